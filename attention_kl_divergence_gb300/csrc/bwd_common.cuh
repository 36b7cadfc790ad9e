// bwd_common.cuh -- helpers shared by the backward kernels (bwd.cu, bwd_decode.cu):
// bounded waits, the dS formulas of both settings, the per-row constants and
// the stores of dS (as hi + lo bf16 terms) and of the gradients.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace streamkl {

namespace {

constexpr int kBwdTile = 64;  // the inner (streamed) tile of both backward kernels
// Bound of the waits that let in-flight TMA copies and MMAs retire before a CTA
// exits (independent of the caller's wait limit).
constexpr uint64_t kDrainNs = 200000000ull;

__device__ __noinline__ bool drain_wait_b(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t code) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, w, code));
}

// dS for one (query, key) pair from the raw dot products z1, z2.
//   la = LSE1 * log2(e);  xb = LSE2 * log2(e) (setting 1) or LSE1 - LSE2 + KL (setting 2)
template <int SETTING>
__device__ __forceinline__ float dscore(float z1, float z2, float c, float scale, float la, float xb, float g) {
    const float p1 = ex2(fmaf(z1, c, -la));
    if (SETTING == 1) {
        const float p2 = ex2(fmaf(z2, c, -xb));
        return g * (p2 - p1);
    } else {
        return g * p1 * fmaf(scale, z1 - z2, -xb);
    }
}

// dS for two queries of one key, FP32x2: nla = -la, nxb = -xb, gs = g * scale
// (the softmax scale of both gradient GEMMs applied here once).
template <int SETTING>
__device__ __forceinline__ float2 dscore2(float2 z1, float2 z2, float2 cc, float2 sc, float2 nla, float2 nxb,
                                          float2 gs) {
    const float2 x1 = __ffma2_rn(z1, cc, nla);
    const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
    if (SETTING == 1) {
        const float2 x2 = __ffma2_rn(z2, cc, nxb);
        const float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
        return __fmul2_rn(gs, __ffma2_rn(p1, make_float2(-1.f, -1.f), p2));  // g s (p2 - p1)
    } else {
        const float2 df = __ffma2_rn(z2, make_float2(-1.f, -1.f), z1);  // z1 - z2
        return __fmul2_rn(__fmul2_rn(gs, p1), __ffma2_rn(df, sc, nxb));  // g s p1 (scale (z1 - z2) - xb)
    }
}

// Per-row constants of the recompute, for row `row` (flat into [B*H*Nq]).
template <int SETTING>
__device__ __forceinline__ void row_constants(const BwdParams& p, size_t row, bool valid, float& la, float& xb,
                                              float& g) {
    constexpr float kLog2e = 1.4426950408889634f;
    if (!valid) {
        la = xb = g = 0.f;
        return;
    }
    const float l1 = p.LSE1[row], l2 = p.LSE2[row];
    la = l1 * kLog2e;
    xb = SETTING == 1 ? l2 * kLog2e : (l1 - l2) + p.KL[row];
    g = p.g[row];
}

// Per-row constants of the joint recompute (both settings at once):
//   la = LSE1 * log2(e), lb = LSE2 * log2(e), xb = LSE1 - LSE2 + KL, g.
__device__ __forceinline__ void row_constants_joint(const BwdParams& p, size_t row, bool valid, float& la,
                                                    float& lb, float& xb, float& g) {
    constexpr float kLog2e = 1.4426950408889634f;
    if (!valid) {
        la = lb = xb = g = 0.f;
        return;
    }
    const float l1 = p.LSE1[row], l2 = p.LSE2[row];
    la = l1 * kLog2e;
    lb = l2 * kLog2e;
    xb = (l1 - l2) + p.KL[row];
    g = p.g[row];
}

// dS of both settings for two pairs from one recompute, FP32x2:
//   d1 = g s P1 (s (z1 - z2) - xb)   setting 2: gradients to the teacher
//   d2 = g s (P2 - P1)               setting 1: gradients to the student
// with nla = -la, nlb = -lb, nxb = -xb, gs = g * scale.
__device__ __forceinline__ void dscore_joint2(float2 z1, float2 z2, float2 cc, float2 sc, float2 nla, float2 nlb,
                                              float2 nxb, float2 gs, float2& d1, float2& d2) {
    const float2 neg = make_float2(-1.f, -1.f);
    const float2 x1 = __ffma2_rn(z1, cc, nla);
    const float2 x2 = __ffma2_rn(z2, cc, nlb);
    const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
    const float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
    d2 = __fmul2_rn(gs, __ffma2_rn(p1, neg, p2));
    const float2 df = __ffma2_rn(z2, neg, z1);
    d1 = __fmul2_rn(__fmul2_rn(gs, p1), __ffma2_rn(df, sc, nxb));
}

// Write 32 dS values as two bf16 terms, hi = bf16(v) and lo = bf16(v - hi),
// each as four 16-byte chunks of a 128-byte swizzled row of its own tile.
// The gradient GEMMs consume hi and lo with the same other operand, so dS
// enters them with ~16 significant bits instead of bf16's 8.
__device__ __forceinline__ void store_ds_chunk(uint32_t tile_hi, uint32_t tile_lo, int row, int chunk0,
                                               const float (&v)[32]) {
    const uint32_t roff = row * 128;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float a = v[cc * 8 + 2 * k], b = v[cc * 8 + 2 * k + 1];
            hi[k] = pack_bf16(a, b);
            const float2 h = make_float2(__uint_as_float(hi[k] << 16), __uint_as_float(hi[k] & 0xffff0000u));
            const float2 r = __ffma2_rn(h, make_float2(-1.f, -1.f), make_float2(a, b));  // exact: v - bf16(v)
            lo[k] = pack_bf16(r.x, r.y);
        }
        const uint32_t off = roff + (((chunk0 + cc) ^ (row & 7)) << 4);
        st_shared_v4(tile_hi + off, hi[0], hi[1], hi[2], hi[3]);
        st_shared_v4(tile_lo + off, lo[0], lo[1], lo[2], lo[3]);
    }
}

// Store 32 gradient values (scaled) at columns [c0, c0 + 32) of a row, as
// float32 or as bf16 (round to nearest even).  Each thread writes its own
// row, so a warp's store instruction touches 32 rows: whole 32-byte sectors
// (when the row is 32-byte aligned) keep those writes sector-sized.
__device__ __forceinline__ void store_grad32(void* row, int c0, const float (&v)[32], float scale, bool bf16) {
    if (bf16) {
        uint16_t* out = reinterpret_cast<uint16_t*>(row) + c0;
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pack_bf16(v[2 * e] * scale, v[2 * e + 1] * scale);
        if ((reinterpret_cast<uintptr_t>(out) & 31u) == 0) {
            st_global_v8(out, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            st_global_v8(out + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
        } else {
            uint4* o4 = reinterpret_cast<uint4*>(out);
#pragma unroll
            for (int e = 0; e < 4; ++e) o4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
    } else {
        float* out = reinterpret_cast<float*>(row) + c0;
        if ((reinterpret_cast<uintptr_t>(out) & 31u) == 0) {
#pragma unroll
            for (int e = 0; e < 32; e += 8)
                st_global_v8(out + e, __float_as_uint(v[e] * scale), __float_as_uint(v[e + 1] * scale),
                             __float_as_uint(v[e + 2] * scale), __float_as_uint(v[e + 3] * scale),
                             __float_as_uint(v[e + 4] * scale), __float_as_uint(v[e + 5] * scale),
                             __float_as_uint(v[e + 6] * scale), __float_as_uint(v[e + 7] * scale));
        } else {
            float4* o4 = reinterpret_cast<float4*>(out);
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                o4[e / 4] = make_float4(v[e] * scale, v[e + 1] * scale, v[e + 2] * scale, v[e + 3] * scale);
        }
    }
}

}  // namespace

}  // namespace streamkl

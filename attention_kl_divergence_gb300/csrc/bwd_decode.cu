// bwd_decode.cu -- backward for few query rows per key head (at most 16 after
// packing the query heads that share a key head), on sm_103a.
//
// Method: "StreamKL: Fast and Memory-Efficient KL Divergence for Boosting
// Attention Distillation" (gist.science/paper/2606.20005, technical summary),
// Methodology 2 (recompute P_t = exp(S_t - LSE_t); dS of setting 1 or 2; dQ =
// scale dS K, dK = scale dS^T Q) with the key range split across CTAs as in
// Methodology 3's Split-K.  With 16 query rows a key tile carries almost no
// arithmetic, and the backward is bound by streaming K1, K2 in and dK out.
//
//   bwd_decode_kernel  one CTA per (batch, key head, key range): keys on the
//     MMA M side (128 keys x 16 query columns, like the decode forward).  Per
//     128-key tile: S1^T, S2^T (TMEM); dS^T as bf16 hi + lo in shared memory;
//     dK = dS^T Q_t (two K = 16 MMAs: hi, lo) written out by the update warps;
//     dQ^T = K_t^T dS^T (M = features, N = 32: hi | lo) accumulated in TMEM
//     over the CTA's key range and added into dQ once at the end.
#include <climits>

#include "bwd_common.cuh"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace streamkl {

namespace {

// Shared memory: the packed query tiles (16 rows), a ring of key stages, one
// dS^T tile (hi in columns 0-15, lo in 16-31 of 128-byte swizzled rows), a zero
// atom that pads the dQ^T MMA to M = 128 when d = 64, per-column constants.
template <int D, int NST>
struct DecBwdSmem {
    static constexpr int NQ = kDecodeMaxQ;
    static constexpr int kQBytes = NQ * D * 2;
    static constexpr int kKBytes = kBlockK * D * 2;
    static constexpr int kDsBytes = kBlockK * 128;  // 128 keys x 64 bf16 columns (32 used)
    static constexpr int q1 = 0;
    static constexpr int q2 = ((kQBytes + 1023) / 1024) * 1024;
    static constexpr int k = 2 * q2;  // stage s: K1 at k + 2*s*kKBytes, K2 right after
    static constexpr int ds = k + 2 * NST * kKBytes;
    static constexpr int zero = ds + kDsBytes;
    static constexpr int kZeroBytes = D < 128 ? kBlockK * 128 : 0;
    static constexpr int vec = zero + kZeroBytes;  // [3][16] floats: -la, -xb, g * scale per column
    static constexpr int bars = vec + 3 * NQ * 4;
    static constexpr int bar_q = bars;
    static constexpr int bar_kfull = bar_q + 8;
    static constexpr int bar_kempty = bar_kfull + 8 * NST;
    static constexpr int bar_sfull = bar_kempty + 8 * NST;  // [2]
    static constexpr int bar_sempty = bar_sfull + 16;        // [2]
    static constexpr int bar_dsfull = bar_sempty + 16;
    static constexpr int bar_dsempty = bar_dsfull + 8;
    static constexpr int bar_dkfull = bar_dsempty + 8;       // [2]
    static constexpr int bar_dkempty = bar_dkfull + 16;      // [2]
    static constexpr int bar_dqfull = bar_dkempty + 16;
    static constexpr int bar_done = bar_dqfull + 8;
    static constexpr int misc = bar_done + 8;  // tmem base (4 B), abort flag (4 B)
    static constexpr int total = misc + 16;
    static constexpr int alloc = total + 1024;  // slack for 1024-byte alignment
};

// TMEM columns: S buffers (S1 | S2, 16 columns each), dK accumulators, dQ^T (hi | lo).
constexpr uint32_t kDecTs = 0, kDecTdk = 128, kDecTdq = 384;

template <int D, int NST, int SETTING>
__global__ void __launch_bounds__(192, 1)
    bwd_decode_kernel(const __grid_constant__ CUtensorMap tQ1, const __grid_constant__ CUtensorMap tK1,
                      const __grid_constant__ CUtensorMap tQ2, const __grid_constant__ CUtensorMap tK2,
                      const BwdParams p) {
    using L = DecBwdSmem<D, NST>;
    constexpr int NQ = L::NQ;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_u32(smem_raw));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::misc + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::misc);
    float* vec = reinterpret_cast<float*>(gbase + L::vec);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // (batch, key head, key range); all query heads of the key head are packed
    // into the 16 query columns: column q is query row q % Nq of head h0 + q / Nq
    const int hp = p.kv_group;
    const int nq = hp * p.Nq;
    const int bkv = blockIdx.x / p.num_splits;
    const int split = blockIdx.x - bkv * p.num_splits;
    const int b = bkv / p.H_kv, hk = bkv - b * p.H_kv;
    const int h0 = hk * p.kv_group;
    const size_t row0 = (static_cast<size_t>(b) * p.H + h0) * p.Nq;  // flat row of column 0
    const int per_split = (p.num_k_tiles + p.num_splits - 1) / p.num_splits;
    const int kt_begin = split * per_split;
    const int n_tiles = max(0, min(p.num_k_tiles, kt_begin + per_split) - kt_begin);
    const uint32_t kt_off = SETTING == 1 ? L::kKBytes : 0u;  // trainable keys within a stage
    const uint32_t qt = base + (SETTING == 1 ? L::q2 : L::q1);  // trainable queries

    if (threadIdx.x == 0) {
        mbar_init(base + L::bar_q, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(base + L::bar_kfull + 8 * s, 1);
            mbar_init(base + L::bar_kempty + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(base + L::bar_sfull + 8 * s, 1);
            mbar_init(base + L::bar_sempty + 8 * s, 128);
            mbar_init(base + L::bar_dkfull + 8 * s, 1);
            mbar_init(base + L::bar_dkempty + 8 * s, 128);
        }
        mbar_init(base + L::bar_dsfull, 128);
        mbar_init(base + L::bar_dsempty, 1);
        mbar_init(base + L::bar_dqfull, 1);
        mbar_init(base + L::bar_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    // unused query columns read zeros (the query copies fill only the first nq rows)
    for (int i = threadIdx.x; i < 2 * (D / kSwizzleCols) * (NQ - nq) * 8; i += blockDim.x) {
        const int chunk16 = i & 7, rr = i >> 3;
        const int r = nq + rr % (NQ - nq), tc = rr / (NQ - nq);
        const uint32_t at = base + (tc & 1 ? L::q2 : L::q1) + (tc >> 1) * NQ * 128 + r * 128 + chunk16 * 16;
        st_shared_v4(at, 0u, 0u, 0u, 0u);
    }
    if (L::kZeroBytes > 0)
        for (int i = threadIdx.x; i < L::kZeroBytes / 16; i += blockDim.x)
            st_shared_v4(base + L::zero + 16 * i, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // the tensor core reads these zeros through the async proxy
    // per-column constants; unused columns get g = 0 (their dS is then 0)
    if (threadIdx.x < NQ) {
        const int q = threadIdx.x;
        float la = 0.f, xb = 0.f, g = 0.f;
        if (q < nq) row_constants<SETTING>(p, row0 + q, true, la, xb, g);
        vec[q] = -la;
        vec[NQ + q] = -xb;
        vec[2 * NQ + q] = g * p.scale;
    }
    if (warp == 1) tmem_alloc(base + L::misc, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, p.status, p.wait_ns};

    if (warp == 0) {
        // ------------------------------------------------ TMA
        if (lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&tQ1);
            prefetch_tensormap(&tK1);
            prefetch_tensormap(&tQ2);
            prefetch_tensormap(&tK2);
            const uint64_t once = policy_evict_first();  // every key is read once
            // one box = Nq rows x the group's heads, landing as nq consecutive rows
            mbar_arrive_expect_tx(base + L::bar_q, 2 * nq * D * 2);
#pragma unroll
            for (int c = 0; c < D / kSwizzleCols; ++c) {
                tma_load_4d(base + L::q1 + c * NQ * 128, &tQ1, base + L::bar_q, c * kSwizzleCols, 0, h0, b);
                tma_load_4d(base + L::q2 + c * NQ * 128, &tQ2, base + L::bar_q, c * kSwizzleCols, 0, h0, b);
            }
            int it = 0, s = 0;
            uint32_t ph = 0;
            for (; it < n_tiles; ++it) {
                if (!mbar_wait(base + L::bar_kempty + 8 * s, ph ^ 1, wc, kErrWaitK)) break;
                const uint32_t fb = base + L::bar_kfull + 8 * s;
                mbar_arrive_expect_tx(fb, 2 * L::kKBytes);
                const int k0 = (kt_begin + it) * kBlockK;
                const uint32_t k1s = base + L::k + 2 * s * L::kKBytes, k2s = k1s + L::kKBytes;
#pragma unroll
                for (int c = 0; c < D / kSwizzleCols; ++c) {
                    tma_load_4d_hint(k1s + c * kBlockK * 128, &tK1, fb, c * kSwizzleCols, k0, hk, b, once);
                    tma_load_4d_hint(k2s + c * kBlockK * 128, &tK2, fb, c * kSwizzleCols, k0, hk, b, once);
                }
                if (++s == NST) s = 0, ph ^= 1;
            }
            drain_wait_b(base + L::bar_q, 0, kDrainNs);  // the query tiles' copies have landed
            for (int j = max(0, it - NST); j < it; ++j) {
                drain_wait_b(base + L::bar_kfull + 8 * (j % NST), (j / NST) & 1, kDrainNs);
                if (!*abort_flag) drain_wait_b(base + L::bar_kempty + 8 * (j % NST), (j / NST) & 1, kDrainNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA
        // iteration m issues the scores of tile m, then the gradient MMAs of tile m - 1
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(kBlockK, NQ);          // S^T: 128 keys x 16 columns
            constexpr uint32_t id_dk = idesc_bf16_f32(kBlockK, D, 0, 1);    // dK: 128 keys x d, B MN-major
            constexpr uint32_t id_dq = idesc_bf16_f32(128, 2 * NQ, 1, 1);   // dQ^T: 128 features x (hi | lo)
            const uint32_t dhi = smem_desc_hi();
            const uint32_t q1_lo = smem_desc_lo_k128(base + L::q1), q2_lo = smem_desc_lo_k128(base + L::q2);
            const uint32_t k_lo0 = smem_desc_lo_k128(base + L::k);
            const uint32_t qt_mn = smem_desc_lo_mn128(qt, NQ * 128);               // B of dK: d-atoms 2 KB apart
            const uint32_t ds_k = smem_desc_lo_k128(base + L::ds);                 // A of dK, K = columns
            const uint32_t ds_mn = smem_desc_lo_mn128(base + L::ds, L::kDsBytes);  // B of dQ^T, N = columns
            constexpr uint32_t kStageLo = (2 * L::kKBytes) >> 4, kK2Lo = L::kKBytes >> 4;
            int issued = 0;
            bool started = false;
            // test aid: a wait on a barrier that nothing arrives on (bar_done is
            // only committed on the abort path below) gives up after wait_ns
            const bool stalled = p.inject_stall && blockIdx.x == 0 &&
                                 !mbar_wait(base + L::bar_done, 0, wc, kErrWaitOther);
            if (!stalled && mbar_wait(base + L::bar_q, 0, wc, kErrWaitQ)) {
                tc_fence_after();
                started = true;
                int s = 0, s2 = 0;
                uint32_t kph = 0, k_lo = k_lo0;
                for (int m = 0; m <= n_tiles; ++m) {
                    if (m < n_tiles) {
                        const int buf = m & 1;
                        if (!mbar_wait(base + L::bar_kfull + 8 * s, kph, wc, kErrWaitK)) break;
                        if (!mbar_wait(base + L::bar_sempty + 8 * buf, ((m >> 1) & 1) ^ 1, wc, kErrWaitS)) break;
                        tc_fence_after();
                        const uint32_t d1 = tmem + kDecTs + buf * 2 * NQ, d2 = d1 + NQ;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t ko = ((kk >> 2) * kBlockK * 128 + (kk & 3) * 32) >> 4;
                            const uint32_t qo = ((kk >> 2) * NQ * 128 + (kk & 3) * 32) >> 4;
                            tc_mma_bf16_w(d1, k_lo + ko, dhi, q1_lo + qo, dhi, id_s, kk > 0);
                        }
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t ko = ((kk >> 2) * kBlockK * 128 + (kk & 3) * 32) >> 4;
                            const uint32_t qo = ((kk >> 2) * NQ * 128 + (kk & 3) * 32) >> 4;
                            tc_mma_bf16_w(d2, k_lo + kK2Lo + ko, dhi, q2_lo + qo, dhi, id_s, kk > 0);
                        }
                        tc_commit(base + L::bar_sfull + 8 * buf);
                        if (++s == NST) {
                            s = 0;
                            kph ^= 1;
                            k_lo = k_lo0;
                        } else {
                            k_lo += kStageLo;
                        }
                    }
                    if (m > 0) {
                        const int mm = m - 1, buf = mm & 1;
                        if (!mbar_wait(base + L::bar_dsfull, mm & 1, wc, kErrWaitOther)) break;
                        if (!mbar_wait(base + L::bar_dkempty + 8 * buf, ((mm >> 1) & 1) ^ 1, wc, kErrWaitOther))
                            break;
                        tc_fence_after();
                        // dK = dS^T Q_t: the hi columns (0-15), then the lo columns (16-31), same B
                        const uint32_t tdk = tmem + kDecTdk + buf * 128;
                        tc_mma_bf16_w(tdk, ds_k, dhi, qt_mn, dhi, id_dk, 0u);
                        tc_mma_bf16_w(tdk, ds_k + (32 >> 4), dhi, qt_mn, dhi, id_dk, 1u);
                        tc_commit(base + L::bar_dkfull + 8 * buf);
                        // dQ^T += K_t^T [dS^T_hi | dS^T_lo] over the tile's 128 keys; A = the trainable
                        // key tile MN-major (64-feature atoms: its second block, or the zero atom when d = 64)
                        const uint32_t kt = base + L::k + 2 * s2 * L::kKBytes + kt_off;
                        const uint32_t a_atom = D == 128 ? kBlockK * 128 : base + L::zero - kt;
                        const uint32_t kt_mn = smem_desc_lo_mn128(kt, a_atom);
#pragma unroll
                        for (int kk = 0; kk < kBlockK / 16; ++kk)
                            tc_mma_bf16_w(tmem + kDecTdq, kt_mn + ((kk * 16 * 128) >> 4), dhi,
                                          ds_mn + ((kk * 16 * 128) >> 4), dhi, id_dq, (mm | kk) != 0);
                        tc_commit(base + L::bar_dsempty);
                        tc_commit(base + L::bar_kempty + 8 * s2);
                        if (++s2 == NST) s2 = 0;
                        ++issued;
                    }
                }
                if (issued == n_tiles) tc_commit(base + L::bar_dqfull);
            }
            if (*abort_flag && started) {  // let the issued MMAs retire before TMEM is freed
                tc_commit(base + L::bar_done);
                drain_wait_b(base + L::bar_done, 0, kDrainNs);
            }
        }
    } else {
        // ------------------------------------------------ dS^T, dK out, dQ out
        const int wq = warp & 3;
        const int krow = wq * 32 + lane;  // key within the tile = TMEM lane
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float c = p.scale_log2e;
        const float2 cc = make_float2(c, c), sc2 = make_float2(p.scale, p.scale);
        // query row within its head of each column; unused columns get INT_MIN,
        // below every visibility bound
        int qi[NQ];
        float nla[NQ], nxb[NQ], gs[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            qi[q] = q < nq ? q % p.Nq : INT_MIN;
            nla[q] = vec[q];
            nxb[q] = vec[NQ + q];
            gs[q] = vec[2 * NQ + q];
        }
        const bool bf16 = p.grad_bf16 != 0;
        // dK rows of tile t: scale is already in dS
        auto dk_out = [&](int t) -> bool {
            const int buf = t & 1;
            if (!wait_all(base + L::bar_dkfull + 8 * buf, (t >> 1) & 1, wc, kErrWaitOther)) return false;
            tc_fence_after();
            const int j = (kt_begin + t) * kBlockK + krow;
            void* out = reinterpret_cast<uint8_t*>(p.dK) + (static_cast<size_t>(bkv) * p.Nk + j) * D * (bf16 ? 2 : 4);
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                float v[32];
                tmem_ld32(tl + kDecTdk + buf * 128 + c0, v);
                tc_wait_ld();
                if (j < p.Nk) store_grad32(out, c0, v, 1.0f, bf16);
            }
            tc_fence_before();
            mbar_arrive(base + L::bar_dkempty + 8 * buf);
            return true;
        };
        bool ok = true;
        for (int t = 0; t < n_tiles; ++t) {
            const int buf = t & 1;
            if (!wait_all(base + L::bar_sfull + 8 * buf, (t >> 1) & 1, wc, kErrWaitS)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float z1[NQ], z2[NQ];
            tmem_ld16(tl + kDecTs + buf * 2 * NQ, z1);
            tmem_ld16(tl + kDecTs + buf * 2 * NQ + NQ, z2);
            tc_wait_ld();
            tc_fence_before();
            mbar_arrive(base + L::bar_sempty + 8 * buf);
            const int j = (kt_begin + t) * kBlockK + krow;
            // key j is visible to query row i iff j <= i + diag_off (bottom-right causal)
            const int first_q = p.causal ? j - p.diag_off : INT_MIN + 1;
            const bool key_ok = j < p.Nk;
            float dsv[NQ];
#pragma unroll
            for (int q = 0; q < NQ; q += 2) {
                const float2 d = dscore2<SETTING>(make_float2(z1[q], z1[q + 1]), make_float2(z2[q], z2[q + 1]), cc,
                                                  sc2, make_float2(nla[q], nla[q + 1]),
                                                  make_float2(nxb[q], nxb[q + 1]), make_float2(gs[q], gs[q + 1]));
                dsv[q] = (key_ok && qi[q] >= first_q) ? d.x : 0.f;
                dsv[q + 1] = (key_ok && qi[q + 1] >= first_q) ? d.y : 0.f;
            }
            if (!wait_all(base + L::bar_dsempty, (t & 1) ^ 1, wc, kErrWaitOther)) {
                ok = false;
                break;
            }
            // row krow of the dS^T tile: hi in 16-byte chunks 0-1, lo in chunks 2-3 (128-byte swizzle)
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float a = dsv[2 * k], bb = dsv[2 * k + 1];
                hi[k] = pack_bf16(a, bb);
                const float2 h = make_float2(__uint_as_float(hi[k] << 16), __uint_as_float(hi[k] & 0xffff0000u));
                const float2 r = __ffma2_rn(h, make_float2(-1.f, -1.f), make_float2(a, bb));  // exact: v - bf16(v)
                lo[k] = pack_bf16(r.x, r.y);
            }
            const uint32_t rowa = base + L::ds + krow * 128;
            const int sw = krow & 7;
            st_shared_v4(rowa + ((0 ^ sw) << 4), hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(rowa + ((1 ^ sw) << 4), hi[4], hi[5], hi[6], hi[7]);
            st_shared_v4(rowa + ((2 ^ sw) << 4), lo[0], lo[1], lo[2], lo[3]);
            st_shared_v4(rowa + ((3 ^ sw) << 4), lo[4], lo[5], lo[6], lo[7]);
            fence_proxy_async_smem();
            mbar_arrive(base + L::bar_dsfull);
            if (t > 0 && !dk_out(t - 1)) {
                ok = false;
                break;
            }
        }
        if (ok && n_tiles > 0) ok = dk_out(n_tiles - 1);
        // this CTA's key range's share of dQ, added into dQ (float32)
        if (ok && n_tiles > 0 && wait_all(base + L::bar_dqfull, 0, wc, kErrWaitOther)) {
            tc_fence_after();
            const int f = krow;  // feature = TMEM lane of dQ^T
            float v[32];
            tmem_ld32(tl + kDecTdq, v);
            tc_wait_ld();
            if (f < D) {
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    if (q < nq) red_add_f32(p.dQacc + (row0 + q) * D + f, v[q] + v[NQ + q]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, int SETTING>
cudaError_t launch_dec_impl(const CUtensorMap* maps, const BwdParams& p, int ctas, cudaStream_t st) {
    constexpr int NST = D == 128 ? 3 : 5;
    static_assert(DecBwdSmem<D, NST>::alloc <= 232448, "shared memory");
    auto k = bwd_decode_kernel<D, NST, SETTING>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DecBwdSmem<D, NST>::alloc);
    if (e != cudaSuccess) return e;
    k<<<ctas, 192, DecBwdSmem<D, NST>::alloc, st>>>(maps[0], maps[1], maps[2], maps[3], p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_decode(int d, int setting, const CUtensorMap* maps, const BwdParams& p, int ctas,
                              cudaStream_t stream) {
    if (d == 128) return setting == 1 ? launch_dec_impl<128, 1>(maps, p, ctas, stream)
                                      : launch_dec_impl<128, 2>(maps, p, ctas, stream);
    return setting == 1 ? launch_dec_impl<64, 1>(maps, p, ctas, stream) : launch_dec_impl<64, 2>(maps, p, ctas, stream);
}

}  // namespace streamkl

// bwd_joint.cu -- backward to both sides from one recompute of the scores,
// on sm_103a.
//
// Method: "StreamKL: Fast and Memory-Efficient KL Divergence for Boosting
// Attention Distillation" (gist.science/paper/2606.20005, technical summary),
// Methodology 2: the two settings differentiate the same KL(P1 || P2) through
// P2 (setting 1, student trainable: dS2 = g (P2 - P1)) and through P1
// (setting 2, teacher trainable: dS1 = g P1 ((S1-LSE1) - (S2-LSE2) - KL)).
// When both sides train, both dS come from the same regenerated P1, P2, so
// each kernel here recomputes S1, S2 once and forms both:
//
//   bwd_q_joint_kernel   one 128-row query tile; loops over 64-key tiles;
//                        dQ1 = scale dS1 K1 and dQ2 = scale dS2 K2 in TMEM,
//                        the query tiles in TMEM as the score MMAs' A operand.
//   bwd_kv_joint_kernel  one 128-key tile; loops over 64-row query tiles;
//                        dK1 = scale dS1^T Q1 and dK2 = scale dS2^T Q2 in TMEM.
//
// Tensor memory (512 columns) holds two accumulators per kernel next to the
// scores, so no gradient is added through atomics: every output is written
// once and the results are deterministic.
#include "bwd_common.cuh"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace streamkl {

namespace {

// ---------------------------------------------------------------------------
// bwd_q_joint: CTA = 128 query rows; 64-key tiles (K1 and K2) through a ring.
// Warps: 0 TMA, 1 TMEM + score MMAs, 2-9 recompute/dS (two warpgroups, one
// query row per thread, each taking 32 of the tile's 64 keys), 10 dQ MMAs.
// TMEM: Q1|Q2 as the A operand of the score MMAs (cols 0-127, copied in
// once), S1|S2 (128-255, released as soon as the update warps hold it in
// registers), dQ1 (256-383), dQ2 (384-511).
// Two dS buffers of four tiles each (dS1 hi, lo; dS2 hi, lo); at d = 128 the
// first takes the query tiles' shared memory, free once they are in TMEM.
// ---------------------------------------------------------------------------
template <int D, int NST>
struct QJointSmem {
    static constexpr int kQBytes = kBlockQ * D * 2;    // 128 rows
    static constexpr int kKBytes = kBwdTile * D * 2;   // 64 keys
    static constexpr int kDsBytes = kBlockQ * kBwdTile * 2;
    static constexpr int kDsBuf = 4 * kDsBytes;
    static constexpr bool kOverlay = 2 * kQBytes >= kDsBuf;
    static constexpr int q1 = 0;
    static constexpr int q2 = kQBytes;
    static constexpr int ds0 = kOverlay ? 0 : 2 * kQBytes;
    static constexpr int ds1 = kOverlay ? 2 * kQBytes : ds0 + kDsBuf;
    static constexpr int k = ds1 + kDsBuf;             // stage s: K1 at k + 2*s*kKBytes, K2 right after
    static constexpr int bars = k + 2 * NST * kKBytes;
    static constexpr int bar_q = bars;
    static constexpr int bar_kfull = bar_q + 8;
    static constexpr int bar_kempty = bar_kfull + 8 * NST;
    static constexpr int bar_sfull = bar_kempty + 8 * NST;
    static constexpr int bar_sempty = bar_sfull + 8;
    static constexpr int bar_dsfull = bar_sempty + 8;    // [2]
    static constexpr int bar_dsempty = bar_dsfull + 16;  // [2]
    static constexpr int bar_done = bar_dsempty + 16;
    static constexpr int bar_drain = bar_done + 8;  // the score issuer's own drain on abort
    static constexpr int misc = bar_drain + 8;  // tmem base (4 B), abort flag (4 B)
    static constexpr int total = misc + 16;
    static constexpr int alloc = total + 1024;  // slack for 1024-byte alignment
};

// warp 0 TMA, warp 1 score MMAs (and TMEM), 8 update warps, the dQ-MMA warp last
constexpr int kQJointThreads = 352;

template <int D, int NST>
__global__ void __launch_bounds__(kQJointThreads, 1)
    bwd_q_joint_kernel(const __grid_constant__ CUtensorMap tQ1, const __grid_constant__ CUtensorMap tK1,
                       const __grid_constant__ CUtensorMap tQ2, const __grid_constant__ CUtensorMap tK2,
                       const BwdParams p) {
    using L = QJointSmem<D, NST>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_u32(smem_raw));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::misc + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::misc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // head-major; causal: the heaviest (last) query tiles of a head first
    const int bh = blockIdx.x / p.num_q_tiles;
    const int qi = blockIdx.x - bh * p.num_q_tiles;
    const int qt = p.causal ? (p.num_q_tiles - 1 - qi) : qi;
    const int b = bh / p.H, h = bh - b * p.H;
    const int hk = h / p.kv_group;
    const int q0 = qt * kBlockQ;
    const int q_last = min(q0 + kBlockQ, p.Nq) - 1;
    const int n_tiles = p.causal ? min(p.num_k_tiles, (q_last + p.diag_off) / kBwdTile + 1) : p.num_k_tiles;

    if (threadIdx.x == 0) {
        mbar_init(base + L::bar_q, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(base + L::bar_kfull + 8 * s, 1);
            mbar_init(base + L::bar_kempty + 8 * s, 1);
        }
        mbar_init(base + L::bar_sfull, 1);
        mbar_init(base + L::bar_sempty, 256);
        for (int s = 0; s < 2; ++s) {
            mbar_init(base + L::bar_dsfull + 8 * s, 256);
            mbar_init(base + L::bar_dsempty + 8 * s, 1);
        }
        mbar_init(base + L::bar_done, 1);
        mbar_init(base + L::bar_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(base + L::misc, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, p.status, p.wait_ns};

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&tQ1);
            prefetch_tensormap(&tK1);
            prefetch_tensormap(&tQ2);
            prefetch_tensormap(&tK2);
            const uint64_t keep = policy_evict_last();
            mbar_arrive_expect_tx(base + L::bar_q, 2 * L::kQBytes);
#pragma unroll
            for (int c = 0; c < D / kSwizzleCols; ++c) {
                tma_load_4d(base + L::q1 + c * kBlockQ * 128, &tQ1, base + L::bar_q, c * kSwizzleCols, q0, h, b);
                tma_load_4d(base + L::q2 + c * kBlockQ * 128, &tQ2, base + L::bar_q, c * kSwizzleCols, q0, h, b);
            }
            int it = 0;
            for (; it < n_tiles; ++it) {
                const int s = it % NST;
                if (!mbar_wait(base + L::bar_kempty + 8 * s, ((it / NST) & 1) ^ 1, wc, kErrWaitK)) break;
                const uint32_t fb = base + L::bar_kfull + 8 * s;
                mbar_arrive_expect_tx(fb, 2 * L::kKBytes);
                const int k0 = it * kBwdTile;
                const uint32_t k1s = base + L::k + 2 * s * L::kKBytes, k2s = k1s + L::kKBytes;
#pragma unroll
                for (int c = 0; c < D / kSwizzleCols; ++c) {
                    tma_load_4d_hint(k1s + c * kBwdTile * 128, &tK1, fb, c * kSwizzleCols, k0, hk, b, keep);
                    tma_load_4d_hint(k2s + c * kBwdTile * 128, &tK2, fb, c * kSwizzleCols, k0, hk, b, keep);
                }
            }
            drain_wait_b(base + L::bar_q, 0, kDrainNs);  // the query tiles' copies have landed
            for (int j = max(0, it - NST); j < it; ++j) {
                drain_wait_b(base + L::bar_kfull + 8 * (j % NST), (j / NST) & 1, kDrainNs);
                if (!*abort_flag) drain_wait_b(base + L::bar_kempty + 8 * (j % NST), (j / NST) & 1, kDrainNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ score MMAs
        // Two threads issue the MMAs: this one the scores of tile it, the last
        // warp's first thread the dQ MMAs of earlier tiles, so that a wait or
        // commit in one leaves the tensor pipe to the other's queued work.
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(kBlockQ, kBwdTile);
            const uint32_t t_q = tmem, t_s = tmem + 128;
            bool started = false;
            const uint32_t dhi = smem_desc_hi();
            constexpr uint32_t kStageLo = (2 * L::kKBytes) >> 4, kK2Lo = L::kKBytes >> 4;
            const uint32_t k_lo0 = smem_desc_lo_k128(base + L::k);
            // test aid: a wait on a barrier that nothing arrives on before the end
            const bool stalled = p.inject_stall && blockIdx.x == 0 &&
                                 !mbar_wait(base + L::bar_done, 0, wc, kErrWaitOther);
            if (!stalled && n_tiles > 0 && mbar_wait(base + L::bar_q, 0, wc, kErrWaitQ)) {
                tc_fence_after();
                // the CTA's query tiles become the A operand of every score MMA; the
                // commit after the first score tile also covers these copies, so
                // once that tile is complete their shared memory may be reused
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qo = (kk >> 2) * kBlockQ * 128 + (kk & 3) * 32;
                    tc_cp_128x256b(t_q + kk * 8, smem_desc_k128(base + L::q1 + qo));
                    tc_cp_128x256b(t_q + D / 2 + kk * 8, smem_desc_k128(base + L::q2 + qo));
                }
                started = true;
                int s = 0;
                uint32_t ph = 0, k_lo = k_lo0;
                for (int it = 0; it < n_tiles; ++it) {
                    if (!mbar_wait(base + L::bar_kfull + 8 * s, ph, wc, kErrWaitK)) break;
                    // tile it - 1's scores are in the update warps' registers
                    if (!mbar_wait(base + L::bar_sempty, (it & 1) ^ 1, wc, kErrWaitS)) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ko = ((kk >> 2) * kBwdTile * 128 + (kk & 3) * 32) >> 4;
                        tc_mma_bf16_ta_w(t_s, t_q + kk * 8, k_lo + ko, dhi, id_s, kk > 0);
                    }
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ko = ((kk >> 2) * kBwdTile * 128 + (kk & 3) * 32) >> 4;
                        tc_mma_bf16_ta_w(t_s + 64, t_q + D / 2 + kk * 8, k_lo + kK2Lo + ko, dhi, id_s, kk > 0);
                    }
                    tc_commit(base + L::bar_sfull);
                    if (++s == NST) {
                        s = 0;
                        ph ^= 1;
                        k_lo = k_lo0;
                    } else {
                        k_lo += kStageLo;
                    }
                }
            }
            if (*abort_flag && started) {  // let the issued copies and MMAs retire before TMEM is freed
                tc_commit(base + L::bar_drain);
                drain_wait_b(base + L::bar_drain, 0, kDrainNs);
            }
        }
    } else if (warp == kQJointThreads / 32 - 1) {
        // ------------------------------------------------ dQ MMAs
        // tile it's dS (from the update warps) -> dQ1 += dS1 K1, dQ2 += dS2 K2
        // (each dS = hi + lo); then the tile's dS buffer and key stage are
        // released.  (Tile it's scores finished before its dS existed, so the
        // stage's release also covers the score MMAs that read it.)
        if (lane == 0) {
            constexpr uint32_t id_dq = idesc_bf16_f32(kBlockQ, D, 0, 1);
            const uint32_t t_dq1 = tmem + 256, t_dq2 = tmem + 384;
            const uint32_t dhi = smem_desc_hi();
            constexpr uint32_t kStageLo = (2 * L::kKBytes) >> 4, kK2Lo = L::kKBytes >> 4;
            // B of dQ_t = K_t, MN-major: K1 at the stage, K2 right after it
            const uint32_t kmn_lo0 = smem_desc_lo_mn128(base + L::k, kBwdTile * 128);
            const uint32_t ds_lo[2] = {smem_desc_lo_k128(base + L::ds0), smem_desc_lo_k128(base + L::ds1)};
            int issued = 0, s = 0;
            uint32_t kmn_lo = kmn_lo0;
            for (int it = 0; it < n_tiles; ++it) {
                const int dsb = it & 1;
                if (!mbar_wait(base + L::bar_dsfull + 8 * dsb, (it >> 1) & 1, wc, kErrWaitOther)) break;
                tc_fence_after();
                const uint32_t dl = ds_lo[dsb];
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kBwdTile / 16; ++kk)
                        tc_mma_bf16_w(t_dq1, dl + ((part * L::kDsBytes + kk * 32) >> 4), dhi,
                                      kmn_lo + ((kk * 16 * 128) >> 4), dhi, id_dq, (it | kk | part) != 0);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kBwdTile / 16; ++kk)
                        tc_mma_bf16_w(t_dq2, dl + (((2 + part) * L::kDsBytes + kk * 32) >> 4), dhi,
                                      kmn_lo + kK2Lo + ((kk * 16 * 128) >> 4), dhi, id_dq, (it | kk | part) != 0);
                tc_commit(base + L::bar_dsempty + 8 * dsb);
                tc_commit(base + L::bar_kempty + 8 * s);
                if (++s == NST) {
                    s = 0;
                    kmn_lo = kmn_lo0;
                } else {
                    kmn_lo += kStageLo;
                }
                ++issued;
            }
            if (issued == n_tiles) tc_commit(base + L::bar_done);
            if (*abort_flag && issued > 0) {  // let the issued MMAs retire before TMEM is freed
                tc_commit(base + L::bar_done);
                drain_wait_b(base + L::bar_done, 0, kDrainNs);
            }
        }
    } else {
        // Two warpgroups: warps 2-5 take keys 0-31 of every tile, warps 6-9 keys 32-63.
        const int wg = (warp - 2) >> 2;
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const int i = q0 + row;
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float c = p.scale_log2e;
        const size_t grow = static_cast<size_t>(bh) * p.Nq + i;
        float la, lb, xb, g;
        row_constants_joint(p, grow, i < p.Nq, la, lb, xb, g);
        const float2 cc = make_float2(c, c), sc2 = make_float2(p.scale, p.scale), nla = make_float2(-la, -la),
                     nlb = make_float2(-lb, -lb), nxb = make_float2(-xb, -xb),
                     gs = make_float2(g * p.scale, g * p.scale);
        const int limit = p.causal ? min(i + p.diag_off, p.Nk - 1) : p.Nk - 1;
        bool ok = true;
        for (int it = 0; it < n_tiles; ++it) {
            if (!wait_all(base + L::bar_sfull, it & 1, wc, kErrWaitS)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t t1 = tl + 128 + wg * 32, t2 = t1 + 64;
            float z1[32], z2[32];
            tmem_ld32(t1, z1);
            tmem_ld32(t2, z2);
            tc_wait_ld();
            tc_fence_before();
            mbar_arrive(base + L::bar_sempty);  // the next score tile may overwrite S now
            const int last = limit - (it * kBwdTile + wg * 32);
            float v1[32], v2[32];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                float2 d1, d2;
                dscore_joint2(make_float2(z1[e], z1[e + 1]), make_float2(z2[e], z2[e + 1]), cc, sc2, nla, nlb, nxb,
                              gs, d1, d2);
                v1[e] = d1.x;
                v1[e + 1] = d1.y;
                v2[e] = d2.x;
                v2[e + 1] = d2.y;
            }
            if (last < 31) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e > last) v1[e] = v2[e] = 0.f;
            }
            const int dsb = it & 1;
            if (!wait_all(base + L::bar_dsempty + 8 * dsb, ((it >> 1) & 1) ^ 1, wc, kErrWaitOther)) {
                ok = false;
                break;
            }
            const uint32_t dss = base + (dsb ? L::ds1 : L::ds0);
            store_ds_chunk(dss, dss + L::kDsBytes, row, wg * 4, v1);
            store_ds_chunk(dss + 2 * L::kDsBytes, dss + 3 * L::kDsBytes, row, wg * 4, v2);
            fence_proxy_async_smem();
            mbar_arrive(base + L::bar_dsfull + 8 * dsb);
        }
        // epilogue: dQ1 and dQ2 rows (the scale is in dS); each warpgroup writes half the columns
        if (ok && wait_all(base + L::bar_done, 0, wc, kErrWaitOther)) {
            tc_fence_after();
            const size_t esz = p.grad_bf16 ? 2 : 4;
            void* out1 = reinterpret_cast<uint8_t*>(p.dQ) + grow * D * esz;
            void* out2 = reinterpret_cast<uint8_t*>(p.dQb) + grow * D * esz;
#pragma unroll 1
            for (int c0 = wg * (D / 2); c0 < (wg + 1) * (D / 2); c0 += 32) {
                float v[32];
                tmem_ld32(tl + 256 + c0, v);
                tc_wait_ld();
                if (i < p.Nq) store_grad32(out1, c0, v, 1.0f, p.grad_bf16 != 0);
                tmem_ld32(tl + 384 + c0, v);
                tc_wait_ld();
                if (i < p.Nq) store_grad32(out2, c0, v, 1.0f, p.grad_bf16 != 0);
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

// ---------------------------------------------------------------------------
// bwd_kv_joint: CTA = 128 keys; 64-row query tiles (Q1 and Q2 together)
// through a ring.  Warps: 0 TMA + per-row constants, 1 TMEM + score MMAs,
// 2-9 recompute/dS (two warpgroups, one key per thread, each taking 32 of the
// tile's 64 query rows), 10 gradient MMAs.
// TMEM: K1|K2 as the A operand of the score MMAs (cols 0-127, copied in
// once), S1^T|S2^T (128-255, released as soon as the update warps hold it in
// registers), dK1 (256-383), dK2 (384-511).
// Two dS buffers of four tiles each (dS1 hi, lo; dS2 hi, lo); at d = 128 the
// first takes the key tiles' shared memory, free once they are in TMEM.
// ---------------------------------------------------------------------------
template <int D, int NST>
struct KvJointSmem {
    static constexpr int kKBytes = kBlockK * D * 2;    // 128 keys
    static constexpr int kQBytes = kBwdTile * D * 2;   // 64 query rows of one tensor
    static constexpr int kDsBytes = kBlockK * kBwdTile * 2;
    static constexpr int kDsBuf = 4 * kDsBytes;
    static constexpr bool kOverlay = 2 * kKBytes >= kDsBuf;
    static constexpr int k1 = 0;
    static constexpr int k2 = kKBytes;
    static constexpr int ds0 = kOverlay ? 0 : 2 * kKBytes;
    static constexpr int ds1 = kOverlay ? 2 * kKBytes : ds0 + kDsBuf;
    static constexpr int q = ds1 + kDsBuf;            // slot s: Q1 at q + 2*s*kQBytes, Q2 right after
    static constexpr int kNv = 2;
    static constexpr int vec = q + 2 * NST * kQBytes;  // [kNv][4][64] floats
    static constexpr int bars = vec + kNv * 4 * kBwdTile * 4;
    static constexpr int bar_k = bars;
    static constexpr int bar_qfull = bar_k + 8;
    static constexpr int bar_qempty = bar_qfull + 8 * NST;
    static constexpr int bar_vfull = bar_qempty + 8 * NST;
    static constexpr int bar_vempty = bar_vfull + 8 * kNv;
    static constexpr int bar_sfull = bar_vempty + 8 * kNv;
    static constexpr int bar_sempty = bar_sfull + 8;
    static constexpr int bar_dsfull = bar_sempty + 8;   // [2]
    static constexpr int bar_dsempty = bar_dsfull + 16;  // [2]
    static constexpr int bar_done = bar_dsempty + 16;
    static constexpr int bar_drain = bar_done + 8;  // the score issuer's own drain on abort
    static constexpr int misc = bar_drain + 8;
    static constexpr int total = misc + 16;
    static constexpr int alloc = total;  // no slack: the kernel checks the base is 1024-byte aligned
};

constexpr int kKvJointThreads = 352;

template <int D, int NST>
__global__ void __launch_bounds__(kKvJointThreads, 1)
    bwd_kv_joint_kernel(const __grid_constant__ CUtensorMap tQ1, const __grid_constant__ CUtensorMap tK1,
                        const __grid_constant__ CUtensorMap tQ2, const __grid_constant__ CUtensorMap tK2,
                        const BwdParams p) {
    using L = KvJointSmem<D, NST>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    if (base & 1023u) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, kErrSmemAlign);
        return;
    }
    uint8_t* gbase = smem_raw;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::misc + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::misc);
    float* vec = reinterpret_cast<float*>(gbase + L::vec);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kGradWarp = kKvJointThreads / 32 - 1;

    // head-major; key tile 0 sees the most query rows under a causal mask and
    // comes first; a key head's CTA visits every query tile of each query head
    // of its group, so dK sums the group's gradients
    const int bkv = blockIdx.x / p.num_k_tiles;
    const int nt = blockIdx.x - bkv * p.num_k_tiles;
    const int b = bkv / p.H_kv, hk = bkv - b * p.H_kv;
    const int n0 = nt * kBlockK;
    const int m_start = p.causal ? max(0, (n0 - p.diag_off) / kBwdTile) : 0;
    const int per_head = p.num_q_tiles - m_start;
    const int n_tiles = per_head * p.kv_group;
    auto qhead = [&](int m) { return p.kv_group == 1 ? hk : hk * p.kv_group + m / per_head; };
    auto qtile = [&](int m) { return m_start + (p.kv_group == 1 ? m : m % per_head); };

    if (threadIdx.x == 0) {
        mbar_init(base + L::bar_k, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(base + L::bar_qfull + 8 * s, 1);
            mbar_init(base + L::bar_qempty + 8 * s, 1);
        }
        for (int s = 0; s < L::kNv; ++s) {
            mbar_init(base + L::bar_vfull + 8 * s, 32);
            mbar_init(base + L::bar_vempty + 8 * s, 256);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(base + L::bar_dsfull + 8 * s, 256);
            mbar_init(base + L::bar_dsempty + 8 * s, 1);
        }
        mbar_init(base + L::bar_sfull, 1);
        mbar_init(base + L::bar_sempty, 256);
        mbar_init(base + L::bar_done, 1);
        mbar_init(base + L::bar_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(base + L::misc, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, p.status, p.wait_ns};

    if (warp == 0) {
        // ------------------------------------------------ TMA + row constants
        if (lane == 0) {
            prefetch_tensormap(&tQ1);
            prefetch_tensormap(&tK1);
            prefetch_tensormap(&tQ2);
            prefetch_tensormap(&tK2);
            mbar_arrive_expect_tx(base + L::bar_k, 2 * L::kKBytes);
#pragma unroll
            for (int c = 0; c < D / kSwizzleCols; ++c) {
                tma_load_4d(base + L::k1 + c * kBlockK * 128, &tK1, base + L::bar_k, c * kSwizzleCols, n0, hk, b);
                tma_load_4d(base + L::k2 + c * kBlockK * 128, &tK2, base + L::bar_k, c * kSwizzleCols, n0, hk, b);
            }
        }
        const uint64_t keep = policy_evict_last();
        int n_q = 0;  // query slots whose copies were issued
        int st = 0, sv = 0;
        uint32_t pt = 0, pv = 0;
        for (int m = 0; m < n_tiles; ++m) {
            const int r0 = qtile(m) * kBwdTile;
            const int h = qhead(m);
            if (!wait_all(base + L::bar_qempty + 8 * st, pt ^ 1, wc, kErrWaitOther)) break;
            if (lane == 0) {
                const uint32_t fb = base + L::bar_qfull + 8 * st, dst = base + L::q + 2 * st * L::kQBytes;
                mbar_arrive_expect_tx(fb, 2 * L::kQBytes);
#pragma unroll
                for (int c = 0; c < D / kSwizzleCols; ++c) {
                    tma_load_4d_hint(dst + c * kBwdTile * 128, &tQ1, fb, c * kSwizzleCols, r0, h, b, keep);
                    tma_load_4d_hint(dst + L::kQBytes + c * kBwdTile * 128, &tQ2, fb, c * kSwizzleCols, r0, h, b,
                                     keep);
                }
            }
            ++n_q;
            if (!wait_all(base + L::bar_vempty + 8 * sv, pv ^ 1, wc, kErrWaitOther)) break;
            // per query row: -la, -lb, -xb and g * scale (the softmax scale of the
            // gradients is folded into dS)
            float* v = vec + sv * 4 * kBwdTile;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int r = lane + 32 * k;
                const int i = r0 + r;
                float la, lb, xb, g;
                row_constants_joint(p, (static_cast<size_t>(b) * p.H + h) * p.Nq + i, i < p.Nq, la, lb, xb, g);
                v[r] = -la;
                v[kBwdTile + r] = -lb;
                v[2 * kBwdTile + r] = -xb;
                v[3 * kBwdTile + r] = g * p.scale;
            }
            mbar_arrive(base + L::bar_vfull + 8 * sv);
            if (++st == NST) st = 0, pt ^= 1;
            if (++sv == L::kNv) sv = 0, pv ^= 1;
        }
        if (lane == 0) {  // every issued copy has landed (and, unless aborting, been consumed)
            drain_wait_b(base + L::bar_k, 0, kDrainNs);
            for (int j = max(0, n_q - NST); j < n_q; ++j) {
                const uint32_t bo = 8 * (j % NST), ph = (j / NST) & 1;
                drain_wait_b(base + L::bar_qfull + bo, ph, kDrainNs);
                if (!*abort_flag) drain_wait_b(base + L::bar_qempty + bo, ph, kDrainNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ score MMAs
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(kBlockK, kBwdTile);
            const uint32_t t_k = tmem, t_s = tmem + 128;
            bool started = false;
            const bool stalled = p.inject_stall && blockIdx.x == 0 &&
                                 !mbar_wait(base + L::bar_done, 0, wc, kErrWaitOther);
            if (!stalled && n_tiles > 0 && mbar_wait(base + L::bar_k, 0, wc, kErrWaitK)) {
                tc_fence_after();
                // the CTA's key tiles become the A operand of every score MMA; the
                // commit after the first score tile also covers these copies, so
                // once that tile is complete their shared memory may be reused
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ko = (kk >> 2) * kBlockK * 128 + (kk & 3) * 32;
                    tc_cp_128x256b(t_k + kk * 8, smem_desc_k128(base + L::k1 + ko));
                    tc_cp_128x256b(t_k + D / 2 + kk * 8, smem_desc_k128(base + L::k2 + ko));
                }
                started = true;
                const uint32_t dhi = smem_desc_hi();
                constexpr uint32_t kSlotLo = (2 * L::kQBytes) >> 4, kQ2Lo = L::kQBytes >> 4;
                const uint32_t q_lo0 = smem_desc_lo_k128(base + L::q);
                int st = 0;
                uint32_t pt = 0, q_lo = q_lo0;
                for (int m = 0; m < n_tiles; ++m) {
                    if (!mbar_wait(base + L::bar_qfull + 8 * st, pt, wc, kErrWaitQ)) break;
                    if (!mbar_wait(base + L::bar_sempty, (m & 1) ^ 1, wc, kErrWaitS)) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t qo = ((kk >> 2) * kBwdTile * 128 + (kk & 3) * 32) >> 4;
                        tc_mma_bf16_ta_w(t_s, t_k + kk * 8, q_lo + qo, dhi, id_s, kk > 0);
                    }
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t qo = ((kk >> 2) * kBwdTile * 128 + (kk & 3) * 32) >> 4;
                        tc_mma_bf16_ta_w(t_s + 64, t_k + D / 2 + kk * 8, q_lo + kQ2Lo + qo, dhi, id_s, kk > 0);
                    }
                    tc_commit(base + L::bar_sfull);
                    if (++st == NST) {
                        st = 0;
                        pt ^= 1;
                        q_lo = q_lo0;
                    } else {
                        q_lo += kSlotLo;
                    }
                }
            }
            if (*abort_flag && started) {  // let the issued copies and MMAs retire before TMEM is freed
                tc_commit(base + L::bar_drain);
                drain_wait_b(base + L::bar_drain, 0, kDrainNs);
            }
        }
    } else if (warp == kGradWarp) {
        // ------------------------------------------------ gradient MMAs
        // dK1 += dS1^T Q1 and dK2 += dS2^T Q2 (A = dS^T K-major over queries,
        // B = the query tile MN-major; each dS = hi + lo), then the tile's dS
        // buffer and query slot are released.
        if (lane == 0) {
            constexpr uint32_t id_dk = idesc_bf16_f32(kBlockK, D, 0, 1);
            const uint32_t t_dk1 = tmem + 256, t_dk2 = tmem + 384;
            const uint32_t dhi = smem_desc_hi();
            constexpr uint32_t kSlotLo = (2 * L::kQBytes) >> 4, kQ2Lo = L::kQBytes >> 4;
            const uint32_t qmn_lo0 = smem_desc_lo_mn128(base + L::q, kBwdTile * 128);
            const uint32_t ds_lo[2] = {smem_desc_lo_k128(base + L::ds0), smem_desc_lo_k128(base + L::ds1)};
            int issued = 0, st = 0;
            uint32_t q_lo = qmn_lo0;
            for (int m = 0; m < n_tiles; ++m) {
                const int dsb = m & 1;
                if (!mbar_wait(base + L::bar_dsfull + 8 * dsb, (m >> 1) & 1, wc, kErrWaitOther)) break;
                tc_fence_after();
                const uint32_t dl = ds_lo[dsb];
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kBwdTile / 16; ++kk)
                        tc_mma_bf16_w(t_dk1, dl + ((part * L::kDsBytes + kk * 32) >> 4), dhi,
                                      q_lo + ((kk * 16 * 128) >> 4), dhi, id_dk, (kk | part | m) != 0);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kBwdTile / 16; ++kk)
                        tc_mma_bf16_w(t_dk2, dl + (((2 + part) * L::kDsBytes + kk * 32) >> 4), dhi,
                                      q_lo + kQ2Lo + ((kk * 16 * 128) >> 4), dhi, id_dk, (kk | part | m) != 0);
                tc_commit(base + L::bar_dsempty + 8 * dsb);
                tc_commit(base + L::bar_qempty + 8 * st);
                if (++st == NST) {
                    st = 0;
                    q_lo = qmn_lo0;
                } else {
                    q_lo += kSlotLo;
                }
                ++issued;
            }
            if (issued == n_tiles) tc_commit(base + L::bar_done);
            if (*abort_flag && issued > 0) {  // let the issued MMAs retire before TMEM is freed
                tc_commit(base + L::bar_done);
                drain_wait_b(base + L::bar_done, 0, kDrainNs);
            }
        }
    } else {
        // ------------------------------------------------ recompute + dS^T of both settings
        const int wg = (warp - 2) >> 2;
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const int j = n0 + row;  // key index
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float c = p.scale_log2e;
        const float2 cc = make_float2(c, c), sc2 = make_float2(p.scale, p.scale);
        const bool key_ok = j < p.Nk;
        bool ok = true;
        for (int m = 0; m < n_tiles; ++m) {
            const int sv = m % L::kNv;
            if (!wait_all(base + L::bar_sfull, m & 1, wc, kErrWaitS) ||
                !wait_all(base + L::bar_vfull + 8 * sv, (m / L::kNv) & 1, wc, kErrWaitQ)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int r0 = qtile(m) * kBwdTile + wg * 32;  // first query row of this chunk
            const uint32_t t1 = tl + 128 + wg * 32, t2 = t1 + 64;
            float z1[32], z2[32];
            tmem_ld32(t1, z1);
            tmem_ld32(t2, z2);
            tc_wait_ld();
            tc_fence_before();
            mbar_arrive(base + L::bar_sempty);  // the next score tile may overwrite S now
            const float4* v4 = reinterpret_cast<const float4*>(vec + sv * 4 * kBwdTile + wg * 32);
            float d1v[32], d2v[32];
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
                const float4 a = v4[e4], bb = v4[kBwdTile / 4 + e4], x = v4[kBwdTile / 2 + e4],
                             gg = v4[3 * kBwdTile / 4 + e4];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int e = 4 * e4 + 2 * k;
                    const float2 nla = k ? make_float2(a.z, a.w) : make_float2(a.x, a.y);
                    const float2 nlb = k ? make_float2(bb.z, bb.w) : make_float2(bb.x, bb.y);
                    const float2 nxb = k ? make_float2(x.z, x.w) : make_float2(x.x, x.y);
                    const float2 gs = k ? make_float2(gg.z, gg.w) : make_float2(gg.x, gg.y);
                    float2 d1, d2;
                    dscore_joint2(make_float2(z1[e], z1[e + 1]), make_float2(z2[e], z2[e + 1]), cc, sc2, nla, nlb,
                                  nxb, gs, d1, d2);
                    d1v[e] = d1.x;
                    d1v[e + 1] = d1.y;
                    d2v[e] = d2.x;
                    d2v[e + 1] = d2.y;
                }
            }
            mbar_arrive(base + L::bar_vempty + 8 * sv);
            // query i = r0 + e sees key j iff j <= i + diag_off; keys past Nk contribute nothing
            const int first = p.causal ? (j - p.diag_off) - r0 : -1;
            if (first > 0 || !key_ok) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e < first || !key_ok) d1v[e] = d2v[e] = 0.f;
            }
            const int dsb = m & 1;
            if (!wait_all(base + L::bar_dsempty + 8 * dsb, ((m >> 1) & 1) ^ 1, wc, kErrWaitOther)) {
                ok = false;
                break;
            }
            const uint32_t dss = base + (dsb ? L::ds1 : L::ds0);
            store_ds_chunk(dss, dss + L::kDsBytes, row, wg * 4, d1v);
            store_ds_chunk(dss + 2 * L::kDsBytes, dss + 3 * L::kDsBytes, row, wg * 4, d2v);
            fence_proxy_async_smem();
            mbar_arrive(base + L::bar_dsfull + 8 * dsb);
        }
        // epilogue: dK1 and dK2 rows (the scale is in dS); each warpgroup writes half the columns
        if (ok && wait_all(base + L::bar_done, 0, wc, kErrWaitOther)) {
            tc_fence_after();
            const size_t esz = p.grad_bf16 ? 2 : 4;
            const size_t krow = static_cast<size_t>(bkv) * p.Nk + j;
            void* out1 = reinterpret_cast<uint8_t*>(p.dK) + krow * D * esz;
            void* out2 = reinterpret_cast<uint8_t*>(p.dKb) + krow * D * esz;
#pragma unroll 1
            for (int c0 = wg * (D / 2); c0 < (wg + 1) * (D / 2); c0 += 32) {
                float v[32];
                tmem_ld32(tl + 256 + c0, v);
                tc_wait_ld();
                if (key_ok) store_grad32(out1, c0, v, 1.0f, p.grad_bf16 != 0);
                tmem_ld32(tl + 384 + c0, v);
                tc_wait_ld();
                if (key_ok) store_grad32(out2, c0, v, 1.0f, p.grad_bf16 != 0);
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

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D>
cudaError_t launch_joint_impl(const CUtensorMap* qm, const CUtensorMap* kvm, const BwdParams& pq,
                              const BwdParams& pkv, int ctas_q, int ctas_kv, cudaStream_t st) {
    constexpr int NQ = D == 128 ? 3 : 4;
    constexpr int NKV = D == 128 ? 3 : 4;
    static_assert(QJointSmem<D, NQ>::alloc <= 232448, "shared memory");
    static_assert(KvJointSmem<D, NKV>::alloc <= 232448, "shared memory");
    auto kq = bwd_q_joint_kernel<D, NQ>;
    auto kkv = bwd_kv_joint_kernel<D, NKV>;
    cudaError_t e = set_smem(kq, QJointSmem<D, NQ>::alloc);
    if (e != cudaSuccess) return e;
    if ((e = set_smem(kkv, KvJointSmem<D, NKV>::alloc)) != cudaSuccess) return e;
    kq<<<ctas_q, kQJointThreads, QJointSmem<D, NQ>::alloc, st>>>(qm[0], qm[1], qm[2], qm[3], pq);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kkv<<<ctas_kv, kKvJointThreads, KvJointSmem<D, NKV>::alloc, st>>>(kvm[0], kvm[1], kvm[2], kvm[3], pkv);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_joint(int d, const CUtensorMap* qmaps, const CUtensorMap* kvmaps, const BwdParams& pq,
                             const BwdParams& pkv, int ctas_q, int ctas_kv, cudaStream_t stream) {
    if (d == 128) return launch_joint_impl<128>(qmaps, kvmaps, pq, pkv, ctas_q, ctas_kv, stream);
    return launch_joint_impl<64>(qmaps, kvmaps, pq, pkv, ctas_q, ctas_kv, stream);
}

}  // namespace streamkl

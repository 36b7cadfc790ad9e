// bwd.cu -- backward kernels of the attention KL divergence on sm_103a.
//
// Method: "StreamKL: Fast and Memory-Efficient KL Divergence for Boosting
// Attention Distillation" (gist.science/paper/2606.20005, technical summary),
// Methodology 2: the probabilities are regenerated tile by tile from the saved
// log-sum-exps, P_t = exp(S_t - LSE_t), and the gradient of sum_i g_i KL_i is
//   setting 1 (teacher fixed, student trainable): dS2 = g (P2 - P1)
//   setting 2 (student fixed, teacher trainable): dS1 = g P1 ((S1-LSE1) - (S2-LSE2) - KL)
// (the log-ratio taken from logit differences and the saved LSEs), followed by
//   dQ_t = scale * dS K_t,   dK_t = scale * dS^T Q_t   for the trainable side t.
//
//   bwd_q_kernel   one 128-row query tile; loops over 64-key tiles; dQ in TMEM.
//   bwd_kv_kernel  one 128-key tile; loops over 64-row query tiles; dK in TMEM.
//                  FUSED also forms dQ^T = K_t^T dS^T per tile pair and adds it
//                  to global dQ with bulk L2 reductions (each QK tile pair
//                  visited once).
// The split mode runs both kernels (each recomputes the scores); the fused
// mode runs bwd_kv_kernel<FUSED> alone after zeroing dQ.
#include <algorithm>

#include "bwd_common.cuh"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace streamkl {

namespace {

// ---------------------------------------------------------------------------
// bwd_q: CTA = 128 query rows; 64-key tiles streamed through a 3-stage ring.
// Warps: 0 TMA, 1 TMEM + MMA, 2-9 recompute/dS (two warpgroups, one query row
// per thread, each taking 32 of the tile's 64 keys).
// TMEM: S1|S2 double buffered (cols 0-255), dQ accumulator (cols 256-383).
// ---------------------------------------------------------------------------
template <int D, int NST>
struct QSmem {
    static constexpr int kQBytes = kBlockQ * D * 2;    // 128 rows
    static constexpr int kKBytes = kBwdTile * D * 2;   // 64 rows
    static constexpr int kDsBytes = kBlockQ * kBwdTile * 2;
    static constexpr int q1 = 0;
    static constexpr int q2 = kQBytes;
    static constexpr int k = 2 * kQBytes;
    static constexpr int kNumDs = 1;                  // dS buffers: the update computes before it stores
    static constexpr int ds = k + 2 * NST * kKBytes;  // buffer b: hi at ds + 2*b*kDsBytes, lo right after
    static constexpr int bars = ds + 2 * kNumDs * kDsBytes;
    static constexpr int bar_q = bars;
    static constexpr int bar_kfull = bar_q + 8;
    static constexpr int bar_kempty = bar_kfull + 8 * NST;
    static constexpr int bar_sfull = bar_kempty + 8 * NST;
    static constexpr int bar_sempty = bar_sfull + 16;
    static constexpr int bar_dsfull = bar_sempty + 16;
    static constexpr int bar_dsempty = bar_dsfull + 16;
    static constexpr int bar_done = bar_dsempty + 16;
    static constexpr int misc = bar_done + 8;
    static constexpr int total = misc + 16;
    static constexpr int alloc = total + 1024;
};

template <int D, int NST, int SETTING>
__global__ void __launch_bounds__(320, 1)
    bwd_q_kernel(const __grid_constant__ CUtensorMap tQ1, const __grid_constant__ CUtensorMap tK1,
                 const __grid_constant__ CUtensorMap tQ2, const __grid_constant__ CUtensorMap tK2,
                 const BwdParams p) {
    using L = QSmem<D, NST>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_u32(smem_raw));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::misc + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::misc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // head-major: resident CTAs share one head's key tiles through L2; causal:
    // the heaviest (last) query tiles of a head first
    const int bh = blockIdx.x / p.num_q_tiles;
    const int qi = blockIdx.x - bh * p.num_q_tiles;
    const int qt = p.causal ? (p.num_q_tiles - 1 - qi) : qi;
    const int b = bh / p.H, h = bh - b * p.H;
    const int hk = h / p.kv_group;  // key head (shared by kv_group query heads)
    const int q0 = qt * kBlockQ;
    const int q_last = min(q0 + kBlockQ, p.Nq) - 1;
    const int n_tiles = p.causal ? min(p.num_k_tiles, (q_last + p.diag_off) / kBwdTile + 1) : p.num_k_tiles;
    // trainable side: setting 1 -> student (Q2, K2), setting 2 -> teacher (Q1, K1)
    const uint32_t kt_off = SETTING == 1 ? L::kKBytes : 0;

    if (threadIdx.x == 0) {
        mbar_init(base + L::bar_q, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(base + L::bar_kfull + 8 * s, 1);
            mbar_init(base + L::bar_kempty + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(base + L::bar_sfull + 8 * s, 1);
            mbar_init(base + L::bar_sempty + 8 * s, 256);
            mbar_init(base + L::bar_dsfull + 8 * s, 256);
            mbar_init(base + L::bar_dsempty + 8 * s, 1);
        }
        mbar_init(base + L::bar_done, 1);
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
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(kBlockQ, kBwdTile);
            constexpr uint32_t id_dq = idesc_bf16_f32(kBlockQ, D, 0, 1);
            const uint32_t t_dq = tmem + 256;
            int issued = 0;
            bool started = false;
            // few instructions per MMA: descriptor low words advance by compile-time
            // offsets (the high word is one constant); ring positions are counters
            const uint32_t dhi = smem_desc_hi();
            constexpr uint32_t kStageLo = (2 * L::kKBytes) >> 4, kK2Lo = L::kKBytes >> 4;
            const uint32_t q1_lo = smem_desc_lo_k128(base + L::q1), q2_lo = smem_desc_lo_k128(base + L::q2);
            const uint32_t k_lo0 = smem_desc_lo_k128(base + L::k);
            const uint32_t kt_lo0 = smem_desc_lo_mn128(base + L::k + kt_off, kBwdTile * 128);
            const uint32_t ds_lo = smem_desc_lo_k128(base + L::ds);
            static_assert(L::kNumDs == 1, "one dS buffer");
            auto issue_s = [&](int buf, uint32_t k_lo) {
                const uint32_t d1 = tmem + buf * 128, d2 = d1 + 64;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qo = ((kk >> 2) * kBlockQ * 128 + (kk & 3) * 32) >> 4;
                    const uint32_t ko = ((kk >> 2) * kBwdTile * 128 + (kk & 3) * 32) >> 4;
                    tc_mma_bf16_w(d1, q1_lo + qo, dhi, k_lo + ko, dhi, id_s, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qo = ((kk >> 2) * kBlockQ * 128 + (kk & 3) * 32) >> 4;
                    const uint32_t ko = ((kk >> 2) * kBwdTile * 128 + (kk & 3) * 32) >> 4;
                    tc_mma_bf16_w(d2, q2_lo + qo, dhi, k_lo + kK2Lo + ko, dhi, id_s, kk > 0);
                }
                tc_commit(base + L::bar_sfull + 8 * buf);
            };
            // test aid: a wait on a barrier that nothing arrives on before the end
            const bool stalled = p.inject_stall && blockIdx.x == 0 &&
                                 !mbar_wait(base + L::bar_done, 0, wc, kErrWaitOther);
            bool ok = !stalled && mbar_wait(base + L::bar_q, 0, wc, kErrWaitQ) &&
                      mbar_wait(base + L::bar_kfull, 0, wc, kErrWaitK);
            if (ok) {
                tc_fence_after();
                issue_s(0, k_lo0);
                started = true;
                int sn = NST > 1 ? 1 : 0, s = 0;    // stages of tiles it + 1 and it
                uint32_t pn = NST > 1 ? 0 : 1;      // phase of tile it + 1's stage
                for (int it = 0; it < n_tiles; ++it) {
                    if (it + 1 < n_tiles) {
                        const int n1 = it + 1;
                        if (!mbar_wait(base + L::bar_kfull + 8 * sn, pn, wc, kErrWaitK)) break;
                        if (!mbar_wait(base + L::bar_sempty + 8 * (n1 & 1), ((n1 >> 1) & 1) ^ 1, wc, kErrWaitS))
                            break;
                        tc_fence_after();
                        issue_s(n1 & 1, k_lo0 + sn * kStageLo);
                        if (++sn == NST) sn = 0, pn ^= 1;
                    }
                    if (!mbar_wait(base + L::bar_dsfull, it & 1, wc, kErrWaitOther)) break;
                    tc_fence_after();
                    const uint32_t kt_lo = kt_lo0 + s * kStageLo;
#pragma unroll
                    for (int part = 0; part < 2; ++part)  // dS = hi + lo
#pragma unroll
                        for (int kk = 0; kk < kBwdTile / 16; ++kk)
                            tc_mma_bf16_w(t_dq, ds_lo + ((part * L::kDsBytes + kk * 32) >> 4), dhi,
                                          kt_lo + ((kk * 16 * 128) >> 4), dhi, id_dq, (it | kk | part) != 0);
                    tc_commit(base + L::bar_dsempty);
                    tc_commit(base + L::bar_kempty + 8 * s);
                    if (++s == NST) s = 0;
                    ++issued;
                }
                if (issued == n_tiles) tc_commit(base + L::bar_done);
            }
            if (*abort_flag && started) {  // let the issued MMAs retire before TMEM is freed
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
        float la, xb, g;
        row_constants<SETTING>(p, grow, i < p.Nq, la, xb, g);
        // the row's constants as FP32x2 pairs; the softmax scale of dQ is folded into g
        const float2 cc = make_float2(c, c), sc2 = make_float2(p.scale, p.scale), nla = make_float2(-la, -la),
                     nxb = make_float2(-xb, -xb), gs = make_float2(g * p.scale, g * p.scale);
        const int limit = p.causal ? min(i + p.diag_off, p.Nk - 1) : p.Nk - 1;
        bool ok = true;
        for (int it = 0; it < n_tiles; ++it) {
            const int buf = it & 1;
            if (!wait_all(base + L::bar_sfull + 8 * buf, (it >> 1) & 1, wc, kErrWaitS)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t t1 = tl + buf * 128 + wg * 32, t2 = t1 + 64;
            const int dsb = it % L::kNumDs;
            const uint32_t dss = base + L::ds + 2 * dsb * L::kDsBytes;
            float z1[32], z2[32];
            tmem_ld32(t1, z1);
            tmem_ld32(t2, z2);
            tc_wait_ld();
            tc_fence_before();
            mbar_arrive(base + L::bar_sempty + 8 * buf);
            const int last = limit - (it * kBwdTile + wg * 32);
            float v[32];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const float2 d = dscore2<SETTING>(make_float2(z1[e], z1[e + 1]), make_float2(z2[e], z2[e + 1]), cc,
                                                  sc2, nla, nxb, gs);
                v[e] = d.x;
                v[e + 1] = d.y;
            }
            if (last < 31) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e > last) v[e] = 0.f;
            }
            if (!wait_all(base + L::bar_dsempty + 8 * dsb, ((it / L::kNumDs) & 1) ^ 1, wc, kErrWaitOther)) {
                ok = false;
                break;
            }
            store_ds_chunk(dss, dss + L::kDsBytes, row, wg * 4, v);
            fence_proxy_async_smem();
            mbar_arrive(base + L::bar_dsfull + 8 * dsb);
        }
        // epilogue: dQ row = scale * accumulator; each warpgroup writes half the columns
        if (ok && wait_all(base + L::bar_done, 0, wc, kErrWaitOther)) {
            tc_fence_after();
            void* out = reinterpret_cast<uint8_t*>(p.dQ) + grow * D * (p.grad_bf16 ? 2 : 4);
#pragma unroll 1
            for (int c0 = wg * (D / 2); c0 < (wg + 1) * (D / 2); c0 += 32) {
                float v[32];
                tmem_ld32(tl + 256 + c0, v);
                tc_wait_ld();
                if (i < p.Nq) store_grad32(out, c0, v, 1.0f, p.grad_bf16 != 0);  // the scale is in dS
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
// bwd_kv: CTA = 128 keys; 64-row query tiles streamed through a 3-stage ring.
// Warps: 0 TMA + per-row constants, 1 TMEM + MMA, 2-9 recompute/dS (two
// warpgroups, one key per thread, each taking 32 of the tile's 64 query rows),
// 10-13 (FUSED) dQ^T accumulator -> bulk reduce-add into global dQ.
// TMEM: K1|K2 as the A operand of the score MMAs (cols 0-127, copied in once),
// S1^T|S2^T (128-255, one buffer, released as soon as the update warps hold it
// in registers), dK (256-383), dQ^T for the hi|lo halves of dS (384-511).
// An M = 128 MMA reading A from shared memory costs ~90 cycles whatever N <= 128
// is; with A in tensor memory an N = 128 MMA runs at the full rate.
// ---------------------------------------------------------------------------
template <int D, int NST>
struct KvSmem {
    static constexpr int kKBytes = kBlockK * D * 2;    // 128 keys
    static constexpr int kQBytes = kBwdTile * D * 2;   // 64 query rows of one tensor
    static constexpr int kDsBytes = kBlockK * kBwdTile * 2;
    // Three rings: the trainable side's query tiles (read by the score and the
    // dK MMAs, so freed after dK), the other side's (read by the score MMAs
    // only, so freed right after them: half as deep does), and the per-row
    // constants (freed once the update warps have read them).
    static constexpr int kQt = NST, kQn = NST / 2, kNv = NST >= 8 ? 4 : 3;
    static constexpr int k1 = 0;
    static constexpr int k2 = kKBytes;
    static constexpr int qt = 2 * kKBytes;
    static constexpr int qn = qt + kQt * kQBytes;
    static constexpr int kNumDs = 2;                   // dS buffers (hi + lo each)
    static constexpr int ds = qn + kQn * kQBytes;      // buffer b: hi at ds + 2*b*kDsBytes, lo right after
    // d = 64: a zero 64-feature atom pads the dQ^T MMA's A operand (K_t^T) to M = 128
    static constexpr int zero = ds + 2 * kNumDs * kDsBytes;
    static constexpr int kZeroBytes = D < 128 ? kBlockK * 128 : 0;
    static constexpr int vec = zero + kZeroBytes;  // [kNv][3][64] floats
    static constexpr int bars = vec + kNv * 3 * kBwdTile * 4;
    static constexpr int bar_k = bars;
    static constexpr int bar_qtfull = bar_k + 8;
    static constexpr int bar_qtempty = bar_qtfull + 8 * kQt;
    static constexpr int bar_qnfull = bar_qtempty + 8 * kQt;
    static constexpr int bar_qnempty = bar_qnfull + 8 * kQn;
    static constexpr int bar_vfull = bar_qnempty + 8 * kQn;
    static constexpr int bar_vempty = bar_vfull + 8 * kNv;
    static constexpr int bar_sfull = bar_vempty + 8 * kNv;
    static constexpr int bar_sempty = bar_sfull + 8;
    static constexpr int bar_dsfull = bar_sempty + 8;
    static constexpr int bar_dsempty = bar_dsfull + 8 * kNumDs;
    static constexpr int bar_dqfull = bar_dsempty + 8 * kNumDs;
    static constexpr int bar_dqempty = bar_dqfull + 8;
    static constexpr int bar_done = bar_dqempty + 8;
    static constexpr int bar_drain = bar_done + 8;  // the score issuer's own drain on abort
    static constexpr int misc = bar_drain + 8;
    static constexpr int total = misc + 16;
    static constexpr int alloc = total;  // no slack: the kernel checks the base is 1024-byte aligned
};

// Threads of bwd_kv_kernel: 10 warps (TMA, score MMAs, 8 update), 4 dQ
// epilogue warps when fused, and the gradient-MMA warp last.
template <bool FUSED>
__host__ __device__ constexpr int kv_threads() { return FUSED ? 480 : 352; }

template <int D, int NST, int SETTING, bool FUSED>
__global__ void __launch_bounds__(kv_threads<FUSED>(), 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tQ1, const __grid_constant__ CUtensorMap tK1,
                  const __grid_constant__ CUtensorMap tQ2, const __grid_constant__ CUtensorMap tK2,
                  const BwdParams p) {
    using L = KvSmem<D, NST>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // The layout uses every byte it asked for, so the dynamic shared memory
    // base itself must be 1024-byte aligned (128-byte swizzle atoms); if it is
    // not, report it and leave before touching any barrier or tensor memory.
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
    constexpr int kGradWarp = kv_threads<FUSED>() / 32 - 1;  // issues the gradient MMAs

    // head-major: resident CTAs share one head's query tiles through L2; key
    // tile 0 sees the most query rows under a causal mask and comes first
    // (a key head serves kv_group query heads: the CTA visits every query tile of each of them,
    // so dK sums the group's gradients without a second pass)
    const int bkv = blockIdx.x / p.num_k_tiles;  // flat (batch, key head)
    const int nt = blockIdx.x - bkv * p.num_k_tiles;
    const int b = bkv / p.H_kv, hk = bkv - b * p.H_kv;
    const int n0 = nt * kBlockK;
    // first 64-row query tile with a row that sees key n0 (row i sees keys j <= i + diag_off)
    const int m_start = p.causal ? max(0, (n0 - p.diag_off) / kBwdTile) : 0;
    const int per_head = p.num_q_tiles - m_start;  // query tiles of one query head that see this key tile
    const int n_tiles = per_head * p.kv_group;
    // iteration m -> (query head, query tile)
    auto qhead = [&](int m) { return p.kv_group == 1 ? hk : hk * p.kv_group + m / per_head; };
    auto qtile = [&](int m) { return m_start + (p.kv_group == 1 ? m : m % per_head); };
    const uint32_t kt_tile = base + (SETTING == 1 ? L::k2 : L::k1);  // trainable keys

    if (threadIdx.x == 0) {
        mbar_init(base + L::bar_k, 1);
        for (int s = 0; s < L::kQt; ++s) {
            mbar_init(base + L::bar_qtfull + 8 * s, 1);
            mbar_init(base + L::bar_qtempty + 8 * s, 1);
        }
        for (int s = 0; s < L::kQn; ++s) {
            mbar_init(base + L::bar_qnfull + 8 * s, 1);
            mbar_init(base + L::bar_qnempty + 8 * s, 1);
        }
        for (int s = 0; s < L::kNv; ++s) {
            mbar_init(base + L::bar_vfull + 8 * s, 32);
            mbar_init(base + L::bar_vempty + 8 * s, 256);
        }
        for (int s = 0; s < L::kNumDs; ++s) {
            mbar_init(base + L::bar_dsfull + 8 * s, 256);
            mbar_init(base + L::bar_dsempty + 8 * s, 1);
        }
        mbar_init(base + L::bar_sfull, 1);
        mbar_init(base + L::bar_sempty, 256);
        mbar_init(base + L::bar_dqfull, 1);
        mbar_init(base + L::bar_dqempty, 128);
        mbar_init(base + L::bar_done, 1);
        mbar_init(base + L::bar_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (L::kZeroBytes > 0) {
        for (int k = threadIdx.x; k < L::kZeroBytes / 16; k += blockDim.x)
            st_shared_v4(base + L::zero + 16 * k, 0u, 0u, 0u, 0u);
        fence_proxy_async_smem();  // the tensor core reads it through the async proxy
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
        const CUtensorMap* tqt = SETTING == 1 ? &tQ2 : &tQ1;  // the trainable side's queries
        const CUtensorMap* tqn = SETTING == 1 ? &tQ1 : &tQ2;
        int n_qt = 0, n_qn = 0;  // tiles whose copies were issued, per ring
        int st = 0, sn = 0, sv = 0;
        uint32_t pt = 0, pn = 0, pv = 0;
        for (int m = 0; m < n_tiles; ++m) {
            const int r0 = qtile(m) * kBwdTile;
            const int h = qhead(m);
            if (!wait_all(base + L::bar_qtempty + 8 * st, pt ^ 1, wc, kErrWaitOther)) break;
            if (lane == 0) {
                const uint32_t fb = base + L::bar_qtfull + 8 * st, dst = base + L::qt + st * L::kQBytes;
                mbar_arrive_expect_tx(fb, L::kQBytes);
#pragma unroll
                for (int c = 0; c < D / kSwizzleCols; ++c)
                    tma_load_4d_hint(dst + c * kBwdTile * 128, tqt, fb, c * kSwizzleCols, r0, h, b, keep);
            }
            ++n_qt;
            if (!wait_all(base + L::bar_qnempty + 8 * sn, pn ^ 1, wc, kErrWaitOther)) break;
            if (lane == 0) {
                const uint32_t fb = base + L::bar_qnfull + 8 * sn, dst = base + L::qn + sn * L::kQBytes;
                mbar_arrive_expect_tx(fb, L::kQBytes);
#pragma unroll
                for (int c = 0; c < D / kSwizzleCols; ++c)
                    tma_load_4d_hint(dst + c * kBwdTile * 128, tqn, fb, c * kSwizzleCols, r0, h, b, keep);
            }
            ++n_qn;
            if (!wait_all(base + L::bar_vempty + 8 * sv, pv ^ 1, wc, kErrWaitOther)) break;
            // per query row: -la, -xb and g * scale (the softmax scale of both
            // gradients is folded into dS, so neither epilogue multiplies)
            float* v = vec + sv * 3 * kBwdTile;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int r = lane + 32 * k;
                const int i = r0 + r;
                float la, xb, g;
                row_constants<SETTING>(p, (static_cast<size_t>(b) * p.H + h) * p.Nq + i, i < p.Nq, la, xb, g);
                v[r] = -la;
                v[kBwdTile + r] = -xb;
                v[2 * kBwdTile + r] = g * p.scale;
            }
            mbar_arrive(base + L::bar_vfull + 8 * sv);
            if (++st == L::kQt) st = 0, pt ^= 1;
            if (++sn == L::kQn) sn = 0, pn ^= 1;
            if (++sv == L::kNv) sv = 0, pv ^= 1;
        }
        if (lane == 0) {  // every issued copy has landed (and, unless aborting, been consumed)
            drain_wait_b(base + L::bar_k, 0, kDrainNs);
            for (int j = max(0, n_qt - L::kQt); j < n_qt; ++j) {
                const uint32_t bo = 8 * (j % L::kQt), ph = (j / L::kQt) & 1;
                drain_wait_b(base + L::bar_qtfull + bo, ph, kDrainNs);
                if (!*abort_flag) drain_wait_b(base + L::bar_qtempty + bo, ph, kDrainNs);
            }
            for (int j = max(0, n_qn - L::kQn); j < n_qn; ++j) {
                const uint32_t bo = 8 * (j % L::kQn), ph = (j / L::kQn) & 1;
                drain_wait_b(base + L::bar_qnfull + bo, ph, kDrainNs);
                if (!*abort_flag) drain_wait_b(base + L::bar_qnempty + bo, ph, kDrainNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ score MMAs
        // Two threads issue the MMAs: this one the scores of tile m, the
        // gradient warp's first thread the dK / dQ^T MMAs of earlier tiles.  A
        // thread waiting on a barrier or committing leaves the tensor pipe to
        // the other's queued work, and neither waits on the other's barriers.
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(kBlockK, kBwdTile);
            const uint32_t t_k = tmem, t_s = tmem + 128;
            bool started = false;
            // test aid: a wait on a barrier that nothing arrives on before the end
            const bool stalled = p.inject_stall && blockIdx.x == 0 &&
                                 !mbar_wait(base + L::bar_done, 0, wc, kErrWaitOther);
            if (!stalled && n_tiles > 0 && mbar_wait(base + L::bar_k, 0, wc, kErrWaitK)) {
                tc_fence_after();
                // the CTA's key tiles become the A operand of every score MMA
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ko = (kk >> 2) * kBlockK * 128 + (kk & 3) * 32;
                    tc_cp_128x256b(t_k + kk * 8, smem_desc_k128(base + L::k1 + ko));
                    tc_cp_128x256b(t_k + D / 2 + kk * 8, smem_desc_k128(base + L::k2 + ko));
                }
                started = true;
                // descriptor low words advance by compile-time offsets (the high word is
                // one constant); ring positions are counters rather than divisions
                const uint32_t dhi = smem_desc_hi();
                constexpr uint32_t kSlotLo = L::kQBytes >> 4;
                const uint32_t qt_lo0 = smem_desc_lo_k128(base + L::qt), qn_lo0 = smem_desc_lo_k128(base + L::qn);
                int st = 0, sn = 0;
                uint32_t pt = 0, pn = 0, qt_lo = qt_lo0, qn_lo = qn_lo0;
                for (int m = 0; m < n_tiles; ++m) {
                    if (!mbar_wait(base + L::bar_qtfull + 8 * st, pt, wc, kErrWaitQ)) break;
                    if (!mbar_wait(base + L::bar_qnfull + 8 * sn, pn, wc, kErrWaitQ)) break;
                    if (!mbar_wait(base + L::bar_sempty, (m & 1) ^ 1, wc, kErrWaitS)) break;
                    tc_fence_after();
                    const uint32_t q1_lo = SETTING == 1 ? qn_lo : qt_lo, q2_lo = SETTING == 1 ? qt_lo : qn_lo;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t qo = ((kk >> 2) * kBwdTile * 128 + (kk & 3) * 32) >> 4;
                        tc_mma_bf16_ta_w(t_s, t_k + kk * 8, q1_lo + qo, dhi, id_s, kk > 0);
                    }
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t qo = ((kk >> 2) * kBwdTile * 128 + (kk & 3) * 32) >> 4;
                        tc_mma_bf16_ta_w(t_s + 64, t_k + D / 2 + kk * 8, q2_lo + qo, dhi, id_s, kk > 0);
                    }
                    tc_commit(base + L::bar_sfull);
                    tc_commit(base + L::bar_qnempty + 8 * sn);  // the other side's tile is done with
                    if (++st == L::kQt) {
                        st = 0;
                        pt ^= 1;
                        qt_lo = qt_lo0;
                    } else {
                        qt_lo += kSlotLo;
                    }
                    if (++sn == L::kQn) {
                        sn = 0;
                        pn ^= 1;
                        qn_lo = qn_lo0;
                    } else {
                        qn_lo += kSlotLo;
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
        // tile m's dS (from the update warps) -> dK += dS^T Q_t, and when fused
        // [dQ^T_hi | dQ^T_lo] = K_t^T [dS^T_hi | dS^T_lo]; then the tile's dS buffer
        // and query stage are released.  (Tile m's scores finished before its dS
        // existed, so these commits also cover the score MMAs that read the stage.)
        if (lane == 0) {
            constexpr uint32_t id_dk = idesc_bf16_f32(kBlockK, D, 0, 1);
            constexpr uint32_t id_dq = idesc_bf16_f32(128, 2 * kBwdTile, 1, 1);  // M = 128 features (d = 64: padded)
            // A = K_t^T as 64-feature atoms: the tile's second block, or the zero atom when d = 64
            const uint32_t a_atom = D == 128 ? kBlockK * 128 : base + L::zero - kt_tile;
            const uint32_t t_dk = tmem + 256, t_dq = tmem + 384;
            const uint32_t dhi = smem_desc_hi();
            constexpr uint32_t kSlotLo = L::kQBytes >> 4, kDsLo = (2 * L::kDsBytes) >> 4;
            const uint32_t qt_lo0 = smem_desc_lo_mn128(base + L::qt, kBwdTile * 128);
            const uint32_t ds_lo0 = smem_desc_lo_k128(base + L::ds);
            const uint32_t dsmn_lo0 = smem_desc_lo_mn128(base + L::ds, L::kDsBytes);
            const uint32_t kt_lo = smem_desc_lo_mn128(kt_tile, a_atom);
            int issued = 0, s2 = 0, dsb = 0;
            uint32_t dsph = 0, qt_lo = qt_lo0;
            // the key tiles (A of dQ^T) have landed before any dS exists; the wait states it
            if (mbar_wait(base + L::bar_k, 0, wc, kErrWaitK)) {
                for (int m = 0; m < n_tiles; ++m) {
                    if (!mbar_wait(base + L::bar_dsfull + 8 * dsb, dsph, wc, kErrWaitOther)) break;
                    tc_fence_after();
                    const uint32_t ds_lo = ds_lo0 + (dsb ? kDsLo : 0u);
                    // dK += dS^T Q_t : A = dS^T (K-major over queries), B = Q_t (MN-major); dS = hi + lo
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int kk = 0; kk < kBwdTile / 16; ++kk)
                            tc_mma_bf16_w(t_dk, ds_lo + ((part * L::kDsBytes + kk * 32) >> 4), dhi,
                                          qt_lo + ((kk * 16 * 128) >> 4), dhi, id_dk, (kk | part | m) != 0);
                    if (FUSED) {
                        // A = K_t (MN-major), B = the hi and lo tiles as two 64-query atoms of one
                        // N = 128 operand, K = 128 keys
                        if (!mbar_wait(base + L::bar_dqempty, (m & 1) ^ 1, wc, kErrWaitOther)) break;
                        tc_fence_after();
                        const uint32_t dsmn_lo = dsmn_lo0 + (dsb ? kDsLo : 0u);
#pragma unroll
                        for (int kk = 0; kk < kBlockK / 16; ++kk)
                            tc_mma_bf16_w(t_dq, kt_lo + ((kk * 16 * 128) >> 4), dhi, dsmn_lo + ((kk * 16 * 128) >> 4),
                                          dhi, id_dq, kk > 0);
                        tc_commit(base + L::bar_dqfull);
                    }
                    tc_commit(base + L::bar_dsempty + 8 * dsb);
                    tc_commit(base + L::bar_qtempty + 8 * s2);
                    if (L::kNumDs == 1) {
                        dsph ^= 1;
                    } else {
                        dsph ^= dsb;  // a buffer's phase flips each time it comes round again
                        dsb ^= 1;
                    }
                    if (++s2 == L::kQt) {
                        s2 = 0;
                        qt_lo = qt_lo0;
                    } else {
                        qt_lo += kSlotLo;
                    }
                    ++issued;
                }
                if (issued == n_tiles) tc_commit(base + L::bar_done);
            }
            if (*abort_flag && issued > 0) {  // let the issued MMAs retire before TMEM is freed
                tc_commit(base + L::bar_done);
                drain_wait_b(base + L::bar_done, 0, kDrainNs);
            }
        }
    } else if (warp < 10) {
        // ------------------------------------------------ recompute + dS^T
        // Two warpgroups: warps 2-5 take query rows 0-31 of every tile, warps
        // 6-9 rows 32-63; one key per thread.
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
            const int dsb = m % L::kNumDs;
            const uint32_t dss = base + L::ds + 2 * dsb * L::kDsBytes;
            float z1[32], z2[32];
            tmem_ld32(t1, z1);
            tmem_ld32(t2, z2);
            tc_wait_ld();
            tc_fence_before();
            mbar_arrive(base + L::bar_sempty);  // the next score tile may overwrite S now
            // per-query constants of this chunk: 128-bit broadcast loads
            const float4* v4 = reinterpret_cast<const float4*>(vec + sv * 3 * kBwdTile + wg * 32);
            float dsv[32];
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
                const float4 a = v4[e4], x = v4[kBwdTile / 4 + e4], gg = v4[kBwdTile / 2 + e4];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int e = 4 * e4 + 2 * k;
                    const float2 nla = k ? make_float2(a.z, a.w) : make_float2(a.x, a.y);
                    const float2 nxb = k ? make_float2(x.z, x.w) : make_float2(x.x, x.y);
                    const float2 gs = k ? make_float2(gg.z, gg.w) : make_float2(gg.x, gg.y);
                    const float2 d = dscore2<SETTING>(make_float2(z1[e], z1[e + 1]), make_float2(z2[e], z2[e + 1]),
                                                      cc, sc2, nla, nxb, gs);
                    dsv[e] = d.x;
                    dsv[e + 1] = d.y;
                }
            }
            mbar_arrive(base + L::bar_vempty + 8 * sv);  // this tile's row constants are read
            // query i = r0 + e sees key j iff j <= i + diag_off; keys past Nk contribute nothing
            const int first = p.causal ? (j - p.diag_off) - r0 : -1;
            if (first > 0 || !key_ok) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e < first || !key_ok) dsv[e] = 0.f;
            }
            if (!wait_all(base + L::bar_dsempty + 8 * dsb, ((m / L::kNumDs) & 1) ^ 1, wc, kErrWaitOther)) {
                ok = false;
                break;
            }
            store_ds_chunk(dss, dss + L::kDsBytes, row, wg * 4, dsv);
            fence_proxy_async_smem();
            mbar_arrive(base + L::bar_dsfull + 8 * dsb);
        }
        // epilogue: dK row = scale * accumulator; each warpgroup writes half the columns
        if (ok && wait_all(base + L::bar_done, 0, wc, kErrWaitOther)) {
            tc_fence_after();
            void* out = reinterpret_cast<uint8_t*>(p.dK) +
                        (static_cast<size_t>(bkv) * p.Nk + j) * D * (p.grad_bf16 ? 2 : 4);
#pragma unroll 1
            for (int c0 = wg * (D / 2); c0 < (wg + 1) * (D / 2); c0 += 32) {
                float v[32];
                tmem_ld32(tl + 256 + c0, v);
                tc_wait_ld();
                if (key_ok) store_grad32(out, c0, v, 1.0f, p.grad_bf16 != 0);  // the scale is in dS
            }
        }
    } else if (FUSED) {
        // ------------------------------------------------ dQ^T -> bulk L2 reduction into dQ
        // Each tile's 64 x d float32 block of dQ is staged in shared memory as
        // 64 contiguous rows (the non-trainable key tile's space: that tile
        // only fed the copy into tensor memory) and added to global dQ by bulk
        // reduce-adds, one per 32-row half, so that staging one half overlaps
        // the reduction still reading the other.
        const int wq = warp & 3;
        const int f = wq * 32 + lane;  // feature = TMEM lane
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const uint32_t stage = base + (SETTING == 1 ? L::k1 : L::k2);
        const bool leader = warp == 10 && lane == 0;
        bool other_pending = false;  // the last bulk group issued was the other half's
        for (int m = 0; m < n_tiles; ++m) {
            // the four epilogue warps decide together, so none is left at a named barrier
            if (!bar_sync_and(3, 128, wait_all(base + L::bar_dqfull, m & 1, wc, kErrWaitOther))) break;
            tc_fence_after();
            float v0[32], v1[32];
            if (wq * 32 < D) {  // d = 64: TMEM lanes 64-127 hold the zero padding
                float lo[32];
                tmem_ld32(tl + 384, v0);  // hi half, query rows 0-31
                tmem_ld32(tl + 448, lo);  // lo half, query rows 0-31
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 t = __fadd2_rn(make_float2(v0[e], v0[e + 1]), make_float2(lo[e], lo[e + 1]));
                    v0[e] = t.x;
                    v0[e + 1] = t.y;
                }
                tmem_ld32(tl + 416, v1);  // hi half, query rows 32-63
                tmem_ld32(tl + 480, lo);  // lo half, query rows 32-63
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 t = __fadd2_rn(make_float2(v1[e], v1[e + 1]), make_float2(lo[e], lo[e + 1]));
                    v1[e] = t.x;
                    v1[e + 1] = t.y;
                }
            }
            tc_fence_before();
            mbar_arrive(base + L::bar_dqempty);
            const int r0 = qtile(m) * kBwdTile;
            const int nrow = min(kBwdTile, p.Nq - r0);
            float* dst = p.dQacc + ((static_cast<size_t>(b) * p.H + qhead(m)) * p.Nq + r0) * D;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const uint32_t sh = stage + hf * 32 * (D * 4);
                // the reduction that last read this half has finished reading; when the
                // other half's reduction was the last one issued it may still run
                if (leader) {
                    if (other_pending)
                        bulk_wait_read_1();
                    else
                        bulk_wait_read_all();
                }
                asm volatile("bar.sync 2, 128;" ::: "memory");
                if (f < D) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(sh + e * (D * 4) + f * 4), "f"(hf ? v1[e] : v0[e])
                                     : "memory");
                }
                fence_proxy_async_smem();
                asm volatile("bar.sync 2, 128;" ::: "memory");
                const int rows = min(32, nrow - 32 * hf);
                other_pending = rows > 0;
                if (leader && rows > 0) {
                    bulk_reduce_add_f32(dst + hf * 32 * D, sh, static_cast<uint32_t>(rows * D * 4));
                    bulk_commit();
                }
            }
        }
        if (leader) bulk_wait_all();  // every reduction has landed before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// float32 -> bf16 (round to nearest even), 8 elements per thread and step.
__global__ void __launch_bounds__(256) to_bf16_kernel(const float4* __restrict__ in, uint4* __restrict__ out,
                                                      size_t n8) {
    for (size_t k = blockIdx.x * size_t(blockDim.x) + threadIdx.x; k < n8; k += size_t(gridDim.x) * blockDim.x) {
        const float4 a = in[2 * k], b = in[2 * k + 1];
        out[k] = make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(b.x, b.y), pack_bf16(b.z, b.w));
    }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D, int SETTING>
cudaError_t launch_q_impl(const CUtensorMap* maps, const BwdParams& p, int ctas, cudaStream_t st) {
    constexpr int NST = D == 128 ? 4 : 6;
    static_assert(QSmem<D, NST>::alloc <= 232448, "shared memory");
    auto k = bwd_q_kernel<D, NST, SETTING>;
    cudaError_t e = set_smem(k, QSmem<D, NST>::alloc);
    if (e != cudaSuccess) return e;
    k<<<ctas, 320, QSmem<D, NST>::alloc, st>>>(maps[0], maps[1], maps[2], maps[3], p);
    return cudaGetLastError();
}

template <int D, int SETTING, bool FUSED>
cudaError_t launch_kv_impl(const CUtensorMap* maps, const BwdParams& p, int ctas, cudaStream_t st) {
    constexpr int NST = D == 128 ? 4 : 8;  // trainable-side query ring; the other side's is half as deep
    static_assert(KvSmem<D, NST>::alloc <= 232448, "shared memory");
    auto k = bwd_kv_kernel<D, NST, SETTING, FUSED>;
    cudaError_t e = set_smem(k, KvSmem<D, NST>::alloc);
    if (e != cudaSuccess) return e;
    k<<<ctas, kv_threads<FUSED>(), KvSmem<D, NST>::alloc, st>>>(maps[0], maps[1], maps[2], maps[3], p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_q(int d, int setting, const CUtensorMap* maps, const BwdParams& p, int ctas,
                         cudaStream_t stream) {
    if (d == 128) return setting == 1 ? launch_q_impl<128, 1>(maps, p, ctas, stream)
                                      : launch_q_impl<128, 2>(maps, p, ctas, stream);
    return setting == 1 ? launch_q_impl<64, 1>(maps, p, ctas, stream) : launch_q_impl<64, 2>(maps, p, ctas, stream);
}

cudaError_t launch_to_bf16(const float* in, void* out, size_t n, int sms, cudaStream_t stream) {
    const size_t n8 = n / 8;  // n is a multiple of 64 (rows of d = 64 or 128 elements)
    const int blocks = static_cast<int>(std::min<size_t>((n8 + 255) / 256, size_t(sms) * 8));
    to_bf16_kernel<<<blocks > 0 ? blocks : 1, 256, 0, stream>>>(reinterpret_cast<const float4*>(in),
                                                               reinterpret_cast<uint4*>(out), n8);
    return cudaGetLastError();
}

cudaError_t launch_bwd_kv(int d, int setting, bool fused, const CUtensorMap* maps, const BwdParams& p, int ctas,
                          cudaStream_t stream) {
    if (d == 128) {
        if (fused)
            return setting == 1 ? launch_kv_impl<128, 1, true>(maps, p, ctas, stream)
                                : launch_kv_impl<128, 2, true>(maps, p, ctas, stream);
        return setting == 1 ? launch_kv_impl<128, 1, false>(maps, p, ctas, stream)
                            : launch_kv_impl<128, 2, false>(maps, p, ctas, stream);
    }
    if (fused)
        return setting == 1 ? launch_kv_impl<64, 1, true>(maps, p, ctas, stream)
                            : launch_kv_impl<64, 2, true>(maps, p, ctas, stream);
    return setting == 1 ? launch_kv_impl<64, 1, false>(maps, p, ctas, stream)
                        : launch_kv_impl<64, 2, false>(maps, p, ctas, stream);
}

}  // namespace streamkl

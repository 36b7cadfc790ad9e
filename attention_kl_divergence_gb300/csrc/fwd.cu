// fwd.cu -- forward kernels of the attention KL divergence on sm_103a.
//
//   fwd_tile_kernel   one 128-row query tile x a range of 128-key tiles: both
//                     score GEMMs on tcgen05 (TMEM accumulators, TMA-staged
//                     bf16 operands), the five-scalar online update in
//                     registers, causal tiles beyond the frontier skipped.
//   fwd_decode_kernel Nq <= 16: keys on the MMA M side (swap of A and B), so
//                     one CTA streams 128 keys per step for every query; the
//                     key range is split across CTAs.
//   combine_kernel    merges the per-split partial states of a row.
//
// Method: "StreamKL: Fast and Memory-Efficient KL Divergence for Boosting
// Attention Distillation" (gist.science/paper/2606.20005, technical summary),
// Methodology 1 (online formulation: m1, m2, l1, l2, acc with acc rescaled by
// the teacher maximum; KL = acc/l1 + LSE2 - LSE1) and Methodology 3 (Split-K).
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace streamkl {

namespace {

constexpr float kTau = 8.0f;  // lazy rescale: tolerate running maxima up to 2^8 stale
// Update warpgroups of the tile kernel: each takes 128 / (32 * kFwdGroups)
// 32-column chunks of every score tile and keeps its own running state per row.
constexpr int kFwdGroups = 2;
// warp 0 TMA, warp 1 the S1 MMAs, the update warpgroups, and a last warp for the S2 MMAs
constexpr int kFwdThreads = 64 + 128 * kFwdGroups + 32;
constexpr int kFwdS2Warp = kFwdThreads / 32 - 1;
// Bound of the waits that let in-flight TMA copies and MMAs retire before a CTA
// exits (independent of the caller's wait limit).
constexpr uint64_t kDrainNs = 200000000ull;

// Shared-memory plan of the tile kernel.  Every operand tile starts on a
// 1024-byte boundary (128-byte swizzle atoms of 8 rows).
template <int D, int NST>
struct TileSmem {
    static constexpr int kQBytes = kBlockQ * D * 2;
    static constexpr int kKBytes = kBlockK * D * 2;
    static constexpr int q1 = 0;
    static constexpr int q2 = kQBytes;
    static constexpr int k = 2 * kQBytes;  // stage s: K1 at k + 2*s*kKBytes, K2 right after
    static constexpr int bars = k + 2 * NST * kKBytes;
    // barriers: q_full, k_full[NST], k_empty[NST], s_full[2], s_empty[2]
    static constexpr int bar_q = bars;
    static constexpr int bar_kfull = bars + 8;
    static constexpr int bar_kempty = bar_kfull + 8 * NST;
    static constexpr int bar_sfull = bar_kempty + 8 * NST;
    static constexpr int bar_sempty = bar_sfull + 16;
    static constexpr int bar_done = bar_sempty + 16;  // drain barriers of aborted MMA issuers (S1, S2)
    static constexpr int misc = bar_done + 16;    // tmem base (4 B), abort flag (4 B)
    static constexpr int red = misc + 16;         // [groups - 1][5][128] floats: the other groups' row states
    static constexpr int total = red + (kFwdGroups - 1) * 5 * 128 * 4;
    static constexpr int alloc = total + 1024;    // slack for 1024-byte alignment
};

__device__ __noinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// One W-column piece of a score row: online update of the five scalars.
// MASKED: only columns e <= last are visible (causal frontier or key tail).
// The unmasked path (every tile but the diagonal and tail ones) runs on packed
// FP32x2 arithmetic and three-input maxima.
template <bool MASKED, int W>
__device__ __forceinline__ void update_chunk(const float (&z1)[W], const float (&z2)[W], int last, RowState& st,
                                             float c, float tau) {
    static_assert(W % 4 == 0, "pieces of whole 4-column groups");
    if (MASKED && last < 0) return;  // the whole chunk lies beyond the row's last key
    float cm1, cm2;
    if (MASKED) {
        cm1 = cm2 = -INFINITY;
#pragma unroll
        for (int e = 0; e < W; ++e) {
            if (e <= last) {
                cm1 = fmaxf(cm1, z1[e]);
                cm2 = fmaxf(cm2, z2[e]);
            }
        }
    } else {
        float a1 = -INFINITY, b1 = -INFINITY, a2 = -INFINITY, b2 = -INFINITY;
#pragma unroll
        for (int e = 0; e < W; e += 4) {
            a1 = max3f(a1, z1[e], z1[e + 1]);
            b1 = max3f(b1, z1[e + 2], z1[e + 3]);
            a2 = max3f(a2, z2[e], z2[e + 1]);
            b2 = max3f(b2, z2[e + 2], z2[e + 3]);
        }
        cm1 = fmaxf(a1, b1);
        cm2 = fmaxf(a2, b2);
    }
    if (cm1 > st.m1 + tau) {
        float a = ex2(c * (st.m1 - cm1));  // 0 on the first visible chunk (m1 = -inf)
        st.l1 *= a;
        st.acc *= a;
        st.m1 = cm1;
    }
    if (cm2 > st.m2 + tau) {
        float a = ex2(c * (st.m2 - cm2));
        st.l2 *= a;
        st.m2 = cm2;
    }
    if (MASKED && st.m1 == -INFINITY) return;  // nothing visible yet
    const float n1 = -c * st.m1, n2 = -c * st.m2;
    if (MASKED) {
        float s1 = 0.f, s2 = 0.f, sa = 0.f;
#pragma unroll
        for (int e = 0; e < W; ++e) {
            if (e <= last) {
                const float p1 = ex2(fmaf(z1[e], c, n1));
                s1 += p1;
                s2 += ex2(fmaf(z2[e], c, n2));
                sa = fmaf(p1, z1[e] - z2[e], sa);
            }
        }
        st.l1 += s1;
        st.l2 += s2;
        st.acc += sa;
        return;
    }
    const float2 cc = make_float2(c, c), nn1 = make_float2(n1, n1), nn2 = make_float2(n2, n2);
    const float2 neg = make_float2(-1.f, -1.f);
    float2 s1[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float2 s2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float2 sa[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int e = 0; e < W; e += 2) {
        const int k = (e >> 1) & 1;
        const float2 u1 = make_float2(z1[e], z1[e + 1]), u2 = make_float2(z2[e], z2[e + 1]);
        const float2 x1 = __ffma2_rn(u1, cc, nn1);
        const float2 x2 = __ffma2_rn(u2, cc, nn2);
        const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
        const float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
        const float2 df = __ffma2_rn(u2, neg, u1);  // z1 - z2
        s1[k] = __fadd2_rn(s1[k], p1);
        s2[k] = __fadd2_rn(s2[k], p2);
        sa[k] = __ffma2_rn(p1, df, sa[k]);
    }
    st.l1 += (s1[0].x + s1[0].y) + (s1[1].x + s1[1].y);
    st.l2 += (s2[0].x + s2[0].y) + (s2[1].x + s2[1].y);
    st.acc += (sa[0].x + sa[0].y) + (sa[1].x + sa[1].y);
}

__device__ __forceinline__ void store_row(const FwdParams& p, size_t row, int split, const RowState& st,
                                          bool failed) {
    if (p.num_splits == 1) {
        float kl, l1, l2;
        finish_row(st, p.scale, kl, l1, l2);
        if (failed) kl = l1 = l2 = __int_as_float(0x7fc00000);
        p.KL[row] = kl;
        p.LSE1[row] = l1;
        p.LSE2[row] = l2;
    } else {
        const size_t R = static_cast<size_t>(p.B) * p.H * p.Nq;
        const size_t S = static_cast<size_t>(p.num_splits);
        float v[5] = {st.m1, st.l1, st.acc, st.m2, st.l2};
        if (failed) v[1] = v[4] = __int_as_float(0x7fc00000);
#pragma unroll
        for (int f = 0; f < 5; ++f) p.part[(f * S + split) * R + row] = v[f];
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Tile forward.  Warp 0 issues TMA, warp 1 owns TMEM and issues the MMAs, the
// remaining kFwdGroups warpgroups run the online update (one query row per
// thread, each group taking its share of the tile's columns).  TMEM: two
// buffers x (S1 | S2), 128 columns each.
// ---------------------------------------------------------------------------
template <int D, int NST>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_tile_kernel(const __grid_constant__ CUtensorMap tQ1, const __grid_constant__ CUtensorMap tK1,
                    const __grid_constant__ CUtensorMap tQ2, const __grid_constant__ CUtensorMap tK2,
                    const FwdParams p) {
    using L = TileSmem<D, NST>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_u32(smem_raw));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::misc + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::misc);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- which (head, query tile, split) this CTA owns.  Head-major order:
    // the CTAs resident at one time share one head's key tiles through L2.
    // Causal: the heaviest (last) query tiles of a head come first.
    const int per_head = p.num_q_tiles * p.num_splits;
    const int bh = blockIdx.x / per_head;
    const int rem = blockIdx.x - bh * per_head;
    const int qi = rem / p.num_splits;
    const int split = rem - qi * p.num_splits;
    const int qt = p.causal ? (p.num_q_tiles - 1 - qi) : qi;
    const int b = bh / p.H, h = bh - b * p.H;
    const int hk = h / p.kv_group;  // key head (shared by kv_group query heads)
    const int q0 = qt * kBlockQ;
    const int q_last = min(q0 + kBlockQ, p.Nq) - 1;
    const int kt_total = p.causal ? min(p.num_k_tiles, (q_last + p.diag_off) / kBlockK + 1) : p.num_k_tiles;
    const int per_split = (kt_total + p.num_splits - 1) / p.num_splits;
    const int kt_begin = split * per_split;
    const int n_tiles = max(0, min(kt_total, kt_begin + per_split) - kt_begin);

    if (threadIdx.x == 0) {
        mbar_init(base + L::bar_q, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(base + L::bar_kfull + 8 * s, 1);
            mbar_init(base + L::bar_kempty + 8 * s, 2);  // both issuers' MMAs have read the stage
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(base + L::bar_sfull + 8 * s, 2);  // S1 and S2 of the buffer are complete
            mbar_init(base + L::bar_sempty + 8 * s, 128 * kFwdGroups);
        }
        mbar_init(base + L::bar_done, 1);
        mbar_init(base + L::bar_done + 8, 1);
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
        // ------------------------------------------------------------ TMA
        if (lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&tQ1);
            prefetch_tensormap(&tK1);
            prefetch_tensormap(&tQ2);
            prefetch_tensormap(&tK2);
            const uint64_t keep = policy_evict_last();  // K tiles are re-read by every query tile
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
                const int k0 = (kt_begin + it) * kBlockK;
                const uint32_t k1s = base + L::k + 2 * s * L::kKBytes, k2s = k1s + L::kKBytes;
#pragma unroll
                for (int c = 0; c < D / kSwizzleCols; ++c) {
                    tma_load_4d_hint(k1s + c * kBlockK * 128, &tK1, fb, c * kSwizzleCols, k0, hk, b, keep);
                    tma_load_4d_hint(k2s + c * kBlockK * 128, &tK2, fb, c * kSwizzleCols, k0, hk, b, keep);
                }
            }
            // drain: every issued copy has landed and every stage was released
            drain_wait(base + L::bar_q, 0, kDrainNs);  // the query tiles' copies have landed
            for (int j = max(0, it - NST); j < it; ++j) {
                drain_wait(base + L::bar_kfull + 8 * (j % NST), (j / NST) & 1, kDrainNs);
                if (!*abort_flag) drain_wait(base + L::bar_kempty + 8 * (j % NST), (j / NST) & 1, kDrainNs);
            }
        }
    } else if (warp == 1 || warp == kFwdS2Warp) {
        // ------------------------------------------------------------ MMA
        // Two threads issue the MMAs, S1 = Q1 K1^T (warp 1) and S2 = Q2 K2^T
        // (the last warp), each committing its own arrival on the shared
        // barriers: the update warpgroups share their schedulers and keep them
        // busy, and two issuers keep the tensor pipe fed when one is held up.
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBlockQ, kBlockK);
            const bool second = warp != 1;
            const uint32_t done_bar = base + L::bar_done + (second ? 8 : 0);
            int issued = 0;
            // test aid: a wait on a barrier that nothing arrives on (bar_done is
            // only committed on the abort path below) gives up after wait_ns
            const bool stalled = p.inject_stall && blockIdx.x == 0 && !second &&
                                 !mbar_wait(base + L::bar_done, 0, wc, kErrWaitOther);
            if (!stalled && mbar_wait(base + L::bar_q, 0, wc, kErrWaitQ)) {
                tc_fence_after();
                // few instructions per MMA: descriptor low words advance by
                // compile-time offsets (the high word is one constant) and ring
                // positions are counters rather than divisions
                const uint32_t dhi = smem_desc_hi();
                const uint32_t q_lo = smem_desc_lo_k128(base + (second ? L::q2 : L::q1));
                const uint32_t k_lo0 = smem_desc_lo_k128(base + L::k) + (second ? (L::kKBytes >> 4) : 0u);
                constexpr uint32_t kStageLo = (2 * L::kKBytes) >> 4;
                const uint32_t dcol = second ? kBlockK : 0u;
                int s = 0;
                uint32_t kph = 0, k_lo = k_lo0;
                for (int it = 0; it < n_tiles; ++it) {
                    const int buf = it & 1;
                    if (!mbar_wait(base + L::bar_kfull + 8 * s, kph, wc, kErrWaitK)) break;
                    if (!mbar_wait(base + L::bar_sempty + 8 * buf, ((it >> 1) & 1) ^ 1, wc, kErrWaitS)) break;
                    tc_fence_after();
                    const uint32_t d = tmem + buf * 2 * kBlockK + dcol;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t qo = ((kk >> 2) * kBlockQ * 128 + (kk & 3) * 32) >> 4;
                        const uint32_t ko = ((kk >> 2) * kBlockK * 128 + (kk & 3) * 32) >> 4;
                        tc_mma_bf16_w(d, q_lo + qo, dhi, k_lo + ko, dhi, idesc, kk > 0);
                    }
                    tc_commit(base + L::bar_sfull + 8 * buf);
                    tc_commit(base + L::bar_kempty + 8 * s);
                    ++issued;
                    if (++s == NST) {
                        s = 0;
                        kph ^= 1;
                        k_lo = k_lo0;
                    } else {
                        k_lo += kStageLo;
                    }
                }
            }
            if (*abort_flag && issued > 0) {  // let the issued MMAs retire before TMEM is freed
                tc_commit(done_bar);
                drain_wait(done_bar, 0, kDrainNs);
            }
        }
    } else {
        // ------------------------------------------------------------ online update (warps 2 .. 2 + 4 groups)
        // kFwdGroups warpgroups split every tile's 128 columns; each keeps its
        // own running state per row, and the states of a row are merged at the
        // end (the same log-sum-exp merge as the Split-K combine).
        constexpr int kChunks = 4 / kFwdGroups;  // 32-column chunks per group and tile
        const int wg = (warp - 2) >> 2;
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const int i = q0 + row;
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float c = p.scale_log2e;
        const float tau = kTau / c;
        const int limit = p.causal ? min(i + p.diag_off, p.Nk - 1) : p.Nk - 1;  // last visible key
        RowState st{-INFINITY, 0.f, 0.f, -INFINITY, 0.f};
        bool ok = true;
        for (int it = 0; it < n_tiles; ++it) {
            const int buf = it & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(base + L::bar_sfull + 8 * buf, (it >> 1) & 1, wc, kErrWaitS))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int jrem = limit - (kt_begin + it) * kBlockK;  // last visible column of this tile
            const uint32_t t1 = tl + buf * 2 * kBlockK, t2 = t1 + kBlockK;
#pragma unroll 1
            for (int cc = 0; cc < kChunks; ++cc) {
                const int ch = kChunks * wg + cc;
                float z1[32], z2[32];
                tmem_ld32(t1 + ch * 32, z1);
                tmem_ld32(t2 + ch * 32, z2);
                tc_wait_ld();
                if (cc == kChunks - 1) {
                    tc_fence_before();
                    mbar_arrive(base + L::bar_sempty + 8 * buf);
                }
                const int last = jrem - ch * 32;
                if (last >= 31)
                    update_chunk<false, 32>(z1, z2, 31, st, c, tau);
                else
                    update_chunk<true, 32>(z1, z2, last, st, c, tau);
            }
        }
        float* red = reinterpret_cast<float*>(gbase + L::red);
        if (wg > 0) {
            float* r = red + (wg - 1) * 5 * 128;
            r[row] = st.m1;
            r[128 + row] = st.l1;
            r[256 + row] = st.acc;
            r[384 + row] = st.m2;
            r[512 + row] = st.l2;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(128 * kFwdGroups) : "memory");  // the update warps only
        if (wg == 0) {
            for (int k = 0; k < kFwdGroups - 1; ++k) {
                const float* r = red + k * 5 * 128;
                const RowState o{r[row], r[128 + row], r[256 + row], r[384 + row], r[512 + row]};
                merge_state(st, o, c);
            }
            if (i < p.Nq) store_row(p, static_cast<size_t>(bh) * p.Nq + i, split, st, !ok || *abort_flag);
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
// Decode forward, Nq <= 16 (causal or not).  S^T = K Q^T: M = 128 keys (TMEM lanes),
// N = 16 query columns.  Each thread owns one key per step and keeps a running
// state per query; the 128 states are merged at the end of the key range.
// Query heads that share a key head are packed into the 16 columns
// (heads_per_cta heads x Nq rows, head-major), so a shared key tile is
// streamed once for all of them.
// ---------------------------------------------------------------------------
template <int D, int NST>
struct DecodeSmem {
    static constexpr int kQBytes = kDecodeMaxQ * D * 2;  // 16 rows
    static constexpr int kKBytes = kBlockK * D * 2;
    static constexpr int q1 = 0;
    static constexpr int q2 = ((kQBytes + 1023) / 1024) * 1024;
    static constexpr int k = q2 + q2;
    static constexpr int bars = k + 2 * NST * kKBytes;
    static constexpr int bar_q = bars;
    static constexpr int bar_kfull = bars + 8;
    static constexpr int bar_kempty = bar_kfull + 8 * NST;
    static constexpr int bar_sfull = bar_kempty + 8 * NST;
    static constexpr int bar_sempty = bar_sfull + 16;
    static constexpr int bar_done = bar_sempty + 16;
    static constexpr int misc = bar_done + 8;
    static constexpr int red = misc + 16;                    // [4 warps][16 q][5] floats
    static constexpr int total = red + 4 * kDecodeMaxQ * 5 * 4;
    static constexpr int alloc = total + 1024;
};

template <int D, int NST>
__global__ void __launch_bounds__(192, 1)
    fwd_decode_kernel(const __grid_constant__ CUtensorMap tQ1, const __grid_constant__ CUtensorMap tK1,
                      const __grid_constant__ CUtensorMap tQ2, const __grid_constant__ CUtensorMap tK2,
                      const FwdParams p) {
    using L = DecodeSmem<D, NST>;
    constexpr int NQ = kDecodeMaxQ;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_u32(smem_raw));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::misc + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::misc);
    float* red = reinterpret_cast<float*>(gbase + L::red);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hp = p.heads_per_cta;
    const int nq = hp * p.Nq;  // packed query columns in use
    const int gi = blockIdx.x / p.num_splits;
    const int split = blockIdx.x - gi * p.num_splits;
    const int groups = p.H / hp;
    const int b = gi / groups, h0 = (gi - b * groups) * hp;
    const int hk = h0 / p.kv_group;  // key head shared by the packed query heads
    const size_t row0 = (static_cast<size_t>(b) * p.H + h0) * p.Nq;  // output row of column 0
    const int per_split = (p.num_k_tiles + p.num_splits - 1) / p.num_splits;
    const int kt_begin = split * per_split;
    const int n_tiles = max(0, min(p.num_k_tiles, kt_begin + per_split) - kt_begin);

    if (threadIdx.x == 0) {
        mbar_init(base + L::bar_q, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(base + L::bar_kfull + 8 * s, 1);
            mbar_init(base + L::bar_kempty + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(base + L::bar_sfull + 8 * s, 1);
            mbar_init(base + L::bar_sempty + 8 * s, 128);
        }
        mbar_init(base + L::bar_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    // unused query columns read zeros (the copies below fill only the first nq rows)
    for (int i = threadIdx.x; i < 2 * (D / kSwizzleCols) * (NQ - nq) * 8; i += blockDim.x) {
        const int chunk16 = i & 7, rr = i >> 3;
        const int r = nq + rr % (NQ - nq), tc = rr / (NQ - nq);  // tc: tensor * column blocks
        const uint32_t at = base + (tc & 1 ? L::q2 : L::q1) + (tc >> 1) * NQ * 128 + r * 128 + chunk16 * 16;
        st_shared_v4(at, 0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    if (warp == 1) tmem_alloc(base + L::misc, 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, p.status, p.wait_ns};

    if (warp == 0) {
        if (lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&tQ1);
            prefetch_tensormap(&tK1);
            prefetch_tensormap(&tQ2);
            prefetch_tensormap(&tK2);
            const uint64_t stream_once = policy_evict_first();  // each key is read exactly once
            // one box = Nq rows x heads_per_cta heads, landing as nq consecutive rows
            mbar_arrive_expect_tx(base + L::bar_q, 2 * nq * D * 2);
#pragma unroll
            for (int c = 0; c < D / kSwizzleCols; ++c) {
                tma_load_4d(base + L::q1 + c * NQ * 128, &tQ1, base + L::bar_q, c * kSwizzleCols, 0, h0, b);
                tma_load_4d(base + L::q2 + c * NQ * 128, &tQ2, base + L::bar_q, c * kSwizzleCols, 0, h0, b);
            }
            int it = 0;
            for (; it < n_tiles; ++it) {
                const int s = it % NST;
                if (!mbar_wait(base + L::bar_kempty + 8 * s, ((it / NST) & 1) ^ 1, wc, kErrWaitK)) break;
                const uint32_t fb = base + L::bar_kfull + 8 * s;
                mbar_arrive_expect_tx(fb, 2 * L::kKBytes);
                const int k0 = (kt_begin + it) * kBlockK;
                const uint32_t k1s = base + L::k + 2 * s * L::kKBytes, k2s = k1s + L::kKBytes;
#pragma unroll
                for (int c = 0; c < D / kSwizzleCols; ++c) {
                    tma_load_4d_hint(k1s + c * kBlockK * 128, &tK1, fb, c * kSwizzleCols, k0, hk, b, stream_once);
                    tma_load_4d_hint(k2s + c * kBlockK * 128, &tK2, fb, c * kSwizzleCols, k0, hk, b, stream_once);
                }
            }
            drain_wait(base + L::bar_q, 0, kDrainNs);  // the query tiles' copies have landed
            for (int j = max(0, it - NST); j < it; ++j) {
                drain_wait(base + L::bar_kfull + 8 * (j % NST), (j / NST) & 1, kDrainNs);
                if (!*abort_flag) drain_wait(base + L::bar_kempty + 8 * (j % NST), (j / NST) & 1, kDrainNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBlockK, NQ);
            int issued = 0;
            // test aid: a wait on a barrier that nothing arrives on (bar_done is
            // only committed on the abort path below) gives up after wait_ns
            const bool stalled = p.inject_stall && blockIdx.x == 0 &&
                                 !mbar_wait(base + L::bar_done, 0, wc, kErrWaitOther);
            if (!stalled && mbar_wait(base + L::bar_q, 0, wc, kErrWaitQ)) {
                tc_fence_after();
                for (int it = 0; it < n_tiles; ++it) {
                    const int s = it % NST, buf = it & 1;
                    if (!mbar_wait(base + L::bar_kfull + 8 * s, (it / NST) & 1, wc, kErrWaitK)) break;
                    if (!mbar_wait(base + L::bar_sempty + 8 * buf, ((it >> 1) & 1) ^ 1, wc, kErrWaitS)) break;
                    tc_fence_after();
                    const uint32_t d1 = tmem + buf * 2 * NQ, d2 = d1 + NQ;
                    const uint32_t k1s = base + L::k + 2 * s * L::kKBytes, k2s = k1s + L::kKBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ko = (kk >> 2) * kBlockK * 128 + (kk & 3) * 32;
                        const uint32_t qo = (kk >> 2) * NQ * 128 + (kk & 3) * 32;
                        tc_mma_bf16(d1, smem_desc_k128(k1s + ko), smem_desc_k128(base + L::q1 + qo), idesc, kk > 0);
                    }
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ko = (kk >> 2) * kBlockK * 128 + (kk & 3) * 32;
                        const uint32_t qo = (kk >> 2) * NQ * 128 + (kk & 3) * 32;
                        tc_mma_bf16(d2, smem_desc_k128(k2s + ko), smem_desc_k128(base + L::q2 + qo), idesc, kk > 0);
                    }
                    tc_commit(base + L::bar_sfull + 8 * buf);
                    tc_commit(base + L::bar_kempty + 8 * s);
                    ++issued;
                }
            }
            if (*abort_flag && issued > 0) {
                tc_commit(base + L::bar_done);
                drain_wait(base + L::bar_done, 0, kDrainNs);
            }
        }
    } else {
        const int wq = warp & 3;
        const int krow = wq * 32 + lane;  // key within the tile = TMEM lane
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float c = p.scale_log2e;
        const float tau = kTau / c;
        // query index within its head of each packed column; unused columns
        // get INT_MIN, below every causal bound
        int qi[NQ];
        float m1[NQ], l1[NQ], ac[NQ], m2[NQ], l2[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            qi[q] = q < nq ? q % p.Nq : INT_MIN;
            m1[q] = -INFINITY;
            m2[q] = -INFINITY;
            l1[q] = l2[q] = ac[q] = 0.f;
        }
        bool ok = true;
        for (int it = 0; it < n_tiles; ++it) {
            const int buf = it & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(base + L::bar_sfull + 8 * buf, (it >> 1) & 1, wc, kErrWaitS))) {
                ok = false;
                break;
            }
            tc_fence_after();
            float z1[NQ], z2[NQ];
            tmem_ld16(tl + buf * 2 * NQ, z1);
            tmem_ld16(tl + buf * 2 * NQ + NQ, z2);
            tc_wait_ld();
            tc_fence_before();
            mbar_arrive(base + L::bar_sempty + 8 * buf);
            const int j = (kt_begin + it) * kBlockK + krow;
            if (j >= p.Nk) continue;  // key tail
            // causal (bottom-right): query i sees key j iff j <= i + diag_off; keys up to
            // diag_off are seen by every query
            const int first_q = p.causal ? j - p.diag_off : 0;
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                if (qi[q] >= first_q) {
                    if (z1[q] > m1[q] + tau) {
                        const float a = ex2(c * (m1[q] - z1[q]));
                        l1[q] *= a;
                        ac[q] *= a;
                        m1[q] = z1[q];
                    }
                    if (z2[q] > m2[q] + tau) {
                        l2[q] *= ex2(c * (m2[q] - z2[q]));
                        m2[q] = z2[q];
                    }
                    const float p1 = ex2(c * (z1[q] - m1[q]));
                    l1[q] += p1;
                    ac[q] = fmaf(p1, z1[q] - z2[q], ac[q]);
                    l2[q] += ex2(c * (z2[q] - m2[q]));
                }
            }
        }
        // merge the 128 per-key states of every query: warp butterfly, then warps
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            if (q < nq) {
                RowState s{m1[q], l1[q], ac[q], m2[q], l2[q]};
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    RowState t{__shfl_xor_sync(0xffffffffu, s.m1, o), __shfl_xor_sync(0xffffffffu, s.l1, o),
                               __shfl_xor_sync(0xffffffffu, s.acc, o), __shfl_xor_sync(0xffffffffu, s.m2, o),
                               __shfl_xor_sync(0xffffffffu, s.l2, o)};
                    merge_state(s, t, c);
                }
                if (lane == 0) {
                    float* r = red + (wq * NQ + q) * 5;
                    r[0] = s.m1;
                    r[1] = s.l1;
                    r[2] = s.acc;
                    r[3] = s.m2;
                    r[4] = s.l2;
                }
            }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four update warps only
        if (wq == 0 && lane < nq) {
            const int q = lane;
            RowState s{-INFINITY, 0.f, 0.f, -INFINITY, 0.f};
            for (int w = 0; w < 4; ++w) {
                const float* r = red + (w * NQ + q) * 5;
                RowState t{r[0], r[1], r[2], r[3], r[4]};
                merge_state(s, t, c);
            }
            store_row(p, row0 + q, split, s, !ok || *abort_flag);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

// ---------------------------------------------------------------------------
// Split-K combine: one thread per row merges its partial states and finishes.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
    const int row = blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
    const size_t R = static_cast<size_t>(p.rows);
    const size_t S = static_cast<size_t>(p.num_splits);
    RowState s{-INFINITY, 0.f, 0.f, -INFINITY, 0.f};
    for (int k = 0; k < p.num_splits; ++k) {
        RowState t{p.part[(0 * S + k) * R + row], p.part[(1 * S + k) * R + row], p.part[(2 * S + k) * R + row],
                   p.part[(3 * S + k) * R + row], p.part[(4 * S + k) * R + row]};
        merge_state(s, t, p.scale_log2e);
    }
    float kl, l1, l2;
    finish_row(s, p.scale, kl, l1, l2);
    p.KL[row] = kl;
    p.LSE1[row] = l1;
    p.LSE2[row] = l2;
}

// ---------------------------------------------------------------------------
// Host-side launchers
// ---------------------------------------------------------------------------
namespace {
template <typename K>
cudaError_t ensure_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}
}  // namespace

cudaError_t launch_fwd_tile(int d, const CUtensorMap* maps, const FwdParams& p, int ctas, cudaStream_t stream) {
    cudaError_t e;
    if (d == 128) {
        constexpr int NST = 2;
        auto k = fwd_tile_kernel<128, NST>;
        if ((e = ensure_smem(k, TileSmem<128, NST>::alloc)) != cudaSuccess) return e;
        k<<<ctas, kFwdThreads, TileSmem<128, NST>::alloc, stream>>>(maps[0], maps[1], maps[2], maps[3], p);
    } else {
        constexpr int NST = 4;
        auto k = fwd_tile_kernel<64, NST>;
        if ((e = ensure_smem(k, TileSmem<64, NST>::alloc)) != cudaSuccess) return e;
        k<<<ctas, kFwdThreads, TileSmem<64, NST>::alloc, stream>>>(maps[0], maps[1], maps[2], maps[3], p);
    }
    return cudaGetLastError();
}

cudaError_t launch_fwd_decode(int d, const CUtensorMap* maps, const FwdParams& p, int ctas, cudaStream_t stream) {
    cudaError_t e;
    if (d == 128) {
        constexpr int NST = 3;
        auto k = fwd_decode_kernel<128, NST>;
        if ((e = ensure_smem(k, DecodeSmem<128, NST>::alloc)) != cudaSuccess) return e;
        k<<<ctas, 192, DecodeSmem<128, NST>::alloc, stream>>>(maps[0], maps[1], maps[2], maps[3], p);
    } else {
        constexpr int NST = 6;
        auto k = fwd_decode_kernel<64, NST>;
        if ((e = ensure_smem(k, DecodeSmem<64, NST>::alloc)) != cudaSuccess) return e;
        k<<<ctas, 192, DecodeSmem<64, NST>::alloc, stream>>>(maps[0], maps[1], maps[2], maps[3], p);
    }
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    const int threads = 256;
    combine_kernel<<<(p.rows + threads - 1) / threads, threads, 0, stream>>>(p);
    return cudaGetLastError();
}

int fwd_tile_stages(int d) { return d == 128 ? 2 : 4; }

}  // namespace streamkl

// api.cu -- the C ABI of libstreamkl: argument validation, launch planning,
// TMA tensor maps and kernel launches on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/streamkl.h"
#include "common.cuh"
#include "kernels.h"

using namespace streamkl;

namespace {

constexpr int kMaxSplits = 64;
constexpr int64_t kDefaultWaitNs = 2000000000LL;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Structural checks that need no device.
streamkl_status check_shape(const streamkl_shape* s, int causal) {
    if (!s) return STREAMKL_ERR_INVALID_ARG;
    if (s->B < 1 || s->H < 1 || s->Nq < 1 || s->Nk < 1 || s->d < 1) return STREAMKL_ERR_INVALID_ARG;
    if (s->d != 64 && s->d != 128) return STREAMKL_ERR_UNSUPPORTED;
    if (causal && s->Nq > s->Nk) return STREAMKL_ERR_INVALID_ARG;
    const int64_t st[6] = {s->q_stride_b, s->q_stride_h, s->q_stride_n, s->k_stride_b, s->k_stride_h, s->k_stride_n};
    for (int64_t v : st)
        if (v < 1 || (v % 8) != 0 || v > (int64_t(1) << 38)) return STREAMKL_ERR_INVALID_ARG;
    if (s->q_stride_n < s->d || s->k_stride_n < s->d) return STREAMKL_ERR_INVALID_ARG;
    if (int64_t(s->B) * s->H > (int64_t(1) << 24)) return STREAMKL_ERR_UNSUPPORTED;
    if (s->H_kv < 0 || (s->H_kv > 0 && s->H % s->H_kv != 0)) return STREAMKL_ERR_INVALID_ARG;
    return STREAMKL_OK;
}

int kv_heads(const streamkl_shape* s) { return s->H_kv > 0 ? s->H_kv : s->H; }

streamkl_status device_sms(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return STREAMKL_ERR_CUDA;
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return STREAMKL_ERR_CUDA;
    return STREAMKL_OK;
}

// Key splits for `units` independent rows-tiles of `k_tiles` key tiles each
// on `slots` resident CTAs: minimise waves * (tiles per split + 1 tile of
// fixed cost), preferring fewer splits on ties.
int choose_splits(int64_t units, int k_tiles, int slots) {
    // (used by the tile forward and the key-split backward; decode_splits below for the decode forward)
    if (units >= slots || k_tiles < 2) return 1;
    int best = 1;
    int64_t best_cost = INT64_MAX;
    const int smax = k_tiles < kMaxSplits ? k_tiles : kMaxSplits;
    for (int s = 1; s <= smax; ++s) {
        const int64_t waves = (units * s + slots - 1) / slots;
        const int64_t cost = waves * ((k_tiles + s - 1) / s + 1);
        if (cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// Key splits of the decode forward, which streams every key byte once and is
// bound by HBM: measured on GB300, about 0.7 x SMs streaming CTAs saturate it
// (32 CTAs 2.7 TB/s, 64 5.2, 96-128 6.1), so the key range is split only until
// that many CTAs exist.  More splits add partial states and a second wave
// (B4 H32, 16 rows: 1 split 1.25 ms, 13 splits 1.32 ms).
int decode_splits(int64_t units, int k_tiles, int sms) {
    const int64_t saturate = (int64_t(sms) * 7 + 9) / 10;
    if (units >= saturate) return 1;
    int64_t s = (saturate + units - 1) / units;
    if (s > k_tiles) s = k_tiles;
    if (s > kMaxSplits) s = kMaxSplits;
    return s < 1 ? 1 : static_cast<int>(s);
}

struct FwdPlan {
    bool decode;
    int heads_per_cta;  // decode: query heads sharing a key head packed into one CTA
    int num_splits;
    int ctas;
    int num_q_tiles;
    int num_k_tiles;
    size_t ws_bytes;
};

streamkl_status plan_fwd(const streamkl_shape* s, int causal, const streamkl_options* opt, FwdPlan* pl) {
    streamkl_status st = check_shape(s, causal);
    if (st != STREAMKL_OK) return st;
    if (opt && (opt->num_splits < 0 || (opt->grad_bf16 != 0 && opt->grad_bf16 != 1) ||
                (opt->debug_flags & ~STREAMKL_DEBUG_INJECT_STALL)))
        return STREAMKL_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = device_sms(&sms)) != STREAMKL_OK) return st;
    const int64_t BH = int64_t(s->B) * s->H;
    pl->decode = s->Nq <= kDecodeMaxQ;
    pl->num_q_tiles = pl->decode ? 1 : (s->Nq + kBlockQ - 1) / kBlockQ;
    pl->num_k_tiles = (s->Nk + kBlockK - 1) / kBlockK;
    // decode: the largest divisor of the group whose queries fit the 16 columns
    pl->heads_per_cta = 1;
    if (pl->decode) {
        const int group = s->H / kv_heads(s);
        for (int c = group; c > 1; --c)
            if (group % c == 0 && c * s->Nq <= kDecodeMaxQ) {
                pl->heads_per_cta = c;
                break;
            }
    }
    const int64_t units = BH / pl->heads_per_cta * pl->num_q_tiles;
    int splits;
    if (opt && opt->num_splits > 0)
        splits = opt->num_splits < pl->num_k_tiles ? opt->num_splits : pl->num_k_tiles;
    else if (pl->decode)
        splits = decode_splits(units, pl->num_k_tiles, sms);
    else
        splits = choose_splits(units, pl->num_k_tiles, sms);
    if (splits > kMaxSplits) splits = kMaxSplits;
    const int64_t ctas = units * splits;
    if (ctas > INT32_MAX) return STREAMKL_ERR_UNSUPPORTED;
    pl->num_splits = splits;
    pl->ctas = static_cast<int>(ctas);
    pl->ws_bytes = kStatusBytes;
    if (splits > 1) pl->ws_bytes += size_t(5) * splits * size_t(BH) * s->Nq * sizeof(float);
    return STREAMKL_OK;
}

struct BwdPlan {
    bool fused;
    bool keysplit;  // at most 16 query rows per key head: key-split kernel
    bool bf16;
    int ctas_q;
    int ctas_kv;
    int splits;     // key-split kernel: key-range splits per key head
    int ctas_dec;
    size_t ws_bytes;
};

// Mode choice.  The pages use the fused kernel (dQ through atomics) while the
// float32 dQ buffer fits in L2 and separate kernels beyond.  Measured on
// GB300 the fused kernel is faster at every size tried (setting 1: 8K causal
// 1.21 vs 2.14 ms, 64K causal 73.4 vs 118.1 ms: the split pays a second
// recompute of both score tiles, which costs more than the L2 reductions), so
// the automatic choice is fused unless every query row of a key head fits one
// CTA's 16 columns (the key-split kernel); the split stays selectable.
streamkl_status plan_bwd(const streamkl_shape* s, int setting, int causal, const streamkl_options* opt,
                         BwdPlan* pl) {
    streamkl_status st = check_shape(s, causal);
    if (st != STREAMKL_OK) return st;
    if (setting != 1 && setting != 2) return STREAMKL_ERR_INVALID_ARG;
    const int mode = opt ? opt->bwd_mode : 0;
    if (mode < 0 || mode > 3) return STREAMKL_ERR_INVALID_ARG;
    if (opt && ((opt->grad_bf16 != 0 && opt->grad_bf16 != 1) || (opt->debug_flags & ~STREAMKL_DEBUG_INJECT_STALL)))
        return STREAMKL_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return STREAMKL_ERR_CUDA;
    const int64_t BH = int64_t(s->B) * s->H;
    // every query row of a key head fits the 16 columns of one CTA: the key-split kernel
    const bool fits = int64_t(s->Nq) * (s->H / kv_heads(s)) <= kDecodeMaxQ;
    if (mode == 3 && !fits) return STREAMKL_ERR_UNSUPPORTED;
    pl->keysplit = mode == 3 || (mode == 0 && fits);
    if (mode == 0)
        pl->fused = !pl->keysplit;
    else
        pl->fused = mode == 1;
    pl->splits = 1;
    pl->ctas_dec = 0;
    if (pl->keysplit) {
        int sms = 0;
        if ((st = device_sms(&sms)) != STREAMKL_OK) return st;
        const int64_t units = int64_t(s->B) * kv_heads(s);
        const int k_tiles = (s->Nk + kBlockK - 1) / kBlockK;
        if (opt && opt->num_splits > 0)
            pl->splits = opt->num_splits < k_tiles ? opt->num_splits : k_tiles;
        else
            pl->splits = choose_splits(units, k_tiles, sms);
        if (units * pl->splits > INT32_MAX) return STREAMKL_ERR_UNSUPPORTED;
        pl->ctas_dec = static_cast<int>(units * pl->splits);
    }
    const int64_t ctas_kv = int64_t(s->B) * kv_heads(s) * ((s->Nk + kBlockK - 1) / kBlockK);
    const int64_t ctas_q = BH * ((s->Nq + kBlockQ - 1) / kBlockQ);
    if (ctas_kv > INT32_MAX || ctas_q > INT32_MAX) return STREAMKL_ERR_UNSUPPORTED;
    pl->ctas_kv = static_cast<int>(ctas_kv);
    pl->ctas_q = static_cast<int>(ctas_q);
    pl->bf16 = opt && opt->grad_bf16 == 1;
    pl->ws_bytes = kStatusBytes;
    // bf16 gradients from a mode that adds dQ up: dQ is accumulated in float32 in the workspace first
    if ((pl->fused || pl->keysplit) && pl->bf16) pl->ws_bytes += size_t(BH) * s->Nq * s->d * sizeof(float);
    return STREAMKL_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 4-D map over [B, H, N, d] bf16 with a (64 x rows x heads) box, 128-byte
// swizzle; rows outside [0, N) read as zero.  A box of several heads lands
// in shared memory as heads * rows consecutive 128-byte rows, head-major.
bool make_map(CUtensorMap* m, const void* ptr, const streamkl_shape* s, bool is_q, int box_rows,
              int box_heads = 1) {
    auto enc = encode_fn();
    if (!enc) return false;
    const int64_t N = is_q ? s->Nq : s->Nk;
    const int64_t sb = is_q ? s->q_stride_b : s->k_stride_b;
    const int64_t sh = is_q ? s->q_stride_h : s->k_stride_h;
    const int64_t sn = is_q ? s->q_stride_n : s->k_stride_n;
    cuuint64_t dims[4] = {cuuint64_t(s->d), cuuint64_t(N), cuuint64_t(is_q ? s->H : kv_heads(s)), cuuint64_t(s->B)};
    cuuint64_t strides[3] = {cuuint64_t(sn * 2), cuuint64_t(sh * 2), cuuint64_t(sb * 2)};
    cuuint32_t box[4] = {cuuint32_t(kSwizzleCols), cuuint32_t(box_rows), cuuint32_t(box_heads), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

float resolve_scale(float scale, int d) {
    if (!(scale > 0.f) || std::isinf(scale)) return 1.0f / std::sqrt(static_cast<float>(d));
    return scale;
}

int64_t wait_limit(const streamkl_options* opt) {
    return (opt && opt->wait_limit_ns > 0) ? opt->wait_limit_ns : kDefaultWaitNs;
}

}  // namespace

extern "C" {

int streamkl_version(void) { return 200; }  // 0.2.0: joint backward, size queries, allocation-free status

const char* streamkl_status_string(streamkl_status s) {
    switch (s) {
        case STREAMKL_OK: return "ok";
        case STREAMKL_ERR_INVALID_ARG: return "invalid argument";
        case STREAMKL_ERR_UNSUPPORTED: return "unsupported configuration";
        case STREAMKL_ERR_WORKSPACE: return "workspace missing or too small";
        case STREAMKL_ERR_CUDA: return "CUDA error";
        case STREAMKL_ERR_TIMEOUT: return "a kernel wait timed out";
    }
    return "unknown status";
}

streamkl_status streamkl_fwd_plan(const streamkl_shape* shape, int causal, const streamkl_options* opt,
                                  streamkl_plan* plan) {
    if (!plan) return STREAMKL_ERR_INVALID_ARG;
    FwdPlan pl{};
    streamkl_status st = plan_fwd(shape, causal, opt, &pl);
    if (st != STREAMKL_OK) return st;
    plan->path = pl.decode ? 1 : 0;
    plan->num_splits = pl.num_splits;
    plan->num_ctas = pl.ctas;
    plan->launches = pl.num_splits > 1 ? 2 : 1;
    plan->workspace_bytes = pl.ws_bytes;
    return STREAMKL_OK;
}

streamkl_status streamkl_fwd(const streamkl_shape* shape, const void* Q1, const void* K1, const void* Q2,
                             const void* K2, float scale, int causal, float* KL, float* LSE1, float* LSE2,
                             void* workspace, size_t workspace_bytes, const streamkl_options* opt,
                             streamkl_stream_t stream) {
    streamkl_status st = check_shape(shape, causal);
    if (st != STREAMKL_OK) return st;
    const void* ptrs[7] = {Q1, K1, Q2, K2, KL, LSE1, LSE2};
    for (const void* q : ptrs)
        if (!q) return STREAMKL_ERR_INVALID_ARG;
    for (int k = 0; k < 4; ++k)
        if (!aligned16(ptrs[k])) return STREAMKL_ERR_INVALID_ARG;
    for (int k = 4; k < 7; ++k)
        if ((reinterpret_cast<uintptr_t>(ptrs[k]) & 3u) != 0) return STREAMKL_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace)) return STREAMKL_ERR_WORKSPACE;
    FwdPlan pl{};
    if ((st = plan_fwd(shape, causal, opt, &pl)) != STREAMKL_OK) return st;
    if (workspace_bytes < pl.ws_bytes) return STREAMKL_ERR_WORKSPACE;

    // decode: one query box is the Nq rows of heads_per_cta heads
    const int qrows = pl.decode ? shape->Nq : kBlockQ;
    const int qheads = pl.heads_per_cta;
    CUtensorMap maps[4];
    if (!make_map(&maps[0], Q1, shape, true, qrows, qheads) || !make_map(&maps[1], K1, shape, false, kBlockK) ||
        !make_map(&maps[2], Q2, shape, true, qrows, qheads) || !make_map(&maps[3], K2, shape, false, kBlockK))
        return STREAMKL_ERR_CUDA;

    const float sc = resolve_scale(scale, shape->d);
    FwdParams p{};
    p.B = shape->B;
    p.H = shape->H;
    p.Nq = shape->Nq;
    p.Nk = shape->Nk;
    p.num_q_tiles = pl.num_q_tiles;
    p.num_k_tiles = pl.num_k_tiles;
    p.num_splits = pl.num_splits;
    p.causal = causal ? 1 : 0;
    p.diag_off = shape->Nk - shape->Nq;
    p.kv_group = shape->H / kv_heads(shape);
    p.heads_per_cta = pl.heads_per_cta;
    p.scale = sc;
    p.scale_log2e = sc * 1.4426950408889634f;
    p.KL = KL;
    p.LSE1 = LSE1;
    p.LSE2 = LSE2;
    p.part = pl.num_splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kStatusBytes) : nullptr;
    p.status = static_cast<unsigned int*>(workspace);
    p.wait_ns = static_cast<unsigned long long>(wait_limit(opt));
    p.inject_stall = (opt && (opt->debug_flags & STREAMKL_DEBUG_INJECT_STALL)) ? 1 : 0;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = pl.decode ? launch_fwd_decode(shape->d, maps, p, pl.ctas, s)
                              : launch_fwd_tile(shape->d, maps, p, pl.ctas, s);
    if (e != cudaSuccess) return STREAMKL_ERR_CUDA;
    if (pl.num_splits > 1) {
        CombineParams c{};
        c.rows = static_cast<int>(int64_t(shape->B) * shape->H * shape->Nq);
        c.num_splits = pl.num_splits;
        c.scale = sc;
        c.scale_log2e = p.scale_log2e;
        c.part = p.part;
        c.KL = KL;
        c.LSE1 = LSE1;
        c.LSE2 = LSE2;
        if (launch_combine(c, s) != cudaSuccess) return STREAMKL_ERR_CUDA;
    }
    return STREAMKL_OK;
}

streamkl_status streamkl_bwd_plan(const streamkl_shape* shape, int setting, int causal,
                                  const streamkl_options* opt, streamkl_plan* plan) {
    if (!plan) return STREAMKL_ERR_INVALID_ARG;
    BwdPlan pl{};
    streamkl_status st = plan_bwd(shape, setting, causal, opt, &pl);
    if (st != STREAMKL_OK) return st;
    plan->path = pl.keysplit ? 4 : pl.fused ? 2 : 3;
    plan->num_splits = pl.splits;
    plan->num_ctas = pl.keysplit ? pl.ctas_dec : pl.ctas_kv;
    // fused and key-split: zero dQ + kernel (+ bf16 conversion); split: two kernels
    plan->launches = ((pl.fused || pl.keysplit) && pl.bf16) ? 3 : 2;
    plan->workspace_bytes = pl.ws_bytes;
    return STREAMKL_OK;
}

size_t streamkl_fwd_workspace_bytes(const streamkl_shape* shape, int causal) {
    FwdPlan pl{};
    return plan_fwd(shape, causal, nullptr, &pl) == STREAMKL_OK ? pl.ws_bytes : 0;
}

size_t streamkl_bwd_workspace_bytes(const streamkl_shape* shape, int setting, int causal) {
    BwdPlan pl{};
    return plan_bwd(shape, setting, causal, nullptr, &pl) == STREAMKL_OK ? pl.ws_bytes : 0;
}

streamkl_status streamkl_bwd(const streamkl_shape* shape, int setting, const float* g, const void* Q1,
                             const void* K1, const void* Q2, const void* K2, const float* KL, const float* LSE1,
                             const float* LSE2, float scale, int causal, void* dQ, void* dK, void* workspace,
                             size_t workspace_bytes, const streamkl_options* opt, streamkl_stream_t stream) {
    streamkl_status st = check_shape(shape, causal);
    if (st != STREAMKL_OK) return st;
    if (setting != 1 && setting != 2) return STREAMKL_ERR_INVALID_ARG;
    const void* qk[4] = {Q1, K1, Q2, K2};
    for (const void* q : qk)
        if (!q || !aligned16(q)) return STREAMKL_ERR_INVALID_ARG;
    const void* rows[4] = {g, KL, LSE1, LSE2};
    for (const void* q : rows)
        if (!q || (reinterpret_cast<uintptr_t>(q) & 3u) != 0) return STREAMKL_ERR_INVALID_ARG;
    if (!dQ || !dK || !aligned16(dQ) || !aligned16(dK)) return STREAMKL_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace)) return STREAMKL_ERR_WORKSPACE;
    BwdPlan pl{};
    if ((st = plan_bwd(shape, setting, causal, opt, &pl)) != STREAMKL_OK) return st;
    if (workspace_bytes < pl.ws_bytes) return STREAMKL_ERR_WORKSPACE;

    const float sc = resolve_scale(scale, shape->d);
    BwdParams p{};
    p.B = shape->B;
    p.H = shape->H;
    p.Nq = shape->Nq;
    p.Nk = shape->Nk;
    p.causal = causal ? 1 : 0;
    p.diag_off = shape->Nk - shape->Nq;
    p.H_kv = kv_heads(shape);
    p.kv_group = shape->H / p.H_kv;
    p.scale = sc;
    p.scale_log2e = sc * 1.4426950408889634f;
    p.g = g;
    p.KL = KL;
    p.LSE1 = LSE1;
    p.LSE2 = LSE2;
    p.dQ = dQ;
    p.dK = dK;
    p.grad_bf16 = pl.bf16 ? 1 : 0;
    p.dQacc = (pl.fused || pl.keysplit)
                  ? (pl.bf16 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kStatusBytes)
                             : static_cast<float*>(dQ))
                  : nullptr;
    p.status = static_cast<unsigned int*>(workspace);
    p.wait_ns = static_cast<unsigned long long>(wait_limit(opt));
    p.inject_stall = (opt && (opt->debug_flags & STREAMKL_DEBUG_INJECT_STALL)) ? 1 : 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t dq_elems = size_t(shape->B) * shape->H * shape->Nq * shape->d;

    if (pl.keysplit) {
        // Q boxes: the Nq rows of all kv_group heads of a key head; K boxes of 128 rows
        CUtensorMap dm[4];
        if (!make_map(&dm[0], Q1, shape, true, shape->Nq, p.kv_group) ||
            !make_map(&dm[1], K1, shape, false, kBlockK) ||
            !make_map(&dm[2], Q2, shape, true, shape->Nq, p.kv_group) || !make_map(&dm[3], K2, shape, false, kBlockK))
            return STREAMKL_ERR_CUDA;
        BwdParams pd = p;
        pd.num_q_tiles = 1;
        pd.num_k_tiles = (shape->Nk + kBlockK - 1) / kBlockK;
        pd.num_splits = pl.splits;
        if (cudaMemsetAsync(p.dQacc, 0, dq_elems * sizeof(float), s) != cudaSuccess) return STREAMKL_ERR_CUDA;
        if (launch_bwd_decode(shape->d, setting, dm, pd, pl.ctas_dec, s) != cudaSuccess) return STREAMKL_ERR_CUDA;
        if (pl.bf16) {
            int sms = 0;
            if (device_sms(&sms) != STREAMKL_OK) return STREAMKL_ERR_CUDA;
            if (launch_to_bf16(p.dQacc, dQ, dq_elems, sms, s) != cudaSuccess) return STREAMKL_ERR_CUDA;
        }
        return STREAMKL_OK;
    }

    // key-tile kernel: Q boxes of 64 rows, K boxes of 128 rows
    CUtensorMap kv[4];
    if (!make_map(&kv[0], Q1, shape, true, 64) || !make_map(&kv[1], K1, shape, false, kBlockK) ||
        !make_map(&kv[2], Q2, shape, true, 64) || !make_map(&kv[3], K2, shape, false, kBlockK))
        return STREAMKL_ERR_CUDA;
    BwdParams pkv = p;
    pkv.num_q_tiles = (shape->Nq + 63) / 64;
    pkv.num_k_tiles = (shape->Nk + kBlockK - 1) / kBlockK;
    if (pl.fused) {
        if (cudaMemsetAsync(p.dQacc, 0, dq_elems * sizeof(float), s) != cudaSuccess) return STREAMKL_ERR_CUDA;
        if (launch_bwd_kv(shape->d, setting, true, kv, pkv, pl.ctas_kv, s) != cudaSuccess) return STREAMKL_ERR_CUDA;
        if (pl.bf16) {
            int sms = 0;
            if (device_sms(&sms) != STREAMKL_OK) return STREAMKL_ERR_CUDA;
            if (launch_to_bf16(p.dQacc, dQ, dq_elems, sms, s) != cudaSuccess) return STREAMKL_ERR_CUDA;
        }
        return STREAMKL_OK;
    }
    // query-tile kernel: Q boxes of 128 rows, K boxes of 64 rows
    CUtensorMap qm[4];
    if (!make_map(&qm[0], Q1, shape, true, kBlockQ) || !make_map(&qm[1], K1, shape, false, 64) ||
        !make_map(&qm[2], Q2, shape, true, kBlockQ) || !make_map(&qm[3], K2, shape, false, 64))
        return STREAMKL_ERR_CUDA;
    BwdParams pq = p;
    pq.num_q_tiles = (shape->Nq + kBlockQ - 1) / kBlockQ;
    pq.num_k_tiles = (shape->Nk + 63) / 64;
    if (launch_bwd_q(shape->d, setting, qm, pq, pl.ctas_q, s) != cudaSuccess) return STREAMKL_ERR_CUDA;
    if (launch_bwd_kv(shape->d, setting, false, kv, pkv, pl.ctas_kv, s) != cudaSuccess) return STREAMKL_ERR_CUDA;
    return STREAMKL_OK;
}

streamkl_status streamkl_bwd_joint_plan(const streamkl_shape* shape, int causal, const streamkl_options* opt,
                                        streamkl_plan* plan) {
    if (!plan) return STREAMKL_ERR_INVALID_ARG;
    streamkl_status st = check_shape(shape, causal);
    if (st != STREAMKL_OK) return st;
    if (opt && (opt->bwd_mode != 0 || (opt->grad_bf16 != 0 && opt->grad_bf16 != 1) ||
                (opt->debug_flags & ~STREAMKL_DEBUG_INJECT_STALL)))
        return STREAMKL_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return STREAMKL_ERR_CUDA;
    const int64_t ctas_kv = int64_t(shape->B) * kv_heads(shape) * ((shape->Nk + kBlockK - 1) / kBlockK);
    const int64_t ctas_q = int64_t(shape->B) * shape->H * ((shape->Nq + kBlockQ - 1) / kBlockQ);
    if (ctas_kv > INT32_MAX || ctas_q > INT32_MAX) return STREAMKL_ERR_UNSUPPORTED;
    plan->path = 5;
    plan->num_splits = 1;
    plan->num_ctas = static_cast<int>(ctas_kv);
    plan->launches = 2;
    plan->workspace_bytes = kStatusBytes;
    return STREAMKL_OK;
}

streamkl_status streamkl_bwd_joint(const streamkl_shape* shape, const float* g, const void* Q1, const void* K1,
                                   const void* Q2, const void* K2, const float* KL, const float* LSE1,
                                   const float* LSE2, float scale, int causal, void* dQ1, void* dK1, void* dQ2,
                                   void* dK2, void* workspace, size_t workspace_bytes, const streamkl_options* opt,
                                   streamkl_stream_t stream) {
    streamkl_status st = check_shape(shape, causal);
    if (st != STREAMKL_OK) return st;
    const void* qk[4] = {Q1, K1, Q2, K2};
    for (const void* q : qk)
        if (!q || !aligned16(q)) return STREAMKL_ERR_INVALID_ARG;
    const void* rows[4] = {g, KL, LSE1, LSE2};
    for (const void* q : rows)
        if (!q || (reinterpret_cast<uintptr_t>(q) & 3u) != 0) return STREAMKL_ERR_INVALID_ARG;
    const void* grads[4] = {dQ1, dK1, dQ2, dK2};
    for (const void* q : grads)
        if (!q || !aligned16(q)) return STREAMKL_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace)) return STREAMKL_ERR_WORKSPACE;
    streamkl_plan plan{};
    if ((st = streamkl_bwd_joint_plan(shape, causal, opt, &plan)) != STREAMKL_OK) return st;
    if (workspace_bytes < plan.workspace_bytes) return STREAMKL_ERR_WORKSPACE;

    const float sc = resolve_scale(scale, shape->d);
    BwdParams p{};
    p.B = shape->B;
    p.H = shape->H;
    p.Nq = shape->Nq;
    p.Nk = shape->Nk;
    p.causal = causal ? 1 : 0;
    p.diag_off = shape->Nk - shape->Nq;
    p.H_kv = kv_heads(shape);
    p.kv_group = shape->H / p.H_kv;
    p.scale = sc;
    p.scale_log2e = sc * 1.4426950408889634f;
    p.g = g;
    p.KL = KL;
    p.LSE1 = LSE1;
    p.LSE2 = LSE2;
    p.dQ = dQ1;
    p.dK = dK1;
    p.dQb = dQ2;
    p.dKb = dK2;
    p.grad_bf16 = (opt && opt->grad_bf16 == 1) ? 1 : 0;
    p.dQacc = nullptr;
    p.status = static_cast<unsigned int*>(workspace);
    p.wait_ns = static_cast<unsigned long long>(wait_limit(opt));
    p.inject_stall = (opt && (opt->debug_flags & STREAMKL_DEBUG_INJECT_STALL)) ? 1 : 0;

    // query-tile kernel: Q boxes of 128 rows, K boxes of 64 rows; key-tile kernel: the reverse
    CUtensorMap qm[4], kv[4];
    if (!make_map(&qm[0], Q1, shape, true, kBlockQ) || !make_map(&qm[1], K1, shape, false, 64) ||
        !make_map(&qm[2], Q2, shape, true, kBlockQ) || !make_map(&qm[3], K2, shape, false, 64) ||
        !make_map(&kv[0], Q1, shape, true, 64) || !make_map(&kv[1], K1, shape, false, kBlockK) ||
        !make_map(&kv[2], Q2, shape, true, 64) || !make_map(&kv[3], K2, shape, false, kBlockK))
        return STREAMKL_ERR_CUDA;
    BwdParams pq = p, pkv = p;
    pq.num_q_tiles = (shape->Nq + kBlockQ - 1) / kBlockQ;
    pq.num_k_tiles = (shape->Nk + 63) / 64;
    pkv.num_q_tiles = (shape->Nq + 63) / 64;
    pkv.num_k_tiles = (shape->Nk + kBlockK - 1) / kBlockK;
    const int ctas_q = static_cast<int>(int64_t(shape->B) * shape->H * pq.num_q_tiles);
    if (launch_bwd_joint(shape->d, qm, kv, pq, pkv, ctas_q, plan.num_ctas, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return STREAMKL_ERR_CUDA;
    return STREAMKL_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward without any allocation: the scratch lives in this file-scope device
// array (every GPU that loads the library holds it until the process exits).
// Host code only ever sees the array's host-side stand-in; its device address
// comes from cudaGetSymbolAddress, with the device of the call current.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = STREAMKL_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.  It is looked up
// on every call (a host-side table lookup once the device code is loaded, and
// no allocation), so no address can outlive the context it belongs to: after
// a cudaDeviceReset the next call resolves the array in the new context.  The
// first call on a device also loads the library's device code there.
streamkl_status noalloc_scratch(void** out) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return STREAMKL_ERR_CUDA;
    *out = ptr;
    return STREAMKL_OK;
}

// Read the device error word at `word_dev` after `stream` drains, clear it if
// set, and map it to a status (shared by both status queries).
streamkl_status read_error_word(void* word_dev, cudaStream_t s, uint32_t* device_error) {
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, word_dev, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return STREAMKL_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return STREAMKL_ERR_CUDA;
    if (word != 0 && cudaMemsetAsync(word_dev, 0, sizeof(word), s) != cudaSuccess) return STREAMKL_ERR_CUDA;
    if (device_error) *device_error = word;
    return word ? STREAMKL_ERR_TIMEOUT : STREAMKL_OK;
}

}  // namespace

extern "C" {

streamkl_status streamkl_fwd_noalloc(const streamkl_shape* shape, const void* Q1, const void* K1, const void* Q2,
                                     const void* K2, float scale, int causal, float* KL, float* LSE1, float* LSE2,
                                     const streamkl_options* opt, streamkl_stream_t stream) {
    FwdPlan pl{};
    streamkl_status st = plan_fwd(shape, causal, opt, &pl);
    if (st != STREAMKL_OK) return st;
    if (pl.ws_bytes > kNoAllocScratchBytes) return STREAMKL_ERR_WORKSPACE;
    void* scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != STREAMKL_OK) return st;
    // the error word must start this call at zero; the partial states need no
    // clearing (every one is written before the combine reads it)
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, kStatusBytes, s) != cudaSuccess) return STREAMKL_ERR_CUDA;
    return streamkl_fwd(shape, Q1, K1, Q2, K2, scale, causal, KL, LSE1, LSE2, scratch, kNoAllocScratchBytes, opt,
                        stream);
}

streamkl_status streamkl_workspace_status(void* workspace, streamkl_stream_t stream, uint32_t* device_error) {
    if (!workspace) return STREAMKL_ERR_INVALID_ARG;
    return read_error_word(workspace, reinterpret_cast<cudaStream_t>(stream), device_error);
}

streamkl_status streamkl_noalloc_status(streamkl_stream_t stream, uint32_t* device_error) {
    void* scratch = nullptr;
    streamkl_status st = noalloc_scratch(&scratch);
    if (st != STREAMKL_OK) return st;
    return read_error_word(scratch, reinterpret_cast<cudaStream_t>(stream), device_error);
}

}  // extern "C"

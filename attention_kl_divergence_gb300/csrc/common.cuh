// common.cuh -- tile sizes, kernel parameter blocks and the per-row finish of
// the online recurrence, shared by the forward, decode, combine and backward
// kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace streamkl {

constexpr int kBlockQ = 128;        // query rows per tile = TMEM lanes = MMA M
constexpr int kBlockK = 128;        // keys per tile = MMA N of the score GEMMs
constexpr int kSwizzleCols = 64;    // bf16 columns per 128-byte swizzled row
constexpr int kDecodeMaxQ = 16;     // the decode kernel handles Nq <= 16
constexpr int kStatusBytes = 256;   // workspace prefix holding the error word

// Device error word bits (set by kernels, read by streamkl_workspace_status).
constexpr uint32_t kErrWaitQ = 1u << 0;      // Q tile never arrived
constexpr uint32_t kErrWaitK = 1u << 1;      // K tile never arrived / stage never freed
constexpr uint32_t kErrWaitS = 1u << 2;      // score tile never produced / consumed
constexpr uint32_t kErrWaitOther = 1u << 3;  // any other barrier
constexpr uint32_t kErrSmemAlign = 1u << 4;  // dynamic shared memory not 1024-byte aligned

// Forward (tile kernel and decode kernel share this block).
struct FwdParams {
    int B, H, Nq, Nk;
    int num_q_tiles;     // ceil(Nq / q rows per tile)
    int num_k_tiles;     // ceil(Nk / kBlockK)
    int num_splits;      // key-range splits per query tile (1 = write final outputs)
    int causal;          // bottom-right causal mask
    int diag_off;        // Nk - Nq
    int kv_group;        // query heads per key head (1 = no sharing)
    int heads_per_cta;   // decode: query heads of one key head packed into a CTA's query columns
    float scale;         // softmax scale
    float scale_log2e;   // scale * log2(e): raw dot product -> base-2 exponent
    float* KL;           // [B*H*Nq]
    float* LSE1;
    float* LSE2;
    float* part;         // partial states [5][num_splits][B*H*Nq] when num_splits > 1
    unsigned int* status;
    unsigned long long wait_ns;
    int inject_stall;    // CTA 0's MMA issuer waits on a barrier nothing arrives on
};

// Backward (both kernels).  Tile counts are in the kernel's own tile units.
struct BwdParams {
    int B, H, Nq, Nk;
    int num_q_tiles;     // bwd_q: 128-row tiles; bwd_kv: 64-row tiles
    int num_k_tiles;     // bwd_q: 64-key tiles;  bwd_kv: 128-key tiles
    int causal;
    int diag_off;        // Nk - Nq
    int H_kv;            // key heads
    int kv_group;        // query heads per key head
    int num_splits;      // key-split backward: key-range splits per key head
    float scale;
    float scale_log2e;
    const float* g;      // [B*H*Nq] upstream gradient dL/dKL
    const float* KL;
    const float* LSE1;
    const float* LSE2;
    void* dQ;            // [B*H*Nq, d] float32 or bf16 (grad_bf16); joint backward: the teacher's dQ1
    void* dK;            // [B*H_kv*Nk, d] float32 or bf16; joint backward: the teacher's dK1
    void* dQb;           // joint backward only: the student's dQ2, laid out like dQ
    void* dKb;           // joint backward only: the student's dK2, laid out like dK
    float* dQacc;        // fused mode: float32 [B*H*Nq, d] the dQ tiles are added into
    int grad_bf16;
    unsigned int* status;
    unsigned long long wait_ns;
    int inject_stall;
};

// Combine of Split-K partial states.
struct CombineParams {
    int rows;            // B*H*Nq
    int num_splits;
    float scale;
    float scale_log2e;
    const float* part;
    float* KL;
    float* LSE1;
    float* LSE2;
};

// Partial state of one row over a key range, in the units the kernels keep:
//   m1, m2  running reference maxima of the raw dot products z = <q, k>
//   l1, l2  sum_j 2^(c (z_t[j] - m_t)),  c = scale * log2(e)
//   acc     sum_j 2^(c (z1[j] - m1)) * (z1[j] - z2[j])
// An empty range has m = -inf and l = acc = 0.
struct RowState {
    float m1, l1, acc, m2, l2;
};

__device__ __forceinline__ void merge_state(RowState& a, const RowState& b, float c) {
    // log-sum-exp merge; acc follows the teacher maximum only
    float m1 = fmaxf(a.m1, b.m1), m2 = fmaxf(a.m2, b.m2);
    float wa1 = (a.m1 == -INFINITY) ? 0.f : exp2f(c * (a.m1 - m1));
    float wb1 = (b.m1 == -INFINITY) ? 0.f : exp2f(c * (b.m1 - m1));
    float wa2 = (a.m2 == -INFINITY) ? 0.f : exp2f(c * (a.m2 - m2));
    float wb2 = (b.m2 == -INFINITY) ? 0.f : exp2f(c * (b.m2 - m2));
    a.l1 = a.l1 * wa1 + b.l1 * wb1;
    a.acc = a.acc * wa1 + b.acc * wb1;
    a.l2 = a.l2 * wa2 + b.l2 * wb2;
    a.m1 = m1;
    a.m2 = m2;
}

// Finish (Methodology 1): LSE_t = scale*m_t + ln l_t and
// KL = scale * acc / l1 + LSE2 - LSE1.
__device__ __forceinline__ void finish_row(const RowState& s, float scale, float& kl, float& lse1, float& lse2) {
    lse1 = scale * s.m1 + logf(s.l1);
    lse2 = scale * s.m2 + logf(s.l2);
    kl = scale * (s.acc / s.l1) + (lse2 - lse1);
}

}  // namespace streamkl

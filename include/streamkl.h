/*
 * streamkl.h -- C ABI of libstreamkl: the fused attention KL divergence on
 * one GB300 (sm_103a) GPU.
 *
 * Method: "StreamKL: Fast and Memory-Efficient KL Divergence for Boosting
 * Attention Distillation" (gist.science/paper/2606.20005, technical summary).
 * For every query row i of every (batch b, head h):
 *
 *     S_t = scale * Q_t K_t^T        t = 1 (teacher), 2 (student)
 *     P_t = softmax(S_t) over the keys row i may see
 *     KL[i] = sum_j P1[i,j] * (log P1[i,j] - log P2[i,j])        (Problem Statement)
 *
 * computed without ever holding an Nq x Nk matrix: the forward streams key
 * tiles through five running scalars per row (Methodology 1, "Online
 * Formulation") and saves only KL, LSE1, LSE2; the backward regenerates
 * P_t = exp(S_t - LSE_t) tile by tile (Methodology 2, "Recomputation
 * Strategy").  Small query counts split the key range across CTAs and merge
 * the partial states (Methodology 3, "Split-K Variant").
 *
 * Conventions shared by every entry point
 *  - Q1, K1, Q2, K2 are bf16 device tensors laid out [B, H, N, d] with d
 *    contiguous (K1, K2 have H_kv heads when keys are shared across a group
 *    of query heads); the element strides of the B, H and N axes are given in
 *    streamkl_shape and must be multiples of 8 elements (16 bytes).  Q1 and
 *    Q2 share one set of strides, K1 and K2 another.  Base pointers must be
 *    16-byte aligned.  d must be 64 or 128.
 *  - KL, LSE1, LSE2 and g are float32 [B, H, Nq], contiguous.  dQ is
 *    [B, H, Nq, d] and dK [B, H_kv, Nk, d], contiguous, float32 (or bf16 on
 *    request); with shared keys dK sums the gradients of every query head of
 *    the group.
 *  - Logarithms are natural.  LSE_t[i] = log sum_j exp(S_t[i,j]) includes the
 *    softmax scale.
 *  - causal != 0 aligns the mask bottom-right: row i sees keys
 *    j <= i + (Nk - Nq).  It requires Nq <= Nk, so no row is empty.
 *  - scale <= 0 (or NaN) selects the default d^-1/2.
 *  - The caller owns every buffer, inputs, outputs and workspace alike.  The
 *    library allocates no device memory, keeps no state between calls and
 *    runs everything asynchronously on the caller's stream.  Arguments are
 *    validated before anything is launched; on an error nothing is launched
 *    and no output is touched.
 *  - streamkl_fwd, streamkl_bwd and streamkl_bwd_joint only enqueue
 *    asynchronous work (kernels and a memset) on the caller's stream: with
 *    buffers allocated beforehand, a sequence of them can be captured into a
 *    CUDA graph and replayed.
 *  - Workspace: the first 256 bytes hold a device error word that kernels set
 *    (they never clear it) when a bounded wait inside them gives up.  Zero the
 *    workspace once when it is allocated; streamkl_workspace_status reads and
 *    clears the word.  A workspace must not be shared by calls that may run
 *    at the same time on different streams.
 */
#ifndef STREAMKL_H
#define STREAMKL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define STREAMKL_API __attribute__((visibility("default")))
#else
#define STREAMKL_API
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* streamkl_stream_t;

typedef enum {
    STREAMKL_OK = 0,
    STREAMKL_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, bad setting */
    STREAMKL_ERR_UNSUPPORTED = 2, /* valid but not implemented here (e.g. d not 64/128) */
    STREAMKL_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the size query said */
    STREAMKL_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed */
    STREAMKL_ERR_TIMEOUT = 5      /* a kernel's bounded wait gave up (device error word) */
} streamkl_status;

typedef struct {
    int32_t B, H, Nq, Nk, d;
    int64_t q_stride_b, q_stride_h, q_stride_n; /* element strides of Q1 and Q2 */
    int64_t k_stride_b, k_stride_h, k_stride_n; /* element strides of K1 and K2 */
    int32_t H_kv; /* key heads: 0 (or H) = one per query head; otherwise H_kv divides H and
                     query head h uses key head h / (H / H_kv) (keys shared by a group) */
} streamkl_shape;

/* Optional knobs; pass NULL for the defaults. */
typedef struct {
    int32_t num_splits;    /* forward and key-split backward: 0 = automatic,        */
                           /*   n >= 1 forces n key-range splits                    */
    int32_t bwd_mode;      /* backward: 0 = automatic, 1 = fused (atomic dQ),        */
                           /*           2 = separate dQ and dK kernels,               */
                           /*           3 = key-split (needs Nq * H / H_kv <= 16)     */
    int64_t wait_limit_ns; /* limit of every in-kernel wait; 0 = default (2 s)      */
    int32_t debug_flags;   /* 0 in normal use; see STREAMKL_DEBUG_*                  */
    int32_t grad_bf16;     /* backward: 0 = float32 dQ/dK, 1 = bf16 dQ/dK            */
} streamkl_options;

/* Test aid for the bounded waits: the first CTA of the main kernel waits on a
 * barrier that nothing arrives on.  The wait gives up after wait_limit_ns,
 * the kernel records STREAMKL_ERR_TIMEOUT in the workspace error word and
 * returns; the outputs of that call are undefined. */
#define STREAMKL_DEBUG_INJECT_STALL 1

/* What a call will launch for a given shape (filled by the plan queries). */
typedef struct {
    int32_t path;       /* 0 = tile forward, 1 = decode (Nq <= 16, causal or not) forward,
                           2 = fused backward, 3 = separate-kernel backward,
                           4 = key-split backward (at most 16 query rows per key head;
                               the automatic choice there),
                           5 = joint backward (both sides, streamkl_bwd_joint) */
    int32_t num_splits; /* key splits of the forward (1 = no combine step) or of the
                           key-split backward */
    int32_t num_ctas;   /* CTAs of the main kernel                          */
    int32_t launches;   /* kernels launched per call                        */
    size_t workspace_bytes;
} streamkl_plan;

/* Plan of streamkl_fwd for this shape on the current device.  Needs a CUDA
 * device (the split count depends on its SM count).  Errors: INVALID_ARG,
 * UNSUPPORTED, CUDA. */
STREAMKL_API streamkl_status streamkl_fwd_plan(const streamkl_shape* shape, int causal, const streamkl_options* opt,
                                  streamkl_plan* plan);

/* Forward (Methodology 1 and 3).  Writes KL, LSE1, LSE2 for every row.
 * workspace must hold at least streamkl_fwd_plan(...).workspace_bytes bytes
 * (256 for the status word plus 20 bytes per row and split when the key
 * range is split).  Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
STREAMKL_API streamkl_status streamkl_fwd(const streamkl_shape* shape, const void* Q1, const void* K1, const void* Q2,
                             const void* K2, float scale, int causal, float* KL, float* LSE1, float* LSE2,
                             void* workspace, size_t workspace_bytes, const streamkl_options* opt,
                             streamkl_stream_t stream);

/* Plan of streamkl_bwd (fused vs separate kernels, workspace). */
STREAMKL_API streamkl_status streamkl_bwd_plan(const streamkl_shape* shape, int setting, int causal,
                                  const streamkl_options* opt, streamkl_plan* plan);

/* Backward (Methodology 2).  Gradient of sum_i g[i] * KL[i] with respect to
 * the trainable side:
 *   setting 1 (teacher fixed): dQ = dL/dQ2, dK = dL/dK2, dS2 = g (P2 - P1)
 *   setting 2 (student fixed): dQ = dL/dQ1, dK = dL/dK1,
 *                              dS1 = g P1 ((S1 - LSE1) - (S2 - LSE2) - KL)
 * and dQ = scale * dS K, dK = scale * dS^T Q.  KL, LSE1, LSE2 are the
 * forward's outputs for the same inputs.  dQ and dK are overwritten; they are
 * float32 unless opt->grad_bf16 selects bf16 (the fused mode then also needs
 * 4 bytes per dQ element of workspace to accumulate in float32).
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
STREAMKL_API streamkl_status streamkl_bwd(const streamkl_shape* shape, int setting, const float* g, const void* Q1,
                             const void* K1, const void* Q2, const void* K2, const float* KL, const float* LSE1,
                             const float* LSE2, float scale, int causal, void* dQ, void* dK, void* workspace,
                             size_t workspace_bytes, const streamkl_options* opt, streamkl_stream_t stream);

/* Joint backward (Methodology 2, both settings at once): the gradient of
 * sum_i g[i] * KL[i] with respect to all four inputs, where the teacher's
 * gradients differentiate through P1 with P2 held fixed (setting 2) and the
 * student's through P2 with P1 held fixed (setting 1):
 *   dQ1 = scale * dS1 K1,  dK1 = scale * dS1^T Q1,  dS1 = g P1 ((S1 - LSE1) - (S2 - LSE2) - KL)
 *   dQ2 = scale * dS2 K2,  dK2 = scale * dS2^T Q2,  dS2 = g (P2 - P1)
 * Results equal streamkl_bwd with setting 2 (dQ1, dK1) and setting 1 (dQ2,
 * dK2), but the scores are regenerated once per kernel for both: a query-tile
 * kernel accumulates dQ1 and dQ2, a key-tile kernel dK1 and dK2, each output
 * written once (no atomics: the results are deterministic).  Layouts, dtypes
 * (opt->grad_bf16) and shared keys as for streamkl_bwd; dQ1/dQ2 are
 * [B, H, Nq, d], dK1/dK2 [B, H_kv, Nk, d].  opt->bwd_mode must be 0 and
 * num_splits is ignored.  The workspace holds the 256-byte error word only
 * (streamkl_bwd_joint_plan: path 5, 2 launches).  For at most 16 query rows
 * per key head (decode shapes) two streamkl_bwd calls, which take the
 * key-split kernel there, are faster.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
STREAMKL_API streamkl_status streamkl_bwd_joint_plan(const streamkl_shape* shape, int causal,
                                                     const streamkl_options* opt, streamkl_plan* plan);
STREAMKL_API streamkl_status streamkl_bwd_joint(const streamkl_shape* shape, const float* g, const void* Q1,
                                                const void* K1, const void* Q2, const void* K2, const float* KL,
                                                const float* LSE1, const float* LSE2, float scale, int causal,
                                                void* dQ1, void* dK1, void* dQ2, void* dK2, void* workspace,
                                                size_t workspace_bytes, const streamkl_options* opt,
                                                streamkl_stream_t stream);

/* Workspace sizes alone, with the default options (opt == NULL): the
 * workspace_bytes field of streamkl_fwd_plan / streamkl_bwd_plan.  They return
 * 0 when the shape, causal flag or setting is invalid or no CUDA device is
 * current (a valid call always needs at least the 256-byte status word).
 * Options that change the size (forced splits, bf16 gradients) need the plan
 * queries. */
STREAMKL_API size_t streamkl_fwd_workspace_bytes(const streamkl_shape* shape, int causal);
STREAMKL_API size_t streamkl_bwd_workspace_bytes(const streamkl_shape* shape, int setting, int causal);

/* Size of the library's own built-in scratch buffer used by streamkl_fwd_noalloc. */
#define STREAMKL_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Forward for callers that cannot allocate device memory themselves -- for
 * example a host program or plugin that is handed tensor pointers by a
 * runtime that owns all device memory and offers it no allocator, or a
 * caller that must not allocate once its memory plan is fixed.  This entry
 * point has no counterpart in the paper; it is streamkl_fwd with the
 * workspace replaced by a fixed buffer that lives inside the library.
 *
 * Same arguments, outputs and validation as streamkl_fwd, minus the
 * workspace.  Neither this call nor anything it launches allocates device
 * memory: the scratch (the device error word plus the Split-K partial
 * states) is a file-scope device array of STREAMKL_NOALLOC_SCRATCH_BYTES
 * bytes that every GPU which loads the library holds until the process
 * exits.  A shape whose plan needs more scratch than that (20 bytes per
 * query row and key split, plus 256) returns STREAMKL_ERR_WORKSPACE and
 * launches nothing.  Every call looks up the array's device address on the
 * current device (a table lookup, no allocation); the first call on a device
 * also loads the library's device code there, so make that first call before
 * any stream capture.  All calls share the one array, so calls that may
 * overlap on the GPU (different streams, or different host threads) race on
 * it and must be serialised by the caller.
 *
 * A bounded wait inside the kernels that gives up (see wait_limit_ns) does
 * not change the return value, which only covers validation and launch: the
 * rows that the giving-up CTA owned come back as NaN, and the scratch's
 * device error word is set.  Read it with streamkl_noalloc_status after the
 * call and before the next one, which clears the word when it starts.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
STREAMKL_API streamkl_status streamkl_fwd_noalloc(const streamkl_shape* shape, const void* Q1, const void* K1,
                                                  const void* Q2, const void* K2, float scale, int causal, float* KL,
                                                  float* LSE1, float* LSE2, const streamkl_options* opt,
                                                  streamkl_stream_t stream);

/* streamkl_workspace_status for the built-in scratch of streamkl_fwd_noalloc
 * on the current device: synchronises `stream`, reads the device error word
 * into *device_error (if not NULL), clears it, and returns
 * STREAMKL_ERR_TIMEOUT if it was set, STREAMKL_OK otherwise (CUDA on a failed
 * copy).  Allocates nothing. */
STREAMKL_API streamkl_status streamkl_noalloc_status(streamkl_stream_t stream, uint32_t* device_error);

/* Synchronises `stream`, reads the workspace's device error word into
 * *device_error (if not NULL), clears it, and returns STREAMKL_ERR_TIMEOUT if
 * it was set, STREAMKL_OK otherwise (or CUDA on a failed copy). */
STREAMKL_API streamkl_status streamkl_workspace_status(void* workspace, streamkl_stream_t stream, uint32_t* device_error);

/* Static description of a status code; never NULL. */
STREAMKL_API const char* streamkl_status_string(streamkl_status status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
STREAMKL_API int streamkl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* STREAMKL_H */

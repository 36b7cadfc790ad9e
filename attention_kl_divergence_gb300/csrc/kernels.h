// kernels.h -- host-side launchers of the CUDA kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace streamkl {

// maps = {Q1, K1, Q2, K2}; Q maps use 128-row boxes (tile) or 16-row boxes (decode).
cudaError_t launch_fwd_tile(int d, const CUtensorMap* maps, const FwdParams& p, int ctas, cudaStream_t stream);
cudaError_t launch_fwd_decode(int d, const CUtensorMap* maps, const FwdParams& p, int ctas, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);
int fwd_tile_stages(int d);

// Backward.  bwd_q maps: Q boxes of 128 rows, K boxes of 64 rows; bwd_kv maps:
// Q boxes of 64 rows, K boxes of 128 rows.
cudaError_t launch_bwd_q(int d, int setting, const CUtensorMap* maps, const BwdParams& p, int ctas,
                         cudaStream_t stream);
cudaError_t launch_to_bf16(const float* in, void* out, size_t n, int sms, cudaStream_t stream);
cudaError_t launch_bwd_kv(int d, int setting, bool fused, const CUtensorMap* maps, const BwdParams& p, int ctas,
                          cudaStream_t stream);
// Key-split backward for at most 16 query rows per key head: Q maps with boxes
// of Nq rows x kv_group heads, K maps with 128-row boxes; p.num_splits set.
// Joint backward (both sides from one recompute of the scores per kernel):
// qmaps as for bwd_q, kvmaps as for bwd_kv; p.dQ/p.dK take the teacher's
// gradients, p.dQb/p.dKb the student's.
cudaError_t launch_bwd_joint(int d, const CUtensorMap* qmaps, const CUtensorMap* kvmaps, const BwdParams& pq,
                             const BwdParams& pkv, int ctas_q, int ctas_kv, cudaStream_t stream);
cudaError_t launch_bwd_decode(int d, int setting, const CUtensorMap* maps, const BwdParams& p, int ctas,
                              cudaStream_t stream);

}  // namespace streamkl

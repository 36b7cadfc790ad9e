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

}  // namespace streamkl

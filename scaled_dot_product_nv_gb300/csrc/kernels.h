// Host-side launchers of the nv_sdpa kernels (one translation unit each) and the
// tiling constants the planner needs from them.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace nvsdpa {

// tiled_simt.cu
size_t tiled_simt_smem_bytes(int64_t d, int64_t dv);
int64_t tiled_simt_rows_per_cta();
int64_t tiled_simt_keys_per_tile();
int64_t merge_max_blocks();
cudaError_t launch_tiled_simt(int dtype, const Params& p, cudaStream_t st);
cudaError_t launch_merge(int dtype, const Params& p, cudaStream_t st);
cudaError_t launch_fill_no_keys(int dtype, const Params& p, cudaStream_t st);

}  // namespace nvsdpa

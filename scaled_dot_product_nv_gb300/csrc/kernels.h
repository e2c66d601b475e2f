// Host-side launchers of the nv_sdpa kernels (one translation unit each) and the
// tiling constants the planner needs from them.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"

namespace nvsdpa {

// tensor_map.cu
constexpr int kDefaultSmCount = 152;  // GB300 (2 dies x 76 SMs), when no device can be asked
// SM count of the current device, read once per device (kDefaultSmCount if none).
int device_sm_count();
// A tiled TMA map of a 16-bit tensor of `rank` dims (innermost first, strides in elements
// for dims 1..rank-1), boxes of 64 x box_rows x 1 ..., 128-byte swizzle, zero fill.
bool encode_tiled_16bit(CUtensorMap* m, int dtype, const void* ptr, int rank, const int64_t* dims,
                        const int64_t* strides_elems, int box_rows);
// The contiguous [outer][rows][inner] case of encode_tiled_16bit.
bool encode_3d(CUtensorMap* m, int dtype, const void* ptr, int64_t inner, int64_t rows, int64_t outer,
               int box_rows);
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per device (thread-safe bitmask).
cudaError_t set_max_dynamic_smem_once(std::atomic<unsigned long long>& configured, const void* fn, int bytes);

// Every kernel of the library is launched as the programmatic dependent of the stream's
// previous kernel: its CTAs may be placed while that kernel's last CTAs run, once all of
// them have signalled (griddepcontrol.launch_dependents), or have exited.  Each kernel
// executes griddepcontrol.wait -- which returns once the previous grid has finished and
// its writes are visible -- before it reads or writes global memory or takes TMEM, so
// the order of the stream's results is that of plain launches; only the launch latency
// and the CTAs' set-up overlap the previous kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// tiled_simt.cu
size_t tiled_simt_smem_bytes(int64_t d, int64_t dv);
int64_t tiled_simt_rows_per_cta();
int64_t tiled_simt_keys_per_tile();
int64_t merge_max_blocks();
cudaError_t launch_tiled_simt(int dtype, const Params& p, cudaStream_t st);
cudaError_t launch_merge(int dtype, const Params& p, cudaStream_t st);
cudaError_t launch_fill_no_keys(int dtype, const Params& p, cudaStream_t st);

// prefill_tc.cu
bool prefill_tc_supported(int dtype, int64_t d, int64_t dv);
int prefill_tc_bn(int64_t d, int64_t dv);
int prefill_tc_q_tiles(int64_t d, int64_t dv, int64_t G);
size_t prefill_tc_smem_bytes(int64_t d, int64_t dv, int bn, int nq, int stg);
int64_t prefill_tc_rows_per_cta(int64_t d, int64_t dv, int64_t G);
size_t prefill_tc_mask_words(int64_t Lk);
// How a tensor-core prefill call is tiled: key tile, Q tiles per CTA, K / V ring depth,
// packed rows or head-local tiles (strided q / out go through 5-D maps), and the grid.
// With nblk > 0, the split-KV form (decode-sized row groups): one Q tile of packed rows
// per CTA and key block.
struct PrefillGeom {
  int bn, nq, stg, head_local, qo5, split, tmem_cols, q_rows, unpadded;
  int64_t n_it, n_rt, grid;
};
PrefillGeom prefill_tc_geometry(int64_t B, int64_t Hkv, int64_t g, int64_t Lq, int64_t d, int64_t dv,
                                bool qo_packed, bool additive, int64_t nblk);
// split: the split-KV form over p.nblk blocks of p.keys_per_blk keys (partials to
// p.part_o / p.part_ml when nblk > 1; the merge pass is the caller's)
cudaError_t launch_prefill_tc(int dtype, const Params& p, uint32_t* mask_bits, bool split, cudaStream_t st);

// decode_mma.cu
bool decode_mma_supported(int dtype, int64_t d, int64_t dv);
int64_t decode_mma_rows_per_warp();
int64_t decode_mma_key_tile();
size_t decode_mma_smem_bytes(int64_t d, int64_t dv);
int decode_mma_ctas_per_sm(int64_t d, int64_t dv);
int decode_mma_warps_per_cta(int64_t d, int64_t dv);
int decode_mma_cta_warps(int64_t warp_units, int64_t d, int64_t dv);
int64_t decode_mma_grid(int64_t warp_units, int64_t d, int64_t dv);
cudaError_t launch_decode_mma(int dtype, const Params& p, cudaStream_t st);
// decode_paged.cu
cudaError_t launch_decode_paged(int dtype, const Params& p, cudaStream_t st);

}  // namespace nvsdpa

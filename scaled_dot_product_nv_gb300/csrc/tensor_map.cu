// Host side of the TMA tensor maps the kernels load through, and the per-device facts
// the launchers need (SM count, one-time function attributes).
//
// cuTensorMapEncodeTiled is a driver entry point; it is looked up once through the
// runtime (no link against libcuda) and shared by every kernel's launcher.
#include <atomic>

#include "kernels.h"

namespace nvsdpa {
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

std::atomic<EncodeTiled> g_encode{nullptr};

EncodeTiled encoder() {
  EncodeTiled fn = g_encode.load(std::memory_order_acquire);
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiled>(ptr);
      g_encode.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

constexpr int kMaxDev = 64;
std::atomic<int> g_sm_count[kMaxDev];

}  // namespace

bool encode_tiled_16bit(CUtensorMap* m, int dtype, const void* ptr, int rank, const int64_t* dims,
                        const int64_t* strides_elems, int box_rows) {
  EncodeTiled enc = encoder();
  if (!enc || rank < 2 || rank > 5) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t box[5], estr[5];
  for (int i = 0; i < rank; ++i) {
    if (dims[i] < 1 || dims[i] > (int64_t(1) << 32)) return false;
    gd[i] = (cuuint64_t)dims[i];
    box[i] = i == 0 ? 64u : (i == 1 ? (cuuint32_t)box_rows : 1u);
    estr[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) {
    const int64_t bytes = strides_elems[i] * 2;
    if (bytes <= 0 || bytes % 16 != 0) return false;
    gs[i] = (cuuint64_t)bytes;
  }
  if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
  return enc(m, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
             (cuuint32_t)rank, const_cast<void*>(ptr), gd, gs, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d(CUtensorMap* m, int dtype, const void* ptr, int64_t inner, int64_t rows, int64_t outer,
               int box_rows) {
  const int64_t dims[3] = {inner, rows, outer};
  const int64_t strides[2] = {inner, inner * rows};
  return encode_tiled_16bit(m, dtype, ptr, 3, dims, strides, box_rows);
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();  // leave no sticky-looking error behind for the caller
    return kDefaultSmCount;
  }
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return kDefaultSmCount;
  }
  g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t set_max_dynamic_smem_once(std::atomic<unsigned long long>& configured, const void* fn, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < kMaxDev ? 1ull << dev : 0ull;
  if (bit && (configured.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  // Two threads may both get here for one device: setting the attribute twice is harmless.
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (bit) configured.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

}  // namespace nvsdpa

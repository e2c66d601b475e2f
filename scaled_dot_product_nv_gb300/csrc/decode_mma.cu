// Decode (Lq <= 8) pass 1 for f16/bf16: stream one block of keys of one KV head from
// HBM through a TMA ring and reduce it against the (up to 16) query rows that share
// that KV head, writing either the final output (one block) or a partial
// (m, l, o) per row for the log-sum-exp merge (sdpa_merge_partials).
//
// This is the split-KV two-pass scheme whose kernels are named in "nuvec-core 0.6.1
// tests/attention_plan.rs" (the vector 2-pass pair, one grid layer per key block); the
// arithmetic per block is the online softmax of "lattice-inference 0.4.0
// src/attention/flash.rs" (run_tiled_attention_head).  The GB300 design:
//
// * The path is bound by reading K and V once.  A producer warp keeps a 3-stage ring of
//   64-key K and V tiles in flight with 3-D TMA (128-byte swizzle, zero fill past Lk);
//   two CTAs per SM keep ~190 KB of loads outstanding per SM.
// * Four compute warps take 16 keys of each tile.  The query rows (g heads x Lq, padded
//   to 16) are the M side of mma.sync.m16n8k16 (f16/bf16 in, f32 accumulate): S = Q K^T
//   over the warp's 16 keys, the online softmax on the accumulator fragments (row max
//   over a lane quad), P re-packed in registers as the A operand of O += P V with V
//   read by ldmatrix.trans.  Tensor-core math keeps the SMs far from the ALU limit that
//   FP32 dot products would hit at 8 query rows per key.
// * At the end of the block the four warps' (m, l, O) are merged through shared memory.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace nvsdpa {
namespace {

using namespace sm100;

constexpr int kRowsDec = 16;     // query rows per CTA (the M of m16n8k16)
constexpr int kKT = 64;          // keys per TMA tile
constexpr int kWarpsC = 4;       // compute warps
constexpr int kDecThreads = (kWarpsC + 1) * 32;
constexpr int kDecStages = 3;
constexpr float kRescaleLog2Dec = 8.0f;
constexpr uint64_t kDrainLimitDec = 1ull << 18;  // polls of <= ~10 us each

struct DecArgs {
  CUtensorMap tmk, tmv;
  Params p;
  int n_rc;       // row chunks of 16 rows per KV head
  int dpanels, dvpanels;
};

template <typename T> struct MmaOp;
template <> struct MmaOp<__half> {
  __device__ static __forceinline__ void run(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) { return pack_f16(lo, hi); }
};
template <> struct MmaOp<__nv_bfloat16> {
  __device__ static __forceinline__ void run(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) { return pack_bf16(lo, hi); }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Byte address of (row, 16-byte chunk) in a [rows][128 B] panel written by TMA with the
// 128-byte swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128(uint32_t panel, int row, int chunk) {
  return panel + row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <typename T, int DMAX, int DV>
__global__ void __launch_bounds__(kDecThreads, (DMAX <= 128 && DV <= 128) ? 2 : 1)
sdpa_decode_mma(const __grid_constant__ DecArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Params& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  const uint32_t k_bytes = a.dpanels * kKT * 128, v_bytes = a.dvpanels * kKT * 128;
  const uint32_t stage_bytes = k_bytes + v_bytes;
  const uint32_t s0 = smem_addr(base);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kDecStages * stage_bytes);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 2 * kDecStages);
  auto full = [&](int s) { return smem_addr(bars + s); };
  auto empty = [&](int s) { return smem_addr(bars + kDecStages + s); };

  // the merge pass may be scheduled once every CTA of this grid is running
  asm volatile("griddepcontrol.launch_dependents;");
  // ---- work unit
  int64_t x = blockIdx.x;
  const int64_t rc = x % a.n_rc; x /= a.n_rc;
  const int64_t blk = x % p.nblk;
  const int64_t bh = x / p.nblk;
  const int64_t b = bh / p.Hkv, hkv = bh % p.Hkv;
  const int64_t j_begin = blk * p.keys_per_blk;
  const int64_t j_end = (j_begin + p.keys_per_blk < p.Lk) ? j_begin + p.keys_per_blk : p.Lk;
  const int n_tiles = (int)((j_end - j_begin + kKT - 1) / kKT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kWarpsC);
    }
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t limit = p.wait_limit;

  // merge buffers (reuse the ring after it drains): per warp m[16], l[16], o[16][DV]
  float* mo = reinterpret_cast<float*>(base);

  if (warp == kWarpsC) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&a.tmk);
      tma_prefetch_desc(&a.tmv);
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kDecStages;
        if (!mbar_wait(empty(s), ((t / kDecStages) & 1) ^ 1, limit, abort)) {
          *abort = 1;
          record_status(p, kStatTimeoutSlotFree);
          break;
        }
        mbar_arrive_expect_tx(full(s), stage_bytes);
        const int key0 = (int)(j_begin + (int64_t)t * kKT);
        for (int pn = 0; pn < a.dpanels; ++pn)
          tma_load_3d(s0 + s * stage_bytes + pn * kKT * 128, &a.tmk, full(s), pn * 64, key0, (int)bh);
        for (int pn = 0; pn < a.dvpanels; ++pn)
          tma_load_3d(s0 + s * stage_bytes + k_bytes + pn * kKT * 128, &a.tmv, full(s), pn * 64, key0, (int)bh);
        issued = t + 1;
      }
      for (int t = issued > kDecStages ? issued - kDecStages : 0; t < issued; ++t)
        mbar_wait(full(t % kDecStages), (t / kDecStages) & 1, kDrainLimitDec, nullptr);
    }
    __syncwarp();
    __syncthreads();  // ring drained: the compute warps may reuse it for the merge
    __syncthreads();  // merge buffers written
    return;
  }

  // ================================================================ compute warps
  // This lane's two query rows (gid and gid + 8 of the chunk).
  const int64_t rows_here = (p.G - rc * kRowsDec < kRowsDec) ? p.G - rc * kRowsDec : kRowsDec;
  int64_t ri[2], last[2];
  bool rok[2];
  const uint8_t* mrow[2];
#pragma unroll
  for (int hrow = 0; hrow < 2; ++hrow) {
    const int r = gid + 8 * hrow;
    rok[hrow] = r < rows_here;
    const int64_t rho = rc * kRowsDec + r;
    ri[hrow] = rok[hrow] ? rho % p.Lq : 0;
    last[hrow] = (p.mask_kind == kMaskCausal) ? causal_last_key(p, ri[hrow]) : p.Lk - 1;
    mrow[hrow] = (p.mask_kind == kMaskBool) ? p.mask + ri[hrow] * p.Lk : nullptr;
  }

  // Q fragments (A operand, row-major m16 x k16 per k-block), straight from global memory.
  constexpr int kKB = DMAX / 16;  // k-blocks of the d bucket
  const int nkb = (int)((p.d + 15) / 16);
  uint32_t qa[kKB][4];
  const T* qbase = reinterpret_cast<const T*>(p.q) + (bh * p.G + rc * kRowsDec) * p.d;
#pragma unroll
  for (int kb = 0; kb < kKB; ++kb) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = gid + 8 * (e & 1);
      const int c = kb * 16 + 2 * tig + 8 * (e >> 1);
      uint32_t v = 0;
      if (kb < nkb && r < rows_here && c < p.d) v = *reinterpret_cast<const uint32_t*>(qbase + r * p.d + c);
      qa[kb][e] = v;
    }
  }

  constexpr int NT = DV / 8;  // n-tiles of the output
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

  bool ok = true;
  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % kDecStages;
    ok = __all_sync(0xffffffffu, mbar_wait(full(s), (t / kDecStages) & 1, limit, abort));
    if (!ok) {
      *abort = 1;
      record_status(p, kStatTimeoutTmaFull);
      break;
    }
    const uint32_t kst = s0 + s * stage_bytes, vst = kst + k_bytes;
    // ---- S = Q K^T over this warp's 16 keys
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int krow = warp * 16 + (lane >> 4) * 8 + (lane & 7);
#pragma unroll
    for (int kb = 0; kb < kKB; ++kb) {
      if (kb < nkb) {
        uint32_t b0, b1, b2, b3;
        const int chunk = (kb & 3) * 2 + ((lane >> 3) & 1);
        ldsm_x4(sw128(kst + (kb >> 2) * kKT * 128, krow, chunk), b0, b1, b2, b3);
        MmaOp<T>::run(sc[0], qa[kb], b0, b1);
        MmaOp<T>::run(sc[1], qa[kb], b2, b3);
      }
    }
    // ---- mask, online softmax (rows gid / gid + 8; keys spread over the lane quad)
    const int64_t jt = j_begin + (int64_t)t * kKT + warp * 16;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hrow = e >> 1;
        const int64_t j = jt + nt * 8 + 2 * tig + (e & 1);
        bool vis = rok[hrow] && j < j_end && j <= last[hrow];
        if (mrow[hrow] && vis) vis = mrow[hrow][j] != 0;
        const float v = vis ? sc[nt][e] * p.scale_log2 : -INFINITY;
        sc[nt][e] = v;
        mx[hrow] = fmaxf(mx[hrow], v);
      }
    }
    float alpha[2];
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      mx[hrow] = fmaxf(mx[hrow], __shfl_xor_sync(0xffffffffu, mx[hrow], 1));
      mx[hrow] = fmaxf(mx[hrow], __shfl_xor_sync(0xffffffffu, mx[hrow], 2));
      const float m_new = fmaxf(m[hrow], mx[hrow]);
      alpha[hrow] = 1.f;
      if (m_new > m[hrow] + kRescaleLog2Dec) {
        alpha[hrow] = ex2(m[hrow] - m_new);
        m[hrow] = m_new;
      }
    }
    uint32_t pa[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int hrow = 0; hrow < 2; ++hrow) {
        const bool none = (m[hrow] == -INFINITY);
        const float p0 = none ? 0.f : ex2(sc[nt][2 * hrow] - m[hrow]);
        const float p1 = none ? 0.f : ex2(sc[nt][2 * hrow + 1] - m[hrow]);
        l[hrow] = l[hrow] * (nt == 0 ? alpha[hrow] : 1.f) + p0 + p1;
        pa[nt * 2 + hrow] = MmaOp<T>::pack(p0, p1);
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      o[j][0] *= alpha[0];
      o[j][1] *= alpha[0];
      o[j][2] *= alpha[1];
      o[j][3] *= alpha[1];
    }
    // ---- O += P V: V tile rows = keys, ldmatrix.trans gives the k16 x n8 B fragments
    const int vrow = warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
    for (int j2 = 0; j2 < NT / 2; ++j2) {
      const int chunk = 2 * j2 + (lane >> 4);  // 16-byte chunk of dv (8 columns)
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(sw128(vst + (chunk >> 3) * kKT * 128, vrow, chunk & 7), b0, b1, b2, b3);
      MmaOp<T>::run(o[2 * j2], pa, b0, b1);
      MmaOp<T>::run(o[2 * j2 + 1], pa, b2, b3);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }

  // ---- merge the four warps through shared memory
  __syncthreads();  // (1) every warp is done with the ring, the producer drained it
#pragma unroll
  for (int hrow = 0; hrow < 2; ++hrow) {
    l[hrow] += __shfl_xor_sync(0xffffffffu, l[hrow], 1);
    l[hrow] += __shfl_xor_sync(0xffffffffu, l[hrow], 2);
  }
  float* wm = mo + warp * (2 * kRowsDec + kRowsDec * DV);
  float* wl = wm + kRowsDec;
  float* wo = wl + kRowsDec;
  if (tig == 0) {
    wm[gid] = m[0];
    wm[gid + 8] = m[1];
    wl[gid] = l[0];
    wl[gid + 8] = l[1];
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int c = j * 8 + 2 * tig;
    wo[gid * DV + c] = o[j][0];
    wo[gid * DV + c + 1] = o[j][1];
    wo[(gid + 8) * DV + c] = o[j][2];
    wo[(gid + 8) * DV + c + 1] = o[j][3];
  }
  __syncthreads();  // (2)
  ok = ok && !*abort;
  if (!ok) return;
  // 128 compute threads: thread -> (row, column group)
  const int tid = threadIdx.x;
  const int dv = (int)p.dv;
  for (int idx = tid; idx < kRowsDec * (DV / 4); idx += kWarpsC * 32) {
    const int r = idx / (DV / 4), c4 = (idx % (DV / 4)) * 4;
    if (r >= rows_here || c4 >= dv) continue;
    const int stride = 2 * kRowsDec + kRowsDec * DV;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarpsC; ++w) M = fmaxf(M, mo[w * stride + r]);
    const int64_t rho = rc * kRowsDec + r;
    const int64_t row_global = (b * p.Hq + hkv * p.g + rho / p.Lq) * p.Lq + rho % p.Lq;
    float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarpsC; ++w) {
        const float mw = mo[w * stride + r];
        const float sw = (mw == -INFINITY) ? 0.f : ex2(mw - M);
        L += mo[w * stride + kRowsDec + r] * sw;
        const float* src = mo + w * stride + 2 * kRowsDec + r * DV + c4;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] += src[e] * sw;
      }
    }
    if (p.nblk == 1) {
      const int64_t h = hkv * p.g + rho / p.Lq;
      const float sk = sink_log2<T>(p, h);
      const float Mf = fmaxf(M, sk);
      float f = 0.f, Lf = 0.f;
      if (Mf != -INFINITY) {
        const float am = (M == -INFINITY) ? 0.f : ex2(M - Mf);
        Lf = L * am + ex2(sk - Mf);
        f = am / Lf;
      }
      T* orow = reinterpret_cast<T*>(p.out) + row_global * p.dv + c4;
      uint2 v;
      v.x = MmaOp<T>::pack(acc[0] * f, acc[1] * f);
      v.y = MmaOp<T>::pack(acc[2] * f, acc[3] * f);
      *reinterpret_cast<uint2*>(orow) = v;
      if (c4 == 0 && p.lse) p.lse[row_global] = (Mf == -INFINITY) ? -INFINITY : (Mf + log2f(Lf)) * kLn2;
    } else {
      float* po = p.part_o + (row_global * p.nblk + blk) * p.dv + c4;
      *reinterpret_cast<float4*>(po) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      if (c4 == 0) {
        p.part_ml[(row_global * p.nblk + blk) * 2 + 0] = M;
        p.part_ml[(row_global * p.nblk + blk) * 2 + 1] = L;
      }
    }
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

EncodeTiled get_encode_dec() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  }
  return fn;
}

bool encode_kv(CUtensorMap* m, int dtype, const void* ptr, int64_t inner, int64_t rows, int64_t outer) {
  EncodeTiled enc = get_encode_dec();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)(inner * 2), (cuuint64_t)(inner * rows * 2)};
  cuuint32_t box[3] = {64, (cuuint32_t)kKT, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int DMAX, int DV>
cudaError_t launch_dec_t(const DecArgs& a, size_t smem, int64_t grid, cudaStream_t st) {
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(configured >> dev & 1ull)) {
    e = cudaFuncSetAttribute(sdpa_decode_mma<T, DMAX, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured |= 1ull << dev;
  }
  sdpa_decode_mma<T, DMAX, DV><<<(unsigned)grid, kDecThreads, smem, st>>>(a);
  return cudaGetLastError();
}

// (d, dv) buckets with a kernel: the smallest bucket covering the head is used; the
// TMA tiles zero-fill the columns between the head size and the bucket.
constexpr int kDecBuckets[][2] = {{64, 64}, {128, 64}, {128, 128}, {192, 128}, {192, 192}, {256, 256}};

int dec_bucket(int64_t d, int64_t dv) {
  for (int i = 0; i < 6; ++i)
    if (d <= kDecBuckets[i][0] && dv <= kDecBuckets[i][1]) return i;
  return -1;
}

template <typename T>
cudaError_t launch_dec_bucket(const DecArgs& a, size_t smem, int64_t grid, cudaStream_t st) {
  switch (dec_bucket(a.p.d, a.p.dv)) {
    case 0: return launch_dec_t<T, 64, 64>(a, smem, grid, st);
    case 1: return launch_dec_t<T, 128, 64>(a, smem, grid, st);
    case 2: return launch_dec_t<T, 128, 128>(a, smem, grid, st);
    case 3: return launch_dec_t<T, 192, 128>(a, smem, grid, st);
    case 4: return launch_dec_t<T, 192, 192>(a, smem, grid, st);
    case 5: return launch_dec_t<T, 256, 256>(a, smem, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool decode_mma_supported(int dtype, int64_t d, int64_t dv) {
  return (dtype == 1 || dtype == 2) && d % 16 == 0 && dv % 16 == 0 && dec_bucket(d, dv) >= 0;
}

int64_t decode_mma_rows_per_cta() { return kRowsDec; }
int64_t decode_mma_key_tile() { return kKT; }
int decode_mma_ctas_per_sm(int64_t d, int64_t dv) {
  const int bk = dec_bucket(d, dv);
  return (bk >= 0 && kDecBuckets[bk][0] <= 128 && kDecBuckets[bk][1] <= 128 &&
          decode_mma_smem_bytes(d, dv) <= 113 * 1024) ? 2 : 1;
}

size_t decode_mma_smem_bytes(int64_t d, int64_t dv) {
  const int64_t dp = (d + 63) / 64, dvp = (dv + 63) / 64;
  const int bk = dec_bucket(d, dv);
  const int64_t dvt = bk >= 0 ? kDecBuckets[bk][1] : 256;
  int64_t ring = kDecStages * (dp + dvp) * kKT * 128;
  const int64_t merge = kWarpsC * (2 * kRowsDec + kRowsDec * dvt) * 4;
  if (merge > ring) ring = merge;
  return (size_t)(ring + 1024 + 64);
}

cudaError_t launch_decode_mma(int dtype, const Params& p, cudaStream_t st) {
  DecArgs a;
  memset(&a, 0, sizeof(a));
  a.p = p;
  const int64_t BH = p.B * p.Hkv;
  if (!encode_kv(&a.tmk, dtype, p.k, p.d, p.Lk, BH) || !encode_kv(&a.tmv, dtype, p.v, p.dv, p.Lk, BH))
    return cudaErrorInvalidValue;
  a.n_rc = (int)((p.G + kRowsDec - 1) / kRowsDec);
  a.dpanels = (int)((p.d + 63) / 64);
  a.dvpanels = (int)((p.dv + 63) / 64);
  const int64_t grid = BH * p.nblk * a.n_rc;
  const size_t smem = decode_mma_smem_bytes(p.d, p.dv);
  return dtype == 1 ? launch_dec_bucket<__half>(a, smem, grid, st) : launch_dec_bucket<__nv_bfloat16>(a, smem, grid, st);
}

}  // namespace nvsdpa

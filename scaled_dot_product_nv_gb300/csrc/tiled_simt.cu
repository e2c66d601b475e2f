// FP32-FMA tiled online-softmax attention (all dtypes), the split-KV merge pass and
// the no-key fill.
//
// The tiled kernel follows the online softmax of "lattice-inference 0.4.0
// src/attention/flash.rs" (run_tiled_attention_head): per key tile, scores, the row
// maximum, the rescale alpha = exp(m_old - m_new) of the running sum and output, and a
// final division by the sum -- with masked keys at minus infinity and an all-masked
// row giving zeros.  Here the scores are kept in log2 units (scale * log2 e folded into
// one multiplier) and exponentials are 2^x.
//
// Work split: one CTA takes 32 query rows that share one KV head -- the g = Hq/Hkv
// query heads of that KV head times their Lq rows, head-major -- and the keys of one
// key block.  With one block it writes the normalised output; with several it writes
// (m, l, o) partials that sdpa_merge_partials combines (the split-KV two-pass scheme
// of the vector kernels named in "nuvec-core 0.6.1 tests/attention_plan.rs").
#include "common.cuh"
#include "kernels.h"

namespace nvsdpa {

namespace {

constexpr int kRows = 32;      // query rows per CTA (one per lane)
constexpr int kKeys = 32;      // keys per tile (8 per warp)
constexpr int kThreads = 128;  // 4 warps
constexpr int kMaxDvPerThread = 64;  // dv <= 256 over 4 warps

template <typename T>
__global__ void __launch_bounds__(kThreads)
sdpa_tiled_simt(const Params p) {
  extern __shared__ float smem[];
  const int d = (int)p.d, dv = (int)p.dv;
  const int ldq = d + 1;  // odd row stride: lane-per-row reads hit distinct banks
  float* Qs = smem;                         // [kRows][d+1]
  float* Ks = Qs + kRows * ldq;             // [kKeys][d+1]
  float* Vs = Ks + kKeys * ldq;             // [kKeys][dv]
  float* Ps = Vs + kKeys * dv;              // [kRows][kKeys+1]
  float* red_max = Ps + kRows * (kKeys + 1);  // [4][32]
  float* red_sum = red_max + 4 * 32;          // [4][32]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the stream's previous kernel has finished before any global access; the merge pass
  // (or the next call) may be scheduled once every CTA of this grid is running
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  int64_t x = blockIdx.x;
  const int64_t rt = x % p.row_tiles; x /= p.row_tiles;
  const int64_t blk = x % p.nblk;
  const int64_t bh = x / p.nblk;  // b * Hkv + hkv
  const int64_t b = bh / p.Hkv, hkv = bh % p.Hkv;
  const int64_t Lkb = seq_keys(p, b);  // keys of this sequence
  const T* Kg = reinterpret_cast<const T*>(p.k);
  const T* Vg = reinterpret_cast<const T*>(p.v);
  const T* Qg = reinterpret_cast<const T*>(p.q);

  // This lane's query row, its absolute position and the keys [lo, hi) it may see.
  const int64_t rho = rt * kRows + lane;
  const bool row_ok = rho < p.G;
  const int64_t hh = row_ok ? rho / p.Lq : 0, i = row_ok ? rho % p.Lq : 0;
  const int64_t h = hkv * p.g + hh;
  const int64_t row_global = (b * p.Hq + h) * p.Lq + i;
  const int64_t pos = i + Lkb - p.Lq;
  const int64_t my_lo = row_key_lo(p, pos), my_hi = row_key_hi(p, pos, Lkb);

  // Stage the 32 query rows (zeros past the last row).
  for (int idx = tid; idx < kRows * d; idx += kThreads) {
    const int r = idx / d, c = idx % d;
    const int64_t rr = rt * kRows + r;
    float val = 0.f;
    if (rr < p.G) val = to_f32<T>(Qg[q_offset(p, b, hkv * p.g + rr / p.Lq, rr % p.Lq) + c]);
    Qs[r * ldq + c] = val;
  }

  // The keys any row of the tile may see, [tile_lo, tile_hi): block blk of the plan's
  // split starts keys_per_blk * blk keys after tile_lo (rows wrap at Lq when a tile spans
  // heads, so the tile's positions are those of its first and last rows, or all of them).
  const int64_t r0 = rt * kRows;
  const int64_t r1 = (r0 + kRows - 1 < p.G - 1) ? r0 + kRows - 1 : p.G - 1;
  const bool one_head = r0 / p.Lq == r1 / p.Lq;
  const int64_t imin = one_head ? r0 % p.Lq : 0, imax = one_head ? r1 % p.Lq : p.Lq - 1;
  const int64_t tile_lo = row_key_lo(p, imin + Lkb - p.Lq);
  const int64_t tile_hi = row_key_hi(p, imax + Lkb - p.Lq, Lkb);
  const int64_t j_begin = tile_lo + blk * p.keys_per_blk;
  int64_t j_end = j_begin + p.keys_per_blk;
  if (j_end > tile_hi) j_end = tile_hi;
  const uint8_t* mrow = (p.mask_kind == kMaskBool) ? p.mask + i * p.Lk : nullptr;
  const bool add = p.mask_kind == kMaskAdd;

  float m = -INFINITY, l = 0.f;
  float o[kMaxDvPerThread];
#pragma unroll
  for (int kk = 0; kk < kMaxDvPerThread; ++kk) o[kk] = 0.f;

  for (int64_t j0 = j_begin; j0 < j_end; j0 += kKeys) {
    __syncthreads();  // previous tile fully consumed (and Qs staged on the first pass)
    for (int idx = tid; idx < kKeys * d; idx += kThreads) {
      const int r = idx / d, c = idx % d;
      const int64_t j = j0 + r;
      Ks[r * ldq + c] = j < j_end ? to_f32<T>(Kg[kv_offset(p, b, hkv, j, p.k_sb, p.k_sh, p.k_sl, p.d) + c]) : 0.f;
    }
    for (int idx = tid; idx < kKeys * dv; idx += kThreads) {
      const int r = idx / dv, c = idx % dv;
      const int64_t j = j0 + r;
      Vs[r * dv + c] = j < j_end ? to_f32<T>(Vg[kv_offset(p, b, hkv, j, p.v_sb, p.v_sh, p.v_sl, p.dv) + c]) : 0.f;
    }
    __syncthreads();

    // Scores of this lane's row against the warp's 8 keys.
    float s[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) s[jj] = 0.f;
    const float* qrow = Qs + lane * ldq;
    const float* kbase = Ks + (warp * 8) * ldq;
    for (int c = 0; c < d; ++c) {
      const float qc = qrow[c];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) s[jj] = fmaf(qc, kbase[jj * ldq + c], s[jj]);
    }
    float tmax = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int64_t j = j0 + warp * 8 + jj;
      bool vis = row_ok && j < j_end && j >= my_lo && j < my_hi;
      if (mrow) vis = vis && mrow[j] != 0;
      float sv = -INFINITY;
      if (vis) sv = add ? fmaf(s[jj], p.scale_log2, amask_log2<T>(p, b, h, i, j)) : s[jj] * p.scale_log2;
      s[jj] = sv;
      tmax = fmaxf(tmax, s[jj]);
    }
    red_max[warp * 32 + lane] = tmax;
    __syncthreads();
    tmax = fmaxf(fmaxf(red_max[lane], red_max[32 + lane]), fmaxf(red_max[64 + lane], red_max[96 + lane]));
    const float m_new = fmaxf(m, tmax);
    float alpha, tsum = 0.f;
    if (m_new == -INFINITY) {  // nothing visible yet: keep zeros, no NaN
      alpha = 1.f;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) Ps[lane * (kKeys + 1) + warp * 8 + jj] = 0.f;
    } else {
      alpha = ex2(m - m_new);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float pj = ex2(s[jj] - m_new);
        Ps[lane * (kKeys + 1) + warp * 8 + jj] = pj;
        tsum += pj;
      }
    }
    red_sum[warp * 32 + lane] = tsum;
    __syncthreads();
    tsum = (red_sum[lane] + red_sum[32 + lane]) + (red_sum[64 + lane] + red_sum[96 + lane]);
    l = l * alpha + tsum;
    m = m_new;
    const float* prow = Ps + lane * (kKeys + 1);
#pragma unroll
    for (int kk = 0; kk < kMaxDvPerThread; ++kk) {
      const int c = warp + 4 * kk;
      if (c < dv) {
        float acc = o[kk] * alpha;
#pragma unroll 8
        for (int j = 0; j < kKeys; ++j) acc = fmaf(prow[j], Vs[j * dv + c], acc);
        o[kk] = acc;
      }
    }
  }
  if (!row_ok) return;

  if (p.nblk == 1) {
    const float sk = sink_log2<T>(p, h);
    const float M = fmaxf(m, sk);
    T* orow = reinterpret_cast<T*>(p.out) + o_offset(p, b, h, i);
    if (M == -INFINITY) {
#pragma unroll
      for (int kk = 0; kk < kMaxDvPerThread; ++kk) {
        const int c = warp + 4 * kk;
        if (c < dv) orow[c] = from_f32<T>(0.f);
      }
      if (warp == 0 && p.lse) p.lse[row_global] = -INFINITY;
      return;
    }
    const float a = ex2(m - M);
    const float L = l * a + ex2(sk - M);
    const float f = a / L;
#pragma unroll
    for (int kk = 0; kk < kMaxDvPerThread; ++kk) {
      const int c = warp + 4 * kk;
      if (c < dv) orow[c] = from_f32<T>(o[kk] * f);
    }
    if (warp == 0 && p.lse) p.lse[row_global] = (M + log2f(L)) * kLn2;
  } else {
    float* po = p.part_o + (row_global * p.nblk + blk) * p.dv;
#pragma unroll
    for (int kk = 0; kk < kMaxDvPerThread; ++kk) {
      const int c = warp + 4 * kk;
      if (c < dv) po[c] = o[kk];
    }
    if (warp == 0) {
      p.part_ml[(row_global * p.nblk + blk) * 2 + 0] = m;
      p.part_ml[(row_global * p.nblk + blk) * 2 + 1] = l;
    }
  }
}

// Pass 2 of split-KV: one CTA (8 warps) per query row merges its nblk partials,
//   M = max(max_blk m_blk, sink),  L = sum_blk l_blk 2^(m_blk - M) + 2^(sink - M),
//   out = sum_blk o_blk 2^(m_blk - M) / L,  lse = (M + log2 L) ln 2.
// Warp w takes blocks w, w+8, ...; each lane owns 4 columns per 128.  The loads of a
// batch of blocks are all issued before any is used, so a row costs about one memory
// latency instead of one per block.  Launched as a programmatic dependent of pass 1:
// griddepcontrol.wait holds it until pass 1 has finished and its writes are visible.
constexpr int kMergeWarps = 8;
constexpr int kMaxBlk = 1024;
constexpr int kMergeBatch = 12;  // blocks per warp whose loads are in flight together

template <typename T>
__global__ void __launch_bounds__(kMergeWarps * 32)
sdpa_merge_partials(const Params p) {
  __shared__ float red[kMergeWarps];
  __shared__ float part[kMergeWarps][256 + 1];  // per-warp partial sums of one row, + L
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");  // (the next call's set-up may overlap)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = blockIdx.x;
  const int64_t h = (row / p.Lq) % p.Hq;
  const int nb = (int)p.nblk;
  const int dv = (int)p.dv;
  const float* ml = p.part_ml + row * p.nblk * 2;
  const float* po = p.part_o + row * p.nblk * p.dv;
  const float sk = sink_log2<T>(p, h);

  // Warp w takes blocks w, w + 8, w + 16, ... and lane l columns 4 l .. 4 l + 3 of each
  // 128-column group; a batch is kMergeBatch such blocks, loaded together.
  float mk[kMergeBatch], lk[kMergeBatch];
  float4 o[kMergeBatch];
  auto load_batch = [&](int k0, int c0) {
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int k = k0 + u * kMergeWarps;
      const bool in = k < nb;
      mk[u] = in ? ml[2 * k] : -INFINITY;
      lk[u] = in ? ml[2 * k + 1] : 0.f;
      o[u] = (in && c0 < dv) ? *reinterpret_cast<const float4*>(po + (int64_t)k * p.dv + c0)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  // The first batch and this thread's share of the block maxima are loaded before any
  // of them is used: up to 8 x kMergeBatch blocks cost one trip to memory.
  float M = sk;
  for (int k = threadIdx.x; k < nb; k += kMergeWarps * 32) M = fmaxf(M, ml[2 * k]);
  load_batch(warp, lane * 4);
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red[warp] = M;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, red[w]);
  T* orow = reinterpret_cast<T*>(p.out) + o_offset(p, row / (p.Lq * p.Hq), h, row % p.Lq);
  if (M == -INFINITY) {
    for (int c = threadIdx.x; c < dv; c += kMergeWarps * 32) orow[c] = from_f32<T>(0.f);
    if (threadIdx.x == 0 && p.lse) p.lse[row] = -INFINITY;
    return;
  }
  float L = 0.f;
  for (int c0 = lane * 4; c0 < dv; c0 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = warp; k0 < nb; k0 += kMergeWarps * kMergeBatch) {
      if (c0 != lane * 4 || k0 != warp) load_batch(k0, c0);
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const float w = (mk[u] == -INFINITY) ? 0.f : ex2(mk[u] - M);
        acc.x = fmaf(o[u].x, w, acc.x);
        acc.y = fmaf(o[u].y, w, acc.y);
        acc.z = fmaf(o[u].z, w, acc.z);
        acc.w = fmaf(o[u].w, w, acc.w);
        if (c0 == lane * 4) L = fmaf(lk[u], w, L);
      }
    }
    part[warp][c0] = acc.x;
    part[warp][c0 + 1] = acc.y;
    part[warp][c0 + 2] = acc.z;
    part[warp][c0 + 3] = acc.w;
  }
  if (lane == 0) part[warp][256] = L;
  __syncthreads();
  float Lt = ex2(sk - M);
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) Lt += part[w][256];
  const float inv = 1.f / Lt;
  for (int c = threadIdx.x; c < dv; c += kMergeWarps * 32) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) s += part[w][c];
    orow[c] = from_f32<T>(s * inv);
  }
  if (threadIdx.x == 0 && p.lse) p.lse[row] = (M + log2f(Lt)) * kLn2;
}

// Pass 2 for few key blocks (nblk <= kWarpMergeMax): one warp per query row, eight rows
// per CTA, the same sums as above.  Lane k (< nblk) loads block k's (m, l); every lane
// loads its four columns of each 128-column group from every block; all of these loads
// are in flight together, so a row costs one trip to memory, and no CTA barrier is
// needed.
constexpr int kWarpMergeMax = 16;

template <typename T>
__global__ void __launch_bounds__(kMergeWarps * 32)
sdpa_merge_partials_warp(const Params p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");  // (the next call's set-up may overlap)
  const int lane = threadIdx.x & 31;
  const int64_t rows = p.B * p.Hq * p.Lq;
  const int64_t row = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int64_t h = (row / p.Lq) % p.Hq;
  const int nb = (int)p.nblk;
  const int dv = (int)p.dv;
  const float* ml = p.part_ml + row * p.nblk * 2;
  const float* po = p.part_o + row * p.nblk * p.dv;
  const float mk = lane < nb ? ml[2 * lane] : -INFINITY;
  const float lk = lane < nb ? ml[2 * lane + 1] : 0.f;
  float4 o[2][kWarpMergeMax];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int c0 = j * 128 + lane * 4;
#pragma unroll
    for (int k = 0; k < kWarpMergeMax; ++k)
      o[j][k] = (k < nb && c0 < dv) ? *reinterpret_cast<const float4*>(po + (int64_t)k * p.dv + c0)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float sk = sink_log2<T>(p, h);
  float M = fmaxf(mk, sk);
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  T* orow = reinterpret_cast<T*>(p.out) + o_offset(p, row / (p.Lq * p.Hq), h, row % p.Lq);
  if (M == -INFINITY) {
    for (int c = lane; c < dv; c += 32) orow[c] = from_f32<T>(0.f);
    if (lane == 0 && p.lse) p.lse[row] = -INFINITY;
    return;
  }
  const float w = (mk == -INFINITY) ? 0.f : ex2(mk - M);  // block lane's weight
  float L = lk * w;
#pragma unroll
  for (int off = 16; off; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  L += ex2(sk - M);
  const float inv = 1.f / L;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kWarpMergeMax; ++k) {
      const float wk = __shfl_sync(0xffffffffu, w, k);  // 0 past nblk
      acc.x = fmaf(o[j][k].x, wk, acc.x);
      acc.y = fmaf(o[j][k].y, wk, acc.y);
      acc.z = fmaf(o[j][k].z, wk, acc.z);
      acc.w = fmaf(o[j][k].w, wk, acc.w);
    }
    const int c0 = j * 128 + lane * 4;
    if (c0 < dv) {
      orow[c0] = from_f32<T>(acc.x * inv);
      orow[c0 + 1] = from_f32<T>(acc.y * inv);
      orow[c0 + 2] = from_f32<T>(acc.z * inv);
      orow[c0 + 3] = from_f32<T>(acc.w * inv);
    }
  }
  if (lane == 0 && p.lse) p.lse[row] = (M + log2f(L)) * kLn2;
}

// Lk == 0: every row sees no key.  out = 0; lse = the sink, or -inf without sinks.
template <typename T>
__global__ void sdpa_fill_no_keys(const Params p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t rows = p.B * p.Hq * p.Lq;
  const int64_t n = rows * p.dv;
  T* out = reinterpret_cast<T*>(p.out);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = e / p.dv, c = e % p.dv;
    const int64_t i = row % p.Lq, h = (row / p.Lq) % p.Hq, b = row / (p.Lq * p.Hq);
    out[o_offset(p, b, h, i) + c] = from_f32<T>(0.f);
    if (p.lse && c == 0)
      p.lse[row] = p.has_sinks ? to_f32<T>(reinterpret_cast<const T*>(p.sinks)[h]) : -INFINITY;
  }
}

template <typename T>
cudaError_t launch_simt_t(const Params& p, cudaStream_t st) {
  const size_t smem = tiled_simt_smem_bytes(p.d, p.dv);
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = set_max_dynamic_smem_once(configured, (const void*)sdpa_tiled_simt<T>,
                                            (int)tiled_simt_smem_bytes(256, 256));
  if (e != cudaSuccess) return e;
  const int64_t grid = p.B * p.Hkv * p.nblk * p.row_tiles;
  return launch_dependent(sdpa_tiled_simt<T>, dim3((unsigned)grid), dim3(kThreads), smem, st, p);
}

template <typename T>
cudaError_t launch_merge_t(const Params& p, cudaStream_t st) {
  const int64_t rows = p.B * p.Hq * p.Lq;
  // (its grid is set up while pass 1 drains)
  if (p.nblk <= kWarpMergeMax && p.dv <= 256)
    return launch_dependent(sdpa_merge_partials_warp<T>, dim3((unsigned)((rows + kMergeWarps - 1) / kMergeWarps)),
                            dim3(kMergeWarps * 32), 0, st, p);
  return launch_dependent(sdpa_merge_partials<T>, dim3((unsigned)rows), dim3(kMergeWarps * 32), 0, st, p);
}

template <typename T>
cudaError_t launch_fill_t(const Params& p, cudaStream_t st) {
  const int64_t n = p.B * p.Hq * p.Lq * p.dv;
  int64_t grid = (n + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return launch_dependent(sdpa_fill_no_keys<T>, dim3((unsigned)grid), dim3(256), 0, st, p);
}

}  // namespace

size_t tiled_simt_smem_bytes(int64_t d, int64_t dv) {
  return sizeof(float) * (size_t)(kRows * (d + 1) + kKeys * (d + 1) + kKeys * dv +
                                  kRows * (kKeys + 1) + 2 * 4 * 32);
}

int64_t tiled_simt_rows_per_cta() { return kRows; }
int64_t tiled_simt_keys_per_tile() { return kKeys; }
int64_t merge_max_blocks() { return kMaxBlk; }

cudaError_t launch_tiled_simt(int dtype, const Params& p, cudaStream_t st) {
  switch (dtype) {
    case 0: return launch_simt_t<float>(p, st);
    case 1: return launch_simt_t<__half>(p, st);
    default: return launch_simt_t<__nv_bfloat16>(p, st);
  }
}

cudaError_t launch_merge(int dtype, const Params& p, cudaStream_t st) {
  switch (dtype) {
    case 0: return launch_merge_t<float>(p, st);
    case 1: return launch_merge_t<__half>(p, st);
    default: return launch_merge_t<__nv_bfloat16>(p, st);
  }
}

cudaError_t launch_fill_no_keys(int dtype, const Params& p, cudaStream_t st) {
  switch (dtype) {
    case 0: return launch_fill_t<float>(p, st);
    case 1: return launch_fill_t<__half>(p, st);
    default: return launch_fill_t<__nv_bfloat16>(p, st);
  }
}

}  // namespace nvsdpa

// The decode kernel template (pass 1 of split-KV, f16/bf16), shared by the translation
// units that instantiate it: decode_mma.cu (keys and values as strided [B, Hkv, Lk, D]
// views) and decode_paged.cu (keys and values in paged caches).  See decode_mma.cu for
// the design.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace nvsdpa {
namespace dec {

using namespace sm100;

// How a decode kernel reads keys and values.
enum {
  kKvTma = 0,        // strided [B][Hkv][Lk][D] views, one 4-D TMA box per tile and panel
  kKvPagedTma = 1,   // paged caches, TMA boxes of gcd(block size, key tile) rows, each from
                     // its block (block size a multiple of 8)
  kKvPagedRows = 2   // paged caches, 16-byte copies of every key row (any block size)
};

using namespace sm100;

constexpr int kRowsDec = 16;     // query rows per warp (the M of m16n8k16)
constexpr int kKTMax = 32;       // the largest key tile of any bucket (key blocks are multiples of 64)
constexpr float kRescaleLog2Dec = 8.0f;
constexpr uint64_t kDrainLimitDec = 1ull << 18;  // polls of <= ~10 us each

struct DecArgs {
  CUtensorMap tmk, tmv;   // the K and V views, or (paged) the caches as [blocks][Hkv][page][D]
  Params p;
  int n_rc;       // row tiles of 16 rows per KV head
  int dpanels, dvpanels;
  int sub_rows;   // kKvPagedTma: rows of one TMA box, gcd(page, key tile)
  int wpc;        // warps per CTA of this launch (at most the bucket's WPC)
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

// The transpose of an 8 x 8 matrix of 16-bit values held as an m8n8 fragment (thread t
// holds row t / 4, columns 2 (t % 4) and 2 (t % 4) + 1): the same fragment of the transpose.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Byte address of (row, 16-byte chunk) in a [rows][128 B] panel written by TMA with the
// 128-byte swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128(uint32_t panel, int row, int chunk) {
  return panel + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// Shape of each (d, dv) bucket's kernel: keys per tile, warps per CTA and ring stages
// per warp, so that about 192 KB of loads are in flight per SM.  The per-warp mma.sync
// work is what bounds the stream, so heads up to 128 run 8 warps (two per scheduler) on
// 16-key tiles; larger heads, whose accumulators would not fit 8 warps' registers, run
// 3-4 warps on 32-key tiles.  (Measured on the 8 x 32/4 x 32769-key f16 decode: 4 warps
// of 32-key tiles 4430 GB/s, 8 warps of 16-key tiles 5390 GB/s; 6, 7, 10 or 12 warps
// lose to an uneven share of key blocks or to register spills.)
template <int DMAX, int DV> struct DecShape {
  static constexpr bool kSmallHead = DMAX <= 128 && DV <= 128;
  static constexpr int KT = kSmallHead ? 16 : 32;
  static constexpr int kStageBytes = (DMAX / 64 + DV / 64) * KT * 128;
  static constexpr int WPC = kSmallHead ? 8 : (DMAX >= 256) ? 3 : 4;
  static constexpr int ST = (WPC * 3 * kStageBytes <= 192 * 1024) ? 3 : 2;
  static constexpr int kSmem = WPC * ST * kStageBytes + 1024 + WPC * ST * 8 + 64;
  static constexpr int kCtasPerSm = (kSmem <= 113 * 1024) ? 2 : 1;
};

// SW (up to 8 query rows per KV head, heads up to 128): the products are taken transposed,
// S^T = K Q^T and O^T = V^T P^T, so that the 16 rows of each m16n8k16 are keys and value
// columns, and the 8 query rows are its N side -- no padding rows, half the products of
// the row-major form.  P^T reaches the B operand of O^T by an in-register 8 x 8 transpose.
template <typename T, int DMAX, int DV, int KV, bool SW>
__global__ void __launch_bounds__(DecShape<DMAX, DV>::WPC * 32, DecShape<DMAX, DV>::kCtasPerSm)
sdpa_decode_mma(const __grid_constant__ DecArgs a) {
  static_assert(!SW || (DMAX <= 128 && DV <= 128 && DecShape<DMAX, DV>::KT == 16), "the transposed form");
  using Sh = DecShape<DMAX, DV>;
  constexpr int ST = Sh::ST;
  constexpr int kKT = Sh::KT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Params& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  const uint32_t k_bytes = a.dpanels * kKT * 128, v_bytes = a.dvpanels * kKT * 128;
  const uint32_t stage_bytes = k_bytes + v_bytes;
  const uint32_t ring = smem_addr(base) + warp * ST * stage_bytes;  // this warp's stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + a.wpc * ST * stage_bytes);
  auto full = [&](int s) { return smem_addr(bars + warp * ST + s); };

  // the stream's previous kernel has finished before any global access; the merge pass
  // may be scheduled once every CTA of this grid is running
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.wpc * ST; ++i) mbar_init(smem_addr(bars + i), 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- this warp's work: (b, KV head, row tile) and a contiguous run of its key blocks
  const int64_t gw = (int64_t)blockIdx.x * a.wpc + warp;
  if (gw >= p.B * p.Hkv * a.n_rc * p.spans) return;
  const int64_t span = gw % p.spans;
  const int64_t unit = gw / p.spans;
  const int64_t rc = unit % a.n_rc;
  const int64_t bh = unit / a.n_rc;
  const int64_t b = bh / p.Hkv, hkv = bh % p.Hkv;
  const int64_t Lkb = seq_keys(p, b);
  const int64_t rows_here = (p.G - rc * kRowsDec < kRowsDec) ? p.G - rc * kRowsDec : kRowsDec;

  // The keys any row of the tile may see, [u_lo, u_hi): the blocks of the plan's split are
  // cut from u_lo (with a window, the band's first key), so that a one-query row's blocks
  // are those of a call over exactly its band.
  const int64_t r0 = rc * kRowsDec, r1 = r0 + rows_here - 1;
  const bool one_head = r0 / p.Lq == r1 / p.Lq;
  const int64_t imin = one_head ? r0 % p.Lq : 0, imax = one_head ? r1 % p.Lq : p.Lq - 1;
  // (paged TMA boxes hold whole slices of a block: the range starts on a key-tile
  // boundary there, the keys before the band masked)
  int64_t u_lo = row_key_lo(p, imin + Lkb - p.Lq);
  if constexpr (KV == kKvPagedTma) u_lo -= u_lo % kKT;
  const int64_t u_hi = row_key_hi(p, imax + Lkb - p.Lq, Lkb);
  const int64_t c_begin = span * p.nblk / p.spans, c_end = (span + 1) * p.nblk / p.spans;
  const int64_t key_begin = u_lo + c_begin * p.keys_per_blk;
  int64_t key_end = u_lo + c_end * p.keys_per_blk;
  if (key_end > u_hi) key_end = u_hi;
  const int n_tiles = key_end > key_begin ? (int)((key_end - key_begin + kKT - 1) / kKT) : 0;
  const int tpb = (int)(p.keys_per_blk / kKT);  // tiles per (full) key block
  const uint64_t limit = p.wait_limit;

  // Paged TMA: lane l holds the (clamped) table entry of page ebase + l; a tile's boxes
  // take their block from it by a shuffle, refilled 32 pages at a time.
  int64_t ebase = -(int64_t(1) << 40);
  int ent = 0;
  // (keys and pages in 32 bits when the table's capacity fits: a 64-bit division per tile
  // costs more than the tile's other integer work)
  const bool cap32 = p.max_pages * p.page <= 0x7fffffff;
  auto page_of = [&](int64_t key, int& pos) -> int64_t {  // page index and position in it
    if (cap32) {
      const uint32_t k32 = (uint32_t)key, pg32 = k32 / (uint32_t)p.page;
      pos = (int)(k32 - pg32 * (uint32_t)p.page);
      return pg32;
    }
    pos = (int)(key % p.page);
    return key / p.page;
  };
  int64_t next_key = -1, next_pg = 0;  // the next tile's first key, its page and position
  int next_pos = 0;
  auto page_entry = [&](int64_t pg) -> int {  // every lane, the same page
    if (pg >= p.max_pages) pg = p.max_pages - 1;  // only past the sequence's end
    if (pg < ebase || pg >= ebase + 32) {
      ebase = pg;
      const int64_t idx = pg + lane < p.max_pages ? pg + lane : p.max_pages - 1;
      int64_t e = p.table[b * p.max_pages + idx];
      ent = (int)(e < 0 ? 0 : (e >= p.num_pages ? p.num_pages - 1 : e));
    }
    return __shfl_sync(0xffffffffu, ent, (int)(pg - ebase));
  };

  // tile i of the run into ring slot i % ST (called by every lane): by TMA from lane 0,
  // or (kKvPagedRows) by 16-byte copies of every lane, key row by key row through the page
  // table, rows outside [key_begin, key_end) and columns past the head zero-filled
  const uint64_t l2_once = l2_policy_evict_first();  // each key and value is read once
  const T* kg = reinterpret_cast<const T*>(p.k);
  const T* vg = reinterpret_cast<const T*>(p.v);
  auto issue = [&](int i) {
    const int s = i % ST;
    const int64_t key0 = key_begin + (int64_t)i * kKT;
    if constexpr (KV == kKvTma) {
      if (lane == 0) {
        mbar_arrive_expect_tx(full(s), stage_bytes);
        for (int pn = 0; pn < a.dpanels; ++pn)
          tma_load_4d_hint(ring + s * stage_bytes + pn * kKT * 128, &a.tmk, full(s), pn * 64, (int)key0, (int)hkv,
                           (int)b, l2_once);
        for (int pn = 0; pn < a.dvpanels; ++pn)
          tma_load_4d_hint(ring + s * stage_bytes + k_bytes + pn * kKT * 128, &a.tmv, full(s), pn * 64, (int)key0,
                           (int)hkv, (int)b, l2_once);
      }
    } else if constexpr (KV == kKvPagedTma) {
      const int R = a.sub_rows;
      if (lane == 0) mbar_arrive_expect_tx(full(s), stage_bytes);
      // the page and position of key0: carried over from the previous tile (tiles are
      // issued in order, kKT keys apart), divided out only for the run's first
      if (key0 != next_key) next_pg = page_of(key0, next_pos);
      int64_t pg = next_pg;
      int pos = next_pos;
      for (int u = 0; u * R < kKT; ++u) {
        const int blk = page_entry(pg);
        if (lane == 0) {
          for (int pn = 0; pn < a.dpanels; ++pn)
            tma_load_4d_hint(ring + s * stage_bytes + pn * kKT * 128 + u * R * 128, &a.tmk, full(s), pn * 64, pos,
                             (int)hkv, blk, l2_once);
          for (int pn = 0; pn < a.dvpanels; ++pn)
            tma_load_4d_hint(ring + s * stage_bytes + k_bytes + pn * kKT * 128 + u * R * 128, &a.tmv, full(s),
                             pn * 64, pos, (int)hkv, blk, l2_once);
        }
        // (a box never crosses a page: R divides the page size)
        pos += R;
        if (pos >= (int)p.page) {
          pos -= (int)p.page;
          ++pg;
        }
      }
      next_key = key0 + kKT;
      next_pg = pg;
      next_pos = pos;
    } else {
      const int ck = (int)(p.d / 8), cv = (int)(p.dv / 8);  // 16-byte chunks of a K / V row
      const int pk = a.dpanels * 8, pv = a.dvpanels * 8;    // chunks of a panelled smem row
      const int per_row = pk + pv;
      for (int e = lane; e < kKT * per_row; e += 32) {
        const int r = e / per_row, cc = e - r * per_row;
        const int64_t j = key0 + r;
        const bool is_k = cc < pk;
        const int ch = is_k ? cc : cc - pk;               // chunk within the K or V row
        const bool in = j < key_end && ch < (is_k ? ck : cv);
        const T* src = kg;
        if (in)
          src = is_k ? kg + kv_offset(p, b, hkv, j, 0, 0, 0, p.d) + ch * 8
                     : vg + kv_offset(p, b, hkv, j, 0, 0, 0, p.dv) + ch * 8;
        const uint32_t panel = ring + s * stage_bytes + (is_k ? 0u : k_bytes) + (ch >> 3) * kKT * 128;
        cp_async16_zfill(sw128(panel, r, ch & 7), src, in ? 16u : 0u);
      }
    }
  };
  // waits until tile i has landed in its slot (bounded for TMA; the row copies are this
  // warp's own and always complete).  A paged TMA tile reads whole block slices, so the
  // value rows past the sequence's end (whatever the cache holds there, NaN included)
  // are cleared before any product reads them.
  auto landed = [&](int i) -> bool {
    if constexpr (KV == kKvPagedRows) {
      __syncwarp();
      return true;
    } else {
      if (!__all_sync(0xffffffffu, mbar_wait(full(i % ST), (i / ST) & 1, limit, nullptr))) return false;
      if constexpr (KV == kKvPagedTma) {
        const int64_t key0 = key_begin + (int64_t)i * kKT;
        if (key0 + kKT > Lkb) {
          const int first = key0 >= Lkb ? 0 : (int)(Lkb - key0);
          const uint32_t vst = ring + (i % ST) * stage_bytes + k_bytes;
          for (int e = lane; e < (kKT - first) * a.dvpanels * 8; e += 32) {
            const int r = first + e / (a.dvpanels * 8), cc = e % (a.dvpanels * 8);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sw128(vst + (cc >> 3) * kKT * 128, r, cc & 7)),
                         "r"(0u)
                         : "memory");
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }
      }
      return true;
    }
  };
  if (KV != kKvPagedRows && lane == 0) {
    tma_prefetch_desc(&a.tmk);
    tma_prefetch_desc(&a.tmv);
  }

  // This lane's two query rows (gid and gid + 8 of the row tile; SW: 2 tig and 2 tig + 1):
  // the keys [lo, hi) each may see (32-bit: the planner sends no longer sequence here) and
  // its mask row (boolean bytes or additive values, by mask kind).
  int lo[2], hi[2];
  bool rok[2];
  const void* mk[2];
  const bool bool_mask = p.mask_kind == kMaskBool, add_mask = p.mask_kind == kMaskAdd;
#pragma unroll
  for (int hrow = 0; hrow < 2; ++hrow) {
    const int r = SW ? 2 * tig + hrow : gid + 8 * hrow;
    rok[hrow] = r < rows_here;
    const int64_t rho = rc * kRowsDec + (rok[hrow] ? r : 0);
    const int64_t i = rho % p.Lq, h = hkv * p.g + rho / p.Lq;
    const int64_t pos = i + Lkb - p.Lq;
    lo[hrow] = (int)row_key_lo(p, pos);
    hi[hrow] = (int)row_key_hi(p, pos, Lkb);
    mk[hrow] = bool_mask ? static_cast<const void*>(p.mask + i * p.Lk)
                         : (add_mask ? static_cast<const void*>(reinterpret_cast<const T*>(p.amask) + b * p.am_sb +
                                                                h * p.am_sh + i * p.Lk)
                                     : nullptr);
  }

  // Q fragments (A operand, row-major m16 x k16 per k-block; SW: B operand, Q^T k16 x n8,
  // query row gid), straight from global memory.
  constexpr int kKB = DMAX / 16;  // k-blocks of the d bucket
  const int nkb = (int)((p.d + 15) / 16);
  uint32_t qa[kKB][SW ? 2 : 4];
  if constexpr (SW) {
    const bool gok = gid < rows_here;
    const int64_t rho = rc * kRowsDec + (gok ? gid : 0);
    const T* qrow = reinterpret_cast<const T*>(p.q) + q_offset(p, b, hkv * p.g + rho / p.Lq, rho % p.Lq);
#pragma unroll
    for (int kb = 0; kb < kKB; ++kb) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = kb * 16 + 2 * tig + 8 * e;
        uint32_t v = 0;
        if (kb < nkb && gok && c < p.d) v = *reinterpret_cast<const uint32_t*>(qrow + c);
        qa[kb][e] = v;
      }
    }
  } else {
    const T* qrow[2];
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      const int64_t rho = rc * kRowsDec + (rok[hrow] ? gid + 8 * hrow : 0);
      qrow[hrow] = reinterpret_cast<const T*>(p.q) + q_offset(p, b, hkv * p.g + rho / p.Lq, rho % p.Lq);
    }
#pragma unroll
    for (int kb = 0; kb < kKB; ++kb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hrow = e & 1;
        const int c = kb * 16 + 2 * tig + 8 * (e >> 1);
        uint32_t v = 0;
        if (kb < nkb && rok[hrow] && c < p.d) v = *reinterpret_cast<const uint32_t*>(qrow[hrow] + c);
        qa[kb][e] = v;
      }
    }
  }

  constexpr int NT = SW ? DV / 16 : DV / 8;  // n-tiles of the output (SW: m-tiles of O^T)
  const int dv = (int)p.dv;
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  int consumed = 0;

  // The partial of key block c from this warp's running (m, l, o) -- or, with a single
  // block, the final output -- and a fresh start for the next block.
  auto flush = [&](int64_t c) {
    float L[2];
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      if constexpr (SW) {
        // (a row's keys are spread over the 8 lanes of one tig)
        L[hrow] = l[hrow] + __shfl_xor_sync(0xffffffffu, l[hrow], 4);
        L[hrow] += __shfl_xor_sync(0xffffffffu, L[hrow], 8);
        L[hrow] += __shfl_xor_sync(0xffffffffu, L[hrow], 16);
      } else {
        L[hrow] = l[hrow] + __shfl_xor_sync(0xffffffffu, l[hrow], 1);
        L[hrow] += __shfl_xor_sync(0xffffffffu, L[hrow], 2);
      }
    }
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      if (!rok[hrow]) continue;
      const int64_t rho = rc * kRowsDec + (SW ? 2 * tig + hrow : gid + 8 * hrow);
      const int64_t ri = rho % p.Lq, hr = hkv * p.g + rho / p.Lq;
      const int64_t row_global = (b * p.Hq + hr) * p.Lq + ri;
      const float M = m[hrow];
      if (p.nblk == 1) {
        const float sk = sink_log2<T>(p, hr);
        const float Mf = fmaxf(M, sk);
        float f = 0.f, Lf = 0.f;
        if (Mf != -INFINITY) {
          const float am = (M == -INFINITY) ? 0.f : ex2(M - Mf);
          Lf = L[hrow] * am + ex2(sk - Mf);
          f = am / Lf;
        }
        T* orow = reinterpret_cast<T*>(p.out) + o_offset(p, b, hr, ri);
        if constexpr (SW) {
          // O^T fragment: value columns 16 j + gid and 16 j + gid + 8 of rows 2 tig, 2 tig + 1
#pragma unroll
          for (int j = 0; j < NT; ++j) {
#pragma unroll
            for (int hv = 0; hv < 2; ++hv) {
              const int cc = j * 16 + gid + 8 * hv;
              if (cc < dv) orow[cc] = from_f32<T>(o[j][2 * hv + hrow] * f);
            }
          }
          if (gid == 0 && p.lse) p.lse[row_global] = (Mf == -INFINITY) ? -INFINITY : (Mf + log2f(Lf)) * kLn2;
        } else {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const int cc = j * 8 + 2 * tig;
            if (cc < dv)
              *reinterpret_cast<uint32_t*>(orow + cc) = MmaOp<T>::pack(o[j][2 * hrow] * f, o[j][2 * hrow + 1] * f);
          }
          if (tig == 0 && p.lse) p.lse[row_global] = (Mf == -INFINITY) ? -INFINITY : (Mf + log2f(Lf)) * kLn2;
        }
      } else {
        float* po = p.part_o + (row_global * p.nblk + c) * p.dv;
        if constexpr (SW) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
#pragma unroll
            for (int hv = 0; hv < 2; ++hv) {
              const int cc = j * 16 + gid + 8 * hv;
              if (cc < dv) po[cc] = o[j][2 * hv + hrow];
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const int cc = j * 8 + 2 * tig;
            if (cc < dv) *reinterpret_cast<float2*>(po + cc) = make_float2(o[j][2 * hrow], o[j][2 * hrow + 1]);
          }
        }
        if (SW ? gid == 0 : tig == 0) {
          p.part_ml[(row_global * p.nblk + c) * 2 + 0] = M;
          p.part_ml[(row_global * p.nblk + c) * 2 + 1] = L[hrow];
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  };

  // the first ST tiles of the run (issued after the setup's global loads, so that the
  // loop's first wait follows the copies closely)
  int issued = n_tiles < ST ? n_tiles : ST;
  for (int i = 0; i < ST; ++i) {
    if (i < issued) issue(i);
    if constexpr (KV == kKvPagedRows) cp_async_commit();  // one group per slot, empty ones included
  }

  bool ok = true;
  // this tile's key block (c_begin + blk_rel) and the block's last key + 1.  The paged
  // forms count them along (a division per tile slowed their streams, 5,043 -> 5,564
  // GB/s); the strided form divides (counting along measured 1.5 % slower there).
  int blk_rel = 0, in_blk = 0;
  int j_end = 0;
  auto block_end = [&](int rel) {
    const int64_t jb_end = u_lo + (c_begin + rel + 1) * p.keys_per_blk;
    return (int)(jb_end < key_end ? jb_end : key_end);
  };
  if (KV != kKvTma && n_tiles > 0) j_end = block_end(0);
  for (int gt = 0; gt < n_tiles; ++gt) {
    const int s = gt % ST;
    if constexpr (KV == kKvPagedRows) cp_async_wait<ST - 1>();
    if (!landed(gt)) {
      if (lane == 0) record_status(p, kStatTimeoutTmaFull);
      ok = false;
      break;
    }
    consumed = gt + 1;
    if constexpr (KV == kKvTma) {
      blk_rel = gt / tpb;
      j_end = block_end(blk_rel);
    }
    const int64_t c = c_begin + blk_rel;  // key block of this tile
    const uint32_t kst = ring + s * stage_bytes, vst = kst + k_bytes;
    if constexpr (SW) {
      // ---- S^T = K Q^T: per 16 keys one m16 (keys) x n8 (query rows) tile; sc[e] holds
      // key gid + 8 (e >> 1), row 2 tig + (e & 1)
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int kb = 0; kb < kKB; ++kb) {
        if (kb < nkb) {
          uint32_t af[4];
          ldsm_x4(sw128(kst + (kb >> 2) * kKT * 128, krow, (kb & 3) * 2 + (lane >> 4)), af[0], af[1], af[2], af[3]);
          MmaOp<T>::run(sc, af, qa[kb][0], qa[kb][1]);
        }
      }
      // ---- mask, online softmax (a row's 16 keys over the 8 lanes of its tig)
      const int jt = (int)(key_begin + (int64_t)gt * kKT);
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hrow = e & 1;
        const int j = jt + gid + 8 * (e >> 1);
        bool vis = rok[hrow] && j < j_end && j >= lo[hrow] && j < hi[hrow];
        if (bool_mask && vis) vis = static_cast<const uint8_t*>(mk[hrow])[j] != 0;
        float v = -INFINITY;
        if (vis) v = add_mask ? fmaf(sc[e], p.scale_log2, to_f32<T>(static_cast<const T*>(mk[hrow])[j]) * kLog2e)
                              : sc[e] * p.scale_log2;
        sc[e] = v;
        mx[hrow] = fmaxf(mx[hrow], v);
      }
      float alpha[2];
#pragma unroll
      for (int hrow = 0; hrow < 2; ++hrow) {
        mx[hrow] = fmaxf(mx[hrow], __shfl_xor_sync(0xffffffffu, mx[hrow], 4));
        mx[hrow] = fmaxf(mx[hrow], __shfl_xor_sync(0xffffffffu, mx[hrow], 8));
        mx[hrow] = fmaxf(mx[hrow], __shfl_xor_sync(0xffffffffu, mx[hrow], 16));
        const float m_new = fmaxf(m[hrow], mx[hrow]);
        alpha[hrow] = 1.f;
        if (m_new > m[hrow] + kRescaleLog2Dec) {
          alpha[hrow] = ex2(m[hrow] - m_new);
          m[hrow] = m_new;
        }
        l[hrow] *= alpha[hrow];
      }
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hrow = e & 1;
        pv[e] = (m[hrow] == -INFINITY) ? 0.f : ex2(sc[e] - m[hrow]);
        l[hrow] += pv[e];
      }
      // P^T as the B operand of O^T += V^T P^T: the 8 x 8 blocks (keys 0-7, keys 8-15) x
      // rows, transposed in registers
      const uint32_t pb0 = movmatrix_t(MmaOp<T>::pack(pv[0], pv[1]));
      const uint32_t pb1 = movmatrix_t(MmaOp<T>::pack(pv[2], pv[3]));
      if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          o[j][0] *= alpha[0];
          o[j][1] *= alpha[1];
          o[j][2] *= alpha[0];
          o[j][3] *= alpha[1];
        }
      }
      // ---- O^T += V^T P^T: per 16 value columns, A = V^T from the V tile by ldmatrix.trans
      const int vrow = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int chunk = 2 * j + ((lane >> 3) & 1);  // 16-byte chunk of dv (8 columns)
        uint32_t af[4];
        ldsm_x4_t(sw128(vst + (chunk >> 3) * kKT * 128, vrow, chunk & 7), af[0], af[1], af[2], af[3]);
        MmaOp<T>::run(o[j], af, pb0, pb1);
      }
    } else {
      // ---- S = Q K^T over the tile's keys (n-tiles of 8 keys)
      constexpr int NS = kKT / 8;  // n-tiles of S
      float sc[NS][4];
  #pragma unroll
      for (int nt = 0; nt < NS; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
  #pragma unroll
      for (int kb = 0; kb < kKB; ++kb) {
        if (kb < nkb) {
          const int chunk = (kb & 3) * 2 + ((lane >> 3) & 1);
  #pragma unroll
          for (int h16 = 0; h16 < kKT / 16; ++h16) {
            uint32_t b0, b1, b2, b3;
            const int krow = h16 * 16 + (lane >> 4) * 8 + (lane & 7);
            ldsm_x4(sw128(kst + (kb >> 2) * kKT * 128, krow, chunk), b0, b1, b2, b3);
            MmaOp<T>::run(sc[2 * h16], qa[kb], b0, b1);
            MmaOp<T>::run(sc[2 * h16 + 1], qa[kb], b2, b3);
          }
        }
      }
      // ---- mask, online softmax (rows gid / gid + 8; keys spread over the lane quad)
      const int jt = (int)(key_begin + (int64_t)gt * kKT);
      float mx[2] = {-INFINITY, -INFINITY};
  #pragma unroll
      for (int nt = 0; nt < NS; ++nt) {
  #pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int hrow = e >> 1;
          const int j = jt + nt * 8 + 2 * tig + (e & 1);
          bool vis = rok[hrow] && j < j_end && j >= lo[hrow] && j < hi[hrow];
          if (bool_mask && vis) vis = static_cast<const uint8_t*>(mk[hrow])[j] != 0;
          float v = -INFINITY;
          if (vis) v = add_mask ? fmaf(sc[nt][e], p.scale_log2, to_f32<T>(static_cast<const T*>(mk[hrow])[j]) * kLog2e)
                                : sc[nt][e] * p.scale_log2;
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
      // P as the A operand of the k16 steps: pa[ks] covers keys 16 ks .. 16 ks + 15
      uint32_t pa[kKT / 16][4];
  #pragma unroll
      for (int hrow = 0; hrow < 2; ++hrow) l[hrow] *= alpha[hrow];
  #pragma unroll
      for (int nt = 0; nt < NS; ++nt) {
  #pragma unroll
        for (int hrow = 0; hrow < 2; ++hrow) {
          const bool none = (m[hrow] == -INFINITY);
          const float p0 = none ? 0.f : ex2(sc[nt][2 * hrow] - m[hrow]);
          const float p1 = none ? 0.f : ex2(sc[nt][2 * hrow + 1] - m[hrow]);
          l[hrow] += p0 + p1;
          pa[nt >> 1][(nt & 1) * 2 + hrow] = MmaOp<T>::pack(p0, p1);
        }
      }
      if (alpha[0] != 1.f || alpha[1] != 1.f) {
  #pragma unroll
        for (int j = 0; j < NT; ++j) {
          o[j][0] *= alpha[0];
          o[j][1] *= alpha[0];
          o[j][2] *= alpha[1];
          o[j][3] *= alpha[1];
        }
      }
      // ---- O += P V: V tile rows = keys, ldmatrix.trans gives the k16 x n8 B fragments
  #pragma unroll
      for (int ks = 0; ks < kKT / 16; ++ks) {
        const int vrow = ks * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
  #pragma unroll
        for (int j2 = 0; j2 < NT / 2; ++j2) {
          const int chunk = 2 * j2 + (lane >> 4);  // 16-byte chunk of dv (8 columns)
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sw128(vst + (chunk >> 3) * kKT * 128, vrow, chunk & 7), b0, b1, b2, b3);
          MmaOp<T>::run(o[2 * j2], pa[ks], b0, b1);
          MmaOp<T>::run(o[2 * j2 + 1], pa[ks], b2, b3);
        }
      }
    }
    // ---- the slot is read: refill it with tile gt + ST (the async proxy's write must
    // follow this warp's reads of the slot)
    __syncwarp();
    if (gt + ST < n_tiles) {
      if (KV != kKvPagedRows && lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(gt + ST);
      issued = gt + ST + 1;
    }
    if constexpr (KV == kKvPagedRows) cp_async_commit();

    // ---- end of a key block: write its partial (or the output when it is the only one)
    if constexpr (KV == kKvTma) {
      if ((gt + 1) % tpb == 0 || gt + 1 == n_tiles) flush(c);
    } else if (++in_blk == tpb || gt + 1 == n_tiles) {
      flush(c);
      in_blk = 0;
      ++blk_rel;
      j_end = block_end(blk_rel);
    }
  }
  if (ok) {
    // key blocks of this run that hold no key of this tile's rows (past a sequence's
    // length, outside a window) still get their (empty) partial, or the final output
    for (int64_t c = c_begin + (n_tiles + tpb - 1) / tpb; c < c_end; ++c) flush(c);
  }
  // a wait that gave up leaves copies in flight: they land before the warp leaves
  if constexpr (KV == kKvPagedRows) {
    cp_async_wait<0>();
  } else if (lane == 0) {
    for (int i = consumed; i < issued; ++i) mbar_wait(full(i % ST), (i / ST) & 1, kDrainLimitDec, nullptr);
  }
  __syncwarp();
}

template <typename T, int DMAX, int DV, int KV, bool SW>
cudaError_t launch_dec_t(const DecArgs& a, int64_t grid, cudaStream_t st) {
  using Sh = DecShape<DMAX, DV>;
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = set_max_dynamic_smem_once(configured, (const void*)sdpa_decode_mma<T, DMAX, DV, KV, SW>, Sh::kSmem);
  if (e != cudaSuccess) return e;
  if (a.wpc < 1 || a.wpc > Sh::WPC) return cudaErrorInvalidValue;
  constexpr int ST = Sh::ST;
  const int smem = a.wpc * ST * Sh::kStageBytes + 1024 + a.wpc * ST * 8 + 64;  // (Sh::kSmem at WPC warps)
  return launch_dependent(sdpa_decode_mma<T, DMAX, DV, KV, SW>, dim3((unsigned)grid), dim3(a.wpc * 32), (size_t)smem,
                          st, a);
}

// (d, dv) buckets with a kernel: the smallest bucket covering the head is used; the
// TMA tiles zero-fill the columns between the head size and the bucket.
constexpr int kDecBuckets[][2] = {{64, 64}, {128, 64}, {128, 128}, {192, 128}, {192, 192}, {256, 256}};

inline int dec_bucket(int64_t d, int64_t dv) {
  for (int i = 0; i < 6; ++i)
    if (d <= kDecBuckets[i][0] && dv <= kDecBuckets[i][1]) return i;
  return -1;
}

struct DecInfo {
  int wpc, ctas_per_sm, smem, kt;
};
template <int DMAX, int DV>
constexpr DecInfo dec_info_t() {
  return {DecShape<DMAX, DV>::WPC, DecShape<DMAX, DV>::kCtasPerSm, DecShape<DMAX, DV>::kSmem, DecShape<DMAX, DV>::KT};
}
inline DecInfo dec_info(int64_t d, int64_t dv) {
  switch (dec_bucket(d, dv)) {
    case 0: return dec_info_t<64, 64>();
    case 1: return dec_info_t<128, 64>();
    case 2: return dec_info_t<128, 128>();
    case 3: return dec_info_t<192, 128>();
    case 4: return dec_info_t<192, 192>();
    case 5: return dec_info_t<256, 256>();
    default: return {0, 0, 0, 0};
  }
}

template <typename T, int KV>
cudaError_t launch_dec_bucket(const DecArgs& a, int64_t grid, cudaStream_t st) {
  const bool sw = a.p.G <= 8;
  switch (dec_bucket(a.p.d, a.p.dv)) {
    // (up to 8 query rows per KV head: the transposed products)
    case 0: return sw ? launch_dec_t<T, 64, 64, KV, true>(a, grid, st) : launch_dec_t<T, 64, 64, KV, false>(a, grid, st);
    case 1: return sw ? launch_dec_t<T, 128, 64, KV, true>(a, grid, st) : launch_dec_t<T, 128, 64, KV, false>(a, grid, st);
    case 2:
      return sw ? launch_dec_t<T, 128, 128, KV, true>(a, grid, st) : launch_dec_t<T, 128, 128, KV, false>(a, grid, st);
    case 3: return launch_dec_t<T, 192, 128, KV, false>(a, grid, st);
    case 4: return launch_dec_t<T, 192, 192, KV, false>(a, grid, st);
    case 5: return launch_dec_t<T, 256, 256, KV, false>(a, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

// Launches pass 1 with K/V read in mode KV (the tensor maps already in `a`).
template <int KV>
cudaError_t launch_dec_kv(int dtype, DecArgs& a, cudaStream_t st) {
  const Params& p = a.p;
  const int kt = dec_info(p.d, p.dv).kt;
  a.n_rc = (int)((p.G + kRowsDec - 1) / kRowsDec);
  a.dpanels = (int)((p.d + 63) / 64);
  a.dvpanels = (int)((p.dv + 63) / 64);
  // every warp walks whole key blocks: a block size that is not a whole number of tiles,
  // or a run count outside [1, blocks], is a planner error
  if (!kt || p.spans < 1 || p.spans > p.nblk || p.keys_per_blk % kt != 0) return cudaErrorInvalidValue;
  const int64_t warp_units = p.B * p.Hkv * a.n_rc * p.spans;
  a.wpc = decode_mma_cta_warps(warp_units, p.d, p.dv);
  const int64_t grid = (warp_units + a.wpc - 1) / a.wpc;
  return dtype == 1 ? launch_dec_bucket<__half, KV>(a, grid, st) : launch_dec_bucket<__nv_bfloat16, KV>(a, grid, st);
}


}  // namespace dec
}  // namespace nvsdpa

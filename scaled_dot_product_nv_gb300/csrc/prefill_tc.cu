// Prefill attention on the 5th-generation tensor cores (tcgen05) for f16/bf16.
//
// The algorithm is the tiled online softmax of "lattice-inference 0.4.0
// src/attention/flash.rs" (run_tiled_attention_head): per key tile, S = Q K^T, the row
// maximum, rescale of the running sum and output, P V accumulated, one division at the
// end; masked keys at minus infinity and all-masked rows giving zeros.  The blocking,
// the memory movement and the exponent bookkeeping are this kernel's own:
//
// * One CTA owns NQ x 128 query rows of one KV head (rows of the g query heads sharing
//   it, head-major -- contiguous in memory) and walks their visible key tiles of BN keys.
//   With two Q tiles these are, where the shape allows, the same 128 positions of two
//   query heads: both tiles then see the same key tiles, and under the causal mask
//   neither waits out the other's extra diagonal tile alone.
// * Warp 0 (one lane) streams the Q tile(s) once and K/V tiles through a 2-stage ring
//   with 3-D TMA (128-byte swizzle, zero fill out of range); completion on mbarriers.
// * Warp 1 allocates the 512 TMEM columns; one lane issues every tcgen05.mma:
//     S = Q K_t^T      (A, B from shared memory, f32 accumulator in TMEM)
//     O += P V_t       (A = P from TMEM, B = V from shared memory, MN-major)
//   and signals completions with tcgen05.commit.
// * NQ softmax warpgroups (4 warps, one query row per thread = one TMEM lane) read S,
//   mask it, keep the running max in log2 units, write P = 2^(s - m) as 16-bit pairs
//   over the TMEM columns of S, and rescale O only when the max grew by more than 2^8
//   (otherwise the stale max stays: exact after the final division, weights <= 2^8).
//   The epilogue folds in the sink logit, divides once, rounds once to the output type
//   and writes the log-sum-exp.
//   - NQ = 1 (any head up to 256): S is double-buffered, so S_{t+1} is computed while
//     the warpgroup works on S_t.
//   - NQ = 2 (d, dv <= 128): two Q tiles share each K/V tile; the MMA issue order
//     S0 S1 | P0V, S0' | P1V, S1' | ... lets one warpgroup's softmax run while the
//     tensor pipe works for the other (ping-pong), with two warps per scheduler.
// * Causal: key tiles wholly above the (bottom-right aligned) diagonal are never loaded,
//   and a warp takes the unmasked fast path on every tile it sees completely.  Boolean
//   masks arrive as a bit-packed copy made by sdpa_pack_mask_bits, which this kernel
//   overlaps as its programmatic dependent.
// * Every mbarrier wait is bounded; a wait that runs out records a status bit, raises
//   a shared abort flag that the other roles also watch, and the CTA drains its
//   in-flight copies and MMAs before freeing TMEM and exiting.
#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace nvsdpa {
namespace {

using namespace sm100;

constexpr int kBM = 128;
constexpr int kStages = 3;  // the deepest K / V ring (barrier slots)
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint64_t kDrainLimit = 1ull << 18;  // polls of <= ~10 us each
constexpr int64_t kTcMaxSmem = 227 * 1024;  // opt-in dynamic shared memory per CTA

struct TcArgs {
  CUtensorMap tmq, tmk, tmv;  // 64-byte aligned by type
  CUtensorMap tmo;            // the output, for TMA stores of whole tiles (when tma_out)
  Params p;
  const uint32_t* mask_bits;  // [Lq][mask_words], bit j%32 of word j/32 = key j visible
  int64_t mask_words;
  int n_rt;          // CTA row blocks (NQ x 128 rows) per (b, kv head)
  int dpanels;       // 64-element panels of d
  int dvpanels;      // 64-element panels of dv
  int ksteps_qk;     // ceil(d / 16)
  int n_pv;          // dv rounded up to 16 (MMA N of P V)
  int itile_order;   // Lq % (NQ x 128) == 0: launch the late (heavier, causal) blocks first
  int head_local;    // each Q tile is 128 positions of one query head (NQ = 2: the same
                     // positions of two heads, equal key extents), late positions first
  int qo5;           // Q and out are read / written through 5-D [B][Hkv][g][Lq][D] maps
                     // (strided layouts); otherwise 3-D [B*Hkv][G][D] maps of packed rows
  int n_it;          // head_local: 128-position blocks per head
  int tma_out;       // the output tile fits the Q tile's shared memory: store it by TMA
  int64_t amask_total;  // elements of the additive mask (loads never pass its end)
  int split;         // NQ = 1, packed rows: CTA x is key block x % nblk of its row block, and
                     // (nblk > 1) its rows' partials go to part_o / part_ml for the merge
  int blk_tiles;     // split: key tiles per block (keys_per_blk / BN)
  int tmem_cols;     // TMEM columns allocated: 512, or 256 where two CTAs share the SM
  int q_rows;        // rows of a Q tile's buffer: 128, or 64 (split-KV, at most 64 rows; the
                     // MMA's rows past 64 read the next panel's, whose scores are masked)
  int unpadded;      // the dynamic shared memory was requested without alignment slack:
                     // its start must already be 1024-byte aligned (checked)
};

// barrier slots
// (NQ = 2: K and V of a stage land on kv_full and are released together; NQ = 1: K on
// kv_full / kv_empty, V on v_full / v_empty, each released as soon as its last reader
// is done)
enum { kBarQ = 0, kBarKvFull = 1, kBarKvEmpty = 1 + kStages, kBarSFull = 1 + 2 * kStages,
       kBarPFull = 3 + 2 * kStages, kBarPvDone = 5 + 2 * kStages, kBarDrain = 7 + 2 * kStages,
       kBarVFull = 8 + 2 * kStages, kBarVEmpty = 8 + 3 * kStages, kBarMFull = 8 + 4 * kStages,
       kNumBars = 10 + 4 * kStages };

// Additive masks: each row's values of kAmTiles key tiles at a time are staged in shared
// memory by one bulk copy per row, issued by the row's own softmax thread two chunks ahead
// (16-byte aligned: from the 8-element boundary at or below the first column, 8 elements
// more than the tiles span), in two buffers.
constexpr int kAmTiles = 2;
template <int BN>
__host__ __device__ constexpr int am_row_bytes() { return (kAmTiles * BN + 8) * 2; }
template <int BN>
__host__ __device__ constexpr int am_bytes() { return 2 * 128 * am_row_bytes<BN>(); }

__device__ __forceinline__ void fail(const Params& p, volatile int* abort, uint32_t bit) {
  *abort = 1;
  record_status(p, bit);
}

template <typename T> struct TypeCode;
template <> struct TypeCode<__half> { static constexpr uint32_t v = 0; };
template <> struct TypeCode<__nv_bfloat16> { static constexpr uint32_t v = 1; };

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) { return pack_f16(lo, hi); }
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  return pack_bf16(lo, hi);
}

// The positions [imin, imax] of a Q tile's valid rows, or false if it has none.  Packed:
// rows [r0, r0 + 128) of the KV head's G rows (head-major; a tile spanning two heads
// covers every position).  Head-local: positions [i0, i0 + 128) of one query head.
__device__ __forceinline__ bool tile_positions(const TcArgs& a, int r0, int i0, int64_t& imin,
                                               int64_t& imax) {
  const Params& p = a.p;
  if (a.head_local) {
    if (i0 >= p.Lq) return false;
    imin = i0;
    imax = (i0 + kBM < p.Lq ? i0 + kBM : p.Lq) - 1;
    return true;
  }
  if (r0 >= p.G) return false;
  const int64_t r1 = (r0 + kBM < p.G ? r0 + kBM : p.G) - 1;
  const bool one = r0 / p.Lq == r1 / p.Lq;
  imin = one ? r0 % p.Lq : 0;
  imax = one ? r1 % p.Lq : p.Lq - 1;
  return true;
}

// Key tiles of BN keys [first, end) that a Q tile needs: the causal bound of its last
// position and the window band of its first (end = first = 0 when it needs none).
template <int BN>
__device__ __forceinline__ void tile_key_range(const TcArgs& a, int r0, int i0, int& first, int& end) {
  const Params& p = a.p;
  int64_t imin, imax;
  first = end = 0;
  if (!tile_positions(a, r0, i0, imin, imax)) return;
  const int64_t hi = row_key_hi(p, imax + p.Lk - p.Lq, p.Lk);
  const int64_t lo = row_key_lo(p, imin + p.Lk - p.Lq);
  if (hi <= lo) return;
  first = (int)(lo / BN);
  end = (int)((hi + BN - 1) / BN);
}

// The 32-bit visibility word of columns [c0, c0 + 32) of a row that sees columns
// [lo, hi) of the tile.
__device__ __forceinline__ uint32_t col_bound(int c0, int lo, int hi) {
  const int a = lo - c0, b = hi - c0;
  const uint32_t below_hi = b >= 32 ? 0xffffffffu : (b <= 0 ? 0u : (1u << b) - 1u);
  const uint32_t below_lo = a >= 32 ? 0xffffffffu : (a <= 0 ? 0u : (1u << a) - 1u);
  return below_hi & ~below_lo;
}

// Mask handling of a prefill kernel instantiation: the key bounds alone (none, causal,
// window), a bit-packed boolean mask, or an additive mask.
enum { kMmBounds = 0, kMmBits = 1, kMmAdd = 2 };

// Words of additive-mask values a softmax step holds: BN / 2 pairs (one word unused
// otherwise).
template <int BN, int MM>
__host__ __device__ constexpr int av_words() { return MM == kMmAdd ? BN / 2 : 1; }

// One query row's softmax step on its t-th key tile, key tile kt of the sequence.  tS /
// tO: TMEM addresses (lane base included) of this tile's S columns and of O; the row
// sees keys [first_key, last_key]; mrow: its mask row (MM = kMmBits: bit-packed words,
// kMmAdd: unused; the tile's additive values are in av), unused otherwise.  PF: the tile's
// words were loaded ahead by the caller into mw.  wait_pv: O may still be receiving
// P_{t-1} V_{t-1} (the one-tile variant), so a rescale waits for it on pv_bar; last: the
// walk's last tile, which waits in any case.  Returns false if a wait gave up.
template <typename T, int BN, int NQ, int MM, bool PF>
__device__ __forceinline__ bool softmax_tile(const TcArgs& a, int t, int kt, uint32_t tS, uint32_t tO,
                                             bool row_ok, int first_key, int last_key, const void* mrow_any,
                                             const uint32_t (&mw)[BN / 32], const uint32_t (&av)[av_words<BN, MM>()],
                                             float& m_run, float& l_run, uint32_t pv_bar, bool wait_pv, bool last,
                                             uint64_t limit, volatile int* abort) {
  const Params& p = a.p;
  const uint32_t* mrow = static_cast<const uint32_t*>(mrow_any);
  uint32_t sr[BN];
  if constexpr (BN == 128) tmem_ld128_sync(tS, sr);
  else tmem_ld64_sync(tS, sr);
  const int j0 = kt * BN;
  // columns [vis_lo, vis_hi) pass the causal / key-count bound and the window band
  const int vh = last_key - j0 + 1, vl = first_key - j0;
  const int vis_hi = vh < 0 ? 0 : (vh > BN ? BN : vh);
  const int vis_lo = vl < 0 ? 0 : (vl > BN ? BN : vl);
  const bool masked = !row_ok || MM != kMmBounds || vis_hi < BN || vis_lo > 0;
  // warp-uniform fast path: nothing masked and scale >= 0, so the maximum of the raw
  // scores gives the scaled maximum and 2^(s*c - m) is one FFMA and one MUFU op
  const bool fast = !__any_sync(0xffffffffu, masked) && p.scale_log2 >= 0.f;
  float alpha = 1.f;
  bool need;
  if (fast) {
    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int e = 0; e < BN; e += 8) {
      m4[0] = fmax3(m4[0], __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
      m4[1] = fmax3(m4[1], __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
      m4[2] = fmax3(m4[2], __uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5]));
      m4[3] = fmax3(m4[3], __uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7]));
    }
    const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
    const float m_new = fmaxf(m_run, mt);
    need = m_new > m_run + kRescaleLog2;
    if (need) {
      alpha = ex2(m_run - m_new);
      m_run = m_new;
    }
    // P = 2^(s*c - m): one two-wide FFMA per pair of scores, the sum two-wide as well
    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(-m_run, -m_run);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int c2i = 0; c2i < BN / 64; ++c2i) {
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int idx = c2i * 64 + 2 * e;
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[idx]), __uint_as_float(sr[idx + 1])), c2, nm2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        acc[e & 3] = f2_add(acc[e & 3], f2_pack(p0, p1));
        pk[e] = pack2<T>(p0, p1);
      }
      tmem_st32(tS + c2i * 32, pk);
    }
    float a0, a1, b0, b1;
    f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
    f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
    l_run = l_run * alpha + ((a0 + a1) + (b0 + b1));
  } else {
    // RAW (scale > 0, no additive term): the maximum is taken over the raw visible scores
    // and scaled once, and P = 2^(s*c - m) is one FFMA as on the fast path (a hidden score
    // is -inf, and -inf * c stays -inf); otherwise the scores are scaled (and the additive
    // term added) first.
    auto masked_tile = [&](auto raw_tag) {
      constexpr bool RAW = decltype(raw_tag)::value;
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t bits = 0xffffffffu;
        if constexpr (MM == kMmBits) bits = PF ? mw[c] : (row_ok ? __ldg(mrow + j0 / 32 + c) : 0u);
        // the visible columns of this word: mask bits, causal / key-count bound, window
        // band, the row
        const uint32_t vb = row_ok ? (bits & col_bound(c * 32, vis_lo, vis_hi)) : 0u;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = c * 32 + e;
          float x0 = __uint_as_float(sr[col]), x1 = __uint_as_float(sr[col + 1]);
          if constexpr (!RAW) {
            f2_unpack(f2_mul(f2_pack(x0, x1), c2), x0, x1);
            if constexpr (MM == kMmAdd) {
              // the additive term, in log2 units (masked columns are replaced below)
              const uint32_t wv = av[col >> 1];
              x0 = fmaf(to_f32<T>(*reinterpret_cast<const T*>(&wv)), kLog2e, x0);
              x1 = fmaf(to_f32<T>(*(reinterpret_cast<const T*>(&wv) + 1)), kLog2e, x1);
            }
          }
          x0 = (vb & (1u << e)) ? x0 : -INFINITY;
          x1 = (vb & (2u << e)) ? x1 : -INFINITY;
          sr[col] = __float_as_uint(x0);
          sr[col + 1] = __float_as_uint(x1);
          m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], x0, x1);
        }
      }
      float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      if constexpr (RAW) mt *= p.scale_log2;
      const float m_new = fmaxf(m_run, mt);
      need = m_new > m_run + kRescaleLog2;
      if (need) {
        alpha = ex2(m_run - m_new);
        m_run = m_new;
      }
      // P = 2^(s - m); while no key of the row has been visible every s is -inf and
      // 2^(s + 0) = 0
      const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
      const uint64_t nm2 = f2_pack(neg_m, neg_m);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int c2i = 0; c2i < BN / 64; ++c2i) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int idx = c2i * 64 + 2 * e;
          float y0, y1;
          const uint64_t sv = f2_pack(__uint_as_float(sr[idx]), __uint_as_float(sr[idx + 1]));
          if constexpr (RAW) f2_unpack(f2_fma(sv, c2, nm2), y0, y1);
          else f2_unpack(f2_add(sv, nm2), y0, y1);
          const float p0 = ex2(y0), p1 = ex2(y1);
          acc[e & 3] = f2_add(acc[e & 3], f2_pack(p0, p1));
          pk[e] = pack2<T>(p0, p1);
        }
        tmem_st32(tS + c2i * 32, pk);
      }
      float a0, a1, b0, b1;
      f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
      f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
      l_run = l_run * alpha + ((a0 + a1) + (b0 + b1));
    };
    // (the two-tile variant, at its register limit, keeps the one general form)
    if (NQ == 1 && MM != kMmAdd && p.scale_log2 > 0.f) masked_tile(std::true_type{});
    else masked_tile(std::false_type{});
  }
  tmem_st_wait();
  const bool rescale = t > 0 && __any_sync(0xffffffffu, need);
  if (t > 0 && wait_pv && (rescale || last)) {
    // O is rescaled only once P_{t-1} V_{t-1} has landed in it.  The wait tests a phase
    // parity, which is exact while the newest completed phase of pv_done is t-2 or t-1:
    // it is at most t-1 (P_t is not released yet), and at least t-2 because S_t, whose
    // completion this thread has seen, was issued after P_{t-2} V_{t-2} and its commit
    // tracks every earlier MMA -- so tiles that need no rescale skip the wait.  The last
    // tile waits all the same: the epilogue's wait for the last P V is then exact too.
    if (!__all_sync(0xffffffffu, mbar_wait(pv_bar, (t - 1) & 1, limit, abort))) return false;
    tc_fence_after();
  }
  if (rescale) {
    for (int c = 0; c < (a.n_pv + 31) / 32; ++c) {
      uint32_t o[32];
      tmem_ld32_sync(tO + c * 32, o);
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
      tmem_st32(tO + c * 32, o);
    }
    tmem_st_wait();
  }
  return true;
}

// Final output of one query row: sink folded in, one division, one rounding; lse.
template <typename T>
__device__ __forceinline__ void epilogue_row(const Params& p, uint32_t tO, bool have_o, bool row_ok,
                                             int64_t b, int64_t h, int64_t i, float m_run, float l_run) {
  const float sk = sink_log2<T>(p, h);
  const float M = fmaxf(m_run, sk);
  float f = 0.f, L = 0.f;
  if (M != -INFINITY) {
    const float am = ex2(m_run - M);
    L = l_run * am + ex2(sk - M);
    f = am / L;
  }
  T* orow = reinterpret_cast<T*>(p.out) + o_offset(p, b, h, i);
  const int64_t lse_row = (b * p.Hq + h) * p.Lq + i;
  const int dv = (int)p.dv;
  // 128 columns of O per TMEM load (the O region is 128-column aligned and inside the
  // allocation for every head this kernel takes)
  for (int c0 = 0; c0 < dv; c0 += 128) {
    uint32_t o[128];
    if (have_o) {
      tmem_ld128_sync(tO + c0, o);
    } else {
#pragma unroll
      for (int e = 0; e < 128; ++e) o[e] = 0u;
    }
    if (row_ok) {
#pragma unroll
      for (int e8 = 0; e8 < 16; ++e8) {
        const int col = c0 + e8 * 8;
        if (col < dv) {
          uint4 v;
          v.x = pack2<T>(__uint_as_float(o[e8 * 8 + 0]) * f, __uint_as_float(o[e8 * 8 + 1]) * f);
          v.y = pack2<T>(__uint_as_float(o[e8 * 8 + 2]) * f, __uint_as_float(o[e8 * 8 + 3]) * f);
          v.z = pack2<T>(__uint_as_float(o[e8 * 8 + 4]) * f, __uint_as_float(o[e8 * 8 + 5]) * f);
          v.w = pack2<T>(__uint_as_float(o[e8 * 8 + 6]) * f, __uint_as_float(o[e8 * 8 + 7]) * f);
          *reinterpret_cast<uint4*>(orow + col) = v;
        }
      }
    }
  }
  if (row_ok && p.lse) p.lse[lse_row] = (M == -INFINITY) ? -INFINITY : (M + log2f(L)) * kLn2;
}

// The same, for one TMA store of the whole tile (the two-tile variant): the row is written (scaled and rounded)
// into `stage`, the tile's shared-memory image in the 128-byte-swizzled layout of the
// loads (64-column panels of 128 rows x 128 B, 16-byte chunk c of row r at
// (c ^ (r mod 8)) * 16); the log-sum-exp is written directly.
template <typename T>
__device__ __forceinline__ void epilogue_row_smem(const Params& p, uint32_t tO, bool have_o, bool row_ok,
                                                  int64_t b, int64_t h, int64_t i, float m_run, float l_run,
                                                  uint8_t* stage, int r) {
  const float sk = sink_log2<T>(p, h);
  const float M = fmaxf(m_run, sk);
  float f = 0.f, L = 0.f;
  if (M != -INFINITY) {
    const float am = ex2(m_run - M);
    L = l_run * am + ex2(sk - M);
    f = am / L;
  }
  const int dv = (int)p.dv;
  for (int c0 = 0; c0 < dv; c0 += 128) {
    uint32_t o[128];
    if (have_o) {
      tmem_ld128_sync(tO + c0, o);
    } else {
#pragma unroll
      for (int e = 0; e < 128; ++e) o[e] = 0u;
    }
#pragma unroll
    for (int e8 = 0; e8 < 16; ++e8) {
      const int col = c0 + e8 * 8;
      if (col < dv) {
        uint4 v;
        v.x = pack2<T>(__uint_as_float(o[e8 * 8 + 0]) * f, __uint_as_float(o[e8 * 8 + 1]) * f);
        v.y = pack2<T>(__uint_as_float(o[e8 * 8 + 2]) * f, __uint_as_float(o[e8 * 8 + 3]) * f);
        v.z = pack2<T>(__uint_as_float(o[e8 * 8 + 4]) * f, __uint_as_float(o[e8 * 8 + 5]) * f);
        v.w = pack2<T>(__uint_as_float(o[e8 * 8 + 6]) * f, __uint_as_float(o[e8 * 8 + 7]) * f);
        const int pn = col >> 6, c = (col >> 3) & 7;
        *reinterpret_cast<uint4*>(stage + pn * (kBM * 128) + r * 128 + ((c ^ (r & 7)) << 4)) = v;
      }
    }
  }
  if (row_ok && p.lse) p.lse[(b * p.Hq + h) * p.Lq + i] = (M == -INFINITY) ? -INFINITY : (M + log2f(L)) * kLn2;
}

// The same, for a TMA store of the tile panel by panel: epilogue_factor gives the row's
// output factor (sink folded in, one division) and writes its log-sum-exp;
// epilogue_panel_smem writes the row's 64 columns of panel pn (scaled, rounded once) into
// `stage`, the tile's shared-memory image in the 128-byte-swizzled layout of the loads
// (64-column panels of 128 rows x 128 B, 16-byte chunk c of row r at (c ^ (r mod 8)) * 16).
template <typename T>
__device__ __forceinline__ float epilogue_factor(const Params& p, bool row_ok, int64_t b, int64_t h, int64_t i,
                                                 float m_run, float l_run) {
  const float sk = sink_log2<T>(p, h);
  const float M = fmaxf(m_run, sk);
  float f = 0.f, L = 0.f;
  if (M != -INFINITY) {
    const float am = ex2(m_run - M);
    L = l_run * am + ex2(sk - M);
    f = am / L;
  }
  if (row_ok && p.lse) p.lse[(b * p.Hq + h) * p.Lq + i] = (M == -INFINITY) ? -INFINITY : (M + log2f(L)) * kLn2;
  return f;
}

template <typename T>
__device__ __forceinline__ void epilogue_panel_smem(const Params& p, uint32_t tO, bool have_o, float f, uint8_t* stage,
                                                    int r, int pn) {
  const int dv = (int)p.dv, c0 = pn * 64;
  uint32_t o[64];
  if (have_o) {
    tmem_ld64_sync(tO + c0, o);
  } else {
#pragma unroll
    for (int e = 0; e < 64; ++e) o[e] = 0u;
  }
#pragma unroll
  for (int e8 = 0; e8 < 8; ++e8) {
    if (c0 + e8 * 8 < dv) {
      uint4 v;
      v.x = pack2<T>(__uint_as_float(o[e8 * 8 + 0]) * f, __uint_as_float(o[e8 * 8 + 1]) * f);
      v.y = pack2<T>(__uint_as_float(o[e8 * 8 + 2]) * f, __uint_as_float(o[e8 * 8 + 3]) * f);
      v.z = pack2<T>(__uint_as_float(o[e8 * 8 + 4]) * f, __uint_as_float(o[e8 * 8 + 5]) * f);
      v.w = pack2<T>(__uint_as_float(o[e8 * 8 + 6]) * f, __uint_as_float(o[e8 * 8 + 7]) * f);
      *reinterpret_cast<uint4*>(stage + pn * (kBM * 128) + r * 128 + ((e8 ^ (r & 7)) << 4)) = v;
    }
  }
}

// Split-KV: the partial of key block c for one query row -- its running maximum m (log2
// units), the sum l of 2^(s - m) and the unnormalised O, all relative to the same m
// (zeros and m = -inf when the block holds no key the row sees) -- for the merge pass.
__device__ __forceinline__ void partial_row(const Params& p, uint32_t tO, bool have_o, bool row_ok, int64_t b,
                                            int64_t h, int64_t i, int64_t c, float m_run, float l_run) {
  const int64_t row_global = (b * p.Hq + h) * p.Lq + i;
  const int64_t slot = row_global * p.nblk + c;
  float* po = p.part_o + slot * p.dv;
  const int dv = (int)p.dv;
  for (int c0 = 0; c0 < dv; c0 += 32) {
    uint32_t o[32];
    if (have_o) {
      tmem_ld32_sync(tO + c0, o);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0u;
    }
    if (row_ok) {
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const int col = c0 + e4 * 4;
        if (col < dv)
          *reinterpret_cast<uint4*>(po + col) = make_uint4(o[e4 * 4], o[e4 * 4 + 1], o[e4 * 4 + 2], o[e4 * 4 + 3]);
      }
    }
  }
  if (row_ok) {
    p.part_ml[slot * 2 + 0] = have_o ? m_run : -INFINITY;
    p.part_ml[slot * 2 + 1] = have_o ? l_run : 0.f;
  }
}

template <int NQ>
constexpr int tc_threads() { return (2 + 4 * NQ) * 32; }

// CTAs per SM a variant is compiled for: the 64-key one-tile variant with the key bounds
// alone serves the split-KV decode of heads up to 128, two CTAs per SM (each with 256
// TMEM columns and under half the shared memory); every other variant owns its SM.
template <int BN, int NQ, int MM>
constexpr int tc_ctas_per_sm() { return (BN == 64 && NQ == 1 && MM == kMmBounds) ? 2 : 1; }

template <typename T, int BN, int NQ, int MM, int STG>
__global__ void __launch_bounds__(tc_threads<NQ>(), (tc_ctas_per_sm<BN, NQ, MM>())) sdpa_prefill_tc(const __grid_constant__ TcArgs a) {
  static_assert(NQ == 1 || NQ == 2, "one or two Q tiles per CTA");
  static_assert(NQ == 1 || BN == 128, "the two-tile variant uses 128-key tiles");
  static_assert(STG >= 1 && STG <= kStages && (NQ == 1 || STG == 2), "ring depth");
  static_assert(STG <= 2 || (NQ == 1 && BN == 64 && MM == kMmBounds), "three stages: the two-CTA split-KV form");
  constexpr int kMaxKsteps = (NQ == 2) ? 8 : 16;  // d <= 128 for two tiles, <= 256 otherwise
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (a.unpadded && base != smem_raw) {
    // (the request had no room to align: the CTA does nothing and the call reports it)
    if (threadIdx.x == 0) record_status(a.p, kStatBadConfig);
    return;
  }
  const Params& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t q_bytes = a.dpanels * a.q_rows * 128;  // one Q tile's buffer
  const uint32_t k_bytes = a.dpanels * BN * 128;
  const uint32_t v_bytes = a.dvpanels * BN * 128;
  const uint32_t sQ = smem_addr(base);
  const uint32_t sK = sQ + NQ * q_bytes;
  const uint32_t sV = sK + STG * k_bytes;
  // (additive masks: the two staging buffers of the rows' mask values follow the rings)
  const uint32_t sM = sV + STG * v_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + NQ * q_bytes + STG * (k_bytes + v_bytes) +
                                               (MM == kMmAdd ? am_bytes<BN>() : 0));
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_holder + 1);
  auto bar = [&](int i) { return smem_addr(bars + i); };

  // ---- which rows and keys this CTA owns: (b, kv head) and, per Q tile, either the first
  // of its 128 packed rows (among the G rows of that KV head) or its query head and first
  // position (head-local tiles)
  // (32-bit: the planner sends no call whose rows, keys or CTAs do not fit)
  const int BH = (int)(p.B * p.Hkv);
  int bh, row0[NQ], i0[NQ], hhq[NQ];
  int blk = 0;  // split: this CTA's key block
  if (NQ == 1 && a.split) {
    // split-KV (decode-sized row groups): key block, then row block, then (b, kv head)
    int x = (int)blockIdx.x;
    blk = x % (int)p.nblk; x /= (int)p.nblk;
    row0[0] = (x % a.n_rt) * kBM;
    bh = x / a.n_rt;
    hhq[0] = 0;
    i0[0] = 0;
  } else if (a.head_local) {
    const int per = (int)(p.g / NQ);  // Q-tile groups (heads or head pairs) per KV head
    int x = (int)blockIdx.x;
    const int pr = x % per; x /= per;
    bh = x % BH;
    const int it = a.n_it - 1 - x / BH;  // late (heavier, causal) positions first
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      hhq[q] = pr * NQ + q;
      i0[q] = it * kBM;
      row0[q] = hhq[q] * (int)p.Lq + i0[q];
    }
  } else {
    int rb;  // row block of NQ x 128 consecutive rows
    if (a.itile_order) {
      const int ipt = (int)(p.Lq / (kBM * NQ));  // row blocks per head
      int x = (int)blockIdx.x;
      const int hh = x % (int)p.g; x /= (int)p.g;
      bh = x % BH;
      const int it = ipt - 1 - x / BH;
      rb = hh * ipt + it;
    } else {
      rb = (int)blockIdx.x % a.n_rt;
      bh = (int)blockIdx.x / a.n_rt;
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      row0[q] = (rb * NQ + q) * kBM;
      hhq[q] = 0;
      i0[q] = 0;
    }
  }
  const int hkv = bh % (int)p.Hkv, bb = bh / (int)p.Hkv;
  // key tiles: the CTA walks tiles kt0 + t, t < n_max; Q tile q uses t < n_q[q] (its tiles
  // before kt0 + n_q[q]; a tile of the walk wholly outside a row's band is masked for it)
  int first_q[NQ], end_q[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) tile_key_range<BN>(a, row0[q], i0[q], first_q[q], end_q[q]);
  if (NQ == 1 && a.split) {
    // the key tiles of block blk, cut from key 0 (whatever the rows' bounds)
    const int b0 = blk * a.blk_tiles, b1 = b0 + a.blk_tiles;
    first_q[0] = first_q[0] > b0 ? first_q[0] : b0;
    end_q[0] = end_q[0] < b1 ? end_q[0] : b1;
  }
  int kt0 = 0x7fffffff;
#pragma unroll
  for (int q = 0; q < NQ; ++q)
    if (end_q[q] > first_q[q] && first_q[q] < kt0) kt0 = first_q[q];
  if (kt0 == 0x7fffffff) kt0 = 0;
  int n_q[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) n_q[q] = end_q[q] > first_q[q] ? end_q[q] - kt0 : 0;
  int n_max = 0;
#pragma unroll
  for (int q = 0; q < NQ; ++q) n_max = n_q[q] > n_max ? n_q[q] : n_max;

  // ---- set-up: barriers, TMEM
  // Launched as the programmatic dependent of the stream's previous kernel: nothing
  // global is read or written, and no TMEM is taken, before that kernel has finished
  // (an early CTA holding TMEM could starve one of the previous grid's on the same SM).
  // With a boolean mask the previous kernel is the mask packing, which itself waited
  // for everything before it: the copies of Q, K and V may start at once, and the
  // softmax warps wait for the bits alone.
  if constexpr (MM != kMmBits) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < STG; ++s) {
      mbar_init(bar(kBarKvFull + s), 1);
      mbar_init(bar(kBarKvEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarSFull + b), 1);
      mbar_init(bar(kBarPFull + b), 128);
      mbar_init(bar(kBarPvDone + b), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    for (int b = 0; b < 2; ++b) mbar_init(bar(kBarMFull + b), 128);  // (one arrival per softmax thread)
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_holder), (uint32_t)a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The next kernel of the stream (the merge pass, or the next call) may now place its
  // CTAs as SMs free up; each waits there for this grid to finish.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
  const uint64_t limit = p.wait_limit;
  // TMEM columns: S slot b at b*BN (NQ = 1: the two buffers; NQ = 2: one per Q tile);
  // O of Q tile q at 2*BN + q*128.
  auto tS_col = [&](int slot) { return (uint32_t)(slot * BN); };
  auto tO_col = [&](int q) { return (uint32_t)(2 * BN + q * 128); };

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0 && n_max > 0) {
      tma_prefetch_desc(&a.tmq);
      tma_prefetch_desc(&a.tmk);
      tma_prefetch_desc(&a.tmv);
      // Only Q tiles that see a key are loaded: the epilogue of a tile that sees none
      // stages its zeros in that tile's buffer, which no copy may still be filling.
      uint32_t q_tx = 0;
#pragma unroll
      for (int q = 0; q < NQ; ++q) q_tx += n_q[q] > 0 ? q_bytes : 0u;
      mbar_arrive_expect_tx(bar(kBarQ), q_tx);
      for (int q = 0; q < NQ; ++q)
        if (n_q[q] > 0)
          for (int pn = 0; pn < a.dpanels; ++pn) {
            if (a.qo5)
              tma_load_5d(sQ + q * q_bytes + pn * a.q_rows * 128, &a.tmq, bar(kBarQ), pn * 64, (int)i0[q], hhq[q],
                          (int)hkv, (int)bb);
            else
              tma_load_3d(sQ + q * q_bytes + pn * a.q_rows * 128, &a.tmq, bar(kBarQ), pn * 64, (int)row0[q], (int)bh);
          }
      // A split call reads each key block once, for every row it holds: its keys and
      // values go first out of L2, before the partials the merge pass reads back.
      const uint64_t l2_once = l2_policy_evict_first();
      // one ring slot: wait until its previous tile is released, then load tile t into it
      auto load = [&](int full, int empty, uint32_t ring, uint32_t bytes, const CUtensorMap* tm1, int panels1,
                      uint32_t ring2, const CUtensorMap* tm2, int panels2, int t) {
        const int s = t % STG;
        if (!mbar_wait(bar(empty + s), ((t / STG) & 1) ^ 1, limit, abort)) {
          fail(p, abort, kStatTimeoutSlotFree);
          return false;
        }
        mbar_arrive_expect_tx(bar(full + s), bytes);
        for (int pn = 0; pn < panels1; ++pn) {
          const uint32_t dst = ring + s * (panels1 * BN * 128) + pn * BN * 128;
          if (a.split)
            tma_load_4d_hint(dst, tm1, bar(full + s), pn * 64, (kt0 + t) * BN, (int)hkv, (int)bb, l2_once);
          else
            tma_load_4d(dst, tm1, bar(full + s), pn * 64, (kt0 + t) * BN, (int)hkv, (int)bb);
        }
        for (int pn = 0; pn < panels2; ++pn) {
          const uint32_t dst = ring2 + s * (panels2 * BN * 128) + pn * BN * 128;
          if (a.split)
            tma_load_4d_hint(dst, tm2, bar(full + s), pn * 64, (kt0 + t) * BN, (int)hkv, (int)bb, l2_once);
          else
            tma_load_4d(dst, tm2, bar(full + s), pn * 64, (kt0 + t) * BN, (int)hkv, (int)bb);
        }
        return true;
      };
      int k_issued = 0, v_issued = 0;
      if constexpr (NQ == 2) {
        // K and V of tile t together into stage t % STG
        for (int t = 0; t < n_max; ++t) {
          const int s = t % STG;
          if (!mbar_wait(bar(kBarKvEmpty + s), ((t / STG) & 1) ^ 1, limit, abort)) {
            fail(p, abort, kStatTimeoutSlotFree);
            break;
          }
          mbar_arrive_expect_tx(bar(kBarKvFull + s), k_bytes + v_bytes);
          for (int pn = 0; pn < a.dpanels; ++pn)
            tma_load_4d(sK + s * k_bytes + pn * BN * 128, &a.tmk, bar(kBarKvFull + s), pn * 64, (kt0 + t) * BN,
                        (int)hkv, (int)bb);
          for (int pn = 0; pn < a.dvpanels; ++pn)
            tma_load_4d(sV + s * v_bytes + pn * BN * 128, &a.tmv, bar(kBarKvFull + s), pn * 64, (kt0 + t) * BN,
                        (int)hkv, (int)bb);
          k_issued = v_issued = t + 1;
        }
      } else {
        // K runs one tile ahead of V (S of tile t + 1 is issued before P V of tile t)
        if (load(kBarKvFull, kBarKvEmpty, sK, k_bytes, &a.tmk, a.dpanels, sV, &a.tmv, 0, 0)) {
          k_issued = 1;
          for (int t = 0; t < n_max; ++t) {
            if (t + 1 < n_max) {
              if (!load(kBarKvFull, kBarKvEmpty, sK, k_bytes, &a.tmk, a.dpanels, sV, &a.tmv, 0, t + 1)) break;
              k_issued = t + 2;
            }
            if (!load(kBarVFull, kBarVEmpty, sV, v_bytes, &a.tmv, a.dvpanels, sK, &a.tmk, 0, t)) break;
            v_issued = t + 1;
          }
        }
      }
      // Every copy issued must land before the CTA may exit (a no-op when all were consumed).
      mbar_wait(bar(kBarQ), 0, kDrainLimit, nullptr);
      for (int t = k_issued > STG ? k_issued - STG : 0; t < k_issued; ++t)
        mbar_wait(bar(kBarKvFull + t % STG), (t / STG) & 1, kDrainLimit, nullptr);
      if constexpr (NQ == 1)
        for (int t = v_issued > STG ? v_issued - STG : 0; t < v_issued; ++t)
          mbar_wait(bar(kBarVFull + t % STG), (t / STG) & 1, kDrainLimit, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0 && n_max > 0) {
      const uint32_t idesc_s = idesc_f16(TypeCode<T>::v, 0, 0, kBM, BN);
      const uint32_t idesc_o = idesc_f16(TypeCode<T>::v, 0, 1, kBM, a.n_pv);
      // Descriptors are built once; a K-step or a stage only moves the start address,
      // which sits in the low bits (16-byte units, below 256 KB: no carry out of the
      // field), so issuing an MMA costs one add -- the single issuing thread must keep
      // up with 64-cycle 128x128x16 MMAs.
      const uint64_t qd0 = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t kd0 = smem_desc_sw128(sK, 16, 1024);
      const uint64_t vd0 = smem_desc_sw128(sV, BN * 128, 1024);
      // S = Q_q K_t^T into S slot `slot`, then commit to s_full[slot]
      auto issue_s = [&](int t, int q, int slot) {
        const uint32_t dst = tmem + tS_col(slot);
        const uint64_t ad = qd0 + (uint64_t)(q * (q_bytes >> 4));
        const uint32_t q_pan = (uint32_t)a.q_rows * 8;  // a Q panel in 16-byte units
        const uint64_t bd = kd0 + (uint64_t)((t % STG) * (k_bytes >> 4));
        if (a.ksteps_qk == kMaxKsteps) {
          // the head fills this variant: straight-line issue, no branch between MMAs (the
          // single issuing thread must keep pace with 64-cycle 128x128x16 MMAs)
#pragma unroll
          for (int k = 0; k < kMaxKsteps; ++k)
            mma_ss(dst, ad + (uint64_t)((k >> 2) * q_pan + (k & 3) * 2),
                   bd + (uint64_t)((k >> 2) * (BN * 8) + (k & 3) * 2), idesc_s, k > 0);
        } else {
          for (int k = 0; k < a.ksteps_qk; ++k)
            mma_ss(dst, ad + (uint64_t)((k >> 2) * q_pan + (k & 3) * 2),
                   bd + (uint64_t)((k >> 2) * (BN * 8) + (k & 3) * 2), idesc_s, k > 0);
        }
        mma_commit(bar(kBarSFull + slot));
      };
      // O_q += P (from S slot `slot`) V_t, then commit to pv_done[q]
      auto issue_pv = [&](int t, int q, int slot) {
        const uint32_t dst = tmem + tO_col(q), src = tmem + tS_col(slot);
        const uint64_t bd = vd0 + (uint64_t)((t % STG) * (v_bytes >> 4));
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(dst, src + kk * 8, bd + (uint64_t)(kk * 128), idesc_o, (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(kBarPvDone + q));
      };
      // (the issuer's waits never suspend: see mbar_wait)
      auto wait_kv = [&](int t) {
        if (mbar_wait<false>(bar(kBarKvFull + t % STG), (t / STG) & 1, limit, abort)) {
          tc_fence_after();
          return true;
        }
        fail(p, abort, kStatTimeoutTmaFull);
        return false;
      };
      auto wait_p = [&](int slot, uint32_t parity) {
        if (mbar_wait<false>(bar(kBarPFull + slot), parity, limit, abort)) {
          tc_fence_after();
          return true;
        }
        fail(p, abort, kStatTimeoutMma);
        return false;
      };
      bool ok = mbar_wait<false>(bar(kBarQ), 0, limit, abort);
      if (!ok) fail(p, abort, kStatTimeoutTmaFull);
      ok = ok && wait_kv(0);
      if constexpr (NQ == 1) {
        // K slots are released once their S is done, V slots once their P V is
        auto wait_v = [&](int t) {
          if (mbar_wait<false>(bar(kBarVFull + t % STG), (t / STG) & 1, limit, abort)) {
            tc_fence_after();
            return true;
          }
          fail(p, abort, kStatTimeoutTmaFull);
          return false;
        };
        if (ok) {
          issue_s(0, 0, 0);
          mma_commit(bar(kBarKvEmpty));
        }
        for (int t = 0; ok && t < n_max; ++t) {
          if (t + 1 < n_max) {
            if (!(ok = wait_kv(t + 1))) break;
            issue_s(t + 1, 0, (t + 1) & 1);
            mma_commit(bar(kBarKvEmpty + (t + 1) % STG));
          }
          if (!(ok = wait_p(t & 1, (t >> 1) & 1))) break;
          if (!(ok = wait_v(t))) break;
          issue_pv(t, 0, t & 1);
          mma_commit(bar(kBarVEmpty + t % STG));
        }
      } else {
        if (ok) {
          if (n_q[0] > 0) issue_s(0, 0, 0);
          if (n_q[1] > 0) issue_s(0, 1, 1);
        }
        for (int t = 0; ok && t < n_max; ++t) {
          const bool nxt = t + 1 < n_max;
          if (t < n_q[0]) {
            if (!(ok = wait_p(0, t & 1))) break;
            issue_pv(t, 0, 0);
          }
          if (nxt && !(ok = wait_kv(t + 1))) break;
          if (nxt && t + 1 < n_q[0]) issue_s(t + 1, 0, 0);
          if (t < n_q[1]) {
            if (!(ok = wait_p(1, t & 1))) break;
            issue_pv(t, 1, 1);
          }
          mma_commit(bar(kBarKvEmpty + t % STG));
          if (nxt && t + 1 < n_q[1]) issue_s(t + 1, 1, 1);
        }
      }
      // all MMAs issued by this thread complete before TMEM can be freed
      mma_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, kDrainLimit, nullptr);
    }
    __syncwarp();
  } else {
    // ================================================================ softmax / epilogue
    // (a bit-packed mask is written by the packing grid this kernel may overlap)
    if constexpr (MM == kMmBits) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int q = (warp - 2) / 4;  // which Q tile this warpgroup serves
    const int q4 = warp & 3;       // TMEM lane quarter this warp may access
    const int row = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    // (selects, not an index: the arrays stay in registers)
    const int i0_q = q == 0 ? i0[0] : i0[NQ - 1], row0_q = q == 0 ? row0[0] : row0[NQ - 1];
    const int hhq_q = q == 0 ? hhq[0] : hhq[NQ - 1];
    bool row_ok;
    int i, hh;
    if (a.head_local) {
      i = i0_q + row;
      row_ok = i < p.Lq;
      hh = hhq_q;
      if (!row_ok) i = 0;
    } else {
      const int rho = row0_q + row;
      row_ok = rho < p.G;
      i = row_ok ? rho % (int)p.Lq : 0;
      hh = row_ok ? rho / (int)p.Lq : 0;
    }
    const int h = hkv * (int)p.g + hh;
    // the keys [first_key, last_key] this row may see (key indices fit 32 bits: the
    // planner sends no longer sequence here)
    const int64_t pos = i + p.Lk - p.Lq;
    const int first_key = (int)row_key_lo(p, pos), last_key = (int)row_key_hi(p, pos, p.Lk) - 1;
    const uint32_t* mrow = MM == kMmBits ? a.mask_bits + (int64_t)i * a.mask_words : nullptr;
    const void* mrow_any = mrow;
    if constexpr (MM == kMmAdd)
      mrow_any = reinterpret_cast<const T*>(p.amask) + bb * p.am_sb + h * p.am_sh + (int64_t)i * p.Lk;
    const int n_tiles = q == 0 ? n_q[0] : n_q[NQ - 1];
    const uint32_t tO = tmem + lane_base + tO_col(q);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    if constexpr (NQ == 2) {
      uint32_t no_words[BN / 32];  // (the mask words are loaded inside the softmax)
      for (int t = 0; t < n_tiles; ++t) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + q), t & 1, limit, abort));
        if (!ok) {
          fail(p, abort, kStatTimeoutMma);
          break;
        }
        tc_fence_after();
        // S of this tile was issued after P_{t-1} V_{t-1} of the same Q tile, and a commit
        // tracks every earlier MMA of the issuing thread, so s_full already implies that O
        // holds P_{t-1} V_{t-1}
        uint32_t no_add[av_words<BN, MM>()];  // (additive masks take the one-tile variant)
        ok = softmax_tile<T, BN, NQ, MM, false>(a, t, kt0 + t, tmem + lane_base + tS_col(q), tO, row_ok, first_key,
                                            last_key, mrow_any, no_words, no_add, m_run, l_run, bar(kBarPvDone + q),
                                            false, false, limit, abort);
        if (!ok) {
          fail(p, abort, kStatTimeoutMma);
          break;
        }
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + q));
      }
    } else {
      // this row's bit-packed mask words of a key tile, loaded one tile ahead so that the
      // global-memory latency falls in the wait for S rather than in the softmax
      uint32_t mw[BN / 32];
      auto load_mw = [&](int t, uint32_t (&dst)[BN / 32]) {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          dst[c] = (MM == kMmBits && row_ok) ? __ldg(mrow + ((kt0 + t) * BN) / 32 + c) : 0u;
      };
      if (n_tiles > 0) load_mw(0, mw);
      // this row's additive-mask values (kMmAdd) of tile t, from the staged chunk: its
      // copy starts at the 8-element boundary below the chunk's first column, so the tile's
      // columns start m + (t mod kAmTiles) * BN elements in (m = the row's offset mod 8,
      // the same for every chunk: 8 divides BN)
      const int64_t am_row_off =
          MM == kMmAdd ? (int64_t)(reinterpret_cast<const T*>(mrow_any) - reinterpret_cast<const T*>(p.amask)) : 0;
      const int am_m = (int)(am_row_off & 7);  // (the tensor starts on a 16-byte boundary)
      // this row's slot in the staging buffers.  A slot's pitch is 4 words past a multiple
      // of 32 banks, and a row's tile starts (am_m >> 1) words into it; with the rows in
      // slot order a warp's 32-bit reads of its 32 rows met 4 to a bank.  Slot 8 j + 2 q + e
      // holds lane 8 q + 2 j + e: the four lanes sharing a bank group (same q and e) then
      // start at four different word phases whenever Lk is odd (consecutive queries of one
      // row tile), and the reads are free of conflicts
      const int am_slot = q4 * 32 + 8 * ((lane & 7) >> 1) + 2 * (lane >> 3) + (lane & 1);
      // this row's copy of chunk c (key tiles [kAmTiles c, kAmTiles c + kAmTiles) of the walk)
      // into buffer c & 1: [a0, a0 + row bytes) from the 8-element boundary at or below its
      // first column, clipped to the tensor's last 16-byte boundary; every softmax thread
      // arrives on the buffer's barrier with its bytes, a row past the tile's end with none
      const int n_chunks = MM == kMmAdd ? (n_tiles + kAmTiles - 1) / kAmTiles : 0;
      auto issue_chunk = [&](int c) {
        if constexpr (MM == kMmAdd) {
          const int b = c & 1;
          const int64_t a0 = (am_row_off + (int64_t)(kt0 + kAmTiles * c) * BN) & ~int64_t(7);
          uint32_t n = 0;
          if (row_ok && a0 < a.amask_total) {
            const int64_t avail = (a.amask_total - a0) * 2;
            n = (uint32_t)(avail >= am_row_bytes<BN>() ? am_row_bytes<BN>() : (avail & ~int64_t(15)));
          }
          const uint32_t fb = bar(kBarMFull + b);
          // (the buffer's previous contents were read by this thread alone, by generic loads)
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(fb, n);
          if (n) bulk_load(sM + b * (kBM * am_row_bytes<BN>()) + am_slot * am_row_bytes<BN>(),
                           reinterpret_cast<const T*>(p.amask) + a0, n, fb);
        }
      };
      int chunks_issued = 0, chunks_seen = 0;
      for (; chunks_issued < 2 && chunks_issued < n_chunks; ++chunks_issued) issue_chunk(chunks_issued);
      for (int t = 0; t < n_tiles; ++t) {
        uint32_t mw_next[BN / 32];
        if (t + 1 < n_tiles) load_mw(t + 1, mw_next);
        const int slot = t & 1;
        uint32_t av[av_words<BN, MM>()];
        if constexpr (MM == kMmAdd) {
          const int c = t / kAmTiles, b = c & 1;
          if (t % kAmTiles == 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarMFull + b), (c >> 1) & 1, limit, abort));
            if (!ok) {
              fail(p, abort, kStatTimeoutTmaFull);
              break;
            }
            chunks_seen = c + 1;
          }
          const int e0 = am_m + (t % kAmTiles) * BN;
          const uint32_t rs = sM + b * (kBM * am_row_bytes<BN>()) + am_slot * am_row_bytes<BN>() + (e0 >> 1) * 4;
          uint32_t w[BN / 2 + 1];
#pragma unroll
          for (int k = 0; k < BN / 2 + 1; ++k)
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[k]) : "r"(rs + 4 * k) : "memory");
#pragma unroll
          for (int k = 0; k < BN / 2; ++k) av[k] = (e0 & 1) ? __funnelshift_r(w[k], w[k + 1], 16) : w[k];
          // the tensor's last elements past its last 16-byte boundary are not staged (a bulk
          // copy moves whole 16-byte units): the row that ends there reads them directly
          const int64_t g0 = am_row_off + (int64_t)(kt0 + t) * BN, staged_end = a.amask_total & ~int64_t(7);
          if (row_ok && g0 + BN > staged_end) {
            const unsigned short* mb = reinterpret_cast<const unsigned short*>(p.amask);
            for (int k = 0; k < BN / 2; ++k) {
              const int64_t e = g0 + 2 * k;
              uint32_t lo = av[k] & 0xffffu, hi = av[k] >> 16;
              if (e >= staged_end && e < a.amask_total) lo = __ldg(mb + e);
              if (e + 1 >= staged_end && e + 1 < a.amask_total) hi = __ldg(mb + e + 1);
              av[k] = lo | (hi << 16);
            }
          }
          // the chunk's buffer row is this thread's again once its last tile is read: chunk
          // c + 2 goes into it
          if ((t % kAmTiles == kAmTiles - 1 || t + 1 == n_tiles) && c + 2 < n_chunks) {
            issue_chunk(c + 2);
            chunks_issued = c + 3;
          }
        }
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + slot), (t >> 1) & 1, limit, abort));
        if (!ok) {
          fail(p, abort, kStatTimeoutMma);
          break;
        }
        tc_fence_after();
        // S_t was issued before P_{t-1} V_{t-1}: the softmax waits for that product
        ok = softmax_tile<T, BN, NQ, MM, true>(a, t, kt0 + t, tmem + lane_base + tS_col(slot), tO, row_ok, first_key,
                                           last_key, mrow_any, mw, av, m_run, l_run, bar(kBarPvDone + q), true,
                                           t + 1 == n_tiles, limit, abort);
        if (!ok) {
          fail(p, abort, kStatTimeoutMma);
          break;
        }
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + slot));
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) mw[c] = mw_next[c];
      }
      if constexpr (MM == kMmAdd) {
        // a loop that stopped early leaves chunk copies in flight: they land before the
        // CTA may leave (bounded: a barrier some thread never arrived on gives up)
        for (int c = chunks_seen; c < chunks_issued; ++c)
          mbar_wait(bar(kBarMFull + (c & 1)), (c >> 1) & 1, kDrainLimit, nullptr);
      }
    }
    // ---- epilogue
    if (ok && n_tiles > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarPvDone + q), (n_tiles - 1) & 1, limit, abort));
      if (!ok) fail(p, abort, kStatTimeoutMma);
      tc_fence_after();
    }
    ok = __all_sync(0xffffffffu, ok && !*abort);
    if (NQ == 1 && a.split && p.nblk > 1) {
      // this key block's partial of the row: (m, l) and the unnormalised O
      if (ok) partial_row(p, tO, n_tiles > 0, row_ok, bb, h, i, blk, m_run, l_run);
    } else if (a.tma_out) {
      // The tile goes out through shared memory and one TMA store per panel: the row
      // stores of a warp would touch 32 rows each, and a CTA could not retire before
      // they drained.  The stage is this Q tile's buffer, unread since its last S
      // product completed (before the last P V that the wait above saw done), and never
      // loaded at all when the tile sees no key.  Every thread of the warpgroup reaches
      // the barrier, whatever happened before it.
      uint8_t* stage = base + q * q_bytes;
      const bool leader = warp == 2 + 4 * q && lane == 0;
      if constexpr (NQ == 2) {
        // (the two-tile variant, at its register limit, stages the whole tile first)
        if (ok) epilogue_row_smem<T>(p, tO, n_tiles > 0, row_ok, bb, h, i, m_run, l_run, stage, row);
        fence_proxy_async_smem();
        const bool all_ok = bar_and(1 + q, 128, ok);
        if (all_ok && leader) {
          for (int pn = 0; pn < a.dvpanels; ++pn) {
            if (a.qo5)
              tma_store_5d(&a.tmo, smem_addr(stage + pn * (kBM * 128)), pn * 64, i0_q, hhq_q, (int)hkv, (int)bb);
            else
              tma_store_3d(&a.tmo, smem_addr(stage + pn * (kBM * 128)), pn * 64, row0_q, (int)bh);
          }
          bulk_commit_group();
          bulk_wait_read_all();  // the stage must stay intact until the copy has read it
        }
      } else {
      // Panel by panel: each panel's TMA store runs while the next one is staged.
      const float f = ok ? epilogue_factor<T>(p, row_ok, bb, h, i, m_run, l_run) : 0.f;
      for (int pn = 0; pn < a.dvpanels; ++pn) {
        if (ok) epilogue_panel_smem<T>(p, tO, n_tiles > 0, f, stage, row, pn);
        fence_proxy_async_smem();
        const bool all_ok = bar_and(1 + q, 128, ok);
        if (all_ok && leader) {
          if (a.qo5)
            tma_store_5d(&a.tmo, smem_addr(stage + pn * (kBM * 128)), pn * 64, i0_q, hhq_q, (int)hkv, (int)bb);
          else
            tma_store_3d(&a.tmo, smem_addr(stage + pn * (kBM * 128)), pn * 64, row0_q, (int)bh);
          bulk_commit_group();
        }
      }
      if (leader) bulk_wait_read_all();  // the stage must stay intact until the copies have read it
      }
    } else if (ok) {
      epilogue_row<T>(p, tO, n_tiles > 0, row_ok, bb, h, i, m_run, l_run);
    }
  }

  // ---- tear-down
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
  }
}

// Bool mask [Lq, Lk] bytes -> bits [Lq, words]: bit e of word w = mask[i, 32 w + e] != 0,
// zero past Lk (the key tiles' padding).  A warp packs four words of a row per step: its
// lanes read 32 consecutive bytes per word (any alignment) and one ballot gives the word.
// The attention kernel is launched as a programmatic dependent: it may start once every
// CTA here has begun, and its softmax warps wait for this grid before reading a bit.
constexpr int kPackWarps = 8;
__global__ void __launch_bounds__(kPackWarps * 32)
sdpa_pack_mask_bits(const uint8_t* __restrict__ mask, int64_t Lq, int64_t Lk, int64_t words,
                    uint32_t* __restrict__ bits) {
  // the stream's previous kernel has finished (and its writes are visible) before the
  // mask is read and before the attention kernel may launch: that kernel copies Q, K
  // and V without a wait of its own
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int64_t quads = words / 4;  // words per row is a multiple of 4
  const int64_t n = Lq * quads;
  const int64_t nwarps = (int64_t)gridDim.x * kPackWarps;
  for (int64_t x = (int64_t)blockIdx.x * kPackWarps + (threadIdx.x >> 5); x < n; x += nwarps) {
    const int64_t i = x / quads, w0 = (x % quads) * 4;
    const uint8_t* row = mask + i * Lk;
    uint32_t v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t j = (w0 + k) * 32 + lane;
      v[k] = __ballot_sync(0xffffffffu, j < Lk && row[j] != 0);
    }
    if (lane < 4) bits[i * words + w0 + lane] = lane == 0 ? v[0] : (lane == 1 ? v[1] : (lane == 2 ? v[2] : v[3]));
  }
}

// ------------------------------------------------------------------------- host side

template <typename T, int BN, int NQ, int MM, int STG>
cudaError_t launch_tc_t(const TcArgs& a, size_t smem, int64_t grid, cudaStream_t st) {
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e =
      set_max_dynamic_smem_once(configured, (const void*)sdpa_prefill_tc<T, BN, NQ, MM, STG>, (int)kTcMaxSmem);
  if (e != cudaSuccess) return e;
  // (with a boolean mask: behind the mask packing, whose grid waited for the stream's
  // earlier work; the prologue, the Q loads and the first products overlap the packing,
  // and the softmax warps wait for its bits)
  return launch_dependent(sdpa_prefill_tc<T, BN, NQ, MM, STG>, dim3((unsigned)grid), dim3(tc_threads<NQ>()), smem,
                          st, a);
}

template <typename T, int MM>
cudaError_t launch_tc_mm(int bn, int nq, int stg, const TcArgs& a, size_t smem, int64_t grid, cudaStream_t st) {
  if constexpr (MM == kMmAdd) {
    // (additive masks always take the one-tile variant with 64-key tiles and one stage)
    if (nq != 1 || bn != 64 || stg != 1) return cudaErrorInvalidValue;
    return launch_tc_t<T, 64, 1, MM, 1>(a, smem, grid, st);
  } else {
    if (nq == 2) return stg == 2 ? launch_tc_t<T, 128, 2, MM, 2>(a, smem, grid, st) : cudaErrorInvalidValue;
    if (stg == 3 && bn != 64) return cudaErrorInvalidValue;
    if (bn == 64) {
      if constexpr (MM == kMmBounds) {
        if (stg == 3) return launch_tc_t<T, 64, 1, MM, 3>(a, smem, grid, st);
      }
      return stg == 2 ? launch_tc_t<T, 64, 1, MM, 2>(a, smem, grid, st) : cudaErrorInvalidValue;
    }
    return stg == 2 ? launch_tc_t<T, 128, 1, MM, 2>(a, smem, grid, st) : launch_tc_t<T, 128, 1, MM, 1>(a, smem, grid, st);
  }
}

template <typename T>
cudaError_t launch_tc_cfg(int bn, int nq, int stg, const TcArgs& a, size_t smem, int64_t grid, cudaStream_t st) {
  if (a.p.mask_kind == kMaskBool) return launch_tc_mm<T, kMmBits>(bn, nq, stg, a, smem, grid, st);
  if (a.p.mask_kind == kMaskAdd) return launch_tc_mm<T, kMmAdd>(bn, nq, stg, a, smem, grid, st);
  return launch_tc_mm<T, kMmBounds>(bn, nq, stg, a, smem, grid, st);
}

size_t smem_need(int64_t d, int64_t dv, int bn, int nq, int stg, int q_rows = kBM, bool pad = true) {
  const int64_t dp = (d + 63) / 64, dvp = (dv + 63) / 64;
  return (size_t)(nq * dp * q_rows * 128 + stg * (dp + dvp) * bn * 128) + (pad ? 1024 : 0) /*align*/ +
         256 /*bars*/;
}

// The key tile and the depth of the K / V rings of the one-tile variant: the largest
// tile whose two S buffers and O fit the 512 TMEM columns, with two stages if they fit in
// shared memory, else one (each ring then refills while the other operand's product runs;
// 128-key tiles keep the S products at the full MMA rate, where 64-key ones run at 2/3).
struct TileChoice {
  int bn, stg;
};
TileChoice tile_choice(int64_t d, int64_t dv, int max_stages = 2) {
  const int64_t npv = (dv + 15) / 16 * 16;
  for (int bn : {128, 64})
    for (int stg = max_stages; stg >= 1; --stg)
      if ((int64_t)smem_need(d, dv, bn, 1, stg) <= kTcMaxSmem && 2 * bn + npv <= kTmemCols) return {bn, stg};
  return {0, 0};
}

}  // namespace

int prefill_tc_bn(int64_t d, int64_t dv) { return tile_choice(d, dv).bn; }

int prefill_tc_q_tiles(int64_t d, int64_t dv, int64_t G) {
  // two Q tiles share each K/V tile when both O accumulators fit next to the two S
  // tiles (dv <= 128), both Q tiles and the ring fit in shared memory, and there are
  // more than 128 rows to fill them
  if (dv <= 128 && prefill_tc_bn(d, dv) == 128 && (int64_t)smem_need(d, dv, 128, 2, 2) <= kTcMaxSmem && G > kBM)
    return 2;
  return 1;
}

size_t prefill_tc_smem_bytes(int64_t d, int64_t dv, int bn, int nq, int stg) {
  const size_t s = smem_need(d, dv, bn, nq, stg);
  // at least 120 KB so that one CTA (with its 512 TMEM columns) owns the SM
  return s < 120 * 1024 ? 120 * 1024 : s;
}

int64_t prefill_tc_rows_per_cta(int64_t d, int64_t dv, int64_t G) { return kBM * prefill_tc_q_tiles(d, dv, G); }

bool prefill_tc_supported(int dtype, int64_t d, int64_t dv) {
  return (dtype == 1 || dtype == 2) && d % 8 == 0 && dv % 8 == 0 && d <= 256 && dv <= 256 &&
         prefill_tc_bn(d, dv) != 0;
}

size_t prefill_tc_mask_words(int64_t Lk) {
  // words per mask row: every key tile of up to 128 keys reads whole words
  return (size_t)((Lk + 127) / 128 * 4);
}

PrefillGeom prefill_tc_geometry(int64_t B, int64_t Hkv, int64_t g, int64_t Lq, int64_t d, int64_t dv,
                                bool qo_packed, bool additive, int64_t nblk) {
  PrefillGeom r{};
  if (nblk > 0) {
    // split-KV over nblk key blocks: one Q tile of packed rows per CTA and key block.
    // Heads up to 128: 64-key tiles and 256 TMEM columns, so that two CTAs -- two
    // independent streams of keys -- share each SM, with three-stage rings where the rows
    // fit a 64-row Q buffer (the two CTAs' shared memory then fits only unpadded), else
    // two; wider heads: the one-tile variant's own tiles, one CTA per SM.
    const bool small = d <= 128 && dv <= 128;
    const bool q64 = small && g * Lq <= 64;
    const TileChoice tc = small ? TileChoice{64, q64 ? 3 : 2} : tile_choice(d, dv);
    r.bn = tc.bn;
    r.stg = tc.stg;
    r.tmem_cols = small ? 256 : 512;
    r.q_rows = q64 ? 64 : kBM;
    r.unpadded = q64 ? 1 : 0;
    r.nq = 1;
    r.head_local = 0;
    r.qo5 = 0;
    r.n_it = (Lq + kBM - 1) / kBM;
    r.n_rt = (g * Lq + kBM - 1) / kBM;
    r.grid = B * Hkv * r.n_rt * nblk;
    r.split = 1;
    return r;
  }
  // (an additive mask takes 64-key tiles: a tile's values live in registers)
  const TileChoice tc = tile_choice(d, dv);
  r.bn = additive ? 64 : tc.bn;
  const int64_t G = g * Lq;
  // (an additive mask is staged in shared memory: the one-tile variant has room)
  r.nq = additive ? 1 : prefill_tc_q_tiles(d, dv, G);
  // (an additive mask stages its values next to one-stage K and V rings)
  r.stg = additive ? 1 : ((r.nq == 2 || r.bn == 64) ? 2 : tc.stg);
  // strided q / out: Q tiles of one query head each (pairs of heads need an even group)
  if (!qo_packed && g % 2 != 0) r.nq = 1;
  r.qo5 = qo_packed ? 0 : 1;
  // Packed rows with two Q tiles, an even group and whole 128-position blocks: the two
  // tiles are the same positions of two heads (equal key extents).  Strided: always
  // head-local tiles.
  r.head_local = (!qo_packed || (r.nq == 2 && g % 2 == 0 && Lq % kBM == 0)) ? 1 : 0;
  r.n_it = (Lq + kBM - 1) / kBM;
  r.n_rt = (G + kBM * r.nq - 1) / (kBM * r.nq);
  r.grid = r.head_local ? B * Hkv * (g / r.nq) * r.n_it : B * Hkv * r.n_rt;
  r.tmem_cols = kTmemCols;
  r.q_rows = kBM;
  r.unpadded = 0;
  return r;
}

cudaError_t launch_prefill_tc(int dtype, const Params& p, uint32_t* mask_bits, bool split, cudaStream_t st) {
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.p = p;
  const PrefillGeom geo = prefill_tc_geometry(p.B, p.Hkv, p.g, p.Lq, p.d, p.dv, p.qo_packed != 0,
                                              p.mask_kind == kMaskAdd, split ? p.nblk : 0);
  // the split form reads packed q / out rows, with the key bounds (no mask tensor, window)
  if (split && (!p.qo_packed || p.mask_kind == kMaskBool || p.mask_kind == kMaskAdd || p.window > 0 || p.nblk < 1 ||
                p.keys_per_blk % geo.bn != 0 || (p.nblk > 1 && (!p.part_o || !p.part_ml))))
    return cudaErrorInvalidValue;
  a.split = geo.split;
  a.blk_tiles = split ? (int)(p.keys_per_blk / geo.bn) : 0;
  a.tmem_cols = geo.tmem_cols;
  const int bn = geo.bn, nq = geo.nq, stg = geo.stg;
  const size_t am_extra = p.mask_kind == kMaskAdd ? (size_t)am_bytes<64>() : 0;
  const size_t need = smem_need(p.d, p.dv, bn, nq, stg, geo.q_rows, !geo.unpadded);
  if (!bn || !prefill_tc_bn(p.d, p.dv) || (int64_t)(need + am_extra) > kTcMaxSmem) return cudaErrorInvalidValue;
  a.q_rows = geo.q_rows;
  a.unpadded = geo.unpadded;
  const int64_t BH = p.B * p.Hkv;
  // K and V as 4-D [B][Hkv][Lk][d] views with the caller's strides
  const int64_t kd[4] = {p.d, p.Lk, p.Hkv, p.B}, ks[3] = {p.k_sl, p.k_sh, p.k_sb};
  const int64_t vd[4] = {p.dv, p.Lk, p.Hkv, p.B}, vs[3] = {p.v_sl, p.v_sh, p.v_sb};
  if (!encode_tiled_16bit(&a.tmk, dtype, p.k, 4, kd, ks, bn) || !encode_tiled_16bit(&a.tmv, dtype, p.v, 4, vd, vs, bn))
    return cudaErrorInvalidValue;
  const bool out_fits = (p.dv + 63) / 64 <= (p.d + 63) / 64;  // the output tile fits the Q tile's buffer
  if (geo.qo5) {
    // q and out as 5-D [B][Hkv][g][Lq][D] views: query head h = hkv * g + hh
    const int64_t qd[5] = {p.d, p.Lq, p.g, p.Hkv, p.B}, qs[4] = {p.q_sl, p.q_sh, p.g * p.q_sh, p.q_sb};
    const int64_t od[5] = {p.dv, p.Lq, p.g, p.Hkv, p.B}, os[4] = {p.o_sl, p.o_sh, p.g * p.o_sh, p.o_sb};
    if (!encode_tiled_16bit(&a.tmq, dtype, p.q, 5, qd, qs, kBM)) return cudaErrorInvalidValue;
    a.tma_out = (out_fits && encode_tiled_16bit(&a.tmo, dtype, p.out, 5, od, os, kBM)) ? 1 : 0;
  } else {
    // the packed layout: [B*Hkv][G][D], the rows of one KV head contiguous
    if (!encode_3d(&a.tmq, dtype, p.q, p.d, p.G, BH, geo.q_rows)) return cudaErrorInvalidValue;
    // (the output tile is staged in the Q tile's buffer: a 64-row buffer is too small)
    a.tma_out = (out_fits && geo.q_rows == kBM && encode_3d(&a.tmo, dtype, p.out, p.dv, p.G, BH, kBM)) ? 1 : 0;
  }
  a.n_rt = (int)geo.n_rt;
  a.n_it = (int)geo.n_it;
  a.qo5 = geo.qo5;
  a.dpanels = (int)((p.d + 63) / 64);
  a.dvpanels = (int)((p.dv + 63) / 64);
  a.ksteps_qk = (int)((p.d + 15) / 16);
  a.n_pv = (int)((p.dv + 15) / 16 * 16);
  a.itile_order = (p.Lq % (kBM * nq) == 0) ? 1 : 0;
  a.head_local = geo.head_local;
  if (p.mask_kind == kMaskAdd)
    a.amask_total = (p.am_sb ? p.B * p.am_sb : (p.am_sh ? p.Hq * p.am_sh : p.Lq * p.Lk));
  if (p.mask_kind == kMaskBool) {
    a.mask_words = (int64_t)prefill_tc_mask_words(p.Lk);
    a.mask_bits = mask_bits;
    const int64_t n = p.Lq * (a.mask_words / 4);  // one warp step per four words
    int64_t g = (n + kPackWarps - 1) / kPackWarps;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (g > cap) g = cap;
    cudaError_t e = launch_dependent(sdpa_pack_mask_bits, dim3((unsigned)(g > 0 ? g : 1)), dim3(kPackWarps * 32), 0,
                                     st, p.mask, p.Lq, p.Lk, a.mask_words, mask_bits);
    if (e != cudaSuccess) return e;
  }
  const int64_t grid = geo.grid;
  // (two CTAs per SM: the ring and Q alone; otherwise at least 120 KB, one CTA per SM)
  const size_t smem = (geo.tmem_cols == 256 ? need : prefill_tc_smem_bytes(p.d, p.dv, bn, nq, stg)) + am_extra;
  if (dtype == 1) return launch_tc_cfg<__half>(bn, nq, stg, a, smem, grid, st);
  return launch_tc_cfg<__nv_bfloat16>(bn, nq, stg, a, smem, grid, st);
}

}  // namespace nvsdpa

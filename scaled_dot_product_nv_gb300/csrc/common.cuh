// Shared device-side definitions of the nv_sdpa kernels: element conversions, the
// launch parameters, the per-device status word and the bounded-wait budget.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvsdpa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaskNone = 0, kMaskCausal = 1, kMaskBool = 2, kMaskAdd = 3;

// Bits of the device status word (OR-ed in by a kernel whose bounded wait ran out).
enum : uint32_t {
  kStatTimeoutTmaFull = 1u << 0,   // a consumer waited too long for a TMA load
  kStatTimeoutSlotFree = 1u << 1,  // a producer waited too long for a free stage
  kStatTimeoutMma = 1u << 2,       // a waiter on an MMA commit gave up
  kStatTimeoutTmem = 1u << 3,      // waiting on the TMEM handoff gave up
  kStatBadConfig = 1u << 8,        // the kernel found a launch configuration it cannot run
};

// Everything a kernel needs to know about one call.
struct Params {
  const void* q;
  const void* k;
  const void* v;
  const uint8_t* mask;  // [Lq, Lk] or null
  const void* sinks;    // [Hq] or null
  void* out;            // [B, Hq, Lq, dv]
  float* lse;           // [B, Hq, Lq] or null
  float* part_o;        // split-KV partials [B*Hq*Lq][nblk][dv] (unnormalised)
  float* part_ml;       // [B*Hq*Lq][nblk][2]: running max (log2 units) and sum
  uint32_t* status;     // per-device status word
  int64_t B, Hq, Hkv, Lq, Lk, d, dv;
  int64_t g;            // Hq / Hkv
  int64_t G;            // g * Lq: query rows that share one KV head
  int64_t nblk;         // key blocks per KV head (1 = final output written directly)
  int64_t keys_per_blk; // keys per block (a multiple of every kernel's key tile)
  int64_t row_tiles;    // ceil(G / rows per CTA)
  int64_t spans;        // decode: CTAs sharing the key blocks of one (b, KV head, row tile)
  int mask_kind;
  int has_sinks;
  float scale;          // as passed
  float scale_log2;     // scale * log2(e): scores are kept in log2 units
  uint64_t wait_limit;  // spin budget of every bounded wait
  // Element strides along [B, H, L] of q, k, v and out (the head dimension is contiguous).
  int64_t q_sb, q_sh, q_sl, k_sb, k_sh, k_sl, v_sb, v_sh, v_sl, o_sb, o_sh, o_sl;
  int64_t window;       // > 0: the causal band p - window < j <= p; 0: no band
  const void* amask;    // additive mask [mB][mH][Lq][Lk] in the input type, or null
  int64_t am_sb, am_sh; // its element strides over b and h (0 where it is shared)
  // Paged caches (paged != 0): k, v are [num_pages][Hkv][page][d | dv], key j of sequence b
  // is position j % page of page table[b][j / page], and sequence b has lens[b] keys.
  const int32_t* table;
  const int32_t* lens;
  int64_t page, max_pages, num_pages;
  int paged;
  int qo_packed;        // q and out are contiguous [B, H, L, D] (the G rows of a KV head
                        // form one [G, D] block)
};

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// 2^x on the SFU; exact 0 for x = -inf.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Sink logit of query head h in log2 units, or -inf.
template <typename T>
__device__ __forceinline__ float sink_log2(const Params& p, int64_t h) {
  if (!p.has_sinks) return -INFINITY;
  return to_f32<T>(reinterpret_cast<const T*>(p.sinks)[h]) * kLog2e;
}

// Last key index query row i may see under the causal mask (bottom-right aligned).
__device__ __forceinline__ int64_t causal_last_key(const Params& p, int64_t i) {
  return i + (p.Lk - p.Lq);
}

// Keys of sequence b: Lk, or for paged caches its length clamped to [0, capacity].
__device__ __forceinline__ int64_t seq_keys(const Params& p, int64_t b) {
  if (!p.paged) return p.Lk;
  const int64_t L = p.lens[b];
  const int64_t cap = p.max_pages * p.page;
  return L < 0 ? 0 : (L > cap ? cap : L);
}

// The keys [lo, hi) that the query at absolute position `pos` (= i + Lkb - Lq) may see in
// a sequence of Lkb keys: the causal bound and the band of the window.
__device__ __forceinline__ int64_t row_key_hi(const Params& p, int64_t pos, int64_t Lkb) {
  if (p.mask_kind != kMaskCausal) return Lkb;
  const int64_t h = pos + 1;
  return h < 0 ? 0 : (h > Lkb ? Lkb : h);
}
__device__ __forceinline__ int64_t row_key_lo(const Params& p, int64_t pos) {
  if (p.window <= 0) return 0;
  const int64_t l = pos - p.window + 1;
  return l < 0 ? 0 : l;
}

// Element offset of key (or value) row j of (b, KV head hkv): strided, or through the page
// table (an entry out of range is clamped, never followed).
__device__ __forceinline__ int64_t kv_offset(const Params& p, int64_t b, int64_t hkv, int64_t j,
                                             int64_t sb, int64_t sh, int64_t sl, int64_t width) {
  if (!p.paged) return b * sb + hkv * sh + j * sl;
  int64_t blk = p.table[b * p.max_pages + j / p.page];
  blk = blk < 0 ? 0 : (blk >= p.num_pages ? p.num_pages - 1 : blk);
  return ((blk * p.Hkv + hkv) * p.page + j % p.page) * width;
}

// Element offset of (b, h, i) in q / out.
__device__ __forceinline__ int64_t q_offset(const Params& p, int64_t b, int64_t h, int64_t i) {
  return b * p.q_sb + h * p.q_sh + i * p.q_sl;
}
__device__ __forceinline__ int64_t o_offset(const Params& p, int64_t b, int64_t h, int64_t i) {
  return b * p.o_sb + h * p.o_sh + i * p.o_sl;
}

// Additive-mask term of (b, h, i, j) in log2 units.
template <typename T>
__device__ __forceinline__ float amask_log2(const Params& p, int64_t b, int64_t h, int64_t i, int64_t j) {
  const T* m = reinterpret_cast<const T*>(p.amask);
  return to_f32<T>(m[b * p.am_sb + h * p.am_sh + i * p.Lk + j]) * kLog2e;
}

__device__ __forceinline__ void record_status(const Params& p, uint32_t bits) {
  if (p.status) atomicOr(p.status, bits);
}

}  // namespace nvsdpa

// The C ABI of nv_sdpa: argument checks, the pure planner/router, launches on the
// caller's stream, the per-device status word and the host-buffer entry point.
//
// Checks follow "nuvec-core 0.6.1 tests/attention_plan.rs"
// (invalid_options_are_rejected_by_plan_and_op: the plan and the op reject the same
// inputs) and "nuvec-core 0.5.0 tests/fast.rs" (attention_fallback_matches_a_direct_formula:
// a head count that does not group is an error).  Size products are checked for
// overflow before anything is allocated, like the guards of "lattice-inference 0.4.0
// src/attention/flash.rs" (assert_tiled_scratch_no_overflow).
#include <atomic>
#include <mutex>
#include <vector>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "nv_sdpa.h"
#include "common.cuh"
#include "decode_blocks_table.h"
#include "kernels.h"

#define NV_SDPA_API extern "C" __attribute__((visibility("default")))

namespace nvsdpa {
namespace {

__device__ uint32_t g_status;  // per-device status word (bounded waits record here)

constexpr int kMaxDevices = 64;
std::atomic<uint32_t*> g_status_ptr[kMaxDevices];
std::atomic<uint64_t> g_wait_limit{0};
constexpr uint64_t kDefaultWaitLimit = 1ull << 18;  // polls, each suspending <= ~10 us

int elt_bytes(int dtype) { return dtype == NV_SDPA_F32 ? 4 : 2; }

// The library's own stream-ordered memory pool on each device.  Freed blocks stay in it
// for the next call: a pool whose release threshold is 0 (the default pool's default)
// hands its memory back to the system at every synchronisation, and mapping it again
// costs each call far more than the work it does.  Calls made with the library's memory
// keep at most their own peak of it.
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices];

cudaError_t pool_alloc(void** ptr, size_t bytes, cudaStream_t st) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return ce;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pools[dev]) {
      cudaMemPoolProps props;
      memset(&props, 0, sizeof(props));
      props.allocType = cudaMemAllocationTypePinned;
      props.handleTypes = cudaMemHandleTypeNone;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t created;
      ce = cudaMemPoolCreate(&created, &props);
      if (ce != cudaSuccess) return ce;
      uint64_t keep = UINT64_MAX;
      ce = cudaMemPoolSetAttribute(created, cudaMemPoolAttrReleaseThreshold, &keep);
      if (ce != cudaSuccess) {
        cudaMemPoolDestroy(created);
        return ce;
      }
      g_pools[dev] = created;
    }
    pool = g_pools[dev];
  }
  return cudaMallocFromPoolAsync(ptr, bytes, pool, st);
}

bool mul_ok(int64_t a, int64_t b, int64_t* r) {
  if (__builtin_mul_overflow(a, b, r)) return false;
  return *r <= (int64_t(1) << 62);
}

// Warps sharing one (b, KV head, 16-row tile)'s nblk key blocks in the decode kernel:
// as many as keep every warp of the grid resident at once (at least one, at most one
// per block).
int64_t decode_spans(const nv_sdpa_dims& x, int64_t nblk) {
  const int64_t rows = (x.Hq / x.Hkv) * x.Lq;
  const int64_t rc = (rows + decode_mma_rows_per_warp() - 1) / decode_mma_rows_per_warp();
  const int64_t warp_slots = (int64_t)device_sm_count() * decode_mma_ctas_per_sm(x.d, x.dv) * decode_mma_warps_per_cta(x.d, x.dv);
  int64_t units;
  if (!mul_ok(x.B * x.Hkv, rc, &units) || units < 1) return 1;
  return std::max<int64_t>(1, std::min(nblk, warp_slots / units));
}

// Checks that need no pointer.  Returns NV_SDPA_OK or the status.
int check_dims(const nv_sdpa_dims* dm, int mask_kind, int dtype) {
  if (!dm) return NV_SDPA_ERR_INVALID;
  const nv_sdpa_dims& x = *dm;
  if (dtype != NV_SDPA_F32 && dtype != NV_SDPA_F16 && dtype != NV_SDPA_BF16) return NV_SDPA_ERR_INVALID;
  if (mask_kind != NV_SDPA_MASK_NONE && mask_kind != NV_SDPA_MASK_CAUSAL && mask_kind != NV_SDPA_MASK_BOOL &&
      mask_kind != NV_SDPA_MASK_ADD)
    return NV_SDPA_ERR_INVALID;
  if (x.B < 0 || x.Hq < 0 || x.Lq < 0 || x.Lk < 0 || x.Hkv < 1 || x.d < 1 || x.dv < 1)
    return NV_SDPA_ERR_INVALID;
  if (x.Hq % x.Hkv != 0) return NV_SDPA_ERR_INVALID;
  const int64_t e = elt_bytes(dtype);
  int64_t t;
  // every tensor's byte size must be representable
  if (!mul_ok(x.B, x.Hq, &t) || !mul_ok(t, x.Lq, &t) || !mul_ok(t, std::max(x.d, x.dv), &t) || !mul_ok(t, e, &t))
    return NV_SDPA_ERR_INVALID;
  if (!mul_ok(x.B, x.Hkv, &t) || !mul_ok(t, x.Lk, &t) || !mul_ok(t, std::max(x.d, x.dv), &t) || !mul_ok(t, e, &t))
    return NV_SDPA_ERR_INVALID;
  if (!mul_ok(x.Lq, x.Lk, &t)) return NV_SDPA_ERR_INVALID;
  // head sizes this build has kernels for
  if (x.d > 256 || x.dv > 256 || x.d % 8 || x.dv % 8) return NV_SDPA_ERR_UNSUPPORTED;
  return NV_SDPA_OK;
}

// The options of one call, resolved: strides (contiguous when not given), the window
// and the additive mask's broadcast.
struct Resolved {
  int64_t qs[3], ks[3], vs[3], os[3];  // element strides along [B, H, L]
  int64_t window;                      // 0 = none
  const void* amask;
  int64_t am_sb, am_sh;
  bool qo_packed;                      // q and out contiguous
};

// Strides of one tensor [n0, n1, n2, width]: contiguous when all three are 0.  Checks that
// the largest offset is representable and, for 16-bit types, the 16-byte rule of TMA.
int resolve_strides(const int64_t* given, int64_t n0, int64_t n1, int64_t n2, int64_t width, int dtype,
                    int64_t* out, bool* contiguous) {
  const bool none = !given || (given[0] == 0 && given[1] == 0 && given[2] == 0);
  if (none) {
    out[2] = width;
    out[1] = n2 * width;
    out[0] = n1 * n2 * width;
    *contiguous = true;
    return NV_SDPA_OK;
  }
  for (int k = 0; k < 3; ++k)
    if (given[k] < 0) return NV_SDPA_ERR_INVALID;
  int64_t span = width, t;
  const int64_t n[3] = {n0, n1, n2};
  for (int k = 0; k < 3; ++k) {
    if (n[k] == 0) continue;
    if (!mul_ok(given[k], n[k] - 1, &t) || __builtin_add_overflow(span, t, &span) || span > (int64_t(1) << 60))
      return NV_SDPA_ERR_INVALID;
  }
  for (int k = 0; k < 3; ++k) out[k] = given[k];
  *contiguous = out[2] == width && out[1] == n2 * width && out[0] == n1 * n2 * width;
  if (dtype != NV_SDPA_F32)
    for (int k = 0; k < 3; ++k)
      if (out[k] % 8 != 0) return NV_SDPA_ERR_UNSUPPORTED;
  return NV_SDPA_OK;
}

int resolve_options(const nv_sdpa_dims& x, int mask_kind, int dtype, const nv_sdpa_options* opt, Resolved* r) {
  nv_sdpa_options zero;
  std::memset(&zero, 0, sizeof(zero));
  const nv_sdpa_options& o = opt ? *opt : zero;
  std::memset(r, 0, sizeof(*r));
  if (o.reserved0 != 0 || (o.has_window != 0 && o.has_window != 1)) return NV_SDPA_ERR_INVALID;
  if (o.has_window) {
    // "nuvec-core 0.5.0 tests/fast.rs", window_errors_empty_inputs_and_full_windows: a window
    // of 0, or a window without the causal mask, is an error
    if (o.window < 1 || mask_kind != NV_SDPA_MASK_CAUSAL) return NV_SDPA_ERR_INVALID;
    // a window of at least Lk keys hides no key from any row (the last row's position is
    // Lk - 1): it is the causal call, and runs as one, bit for bit
    r->window = o.window >= x.Lk ? 0 : o.window;
  } else if (o.window != 0) {
    return NV_SDPA_ERR_INVALID;
  }
  if (mask_kind == NV_SDPA_MASK_ADD) {
    const int64_t mb = o.add_mask_b ? o.add_mask_b : 1, mh = o.add_mask_h ? o.add_mask_h : 1;
    if ((mb != 1 && mb != x.B) || (mh != 1 && mh != x.Hq)) return NV_SDPA_ERR_INVALID;
    int64_t t;
    if (!mul_ok(x.Lq, x.Lk, &t) || !mul_ok(t, x.Hq, &t) || !mul_ok(t, x.B, &t)) return NV_SDPA_ERR_INVALID;
    r->amask = o.add_mask;
    r->am_sh = mh == 1 ? 0 : x.Lq * x.Lk;
    r->am_sb = mb == 1 ? 0 : mh * x.Lq * x.Lk;
  } else if (o.add_mask || o.add_mask_b || o.add_mask_h) {
    return NV_SDPA_ERR_INVALID;
  }
  bool qc, kc, vc, oc;
  int st;
  if ((st = resolve_strides(o.q_strides, x.B, x.Hq, x.Lq, x.d, dtype, r->qs, &qc)) != NV_SDPA_OK) return st;
  if ((st = resolve_strides(o.k_strides, x.B, x.Hkv, x.Lk, x.d, dtype, r->ks, &kc)) != NV_SDPA_OK) return st;
  if ((st = resolve_strides(o.v_strides, x.B, x.Hkv, x.Lk, x.dv, dtype, r->vs, &vc)) != NV_SDPA_OK) return st;
  if ((st = resolve_strides(o.out_strides, x.B, x.Hq, x.Lq, x.dv, dtype, r->os, &oc)) != NV_SDPA_OK) return st;
  r->qo_packed = qc && oc;
  return NV_SDPA_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// What the router needs to know about one call beyond its sizes.
struct CallShape {
  nv_sdpa_dims x;   // (paged: Lk = the table's capacity)
  int64_t span;     // keys one row tile's blocks cover: Lk, or the window's reach
  bool qo_packed;   // q and out contiguous
  bool paged;
  bool window;      // a causal sliding window is set
};

CallShape call_shape(const nv_sdpa_dims& x, const Resolved& r) {
  CallShape c{x, x.Lk, r.qo_packed, false, r.window > 0};
  // rows of one tile are at most Lq positions apart: their bands together cover at most
  // window + Lq - 1 keys
  if (r.window > 0 && r.window < x.Lk) c.span = std::min<int64_t>(x.Lk, r.window + std::max<int64_t>(x.Lq, 1) - 1);
  return c;
}

// NV_SDPA_DECODE_BLOCKS=n forces n key blocks on the tensor-core decode: a tuning and
// measurement override (unset, 0 or not a number: the planner's own choice).  Read at
// every plan, so a plan is pure only for a fixed environment.
int64_t decode_blocks_override() {
  const char* s = std::getenv("NV_SDPA_DECODE_BLOCKS");
  if (!s || !*s) return 0;
  char* end = nullptr;
  const long long v = std::strtoll(s, &end, 10);
  return (end && *end == 0 && v > 0) ? (int64_t)v : 0;
}

// The decode key split: blocks of keys_per_blk (a multiple of `quantum`) over `span`
// keys, enough of them that one batch item alone keeps 2 x (SM count) warps streaming,
// each at least 256 keys.  Depends on the head shape and the span alone, never on B.
void split_keys(int64_t span, int64_t units_per_item, int64_t quantum, int64_t* nblk_out, int64_t* kpb_out) {
  const int64_t sms = device_sm_count();
  int64_t nblk = cdiv(2 * sms, std::max<int64_t>(1, units_per_item));
  nblk = std::min(nblk, cdiv(span, 256));
  nblk = std::max<int64_t>(1, std::min(nblk, merge_max_blocks()));
  const int64_t kpb = cdiv(cdiv(span, nblk), quantum) * quantum;
  *kpb_out = kpb;
  *nblk_out = std::max<int64_t>(1, cdiv(span, kpb));
}

// The tensor-core decode's key split from the measured table: the nearest entry (head
// bucket first, then work units per batch item, then span, each by ratio) gives the keys
// per block, and the span is cut into blocks of that many keys (at most the merge pass's
// limit).
void split_keys_measured(int64_t dmax, int64_t units_per_item, int64_t span, int64_t* nblk_out,
                         int64_t* kpb_out) {
  const DecodeBlocksEntry* best = &kDecodeBlocks[0];
  double best_d = 1e300;
  for (const DecodeBlocksEntry& t : kDecodeBlocks) {
    const double dd = 4.0 * std::fabs(std::log2((double)t.dmax / (double)std::max<int64_t>(dmax, 1))) +
                      2.0 * std::fabs(std::log2((double)t.units / (double)std::max<int64_t>(units_per_item, 1))) +
                      std::fabs(std::log2((double)t.span / (double)std::max<int64_t>(span, 1)));
    if (dd < best_d) {
      best_d = dd;
      best = &t;
    }
  }
  int64_t kpb = best->keys_per_blk;
  int64_t nblk = std::max<int64_t>(1, cdiv(span, kpb));
  if (nblk > merge_max_blocks()) {
    nblk = merge_max_blocks();
    kpb = cdiv(cdiv(span, nblk), 64) * 64;
    nblk = cdiv(span, kpb);
  }
  *nblk_out = nblk;
  *kpb_out = kpb;
}

// The router.  Pure for a given device: depends on its arguments and the current
// device's SM count only.  The key-block count depends on the span of keys and the
// per-batch-item work (Hkv x row tiles), never on B, so that a batch item gets the bits
// of the same item run alone.
int make_plan(const CallShape& cs, int mask_kind, int has_sinks, int dtype, nv_sdpa_plan_t* pl) {
  (void)has_sinks;
  const nv_sdpa_dims& x = cs.x;
  std::memset(pl, 0, sizeof(*pl));
  pl->nblk = 1;
  if (x.B == 0 || x.Hq == 0 || x.Lq == 0) {
    pl->path = NV_SDPA_PATH_NOOP;
    pl->kernel = NV_SDPA_KERNEL_NONE;
    return NV_SDPA_OK;
  }
  const int64_t g = x.Hq / x.Hkv, G = g * x.Lq;
  if (x.Lk == 0) {
    pl->path = NV_SDPA_PATH_NO_KEYS;
    pl->kernel = NV_SDPA_KERNEL_FILL;
    pl->grid = 1;
    pl->launches = 1;
    return NV_SDPA_OK;
  }
  pl->path = x.Lq > 8 ? NV_SDPA_PATH_PREFILL : NV_SDPA_PATH_DECODE;
  if (cs.paged && pl->path != NV_SDPA_PATH_DECODE) return NV_SDPA_ERR_UNSUPPORTED;
  // the tensor-core kernels index keys and rows in 32 bits (as TMA coordinates are)
  const bool fits32 = x.Lk < (int64_t(1) << 31) - 1024 && G < (int64_t(1) << 31) - 1024;
  if (!fits32 && dtype != NV_SDPA_F32) return NV_SDPA_ERR_UNSUPPORTED;
  if (pl->path == NV_SDPA_PATH_PREFILL && prefill_tc_supported(dtype, x.d, x.dv)) {
    // tcgen05 kernel: one CTA per 128 or 256 rows of one KV head, all keys (no split)
    const PrefillGeom geo =
        prefill_tc_geometry(x.B, x.Hkv, g, x.Lq, x.d, x.dv, cs.qo_packed, mask_kind == NV_SDPA_MASK_ADD, 0);
    pl->kernel = NV_SDPA_KERNEL_PREFILL_TC;
    pl->rows_per_cta = 128 * geo.nq;
    pl->keys_per_blk = x.Lk;
    if (geo.grid > 0x7fffffff || geo.n_it > 0x7fffffff / 128) return NV_SDPA_ERR_UNSUPPORTED;
    pl->grid = geo.grid;
    pl->launches = 1;
    if (mask_kind == NV_SDPA_MASK_BOOL) {  // bit-packed copy of the mask
      pl->launches = 2;
      pl->scratch_bytes = x.Lq * (int64_t)prefill_tc_mask_words(x.Lk) * 4;
    }
    return NV_SDPA_OK;
  }
  if (pl->path == NV_SDPA_PATH_DECODE && (G > decode_mma_rows_per_warp() || x.d > 128 || x.dv > 128) &&
      cs.qo_packed && !cs.paged &&
      !cs.window && (mask_kind == NV_SDPA_MASK_NONE || mask_kind == NV_SDPA_MASK_CAUSAL) &&
      prefill_tc_supported(dtype, x.d, x.dv)) {
    // More query rows per KV head than one mma.sync row tile (g x Lq > 16), or heads
    // wider than 128: the tcgen05 prefill kernel, split over key blocks, reads each KV
    // head's keys once for up to 128 rows (the mma.sync decode kernel would stream them
    // once per 16 rows, and its products, not HBM, would bound it; for wide heads its
    // accumulators overflow the registers).  Blocks of whole 128-key tiles, cut from key 0,
    // sized from the keys and the head count alone (never B): as many as fill the CTA
    // slots (two per SM for heads up to 128) once for an 8-sequence batch, at least 8
    // tiles each.  (Measured, 8 x 32/4 heads x 8 queries x 32769 keys, f16: 9 blocks
    // 4846 GB/s, 19 blocks 4435, 33 blocks 3890.)
    pl->kernel = NV_SDPA_KERNEL_DECODE_TC;
    pl->rows_per_cta = 128;
    const int64_t n_rt = cdiv(G, 128), tiles = cdiv(x.Lk, 128);
    const int64_t slots = (x.d <= 128 && x.dv <= 128 ? 2 : 1) * (int64_t)device_sm_count();
    const int64_t target = std::max<int64_t>(1, slots / (8 * x.Hkv * n_rt));
    int64_t blk_tiles = std::max<int64_t>(8, cdiv(tiles, target));
    if (const int64_t forced = decode_blocks_override())
      blk_tiles = cdiv(tiles, std::max<int64_t>(1, std::min(forced, tiles)));
    blk_tiles = std::max<int64_t>(blk_tiles, cdiv(tiles, merge_max_blocks()));
    pl->keys_per_blk = blk_tiles * 128;
    pl->nblk = cdiv(tiles, blk_tiles);
    int64_t grid;
    if (!mul_ok(x.B * x.Hkv, n_rt, &grid) || !mul_ok(grid, pl->nblk, &grid) || grid > 0x7fffffff)
      return NV_SDPA_ERR_UNSUPPORTED;
    pl->grid = grid;
    pl->launches = pl->nblk > 1 ? 2 : 1;
    if (pl->nblk > 1) {
      const int64_t rows = x.B * x.Hq * x.Lq;
      if (rows > 0x7fffffff) return NV_SDPA_ERR_UNSUPPORTED;  // the merge grid: one CTA per row
      pl->scratch_bytes = cdiv(rows * pl->nblk * x.dv * 4, 256) * 256 + rows * pl->nblk * 2 * 4;
    }
    return NV_SDPA_OK;
  }
  if (pl->path == NV_SDPA_PATH_DECODE && decode_mma_supported(dtype, x.d, x.dv)) {
    // Tensor-core decode.  The keys of each KV head are cut into blocks that depend on
    // the head shape and the span alone, never on B: their size comes from the table of
    // rates measured on a GB300 (decode_blocks_table.h).  Every block's partial is computed
    // the same way whichever warp computes it, so a batch item gets the bits it would get
    // alone.  How many warps share a (b, KV head, 16-row tile)'s blocks (each walking a
    // contiguous run of them) is free, and is chosen so that all warps run as one wave:
    // fewer, longer streams read K and V best (measured: one wave at 85-95 % of the slots
    // beats two full waves, and far beats eight).
    pl->kernel = NV_SDPA_KERNEL_DECODE_MMA;
    pl->rows_per_cta = decode_mma_rows_per_warp();
    const int64_t rc = cdiv(G, pl->rows_per_cta);
    split_keys_measured(std::max(x.d, x.dv), x.Hkv * rc, cs.span, &pl->nblk, &pl->keys_per_blk);
    if (const int64_t forced = decode_blocks_override()) {
      const int64_t nb = std::max<int64_t>(1, std::min(forced, std::min(cdiv(cs.span, 64), merge_max_blocks())));
      pl->keys_per_blk = cdiv(cdiv(cs.span, nb), 64) * 64;
      pl->nblk = cdiv(cs.span, pl->keys_per_blk);
    }
    int64_t units, warp_units;
    if (!mul_ok(x.B * x.Hkv, rc, &units) || !mul_ok(units, decode_spans(x, pl->nblk), &warp_units))
      return NV_SDPA_ERR_UNSUPPORTED;
    const int64_t grid = decode_mma_grid(warp_units, x.d, x.dv);
    if (grid > 0x7fffffff) return NV_SDPA_ERR_UNSUPPORTED;
    pl->grid = grid;
    pl->launches = pl->nblk > 1 ? 2 : 1;
    if (pl->nblk > 1) {
      const int64_t rows = x.B * x.Hq * x.Lq;
      if (rows > 0x7fffffff) return NV_SDPA_ERR_UNSUPPORTED;  // the merge grid: one CTA per row
      pl->scratch_bytes = cdiv(rows * pl->nblk * x.dv * 4, 256) * 256 + rows * pl->nblk * 2 * 4;
    }
    return NV_SDPA_OK;
  }
  // FP32-FMA tiled kernel, split over key blocks when one CTA per row tile would leave
  // most SMs idle.
  pl->kernel = NV_SDPA_KERNEL_TILED_SIMT;
  pl->rows_per_cta = tiled_simt_rows_per_cta();
  const int64_t row_tiles = cdiv(G, pl->rows_per_cta);
  split_keys(cs.span, x.Hkv * row_tiles, 128, &pl->nblk, &pl->keys_per_blk);
  int64_t grid;
  if (!mul_ok(x.B * x.Hkv, row_tiles, &grid) || !mul_ok(grid, pl->nblk, &grid) || grid > 0x7fffffff)
    return NV_SDPA_ERR_UNSUPPORTED;
  pl->grid = grid;
  pl->launches = pl->nblk > 1 ? 2 : 1;
  if (pl->nblk > 1) {
    const int64_t rows = x.B * x.Hq * x.Lq;
    if (rows > 0x7fffffff) return NV_SDPA_ERR_UNSUPPORTED;  // the merge grid: one CTA per row
    const int64_t o_bytes = cdiv(rows * pl->nblk * x.dv * 4, 256) * 256;
    pl->scratch_bytes = o_bytes + rows * pl->nblk * 2 * 4;
  }
  return NV_SDPA_OK;
}

uint32_t* status_ptr_for_current_device(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  uint32_t* cached = g_status_ptr[dev].load();
  if (!cached) {
    void* ptr = nullptr;
    *err = cudaGetSymbolAddress(&ptr, g_status);
    if (*err != cudaSuccess) return nullptr;
    cached = static_cast<uint32_t*>(ptr);
    g_status_ptr[dev].store(cached);
  }
  return cached;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace nvsdpa

using namespace nvsdpa;

NV_SDPA_API int nv_sdpa_abi_version(void) { return NV_SDPA_ABI_VERSION; }

NV_SDPA_API const char* nv_sdpa_status_string(int s) {
  switch (s) {
    case NV_SDPA_OK: return "ok";
    case NV_SDPA_ERR_INVALID: return "invalid argument";
    case NV_SDPA_ERR_UNSUPPORTED: return "unsupported head size, alignment or launch size";
    case NV_SDPA_ERR_CUDA: return "CUDA runtime error";
    case NV_SDPA_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    default: return "unknown status";
  }
}

namespace nvsdpa {
namespace {
// Every check of a (non-paged) call that needs no device pointer; on success *r holds the
// resolved options and *cs the router's view of the call.  The entry points without
// options take no additive mask.
int check_call(const nv_sdpa_dims* dims, int mask_kind, int dtype, const nv_sdpa_options* opt, Resolved* r,
               CallShape* cs) {
  int st = check_dims(dims, mask_kind, dtype);
  if (st != NV_SDPA_OK) return st;
  if (mask_kind == NV_SDPA_MASK_ADD && (!opt || !opt->add_mask)) return NV_SDPA_ERR_INVALID;
  st = resolve_options(*dims, mask_kind, dtype, opt, r);
  if (st != NV_SDPA_OK) return st;
  *cs = call_shape(*dims, *r);
  return NV_SDPA_OK;
}
}  // namespace
}  // namespace nvsdpa

NV_SDPA_API int nv_sdpa_plan_ex(const nv_sdpa_dims* dims, int mask_kind, int has_sinks, int dtype,
                                const nv_sdpa_options* opt, nv_sdpa_plan_t* plan) {
  if (!plan) return NV_SDPA_ERR_INVALID;
  Resolved r;
  CallShape cs;
  int st = check_call(dims, mask_kind, dtype, opt, &r, &cs);
  if (st != NV_SDPA_OK) return st;
  return make_plan(cs, mask_kind, has_sinks, dtype, plan);
}

NV_SDPA_API int nv_sdpa_plan(const nv_sdpa_dims* dims, int mask_kind, int has_sinks, int dtype,
                             nv_sdpa_plan_t* plan) {
  return nv_sdpa_plan_ex(dims, mask_kind, has_sinks, dtype, nullptr, plan);
}

NV_SDPA_API int nv_sdpa_set_wait_limit(uint64_t spins) {
  g_wait_limit.store(spins);
  return NV_SDPA_OK;
}

namespace nvsdpa {
namespace {

// Launch parameters common to every call: sizes, the split, the scale and the wait budget.
void fill_common(Params* p, const nv_sdpa_dims& x, const nv_sdpa_plan_t& pl, int mask_kind, const void* sinks,
                 float scale) {
  p->B = x.B; p->Hq = x.Hq; p->Hkv = x.Hkv; p->Lq = x.Lq; p->Lk = x.Lk; p->d = x.d; p->dv = x.dv;
  p->g = x.Hq / x.Hkv; p->G = p->g * x.Lq;
  p->nblk = pl.nblk; p->keys_per_blk = pl.keys_per_blk;
  p->row_tiles = pl.rows_per_cta ? (p->G + pl.rows_per_cta - 1) / pl.rows_per_cta : 1;
  p->spans = pl.kernel == NV_SDPA_KERNEL_DECODE_MMA ? decode_spans(x, pl.nblk) : 1;
  p->mask_kind = mask_kind;
  p->sinks = sinks;
  p->has_sinks = sinks != nullptr;
  p->scale = scale;
  p->scale_log2 = (float)((double)scale * 1.4426950408889634);
  const uint64_t wl = g_wait_limit.load();
  p->wait_limit = wl ? wl : kDefaultWaitLimit;
}

// Everything nv_sdpa_ex(), nv_sdpa() and nv_sdpa_noalloc() check before launching, and the
// launch parameters of the call's plan.  Returns NV_SDPA_OK (with *pl and *p filled) or the
// status to return; nothing has been launched or allocated either way.
int prepare_call(const void* q, const void* k, const void* v, const nv_sdpa_dims* dims, int mask_kind,
                 const uint8_t* bool_mask, const void* sinks, float scale, const nv_sdpa_options* opt, void* out,
                 float* lse, int dtype, nv_sdpa_plan_t* pl, Params* p) {
  Resolved r;
  CallShape cs;
  int st = check_call(dims, mask_kind, dtype, opt, &r, &cs);
  if (st != NV_SDPA_OK) return st;
  if (!std::isfinite(scale)) return NV_SDPA_ERR_INVALID;
  const nv_sdpa_dims& x = *dims;
  st = make_plan(cs, mask_kind, sinks != nullptr, dtype, pl);
  if (st != NV_SDPA_OK) return st;
  if (pl->path == NV_SDPA_PATH_NOOP) return NV_SDPA_OK;
  // pointers: required ones present and aligned
  const int64_t e = elt_bytes(dtype);
  if (!out || !aligned(out, 16)) return NV_SDPA_ERR_INVALID;
  if (lse && !aligned(lse, 4)) return NV_SDPA_ERR_INVALID;
  if (sinks && !aligned(sinks, (uintptr_t)e)) return NV_SDPA_ERR_INVALID;
  if (pl->path != NV_SDPA_PATH_NO_KEYS) {
    if (!q || !k || !v || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return NV_SDPA_ERR_INVALID;
    if (mask_kind == NV_SDPA_MASK_BOOL && !bool_mask) return NV_SDPA_ERR_INVALID;
    if (mask_kind == NV_SDPA_MASK_ADD && !aligned(r.amask, 16)) return NV_SDPA_ERR_INVALID;
  }
  *p = Params{};
  p->q = q; p->k = k; p->v = v;
  p->mask = mask_kind == NV_SDPA_MASK_BOOL ? bool_mask : nullptr;
  p->out = out; p->lse = lse;
  fill_common(p, x, *pl, mask_kind, sinks, scale);
  p->q_sb = r.qs[0]; p->q_sh = r.qs[1]; p->q_sl = r.qs[2];
  p->k_sb = r.ks[0]; p->k_sh = r.ks[1]; p->k_sl = r.ks[2];
  p->v_sb = r.vs[0]; p->v_sh = r.vs[1]; p->v_sl = r.vs[2];
  p->o_sb = r.os[0]; p->o_sh = r.os[1]; p->o_sl = r.os[2];
  p->qo_packed = r.qo_packed ? 1 : 0;
  p->window = r.window;
  p->amask = r.amask;
  p->am_sb = r.am_sb;
  p->am_sh = r.am_sh;
  return NV_SDPA_OK;
}

// Launches the kernels of a prepared call on `cs`.  `scratch` holds pl.scratch_bytes
// (the split-KV partials, or the bit-packed boolean mask) or is null when none is needed.
cudaError_t launch_plan(int dtype, const nv_sdpa_plan_t& pl, Params& p, void* scratch, cudaStream_t cs) {
  cudaError_t ce;
  p.status = status_ptr_for_current_device(&ce);
  if (!p.status) return ce != cudaSuccess ? ce : cudaErrorUnknown;
  if (pl.path == NV_SDPA_PATH_NO_KEYS) return launch_fill_no_keys(dtype, p, cs);
  if (scratch) {
    const int64_t rows = p.B * p.Hq * p.Lq;
    const int64_t o_bytes = (rows * pl.nblk * p.dv * 4 + 255) / 256 * 256;
    p.part_o = static_cast<float*>(scratch);
    p.part_ml = reinterpret_cast<float*>(static_cast<char*>(scratch) + o_bytes);
  }
  if (pl.kernel == NV_SDPA_KERNEL_PREFILL_TC)
    return launch_prefill_tc(dtype, p, static_cast<uint32_t*>(scratch), false, cs);
  if (pl.kernel == NV_SDPA_KERNEL_DECODE_TC) {
    ce = launch_prefill_tc(dtype, p, nullptr, true, cs);
  } else if (pl.kernel == NV_SDPA_KERNEL_DECODE_MMA) {
    ce = launch_decode_mma(dtype, p, cs);
  } else {
    ce = launch_tiled_simt(dtype, p, cs);
  }
  if (ce == cudaSuccess && pl.nblk > 1) ce = launch_merge(dtype, p, cs);
  return ce;
}

}  // namespace
}  // namespace nvsdpa

namespace nvsdpa {
namespace {
// Runs a prepared call with its scratch from the library's pool on `stream`.  While the
// stream is being captured into a CUDA graph the scratch comes from cudaMallocAsync
// instead, which capture records as the graph's own allocation and free nodes (the
// library's pool is not one a graph can allocate from).
int run_pooled(int dtype, const nv_sdpa_plan_t& pl, Params& p, void* stream) {
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  if (pl.scratch_bytes) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(cs, &cap) != cudaSuccess) return NV_SDPA_ERR_CUDA;
    const cudaError_t ae = cap == cudaStreamCaptureStatusActive
                               ? cudaMallocAsync(&scratch, (size_t)pl.scratch_bytes, cs)
                               : pool_alloc(&scratch, (size_t)pl.scratch_bytes, cs);
    if (ae != cudaSuccess) return NV_SDPA_ERR_CUDA;
  }
  cudaError_t ce = launch_plan(dtype, pl, p, scratch, cs);
  if (scratch) {
    cudaError_t fe = cudaFreeAsync(scratch, cs);
    if (ce == cudaSuccess) ce = fe;
  }
  return ce == cudaSuccess ? NV_SDPA_OK : NV_SDPA_ERR_CUDA;
}
}  // namespace
}  // namespace nvsdpa

NV_SDPA_API int nv_sdpa_ex(const void* q, const void* k, const void* v, const nv_sdpa_dims* dims,
                           int mask_kind, const uint8_t* bool_mask, const void* sinks, float scale,
                           const nv_sdpa_options* opt, void* out, float* lse, int dtype, void* stream) {
  nv_sdpa_plan_t pl;
  Params p;
  int st = prepare_call(q, k, v, dims, mask_kind, bool_mask, sinks, scale, opt, out, lse, dtype, &pl, &p);
  if (st != NV_SDPA_OK || pl.path == NV_SDPA_PATH_NOOP) return st;
  return run_pooled(dtype, pl, p, stream);
}

NV_SDPA_API int nv_sdpa(const void* q, const void* k, const void* v, const nv_sdpa_dims* dims,
                        int mask_kind, const uint8_t* bool_mask, const void* sinks, float scale,
                        void* out, float* lse, int dtype, void* stream) {
  return nv_sdpa_ex(q, k, v, dims, mask_kind, bool_mask, sinks, scale, nullptr, out, lse, dtype, stream);
}

namespace nvsdpa {
namespace {
// Checks of a paged call that need no device pointer; fills the router's view (Lk = the
// table's capacity).
int check_paged(const nv_sdpa_paged_dims* pd, int mask_kind, int has_window, int64_t window, int dtype,
                nv_sdpa_dims* x, CallShape* cs) {
  if (!pd) return NV_SDPA_ERR_INVALID;
  if (mask_kind != NV_SDPA_MASK_NONE && mask_kind != NV_SDPA_MASK_CAUSAL) return NV_SDPA_ERR_INVALID;
  if (has_window != 0 && has_window != 1) return NV_SDPA_ERR_INVALID;
  if (has_window && (window < 1 || mask_kind != NV_SDPA_MASK_CAUSAL)) return NV_SDPA_ERR_INVALID;
  if (pd->num_blocks < 1 || pd->block_size < 1 || pd->max_blocks < 1) return NV_SDPA_ERR_INVALID;
  int64_t cap, t;
  if (!mul_ok(pd->max_blocks, pd->block_size, &cap) || cap > 0x7fffffff) return NV_SDPA_ERR_INVALID;
  if (!mul_ok(pd->B, pd->max_blocks, &t)) return NV_SDPA_ERR_INVALID;
  const int64_t e = elt_bytes(dtype);
  if (pd->Hkv < 1 || !mul_ok(pd->num_blocks, pd->Hkv, &t) || !mul_ok(t, pd->block_size, &t) ||
      !mul_ok(t, std::max(pd->d, pd->dv), &t) || !mul_ok(t, e, &t))
    return NV_SDPA_ERR_INVALID;
  *x = nv_sdpa_dims{pd->B, pd->Hq, pd->Hkv, pd->Lq, cap, pd->d, pd->dv};
  int st = check_dims(x, mask_kind, dtype);
  if (st != NV_SDPA_OK) return st;
  if (x->Lq > 8) return NV_SDPA_ERR_UNSUPPORTED;  // paged caches serve the decode path
  cs->x = *x;
  cs->span = cap;
  // (+ one key tile: paged tiles start on a tile boundary at or before the band)
  if (has_window && window < cap)
    cs->span = std::min<int64_t>(cap, window + std::max<int64_t>(x->Lq, 1) - 1 + decode_mma_key_tile());
  cs->qo_packed = true;
  cs->paged = true;
  return NV_SDPA_OK;
}
}  // namespace
}  // namespace nvsdpa

NV_SDPA_API int nv_sdpa_paged_plan(const nv_sdpa_paged_dims* dims, int mask_kind, int has_window, int64_t window,
                                   int has_sinks, int dtype, nv_sdpa_plan_t* plan) {
  if (!plan) return NV_SDPA_ERR_INVALID;
  nv_sdpa_dims x;
  CallShape cs;
  int st = check_paged(dims, mask_kind, has_window, window, dtype, &x, &cs);
  if (st != NV_SDPA_OK) return st;
  return make_plan(cs, mask_kind, has_sinks, dtype, plan);
}

NV_SDPA_API int nv_sdpa_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                              const int32_t* seq_lens, const nv_sdpa_paged_dims* dims, int mask_kind,
                              int has_window, int64_t window, const void* sinks, float scale, void* out,
                              float* lse, int dtype, void* stream) {
  nv_sdpa_dims x;
  CallShape cs;
  int st = check_paged(dims, mask_kind, has_window, window, dtype, &x, &cs);
  if (st != NV_SDPA_OK) return st;
  if (!std::isfinite(scale)) return NV_SDPA_ERR_INVALID;
  nv_sdpa_plan_t pl;
  st = make_plan(cs, mask_kind, sinks != nullptr, dtype, &pl);
  if (st != NV_SDPA_OK || pl.path == NV_SDPA_PATH_NOOP) return st;
  const int64_t e = elt_bytes(dtype);
  if (!q || !k_cache || !v_cache || !out || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(out, 16))
    return NV_SDPA_ERR_INVALID;
  if (!block_table || !seq_lens || !aligned(block_table, 4) || !aligned(seq_lens, 4)) return NV_SDPA_ERR_INVALID;
  if (lse && !aligned(lse, 4)) return NV_SDPA_ERR_INVALID;
  if (sinks && !aligned(sinks, (uintptr_t)e)) return NV_SDPA_ERR_INVALID;
  Params p{};
  p.q = q; p.k = k_cache; p.v = v_cache;
  p.out = out; p.lse = lse;
  fill_common(&p, x, pl, mask_kind, sinks, scale);
  p.q_sl = x.d; p.q_sh = x.Lq * x.d; p.q_sb = x.Hq * x.Lq * x.d;
  p.o_sl = x.dv; p.o_sh = x.Lq * x.dv; p.o_sb = x.Hq * x.Lq * x.dv;
  p.qo_packed = 1;
  p.window = has_window ? window : 0;
  p.paged = 1;
  p.table = block_table;
  p.lens = seq_lens;
  p.page = dims->block_size;
  p.max_pages = dims->max_blocks;
  p.num_pages = dims->num_blocks;
  return run_pooled(dtype, pl, p, stream);
}

NV_SDPA_API int nv_sdpa_device_status(void* stream, uint32_t* detail) {
  cudaError_t ce = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return NV_SDPA_ERR_CUDA;
  uint32_t w = 0;
  ce = cudaMemcpyFromSymbol(&w, g_status, sizeof(w));
  if (ce != cudaSuccess) return NV_SDPA_ERR_CUDA;
  if (w) {
    const uint32_t zero = 0;
    ce = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
    if (ce != cudaSuccess) return NV_SDPA_ERR_CUDA;
  }
  if (detail) *detail = w;
  if (!w) return NV_SDPA_OK;
  if (w & kStatBadConfig) return NV_SDPA_ERR_UNSUPPORTED;
  return NV_SDPA_ERR_DEVICE_TIMEOUT;
}

namespace nvsdpa {
namespace {

// Internal streams of the host-buffer entry point, one set per device, created on first
// use and kept for the life of the process: copies in, attention, copies out.
struct HostCopyStreams {
  cudaStream_t h2d = nullptr, d2h = nullptr, comp = nullptr;
};
std::mutex g_copy_streams_mu;
HostCopyStreams g_copy_streams[kMaxDevices];
cudaError_t copy_streams_for_current_device(HostCopyStreams* out) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return ce;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_copy_streams_mu);
  HostCopyStreams& s = g_copy_streams[dev];
  if (!s.h2d && (ce = cudaStreamCreateWithFlags(&s.h2d, cudaStreamNonBlocking)) != cudaSuccess) return ce;
  if (!s.d2h && (ce = cudaStreamCreateWithFlags(&s.d2h, cudaStreamNonBlocking)) != cudaSuccess) return ce;
  if (!s.comp && (ce = cudaStreamCreateWithFlags(&s.comp, cudaStreamNonBlocking)) != cudaSuccess) return ce;
  *out = s;
  return cudaSuccess;
}
// A run of the host-buffer pipeline: batch items [b0, b0 + nb), and within them KV heads
// [h0, h0 + nh) (nb > 1 only with every KV head).
struct HostChunk {
  int64_t b0, nb, h0, nh;
};

// How a host-buffer call is cut.  The (batch item, KV head) units of the tensor-core
// prefill are computed independently (no key split, no cross-unit reduction) and each
// unit's rows of q, k, v, out and lse are contiguous, so a run of units is one call on
// contiguous sub-buffers that gives the same bits.  A large call is cut into up to 8
// runs of at least 12 MiB of inputs, so that copies in, attention and copies out of
// different runs overlap (measured with the 2x32/8 heads, 4096-position causal prefill,
// 96 MiB in: 1.12 ms per call in one piece, 1.01 ms in 2 runs, 0.91 ms in 4, 0.87 ms in
// 6, 0.86 ms in 8); every other case is one run.
std::vector<HostChunk> host_chunks(const nv_sdpa_dims& x, int kernel, size_t h2d_bytes) {
  std::vector<HostChunk> out;
  const int64_t units = x.B * x.Hkv;
  int64_t n = 1;
  if (kernel == NV_SDPA_KERNEL_PREFILL_TC) {
    n = (int64_t)(h2d_bytes / (12u << 20));  // runs of at least 12 MiB of inputs, at most 8
    if (n > 8) n = 8;
    if (n < 1) n = 1;
  }
  if (n > units) n = units;
  if (n == 1) {
    out.push_back({0, x.B, 0, x.Hkv});
  } else if (x.B >= n) {
    for (int64_t c = 0; c < n; ++c) {
      const int64_t b0 = x.B * c / n, b1 = x.B * (c + 1) / n;
      if (b1 > b0) out.push_back({b0, b1 - b0, 0, x.Hkv});
    }
  } else {
    const int64_t per_b = (n + x.B - 1) / x.B;
    for (int64_t b = 0; b < x.B; ++b)
      for (int64_t c = 0; c < per_b; ++c) {
        const int64_t h0 = x.Hkv * c / per_b, h1 = x.Hkv * (c + 1) / per_b;
        if (h1 > h0) out.push_back({b, 1, h0, h1 - h0});
      }
  }
  return out;
}
}  // namespace
}  // namespace nvsdpa

NV_SDPA_API int nv_sdpa_host(const void* q, const void* k, const void* v, const nv_sdpa_dims* dims,
                             int mask_kind, const uint8_t* bool_mask, const void* sinks, float scale,
                             void* out, float* lse, int dtype, void* stream) {
  Resolved r;
  CallShape shape;
  int st = check_call(dims, mask_kind, dtype, nullptr, &r, &shape);
  if (st != NV_SDPA_OK) return st;
  if (!std::isfinite(scale)) return NV_SDPA_ERR_INVALID;
  const nv_sdpa_dims& x = *dims;
  const int64_t e = elt_bytes(dtype);
  const size_t nq = (size_t)(x.B * x.Hq * x.Lq * x.d * e), nk = (size_t)(x.B * x.Hkv * x.Lk * x.d * e),
               nv = (size_t)(x.B * x.Hkv * x.Lk * x.dv * e), no = (size_t)(x.B * x.Hq * x.Lq * x.dv * e),
               nl = (size_t)(x.B * x.Hq * x.Lq * 4), nm = (size_t)(x.Lq * x.Lk), ns = (size_t)(x.Hq * e);
  if ((nq && !q) || (nk && !k) || (nv && !v) || (no && !out)) return NV_SDPA_ERR_INVALID;
  if (mask_kind == NV_SDPA_MASK_BOOL && nm && !bool_mask) return NV_SDPA_ERR_INVALID;
  nv_sdpa_plan_t pl;
  st = make_plan(shape, mask_kind, sinks != nullptr, dtype, &pl);
  if (st != NV_SDPA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool use_mask = mask_kind == NV_SDPA_MASK_BOOL && nm;
  const bool use_lse = lse && nl;
  const bool use_sinks = sinks != nullptr;
  const std::vector<HostChunk> chunks = host_chunks(x, pl.kernel, nq + nk + nv);
  const bool piped = chunks.size() > 1;
  HostCopyStreams cps;
  cudaError_t ce = cudaSuccess;
  if (piped) {
    ce = copy_streams_for_current_device(&cps);
    if (ce != cudaSuccess) return NV_SDPA_ERR_CUDA;
  } else {
    cps.h2d = cps.d2h = cps.comp = cs;
  }
  auto up = [](size_t n) { return (n + 255) / 256 * 256; };
  const size_t oq = 0, ok = oq + up(nq), ov = ok + up(nk), oo = ov + up(nv), ol = oo + up(no),
               om = ol + up(use_lse ? nl : 0), os = om + up(use_mask ? nm : 0), total = os + up(use_sinks ? ns : 0);
  char* dbuf = nullptr;
  ce = pool_alloc(reinterpret_cast<void**>(&dbuf), total ? total : 256, cs);
  if (ce != cudaSuccess) return NV_SDPA_ERR_CUDA;
  std::vector<cudaEvent_t> ev(piped ? 2 + 2 * chunks.size() : 0, nullptr);
  for (size_t i = 0; i < ev.size() && ce == cudaSuccess; ++i)
    ce = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
  cudaEvent_t* ev_in = piped ? ev.data() + 2 : nullptr;
  cudaEvent_t* ev_done = piped ? ev.data() + 2 + chunks.size() : nullptr;
  auto record_wait = [&](cudaEvent_t evt, cudaStream_t from, cudaStream_t to) {
    if (ce == cudaSuccess) ce = cudaEventRecord(evt, from);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(to, evt, 0);
  };
  if (piped) record_wait(ev[0], cs, cps.h2d);
  auto h2d = [&](size_t off, const void* src, size_t n) {
    if (ce == cudaSuccess && n) ce = cudaMemcpyAsync(dbuf + off, src, n, cudaMemcpyHostToDevice, cps.h2d);
  };
  auto d2h = [&](void* dst, size_t off, size_t n) {
    if (ce == cudaSuccess && n) ce = cudaMemcpyAsync(dst, dbuf + off, n, cudaMemcpyDeviceToHost, cps.d2h);
  };
  const size_t uq = (size_t)(x.Hq / x.Hkv * x.Lq * x.d * e), uk = (size_t)(x.Lk * x.d * e),
               uv = (size_t)(x.Lk * x.dv * e), uo = (size_t)(x.Hq / x.Hkv * x.Lq * x.dv * e),
               ul = (size_t)(x.Hq / x.Hkv * x.Lq * 4);
  auto unit0 = [&](const HostChunk& c) { return (size_t)(c.b0 * x.Hkv + c.h0); };
  auto units = [&](const HostChunk& c) { return (size_t)(c.nb * c.nh); };
  if (use_mask) h2d(om, bool_mask, nm);
  if (use_sinks) h2d(os, sinks, ns);
  const int64_t g = x.Hq / x.Hkv;
  // Enqueue order: in(c), attention(c), out(c), ...  A copy here can hold the host
  // until it is done (measured: queueing every copy in first left the first run's
  // attention waiting for the last copy in), so each run's attention and copies out are
  // queued right behind its inputs; the copies out then overlap the next runs' copies in
  // (queued two runs later they had started late and left three runs' outputs to drain
  // after the last attention: 0.857 -> 0.787 ms for the 2x32/8x4096x128 prefill).
  auto do_in = [&](size_t c) {
    const size_t u0 = unit0(chunks[c]), nu = units(chunks[c]);
    h2d(oq + u0 * uq, static_cast<const char*>(q) + u0 * uq, nu * uq);
    h2d(ok + u0 * uk, static_cast<const char*>(k) + u0 * uk, nu * uk);
    h2d(ov + u0 * uv, static_cast<const char*>(v) + u0 * uv, nu * uv);
    if (piped) record_wait(ev_in[c], cps.h2d, cps.comp);
  };
  auto do_attn = [&](size_t c) {
    if (ce != cudaSuccess || st != NV_SDPA_OK) return;
    const HostChunk& hc = chunks[c];
    const size_t u0 = unit0(hc);
    const nv_sdpa_dims cd{hc.nb, hc.nh * g, hc.nh, x.Lq, x.Lk, x.d, x.dv};
    st = nv_sdpa(dbuf + oq + u0 * uq, dbuf + ok + u0 * uk, dbuf + ov + u0 * uv, &cd, mask_kind,
                 use_mask ? reinterpret_cast<const uint8_t*>(dbuf + om) : nullptr,
                 use_sinks ? dbuf + os + (size_t)(hc.h0 * g * e) : nullptr, scale, dbuf + oo + u0 * uo,
                 use_lse ? reinterpret_cast<float*>(dbuf + ol + u0 * ul) : nullptr, dtype, cps.comp);
    if (piped && st == NV_SDPA_OK) record_wait(ev_done[c], cps.comp, cps.d2h);
  };
  auto do_out = [&](size_t c) {
    if (st != NV_SDPA_OK) return;
    const size_t u0 = unit0(chunks[c]), nu = units(chunks[c]);
    d2h(static_cast<char*>(out) + u0 * uo, oo + u0 * uo, nu * uo);
    if (use_lse) d2h(reinterpret_cast<char*>(lse) + u0 * ul, ol + u0 * ul, nu * ul);
  };
  for (size_t c = 0; c < chunks.size(); ++c) {
    do_in(c);
    do_attn(c);
    do_out(c);
  }
  if (piped) {
    if (ce == cudaSuccess) record_wait(ev[1], cps.d2h, cs);
    if (ce != cudaSuccess || st != NV_SDPA_OK) {
      cudaStreamSynchronize(cps.h2d);
      cudaStreamSynchronize(cps.comp);
      cudaStreamSynchronize(cps.d2h);
    }
  }
  if (st == NV_SDPA_OK && ce != cudaSuccess) st = NV_SDPA_ERR_CUDA;
  cudaError_t fe = cudaFreeAsync(dbuf, cs);
  cudaError_t se = cudaStreamSynchronize(cs);
  for (cudaEvent_t evt : ev)
    if (evt) cudaEventDestroy(evt);
  if (st == NV_SDPA_OK && (fe != cudaSuccess || se != cudaSuccess)) st = NV_SDPA_ERR_CUDA;
  return st;
}

// ------------------------------------------------------------------------------------
// nv_sdpa_noalloc: the same attention call for callers that cannot allocate device
// memory.  Some callers run inside a host program whose device memory belongs to
// another allocator -- a serving runtime or framework that reserves the GPU's memory up
// front and forbids allocations outside its own pool -- or in a loop that cannot
// afford an allocation call at all.  nv_sdpa() takes its scratch (split-KV partials,
// the bit-packed boolean mask) from the library's pool; this entry point takes it from the
// fixed array below instead and allocates nothing.
//
// The array is a file-scope device variable: every GPU that loads this library holds
// NV_SDPA_STATIC_SCRATCH_BYTES of it until the process exits.  In host code its name
// is only a host-side stand-in, so its device address is looked up once per device
// (cudaGetSymbolAddress, with that device current) by the first call on that device,
// and that address is what the kernels receive.
static __device__ __align__(256) unsigned char g_nv_sdpa_static_scratch[NV_SDPA_STATIC_SCRATCH_BYTES];

namespace nvsdpa {
namespace {
std::atomic<void*> g_static_scratch_ptr[kMaxDevices];

// Device address of the static scratch on the current device (set up on first use).
void* static_scratch_for_current_device(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    if (*err == cudaSuccess) *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  void* ptr = g_static_scratch_ptr[dev].load();
  if (!ptr) {
    *err = cudaGetSymbolAddress(&ptr, g_nv_sdpa_static_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_static_scratch_ptr[dev].store(ptr);
  }
  return ptr;
}
}  // namespace
}  // namespace nvsdpa

NV_SDPA_API int nv_sdpa_noalloc(const void* q, const void* k, const void* v, const nv_sdpa_dims* dims,
                                int mask_kind, const uint8_t* bool_mask, const void* sinks, float scale,
                                void* out, float* lse, int dtype, void* stream) {
  nv_sdpa_plan_t pl;
  Params p;
  int st = prepare_call(q, k, v, dims, mask_kind, bool_mask, sinks, scale, nullptr, out, lse, dtype, &pl, &p);
  if (st != NV_SDPA_OK || pl.path == NV_SDPA_PATH_NOOP) return st;
  if (pl.scratch_bytes > (int64_t)NV_SDPA_STATIC_SCRATCH_BYTES) return NV_SDPA_ERR_UNSUPPORTED;
  cudaError_t ce = cudaSuccess;
  void* scratch = nullptr;
  if (pl.scratch_bytes) {
    scratch = static_scratch_for_current_device(&ce);
    if (!scratch) return NV_SDPA_ERR_CUDA;
  }
  // every partial (and mask word) that a later kernel of the call reads is written by an
  // earlier one, so the array's previous contents never need clearing
  ce = launch_plan(dtype, pl, p, scratch, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? NV_SDPA_OK : NV_SDPA_ERR_CUDA;
}

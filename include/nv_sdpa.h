/*
 * nv_sdpa -- fused scaled-dot-product attention forward for NVIDIA GB300 (sm_103a).
 *
 * The operation (one head; "nuvec-core 0.5.0 tests/fast.rs", test
 * attention_fallback_matches_a_direct_formula, and the fused-attention tests there):
 *
 *     out[b,h,i,:] = sum_j softmax_j(scale * <q[b,h,i,:], k[b,hk,j,:]> (+ mask)) * v[b,hk,j,:]
 *
 * with hk = h / (Hq / Hkv) (grouped-query heads; "lattice-inference 0.4.0
 * src/attention/flash.rs", kv_head_index), masked keys at a score of minus infinity,
 * rows with no visible key giving zeros ("lattice-inference 0.4.0
 * src/attention/flash.rs", tests all_masked_row_yields_zero_output_not_nan and
 * masked_key_below_finite_sentinel_does_not_dominate), and an optional per-head sink
 * logit that adds exp(sink - m) to the softmax denominator only (a sink is passed
 * per query head in the input dtype in the nuvec fused-attention tests; this library
 * reads it as a logit in score space, not multiplied by scale, with a zero value row).
 *
 * All entry points are plain C.  Device pointers are CUDA device addresses of the
 * current device; `stream` is a cudaStream_t (NULL = the legacy default stream).
 * Every call is asynchronous with respect to the host, like a kernel launch, unless
 * stated otherwise.  No entry point ever falls back to the CPU.  A call's kernels are
 * launched as programmatic dependents of the stream's previous kernel: their CTAs may
 * be placed while that kernel finishes, but each waits for it to complete (its writes
 * visible) before reading or writing any of the call's buffers, so stream order holds
 * as for plain launches.
 *
 * Layouts (all contiguous, row-major, element type = `dtype`):
 *   q    [B, Hq,  Lq, d ]        k [B, Hkv, Lk, d]        v [B, Hkv, Lk, dv]
 *   out  [B, Hq,  Lq, dv]        lse [B, Hq, Lq] float32 (natural log; may be NULL)
 *   bool_mask [Lq, Lk] uint8, nonzero = attend, shared by every batch item and head
 *   sinks [Hq] in `dtype`, or NULL
 *
 * Error behaviour: every argument check runs on the host before anything is launched;
 * a failed check returns its status and launches nothing.  Errors are returned, never
 * raised or printed.  Device-side waits are bounded: a wait that runs out records
 * NV_SDPA_ERR_DEVICE_TIMEOUT in a per-device status word that nv_sdpa_device_status()
 * reads, and the kernel returns instead of hanging.
 */
#ifndef NV_SDPA_H
#define NV_SDPA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NV_SDPA_ABI_VERSION 2

/* Element types of q, k, v, sinks and out. */
typedef enum { NV_SDPA_F32 = 0, NV_SDPA_F16 = 1, NV_SDPA_BF16 = 2 } nv_sdpa_dtype;

/* Mask kinds.  CAUSAL is aligned bottom-right: query row i sees key j iff
 * j <= i + (Lk - Lq) ("nuvec-core 0.5.0 tests/fast.rs", the direct-formula test's
 * visible count i + lk - lq + 1).  With Lq > Lk the first Lq - Lk rows see no key.
 * BOOL reads bool_mask[i * Lk + j] ("nuvec-core 0.5.0 tests/fast.rs", the boolean
 * mask of shape [lq, lk] in the fused-attention tests).  ADD (nv_sdpa_ex only) adds a
 * float mask in the input dtype to the scaled scores, softmax(scale * q.k + mask)
 * (same page, the "additive" mask amask of shape [1, hq, lq, lk]); an entry of -inf
 * hides its key like a false boolean entry. */
typedef enum {
  NV_SDPA_MASK_NONE = 0,
  NV_SDPA_MASK_CAUSAL = 1,
  NV_SDPA_MASK_BOOL = 2,
  NV_SDPA_MASK_ADD = 3
} nv_sdpa_mask;

typedef enum {
  NV_SDPA_OK = 0,
  NV_SDPA_ERR_INVALID = 1,        /* bad argument: shape, pointer, kind, overflow   */
  NV_SDPA_ERR_UNSUPPORTED = 2,    /* valid, but (d, dv) or alignment not built here  */
  NV_SDPA_ERR_CUDA = 3,           /* a CUDA runtime call failed (launch, allocation) */
  NV_SDPA_ERR_DEVICE_TIMEOUT = 4  /* a bounded device-side wait ran out              */
} nv_sdpa_status;

/* Problem sizes.  B, Hq, Lq, Lk >= 0; Hkv >= 1 with Hq % Hkv == 0; 8 <= d, dv <= 256,
 * both multiples of 8 (this covers every head size 64..256 and (96,64), (192,128)). */
typedef struct {
  int64_t B, Hq, Hkv, Lq, Lk, d, dv;
} nv_sdpa_dims;

typedef enum {
  NV_SDPA_PATH_NOOP = 0,     /* B*Hq*Lq == 0: nothing to write                         */
  NV_SDPA_PATH_NO_KEYS = 1,  /* Lk == 0: out = 0, lse = sink or -inf                   */
  NV_SDPA_PATH_PREFILL = 2,  /* Lq > 8: tiled online softmax                           */
  NV_SDPA_PATH_DECODE = 3    /* Lq <= 8: split-KV pass 1 + log-sum-exp merge pass 2    */
} nv_sdpa_path;

typedef enum {
  NV_SDPA_KERNEL_NONE = 0,
  NV_SDPA_KERNEL_FILL = 1,          /* Lk == 0 rows                                     */
  NV_SDPA_KERNEL_PREFILL_TC = 2,    /* tcgen05 + TMEM + TMA prefill, f16/bf16           */
  NV_SDPA_KERNEL_TILED_SIMT = 3,    /* FP32-FMA tiled online softmax (f32; any path)    */
  NV_SDPA_KERNEL_DECODE_MMA = 4,    /* TMA-staged tensor-core decode pass 1, f16/bf16   */
  NV_SDPA_KERNEL_DECODE_TC = 5      /* decode with g*Lq > 16 rows per KV head: the      */
                                    /* tcgen05 prefill kernel split over key blocks     */
} nv_sdpa_kernel;

/* What nv_sdpa() will launch for a problem.  Pure for a given device: a function of its
 * arguments and of the current device's SM count (read once per device; 152, a GB300's,
 * when no device can be asked) -- the same answer on every call and thread, like the
 * pure attention planner of "nuvec-core 0.6.1 tests/attention_plan.rs" (plans_are_pure).
 * The batch size never changes how the keys are split. */
typedef struct {
  int32_t path;          /* nv_sdpa_path                                                */
  int32_t kernel;        /* nv_sdpa_kernel of the main (first) launch                   */
  int64_t nblk;          /* decode/SIMT: key blocks per KV head; >1 adds the merge pass */
  int64_t keys_per_blk;  /* keys each block covers                                      */
  int64_t rows_per_cta;  /* query rows of one KV head handled by one CTA                */
  int64_t grid;          /* CTAs of the main launch                                     */
  int64_t launches;      /* kernels launched by one nv_sdpa() call                      */
  int64_t scratch_bytes; /* device scratch nv_sdpa() allocates on `stream` (partials)   */
} nv_sdpa_plan_t;

/* nv_sdpa: the fused attention forward.
 *   q, k, v   device, dtype, layouts above; must be 16-byte aligned.
 *   dims      host pointer, read during the call only.
 *   mask_kind nv_sdpa_mask.  bool_mask: device [Lq, Lk] uint8 when mask_kind is BOOL,
 *             ignored otherwise.
 *   sinks     device [Hq] of dtype, or NULL for no sinks.
 *   scale     any finite float (0 and negative allowed); multiplies q.k, not the sink.
 *   out       device [B, Hq, Lq, dv] dtype, written once, rounded to nearest even from
 *             the f32 accumulator ("nuvec-core 0.5.0 tests/fast.rs",
 *             half_precision_softmax_is_precise: one rounding at the end).
 *   lse       device [B, Hq, Lq] float32 or NULL: m + ln(sum of weights incl. sink).
 *   dtype     nv_sdpa_dtype.   stream: cudaStream_t.
 * Ownership: the caller owns every buffer.  When the plan needs scratch, the call takes
 * plan.scratch_bytes from the library's own stream-ordered pool on the current device
 * (cudaMallocFromPoolAsync on `stream`) and frees it with cudaFreeAsync on the same
 * stream; the pool keeps freed blocks for later calls (at most the largest call's
 * scratch at a time).  Nothing else is allocated, nothing synchronises.
 * Graphs: while `stream` is being captured, the scratch comes from cudaMallocAsync and
 * is freed in the same capture, so the graph holds its own allocation and free nodes;
 * each replay computes what the captured call would have.  Make one call outside the
 * capture first: it sets the kernels' attributes and looks up the device status word.
 * Returns NV_SDPA_OK or an nv_sdpa_status; on error nothing was launched (INVALID,
 * UNSUPPORTED) or a launch failed (CUDA). */
int nv_sdpa(const void* q, const void* k, const void* v, const nv_sdpa_dims* dims,
            int mask_kind, const uint8_t* bool_mask, const void* sinks, float scale,
            void* out, float* lse, int dtype, void* stream);

/* nv_sdpa_plan: the plan nv_sdpa() follows for these arguments, without launching
 * anything or touching a device.  Applies exactly the checks of nv_sdpa() that do not
 * need pointers (shapes, kinds, dtype, head sizes, size overflow) and returns the same
 * status for them.  `plan` is a host pointer, written on success. */
int nv_sdpa_plan(const nv_sdpa_dims* dims, int mask_kind, int has_sinks, int dtype,
                 nv_sdpa_plan_t* plan);

/* Optional arguments of nv_sdpa_ex() / nv_sdpa_plan_ex().  Zero-initialise the struct and
 * set what is used: an all-zero struct (or a NULL pointer) is exactly nv_sdpa().
 *
 *   has_window, window  A causal sliding window ("nuvec-core 0.5.0 tests/fast.rs", band /
 *             window_mask and windows_run_fused_and_equal_the_boolean_mask): with
 *             has_window = 1, the query at absolute position p = i + Lk - Lq sees key j iff
 *             p - window < j <= p.  Needs mask_kind CAUSAL and window >= 1; anything else
 *             is NV_SDPA_ERR_INVALID (window_errors_empty_inputs_and_full_windows: a
 *             window of 0, or a window without the causal mask, is an error).  A window of
 *             at least Lk is plain causal attention, bit for bit.  Key blocks and tiles
 *             wholly outside every row's band are never read; a one-query (Lq = 1)
 *             f16/bf16 decode cuts its key blocks from the band's first key, so each row
 *             gets the bits of an unmasked call over exactly its window's keys.
 *   add_mask, add_mask_b, add_mask_h  mask_kind ADD: device pointer to the mask, dtype,
 *             contiguous [add_mask_b, add_mask_h, Lq, Lk] with add_mask_b in {1, B} and
 *             add_mask_h in {1, Hq} (a dimension of 1 is shared by every batch item / query
 *             head; 0 reads as 1).  Not multiplied by scale.  Must be NULL for other kinds.
 *   q_strides, k_strides, v_strides, out_strides  Element strides of q, k, v and out
 *             along their first three dimensions [B, H, L] (the head dimension is always
 *             contiguous, stride 1).  All three 0 = the contiguous layout.  This covers
 *             "transposed views of [B, L, H, D]" (strides {L*H*D, D, H*D}) and keys and
 *             values sliced out of a longer cache ("nuvec-core 0.5.0 tests/fast.rs",
 *             attention_kernels_match_the_fallback and the windowed-kernel tests), with
 *             no copy: the tensor-core kernels read them through stride-aware TMA tensor
 *             maps.  Strides must be >= 0; for f16/bf16 every stride must be a multiple
 *             of 8 elements (16 bytes, a TMA rule), else NV_SDPA_ERR_UNSUPPORTED.  The
 *             output must not overlap the inputs; lse stays contiguous [B, Hq, Lq]. */
typedef struct {
  int32_t has_window;
  int32_t reserved0;       /* must be 0 */
  int64_t window;
  const void* add_mask;
  int64_t add_mask_b;
  int64_t add_mask_h;
  int64_t q_strides[3];
  int64_t k_strides[3];
  int64_t v_strides[3];
  int64_t out_strides[3];
} nv_sdpa_options;

/* nv_sdpa_ex: nv_sdpa() with the options above (`opt` is a host pointer, read during the
 * call only; NULL = no options).  Same ownership, scratch and error behaviour. */
int nv_sdpa_ex(const void* q, const void* k, const void* v, const nv_sdpa_dims* dims,
               int mask_kind, const uint8_t* bool_mask, const void* sinks, float scale,
               const nv_sdpa_options* opt, void* out, float* lse, int dtype, void* stream);

/* nv_sdpa_plan_ex: nv_sdpa_plan() for nv_sdpa_ex(): the same checks (those that need no
 * device pointer) and the same status. */
int nv_sdpa_plan_ex(const nv_sdpa_dims* dims, int mask_kind, int has_sinks, int dtype,
                    const nv_sdpa_options* opt, nv_sdpa_plan_t* plan);

/* Paged key/value caches ("nuvec-core 0.5.0 tests/fast.rs", paged and
 * paged_attention_equals_contiguous_attention): sizes of nv_sdpa_paged(). */
typedef struct {
  int64_t B, Hq, Hkv, Lq, d, dv;
  int64_t num_blocks;   /* blocks in each cache, >= 1 */
  int64_t block_size;   /* key positions per block, >= 1 (a multiple of 8 for f16/bf16) */
  int64_t max_blocks;   /* columns of the block table, >= 1 */
} nv_sdpa_paged_dims;

/* nv_sdpa_paged: decode attention (Lq <= 8) over paged caches.
 *   q            device [B, Hq, Lq, d], dtype, contiguous.
 *   k_cache      device [num_blocks, Hkv, block_size, d], dtype, contiguous.
 *   v_cache      device [num_blocks, Hkv, block_size, dv], dtype, contiguous.
 *   block_table  device [B, max_blocks] int32: key j of sequence s is position
 *                j % block_size of block block_table[s, j / block_size].
 *   seq_lens     device [B] int32: sequence s has seq_lens[s] keys.
 *   mask_kind    NONE or CAUSAL (bottom-right against each sequence's own length);
 *                BOOL and ADD are NV_SDPA_ERR_INVALID, as in the pages' paged tests.
 *   has_window, window  as in nv_sdpa_options (CAUSAL only; window >= 1).  Blocks wholly
 *                before a sequence's band are never read.
 *   sinks, scale, out [B, Hq, Lq, dv], lse [B, Hq, Lq]: as in nv_sdpa().
 * The result of sequence s equals contiguous attention over its first seq_lens[s] keys
 * with the same options.  Hostile device inputs are clamped, never dereferenced out of
 * range ("nuvec-core 0.5.0 tests/fast.rs", paged_attention_clamps_hostile_tables_and_lengths):
 * a length to [0, max_blocks * block_size], a block id to [0, num_blocks - 1].  Keys past
 * a sequence's length are never read, whatever the cache holds there.  Lq > 8 is
 * NV_SDPA_ERR_UNSUPPORTED.  Scratch (split-KV partials, sized from the table's capacity)
 * comes from the library's pool on `stream`, as in nv_sdpa(). */
int nv_sdpa_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                  const int32_t* seq_lens, const nv_sdpa_paged_dims* dims, int mask_kind,
                  int has_window, int64_t window, const void* sinks, float scale, void* out,
                  float* lse, int dtype, void* stream);

/* nv_sdpa_paged_plan: the plan nv_sdpa_paged() follows (checks that need no pointer). */
int nv_sdpa_paged_plan(const nv_sdpa_paged_dims* dims, int mask_kind, int has_window, int64_t window,
                       int has_sinks, int dtype, nv_sdpa_plan_t* plan);

/* nv_sdpa_host: the same operation on HOST buffers (same layouts), for callers without
 * device memory of their own.  Takes one device block from the library's pool (as nv_sdpa
 * does its scratch), copies the inputs in, runs nv_sdpa, copies out (and lse, if not
 * NULL) back, frees, and synchronises `stream` before returning.  A large tensor-core
 * prefill (24 MiB of inputs or more) runs as a pipeline over up to 8 runs of (batch item,
 * KV head) units: copies in, attention and copies out on three internal streams of the
 * library, ordered by events, so that the copies of one run overlap the attention of
 * another; the results are the bits of the single call.  Pinned host memory makes the
 * copies fastest.  `bool_mask` and `sinks` are host pointers here too. */
int nv_sdpa_host(const void* q, const void* k, const void* v, const nv_sdpa_dims* dims,
                 int mask_kind, const uint8_t* bool_mask, const void* sinks, float scale,
                 void* out, float* lse, int dtype, void* stream);

/* nv_sdpa_noalloc: nv_sdpa() for callers that cannot allocate device memory -- e.g. a
 * host program whose GPU memory is owned by another allocator (a serving runtime or
 * framework that reserves the device up front and forbids allocations outside its
 * pool), or a loop that cannot afford an allocation call.  No counterpart on the source
 * pages: this is a deployment variant of the same operation.
 * Same arguments, layouts, results and checks as nv_sdpa().  It calls no cudaMalloc,
 * cudaMallocAsync, cudaFree or other allocating routine: the scratch a plan needs
 * (plan.scratch_bytes: split-KV partials, the bit-packed boolean mask) comes from one
 * fixed device array of NV_SDPA_STATIC_SCRATCH_BYTES that the library defines and that
 * every GPU loading the library holds until the process exits.  A call whose plan needs
 * more returns NV_SDPA_ERR_UNSUPPORTED and launches nothing (nv_sdpa_plan() tells in
 * advance).  The first call on a device looks the array's device address up
 * (cudaGetSymbolAddress) with that device current: make that first call before any
 * stream capture.  Every call on a device shares the one array, which keeps the last
 * call's contents (nothing in it needs to start at zero); calls whose kernels overlap
 * on the GPU -- on different streams, or from different host threads -- race on it and
 * must be serialised by the caller. */
#define NV_SDPA_STATIC_SCRATCH_BYTES (32u << 20)
int nv_sdpa_noalloc(const void* q, const void* k, const void* v, const nv_sdpa_dims* dims,
                    int mask_kind, const uint8_t* bool_mask, const void* sinks, float scale,
                    void* out, float* lse, int dtype, void* stream);

/* nv_sdpa_device_status: synchronises `stream`, then reads and clears the current
 * device's status word.  Returns NV_SDPA_OK, NV_SDPA_ERR_DEVICE_TIMEOUT (a bounded wait
 * in a kernel ran out; that launch's outputs are not valid), NV_SDPA_ERR_UNSUPPORTED (a
 * kernel refused a launch configuration it cannot run), or NV_SDPA_ERR_CUDA.
 * If `detail` is not NULL it receives the raw status word (which wait gave up).
 * This is how a device-side failure becomes a returned error instead of a hang or a
 * trap: the pages' kernels report invalid states as errors, never a panic ("nuvec-core
 * 0.5.0 tests/fast.rs", window_errors_empty_inputs_and_full_windows: invalid options
 * are sticky errors).  The status word's device address is cached per device, as are
 * the static scratch of nv_sdpa_noalloc and the kernels' attributes: do not use the
 * library across a cudaDeviceReset of a device it has run on. */
int nv_sdpa_device_status(void* stream, uint32_t* detail);

/* Test hook for the bounded waits: sets the iteration limit of every device-side wait
 * of later launches on this process (0 = the built-in default).  A tiny limit makes
 * the waits run out so that the timeout path can be checked without hanging anything:
 * the failure becomes NV_SDPA_ERR_DEVICE_TIMEOUT from nv_sdpa_device_status(), an error
 * and never a panic, as the pages ask of invalid states ("nuvec-core 0.5.0
 * tests/fast.rs", window_errors_empty_inputs_and_full_windows). */
int nv_sdpa_set_wait_limit(uint64_t spins);

/* A short, static, human-readable name of a status code (errors are returned as codes,
 * never raised or printed: "nuvec-core 0.6.1 tests/attention_plan.rs",
 * invalid_options_are_rejected_by_plan_and_op, where the plan and the op reject the same
 * inputs with an error). */
const char* nv_sdpa_status_string(int status);

/* NV_SDPA_ABI_VERSION of the loaded library. */
int nv_sdpa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NV_SDPA_H */

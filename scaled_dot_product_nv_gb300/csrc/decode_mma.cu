// Decode (Lq <= 8) pass 1 for f16/bf16: stream the keys of one KV head from HBM
// through TMA rings and reduce them against the (up to 16) query rows that share that
// KV head, writing one partial (m, l, o) per row and key block for the log-sum-exp merge
// (sdpa_merge_partials), or the final output when there is a single block.
//
// This is the split-KV two-pass scheme whose kernels are named in "nuvec-core 0.6.1
// tests/attention_plan.rs" (the vector 2-pass pair, one grid layer per key block); the
// arithmetic per block is the online softmax of "lattice-inference 0.4.0
// src/attention/flash.rs" (run_tiled_attention_head).  The GB300 design:
//
// * The path is bound by reading K and V once.  Every warp of a CTA works alone: it owns
//   a ring of ST stages of 16- or 32-key K and V tiles (3-D TMA, 128-byte swizzle, zero fill
//   past Lk), issues its own loads ST tiles ahead, and walks a contiguous run of key
//   blocks of one (b, KV head, 16-row tile).  With no producer warp, no consumer
//   barriers and no cross-warp merge, a block boundary costs a partial's write and
//   nothing else.
// * The key blocks depend on the head shape and Lk alone.  Each block's online softmax
//   starts afresh and runs in the same order in whichever warp takes it, so the number
//   of warps (one wave of them, whatever the batch size) changes no bit of any item.
// * The query rows (g heads x Lq, padded to 16) are the M side of mma.sync.m16n8k16
//   (f16/bf16 in, f32 accumulate): S = Q K^T over the tile's keys, the online softmax
//   on the accumulator fragments (row max over a lane quad), P re-packed in registers as
//   the A operand of O += P V with V read by ldmatrix.trans.  Tensor-core math keeps the
//   SMs far from the ALU limit that FP32 dot products would hit at 8 query rows per key.
#include <algorithm>

#include "decode_kernel.cuh"

namespace nvsdpa {

using namespace dec;

bool decode_mma_supported(int dtype, int64_t d, int64_t dv) {
  return (dtype == 1 || dtype == 2) && d % 16 == 0 && dv % 16 == 0 && dec_bucket(d, dv) >= 0;
}

int64_t decode_mma_rows_per_warp() { return kRowsDec; }
int64_t decode_mma_key_tile() { return kKTMax; }
int decode_mma_warps_per_cta(int64_t d, int64_t dv) { return dec_info(d, dv).wpc; }
int decode_mma_ctas_per_sm(int64_t d, int64_t dv) { return dec_info(d, dv).ctas_per_sm; }
size_t decode_mma_smem_bytes(int64_t d, int64_t dv) { return (size_t)dec_info(d, dv).smem; }

// Warps per CTA: the bucket's full CTA when the warps fill every SM, else fewer, so that
// a small grid spreads over the SMs instead of piling onto a few (each warp streams its
// own keys; an SM's share of the HBM stream grows with the warps it holds only up to the
// bucket's size).
int decode_mma_cta_warps(int64_t warp_units, int64_t d, int64_t dv) {
  const DecInfo di = dec_info(d, dv);
  if (!di.wpc) return 0;
  const int64_t per_sm = (warp_units + (int64_t)device_sm_count() - 1) / (int64_t)device_sm_count();
  return (int)std::max<int64_t>(1, std::min<int64_t>(di.wpc, per_sm));
}

int64_t decode_mma_grid(int64_t warp_units, int64_t d, int64_t dv) {
  const int wpc = decode_mma_cta_warps(warp_units, d, dv);
  return wpc ? (warp_units + wpc - 1) / wpc : 0;
}

cudaError_t launch_decode_mma(int dtype, const Params& p, cudaStream_t st) {
  if (p.paged) return launch_decode_paged(dtype, p, st);
  DecArgs a;
  memset(&a, 0, sizeof(a));
  a.p = p;
  const int kt = dec_info(p.d, p.dv).kt;
  if (!kt) return cudaErrorInvalidValue;
  // K and V as 4-D [B][Hkv][Lk][d] views with the caller's strides (a slice of a longer
  // cache or a transposed [B, L, H, D] layout reads in place)
  const int64_t kd[4] = {p.d, p.Lk, p.Hkv, p.B}, ks[3] = {p.k_sl, p.k_sh, p.k_sb};
  const int64_t vd[4] = {p.dv, p.Lk, p.Hkv, p.B}, vs[3] = {p.v_sl, p.v_sh, p.v_sb};
  if (!encode_tiled_16bit(&a.tmk, dtype, p.k, 4, kd, ks, kt) || !encode_tiled_16bit(&a.tmv, dtype, p.v, 4, vd, vs, kt))
    return cudaErrorInvalidValue;
  return launch_dec_kv<kKvTma>(dtype, a, st);
}

}  // namespace nvsdpa

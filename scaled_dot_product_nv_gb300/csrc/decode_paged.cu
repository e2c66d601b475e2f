// Decode pass 1 over paged key/value caches: the kernel of decode_kernel.cuh reading
// each key tile through the page table ("nuvec-core 0.5.0 tests/fast.rs", paged and
// paged_attention_equals_contiguous_attention).  With a block size that is a multiple of 8
// the tile arrives by TMA in boxes of gcd(block size, key tile) rows, each from its block;
// any other block size falls back to 16-byte copies of every key row.  Entries of the
// table and lengths out of range are clamped, never followed.
#include "decode_kernel.cuh"

namespace nvsdpa {

using namespace dec;

namespace {
int gcd_int(int a, int b) { return b ? gcd_int(b, a % b) : a; }
}  // namespace

cudaError_t launch_decode_paged(int dtype, const Params& p, cudaStream_t st) {
  DecArgs a;
  memset(&a, 0, sizeof(a));
  a.p = p;
  const int kt = dec_info(p.d, p.dv).kt;
  if (!kt) return cudaErrorInvalidValue;
  const int r = gcd_int((int)(p.page % kt), kt);  // gcd(page, key tile)
  if (p.page % 8 == 0 && r % 8 == 0) {
    // the caches as 4-D [blocks][Hkv][page][D] tensors, boxes of r rows
    const int64_t kd[4] = {p.d, p.page, p.Hkv, p.num_pages}, ks[3] = {p.d, p.page * p.d, p.Hkv * p.page * p.d};
    const int64_t vd[4] = {p.dv, p.page, p.Hkv, p.num_pages},
                  vs[3] = {p.dv, p.page * p.dv, p.Hkv * p.page * p.dv};
    if (!encode_tiled_16bit(&a.tmk, dtype, p.k, 4, kd, ks, r) || !encode_tiled_16bit(&a.tmv, dtype, p.v, 4, vd, vs, r))
      return cudaErrorInvalidValue;
    a.sub_rows = r;
    return launch_dec_kv<kKvPagedTma>(dtype, a, st);
  }
  return launch_dec_kv<kKvPagedRows>(dtype, a, st);
}

}  // namespace nvsdpa

"""Decode with more query rows per KV head than one mma.sync row tile (g x Lq > 16): the
tcgen05 prefill kernel split over key blocks of whole 128-key tiles, each block's
partial (m, l, O) merged by the log-sum-exp pass.  Parity with the oracle element by
element, one key block and several, ragged row tiles, wide heads (one-stage K/V rings),
and the bits of each batch item alone ("nuvec-core 0.5.0 tests/fast.rs",
attention_batch_items_equal_each_item_alone)."""
import numpy as np
import pytest

import workloads as W
from helpers import check_case, ensure_built, upload

pytestmark = pytest.mark.gpu


def _plan(nv, c):
    st, pl = nv.nv_sdpa_plan((c.B, c.Hq, c.Hkv, c.Lq, c.Lk, c.d, c.dv), nv.MASKS[c.mask], int(c.sinks),
                             nv.DTYPES[c.dtype])
    assert st == nv.OK
    return pl


CASES = [
    # 8 queries x 8 heads per KV head (64 rows), 33 key tiles in blocks of 8 (the last 1)
    (W.Case(2, 32, 4, 8, 4097, 128, 128, "bf16", "causal", True, None, "n0.5", seed=81, name="g8_lq8_causal"),
     True),
    # wide heads: 128-key tiles with one-stage K and V rings
    (W.Case(1, 16, 2, 4, 3000, 256, 256, "f16", "none", True, None, "u2", seed=82, name="g8_lq4_d256"), True),
    # one key block: the kernel writes the final output itself (no merge)
    (W.Case(2, 8, 2, 8, 700, 128, 128, "f16", "causal", False, None, "n0.5", seed=83, name="one_block"), False),
    # 140 rows per KV head: two row tiles, the second 12 rows; a head pair with dv < d
    (W.Case(1, 20, 1, 7, 2000, 96, 64, "bf16", "causal", True, None, "u0.25", seed=84, name="ragged_rows_d96x64"),
     True),
    # fewer keys than queries under the causal mask: the first rows see no key
    (W.Case(1, 16, 2, 8, 5, 64, 64, "bf16", "causal", True, None, "n0.5", seed=85, name="keys_lt_queries"), False),
    # one query per sequence on 256-wide heads (4 rows per KV head)
    (W.Case(2, 8, 2, 1, 5000, 256, 256, "bf16", "causal", True, None, "n0.5", seed=89, name="lq1_d256"), True),
    # 192-wide heads, a tail block of a few keys
    (W.Case(3, 12, 3, 6, 2177, 192, 192, "bf16", "causal", False, None, "n0.5", seed=86, name="d192_tail"), True),
]


@pytest.mark.parametrize("case,split", CASES, ids=[c.name for c, _ in CASES])
def test_decode_tc_parity(case, split):
    nv = ensure_built()
    pl = _plan(nv, case)
    assert pl["kernel"] == "decode_tc" and (pl["nblk"] > 1) == split, pl
    assert pl["keys_per_blk"] % 128 == 0
    check_case(case)


def test_decode_tc_full_workload_sampled():
    """The 8-query decode workload at full size (8 x 32/4 x 8 x 32769 x 128, f16, causal,
    sinks): sampled rows against the oracle."""
    nv = ensure_built()
    c = W.decode_f16_long_kv().with_(Lq=8, name="decode_lq8_full")
    assert _plan(nv, c)["kernel"] == "decode_tc"
    check_case(c, max_oracle_flops=0)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_decode_tc_items_keep_their_bits(dt):
    import torch
    nv = ensure_built()
    c = W.Case(3, 16, 2, 8, 3333, 128, 128, dt, "causal", True, None, "u0.25", seed=87)
    assert _plan(nv, c)["kernel"] == "decode_tc"
    pb, p1 = _plan(nv, c), _plan(nv, c.with_(B=1))
    assert (pb["nblk"], pb["keys_per_blk"]) == (p1["nblk"], p1["keys_per_blk"])
    x = W.make_inputs(c)
    dev = upload(c, x)
    allb, all_lse = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind="causal", scale=c.scale_f32,
                            sinks=dev["sinks"])
    for b in range(c.B):
        one, one_lse = nv.sdpa(dev["q"][b:b + 1].contiguous(), dev["k"][b:b + 1].contiguous(),
                               dev["v"][b:b + 1].contiguous(), mask_kind="causal", scale=c.scale_f32,
                               sinks=dev["sinks"])
        assert torch.equal(allb[b:b + 1].view(torch.int16), one.view(torch.int16)), b
        assert torch.equal(all_lse[b:b + 1], one_lse), b


@pytest.mark.parametrize("scale", [0.0, -0.3])
def test_decode_tc_zero_and_negative_scale(scale):
    c = W.Case(1, 16, 2, 4, 1500, 128, 128, "bf16", "causal", True, scale, "n0.5", seed=88,
               name=f"decode_tc_scale{scale}")
    nv = ensure_built()
    assert _plan(nv, c)["kernel"] == "decode_tc"
    check_case(c)

"""The merge pass of split-KV decode has two forms: one warp per query row when a row has
at most 16 key blocks, one CTA per row beyond.  Parity with the oracle on both sides of
that boundary (the key-block count forced through the planner's tuning override), for
the head widths the warp form handles in one and two 128-column groups, on the mma.sync
decode, the split tcgen05 decode and the FP32 kernel; and key blocks that some rows see
no key of (partials m = -inf, l = 0), which must weigh nothing."""
import pytest

import workloads as W
from helpers import check_case, ensure_built

pytestmark = pytest.mark.gpu

# 17408 = 16 x 1088 = 17 x 1024 keys: 16 and 17 blocks of whole 64- and 128-key tiles
CASES = [
    W.Case(2, 8, 2, 1, 17408, 128, 128, "f16", "causal", True, None, "n0.5", seed=91, name="mma_d128"),
    W.Case(2, 8, 2, 1, 17408, 96, 64, "bf16", "causal", True, None, "u0.25", seed=92, name="mma_d96x64"),
    W.Case(1, 16, 2, 8, 17408, 256, 256, "bf16", "causal", True, None, "n0.5", seed=93, name="tc_d256"),
    W.Case(1, 16, 2, 8, 17408, 192, 192, "f16", "none", False, None, "n0.5", seed=94, name="tc_d192"),
]


def _plan(nv, c):
    st, pl = nv.nv_sdpa_plan((c.B, c.Hq, c.Hkv, c.Lq, c.Lk, c.d, c.dv), nv.MASKS[c.mask], int(c.sinks),
                             nv.DTYPES[c.dtype])
    assert st == nv.OK and pl["path"] == "decode", pl
    return pl


@pytest.mark.parametrize("nblk", [16, 17])
@pytest.mark.parametrize("case", CASES, ids=[c.name for c in CASES])
def test_merge_forms_at_the_boundary(case, nblk, monkeypatch):
    monkeypatch.setenv("NV_SDPA_DECODE_BLOCKS", str(nblk))
    nv = ensure_built()
    assert _plan(nv, case)["nblk"] == nblk
    check_case(case.with_(name=f"{case.name}_nblk{nblk}"))


@pytest.mark.parametrize("lk,want_blocks", [(4000, 16), (30000, 118)])
def test_merge_forms_f32(lk, want_blocks):
    """The FP32 kernel's own key split: 16 blocks (warp form) and more (CTA form)."""
    nv = ensure_built()
    c = W.Case(1, 4, 2, 2, lk, 64, 64, "f32", "causal", True, None, "u0.25", seed=95, name=f"simt_f32_lk{lk}")
    pl = _plan(nv, c)
    assert pl["kernel"] == "tiled_simt" and pl["nblk"] == want_blocks, pl
    check_case(c)


# The last key block holds 3 keys: query rows 0..4 of 8 see none of them.
EMPTY = [
    (W.Case(2, 4, 2, 8, 1923, 128, 128, "bf16", "causal", False, None, "n0.5", seed=97, name="mma_warp_form"), 16,
     "decode_mma"),
    (W.Case(2, 4, 2, 8, 2051, 128, 128, "f16", "causal", False, None, "n0.5", seed=98, name="mma_cta_form"), 17,
     "decode_mma"),
    (W.Case(1, 16, 2, 8, 1923, 128, 128, "bf16", "causal", False, None, "n0.5", seed=99, name="tc_warp_form"), 16,
     "decode_tc"),
]


@pytest.mark.parametrize("case,nblk,kernel", EMPTY, ids=[e[0].name for e in EMPTY])
def test_merge_blocks_some_rows_cannot_see(case, nblk, kernel, monkeypatch):
    monkeypatch.setenv("NV_SDPA_DECODE_BLOCKS", str(nblk))
    nv = ensure_built()
    pl = _plan(nv, case)
    assert pl["kernel"] == kernel and pl["nblk"] == nblk and (nblk - 1) * pl["keys_per_blk"] == case.Lk - 3, pl
    check_case(case)

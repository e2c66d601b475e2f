"""The online softmax rescales O only when a row's running maximum grows by more than 2^8
(in log2 units), and the one-tile kernels then wait for the previous tile's P V before
touching O; tiles without a rescale do not wait, and the last tile always does.  Keys
whose scores climb by about one such step per key tile force a rescale on every tile, or
on every other one, and the results must still match the oracle element by element
("lattice-inference 0.4.0 src/attention/flash.rs": the tiled online softmax equals the
materialised one).  Covered: the 256-wide prefill (no mask, boolean mask, additive
mask) and the split tcgen05 decode."""
import numpy as np
import pytest

import workloads as W
from helpers import check_case, ensure_built

pytestmark = pytest.mark.gpu


def _climbing_inputs(c, pattern, seed):
    """q: 0.5 + small noise; k_j: (step_j + small noise) in every coordinate, step_j growing
    by `per_tile` every 128 keys (pattern "every") or every other 128 keys ("alternate"),
    so that the scores climb ~11.5 log2 units per climbing tile at d = 256 (scale 1/16)."""
    rng = np.random.default_rng(seed)
    dt = np.float16
    q = (0.5 + 0.05 * rng.standard_normal((c.B, c.Hq, c.Lq, c.d))).astype(dt)
    tile = np.arange(c.Lk) // 128
    climbs = tile if pattern == "every" else (tile + 1) // 2
    per_tile = 256.0 / c.d  # the same score step for narrower heads
    step = climbs * per_tile
    k = (step[None, None, :, None] + 0.05 * rng.standard_normal((c.B, c.Hkv, c.Lk, c.d))).astype(dt)
    v = rng.standard_normal((c.B, c.Hkv, c.Lk, c.dv)).astype(dt)
    sinks = rng.standard_normal(c.Hq).astype(dt) if c.sinks else None
    mask = None
    if c.mask == "bool":
        mask = (rng.random((c.Lq, c.Lk)) < 0.9).astype(np.uint8)
        r = np.arange(min(c.Lq, c.Lk))
        mask[r, r] = 1
    return dict(q=q, k=k, v=v, sinks=sinks, mask=mask)


CASES = [
    W.Case(1, 4, 2, 256, 1801, 256, 256, "f16", "none", True, None, "n0.5", name="prefill_d256"),
    W.Case(1, 4, 2, 256, 1801, 256, 256, "f16", "bool", True, None, "n0.5", name="bool_d256"),
    W.Case(2, 16, 2, 8, 4097, 128, 128, "f16", "causal", True, None, "n0.5", name="decode_tc_d128"),
]


@pytest.mark.parametrize("pattern", ["every", "alternate"])
@pytest.mark.parametrize("case", CASES, ids=[c.name for c in CASES])
def test_rescales_on_every_or_every_other_tile(case, pattern):
    nv = ensure_built()
    st, pl = nv.nv_sdpa_plan((case.B, case.Hq, case.Hkv, case.Lq, case.Lk, case.d, case.dv), nv.MASKS[case.mask],
                             int(case.sinks), nv.DTYPES[case.dtype])
    assert st == nv.OK
    assert pl["kernel"] in ("prefill_tc", "decode_tc") and pl["rows_per_cta"] == 128, pl
    x = _climbing_inputs(case, pattern, seed=sum(map(ord, case.name + pattern)))
    check_case(case, x, name=f"{case.name}_{pattern}")


@pytest.mark.parametrize("pattern", ["every", "alternate"])
def test_rescales_with_an_additive_mask(pattern):
    """The additive path (64-key tiles): the same climbing keys, plus an additive mask of
    small values with a few -inf entries."""
    import torch
    import oracle
    from helpers import TOL, assert_close, from_device, upload
    nv = ensure_built()
    c = W.Case(1, 4, 2, 256, 1801, 256, 256, "f16", "none", True, None, "n0.5", name=f"additive_{pattern}")
    x = _climbing_inputs(c, pattern, seed=77)
    rng = np.random.default_rng(78)
    am = (0.5 * rng.standard_normal((1, c.Hq, c.Lq, c.Lk))).astype(np.float16)
    am[rng.random(am.shape) < 0.05] = -np.inf
    dev = upload(c, x)
    amd = torch.from_numpy(am).cuda()
    out, lse = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind="add", scale=c.scale_f32, add_mask=amd,
                       sinks=dev["sinks"])
    torch.cuda.synchronize()
    want, wlse = oracle.sdpa(W.widen(x["q"], c.dtype), W.widen(x["k"], c.dtype), W.widen(x["v"], c.dtype),
                             mask_kind="add", scale=c.scale_f32, add_mask=W.widen(am, c.dtype),
                             sinks=W.widen(x["sinks"], c.dtype))
    assert_close(c.name + " out", from_device(out, c.dtype), want, TOL[c.dtype])
    assert_close(c.name + " lse", lse.cpu().numpy().astype(np.float64), wlse, TOL[c.dtype])

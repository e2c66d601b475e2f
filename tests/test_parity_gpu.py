"""Parity of the CUDA path with the f64 oracle, through the C ABI, on seeded inputs.

Element by element wherever the oracle finishes in seconds (sizes that still span
several tiles and ragged tails), on sampled rows at the full sizes of the workloads.
Tolerance per dtype: f32 2e-5, f16 4e-3, bf16 2e-2 of max(|want|, 1), the same for
the log-sum-exp."""
import itertools

import numpy as np
import pytest

import workloads as W
from helpers import TOL, assert_close, check_case, ensure_built, oracle_full, run_gpu, upload

pytestmark = pytest.mark.gpu


def _small_cases():
    shapes = [(64, 64), (96, 64), (128, 128), (192, 128), (256, 256), (72, 72), (80, 80)]
    heads = [(4, 2), (8, 1), (6, 6), (32, 4), (2, 1)]
    lens = [(1, 1), (1, 300), (3, 129), (8, 1000), (9, 9), (77, 141), (200, 200), (130, 2049),
            (333, 64), (64, 333)]
    out = []
    n = 0
    for dt, mk, sk in itertools.product(["f32", "f16", "bf16"], ["none", "causal", "bool"],
                                        [False, True]):
        for t in range(3):
            d, dv = shapes[n % len(shapes)]
            hq, hkv = heads[n % len(heads)]
            lq, lk = lens[n % len(lens)]
            out.append(W.Case(1 + n % 2, hq, hkv, lq, lk, d, dv, dt, mk, sk, None,
                              ["u0.25", "u2", "n0.5"][n % 3], seed=100 + n,
                              name=f"small{n:02d}_{dt}_{mk}_s{int(sk)}_d{d}x{dv}_h{hq}x{hkv}_{lq}x{lk}"))
            n += 1
    return out


SMALL = _small_cases()


@pytest.mark.parametrize("case", SMALL, ids=[c.name for c in SMALL])
def test_small_cases(case):
    check_case(case)


def test_tiny_f32_causal():
    check_case(W.tiny_f32_causal())


def test_decode_f16_long_kv_full():
    check_case(W.decode_f16_long_kv(), max_oracle_flops=1e12)


def test_prefill_f16_boolmask_sinks_full():
    check_case(W.prefill_f16_boolmask_sinks(), max_oracle_flops=1e12)


def test_prefill_bf16_gqa_sampled():
    check_case(W.prefill_bf16_gqa())


SWEEP = W.sweep_bf16()


@pytest.mark.parametrize("case", SWEEP, ids=[c.name for c in SWEEP])
def test_sweep_bf16(case):
    check_case(case, max_oracle_flops=3e9)


# ----------------------------------------------------------------------------- edge cases

@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_no_keys_gives_zeros(dt):
    for mk, sk in [("none", False), ("causal", False), ("causal", True)]:
        c = W.Case(1, 2, 2, 3, 0, 64, 64, dt, mk, sk, 0.125, seed=7)
        x = W.make_inputs(c)
        got, lse = run_gpu(c, x)
        assert got.shape == (1, 2, 3, 64) and np.all(got == 0.0)
        if sk:
            np.testing.assert_allclose(lse[0], np.broadcast_to(W.widen(x["sinks"], dt)[:, None], (2, 3)))
        else:
            assert np.all(lse == -np.inf)


def test_no_queries_is_a_noop():
    c = W.Case(1, 2, 2, 0, 9, 64, 64, "bf16", "causal", False, seed=8)
    got, lse = run_gpu(c, W.make_inputs(c))
    assert got.shape == (1, 2, 0, 64)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("lq,lk", [(20, 5), (6, 2), (300, 129)])
def test_causal_with_more_queries_than_keys(dt, lq, lk):
    for sk in [False, True]:
        c = W.Case(2, 4, 2, lq, lk, 64, 64, dt, "causal", sk, None, "n0.5", seed=9)
        got, lse = check_case(c)
        assert np.all(got[:, :, : lq - lk] == 0.0)


@pytest.mark.parametrize("dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("lq", [1, 5, 40, 200])
def test_all_masked_rows_are_zero(dt, lq):
    c = W.Case(1, 4, 2, lq, 300, 128, 128, dt, "bool", False, None, "n0.5", seed=10)
    x = W.make_inputs(c)
    x["mask"][::3] = 0  # every third row sees nothing
    got, lse = check_case(c, x)
    assert np.all(got[:, :, ::3] == 0.0) and np.all(lse[:, :, ::3] == -np.inf)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_large_group_decode(dt):
    # 32 query heads on one KV head with 8 queries each: 256 rows per KV head
    check_case(W.Case(1, 32, 1, 8, 5000, 128, 128, dt, "causal", True, None, "u2", seed=11))


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_extreme_scores_stay_finite(dt):
    # scores of +-100s: the online max must keep every exponent <= 0
    c = W.Case(1, 4, 2, 70, 900, 64, 64, dt, "none", True, 4.0, "n1", seed=12)
    check_case(c)


@pytest.mark.parametrize("d,dv", [(64, 128), (128, 64), (64, 256), (256, 64), (136, 136)])
@pytest.mark.parametrize("lq", [1, 300])
def test_head_pairs_beyond_the_listed_ones(d, dv, lq):
    """Head pairs the ABI accepts beyond the pages' list.  An output tile wider than the Q
    tile (dv > d) leaves the prefill by direct row stores instead of the TMA store; a
    136-wide head needs a ninth K-step and a third, partly filled 64-column panel."""
    c = W.Case(2, 8, 2, lq, 777, d, dv, "bf16", "causal", True, None, "n0.5", seed=15)
    check_case(c, name=f"d{d}x{dv}_lq{lq}")


WAVES = [
    # 352 work tiles of 256 rows (ragged: G = 2600); the first rows see no key at all
    W.Case(4, 16, 8, 1300, 1000, 64, 64, "bf16", "causal", True, None, "n0.5", seed=21,
           name="waves_causal_lk_lt_lq_d64"),
    # 192 tiles of two query heads' rows, heaviest first, boolean mask and sinks
    W.Case(3, 32, 8, 512, 700, 128, 128, "f16", "bool", True, None, "u2", seed=22,
           name="waves_bool_sinks_d128"),
    # 512 tiles of two query heads' rows, no mask, a head pair with dv < d
    W.Case(2, 32, 8, 2048, 2048, 96, 64, "bf16", "none", False, None, "u0.25", seed=23,
           name="waves_none_d96x64"),
    # an odd group (g = 3): 192 tiles of 256 consecutive rows, some across two heads
    W.Case(6, 12, 4, 640, 900, 128, 128, "bf16", "causal", True, None, "n0.5", seed=24,
           name="waves_causal_odd_group_d128"),
]


@pytest.mark.parametrize("case", WAVES, ids=[c.name for c in WAVES])
def test_prefill_more_work_tiles_than_sms(case):
    """More 256-row work tiles than SMs, so CTAs run in several waves, each tile on
    whichever SM frees first."""
    nv = ensure_built()
    _, pl = nv.nv_sdpa_plan((case.B, case.Hq, case.Hkv, case.Lq, case.Lk, case.d, case.dv),
                            nv.MASKS[case.mask], int(case.sinks), nv.DTYPES[case.dtype])
    assert pl["rows_per_cta"] == 256
    check_case(case)


# ----------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("lq,lk", [(300, 300), (1, 8193), (9, 777)])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_batch_items_equal_each_item_alone(lq, lk, dt):
    """"nuvec-core 0.5.0 tests/fast.rs", attention_batch_items_equal_each_item_alone:
    each batch item gets the bits of that item alone."""
    import torch
    nv = ensure_built()
    c = W.Case(3, 8, 2, lq, lk, 128, 128, dt, "causal", True, None, "u0.25", seed=13)
    x = W.make_inputs(c)
    dev = upload(c, x)
    allb, _ = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind="causal", scale=c.scale_f32,
                      sinks=dev["sinks"])
    for b in range(3):
        one, _ = nv.sdpa(dev["q"][b:b + 1].contiguous(), dev["k"][b:b + 1].contiguous(),
                         dev["v"][b:b + 1].contiguous(), mask_kind="causal", scale=c.scale_f32,
                         sinks=dev["sinks"])
        assert torch.equal(allb[b:b + 1].view(torch.int16), one.view(torch.int16)), b


def test_decode_items_keep_their_bits_when_ctas_take_runs_of_key_blocks():
    """The decode grid follows the batch size (one wave of CTAs, each walking a run of key
    blocks) while the key blocks do not: in an 8-item batch a CTA takes several blocks,
    alone one, and the item's output and log-sum-exp keep every bit."""
    import torch
    nv = ensure_built()
    c = W.decode_f16_long_kv()
    shape = (c.B, c.Hq, c.Hkv, c.Lq, c.Lk, c.d, c.dv)
    _, pl_b = nv.nv_sdpa_plan(shape, 1, 1, 1)
    _, pl_1 = nv.nv_sdpa_plan((1,) + shape[1:], 1, 1, 1)
    assert (pl_b["nblk"], pl_b["keys_per_blk"]) == (pl_1["nblk"], pl_1["keys_per_blk"])
    assert pl_b["grid"] < c.B * pl_1["grid"]  # CTAs of the batch walk runs of blocks
    x = W.make_inputs(c)
    dev = upload(c, x)
    allb, all_lse = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind=c.mask, scale=c.scale_f32,
                            sinks=dev["sinks"])
    for b in (0, 3, c.B - 1):
        one, one_lse = nv.sdpa(dev["q"][b:b + 1].contiguous(), dev["k"][b:b + 1].contiguous(),
                               dev["v"][b:b + 1].contiguous(), mask_kind=c.mask, scale=c.scale_f32,
                               sinks=dev["sinks"])
        assert torch.equal(allb[b:b + 1].view(torch.int16), one.view(torch.int16)), b
        assert torch.equal(all_lse[b:b + 1], one_lse), b


def test_run_to_run_deterministic():
    import torch
    nv = ensure_built()
    for c in [W.decode_f16_long_kv(), W.prefill_f16_boolmask_sinks()]:
        x = W.make_inputs(c)
        dev = upload(c, x)
        outs = [nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind=c.mask, scale=c.scale_f32,
                        bool_mask=dev["mask"], sinks=dev["sinks"]) for _ in range(3)]
        for o, l in outs[1:]:
            assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
            assert torch.equal(l, outs[0][1])


def test_host_buffer_entry_point_matches_device_entry_point():
    import torch
    nv = ensure_built()
    c = W.prefill_f16_boolmask_sinks().with_(Lq=200, Lk=333)
    x = W.make_inputs(c)
    dev = upload(c, x)
    o_dev, l_dev = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind=c.mask, scale=c.scale_f32,
                           bool_mask=dev["mask"], sinks=dev["sinks"])
    torch.cuda.synchronize()
    out = np.empty((c.B, c.Hq, c.Lq, c.dv), dtype=np.float16)
    lse = np.empty((c.B, c.Hq, c.Lq), dtype=np.float32)
    st = nv.nv_sdpa_host(x["q"].ctypes.data, x["k"].ctypes.data, x["v"].ctypes.data,
                         (c.B, c.Hq, c.Hkv, c.Lq, c.Lk, c.d, c.dv), 2, x["mask"].ctypes.data,
                         x["sinks"].ctypes.data, c.scale_f32, out.ctypes.data, lse.ctypes.data,
                         1, 0)
    assert st == 0
    np.testing.assert_array_equal(out, o_dev.cpu().numpy())
    np.testing.assert_array_equal(lse, l_dev.cpu().numpy())


@pytest.mark.parametrize("mask,sinks,out_pinned", [("causal", False, True), ("bool", True, True),
                                                   ("causal", False, False)])
def test_large_host_buffer_call_gives_the_device_call_bits(mask, sinks, out_pinned):
    """A large host-buffer call from pinned memory runs as a pipeline over runs of
    (batch item, KV head) units (48 MiB of inputs: 2 batch items x 2 runs of 4 KV heads)
    and gives every output and lse bit of the single device call, with the outputs in
    page-locked or in pageable memory."""
    import torch
    nv = ensure_built()
    c = W.Case(2, 32, 8, 2048, 2048, 128, 128, "bf16", mask, sinks, None, "n0.5", seed=31)
    x = W.make_inputs(c)
    dev = upload(c, x)
    o_dev, l_dev = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind=c.mask, scale=c.scale_f32,
                           bool_mask=dev["mask"], sinks=dev["sinks"])
    torch.cuda.synchronize()
    pin = {n: torch.from_numpy(np.ascontiguousarray(x[n]).view(np.int16)).pin_memory()
           for n in ("q", "k", "v")}
    hout = torch.empty((c.B, c.Hq, c.Lq, c.dv), dtype=torch.int16)
    hlse = torch.empty((c.B, c.Hq, c.Lq), dtype=torch.float32)
    if out_pinned:
        hout, hlse = hout.pin_memory(), hlse.pin_memory()
    st = nv.nv_sdpa_host(pin["q"].data_ptr(), pin["k"].data_ptr(), pin["v"].data_ptr(),
                         (c.B, c.Hq, c.Hkv, c.Lq, c.Lk, c.d, c.dv), nv.MASKS[mask],
                         x["mask"].ctypes.data if mask == "bool" else None,
                         x["sinks"].ctypes.data if sinks else None, c.scale_f32,
                         hout.data_ptr(), hlse.data_ptr(), nv.DTYPES["bf16"], 0)
    assert st == 0
    assert torch.equal(hout, o_dev.view(torch.int16).cpu())
    assert torch.equal(hlse, l_dev.cpu())


def test_lse_only_optional_and_status_clean():
    import torch
    nv = ensure_built()
    c = W.Case(1, 4, 2, 33, 100, 64, 64, "bf16", "causal", False, seed=14)
    dev = upload(c, W.make_inputs(c))
    o1, _ = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind="causal", scale=c.scale_f32)
    o2, none = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind="causal", scale=c.scale_f32,
                       want_lse=False)
    assert none is None and torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert nv.nv_sdpa_device_status(0) == (0, 0)


@pytest.mark.parametrize("case", [
    # one Q tile per CTA, 128-key tiles, long key loop (the 192/128 head)
    W.Case(1, 8, 2, 1024, 4096, 192, 128, "bf16", "none", False, None, "u2", seed=41, name="nq1_d192"),
    # two Q tiles per CTA (ping-pong), causal and unmasked
    W.Case(1, 8, 2, 2048, 4096, 128, 128, "bf16", "causal", True, None, "n0.5", seed=42, name="nq2_causal"),
    W.Case(2, 4, 4, 1000, 3000, 64, 64, "f16", "none", False, None, "n1", seed=43, name="nq2_d64"),
    # 64-key tiles (the 256 head)
    W.Case(1, 4, 1, 700, 3000, 256, 256, "f16", "causal", True, None, "n0.5", seed=44, name="bn64_d256"),
], ids=lambda c: c.name)
def test_pipeline_repeats_are_identical_and_correct(case):
    """Long key loops through every CTA variant of the tensor-core prefill, run several
    times: every run must give the same bits and match the oracle on sampled rows
    (a synchronisation race shows up as run-to-run or oracle differences)."""
    import torch
    nv = ensure_built()
    x = W.make_inputs(case)
    dev = upload(case, x)
    outs = []
    for _ in range(4):
        o, l = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind=case.mask, scale=case.scale_f32,
                       sinks=dev["sinks"])
        outs.append((o.clone(), l.clone()))
    torch.cuda.synchronize()
    assert nv.nv_sdpa_device_status(0) == (nv.OK, 0)
    for o, l in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(l, outs[0][1])
    check_case(case, x)


# ----------------------------------------------------------------------------- scales and mask bytes

def _scale_cases():
    """Every kernel under scale 0 (all scores equal: the mean of the visible V rows) and
    under negative scales (the largest raw score is then the smallest scaled one, which
    the prefill's unmasked fast path must not assume away).  The pages pass arbitrary f32
    scales ("nuvec-core 0.5.0 tests/fast.rs": 0.3 in the fused-attention tests, 0.125 in
    the window tests); here 0, -0.3 and -1/sqrt(d)."""
    base = [
        # (name, case, expected kernel, expected nblk > 1)
        ("prefill_nq2", W.Case(1, 8, 2, 300, 500, 128, 128, "bf16", "none", True, None, "n0.5", seed=61),
         "prefill_tc", False),
        ("prefill_nq2_causal", W.Case(2, 4, 2, 257, 257, 64, 64, "f16", "causal", False, None, "u2", seed=62),
         "prefill_tc", False),
        ("prefill_nq1_d256", W.Case(1, 4, 2, 200, 300, 256, 256, "f16", "none", True, None, "n0.5", seed=63),
         "prefill_tc", False),
        ("prefill_nq1_d192_bool", W.Case(1, 4, 1, 100, 700, 192, 128, "bf16", "bool", False, None, "n0.5",
                                         seed=64), "prefill_tc", False),
        ("decode_split", W.Case(2, 8, 2, 1, 3000, 128, 128, "f16", "causal", True, None, "u2", seed=65),
         "decode_mma", True),
        ("decode_one_block", W.Case(1, 4, 4, 3, 60, 64, 64, "bf16", "none", False, None, "n0.5", seed=66),
         "decode_mma", False),
        ("decode_bool", W.Case(1, 8, 2, 5, 900, 128, 128, "bf16", "bool", True, None, "n0.5", seed=67),
         "decode_mma", True),
        ("f32_prefill", W.Case(1, 4, 2, 40, 700, 64, 64, "f32", "causal", True, None, "n0.5", seed=68),
         "tiled_simt", True),
        ("f32_decode", W.Case(2, 4, 2, 1, 3000, 64, 64, "f32", "none", False, None, "u0.25", seed=69),
         "tiled_simt", True),
    ]
    out = []
    for name, c, kern, split in base:
        for sc in [0.0, -0.3, "-rsqrt"]:
            s = -1.0 / np.sqrt(c.d) if sc == "-rsqrt" else sc
            out.append((f"{name}_scale{sc}", c.with_(scale=s, name=f"{name}_scale{sc}"), kern, split))
    return out


SCALES = _scale_cases()


@pytest.mark.parametrize("name,case,kernel,split", SCALES, ids=[s[0] for s in SCALES])
def test_zero_and_negative_scales(name, case, kernel, split):
    nv = ensure_built()
    st, pl = nv.nv_sdpa_plan((case.B, case.Hq, case.Hkv, case.Lq, case.Lk, case.d, case.dv),
                             nv.MASKS[case.mask], int(case.sinks), nv.DTYPES[case.dtype])
    assert st == nv.OK and pl["kernel"] == kernel and (pl["nblk"] > 1) == split, pl
    check_case(case, name=name)


MASK_BYTES = [
    W.Case(1, 8, 2, 300, 700, 128, 128, "bf16", "bool", True, None, "n0.5", seed=71, name="prefill_nq2"),
    W.Case(1, 4, 2, 150, 333, 256, 256, "f16", "bool", False, None, "n0.5", seed=72, name="prefill_nq1"),
    W.Case(2, 8, 2, 4, 2000, 128, 128, "f16", "bool", True, None, "u2", seed=73, name="decode"),
    W.Case(1, 4, 2, 33, 400, 64, 64, "f32", "bool", False, None, "u0.25", seed=74, name="f32"),
]


@pytest.mark.parametrize("case", MASK_BYTES, ids=[c.name for c in MASK_BYTES])
def test_boolean_mask_reads_any_nonzero_byte_as_attend(case):
    """The mask is bytes, nonzero = attend: entries of 2, 128 and 255 must act like 1."""
    x = W.make_inputs(case)
    rng = np.random.RandomState(case.seed)
    x["mask"] = (x["mask"] * rng.choice(np.array([1, 2, 128, 255], dtype=np.uint8),
                                        size=x["mask"].shape)).astype(np.uint8)
    assert set(np.unique(x["mask"])) == {0, 1, 2, 128, 255}
    check_case(case, x)

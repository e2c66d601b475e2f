"""Parity of the CUDA path with the f64 oracle for the options beyond nv_sdpa(): causal
sliding windows, additive masks, strided views of q / k / v / out, and paged key/value
caches -- through the C ABI (nv_sdpa_ex, nv_sdpa_paged), element by element, with the
outputs in canary-guarded buffers.

Shapes follow the pages' own test grids ("nuvec-core 0.5.0 tests/fast.rs":
windows_run_fused_and_equal_the_boolean_mask, attention_kernels_match_the_fallback,
paged_attention_equals_contiguous_attention, paged_windows_and_sinks_equal_contiguous_attention,
paged_attention_clamps_hostile_tables_and_lengths)."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import (TOL, Guarded, assert_close, ensure_built, from_device, to_device,
                     torch_dtype)

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------------------------- plumbing

def _case(B, Hq, Hkv, Lq, Lk, d, dv, dt, mask, sinks, seed, values="n0.5", scale=None, name=""):
    return W.Case(B, Hq, Hkv, Lq, Lk, d, dv, dt, mask, sinks, scale, values, seed=seed, name=name)


def _view(stored, dt, layout, pad_seed=0):
    """A CUDA view of the [B, H, L, D] array `stored` in the given layout:
    "contig", "bhld_T" (a transposed [B, L, H, D] buffer), or "slice" (rows 5.. of a
    longer [B, H, L + 17, D] cache filled with NaN around them)."""
    import torch
    t = to_device(stored, dt)
    if layout == "contig":
        return t
    if layout == "bhld_T":
        buf = torch.empty((t.shape[0], t.shape[2], t.shape[1], t.shape[3]), dtype=t.dtype, device="cuda")
        buf.copy_(t.transpose(1, 2))
        return buf.transpose(1, 2)
    if layout == "slice":
        buf = torch.full((t.shape[0], t.shape[1], t.shape[2] + 17, t.shape[3]), float("nan"),
                         dtype=t.dtype, device="cuda")
        buf[:, :, 5:5 + t.shape[2]] = t
        return buf[:, :, 5:5 + t.shape[2]]
    raise ValueError(layout)


class _GuardedOut:
    """The output in a canary-guarded buffer, optionally as a transposed [B, L, H, D] view."""

    def __init__(self, case, transposed):
        import torch
        self.transposed = transposed
        shape = (case.B, case.Lq, case.Hq, case.dv) if transposed else (case.B, case.Hq, case.Lq, case.dv)
        self.g = Guarded(shape, torch_dtype(case.dtype))
        self.out = self.g.tensor.transpose(1, 2) if transposed else self.g.tensor
        self.glse = Guarded((case.B, case.Hq, case.Lq), torch.float32)
        self.lse = self.glse.tensor

    def check(self):
        self.g.check("out")
        self.glse.check("lse")


def run_ex(case, x, *, window=None, add_mask=None, layouts=("contig",) * 4):
    """The CUDA path through nv_sdpa_ex with the given options and layouts of q, k, v, out;
    returns (out f64, lse f64) after checking the canaries and the device status."""
    import torch
    nv = ensure_built()
    q = _view(x["q"], case.dtype, layouts[0])
    k = _view(x["k"], case.dtype, layouts[1])
    v = _view(x["v"], case.dtype, layouts[2])
    go = _GuardedOut(case, layouts[3] == "bhld_T")
    sinks = to_device(x["sinks"], case.dtype) if x["sinks"] is not None else None
    mask = to_device(x["mask"], "u8") if x["mask"] is not None else None
    am = to_device(W.to_storage(add_mask, case.dtype), case.dtype) if add_mask is not None else None
    opts = nv.make_options(window=window, add_mask=am.data_ptr() if am is not None else 0,
                           add_mask_b=am.shape[0] if am is not None else 0,
                           add_mask_h=am.shape[1] if am is not None else 0,
                           q_strides=nv._bhl_strides(q), k_strides=nv._bhl_strides(k),
                           v_strides=nv._bhl_strides(v), out_strides=nv._bhl_strides(go.out))
    st = nv.nv_sdpa_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                       (case.B, case.Hq, case.Hkv, case.Lq, case.Lk, case.d, case.dv),
                       nv.MASKS[case.mask], mask.data_ptr() if mask is not None else 0,
                       sinks.data_ptr() if sinks is not None else 0, case.scale_f32, opts,
                       go.out.data_ptr(), go.lse.data_ptr(), nv.DTYPES[case.dtype],
                       torch.cuda.current_stream().cuda_stream)
    assert st == nv.OK, nv.nv_sdpa_status_string(st)
    torch.cuda.synchronize()
    assert nv.nv_sdpa_device_status(0) == (nv.OK, 0)
    go.check()
    return from_device(go.out.contiguous(), case.dtype), go.lse.cpu().numpy().astype(np.float64)


def want_ex(case, x, *, window=None, add_mask=None, rows=None):
    """The oracle on the same stored values (all rows, or the sampled (b, h, i) rows);
    the additive mask is rounded to the input dtype first, as the GPU reads it."""
    kw = dict(mask_kind=case.mask, scale=case.scale_f32, bool_mask=x["mask"],
              sinks=None if x["sinks"] is None else W.widen(x["sinks"], case.dtype), window=window,
              add_mask=None if add_mask is None else W.widen(W.to_storage(add_mask, case.dtype), case.dtype))
    q, k, v = (W.widen(x[n], case.dtype) for n in ("q", "k", "v"))
    if rows is None:
        return oracle.sdpa(q, k, v, **kw)
    return oracle.sdpa_sampled(q, k, v, rows, **kw)


def compare(name, case, got, glse, want, wlse, rows=None):
    tol = TOL[case.dtype]
    if rows is not None:
        got = np.stack([got[b, h, i] for b, h, i in rows])
        glse = np.array([glse[b, h, i] for b, h, i in rows])
    assert_close(name + " out", got, want, tol)
    assert_close(name + " lse", glse, wlse, tol)
    assert np.all(np.isfinite(got)), name + ": non-finite output"


def _rows(case, n=40, seed=0):
    rng = np.random.RandomState(seed)
    out = {(0, 0, 0), (case.B - 1, case.Hq - 1, case.Lq - 1)}
    while len(out) < n:
        out.add((int(rng.randint(case.B)), int(rng.randint(case.Hq)), int(rng.randint(case.Lq))))
    return sorted(out)


def _check(case, x, **kw):
    got, glse = run_ex(case, x, **kw)
    opts = {k: v for k, v in kw.items() if k in ("window", "add_mask")}
    flops = 2.0 * case.B * case.Hq * case.Lq * case.Lk * (case.d + case.dv)
    rows = None if flops <= 3e9 else _rows(case)
    want, wlse = want_ex(case, x, rows=rows, **opts)
    compare(case.name, case, got, glse, want, wlse, rows)
    return got, glse


# ----------------------------------------------------------------------------- windows

# (Lq, Lk, D, Hq, Hkv, W): "nuvec-core 0.5.0 tests/fast.rs", windows_run_fused_and_equal_the_boolean_mask
WINDOW_GRID = [
    (1, 300, 64, 8, 1, 128), (1, 4096, 64, 8, 8, 128), (1, 9000, 128, 8, 1, 3), (1, 2000, 256, 4, 1, 1024),
    (4, 600, 128, 4, 2, 7), (8, 1500, 64, 4, 4, 128), (40, 300, 64, 4, 2, 7), (97, 400, 128, 2, 1, 33),
    (64, 640, 64, 2, 2, 1), (300, 700, 256, 2, 1, 128), (33, 45, 64, 4, 2, 100), (1, 4000, 64, 8, 1, 128),
    (1, 9000, 128, 16, 2, 300), (2, 5000, 256, 4, 2, 1024),
]
WINDOW_CASES = []
for n, (lq, lk, d, hq, hkv, w) in enumerate(WINDOW_GRID):
    for t, dt in enumerate(["f32", "f16", "bf16"]):
        WINDOW_CASES.append((_case(1, hq, hkv, lq, lk, d, d, dt, "causal", (n + t) % 2 == 1, 300 + 3 * n + t,
                                   name=f"win_lq{lq}_lk{lk}_d{d}_h{hq}x{hkv}_w{w}_{dt}"), w))


@pytest.mark.parametrize("case,w", WINDOW_CASES, ids=[c.name for c, _ in WINDOW_CASES])
def test_window_matches_the_oracle(case, w):
    """Keys and values as slices of a longer cache (read in place), as in the pages' test."""
    _check(case, W.make_inputs(case), window=w, layouts=("contig", "slice", "slice", "contig"))


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("lq,lk", [(1, 3000), (5, 700), (300, 300), (200, 1000)])
def test_window_of_at_least_the_keys_is_causal_bit_for_bit(dt, lq, lk):
    """ "nuvec-core 0.5.0 tests/fast.rs", window_errors_empty_inputs_and_full_windows."""
    import torch
    nv = ensure_built()
    c = _case(2, 8, 2, lq, lk, 128, 128, dt, "causal", True, 77, "u2")
    x = W.make_inputs(c)
    base, base_lse = run_ex(c, x)
    for w in (lk, lk + 1, 10 * lk):
        got, lse = run_ex(c, x, window=w)
        assert np.array_equal(got, base) and np.array_equal(lse, base_lse), w
    torch.cuda.synchronize()


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("lk,w,hq,hkv", [(9000, 300, 16, 2), (4000, 128, 8, 1), (2000, 1024, 4, 1),
                                         (50000, 4096, 32, 4)])
def test_windowed_decode_row_equals_its_window_alone(dt, lk, w, hq, hkv):
    """One query: the row gets the bits of an unmasked call over exactly its window's keys
    ("nuvec-core 0.5.0 tests/fast.rs", windows_run_fused_and_equal_the_boolean_mask), and
    the key split follows the window, not the keys."""
    import torch
    nv = ensure_built()
    c = _case(2, hq, hkv, 1, lk, 128, 128, dt, "causal", True, 88, "u2")
    x = W.make_inputs(c)
    got, lse = run_ex(c, x, window=w)
    lo = lk - w
    xs = dict(x, k=np.ascontiguousarray(x["k"][:, :, lo:]), v=np.ascontiguousarray(x["v"][:, :, lo:]))
    cs = c.with_(Lk=w, mask="none")
    one, one_lse = run_ex(cs, xs)
    assert np.array_equal(got, one) and np.array_equal(lse, one_lse)
    _, pw = nv.nv_sdpa_plan_ex((c.B, c.Hq, c.Hkv, 1, lk, 128, 128), 1, 1, nv.DTYPES[dt],
                               nv.make_options(window=w))
    _, p1 = nv.nv_sdpa_plan((c.B, c.Hq, c.Hkv, 1, w, 128, 128), 0, 1, nv.DTYPES[dt])
    assert (pw["nblk"], pw["keys_per_blk"]) == (p1["nblk"], p1["keys_per_blk"])
    torch.cuda.synchronize()


@pytest.mark.parametrize("case,w", [
    (_case(2, 32, 8, 4096, 4096, 128, 128, "bf16", "causal", False, 91, name="win_prefill_nq2_bf16"), 512),
    (_case(1, 16, 2, 2048, 2048, 256, 256, "f16", "causal", True, 92, name="win_prefill_d256_f16"), 700),
    (_case(1, 8, 8, 1000, 3000, 128, 128, "bf16", "causal", True, 93, name="win_prefill_lq_lt_lk"), 129),
], ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_window_prefill_long_sequences(case, w):
    """Long prefills whose key tiles before every row's band are skipped (sampled rows)."""
    _check(case, W.make_inputs(case), window=w)


def test_window_errors_in_plan_and_op():
    """A window of 0 or below, or with a mask kind other than causal, is an error in the
    plan and in the op alike; nothing launches."""
    nv = ensure_built()
    dims = (1, 4, 2, 16, 64, 64, 64)
    fake = 1 << 20
    for mk, w in [(1, 0), (1, -3), (0, 3), (2, 3)]:
        o = nv.make_options()
        o.has_window, o.window = 1, w
        assert nv.nv_sdpa_plan_ex(dims, mk, 0, 2, o)[0] == nv.ERR_INVALID
        assert nv.nv_sdpa_ex(fake, fake, fake, dims, mk, fake, 0, 0.1, o, fake, 0, 2, 0) == nv.ERR_INVALID


# ----------------------------------------------------------------------------- additive masks

ADD_CASES = [
    # (case, mask shape prefix (mB, mH)): tensor-core prefill (two and one Q tiles), decode, f32
    (_case(2, 8, 2, 300, 500, 128, 128, "bf16", "add", True, 401, name="add_prefill_nq2_1xH"), (1, 8)),
    (_case(1, 8, 2, 257, 901, 64, 64, "f16", "add", False, 402, name="add_prefill_nq2_odd_lk"), (1, 1)),
    (_case(2, 4, 2, 200, 333, 256, 256, "f16", "add", True, 403, name="add_prefill_d256_BxH"), (2, 4)),
    (_case(2, 4, 1, 100, 700, 192, 128, "bf16", "add", False, 404, name="add_prefill_d192_Bx1"), (2, 1)),
    (_case(2, 8, 2, 1, 3000, 128, 128, "f16", "add", True, 405, name="add_decode_split"), (1, 8)),
    (_case(1, 4, 4, 3, 200, 64, 64, "bf16", "add", False, 406, name="add_decode_one_block"), (1, 4)),
    (_case(2, 4, 2, 40, 700, 64, 64, "f32", "add", True, 407, name="add_f32"), (2, 4)),
    (_case(1, 4, 2, 2, 33, 96, 64, "f32", "add", False, 408, name="add_f32_decode"), (1, 1)),
]


@pytest.mark.parametrize("case,mshape", ADD_CASES, ids=[c.name for c, _ in ADD_CASES])
def test_additive_mask_matches_the_oracle(case, mshape):
    """softmax(scale q.k + mask): N(0,1) entries, a few -inf (hidden keys), and one row hidden
    entirely (zeros, never NaN) -- "nuvec-core 0.5.0 tests/fast.rs",
    attention_kernels_match_the_fallback (the additive mask [1, hq, lq, lk])."""
    x = W.make_inputs(case)
    s = W.Stream(case.seed + 7)
    am = s.normal(mshape[0] * mshape[1] * case.Lq * case.Lk).reshape(mshape + (case.Lq, case.Lk))
    am[..., ::7] = -np.inf
    am[..., case.Lq // 2, :] = -np.inf
    got, glse = _check(case, x, add_mask=am)
    assert np.all(got[:, :, case.Lq // 2] == 0.0)


@pytest.mark.parametrize("layouts", [("bhld_T", "contig", "contig", "bhld_T"), ("contig",) * 4],
                         ids=["head_local_tiles", "packed_rows"])
def test_additive_mask_staging_over_many_tiles(layouts):
    """The staged additive values over many key tiles (chunks of two 64-key tiles, odd
    counts, a row length that is no multiple of 8 elements, the tensor's last row ending
    mid-chunk), with the rows taken from packed tiles and from head-local tiles (strided q
    and out)."""
    case = _case(2, 8, 2, 260, 1123, 128, 128, "bf16", "add", True, 409, name="add_staging_" + layouts[0])
    x = W.make_inputs(case)
    s = W.Stream(case.seed + 7)
    am = s.normal(case.B * case.Hq * case.Lq * case.Lk).reshape(case.B, case.Hq, case.Lq, case.Lk)
    am[..., ::11] = -np.inf
    got, glse = run_ex(case, x, add_mask=am, layouts=layouts)
    rows = _rows(case, n=60, seed=3)
    want, wlse = want_ex(case, x, rows=rows, add_mask=am)
    compare(case.name, case, got, glse, want, wlse, rows)


# ----------------------------------------------------------------------------- strided views

STRIDE_CASES = [
    # q and out as transposed [B, L, H, D] buffers; k, v transposed or sliced
    (_case(2, 8, 2, 300, 500, 128, 128, "bf16", "causal", True, 501, name="stride_prefill_nq2"),
     ("bhld_T", "bhld_T", "bhld_T", "bhld_T")),
    (_case(1, 6, 2, 200, 300, 128, 128, "f16", "none", False, 502, name="stride_prefill_odd_group"),
     ("bhld_T", "slice", "slice", "bhld_T")),
    (_case(2, 4, 2, 130, 777, 256, 256, "bf16", "bool", True, 503, name="stride_prefill_d256_bool"),
     ("bhld_T", "bhld_T", "slice", "contig")),
    (_case(1, 8, 2, 512, 512, 64, 64, "bf16", "causal", False, 504, name="stride_prefill_q_only"),
     ("bhld_T", "contig", "contig", "contig")),
    (_case(1, 8, 2, 256, 600, 96, 64, "f16", "causal", True, 505, name="stride_prefill_out_only"),
     ("contig", "contig", "contig", "bhld_T")),
    (_case(2, 8, 2, 1, 5000, 128, 128, "f16", "causal", True, 506, name="stride_decode_split"),
     ("bhld_T", "bhld_T", "bhld_T", "bhld_T")),
    (_case(1, 16, 2, 4, 900, 64, 64, "bf16", "none", False, 507, name="stride_decode_lq4"),
     ("bhld_T", "slice", "slice", "bhld_T")),
    (_case(2, 4, 2, 20, 300, 64, 64, "f32", "causal", True, 508, name="stride_f32"),
     ("bhld_T", "bhld_T", "slice", "bhld_T")),
]


@pytest.mark.parametrize("case,layouts", STRIDE_CASES, ids=[c.name for c, _ in STRIDE_CASES])
def test_strided_views_match_the_oracle(case, layouts):
    """Transposed [B, L, H, D] views and slices of longer caches are read in place (the
    keys around a slice hold NaN, which must never be read) -- "nuvec-core 0.5.0
    tests/fast.rs", attention_kernels_match_the_fallback and the windowed-kernel inputs."""
    _check(case, W.make_inputs(case), layouts=layouts)


def test_strided_prefill_big():
    """The 2x32/8 prefill shape with every tensor a transposed view (sampled rows)."""
    c = _case(2, 32, 8, 2048, 2048, 128, 128, "bf16", "causal", False, 509, name="stride_big")
    _check(c, W.make_inputs(c), layouts=("bhld_T",) * 4)


def test_strides_off_the_tma_grid_are_unsupported():
    nv = ensure_built()
    dims = (1, 4, 2, 16, 64, 64, 64)
    o = nv.make_options(k_strides=(2 * 64 * 65, 64 * 65, 65))   # a row stride of 65 elements
    assert nv.nv_sdpa_plan_ex(dims, 0, 0, 2, o)[0] == nv.ERR_UNSUPPORTED
    o = nv.make_options(q_strides=(-1, 64, 64))
    assert nv.nv_sdpa_plan_ex(dims, 0, 0, 2, o)[0] == nv.ERR_INVALID


# ----------------------------------------------------------------------------- paged caches

def _paged_inputs(case, lengths, bs, seed, extra_blocks=3):
    """Caches [num_blocks, Hkv, bs, d] holding each sequence's keys in shuffled blocks (a
    few unused; NaN everywhere no key lives), the block table and the lengths."""
    x = W.make_inputs(case)      # k, v of [B, Hkv, N, d] with N = max length
    N = case.Lk
    per = -(-N // bs)
    nblocks = case.B * per + extra_blocks
    order = np.random.RandomState(seed).permutation(nblocks)
    kdt = x["k"].dtype
    nan = W.to_storage(np.array([np.nan]), case.dtype)[0]
    kc = np.full((nblocks, case.Hkv, bs, case.d), nan, dtype=kdt)
    vc = np.full((nblocks, case.Hkv, bs, case.dv), nan, dtype=kdt)
    table = np.zeros((case.B, per), np.int32)
    for s in range(case.B):
        for j in range(per):
            blk = order[s * per + j]
            table[s, j] = blk
            n = max(0, min(bs, lengths[s] - j * bs))
            kc[blk, :, :n] = x["k"][s, :, j * bs:j * bs + n]
            vc[blk, :, :n] = x["v"][s, :, j * bs:j * bs + n]
    return x, kc, vc, table, np.array(lengths, np.int32)


def run_paged(case, x, kc, vc, table, lens, *, window=None):
    import torch
    nv = ensure_built()
    dt = case.dtype
    q = to_device(x["q"], dt)
    kcd, vcd = to_device(kc, dt), to_device(vc, dt)
    td = torch.from_numpy(table).cuda()
    ld = torch.from_numpy(lens).cuda()
    sinks = to_device(x["sinks"], dt) if x["sinks"] is not None else None
    go = _GuardedOut(case, False)
    st = nv.nv_sdpa_paged(q.data_ptr(), kcd.data_ptr(), vcd.data_ptr(), td.data_ptr(), ld.data_ptr(),
                          (case.B, case.Hq, case.Hkv, case.Lq, case.d, case.dv, kc.shape[0], kc.shape[2],
                           table.shape[1]), nv.MASKS[case.mask], window is not None, window or 0,
                          sinks.data_ptr() if sinks is not None else 0, case.scale_f32, go.out.data_ptr(),
                          go.lse.data_ptr(), nv.DTYPES[dt], torch.cuda.current_stream().cuda_stream)
    assert st == nv.OK, nv.nv_sdpa_status_string(st)
    torch.cuda.synchronize()
    assert nv.nv_sdpa_device_status(0) == (nv.OK, 0)
    go.check()
    return from_device(go.out, dt), go.lse.cpu().numpy().astype(np.float64)


def want_paged(case, x, kc, vc, table, lens, window=None):
    return oracle.sdpa_paged(W.widen(x["q"], case.dtype), W.widen(kc, case.dtype), W.widen(vc, case.dtype),
                             table, lens, mask_kind=case.mask, scale=case.scale_f32,
                             sinks=None if x["sinks"] is None else W.widen(x["sinks"], case.dtype),
                             window=window)


# (B, Hq, Hkv, Lq, d, block size, lengths, window): the pages' paged grids
PAGED_GRID = [
    (1, 4, 4, 1, 128, 16, [37], None), (3, 8, 2, 1, 128, 32, [1, 64, 300], None),
    (2, 4, 1, 4, 64, 16, [4, 77], None), (2, 2, 2, 1, 256, 8, [9, 513], None),
    (2, 8, 2, 1, 128, 32, [1500, 3000], None), (1, 8, 2, 4, 128, 64, [2100], None),
    (1, 4, 2, 1, 256, 16, [1100], None),
    (2, 8, 1, 1, 64, 16, [40, 300], 128), (2, 4, 2, 4, 64, 16, [9, 77], 5),
    (2, 8, 2, 1, 128, 32, [1500, 3000], 128), (1, 4, 4, 1, 256, 8, [513], 256),
    (2, 8, 2, 1, 128, 24, [700, 1234], None),  # a block size that is no power of two
]
PAGED_CASES = []
for n, (B, hq, hkv, lq, d, bs, lens, w) in enumerate(PAGED_GRID):
    for t, dt in enumerate(["f32", "f16", "bf16"]):
        PAGED_CASES.append((_case(B, hq, hkv, lq, max(lens), d, d, dt, "causal", (n + t) % 2 == 0, 600 + 3 * n + t,
                                  name=f"paged_b{B}_h{hq}x{hkv}_lq{lq}_d{d}_bs{bs}_w{w}_{dt}"), bs, lens, w))


@pytest.mark.parametrize("case,bs,lens,w", PAGED_CASES, ids=[c[0].name for c in PAGED_CASES])
def test_paged_matches_the_oracle(case, bs, lens, w):
    """Shuffled blocks, unused blocks and every slot past a length hold NaN: none is read.
    With a window, the blocks wholly before it hold NaN too."""
    x, kc, vc, table, ln = _paged_inputs(case, lens, bs, case.seed)
    if w is not None:
        nan = W.to_storage(np.array([np.nan]), case.dtype)[0]
        for s, L in enumerate(lens):
            first = max(0, L - case.Lq - w + 1)
            for j in range(first // bs):
                kc[table[s, j]] = nan
                vc[table[s, j]] = nan
    got, glse = run_paged(case, x, kc, vc, table, ln, window=w)
    want, wlse = want_paged(case, x, kc, vc, table, ln, window=w)
    compare(case.name, case, got, glse, want, wlse)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("B,hq,hkv,lq,d,bs,max_blocks", [(2, 4, 2, 1, 64, 8, 4), (2, 4, 2, 3, 128, 16, 3),
                                                         (2, 8, 2, 1, 128, 32, 64)])
def test_paged_clamps_hostile_tables_and_lengths(dt, B, hq, hkv, lq, d, bs, max_blocks):
    """Entries past the block count, negative ones, and lengths past the capacity: clamped,
    finite, equal to the oracle's clamped reading ("nuvec-core 0.5.0 tests/fast.rs",
    paged_attention_clamps_hostile_tables_and_lengths)."""
    blocks = 5
    c = _case(B, hq, hkv, lq, bs, d, d, dt, "causal", False, 700 + bs)
    s = W.Stream(c.seed)
    kc = W.to_storage(s.normal(blocks * hkv * bs * d).reshape(blocks, hkv, bs, d), dt)
    vc = W.to_storage(s.normal(blocks * hkv * bs * d).reshape(blocks, hkv, bs, d), dt)
    x = dict(q=W.to_storage(s.normal(B * hq * lq * d).reshape(B, hq, lq, d), dt), sinks=None)
    vals = [lambda i: i % blocks, lambda i: blocks + 1000, lambda i: -5, lambda i: 2**31 - 1]
    table = np.array([vals[i % 4](i) for i in range(B * max_blocks)], np.int64).astype(np.int32)
    table = table.reshape(B, max_blocks)
    lens = np.array([max_blocks * bs + 1, 2**31 - 1][:B], np.int32)
    got, glse = run_paged(c, x, kc, vc, table, lens)
    want, wlse = want_paged(c, x, kc, vc, table, lens)
    compare(f"hostile {dt}", c, got, glse, want, wlse)


def test_paged_equals_contiguous_bits_on_the_same_split():
    """Where both plans cut the keys into the same blocks, paged attention gives the
    contiguous call's bits."""
    import torch
    nv = ensure_built()
    c = _case(2, 8, 2, 1, 200, 128, 128, "f16", "causal", True, 801, "u2")
    x, kc, vc, table, ln = _paged_inputs(c, [200, 200], 16, 801, extra_blocks=0)
    _, pp = nv.nv_sdpa_paged_plan((2, 8, 2, 1, 128, 128, kc.shape[0], 16, table.shape[1]), 1, 0, 0, 1, 1)
    _, pc = nv.nv_sdpa_plan((2, 8, 2, 1, 200, 128, 128), 1, 1, 1)
    assert (pp["nblk"], pp["keys_per_blk"]) == (pc["nblk"], pc["keys_per_blk"])
    got, glse = run_paged(c, x, kc, vc, table, ln)
    one, one_lse = run_ex(c, x)
    assert np.array_equal(got, one) and np.array_equal(glse, one_lse)
    torch.cuda.synchronize()


def test_paged_errors():
    nv = ensure_built()
    fake = 1 << 20
    dims = (1, 4, 2, 1, 64, 64, 4, 8, 2)
    assert nv.nv_sdpa_paged_plan(dims, 2, 0, 0, 0, 1)[0] == nv.ERR_INVALID      # boolean mask
    assert nv.nv_sdpa_paged_plan(dims, 1, 1, 0, 0, 1)[0] == nv.ERR_INVALID      # window 0
    assert nv.nv_sdpa_paged_plan((1, 4, 3, 1, 64, 64, 4, 8, 2), 1, 0, 0, 0, 1)[0] == nv.ERR_INVALID
    assert nv.nv_sdpa_paged_plan((1, 4, 2, 9, 64, 64, 4, 8, 2), 1, 0, 0, 0, 1)[0] == nv.ERR_UNSUPPORTED
    assert nv.nv_sdpa_paged(fake, fake, fake, 0, fake, dims, 1, 0, 0, 0, 0.1, fake, 0, 1, 0) == nv.ERR_INVALID

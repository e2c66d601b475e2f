"""The C ABI without a GPU: the library loads, exports every function its header
declares, and its host-side checks and planner behave as documented.  Nothing here
launches a kernel."""
import os
import re

import pytest

from helpers import ensure_built

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def nv():
    return ensure_built()


def header_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(nv_sdpa\w*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = header_functions()
    for must in ["nv_sdpa", "nv_sdpa_plan", "nv_sdpa_host", "nv_sdpa_device_status",
                 "nv_sdpa_status_string", "nv_sdpa_abi_version", "nv_sdpa_set_wait_limit"]:
        assert must in names


def test_library_exports_every_declared_symbol(nv):
    lib = nv.lib()
    missing = [n for n in header_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_only_abi_symbols_are_exported(nv):
    import subprocess
    r = subprocess.run(["nm", "-D", "--defined-only", nv.LIB_PATH], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("nm not available")
    syms = [l.split()[-1] for l in r.stdout.splitlines() if " T " in l]
    ours = [s for s in syms if s.startswith("nv_sdpa")]
    assert set(ours) == set(header_functions())


def test_abi_version_and_status_strings(nv):
    assert nv.nv_sdpa_abi_version() == 2
    for s in range(5):
        assert nv.nv_sdpa_status_string(s) and "unknown" not in nv.nv_sdpa_status_string(s)
    assert "unknown" in nv.nv_sdpa_status_string(99)


# ----------------------------------------------------------------------------- planner

def plan(nv, dims, mask="none", sinks=0, dtype="bf16"):
    return nv.nv_sdpa_plan(dims, nv.MASKS.get(mask, mask) if isinstance(mask, str) else mask,
                           sinks, nv.DTYPES.get(dtype, dtype) if isinstance(dtype, str) else dtype)


@pytest.mark.parametrize("dims,status", [
    ((1, 4, 3, 16, 16, 64, 64), 1),      # Hq not a multiple of Hkv
    ((1, 4, 0, 16, 16, 64, 64), 1),      # Hkv = 0
    ((-1, 4, 2, 16, 16, 64, 64), 1),     # negative size
    ((1, 4, 2, -1, 16, 64, 64), 1),
    ((1, 4, 2, 16, 16, 0, 64), 1),       # d = 0
    ((1, 4, 2, 16, 16, 64, 0), 1),
    ((1 << 40, 1 << 20, 1, 1 << 10, 16, 64, 64), 1),  # size overflow
    ((1, 4, 2, 16, 16, 512, 512), 2),    # head 512: not built
    ((1, 4, 2, 16, 16, 60, 60), 2),      # not a multiple of 8
    ((1, 4, 2, 16, 16, 64, 264), 2),
])
def test_plan_rejects(nv, dims, status):
    st, pl = plan(nv, dims)
    assert st == status and pl is None


def test_plan_rejects_unknown_kinds(nv):
    assert plan(nv, (1, 4, 2, 16, 16, 64, 64), mask=3)[0] == nv.ERR_INVALID
    assert plan(nv, (1, 4, 2, 16, 16, 64, 64), dtype=3)[0] == nv.ERR_INVALID
    assert plan(nv, (1, 4, 2, 16, 16, 64, 64), dtype=-1)[0] == nv.ERR_INVALID


def test_plan_routes_by_query_length(nv):
    for lq, path in [(0, "noop"), (1, "decode"), (8, "decode"), (9, "prefill"), (4096, "prefill")]:
        st, pl = plan(nv, (2, 32, 8, lq, 4096, 128, 128), mask="causal")
        assert st == 0 and pl["path"] == path, (lq, pl)
    st, pl = plan(nv, (2, 32, 8, 5, 0, 128, 128))
    assert pl["path"] == "no_keys" and pl["kernel"] == "fill" and pl["scratch_bytes"] == 0
    st, pl = plan(nv, (0, 32, 8, 5, 10, 128, 128))
    assert pl["path"] == "noop" and pl["launches"] == 0


def test_every_head_shape_of_the_pages_is_planned(nv):
    shapes = [(64, 64), (72, 72), (80, 80), (96, 96), (128, 128), (192, 192), (256, 256),
              (96, 64), (192, 128)]
    for d, dv in shapes:
        for dt in ["f32", "f16", "bf16"]:
            for lq in [1, 9, 342]:
                st, pl = plan(nv, (1, 16, 2, lq, 1801, d, dv), mask="causal", dtype=dt)
                assert st == 0, (d, dv, dt, lq)


def test_plan_is_pure_and_batch_independent(nv):
    a = [plan(nv, (8, 32, 4, 1, 32769, 128, 128), "causal", 1, "f16")[1] for _ in range(5)]
    assert all(x == a[0] for x in a)
    one = plan(nv, (1, 32, 4, 1, 32769, 128, 128), "causal", 1, "f16")[1]
    # the key split is the same for every batch size: item b gets the bits of item b alone
    assert (one["nblk"], one["keys_per_blk"]) == (a[0]["nblk"], a[0]["keys_per_blk"])


def test_decode_scratch_is_small_next_to_the_keys(nv):
    B, Hq, Hkv, Lk, d = 8, 32, 4, 32769, 128
    st, pl = plan(nv, (B, Hq, Hkv, 1, Lk, d, d), "causal", 1, "f16")
    assert st == 0 and pl["path"] == "decode"
    kv_bytes = 2 * B * Hkv * Lk * d * 2
    assert pl["nblk"] > 1 and 0 < pl["scratch_bytes"] <= 0.02 * kv_bytes
    assert pl["nblk"] * pl["keys_per_blk"] >= Lk > (pl["nblk"] - 1) * pl["keys_per_blk"]


def test_decode_grid_is_one_wave_and_splits_only_by_shape(nv):
    """The decode kernel's warps (up to 8 per CTA, one CTA per SM of 152 for d = dv = 128)
    run as one wave for any batch size, each walking a run of key blocks; a grid of fewer
    warps than 8 per SM takes smaller CTAs, spread over the SMs.  The blocks themselves
    depend on the head shape and Lk only."""
    warp_slots = 8 * 152
    for B in (1, 2, 8, 64):
        st, pl = plan(nv, (B, 32, 4, 1, 32769, 128, 128), "causal", 1, "f16")
        assert st == 0 and pl["path"] == "decode" and pl["kernel"] == "decode_mma"
        assert (pl["nblk"], pl["keys_per_blk"]) == (74, 448)
        units = B * 4
        spans = min(pl["nblk"], max(1, warp_slots // units))
        wpc = max(1, min(8, -(-units * spans // 152)))
        assert pl["grid"] == -(-units * spans // wpc)
        assert pl["grid"] <= max(152, -(-units // 8))
    # one sequence: 4 x 74 warps in CTAs of 2, over 148 SMs
    assert plan(nv, (1, 32, 4, 1, 32769, 128, 128), "causal", 1, "f16")[1]["grid"] == 148


def test_decode_with_many_rows_per_kv_head_takes_the_split_tcgen05_kernel(nv):
    """g x Lq > 16 query rows per KV head, or a head wider than 128: the tcgen05 prefill
    kernel split over blocks of whole 128-key tiles (at least 8), the same blocks for
    every batch size; a window, a boolean mask or 16 rows or fewer of a head up to 128
    keep the mma.sync decode kernel."""
    dims = (8, 32, 4, 8, 32769, 128, 128)
    ref = None
    for B in (1, 2, 8, 64):
        st, pl = plan(nv, (B,) + dims[1:], "causal", 1, "f16")
        assert st == 0 and pl["path"] == "decode" and pl["kernel"] == "decode_tc", pl
        assert pl["keys_per_blk"] % 128 == 0 and pl["keys_per_blk"] >= 8 * 128
        assert pl["nblk"] * pl["keys_per_blk"] >= 32769 > (pl["nblk"] - 1) * pl["keys_per_blk"]
        assert pl["grid"] == B * 4 * pl["nblk"] and pl["launches"] == 2
        ref = ref or (pl["nblk"], pl["keys_per_blk"])
        assert (pl["nblk"], pl["keys_per_blk"]) == ref
    assert plan(nv, dims, "bool", 0, "bf16")[1]["kernel"] == "decode_mma"
    assert plan(nv, (8, 8, 4, 8, 32769, 128, 128), "causal", 0, "bf16")[1]["kernel"] == "decode_mma"  # 16 rows
    st, pl = nv.nv_sdpa_plan_ex(dims, nv.MASKS["causal"], 0, nv.DTYPES["bf16"], nv.make_options(window=512))
    assert st == 0 and pl["kernel"] == "decode_mma"
    assert plan(nv, dims, "causal", 0, "f32")[1]["kernel"] == "tiled_simt"
    # heads wider than 128 take it at any row count (the mma.sync kernel's accumulators
    # would not fit its registers)
    for d, dv in [(256, 256), (192, 192), (192, 128), (64, 256)]:
        st, pl = plan(nv, (8, 16, 2, 1, 32769, d, dv), "causal", 1, "f16")
        assert st == 0 and pl["kernel"] == "decode_tc", (d, dv, pl)


# ----------------------------------------------------------------------------- entry points

def test_nv_sdpa_rejects_before_touching_a_device(nv):
    dims = (1, 4, 2, 16, 16, 64, 64)
    fake = 1 << 20  # aligned, never dereferenced: every call below fails its checks first
    assert nv.nv_sdpa(fake, fake, fake, (1, 4, 3, 16, 16, 64, 64), 0, 0, 0, 1.0, fake, 0, 2, 0) == nv.ERR_INVALID
    assert nv.nv_sdpa(0, fake, fake, dims, 0, 0, 0, 1.0, fake, 0, 2, 0) == nv.ERR_INVALID
    assert nv.nv_sdpa(fake, fake, fake, dims, 0, 0, 0, 1.0, 0, 0, 2, 0) == nv.ERR_INVALID
    assert nv.nv_sdpa(fake + 2, fake, fake, dims, 0, 0, 0, 1.0, fake, 0, 2, 0) == nv.ERR_INVALID
    assert nv.nv_sdpa(fake, fake, fake, dims, 2, 0, 0, 1.0, fake, 0, 2, 0) == nv.ERR_INVALID  # bool, no mask
    assert nv.nv_sdpa(fake, fake, fake, dims, 0, 0, 0, float("nan"), fake, 0, 2, 0) == nv.ERR_INVALID
    assert nv.nv_sdpa(fake, fake, fake, dims, 0, 0, 0, float("inf"), fake, 0, 2, 0) == nv.ERR_INVALID
    assert nv.nv_sdpa(fake, fake, fake, dims, 0, 0, 0, 1.0, fake, 0, 7, 0) == nv.ERR_INVALID
    assert nv.nv_sdpa(fake, fake, fake, (1, 4, 2, 16, 16, 512, 512), 0, 0, 0, 1.0, fake, 0, 2, 0) == nv.ERR_UNSUPPORTED
    # nothing to do: OK without any pointer
    assert nv.nv_sdpa(0, 0, 0, (1, 4, 2, 0, 16, 64, 64), 0, 0, 0, 1.0, 0, 0, 2, 0) == nv.OK


def test_host_entry_point_rejects_bad_arguments(nv):
    assert nv.nv_sdpa_host(0, 0, 0, (1, 4, 2, 16, 16, 64, 64), 0, 0, 0, 1.0, 0, 0, 2, 0) == nv.ERR_INVALID
    assert nv.nv_sdpa_host(0, 0, 0, (1, 4, 3, 16, 16, 64, 64), 0, 0, 0, 1.0, 0, 0, 2, 0) == nv.ERR_INVALID


def test_product_path_fails_loudly_without_the_library(monkeypatch, tmp_path):
    import scaled_dot_product_nv_gb300 as nvmod
    monkeypatch.setattr(nvmod, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(nvmod, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        nvmod.lib()


def test_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "scaled_dot_product_nv_gb300")
    for dp, _, fs in os.walk(pkg):
        for f in fs:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dp, f)).read()
                assert not re.search(r"\boracle\b", src.replace("oracle is", "")), f


def test_wrapper_passes_zero_strides_for_contiguous_tensors(nv):
    """The torch wrapper hands the options struct strides only for tensors that are not
    contiguous: zero strides are the header's contiguous layout, and skipping them keeps
    a windowed call's host time down."""
    import torch
    t = torch.empty(2, 3, 5, 8)
    assert nv._strides_or_none(t, t.is_contiguous()) is None
    v = torch.empty(2, 5, 3, 8).transpose(1, 2)  # a [B, L, H, D] buffer viewed as [B, H, L, D]
    assert not v.is_contiguous()
    assert nv._strides_or_none(v, False) == (5 * 3 * 8, 8, 3 * 8)
    o = nv.make_options(window=7, q_strides=None, k_strides=nv._strides_or_none(v, False))
    assert (o.has_window, o.window) == (1, 7)
    assert list(o.q_strides) == [0, 0, 0] and list(o.k_strides) == [120, 8, 24]
    assert list(o.v_strides) == [0, 0, 0] and list(o.out_strides) == [0, 0, 0]
    with pytest.raises(ValueError):
        nv._bhl_strides(torch.empty(2, 3, 8, 5).transpose(2, 3))  # head dimension not contiguous


def test_wrapper_launches_on_a_given_stream(nv):
    """An explicit stream object's handle is used as is (no current-stream lookup)."""
    class FakeStream:
        cuda_stream = 0x1234
    assert nv._stream_handle(FakeStream(), None) == 0x1234

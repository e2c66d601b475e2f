"""nv_sdpa_noalloc: the attention call for callers that cannot allocate device memory
(a host program whose GPU memory belongs to another allocator, e.g. a serving runtime
that reserves the device up front, or a loop that cannot afford an allocation call).
Its scratch comes from the library's fixed device array instead of cudaMallocAsync.

Checked through the C ABI against nv_sdpa on the same inputs, on two calls in a row
with different inputs (the array keeps the first call's contents when the second
runs).  Both entry points run the same kernels on the same plan, so the results must
agree bit for bit, which is stricter than the parity tolerance.  This file is
collected last on purpose."""
import numpy as np
import pytest

import workloads as W
from helpers import ensure_built, from_device, upload

pytestmark = pytest.mark.gpu

CASES = [
    # split-KV decode: the partials live in the static array
    W.decode_f16_long_kv(),
    # boolean-mask prefill: the bit-packed mask lives in the static array
    W.prefill_f16_boolmask_sinks(),
    # f32 decode on the FFMA kernel, split over key blocks
    W.Case(2, 8, 2, 3, 9000, 64, 64, "f32", "causal", True, None, "u0.25", seed=31,
           name="decode_f32_split"),
]


def _call(nv, fn, case, dev, out, lse):
    import torch
    st = fn(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(),
            (case.B, case.Hq, case.Hkv, case.Lq, case.Lk, case.d, case.dv),
            W.MASK_CODES[case.mask], dev["mask"].data_ptr() if dev["mask"] is not None else 0,
            dev["sinks"].data_ptr() if dev["sinks"] is not None else 0, case.scale_f32,
            out.data_ptr(), lse.data_ptr(), W.DTYPE_CODES[case.dtype],
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("case", CASES, ids=[c.name for c in CASES])
def test_noalloc_matches_nv_sdpa_on_two_calls_in_a_row(case):
    import torch
    nv = ensure_built()
    st, plan = nv.nv_sdpa_plan((case.B, case.Hq, case.Hkv, case.Lq, case.Lk, case.d, case.dv),
                               W.MASK_CODES[case.mask], int(case.sinks), W.DTYPE_CODES[case.dtype])
    assert st == nv.OK and 0 < plan["scratch_bytes"] <= nv.STATIC_SCRATCH_BYTES, plan
    from helpers import torch_dtype
    for call, seed in enumerate([case.seed, case.seed + 1000]):
        c = case.with_(seed=seed)
        dev = upload(c, W.make_inputs(c))
        shape = (c.B, c.Hq, c.Lq, c.dv)
        ref_out = torch.empty(shape, dtype=torch_dtype(c.dtype), device="cuda")
        ref_lse = torch.empty(shape[:3], dtype=torch.float32, device="cuda")
        assert _call(nv, nv.nv_sdpa, c, dev, ref_out, ref_lse) == nv.OK
        out = torch.full(shape, float("nan"), dtype=torch_dtype(c.dtype), device="cuda")
        lse = torch.full(shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        assert _call(nv, nv.nv_sdpa_noalloc, c, dev, out, lse) == nv.OK, f"call {call}"
        assert nv.nv_sdpa_device_status(0) == (nv.OK, 0)
        got = from_device(out, c.dtype)
        assert np.all(np.isfinite(got))
        bits = torch.int16 if c.dtype != "f32" else torch.int32
        assert torch.equal(out.view(bits), ref_out.view(bits)), f"{c.name} call {call}: out bits"
        assert torch.equal(lse, ref_lse), f"{c.name} call {call}: lse bits"


def test_noalloc_rejects_a_plan_beyond_the_static_scratch():
    nv = ensure_built()
    dims = (64, 32, 4, 1, 32769, 128, 128)  # split-KV partials of ~79 MB
    st, plan = nv.nv_sdpa_plan(dims, 1, 1, 1)
    assert st == nv.OK and plan["scratch_bytes"] > nv.STATIC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first and launches nothing
    assert nv.nv_sdpa_noalloc(fake, fake, fake, dims, 1, 0, fake, 0.1, fake, 0, 1, 0) == \
        nv.ERR_UNSUPPORTED


def test_noalloc_calls_replay_from_a_cuda_graph():
    """Captured in a CUDA graph -- the kernels' programmatic dependent launches become
    the graph's programmatic edges -- a boolean-mask prefill (packing + attention) and
    a split-KV decode (pass 1 + merge), replayed three times with new inputs copied into
    the captured buffers each time, give the bits of direct nv_sdpa calls."""
    import torch
    nv = ensure_built()
    cases = [W.Case(1, 8, 2, 200, 700, 128, 128, "f16", "bool", True, None, "n0.5", seed=61, name="g_bool"),
             W.Case(2, 16, 4, 1, 9000, 128, 128, "bf16", "causal", True, None, "n0.5", seed=62, name="g_decode")]
    from helpers import torch_dtype
    devs, outs, lses = [], [], []
    for c in cases:
        devs.append(upload(c, W.make_inputs(c)))
        outs.append(torch.empty((c.B, c.Hq, c.Lq, c.dv), dtype=torch_dtype(c.dtype), device="cuda"))
        lses.append(torch.empty((c.B, c.Hq, c.Lq), dtype=torch.float32, device="cuda"))

    def launch_all():
        for c, dev, o, l in zip(cases, devs, outs, lses):
            st = nv.nv_sdpa_noalloc(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(),
                                    (c.B, c.Hq, c.Hkv, c.Lq, c.Lk, c.d, c.dv), W.MASK_CODES[c.mask],
                                    dev["mask"].data_ptr() if dev["mask"] is not None else 0,
                                    dev["sinks"].data_ptr() if dev["sinks"] is not None else 0, c.scale_f32,
                                    o.data_ptr(), l.data_ptr(), W.DTYPE_CODES[c.dtype],
                                    torch.cuda.current_stream().cuda_stream)
            assert st == nv.OK
    launch_all()  # outside the capture first (the static array's address is looked up)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        launch_all()
    torch.cuda.synchronize()
    for rep in range(3):
        for i, c in enumerate(cases):
            x = W.make_inputs(c.with_(seed=c.seed + 100 * (rep + 1)))
            fresh = upload(c, x)
            for n in ("q", "k", "v"):
                devs[i][n].copy_(fresh[n])
        graph.replay()
        torch.cuda.synchronize()
        for c, dev, o, l in zip(cases, devs, outs, lses):
            want, wl = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind=c.mask, scale=c.scale_f32,
                               bool_mask=dev["mask"], sinks=dev["sinks"])
            torch.cuda.synchronize()
            bits = torch.int16 if c.dtype != "f32" else torch.int32
            assert torch.equal(o.view(bits), want.view(bits)), (c.name, rep)
            assert torch.equal(l, wl), (c.name, rep)
        assert nv.nv_sdpa_device_status(0) == (nv.OK, 0)

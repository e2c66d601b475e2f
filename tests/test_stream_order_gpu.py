"""Stream order across calls.  Every kernel of the library is launched as the programmatic
dependent of the stream's previous kernel, so its CTAs may be placed while that kernel
drains; each waits for the previous grid before it touches global memory.  These tests
chain calls with no host synchronisation in between and compare the results, bit for bit,
with the same chain run one call at a time:
- read after write: each call's query is the previous call's output;
- write after read: a call's output buffer is the memory the previous call read its keys
  (and, for split calls, its merge read its partials) from.
The paths covered are the tensor-core prefill, the boolean-mask prefill (packing kernel
first), the split tcgen05 decode with its merge pass, the mma.sync decode with its merge,
and the FP32 kernel."""
import pytest

from helpers import ensure_built

pytestmark = pytest.mark.gpu

# (name, B, Hq, Hkv, Lq, Lk, d, dtype, mask, expected kernel)
PATHS = [
    ("prefill_tc", 1, 8, 2, 384, 2000, 128, "bf16", "causal", "prefill_tc"),
    ("bool_mask", 1, 4, 2, 256, 700, 128, "f16", "bool", "prefill_tc"),
    ("decode_tc", 2, 16, 2, 8, 5000, 128, "bf16", "causal", "decode_tc"),
    ("decode_mma", 2, 8, 2, 1, 9000, 128, "f16", "causal", "decode_mma"),
    ("tiled_simt", 1, 4, 2, 3, 3000, 64, "f32", "causal", "tiled_simt"),
]


def _inputs(torch, B, Hq, Hkv, Lq, Lk, d, dt, mask, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dt]

    def r(*s):
        return (torch.randn(s, generator=g, device="cuda") * 0.5).to(tdt)
    q, k, v = r(B, Hq, Lq, d), r(B, Hkv, Lk, d), r(B, Hkv, Lk, d)
    m = (torch.rand((Lq, Lk), generator=g, device="cuda") < 0.7).to(torch.uint8) if mask == "bool" else None
    return q, k, v, r(Hq), m


@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
def test_chained_calls_read_after_write(path):
    import torch
    nv = ensure_built()
    name, B, Hq, Hkv, Lq, Lk, d, dt, mask, kern = path
    st, pl = nv.nv_sdpa_plan((B, Hq, Hkv, Lq, Lk, d, d), nv.MASKS[mask], 1, nv.DTYPES[dt])
    assert st == nv.OK and pl["kernel"] == kern, pl
    q0, k, v, s, m = _inputs(torch, B, Hq, Hkv, Lq, Lk, d, dt, mask, 11)
    n = 6

    def chain(sync):
        outs, q = [], q0
        for _ in range(n):
            o, lse = nv.sdpa(q, k, v, mask_kind=mask, bool_mask=m, sinks=s)
            if sync:
                torch.cuda.synchronize()
            outs.append((o, lse))
            q = o  # the next call reads this call's output
        torch.cuda.synchronize()
        return outs

    want = chain(True)
    for rep in range(3):
        got = chain(False)
        for i, ((go, gl), (wo, wl)) in enumerate(zip(got, want)):
            assert torch.equal(go, wo), (rep, i)
            assert torch.equal(gl, wl), (rep, i)


@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
def test_output_over_previous_inputs_write_after_read(path):
    """Call 1 reads its keys from buffer X; call 2, queued right behind it, writes its
    output into X.  Call 1's result must be that of keys read before call 2 ran."""
    import torch
    nv = ensure_built()
    name, B, Hq, Hkv, Lq, Lk, d, dt, mask, kern = path
    q, k, v, s, m = _inputs(torch, B, Hq, Hkv, Lq, Lk, d, dt, mask, 12)
    ref1, ref1_lse = nv.sdpa(q, k, v, mask_kind=mask, bool_mask=m, sinks=s)
    torch.cuda.synchronize()
    n_out = B * Hq * Lq * d
    assert n_out <= k.numel()
    for rep in range(3):
        x = k.clone()  # call 1's keys
        o1, l1 = nv.sdpa(q, x, v, mask_kind=mask, bool_mask=m, sinks=s)
        # call 2 writes its output over the first n_out elements of x
        o2_view = x.view(-1)[:n_out].view(B, Hq, Lq, d)
        nv.sdpa(q, k, v, mask_kind=mask, bool_mask=m, sinks=s, out=o2_view)
        torch.cuda.synchronize()
        assert torch.equal(o1, ref1), rep
        assert torch.equal(l1, ref1_lse), rep
        assert torch.equal(o2_view, ref1), rep

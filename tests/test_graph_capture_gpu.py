"""nv_sdpa, nv_sdpa_ex and nv_sdpa_paged captured into a CUDA graph.

A captured call takes its scratch (split-KV partials, the bit-packed boolean mask) from
cudaMallocAsync, which the capture records as the graph's own allocation and free nodes,
instead of the library's memory pool.  Each replay must then give the bits of the same
call made directly: the kernels and the plan are the same, only where the scratch lives
differs.  Covered: a boolean-mask prefill (packing + attention), a split-KV decode
(pass 1 + merge), a windowed decode through the options struct and a paged decode, all
four in one graph on torch's capture stream, replayed with new inputs copied into the
captured buffers."""
import pytest

import workloads as W
from helpers import ensure_built, torch_dtype, upload

pytestmark = pytest.mark.gpu

BOOL = W.Case(1, 8, 2, 200, 700, 128, 128, "f16", "bool", True, None, "n0.5", seed=71, name="cap_bool")
SPLIT = W.Case(2, 16, 4, 1, 9000, 128, 128, "bf16", "causal", True, None, "n0.5", seed=72, name="cap_split")
WIN = W.Case(2, 16, 4, 1, 9000, 128, 128, "f16", "causal", True, None, "n0.5", seed=73, name="cap_window")
WINDOW = 3000
BS = 16


def _paged(dev, case, order):
    """K and V of `case` cut into blocks of BS keys, stored at the shuffled slots `order`."""
    import torch
    per = -(-case.Lk // BS)

    def pages(t):
        pad = torch.zeros((case.B, case.Hkv, per * BS, t.shape[3]), dtype=t.dtype, device=t.device)
        pad[:, :, :case.Lk] = t
        blocks = pad.view(case.B, case.Hkv, per, BS, t.shape[3]).permute(0, 2, 1, 3, 4)
        cache = torch.zeros((order.numel(), case.Hkv, BS, t.shape[3]), dtype=t.dtype, device=t.device)
        cache[order] = blocks.reshape(case.B * per, case.Hkv, BS, t.shape[3])
        return cache
    return pages(dev["k"]), pages(dev["v"])


def test_captured_calls_replay_with_the_bits_of_direct_calls():
    import torch
    nv = ensure_built()
    # every call below needs scratch, so the capture takes the allocation path
    for c, opts in ((BOOL, None), (SPLIT, None), (WIN, nv.make_options(window=WINDOW))):
        st, pl = nv.nv_sdpa_plan_ex((c.B, c.Hq, c.Hkv, c.Lq, c.Lk, c.d, c.dv), W.MASK_CODES[c.mask], 1,
                                    W.DTYPE_CODES[c.dtype], opts)
        assert st == nv.OK and pl["scratch_bytes"] > 0, (c.name, pl)
    per = -(-WIN.Lk // BS)
    order = torch.randperm(WIN.B * per, generator=torch.Generator().manual_seed(7)).cuda()
    table = order.view(WIN.B, per).to(torch.int32).contiguous()  # block (b, j) sits in slot order[b per + j]
    lens = torch.tensor([WIN.Lk, WIN.Lk - 1234], dtype=torch.int32, device="cuda")
    st, ppl = nv.nv_sdpa_paged_plan((WIN.B, WIN.Hq, WIN.Hkv, 1, WIN.d, WIN.dv, order.numel(), BS, per), 1, 1,
                                    WINDOW, 1, W.DTYPE_CODES[WIN.dtype])
    assert st == nv.OK and ppl["scratch_bytes"] > 0, ppl

    devs = {c.name: upload(c, W.make_inputs(c)) for c in (BOOL, SPLIT, WIN)}
    kc, vc = _paged(devs[WIN.name], WIN, order)
    outs = {n: (torch.empty((c.B, c.Hq, c.Lq, c.dv), dtype=torch_dtype(c.dtype), device="cuda"),
                torch.empty((c.B, c.Hq, c.Lq), dtype=torch.float32, device="cuda"))
            for n, c in (("bool", BOOL), ("split", SPLIT), ("window", WIN), ("paged", WIN))}

    def calls(into):
        b, s, w = devs[BOOL.name], devs[SPLIT.name], devs[WIN.name]
        nv.sdpa(b["q"], b["k"], b["v"], mask_kind="bool", scale=BOOL.scale_f32, bool_mask=b["mask"],
                sinks=b["sinks"], out=into["bool"][0], lse=into["bool"][1])
        nv.sdpa(s["q"], s["k"], s["v"], mask_kind="causal", scale=SPLIT.scale_f32, sinks=s["sinks"],
                out=into["split"][0], lse=into["split"][1])
        nv.sdpa(w["q"], w["k"], w["v"], mask_kind="causal", scale=WIN.scale_f32, window=WINDOW,
                sinks=w["sinks"], out=into["window"][0], lse=into["window"][1])
        nv.sdpa_paged(w["q"], kc, vc, table, lens, mask_kind="causal", scale=WIN.scale_f32, window=WINDOW,
                      sinks=w["sinks"], out=into["paged"][0], lse=into["paged"][1])

    calls(outs)  # outside the capture first: kernel attributes, the status word's address
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls(outs)
    torch.cuda.synchronize()
    want = {n: (torch.empty_like(o), torch.empty_like(l)) for n, (o, l) in outs.items()}
    for rep in range(2):
        for c in (BOOL, SPLIT, WIN):
            fresh = upload(c, W.make_inputs(c.with_(seed=c.seed + 100 * (rep + 1))))
            for n in ("q", "k", "v"):
                devs[c.name][n].copy_(fresh[n])
        nk, nvv = _paged(devs[WIN.name], WIN, order)
        kc.copy_(nk)
        vc.copy_(nvv)
        for o, l in outs.values():
            o.fill_(float("nan"))
            l.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        calls(want)
        torch.cuda.synchronize()
        for n, (o, l) in outs.items():
            bits = torch.int16
            assert torch.equal(o.view(bits), want[n][0].view(bits)), (n, rep)
            assert torch.equal(l, want[n][1]), (n, rep)
        assert bool(torch.isfinite(outs["split"][0].float()).all())
        assert nv.nv_sdpa_device_status(0) == (nv.OK, 0)

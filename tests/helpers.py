"""Shared test plumbing: upload seeded inputs, call the CUDA path through the C ABI,
evaluate the oracle on the same stored values, and compare with the pages' metric."""
from __future__ import annotations

import os

import numpy as np

import workloads as W

# max|a - b| <= tol * max(|b|, 1) per element ("nuvec-core 0.5.0 tests/fast.rs",
# assert_close), with these tolerances per dtype; the same for the log-sum-exp.
TOL = {"f32": 2e-5, "f16": 4e-3, "bf16": 2e-2}


def ensure_built():
    import scaled_dot_product_nv_gb300 as nv
    if not os.path.exists(nv.LIB_PATH):
        from scaled_dot_product_nv_gb300 import _build
        _build.build()
    return nv


def close_mask(got, want, tol):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    same = got == want  # covers matching infinities
    return same | (np.abs(got - want) <= tol * np.maximum(np.abs(want), 1.0))


def assert_close(name, got, want, tol):
    ok = close_mask(got, want, tol)
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        g = np.asarray(got, dtype=np.float64)
        w = np.asarray(want, dtype=np.float64)
        err = np.abs(g - w) / np.maximum(np.abs(w), 1.0)
        err = np.where(np.isnan(err), np.inf, err)
        raise AssertionError(f"{name}: {bad.shape[0]} of {ok.size} elements off; first at {i}: "
                             f"got {g[i]} want {w[i]}; worst scaled error {np.nanmax(err):.3g} "
                             f"(tol {tol})")


# ----------------------------------------------------------------------------- device side

def torch_dtype(dt):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dt]


def to_device(stored, dt):
    """Stored numpy array (float32 / float16 / bf16 bits) -> CUDA tensor of that dtype."""
    import torch
    if dt == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(stored).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(stored))
    return t.cuda()


def from_device(t, dt):
    import torch
    t = t.detach().cpu()
    if dt == "bf16":
        return W.widen(t.view(torch.int16).numpy().view(np.uint16), dt)
    return t.numpy().astype(np.float64)


def upload(case, x):
    dev = dict(q=to_device(x["q"], case.dtype), k=to_device(x["k"], case.dtype),
               v=to_device(x["v"], case.dtype))
    dev["sinks"] = to_device(x["sinks"], case.dtype) if x["sinks"] is not None else None
    dev["mask"] = to_device(x["mask"], "u8") if x["mask"] is not None else None
    return dev


GUARD_BYTES = 4096   # canary band on each side of an output (a multiple of 256: keeps alignment)
CANARY = 0xA5


class Guarded:
    """A CUDA tensor of `shape` inside a larger byte buffer whose bands before and after
    it hold a canary pattern, so that a kernel writing past either end of its output is
    caught (no memory checker runs on the GPU; these bands are the stand-in)."""

    def __init__(self, shape, dtype):
        import torch
        self.shape = tuple(shape)
        n = int(np.prod(self.shape)) if self.shape else 1
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD_BYTES + nbytes + GUARD_BYTES,), CANARY, dtype=torch.uint8,
                              device="cuda")
        self.nbytes = nbytes
        self.tensor = self.raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(self.shape)

    def check(self, what):
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.nbytes:]
        bad_head = int((head != CANARY).sum())
        bad_tail = int((tail != CANARY).sum())
        assert bad_head == 0 and bad_tail == 0, \
            f"{what}: {bad_head} bytes before and {bad_tail} bytes after the buffer were written"


def run_gpu(case, x, dev=None):
    """Runs the CUDA path; returns (out f64 [B,Hq,Lq,dv], lse f64 [B,Hq,Lq]).  The output
    and the log-sum-exp are written into canary-guarded buffers, checked after the call."""
    import torch
    nv = ensure_built()
    dev = dev or upload(case, x)
    gout = Guarded((case.B, case.Hq, case.Lq, case.dv), torch_dtype(case.dtype))
    glse = Guarded((case.B, case.Hq, case.Lq), torch.float32)
    out, lse = nv.sdpa(dev["q"], dev["k"], dev["v"], mask_kind=case.mask, scale=case.scale_f32,
                       bool_mask=dev["mask"], sinks=dev["sinks"], out=gout.tensor, lse=glse.tensor)
    torch.cuda.synchronize()
    st, detail = nv.nv_sdpa_device_status(0)
    assert st == nv.OK, f"device status {st} detail {detail:#x}"
    gout.check("out")
    glse.check("lse")
    return from_device(out, case.dtype), lse.cpu().numpy().astype(np.float64)


def oracle_full(case, x):
    import oracle
    return oracle.sdpa(W.widen(x["q"], case.dtype), W.widen(x["k"], case.dtype),
                       W.widen(x["v"], case.dtype), mask_kind=case.mask, scale=case.scale_f32,
                       bool_mask=x["mask"],
                       sinks=None if x["sinks"] is None else W.widen(x["sinks"], case.dtype))


def oracle_rows(case, x, samples):
    import oracle
    return oracle.sdpa_sampled(W.widen(x["q"], case.dtype), W.widen(x["k"], case.dtype),
                               W.widen(x["v"], case.dtype), samples, mask_kind=case.mask,
                               scale=case.scale_f32, bool_mask=x["mask"],
                               sinks=None if x["sinks"] is None else W.widen(x["sinks"], case.dtype))


def oracle_flops(case):
    return 2.0 * case.B * case.Hq * case.Lq * case.Lk * (case.d + case.dv)


def sample_rows(case, n=48, seed=0):
    """A spread of (b, h, i): first/last rows, tile edges, and seeded random rows."""
    rng = np.random.RandomState(seed)
    out = set()
    edges = [0, 1, case.Lq - 1, min(127, case.Lq - 1), min(128, case.Lq - 1), case.Lq // 2]
    for b in {0, case.B - 1}:
        for h in {0, case.Hq - 1, case.Hq // 2}:
            for i in edges:
                out.add((b, h, max(0, i)))
    while len(out) < n + len(edges):
        out.add((int(rng.randint(case.B)), int(rng.randint(case.Hq)), int(rng.randint(case.Lq))))
    return sorted(out)


def check_case(case, x=None, max_oracle_flops=4e10, name=None):
    """Full element-by-element comparison when the oracle finishes in seconds, else on
    sampled rows computed one by one."""
    x = x or W.make_inputs(case)
    got, glse = run_gpu(case, x)
    tol = TOL[case.dtype]
    name = name or case.name or str(case)
    if oracle_flops(case) <= max_oracle_flops:
        want, wlse = oracle_full(case, x)
        assert_close(name + " out", got, want, tol)
        assert_close(name + " lse", glse, wlse, tol)
    else:
        samples = sample_rows(case)
        want, wlse = oracle_rows(case, x, samples)
        g = np.stack([got[b, h, i] for b, h, i in samples])
        gl = np.array([glse[b, h, i] for b, h, i in samples])
        assert_close(name + " out (sampled)", g, want, tol)
        assert_close(name + " lse (sampled)", gl, wlse, tol)
    assert np.all(np.isfinite(got)), name + ": non-finite output"
    return got, glse

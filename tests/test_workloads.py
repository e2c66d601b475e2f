"""The seeded input generator (no GPU): the LCG against its sequential recurrence,
the dtype casts against torch's, and the workload list."""
import numpy as np
import torch

import workloads as W


def _sequential(seed, n):
    s, out = seed, []
    for _ in range(n):
        s = (s * 6364136223846793005 + 1) % (1 << 64)
        out.append(s >> 32)
    return out


def test_lcg_matches_recurrence_across_blocks():
    for seed in [0, 1, 0xDEADBEEF]:
        st = W.Stream(seed)
        got = list(st.u32(5)) + list(st.u32(W._BLOCK + 3))
        assert got == _sequential(seed, W._BLOCK + 8)


def test_uniform_and_normal_ranges():
    st = W.Stream(7)
    u = st.uniform(100000)
    assert u.min() >= 0.0 and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.01
    z = st.normal(100001)
    assert z.size == 100001 and abs(z.mean()) < 0.02 and abs(z.std() - 1) < 0.02


def test_casts_match_torch_rne():
    x = W.Stream(3).normal(50000) * 100
    for dt, tdt in [("f16", torch.float16), ("bf16", torch.bfloat16), ("f32", torch.float32)]:
        ours = W.widen(W.to_storage(x, dt), dt)
        ref = torch.from_numpy(x.astype(np.float32)).to(tdt).to(torch.float64).numpy()
        np.testing.assert_array_equal(ours, ref)


def test_sweep_is_108_cases_in_order():
    cases = W.sweep_bf16()
    assert len(cases) == 108
    assert [c.mask for c in cases[:4]] == ["causal", "none", "causal", "none"]
    assert all(c.B == 1 + c.Lk % 2 for c in cases)
    assert (cases[0].d, cases[0].Hq, cases[0].Lq, cases[0].Lk) == (64, 16, 1, 1)
    assert (cases[-1].d, cases[-1].dv, cases[-1].Hq, cases[-1].Lq, cases[-1].Lk) == (256, 256, 32, 342, 8193)


def test_make_inputs_shapes_and_mask_diagonal():
    c = W.Case(1, 4, 2, 9, 13, 16, 8, "bf16", "bool", True, None, "n0.5", seed=9)
    x = W.make_inputs(c)
    assert x["q"].shape == (1, 4, 9, 16) and x["q"].dtype == np.uint16
    assert x["v"].shape == (1, 2, 13, 8) and x["sinks"].shape == (4,)
    assert x["mask"].shape == (9, 13) and all(x["mask"][i, i] == 1 for i in range(9))
    y = W.make_inputs(c)
    assert all(np.array_equal(x[k], y[k]) for k in ["q", "k", "v", "sinks", "mask"])

"""Pins of the f64 oracle to facts it does not compute itself (no GPU needed).

Each pin is a function of the attention implementation under test so that the last
test can plant plausible mistakes in the oracle (on the CPU) and show that some pin
catches every one of them.

Sources: the worked examples of "lattice-inference 0.4.0 src/attention/flash.rs"
(tests/golden/*.txt, each citing its test), the direct formula and the empty-key
rules of "nuvec-core 0.5.0 tests/fast.rs", and closed forms of softmax attention.
"""
import decimal
import glob
import math
import os

import numpy as np
import pytest

import oracle
import oracle.attention as osdpa
from workloads import Stream

HERE = os.path.dirname(os.path.abspath(__file__))


def rand(shape, seed, lo=-1.0, hi=1.0):
    s = Stream(seed)
    return (lo + (hi - lo) * s.uniform(int(np.prod(shape)))).reshape(shape)


# ------------------------------------------------------------------ golden fixtures

def parse_fixture(path):
    fx = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            fx[key] = vals
    ints = {k: int(fx[k][0]) for k in ["B", "Hq", "Hkv", "Lq", "Lk", "d", "dv"]}
    arr = lambda k: np.array([float(x) for x in fx[k]])
    case = dict(ints)
    case["mask"] = fx["mask"][0]
    case["scale"] = float(fx["scale"][0])
    case["q"] = arr("q").reshape(ints["B"], ints["Hq"], ints["Lq"], ints["d"])
    case["k"] = arr("k").reshape(ints["B"], ints["Hkv"], ints["Lk"], ints["d"])
    case["v"] = arr("v").reshape(ints["B"], ints["Hkv"], ints["Lk"], ints["dv"])
    case["bool_mask"] = (arr("bool_mask").reshape(ints["Lq"], ints["Lk"]).astype(np.uint8)
                         if "bool_mask" in fx else None)
    case["expect_out"] = arr("expect_out").reshape(ints["B"], ints["Hq"], ints["Lq"], ints["dv"])
    case["tol"] = float(fx["tol"][0])
    return case


FIXTURES = sorted(glob.glob(os.path.join(HERE, "golden", "*.txt")))


def pin_golden(fn, path):
    c = parse_fixture(path)
    out, lse = fn(c["q"], c["k"], c["v"], mask_kind=c["mask"], scale=c["scale"],
                  bool_mask=c["bool_mask"])
    assert np.all(np.isfinite(out)), path
    err = np.max(np.abs(out - c["expect_out"])) if out.size else 0.0
    assert err <= c["tol"], (path, out, c["expect_out"])


@pytest.mark.parametrize("path", FIXTURES, ids=[os.path.basename(p) for p in FIXTURES])
def test_golden_fixture(path):
    pin_golden(oracle.sdpa, path)


def test_fixtures_present():
    assert len(FIXTURES) >= 3


# ------------------------------------------------------------------ closed forms

def pin_single_key(fn):
    """One visible key: the output is that key's value row, for any scale and mask."""
    for scale in [0.125, 3.0, -2.0, 0.0]:
        q = rand((1, 2, 3, 8), 1)
        k = rand((1, 1, 1, 8), 2)
        v = rand((1, 1, 1, 5), 3)
        for mk in ["none", "causal", "bool"]:
            bm = np.ones((3, 1), np.uint8)
            out, lse = fn(q, k, v, mask_kind=mk, scale=scale, bool_mask=bm)
            # causal, bottom-right: every row i sees key 0 since 0 <= i + 1 - 3 fails
            # only for i < 2 -> rows 0, 1 see nothing (zeros), row 2 sees key 0
            if mk == "causal":
                np.testing.assert_array_equal(out[:, :, :2], 0.0)
                np.testing.assert_allclose(out[0, :, 2], np.broadcast_to(v[0, 0, 0], (2, 5)),
                                           rtol=0, atol=1e-15)
            else:
                np.testing.assert_allclose(out[0], np.broadcast_to(v[0, 0, 0], (2, 3, 5)),
                                           rtol=0, atol=1e-15)
            s = scale * np.einsum("hid,d->hi", q[0], k[0, 0, 0])
            if mk != "causal":
                np.testing.assert_allclose(lse[0], s, rtol=1e-14, atol=1e-14)


def pin_single_key_with_sink(fn):
    """One key with score s and a sink logit sigma: out = v / (1 + e^(sigma - s)),
    lse = ln(e^s + e^sigma)."""
    q = rand((1, 2, 1, 4), 11)
    k = rand((1, 2, 1, 4), 12)
    v = rand((1, 2, 1, 3), 13)
    sinks = np.array([0.7, -1.3])
    scale = 0.5
    out, lse = fn(q, k, v, mask_kind="none", scale=scale, sinks=sinks)
    for h in range(2):
        s = scale * float(q[0, h, 0] @ k[0, h, 0])
        w = 1.0 / (1.0 + math.exp(sinks[h] - s))
        np.testing.assert_allclose(out[0, h, 0], w * v[0, h, 0], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(lse[0, h, 0], math.log(math.exp(s) + math.exp(sinks[h])),
                                   rtol=1e-13)


def pin_identical_keys_mean(fn):
    """All keys equal: every visible key gets the same weight -> mean of visible V."""
    Lq, Lk = 4, 7
    q = rand((1, 1, Lq, 6), 21)
    k = np.broadcast_to(rand((1, 1, 1, 6), 22), (1, 1, Lk, 6)).copy()
    v = rand((1, 1, Lk, 5), 23)
    bm = (rand((Lq, Lk), 24, 0, 1) < 0.6).astype(np.uint8)
    bm[:, 0] = 1
    for mk in ["none", "causal", "bool"]:
        out, _ = fn(q, k, v, mask_kind=mk, scale=0.9, bool_mask=bm)
        for i in range(Lq):
            if mk == "none":
                vis = np.arange(Lk)
            elif mk == "causal":
                vis = np.arange(i + Lk - Lq + 1)     # the page's visible count
            else:
                vis = np.nonzero(bm[i])[0]
            np.testing.assert_allclose(out[0, 0, i], v[0, 0, vis].mean(axis=0), rtol=1e-13)


def pin_zero_scale_mean(fn):
    """scale = 0: every score is 0 -> mean of the visible V rows, for any K."""
    q = rand((2, 2, 3, 4), 31)
    k = rand((2, 1, 6, 4), 32)
    v = rand((2, 1, 6, 3), 33)
    out, lse = fn(q, k, v, mask_kind="causal", scale=0.0)
    for i in range(3):
        n = i + 6 - 3 + 1
        np.testing.assert_allclose(out[:, :, i], np.broadcast_to(
            v[:, :, :n].mean(axis=2), (2, 2, 3)), rtol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(n), rtol=1e-14)


def pin_causal_row0(fn):
    """Lq = Lk, causal: query 0 sees only key 0 -> out = V[0]; the last row sees all."""
    q = rand((1, 2, 5, 8), 41)
    k = rand((1, 2, 5, 8), 42)
    v = rand((1, 2, 5, 8), 43)
    out, _ = fn(q, k, v, mask_kind="causal", scale=0.3)
    np.testing.assert_allclose(out[0, :, 0], v[0, :, 0], rtol=0, atol=1e-15)
    full, _ = fn(q, k, v, mask_kind="none", scale=0.3)
    np.testing.assert_allclose(out[0, :, 4], full[0, :, 4], rtol=1e-14)


def pin_decode_causal_sees_all(fn):
    """One query, causal (bottom-right): it sees every key -> equals no mask."""
    q = rand((2, 4, 1, 8), 51)
    k = rand((2, 2, 9, 8), 52)
    v = rand((2, 2, 9, 4), 53)
    a, la = fn(q, k, v, mask_kind="causal", scale=0.4)
    b, lb = fn(q, k, v, mask_kind="none", scale=0.4)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def pin_gqa_equals_repeated_heads(fn):
    """Hq/Hkv grouping == the same call with each KV head repeated g times in order
    (query head h reads KV head h // g)."""
    B, Hq, Hkv, Lq, Lk = 2, 6, 2, 5, 7
    q = rand((B, Hq, Lq, 4), 61)
    k = rand((B, Hkv, Lk, 4), 62)
    v = rand((B, Hkv, Lk, 3), 63)
    g = Hq // Hkv
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    sinks = rand((Hq,), 64)
    for mk in ["none", "causal"]:
        a, la = fn(q, k, v, mask_kind=mk, scale=0.7, sinks=sinks)
        b, lb = fn(q, kr, vr, mask_kind=mk, scale=0.7, sinks=sinks)
        np.testing.assert_array_equal(a, b)
        np.testing.assert_array_equal(la, lb)
    # and distinct heads really do give distinct results
    assert not np.allclose(a[:, 0], a[:, g])


def pin_sink_limits(fn):
    """sink = -inf is no sink at all; a sink far above every score takes all the
    weight: out -> 0 and lse -> sink."""
    q = rand((1, 3, 4, 8), 71)
    k = rand((1, 3, 6, 8), 72)
    v = rand((1, 3, 6, 5), 73)
    a, la = fn(q, k, v, mask_kind="causal", scale=0.5)
    b, lb = fn(q, k, v, mask_kind="causal", scale=0.5, sinks=np.full(3, -np.inf))
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
    big = np.full(3, 60.0)
    c, lc = fn(q, k, v, mask_kind="causal", scale=0.5, sinks=big)
    assert np.max(np.abs(c)) < 1e-20
    np.testing.assert_allclose(lc, 60.0, rtol=1e-15)


def pin_empty_and_all_masked(fn):
    """No keys: zeros, with a causal mask and with sinks too ("nuvec-core 0.5.0
    tests/fast.rs", window_errors_empty_inputs_and_full_windows).  All keys masked:
    zeros and never NaN; lse = -inf, or the sink when there is one.  No queries: an
    empty output."""
    q = rand((1, 2, 3, 64), 81)
    none = np.zeros((1, 2, 0, 64))
    sinks = rand((2,), 82)
    for mk, s in [("none", None), ("causal", None), ("causal", sinks)]:
        out, lse = fn(q, none, none, mask_kind=mk, scale=0.125, sinks=s)
        assert out.shape == (1, 2, 3, 64)
        np.testing.assert_array_equal(out, 0.0)
        if s is None:
            assert np.all(lse == -np.inf)
        else:
            np.testing.assert_allclose(lse[0], np.broadcast_to(sinks[:, None], (2, 3)))
    k = rand((1, 2, 4, 64), 83)
    out, lse = fn(q, k, k, mask_kind="bool", scale=0.125, bool_mask=np.zeros((3, 4), np.uint8),
                  sinks=sinks)
    np.testing.assert_array_equal(out, 0.0)
    np.testing.assert_allclose(lse[0], np.broadcast_to(sinks[:, None], (2, 3)))
    # causal with more queries than keys: the first Lq - Lk rows see no key
    q5 = rand((1, 2, 6, 64), 84)
    out, lse = fn(q5, k, k, mask_kind="causal", scale=0.125)
    np.testing.assert_array_equal(out[:, :, :2], 0.0)
    assert np.all(lse[:, :, :2] == -np.inf) and np.all(np.isfinite(lse[:, :, 2:]))
    out, lse = fn(np.zeros((1, 2, 0, 64)), k, k, mask_kind="causal", scale=0.125)
    assert out.shape == (1, 2, 0, 64) and lse.shape == (1, 2, 0)


# ------------------------------------------------------------------ sliding window

def pin_window_full_equals_causal(fn):
    """A window of at least the keys is plain causal attention, bit for bit ("nuvec-core
    0.5.0 tests/fast.rs", window_errors_empty_inputs_and_full_windows)."""
    q = rand((1, 2, 5, 8), 131)
    k = rand((1, 2, 9, 8), 132)
    v = rand((1, 2, 9, 4), 133)
    c, lc = fn(q, k, v, mask_kind="causal", scale=0.125)
    for w in [9, 10, 1000]:
        a, la = fn(q, k, v, mask_kind="causal", scale=0.125, window=w)
        np.testing.assert_array_equal(a, c)
        np.testing.assert_array_equal(la, lc)
    a, _ = fn(q, k, v, mask_kind="causal", scale=0.125, window=8)
    assert not np.array_equal(a, c)   # a window shorter than the keys does hide some


def pin_window_of_one_sees_its_own_position(fn):
    """W = 1: the query at position p = i + Lk - Lq sees key p alone -> out = v_p and
    lse = s_pp (with a sink: the one-key closed form); rows with p < 0 see nothing."""
    q = rand((1, 2, 6, 4), 141)
    k = rand((1, 1, 4, 4), 142)
    v = rand((1, 1, 4, 3), 143)
    sinks = np.array([0.3, -0.8])
    scale = 0.7
    out, lse = fn(q, k, v, mask_kind="causal", scale=scale, window=1)
    outs, lses = fn(q, k, v, mask_kind="causal", scale=scale, window=1, sinks=sinks)
    for h in range(2):
        for i in range(6):
            p = i + 4 - 6
            if p < 0:
                assert np.all(out[0, h, i] == 0) and lse[0, h, i] == -np.inf
                np.testing.assert_array_equal(outs[0, h, i], 0.0)
                assert lses[0, h, i] == sinks[h]
                continue
            s = scale * float(q[0, h, i] @ k[0, 0, p])
            np.testing.assert_allclose(out[0, h, i], v[0, 0, p], rtol=0, atol=1e-15)
            np.testing.assert_allclose(lse[0, h, i], s, rtol=1e-14, atol=1e-15)
            w = 1.0 / (1.0 + math.exp(sinks[h] - s))
            np.testing.assert_allclose(outs[0, h, i], w * v[0, 0, p], rtol=1e-13, atol=1e-15)


def pin_window_identical_keys_mean(fn):
    """Identical keys: each row is the mean of the V rows in its band, whose size is
    min(W, p + 1) -- the count of keys p - W < j <= p that exist."""
    Lq, Lk, W = 5, 9, 3
    q = rand((1, 1, Lq, 6), 151)
    k = np.broadcast_to(rand((1, 1, 1, 6), 152), (1, 1, Lk, 6)).copy()
    v = rand((1, 1, Lk, 5), 153)
    out, lse = fn(q, k, v, mask_kind="causal", scale=1.1, window=W)
    for i in range(Lq):
        p = i + Lk - Lq
        np.testing.assert_allclose(out[0, 0, i], v[0, 0, p - W + 1:p + 1].mean(axis=0), rtol=1e-13)


def pin_window_rows_equal_one_query_calls(fn):
    """Each row of a windowed call equals an unmasked one-query call over exactly its
    window's keys ("nuvec-core 0.5.0 tests/fast.rs", windows_run_fused_and_equal_the_boolean_mask)."""
    Lq, Lk, W = 4, 11, 5
    q = rand((2, 4, Lq, 8), 161)
    k = rand((2, 2, Lk, 8), 162)
    v = rand((2, 2, Lk, 6), 163)
    sinks = rand((4,), 164)
    out, lse = fn(q, k, v, mask_kind="causal", scale=0.4, window=W, sinks=sinks)
    for i in range(Lq):
        p = i + Lk - Lq
        lo, hi = max(0, p - W + 1), p + 1
        o1, l1 = fn(q[:, :, i:i + 1], k[:, :, lo:hi], v[:, :, lo:hi], mask_kind="none", scale=0.4,
                    sinks=sinks)
        np.testing.assert_allclose(out[:, :, i:i + 1], o1, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(lse[:, :, i:i + 1], l1, rtol=1e-13)


def pin_window_errors(fn):
    """A window of 0, or a window without the causal mask, is an error."""
    q = rand((1, 2, 5, 8), 171)
    k = rand((1, 2, 9, 8), 172)
    bm = np.ones((5, 9), np.uint8)
    for kw in [dict(mask_kind="causal", window=0), dict(mask_kind="causal", window=-2),
               dict(mask_kind="none", window=3), dict(mask_kind="bool", window=3, bool_mask=bm)]:
        with pytest.raises(ValueError):
            fn(q, k, k, scale=0.125, **kw)


# ------------------------------------------------------------------ additive mask

def pin_additive_zero_equals_none(fn):
    q = rand((2, 4, 5, 8), 181)
    k = rand((2, 2, 7, 8), 182)
    v = rand((2, 2, 7, 3), 183)
    a, la = fn(q, k, v, mask_kind="add", scale=0.3, add_mask=np.zeros((1, 4, 5, 7)))
    b, lb = fn(q, k, v, mask_kind="none", scale=0.3)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def pin_additive_neg_inf_equals_bool(fn):
    """0 where the boolean mask is true and -inf where false hides exactly the same keys
    (a row hidden entirely gives zeros, never NaN)."""
    q = rand((1, 2, 6, 8), 191)
    k = rand((1, 1, 9, 8), 192)
    v = rand((1, 1, 9, 4), 193)
    bm = (rand((6, 9), 194, 0, 1) < 0.5).astype(np.uint8)
    bm[2] = 0
    sinks = rand((2,), 195)
    am = np.where(bm != 0, 0.0, -np.inf)[None, None]
    for s in [None, sinks]:
        a, la = fn(q, k, v, mask_kind="add", scale=0.8, add_mask=am, sinks=s)
        b, lb = fn(q, k, v, mask_kind="bool", scale=0.8, bool_mask=bm, sinks=s)
        np.testing.assert_array_equal(a, b)
        np.testing.assert_array_equal(la, lb)
    assert np.all(a[:, :, 2] == 0)


def pin_additive_log_weights(fn):
    """scale = 0 and a mask of log weights: out = sum_j w_j v_j / sum_j w_j and
    lse = ln sum_j w_j, for chosen weights -- the mask is added to the scaled scores
    (not multiplied by the scale), and enters the exponent as itself."""
    w = np.array([1.0, 2.0, 0.5, 4.0, 0.25])
    q = rand((1, 1, 2, 3), 201)
    k = rand((1, 1, 5, 3), 202)
    v = rand((1, 1, 5, 2), 203)
    am = np.broadcast_to(np.log(w), (1, 1, 2, 5)).copy()
    out, lse = fn(q, k, v, mask_kind="add", scale=0.0, add_mask=am)
    want = (w @ v[0, 0]) / w.sum()
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(want, (2, 2)), rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], math.log(w.sum()), rtol=1e-14)


def pin_additive_constant_shift(fn):
    """A constant mask c changes no weight and shifts the log-sum-exp by exactly c."""
    q = rand((1, 2, 4, 8), 211)
    k = rand((1, 2, 6, 8), 212)
    v = rand((1, 2, 6, 5), 213)
    b, lb = fn(q, k, v, mask_kind="none", scale=0.5)
    for c in [3.0, -7.25]:
        a, la = fn(q, k, v, mask_kind="add", scale=0.5, add_mask=np.full((1, 1, 4, 6), c))
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(la, lb + c, rtol=1e-13)


def pin_additive_broadcast(fn):
    """[1, 1, Lq, Lk] acts like the same mask repeated over batch items and heads; a
    [B, Hq, Lq, Lk] mask gives item b, head h its own slice."""
    B, Hq, Hkv, Lq, Lk = 2, 4, 2, 3, 6
    q = rand((B, Hq, Lq, 4), 221)
    k = rand((B, Hkv, Lk, 4), 222)
    v = rand((B, Hkv, Lk, 3), 223)
    m1 = rand((1, 1, Lq, Lk), 224, -2, 2)
    a, la = fn(q, k, v, mask_kind="add", scale=0.6, add_mask=m1)
    b, lb = fn(q, k, v, mask_kind="add", scale=0.6, add_mask=np.broadcast_to(m1, (B, Hq, Lq, Lk)).copy())
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
    full = rand((B, Hq, Lq, Lk), 225, -2, 2)
    a, la = fn(q, k, v, mask_kind="add", scale=0.6, add_mask=full)
    for bb in range(B):
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            o, lo = fn(q[bb:bb + 1, h:h + 1], k[bb:bb + 1, hk:hk + 1], v[bb:bb + 1, hk:hk + 1],
                       mask_kind="add", scale=0.6, add_mask=full[bb:bb + 1, h:h + 1])
            np.testing.assert_array_equal(a[bb:bb + 1, h:h + 1], o)
            np.testing.assert_array_equal(la[bb:bb + 1, h:h + 1], lo)


# ------------------------------------------------------------------ brute force

def decimal_attention(q, k, v, mask_kind, scale, bool_mask=None, sinks=None, prec=60, window=None,
                      add_mask=None):
    """An independent evaluation in 60-digit decimal arithmetic, with no maximum
    subtracted: out_i = sum_j e^(s_ij) v_j / (sum_j e^(s_ij) + e^(sink)).  Visible keys
    follow the pages' statement directly: a causal row i sees its first
    i + Lk - Lq + 1 keys; a boolean mask row lists its own keys."""
    D = decimal.Decimal
    ctx = decimal.Context(prec=prec)
    B, Hq, Lq, d = q.shape
    Hkv, Lk, dv = k.shape[1], k.shape[2], v.shape[3]
    out = np.zeros((B, Hq, Lq, dv))
    lse = np.zeros((B, Hq, Lq))
    for b in range(B):
        for h in range(Hq):
            hk = h * Hkv // Hq
            for i in range(Lq):
                if mask_kind == "causal" and window is not None:
                    # the page's band: position p sees keys p - W < j <= p
                    pos = i + Lk - Lq
                    keys = [j for j in range(Lk) if pos - window < j <= pos]
                elif mask_kind == "causal":
                    keys = range(max(0, min(Lk, i + Lk - Lq + 1)))
                elif mask_kind == "bool":
                    keys = [j for j in range(Lk) if bool_mask[i][j]]
                else:
                    keys = range(Lk)
                num = [D(0)] * dv
                den = D(0)
                for j in keys:
                    dot = D(0)
                    for c in range(d):
                        dot = ctx.add(dot, ctx.multiply(D(float(q[b, h, i, c])), D(float(k[b, hk, j, c]))))
                    logit = ctx.multiply(D(float(scale)), dot)
                    if add_mask is not None:
                        a = add_mask[b if add_mask.shape[0] > 1 else 0, h if add_mask.shape[1] > 1 else 0, i, j]
                        if a == -math.inf:
                            continue
                        logit = ctx.add(logit, D(float(a)))
                    w = ctx.exp(logit)
                    den = ctx.add(den, w)
                    for c in range(dv):
                        num[c] = ctx.add(num[c], ctx.multiply(w, D(float(v[b, hk, j, c]))))
                zsum = den
                if sinks is not None:
                    zsum = ctx.add(zsum, ctx.exp(D(float(sinks[h]))))
                if zsum == 0:
                    lse[b, h, i] = -math.inf
                    continue
                lse[b, h, i] = float(ctx.ln(zsum))
                for c in range(dv):
                    out[b, h, i, c] = float(ctx.divide(num[c], zsum))
    return out, lse


BRUTE_CASES = [
    # the pages' own direct-formula shape: one head, Lq 3, Lk 5, d 4, scale 0.5, causal
    dict(B=1, Hq=1, Hkv=1, Lq=3, Lk=5, d=4, dv=4, mask="causal", scale=0.5, sinks=False),
    dict(B=1, Hq=1, Hkv=1, Lq=3, Lk=5, d=4, dv=4, mask="none", scale=0.5, sinks=True),
    dict(B=2, Hq=4, Hkv=2, Lq=4, Lk=6, d=3, dv=2, mask="bool", scale=1.3, sinks=True),
    dict(B=1, Hq=3, Hkv=1, Lq=6, Lk=4, d=5, dv=3, mask="causal", scale=-0.8, sinks=False),
    dict(B=1, Hq=2, Hkv=2, Lq=2, Lk=9, d=8, dv=6, mask="causal", scale=0.35, sinks=True),
    # a sliding window of 3 (the band p - 3 < j <= p) and an additive mask
    dict(B=1, Hq=2, Hkv=1, Lq=4, Lk=7, d=3, dv=2, mask="causal", scale=0.9, sinks=True, window=3),
    dict(B=2, Hq=2, Hkv=1, Lq=3, Lk=5, d=4, dv=3, mask="add", scale=-0.6, sinks=True, add=(2, 1)),
    dict(B=1, Hq=3, Hkv=3, Lq=2, Lk=6, d=2, dv=2, mask="add", scale=0.4, sinks=False, add=(1, 3)),
]


def pin_brute_force(fn):
    for n, c in enumerate(BRUTE_CASES):
        q = rand((c["B"], c["Hq"], c["Lq"], c["d"]), 100 + n, -2, 2)
        k = rand((c["B"], c["Hkv"], c["Lk"], c["d"]), 200 + n, -2, 2)
        v = rand((c["B"], c["Hkv"], c["Lk"], c["dv"]), 300 + n, -2, 2)
        bm = (rand((c["Lq"], c["Lk"]), 400 + n, 0, 1) < 0.6).astype(np.uint8)
        sinks = rand((c["Hq"],), 500 + n, -1, 1) if c["sinks"] else None
        kw = {}
        if "window" in c:
            kw["window"] = c["window"]
        if "add" in c:
            mb, mh = c["add"]
            am = rand((mb, mh, c["Lq"], c["Lk"]), 600 + n, -3, 3)
            am[..., 1] = -np.inf   # hidden keys
            kw["add_mask"] = am
        a, la = fn(q, k, v, mask_kind=c["mask"], scale=c["scale"], bool_mask=bm, sinks=sinks, **kw)
        b, lb = decimal_attention(q, k, v, c["mask"], c["scale"], bm, sinks, **kw)
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14, err_msg=str(c))
        fin = np.isfinite(lb)
        assert np.array_equal(fin, np.isfinite(la))
        np.testing.assert_allclose(la[fin], lb[fin], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ invariants

def pin_lse_consistency(fn):
    """out_i = sum_vis e^(s_ij - lse_i) v_j and sum_vis e^(s_ij - lse_i) + e^(sink - lse_i) = 1."""
    q = rand((1, 2, 5, 6), 91)
    k = rand((1, 1, 8, 6), 92)
    v = rand((1, 1, 8, 4), 93)
    sinks = rand((2,), 94)
    scale = 0.6
    out, lse = fn(q, k, v, mask_kind="causal", scale=scale, sinks=sinks)
    for h in range(2):
        for i in range(5):
            nvis = i + 8 - 5 + 1
            s = scale * (k[0, 0, :nvis] @ q[0, h, i])
            w = np.exp(s - lse[0, h, i])
            np.testing.assert_allclose(w.sum() + math.exp(sinks[h] - lse[0, h, i]), 1.0, rtol=1e-13)
            np.testing.assert_allclose(w @ v[0, 0, :nvis], out[0, h, i], rtol=1e-12, atol=1e-15)


def pin_key_permutation(fn):
    """Without a causal order, permuting keys (with their V rows and mask columns)
    leaves the result unchanged up to rounding."""
    q = rand((1, 2, 4, 8), 95)
    k = rand((1, 2, 11, 8), 96)
    v = rand((1, 2, 11, 5), 97)
    bm = (rand((4, 11), 98, 0, 1) < 0.5).astype(np.uint8)
    perm = np.random.RandomState(3).permutation(11)
    for mk in ["none", "bool"]:
        a, la = fn(q, k, v, mask_kind=mk, scale=0.8, bool_mask=bm)
        b, lb = fn(q, k[:, :, perm], v[:, :, perm], mask_kind=mk, scale=0.8,
                   bool_mask=bm[:, perm])
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(la, lb, rtol=1e-13, atol=1e-15)


def pin_batch_items_alone(fn):
    """Each batch item equals the item run alone ("nuvec-core 0.5.0 tests/fast.rs",
    attention_batch_items_equal_each_item_alone)."""
    q = rand((3, 4, 5, 8), 101)
    k = rand((3, 2, 7, 8), 102)
    v = rand((3, 2, 7, 8), 103)
    s = rand((4,), 104)
    a, la = fn(q, k, v, mask_kind="causal", scale=0.35, sinks=s)
    for b in range(3):
        o, lo = fn(q[b:b + 1], k[b:b + 1], v[b:b + 1], mask_kind="causal", scale=0.35, sinks=s)
        np.testing.assert_array_equal(a[b:b + 1], o)
        np.testing.assert_array_equal(la[b:b + 1], lo)


def pin_sampled_equals_full(fn_full, fn_sampled):
    q = rand((2, 4, 6, 8), 111)
    k = rand((2, 2, 9, 8), 112)
    v = rand((2, 2, 9, 3), 113)
    bm = (rand((6, 9), 114, 0, 1) < 0.5).astype(np.uint8)
    s = rand((4,), 115)
    full, lf = fn_full(q, k, v, mask_kind="bool", scale=0.4, bool_mask=bm, sinks=s)
    samples = [(1, 3, 5), (0, 0, 0), (1, 0, 2), (0, 3, 4), (1, 3, 1)]
    o, l = fn_sampled(q, k, v, samples, mask_kind="bool", scale=0.4, bool_mask=bm, sinks=s)
    for n, (b, h, i) in enumerate(samples):
        np.testing.assert_allclose(o[n], full[b, h, i], rtol=1e-14, atol=1e-16)
        np.testing.assert_allclose(l[n], lf[b, h, i], rtol=1e-14)


PINS = [pin_single_key, pin_single_key_with_sink, pin_identical_keys_mean, pin_zero_scale_mean,
        pin_causal_row0, pin_decode_causal_sees_all, pin_gqa_equals_repeated_heads,
        pin_sink_limits, pin_empty_and_all_masked, pin_brute_force, pin_lse_consistency,
        pin_key_permutation, pin_batch_items_alone,
        pin_window_full_equals_causal, pin_window_of_one_sees_its_own_position,
        pin_window_identical_keys_mean, pin_window_rows_equal_one_query_calls, pin_window_errors,
        pin_additive_zero_equals_none, pin_additive_neg_inf_equals_bool, pin_additive_log_weights,
        pin_additive_constant_shift, pin_additive_broadcast]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.sdpa)


def test_sampled_oracle_equals_full():
    pin_sampled_equals_full(oracle.sdpa, oracle.sdpa_sampled)


# ------------------------------------------------------------------ paged caches

def build_paged(keys, values, bs, order):
    """Caches [num_blocks, Hkv, bs, d] holding keys/values [B, Hkv, N, d] in blocks of bs
    positions, block j of sequence s stored at order[s * per + j] (the layout of the
    pages' ``paged`` helper, filled here by hand); unused blocks hold NaN."""
    B, Hkv, N, d = keys.shape
    per = -(-N // bs)
    nblocks = max(order) + 1
    kc = np.full((nblocks, Hkv, bs, d), np.nan)
    vc = np.full((nblocks, Hkv, bs, values.shape[3]), np.nan)
    table = np.zeros((B, per), np.int32)
    for s in range(B):
        for j in range(per):
            blk = order[s * per + j]
            table[s, j] = blk
            n = min(bs, N - j * bs)
            kc[blk, :, :n] = keys[s, :, j * bs:j * bs + n]
            vc[blk, :, :n] = values[s, :, j * bs:j * bs + n]
    return kc, vc, table


def pin_paged_equals_contiguous(fn, fnp):
    """Shuffled blocks with a few unused ones: each sequence equals contiguous attention
    over its first len_s keys, bit for bit, with a causal mask (Lq > 1 aligned to that
    sequence's own length), a window and sinks ("nuvec-core 0.5.0 tests/fast.rs",
    paged_attention_equals_contiguous_attention, paged_windows_and_sinks_equal_contiguous_attention)."""
    B, Hq, Hkv, Lq, N, d, bs = 3, 4, 2, 3, 13, 8, 4
    keys = rand((B, Hkv, N, d), 231)
    vals = rand((B, Hkv, N, 5), 232)
    q = rand((B, Hq, Lq, d), 233)
    sinks = rand((Hq,), 234)
    per = -(-N // bs)
    order = list(np.random.RandomState(5).permutation(B * per + 3))
    kc, vc, table = build_paged(keys, vals, bs, order)
    lens = np.array([13, 4, 9], np.int32)
    for kw in [dict(mask_kind="causal"), dict(mask_kind="none", sinks=sinks),
               dict(mask_kind="causal", window=2, sinks=sinks)]:
        out, lse = fnp(q, kc, vc, table, lens, scale=0.3, **kw)
        for s in range(B):
            L = lens[s]
            o, l = fn(q[s:s + 1], keys[s:s + 1, :, :L], vals[s:s + 1, :, :L], scale=0.3, **kw)
            np.testing.assert_array_equal(out[s:s + 1], o)
            np.testing.assert_array_equal(lse[s:s + 1], l)
        assert np.all(np.isfinite(out))


def pin_paged_hostile_tables_are_clamped(fn, fnp):
    """Table entries past the block count or negative, and lengths past the capacity,
    are clamped: the keys are those of the clamped table, gathered here by hand."""
    nblocks, Hkv, bs, d = 3, 2, 4, 8
    kc = rand((nblocks, Hkv, bs, d), 241)
    vc = rand((nblocks, Hkv, bs, 6), 242)
    q = rand((2, 4, 1, d), 243)
    table = np.array([[1, 99, -5, 2], [2, 2**31 - 1, 0, -(2**31)]], np.int64)
    lens = np.array([100, 2**31 - 1], np.int64)        # capacity is 16 keys
    out, lse = fnp(q, kc, vc, table, lens, mask_kind="causal", scale=0.25)
    assert np.all(np.isfinite(out))
    picks = [[1, 2, 0, 2], [2, 2, 0, 0]]
    for s in range(2):
        K = np.concatenate([kc[b] for b in picks[s]], axis=1)[None]   # [1, Hkv, 16, d]
        V = np.concatenate([vc[b] for b in picks[s]], axis=1)[None]
        o, l = fn(q[s:s + 1], K, V, mask_kind="causal", scale=0.25)
        np.testing.assert_array_equal(out[s:s + 1], o)
        np.testing.assert_array_equal(lse[s:s + 1], l)


def pin_paged_block_order(fn, fnp):
    """Key j of a sequence comes from position j % bs of block table[s, j // bs]: with
    one key per block in reverse order, the keys come out reversed block by block."""
    nblocks, bs = 4, 2
    kc = np.zeros((nblocks, 1, bs, 2))
    vc = np.zeros((nblocks, 1, bs, 1))
    for blk in range(nblocks):
        for pos in range(bs):
            vc[blk, 0, pos, 0] = 10 * blk + pos       # a value naming its slot
    q = np.zeros((1, 1, 1, 2))
    table = np.array([[3, 1, 2, 0]])
    # W = 1 with causal and one query: the query sees only the last key, j = len - 1
    for L, want in [(1, 30), (2, 31), (3, 10), (4, 11), (5, 20), (8, 1)]:
        out, _ = fnp(q, kc, vc, table, np.array([L]), mask_kind="causal", scale=1.0, window=1)
        assert out[0, 0, 0, 0] == want, (L, out[0, 0, 0, 0], want)


def pin_paged_empty_sequences(fn, fnp):
    """A sequence of length 0 (or a negative length) gives zeros; lse is the sink, or -inf."""
    kc = rand((2, 1, 4, 8), 251)
    q = rand((2, 2, 1, 8), 252)
    sinks = rand((2,), 253)
    table = np.array([[0, 1], [1, 0]])
    for lens in [np.array([0, -3])]:
        out, lse = fnp(q, kc, kc, table, lens, mask_kind="causal", scale=0.5)
        np.testing.assert_array_equal(out, 0.0)
        assert np.all(lse == -np.inf)
        out, lse = fnp(q, kc, kc, table, lens, mask_kind="causal", scale=0.5, sinks=sinks)
        np.testing.assert_array_equal(out, 0.0)
        np.testing.assert_array_equal(lse[:, :, 0], np.broadcast_to(sinks, (2, 2)))
    with pytest.raises(ValueError):
        fnp(q, kc, kc, table, np.array([3, 3]), mask_kind="bool", scale=0.5)


def pin_paged_never_reads_hidden_blocks(fn, fnp):
    """Blocks wholly before every row's window, and every slot past a length, hold NaN:
    the result equals the one with those slots zeroed, and is finite ("nuvec-core 0.5.0
    tests/fast.rs", paged_windows_and_sinks_equal_contiguous_attention)."""
    B, Hq, Hkv, Lq, N, d, bs, W = 2, 4, 2, 2, 12, 4, 3, 4
    keys = rand((B, Hkv, N, d), 261)
    vals = rand((B, Hkv, N, 3), 262)
    q = rand((B, Hq, Lq, d), 263)
    kc, vc, table = build_paged(keys, vals, bs, list(range(B * (-(-N // bs)))))
    lens = np.array([12, 9])
    clean_k, clean_v = np.nan_to_num(kc), np.nan_to_num(vc)
    for s in range(B):
        first = lens[s] - Lq - W + 1          # the earliest row's band starts here
        for j in range(first // bs):
            kc[table[s, j]] = np.nan
            vc[table[s, j]] = np.nan
    a, la = fnp(q, kc, vc, table, lens, mask_kind="causal", scale=0.5, window=W)
    b, lb = fnp(q, clean_k, clean_v, table, lens, mask_kind="causal", scale=0.5, window=W)
    assert np.all(np.isfinite(a))
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


PAGED_PINS = [pin_paged_never_reads_hidden_blocks, pin_paged_equals_contiguous, pin_paged_hostile_tables_are_clamped, pin_paged_block_order,
              pin_paged_empty_sequences]


@pytest.mark.parametrize("pin", PAGED_PINS, ids=[p.__name__ for p in PAGED_PINS])
def test_oracle_paged_pin(pin):
    pin(oracle.sdpa, oracle.sdpa_paged)


# ------------------------------------------------------------------ planted mistakes

def _all_pins_pass(fn):
    try:
        for path in FIXTURES:
            pin_golden(fn, path)
        for pin in PINS:
            pin(fn)
        for pin in PAGED_PINS:
            pin(fn, osdpa.sdpa_paged)
    except (AssertionError, ValueError, IndexError, TypeError):
        return False
    return True


MUTANTS = {
    # query head h reads KV head h mod Hkv instead of h // g
    "kv_head_modulo": dict(_kv_head=lambda h, Hq, Hkv: h % Hkv),
    # causal aligned top-left (j <= i) instead of bottom-right
    "causal_top_left": dict(visible_mask=lambda mk, Lq, Lk, rows, bm=None, w=None: (
        np.arange(Lk)[None, :] <= np.asarray(rows)[:, None] if mk == "causal"
        else _orig_visible(mk, Lq, Lk, rows, bm, w))),
}


def _orig_visible(*a):
    return _ORIG["visible_mask"](*a)


_ORIG = {"visible_mask": osdpa.visible_mask, "_kv_head": osdpa._kv_head,
         "attend_rows": osdpa.attend_rows}


def _attend_sink_scaled(q_rows, k_head, v_head, vis, scale, sink=None, add=None):
    # the sink multiplied by scale like a score
    return _ORIG["attend_rows"](q_rows, k_head, v_head, vis, scale,
                                None if sink is None else sink * scale, add)


def _attend_no_sink_in_denominator(q_rows, k_head, v_head, vis, scale, sink=None, add=None):
    out, lse = _ORIG["attend_rows"](q_rows, k_head, v_head, vis, scale, None, add)
    return out, lse


def _attend_transposed_value(q_rows, k_head, v_head, vis, scale, sink=None, add=None):
    # values taken from the query side (a transposed operand)
    vv = v_head[::-1].copy()
    return _ORIG["attend_rows"](q_rows, k_head, vv, vis, scale, sink, add)


def _attend_no_scale(q_rows, k_head, v_head, vis, scale, sink=None, add=None):
    return _ORIG["attend_rows"](q_rows, k_head, v_head, vis, 1.0, sink, add)


def _attend_masked_as_finite(q_rows, k_head, v_head, vis, scale, sink=None, add=None):
    # the old finite sentinel: masked scores at -10000 instead of -inf
    s_vis = np.ones_like(vis, dtype=bool)
    kk = np.asarray(k_head, dtype=np.float64)
    out = []
    lse = []
    s = scale * (np.asarray(q_rows, dtype=np.float64) @ kk.T) if kk.shape[0] else np.zeros((len(q_rows), 0))
    if add is not None:
        s = s + add
    s = np.where(vis, s, -10000.0)
    m = s.max(axis=1) if kk.shape[0] else np.full(len(q_rows), -np.inf)
    if sink is not None:
        m = np.maximum(m, sink)
    mm = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - mm[:, None])
    z = p.sum(axis=1) + (np.exp(sink - mm) if sink is not None else 0.0)
    with np.errstate(all="ignore"):
        o = (p @ np.asarray(v_head, dtype=np.float64)) / z[:, None] if kk.shape[0] else np.zeros((len(q_rows), v_head.shape[1]))
    return np.nan_to_num(o), mm + np.log(z)


MUTANTS.update({
    "sink_scaled": dict(attend_rows=_attend_sink_scaled),
    "sink_dropped": dict(attend_rows=_attend_no_sink_in_denominator),
    "values_reversed": dict(attend_rows=_attend_transposed_value),
    "scale_dropped": dict(attend_rows=_attend_no_scale),
    "finite_mask_sentinel": dict(attend_rows=_attend_masked_as_finite),
})


def _visible_window_off_by_one(mk, Lq, Lk, rows, bm=None, w=None):
    # the band one key too wide: p - W <= j <= p
    vis = _orig_visible(mk, Lq, Lk, rows, bm, None)
    if w is not None:
        pos = np.asarray(rows)[:, None] + (Lk - Lq)
        vis &= np.arange(Lk)[None, :] >= pos - w
    return vis


def _visible_window_from_row(mk, Lq, Lk, rows, bm=None, w=None):
    # the window measured from the row index i instead of the absolute position p
    vis = _orig_visible(mk, Lq, Lk, rows, bm, None)
    if w is not None:
        vis &= np.arange(Lk)[None, :] > np.asarray(rows)[:, None] - w
    return vis


def _attend_add_scaled(q_rows, k_head, v_head, vis, scale, sink=None, add=None):
    # the additive mask multiplied by the scale like the scores
    return _ORIG["attend_rows"](q_rows, k_head, v_head, vis, scale, sink,
                                None if add is None else add * scale)


def _attend_add_dropped(q_rows, k_head, v_head, vis, scale, sink=None, add=None):
    return _ORIG["attend_rows"](q_rows, k_head, v_head, vis, scale, sink, None)


def _add_rows_first_slice(add_mask, b, h, rows):
    # every batch item and head reads the mask's first slice
    return None if add_mask is None else np.asarray(add_mask)[0, 0][rows].astype(np.float64)


def _gather_swapped(cache, block_table, seq_lens, s):
    # block and position swapped: block table[s, j % bs], position j // bs
    cache = np.asarray(cache)
    table = np.asarray(block_table, dtype=np.int64)
    nblocks, Hkv, bs, d = cache.shape
    L = int(min(max(int(seq_lens[s]), 0), table.shape[1] * bs))
    j = np.arange(L)
    ids = np.clip(table[s, np.minimum(j % bs, table.shape[1] - 1)], 0, nblocks - 1)
    return cache[ids, :, np.minimum(j // bs, bs - 1), :].transpose(1, 0, 2)


def _gather_unclamped_len(cache, block_table, seq_lens, s):
    # the length taken as given, past the table's capacity (ids still clamped)
    cache = np.asarray(cache)
    table = np.asarray(block_table, dtype=np.int64)
    nblocks, Hkv, bs, d = cache.shape
    L = max(int(seq_lens[s]), 0)
    j = np.arange(min(L, 10**6))
    ids = np.clip(table[s, np.minimum(j // bs, table.shape[1] - 1)], 0, nblocks - 1)
    return cache[ids, :, j % bs, :].transpose(1, 0, 2)


MUTANTS.update({
    "window_off_by_one": dict(visible_mask=_visible_window_off_by_one),
    "window_from_row_index": dict(visible_mask=_visible_window_from_row),
    "window_ignored": dict(visible_mask=lambda mk, Lq, Lk, rows, bm=None, w=None:
                           _orig_visible(mk, Lq, Lk, rows, bm, None)),
    "additive_scaled": dict(attend_rows=_attend_add_scaled),
    "additive_dropped": dict(attend_rows=_attend_add_dropped),
    "additive_first_slice_only": dict(_add_rows=_add_rows_first_slice),
    "paged_block_position_swapped": dict(paged_gather=_gather_swapped),
    "paged_length_unclamped": dict(paged_gather=_gather_unclamped_len),
})


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    for attr, fn in MUTANTS[name].items():
        monkeypatch.setattr(osdpa, attr, fn)
    assert not _all_pins_pass(osdpa.sdpa), f"no pin caught the planted mistake {name}"


def test_unmutated_oracle_passes_every_pin():
    assert _all_pins_pass(osdpa.sdpa)

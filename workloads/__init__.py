"""Seeded synthetic inputs for the fused attention forward.

This module is the one piece of code that both the CUDA path's tests/bench and the
f64 oracle's tests use.  It holds no attention arithmetic: it draws numbers, casts
them to the storage dtype, and describes the workloads by their shapes.

Generator
---------
The 64-bit linear congruential generator of the seeded test helper in
"lattice-inference 0.4.0 src/attention/flash.rs" (its test module's ``Lcg``):

    state <- state * 6364136223846793005 + 1   (mod 2**64)
    u32    = state >> 32

drawn in blocks with jump-ahead so that tens of millions of values come out in
numpy vector operations, bit-identical to the sequential recurrence.  From it:

* ``uniform``: u32 / 2**32, in [0, 1)
* ``normal``:  Box-Muller on consecutive pairs (u1, u2):
               r = sqrt(-2 ln(1 - u1)); z0 = r cos(2 pi u2), z1 = r sin(2 pi u2)
* ``bernoulli(p)``: uniform < p

Values are produced in f64, cast to f32 (round to nearest even), and from there to
f16 (numpy, RNE) or bf16 (RNE on the f32 bits).  Both the oracle and the GPU read
the same stored values.  bf16 is held as its uint16 bit pattern.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = [
    "Stream", "Case", "DTYPE_CODES", "MASK_CODES", "to_storage", "widen",
    "make_inputs", "tiny_f32_causal", "prefill_bf16_gqa", "decode_f16_long_kv",
    "prefill_f16_boolmask_sinks", "sweep_bf16", "named_workloads",
]

_A = np.uint64(6364136223846793005)
_C = np.uint64(1)
_BLOCK = 1 << 20

# Jump-ahead tables for one block: state_{n+i} = P[i] * state_n + Q[i]  (mod 2**64).
_P = np.empty(_BLOCK, dtype=np.uint64)
_Q = np.empty(_BLOCK, dtype=np.uint64)
_P[0], _Q[0] = 1, 0
with np.errstate(over="ignore"):
    _m = 1
    _P[1], _Q[1] = _A, _C
    _m = 2
    while _m < _BLOCK:
        pm, qm = _P[_m - 1] * _A, _Q[_m - 1] * _A + _C  # a^m and c_m
        _P[_m:2 * _m] = _P[:_m] * pm
        _Q[_m:2 * _m] = _P[:_m] * qm + _Q[:_m]
        _m *= 2
    _PB = _P[_BLOCK - 1] * _A            # a^BLOCK
    _QB = _Q[_BLOCK - 1] * _A + _C       # c_BLOCK


class Stream:
    """The LCG above, seeded; every draw continues where the last one stopped."""

    def __init__(self, seed: int):
        self.state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)

    def u32(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.uint32)
        s = self.state
        pos = 0
        with np.errstate(over="ignore"):
            while pos < n:
                take = min(_BLOCK, n - pos)
                # states after 1..take steps
                st = _P[1:take + 1] * s + _Q[1:take + 1] if take < _BLOCK else None
                if st is None:
                    st = np.empty(_BLOCK, dtype=np.uint64)
                    st[:-1] = _P[1:] * s + _Q[1:]
                    st[-1] = _PB * s + _QB
                out[pos:pos + take] = (st >> np.uint64(32)).astype(np.uint32)
                s = st[take - 1]
                pos += take
        self.state = np.uint64(s)
        return out

    def uniform(self, n: int) -> np.ndarray:
        return self.u32(n).astype(np.float64) * (1.0 / 4294967296.0)

    def normal(self, n: int) -> np.ndarray:
        pairs = (n + 1) // 2
        u = self.uniform(2 * pairs).reshape(pairs, 2)
        r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
        t = 2.0 * math.pi * u[:, 1]
        z = np.empty((pairs, 2), dtype=np.float64)
        z[:, 0] = r * np.cos(t)
        z[:, 1] = r * np.sin(t)
        return z.reshape(-1)[:n]

    def bernoulli(self, n: int, p: float) -> np.ndarray:
        return self.uniform(n) < p


# ----------------------------------------------------------------------------- dtypes

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}
MASK_CODES = {"none": 0, "causal": 1, "bool": 2}
ELT_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


def _f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    b = x32.astype(np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(x32)
    rounded = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """f64 values -> the stored array (float32, float16, or bf16 bits as uint16)."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return x32
    if dtype == "f16":
        return x32.astype(np.float16)
    if dtype == "bf16":
        return _f32_to_bf16_bits(x32)
    raise ValueError(dtype)


def widen(stored: np.ndarray, dtype: str) -> np.ndarray:
    """The stored array -> exact f64 values."""
    if dtype in ("f32", "f16"):
        return np.asarray(stored).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(stored, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------- cases

@dataclasses.dataclass(frozen=True)
class Case:
    """One attention call: shapes, dtype, mask kind, sinks, value recipe and seed."""
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    d: int
    dv: int
    dtype: str = "bf16"
    mask: str = "none"        # none | causal | bool
    sinks: bool = False
    scale: Optional[float] = None   # None -> 1/sqrt(d), as f32
    values: str = "u0.25"     # u0.25: U[0,0.25) | u2: U[0,0.25)*8 | n0.5: 0.5*N(0,1)
    mask_p: float = 0.9       # Bernoulli(p) of a true mask entry
    seed: int = 0
    name: str = ""

    @property
    def scale_f32(self) -> float:
        s = self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)
        return float(np.float32(s))

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    def numel(self):
        return dict(q=self.B * self.Hq * self.Lq * self.d,
                    k=self.B * self.Hkv * self.Lk * self.d,
                    v=self.B * self.Hkv * self.Lk * self.dv,
                    out=self.B * self.Hq * self.Lq * self.dv,
                    lse=self.B * self.Hq * self.Lq)

    def with_(self, **kw) -> "Case":
        return dataclasses.replace(self, **kw)


def _draw(stream: Stream, n: int, recipe: str) -> np.ndarray:
    if recipe == "u0.25":
        return stream.uniform(n) / 4.0
    if recipe == "u2":
        return stream.uniform(n) / 4.0 * 8.0
    if recipe == "n0.5":
        return 0.5 * stream.normal(n)
    if recipe == "n1":
        return stream.normal(n)
    raise ValueError(recipe)


def make_inputs(c: Case) -> dict:
    """Draw Q, K, V, sinks, mask in that order from one stream seeded with c.seed.

    Returns stored arrays: q [B,Hq,Lq,d], k [B,Hkv,Lk,d], v [B,Hkv,Lk,dv] in the
    storage dtype, sinks [Hq] (same dtype, N(0,1)) or None, mask [Lq,Lk] uint8
    (1 = attend; Bernoulli(mask_p) with the diagonal j = i forced to 1) or None.
    """
    s = Stream(c.seed)
    n = c.numel()
    q = to_storage(_draw(s, n["q"], c.values), c.dtype).reshape(c.B, c.Hq, c.Lq, c.d)
    k = to_storage(_draw(s, n["k"], c.values), c.dtype).reshape(c.B, c.Hkv, c.Lk, c.d)
    v = to_storage(_draw(s, n["v"], c.values), c.dtype).reshape(c.B, c.Hkv, c.Lk, c.dv)
    sinks = to_storage(s.normal(c.Hq), c.dtype) if c.sinks else None
    mask = None
    if c.mask == "bool":
        m = s.bernoulli(c.Lq * c.Lk, c.mask_p).reshape(c.Lq, c.Lk)
        r = np.arange(min(c.Lq, c.Lk))
        m[r, r] = True
        mask = m.astype(np.uint8)
    return dict(q=q, k=k, v=v, sinks=sinks, mask=mask)


# ----------------------------------------------------------------------------- workloads

def tiny_f32_causal() -> Case:
    """Tiny f32 causal case: 1x2/1 heads, 16 queries and keys, head 64."""
    return Case(1, 2, 1, 16, 16, 64, 64, "f32", "causal", False, None, "u0.25", seed=0,
                name="tiny_f32_causal_b1_h2x1_l16_d64")


def prefill_bf16_gqa() -> Case:
    """Prefill bf16 GQA 32/8, B=2, Lq=Lk=4096, head 128, causal."""
    return Case(2, 32, 8, 4096, 4096, 128, 128, "bf16", "causal", False, None, "n0.5",
                seed=1, name="prefill_bf16_gqa_b2_h32x8_l4096_d128_causal")


def decode_f16_long_kv() -> Case:
    """Decode f16 GQA 32/4, B=8, one query over 32769 keys, head 128, causal, sinks."""
    return Case(8, 32, 4, 1, 32769, 128, 128, "f16", "causal", True, None, "u2",
                seed=2, name="decode_f16_b8_h32x4_lk32769_d128_sinks")


def prefill_f16_boolmask_sinks() -> Case:
    """Prefill f16 16/2 heads, Lq=1024, Lk=1801, head 256, Bernoulli(0.9) mask, sinks."""
    return Case(1, 16, 2, 1024, 1801, 256, 256, "f16", "bool", True, None, "n0.5",
                seed=3, name="prefill_f16_b1_h16x2_lq1024_lk1801_d256_bool_sinks")


def sweep_bf16() -> list:
    """The 108-case bf16 head-shape sweep, in enumeration order (d,dv) -> heads -> Lq -> Lk.

    Case n is causal when n is even, unmasked when odd; B = 1 + (Lk mod 2);
    values U[0,0.25)*8; scale 1/sqrt(d); no sinks; seed 5000 + n.
    """
    out = []
    n = 0
    for d, dv in [(64, 64), (96, 64), (192, 128), (256, 256)]:
        for hq, hkv in [(16, 2), (8, 8), (32, 8)]:
            for lq in [1, 9, 342]:
                for lk in [lq, lq + 777, 8193]:
                    out.append(Case(1 + (lk % 2), hq, hkv, lq, lk, d, dv, "bf16",
                                    "causal" if n % 2 == 0 else "none", False, None, "u2",
                                    seed=5000 + n,
                                    name=f"sweep{n:03d}_d{d}x{dv}_h{hq}x{hkv}_lq{lq}_lk{lk}"))
                    n += 1
    return out


def named_workloads() -> dict:
    return {c.name: c for c in [tiny_f32_causal(), prefill_bf16_gqa(), decode_f16_long_kv(),
                                prefill_f16_boolmask_sinks()]}

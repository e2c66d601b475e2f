"""f64 oracle: scaled-dot-product attention written out from its definition.

TEST INFRASTRUCTURE ONLY (tests, the smoke check and the CPU-baseline leg of the
bench).  Plain numpy, float64 throughout, one head at a time, the full score matrix
materialised.  No blocking, no online softmax, no split over keys: the fused kernels
reach this same result in another order, and this file is the definition they are
checked against.

Sources (page titles and the test or function each step follows)
-----------------------------------------------------------------
* The formula, one head: ``softmax(scale * q k^T) v`` with the row maximum subtracted
  before the exponential and a causal row ``i`` seeing its first ``i + Lk - Lq + 1``
  keys -- "nuvec-core 0.5.0 tests/fast.rs", test
  ``attention_fallback_matches_a_direct_formula``.
* The materialised reference (scores, mask, softmax, weighted sum of V) --
  "lattice-inference 0.4.0 src/attention/flash.rs", test helper
  ``reference_attention_head``.
* Masked keys carry a score of minus infinity, so their weight is exactly zero, and a
  row with no visible key yields zeros, never NaN -- same page,
  ``run_tiled_attention_head`` and tests ``masked_key_below_finite_sentinel_does_not_dominate``,
  ``all_masked_row_yields_zero_output_not_nan``.
* Grouped-query heads: query head ``h`` reads key/value head ``h / (Hq / Hkv)`` --
  same page, ``kv_head_index``.
* Boolean mask ``[Lq, Lk]``, true = attend, shared by every batch item and head;
  sinks are one value per query head, in the input dtype -- "nuvec-core 0.5.0
  tests/fast.rs", the fused-attention tests building ``bmask`` and ``sinks``.
* No keys give zeros (also with a causal mask and with sinks) -- same page, test
  ``window_errors_empty_inputs_and_full_windows``.
* Sliding window (causal only): the query at absolute position ``p = i + Lk - Lq`` sees
  key ``j`` iff ``p - W < j <= p``; a window of 0, or a window with any mask kind but
  causal, is an error -- same page, ``band`` / ``window_mask`` (the window as an explicit
  boolean mask) and ``window_errors_empty_inputs_and_full_windows``.
* Additive mask: a float array of shape ``[1|B, 1|Hq, Lq, Lk]`` in the input dtype,
  added to the scaled scores (``softmax(scale * q k^T + mask)``); it is a mask kind of its
  own, beside none, causal and boolean -- same page, ``attention_kernels_match_the_fallback``
  (``amask`` of shape ``[1, hq, lq, lk]``, the "additive" mask).
* Paged keys and values: caches ``[num_blocks, Hkv, block_size, d]`` and a block table
  ``[B, max_blocks]``; key ``j`` of sequence ``s`` is position ``j % block_size`` of block
  ``table[s, j // block_size]``, and sequence ``s`` has ``seq_lens[s]`` keys; the result
  equals contiguous attention over the gathered keys with the same options (causal
  bottom-right against that sequence's length, windows, sinks) -- same page, ``paged``
  and ``paged_attention_equals_contiguous_attention``,
  ``paged_windows_and_sinks_equal_contiguous_attention``.

Readings where the pages are silent
-----------------------------------
* A sink is one extra logit per query head in *score space* (it is not multiplied by
  ``scale``) whose value row is zero: it only adds ``exp(sink - m)`` to the
  denominator.  This is the one reading under which "no keys give zeros, with sinks
  too" holds.
* ``lse`` is the natural log of the full denominator, sink included, over scaled
  scores: ``lse = m + ln Z``.  A row with no visible key and no sink has
  ``lse = -inf``; with a sink and no visible key, ``lse = sink`` and the output is 0.
* Causal alignment is bottom-right for any ``Lq`` and ``Lk``: row ``i`` sees key ``j``
  iff ``j <= i + Lk - Lq``.  With ``Lq > Lk`` the first rows see no key (zeros).
* ``scale`` is the f32 value the caller passes, widened exactly.
* An additive mask is not multiplied by ``scale``, and entries of ``-inf`` hide a key
  exactly like a false boolean entry (a row whose every key is hidden gives zeros).
* Hostile paged inputs ("nuvec-core 0.5.0 tests/fast.rs",
  ``paged_attention_clamps_hostile_tables_and_lengths`` asks only for finite output equal
  to the CPU fallback's) are clamped: a length to ``[0, max_blocks * block_size]``, a
  block id to ``[0, num_blocks - 1]``.
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

__all__ = ["visible_mask", "attend_rows", "sdpa", "sdpa_sampled", "sdpa_paged", "paged_gather"]

MASK_KINDS = ("none", "causal", "bool", "add")


def check_window(mask_kind: str, window) -> None:
    """A window needs the causal mask and is at least 1 ("nuvec-core 0.5.0 tests/fast.rs",
    window_errors_empty_inputs_and_full_windows)."""
    if window is None:
        return
    if int(window) != window or window < 1:
        raise ValueError(f"window must be a positive integer, got {window!r}")
    if mask_kind != "causal":
        raise ValueError("a window needs the causal mask")


def visible_mask(mask_kind: str, Lq: int, Lk: int, rows: np.ndarray,
                 bool_mask: Optional[np.ndarray] = None, window: Optional[int] = None) -> np.ndarray:
    """Which keys each query row in ``rows`` may attend to: bool ``[len(rows), Lk]``."""
    check_window(mask_kind, window)
    rows = np.asarray(rows, dtype=np.int64)
    j = np.arange(Lk, dtype=np.int64)
    if mask_kind in ("none", "add"):
        return np.ones((rows.size, Lk), dtype=bool)
    if mask_kind == "causal":
        pos = rows[:, None] + (Lk - Lq)          # absolute position of each query
        vis = j[None, :] <= pos
        if window is not None:
            vis &= j[None, :] > pos - int(window)
        return vis
    if mask_kind == "bool":
        if bool_mask is None:
            raise ValueError("bool mask kind needs a mask")
        return np.asarray(bool_mask)[rows, :] != 0
    raise ValueError(f"unknown mask kind {mask_kind!r}")


def attend_rows(q_rows: np.ndarray, k_head: np.ndarray, v_head: np.ndarray,
                vis: np.ndarray, scale: float, sink: Optional[float] = None,
                add: Optional[np.ndarray] = None):
    """Attention of some query rows of one head over all keys of its KV head.

    q_rows [n, d], k_head [Lk, d], v_head [Lk, dv] (f64); vis [n, Lk] bool;
    scale, sink as f64 (sink None = no sink); add [n, Lk] f64 added to the scaled
    scores, or None.  Returns (out [n, dv], lse [n]).
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k_head = np.asarray(k_head, dtype=np.float64)
    v_head = np.asarray(v_head, dtype=np.float64)
    n, Lk, dv = q_rows.shape[0], k_head.shape[0], v_head.shape[1]
    # The sums run over visible keys only: a key that no row sees takes no part at all,
    # whatever its stored values (the pages fill such never-read cache blocks with NaN).
    seen = np.asarray(vis).any(axis=0)
    if not seen.all():
        k_head = np.where(seen[:, None], k_head, 0.0)
        v_head = np.where(seen[:, None], v_head, 0.0)
    # scores s_ij = scale * <q_i, k_j> (+ mask_ij), minus infinity where key j is not visible
    s = np.float64(scale) * (q_rows @ k_head.T) if Lk else np.zeros((n, 0))
    if add is not None:
        s = s + np.asarray(add, dtype=np.float64)
    vis = vis & (s > -np.inf)
    s = np.where(vis, s, -np.inf)
    # row maximum over the visible scores and the sink logit
    m = s.max(axis=1) if Lk else np.full(n, -np.inf)
    if sink is not None:
        m = np.maximum(m, np.float64(sink))
    empty = m == -np.inf
    m_safe = np.where(empty, 0.0, m)
    # unnormalised weights and the denominator
    p = np.where(vis, np.exp(s - m_safe[:, None]), 0.0)
    z = p.sum(axis=1)
    if sink is not None:
        z = z + np.exp(np.float64(sink) - m_safe)
    with np.errstate(divide="ignore", invalid="ignore"):
        out = (p @ v_head) / z[:, None] if Lk else np.zeros((n, dv))
        lse = m + np.log(z)
    out = np.where(empty[:, None], 0.0, out)
    lse = np.where(empty, -np.inf, lse)
    return out, lse


def _kv_head(h: int, Hq: int, Hkv: int) -> int:
    return h // (Hq // Hkv)


def _check(q, k, v):
    B, Hq, Lq, d = q.shape
    Bk, Hkv, Lk, dk = k.shape
    if v.shape[:3] != (B, Hkv, Lk) or Bk != B or dk != d or Hkv == 0 or Hq % Hkv:
        raise ValueError(f"bad shapes q{q.shape} k{k.shape} v{v.shape}")
    return B, Hq, Hkv, Lq, Lk, d, v.shape[3]


def _add_rows(add_mask, b, h, rows):
    """The additive mask's rows for batch item b and query head h ([1|B, 1|Hq] broadcast)."""
    if add_mask is None:
        return None
    a = np.asarray(add_mask)
    return np.asarray(a[b if a.shape[0] > 1 else 0, h if a.shape[1] > 1 else 0][rows],
                      dtype=np.float64)


def _check_add(mask_kind, add_mask, B, Hq, Lq, Lk):
    if mask_kind == "add":
        if add_mask is None:
            raise ValueError("the additive mask kind needs a mask")
        a = np.asarray(add_mask)
        if a.ndim != 4 or a.shape[0] not in (1, B) or a.shape[1] not in (1, Hq) or a.shape[2:] != (Lq, Lk):
            raise ValueError(f"additive mask shape {a.shape} is not [1|B, 1|Hq, Lq, Lk]")
        return add_mask
    return None


def sdpa(q, k, v, *, mask_kind: str, scale: float, bool_mask=None, sinks=None, window=None,
         add_mask=None):
    """Full attention forward in f64.

    q [B,Hq,Lq,d], k [B,Hkv,Lk,d], v [B,Hkv,Lk,dv] (any real dtype, widened to f64);
    mask_kind in {"none","causal","bool","add"}; bool_mask [Lq,Lk] (nonzero = attend);
    add_mask [1|B, 1|Hq, Lq, Lk] (mask kind "add"); window W >= 1 (causal only) or None;
    sinks [Hq] or None.  Returns (out [B,Hq,Lq,dv] f64, lse [B,Hq,Lq] f64).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, Hkv, Lq, Lk, d, dv = _check(q, k, v)
    add_mask = _check_add(mask_kind, add_mask, B, Hq, Lq, Lk)
    out = np.zeros((B, Hq, Lq, dv))
    lse = np.full((B, Hq, Lq), -np.inf)
    rows = np.arange(Lq)
    vis = visible_mask(mask_kind, Lq, Lk, rows, bool_mask, window)
    for b in range(B):
        for h in range(Hq):
            hk = _kv_head(h, Hq, Hkv)
            sink = None if sinks is None else float(np.asarray(sinks, dtype=np.float64)[h])
            out[b, h], lse[b, h] = attend_rows(q[b, h], k[b, hk], v[b, hk], vis, scale, sink,
                                               _add_rows(add_mask, b, h, rows))
    return out, lse


def sdpa_sampled(q, k, v, samples: Iterable, *, mask_kind: str, scale: float,
                 bool_mask=None, sinks=None, window=None, add_mask=None):
    """The same definition at selected outputs only: ``samples`` is a list of
    (b, h, i).  Returns (out [n, dv], lse [n]) in the order of ``samples``.
    Used where the full problem is too large for the oracle to finish in seconds."""
    samples = list(samples)
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    dv = v.shape[3]
    add_mask = _check_add(mask_kind, add_mask, B, Hq, Lq, Lk)
    out = np.zeros((len(samples), dv))
    lse = np.zeros(len(samples))
    groups = {}
    for n, (b, h, i) in enumerate(samples):
        groups.setdefault((b, h), []).append((n, i))
    for (b, h), lst in groups.items():
        idx = np.array([n for n, _ in lst])
        rows = np.array([i for _, i in lst])
        hk = _kv_head(h, Hq, Hkv)
        vis = visible_mask(mask_kind, Lq, Lk, rows, bool_mask, window)
        sink = None if sinks is None else float(np.asarray(sinks, dtype=np.float64)[h])
        o, l = attend_rows(np.asarray(q[b, h][rows], dtype=np.float64),
                           np.asarray(k[b, hk], dtype=np.float64),
                           np.asarray(v[b, hk], dtype=np.float64), vis, scale, sink,
                           _add_rows(add_mask, b, h, rows))
        out[idx], lse[idx] = o, l
    return out, lse


def paged_gather(cache, block_table, seq_lens, s: int):
    """The keys (or values) of sequence ``s`` from a paged cache, in key order:
    ``[Hkv, L_s, d]``.  Key ``j`` is position ``j % block_size`` of block
    ``block_table[s, j // block_size]``; the length and the block ids are clamped into
    range (a length to ``[0, max_blocks * block_size]``, an id to ``[0, num_blocks - 1]``)."""
    cache = np.asarray(cache)
    table = np.asarray(block_table, dtype=np.int64)
    nblocks, Hkv, bs, d = cache.shape
    cap = table.shape[1] * bs
    L = int(min(max(int(seq_lens[s]), 0), cap))
    j = np.arange(L, dtype=np.int64)
    ids = np.clip(table[s, j // bs], 0, nblocks - 1)
    return cache[ids, :, j % bs, :].transpose(1, 0, 2)   # [L, Hkv, d] -> [Hkv, L, d]


def sdpa_paged(q, k_cache, v_cache, block_table, seq_lens, *, mask_kind: str, scale: float,
               sinks=None, window=None):
    """Attention over paged caches: for each sequence s, the plain definition (``sdpa``)
    over its gathered keys and values, with Lk = its (clamped) length.  mask_kind is
    "none" or "causal" (a boolean or additive mask is an error, as in the pages' paged
    tests).  Returns (out [B,Hq,Lq,dv], lse [B,Hq,Lq])."""
    if mask_kind not in ("none", "causal"):
        raise ValueError("paged attention takes no mask array")
    q = np.asarray(q, dtype=np.float64)
    B, Hq, Lq, d = q.shape
    dv = np.asarray(v_cache).shape[3]
    if np.asarray(block_table).shape[0] != B or np.asarray(seq_lens).shape[0] != B:
        raise ValueError("block table and lengths need one row per sequence")
    out = np.zeros((B, Hq, Lq, dv))
    lse = np.full((B, Hq, Lq), -np.inf)
    for s in range(B):
        k = paged_gather(k_cache, block_table, seq_lens, s)[None]
        v = paged_gather(v_cache, block_table, seq_lens, s)[None]
        out[s:s + 1], lse[s:s + 1] = sdpa(q[s:s + 1], k, v, mask_kind=mask_kind, scale=scale,
                                          sinks=sinks, window=window)
    return out, lse

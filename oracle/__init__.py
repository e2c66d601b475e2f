"""The f64 CPU oracle for the fused attention forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The library (``scaled_dot_product_nv_gb300``) never does:
it has no CPU path at all.

The oracle is the plain definition of scaled-dot-product attention: it materialises
the full score matrix of each head in float64 with numpy and shares no code with the
CUDA kernels.  See ``oracle/attention.py`` for the definition, its sources on the pages,
and the readings taken where the pages are silent.  Every function here is pinned by
``tests/test_oracle_pins.py`` (closed forms, a worked example printed on the pages,
invariants and a high-precision brute force) -- no function is "parity unpinned".
"""
from .attention import (attend_rows, paged_gather, sdpa, sdpa_paged, sdpa_sampled,  # noqa: F401
                        visible_mask)

"""Plain, slow CPU oracle for MARBLE's exact masked ring-attention hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call this package:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.
It shares no code with the CUDA implementation; the only shared inputs are the seeded
generators in ``workloads``.

Modules
  mask       -- the per-pair mask predicate (MARBLE post, section 01, the ``mask_mod`` code)
  plan       -- block summaries, tile classification, PTRR, token order, per-step lists,
                needed-KV index (MARBLE post, section 03 "Block classification", "PTRR";
                section 04 "Sparse all-to-all", "Layout transforms")
  attention  -- fp64 softmax(QK^T/sqrt(d) + M)V, its LSE and gradients (Libra Eq. 1)
  ring       -- fp64 ring simulation carrying (O, m, l) across KV shards (RingAttention
                tutorial, "The Online Softmax Formulation"; ring simulation page)
  counts     -- legal-pair counters (Libra Eq. 2 / Eq. 6 style workload counts)

Every function here is pinned by tests in ``tests/test_oracle_*.py`` to values the pages
print, closed forms, invariants or brute force.
"""
from . import mask, plan, attention, ring, counts  # noqa: F401

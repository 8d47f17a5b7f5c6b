"""fp64 CPU oracle for context-parallel exact softmax attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA library never calls
it and shares no code with it: no kernels, headers, helpers, tables or pre/post-processing.

Contents (``oracle.usp``):

* ``attention``: plain softmax attention with a natural-log log-sum-exp, the output pair
  ``(out, lse)`` that each ring step produces (diffusers PR #12693 "Add Unified Sequence Parallel
  attention", the TemplatedRingAttention forward quoted in the LSE-shape discussion; HF docs
  "Context parallelism", section Ring Attention).
* ``merge``: the ring step's LSE-weighted combine in the pages' own sigmoid / log-sigmoid form
  (same PR, same snippet).
* ``seq2head`` / ``head2seq``: the Ulysses all-to-all as index loops over per-rank buffers
  (HF docs "Context parallelism", section Ulysses Attention; diffusers issue #12706 "UAA: Ulysses
  Anything Attention" for uneven per-rank lengths).
* ``ring_positions``: contiguous / zigzag / stripe chunk orderings (sourcepulse USP summary,
  "Highlighted Details" and "Limitations & Caveats"; the pages name them without defining them,
  so the readings are stated in each docstring).
* ``usp_attention``: the whole method (Unified SP: Ulysses all-to-all inside each ring group, ring
  loop with merges, reverse all-to-all; HF docs "Context parallelism", section Unified Attention).

Every function here is pinned by ``tests/test_oracle_*.py`` against something other than itself
(brute force, torch's fp64 SDPA, closed forms, invariants, the split sizes the workloads print).
"""
from .usp import (  # noqa: F401
    NEG_INF,
    attention,
    attention_rows,
    default_split,
    head2seq,
    merge,
    ring_positions,
    seq2head,
    usp_attention,
    virtual_rank_lengths,
    widen_bf16,
)

"""CPU oracle for shared-prefix tree attention (TEST INFRASTRUCTURE ONLY).

This package is the slow, plain, fp64 NumPy statement of what the GPU path
computes.  It exists to check the CUDA library, never to stand in for it: only
the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA path; both take
their inputs from the separate ``workloads`` module.

Sources (three web pages about one Megatron-LM feature):

* "[ENHANCEMENT] Shared-prefix training with context parallelism for exact
  agent trajectories" (issue #7386) -- "Describe the solution you'd like"
  (DFS segments with parent/depth metadata; every query run attends to its
  own ancestor path only; only the sampled-edge sources are projected, and
  each sampled action has a single loss owner) and "Describe alternatives you've
  considered" (independent exact-call sequences are the correctness
  reference).
* "feat(hybrid): add opt-in shared-prefix attention and Mamba execution"
  (#7914) -- introduction (the prompt's K/V is reused, each suffix is
  causally isolated, the backward sums the branches' contributions into
  their shared prefix).
* "TreePackedSeqParams" draft (PR #7387) -- "Summary" (DFS segments, ancestor
  relationships, each query segment attending causally over its ancestors,
  edge-source selection before the vocabulary projection, rejection of
  unsupported input).

Modules: ``tree`` (validation, ancestry, brute-force visibility), ``plan``
(per-query-tile ancestor KV ranges and the backward KV-block table, derived
independently of the C++ planner), ``attention`` (leaf-unrolled forward and
backward, plus the dense tree-mask route for tiny trees), ``gather``
(sampled-edge selection and its adjoint), ``lm_head`` (log-probability of each
sampled action through the vocabulary projection, and its backward),
``fragments`` (bounded fragment planning with repeated ancestors).

Parity status: every function here is pinned by ``tests/test_oracle.py``
against brute force, library routines, finite differences or invariants; no
function is "parity unpinned".  ``tests/test_oracle_mutants.py`` plants
mistakes in a copy of this package and checks that some pin fails for each.
"""
from . import tree, plan, attention, gather, lm_head, fragments  # noqa: F401

"""Float64 CPU oracle for anchor-masked block-sparse cross-attention.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports this package: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` may call it. It shares no code with the CUDA path; the
two meet only in the seeded input draws of ``workloads``.

What it computes, and the passages it follows:

* ``attention.forward`` / ``attention.backward``: the plain definition of
  exact masked cross-attention. Each draft block j (anchor a_j) attends to
  the context keys [0, a_j) of its sample plus the B keys of its own draft
  tokens; the output is softmax(scale * q k^T) v and the backward is the
  analytic softmax gradient. The Split-KV paper (arXiv:2611.05926, abstract)
  describes this as cross-attention of compact draft queries over a longer
  context under a block-sparse mask; the rit.work article on Split-KV
  (section "Split-KV двигает запросы, а не ключи и значения") states that the
  split computation reproduces the single-device result exactly, which is
  why the oracle is the unsplit definition and not the split algorithm.
* ``attention.partial_forward`` / ``attention.merge``: attention restricted to
  a key subset, plus the log-sum-exp merge of such partials. Used only to
  check that any split merges back to ``forward`` (the exactness property).
* ``projection``: the drafter layer's input projections (Q, K, V of the
  draft tokens and K, V of the context through one stacked weight) and
  output projection around the attention, forward and backward, as plain
  float64 matrix products; ``layer_forward`` / ``layer_backward`` compose
  them with ``attention``. The pages name the layer (diffusion drafters whose
  draft blocks cross-attend to the target's context) but not its
  projections; the plain linear maps are the reading taken.
* ``plan``: the realized-attention cost of a KV chunk and the
  longest-processing-time-first assignment (sort by cost, most expensive
  first; give each to the least-loaded worker) that the abstract and the
  rit.work article (paragraph on load imbalance from anchor sampling)
  describe, with the deterministic tie-breaks this library fixes.

The pages print no worked example, formula or table, so every function here
is pinned by mathematics instead: brute force on tiny inputs, a library
special case, finite differences, closed forms, invariants and Graham's
bound (see ``tests/test_oracle_*.py``).
"""
from . import attention, plan, projection  # noqa: F401

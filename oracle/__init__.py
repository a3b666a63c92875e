"""Reference oracle for the KV-cache eviction engine.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.

It is a plain, slow, float64 restatement of what the four pages define:

* ``attention``  -- softmax decode / window attention
  (H2O Guide, "The Existence of Heavy Hitters").
* ``h2o``        -- cumulative attention scores with GQA aggregation
  (H2O Guide, "Formulating Cumulative Attention Scores"; FAQ on GQA).
* ``snapkv``     -- observation-window ring, fresh window sums, max-pool
  (SnapKV, "How it works", "On the adaptation").
* ``dropkv``     -- residual-output scores, Lemma 1, greedy bound
  (DropKV explainer, Lemma 1 paragraph, bound paragraph, worked example).
* ``select``     -- budgeted bottom-k outside the recent window
  (H2O Guide, "Step-by-Step Eviction Lifecycle"; SnapKV tie-breaking).
* ``paged``      -- token table, 16-token blocks, reclamation planning
  (vToken review, Sec. 2 Eq. (1), Sec. 3.2, Sec. 3.3 Stages 1-3, Eq. (2)).
* ``engine``     -- the per-decode-step order of operations across lanes.

Every function names the passage it follows.  Floating point is float64
except where a page fixes the precision (the SnapKV history is float32).

Parity status: every function is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py`` except ``workloads`` generators (which are not
part of this package).
"""

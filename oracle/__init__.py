"""Float64 CPU oracle for ring attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import this package. The product path (the CUDA library and its
Python binding) never imports, links or runs anything here, and nothing here imports the
product package. The two sides share only the seeded input generators in ``workloads``.

What it computes, and from which passages:

* ``layouts``: where each token of a shard sits in the global sequence, for the basic
  (contiguous), zigzag (chunk i and chunk 2D-1-i) and stripe (token t on shard t mod D)
  layouts (ring-flash-attn package card, "What it is and what it does"; Ring Attention
  concept page, "Sequence sharding and the ring topology").
* ``attention``: the plain definition, softmax(scale * Q K^T + mask) V with its log-sum-exp,
  and its textbook gradient. Ring attention is exact, so this is what the method reaches
  (Ring Attention concept page, "Online softmax across ring steps" and "Show Me the Code").
* ``ring``: the explicit ring schedule — rank r holds KV shard (r - s) mod D at step s,
  a normalised (block_out, block_lse) per step, merged by the log-sum-exp rule of
  ``update_out_and_lse`` (nanotron how-to page, "Forward Pass Implementation" and
  "Numerically-Stable Output Fusion"), and the per-step backward that accumulates dq, dk
  and dv against the final out / lse ("Backward Pass and Gradient Accumulation").

Every function is pinned by ``tests/test_oracle_*.py`` to something other than itself:
the two-device worked example, closed forms, brute force and finite differences.
"""

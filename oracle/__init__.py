"""CPU oracle for one GLANCE verify round.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call, link or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

It is a plain, slow restatement of what the pages define, in numpy float64:

* ``marginals``  per-offset log-softmax of the draft logits and the per-offset
  candidate lists (Assumption 1; the plug-in score pi_hat).
* ``tree``       the top-N prefix set under the plug-in score, as a brute-force
  enumeration (tiny V, L) and as a lazy best-first search (full size), and the
  canonical packing into parent/depth/position/ancestor arrays (Definition 1).
* ``attention``  ancestor-masked GQA attention over cached prefix + tree rows.
* ``lmhead``     LM-head projection with per-row greedy argmax and top-2 gap
  (the gap gamma_k of Theorem 1's full statement, Appendix B.1).
* ``walk``       the acceptance walk, A(S) in its set form, and the KV commit.
* ``toy``        a small random-init decoder target with greedy autoregression
  and GLANCE rounds, for Theorem 1 (Section 4.2, Appendix B.1).

It shares no code with the CUDA library and imports nothing from it. The only
code both sides use is the seeded input generator package ``workloads``.
"""

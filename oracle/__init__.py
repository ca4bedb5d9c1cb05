"""Float64 CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, step-by-step
restatement of the verify rule and of the RMSNorm + LM-head contraction,
written from the pages' descriptions.  It exists to check the CUDA library.
Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import it; the product path never does, and it shares no code with
the CUDA kernels or their binding.

Parity status of each function (what pins it, see tests/test_oracle_*.py):
  verify.temperature_softmax   pinned: library softmax, invariants
  verify.top_p_mask            pinned: O(V^2) brute-force definition
  verify.inverse_cdf           pinned: exact enumeration of u pieces
  verify.residual_weights      pinned: marginal = p by exact enumeration
  verify.verify_from_distributions / verify_sequence
                               pinned: enumeration, chi-square, E(k),
                               special cases, greedy argmax match
  verify.kv_commit             pinned: length invariant
  lmhead.lmhead_rmsnorm        pinned: pure-Python triple loop, scale
                               invariance of RMSNorm
  analytics.*                  pinned: the pages' printed speedup table and
                               worked examples (tests/golden/)
  sample.sample_row / sample_tokens
                               pinned: exact u-grid frequencies against a
                               plain-loop softmax and nucleus, greedy ties,
                               padding and flags
  dynk.DynK                    pinned: hand-worked crossings, exact
                               thresholds, window expiry, caps, direct
                               window sums over random histories
  paged.kv_commit_paged        pinned: hand-worked page boundaries, per-token
                               page ownership on random cases, all-or-nothing
                               capacity
Planted mistakes that the pins must catch: tests/test_oracle_mutations*.py.
"""

from . import analytics, dynk, lmhead, paged, sample, verify  # noqa: F401

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
"""

from . import analytics, lmhead, verify  # noqa: F401

"""Closed forms the pages give for the verify rule's yield and speedup.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see ``oracle/__init__.py``).

[SSD §3.2] ("Self-speculative decoding with layer skip and KV reuse") and
[SD §2.3] ("Speculative decoding, the founding scheme"): with i.i.d. per
position acceptance alpha and k drafts, the expected tokens emitted per round
is E(k) = (1 - alpha^(k+1)) / (1 - alpha); with a draft costing c of a full
forward per token the round costs c*k + 1, so the speedup is E(k)/(c*k + 1).
[FS §2.1, §3.3] ("FlashSpec speculative decoding in practice") measures the
speedup as accepted tokens per round over the round's time in target decode
steps (draft + verify + sampling).
"""

from __future__ import annotations


def expected_tokens(alpha: float, k: int) -> float:
    """E(k) = (1 - alpha^(k+1)) / (1 - alpha); k + 1 when alpha == 1."""
    if alpha == 1.0:
        return float(k + 1)
    return (1.0 - alpha ** (k + 1)) / (1.0 - alpha)


def speedup(alpha: float, k: int, c: float) -> float:
    """E(k) / (c*k + 1) [SSD §3.2]."""
    return expected_tokens(alpha, k) / (c * k + 1.0)


def round_speedup(tokens_per_round: float, *step_costs: float) -> float:
    """tokens per round / (sum of the round's costs in target decode steps)
    [FS §2.1, §3.3]."""
    return tokens_per_round / sum(step_costs)


def acceptance_law(betas) -> list:
    """P(n >= i) = prod_{j < i} beta_j for i = 0..k, where beta_j =
    sum_v min(p_j(v), q_j(v)) is position j's acceptance probability."""
    out = [1.0]
    for b in betas:
        out.append(out[-1] * b)
    return out

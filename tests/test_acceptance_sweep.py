"""Acceptance against temperature on synthetic logits, the comparison that
"Speculative decoding, the founding scheme" §5.1 makes with a real draft
model (acceptance near 0.85 at T=0.1, about 0.65 at T=0.7, a little above 0.5
at T=1.0).

A tested position i accepts with probability beta_i = sum_v min(p'_i(v),
q'_i(v)) when its token was drawn from q'_i (the accept rule of "Speculative
decoding, the founding scheme" §2.1-2.2 summed over the draft's draws), so the
realised accept count over all tested positions minus the sum of their
beta_i is a sum of martingale differences: mean 0, variance
sum beta_i (1 - beta_i).  The CPU test checks the oracle's
accept rule against that at full vocabulary size; the GPU test checks the
library's.  beta_i itself depends only on the logits, so the table printed by
running this file (mean beta and the exact E[n+1] = sum_i prod_{j<i} beta_j)
needs no sampling.

Two draft recipes (reading R31): the plain one, draft = target + N(0, sigma^2)
in logit space, whose disagreement a higher temperature divides down, so its
acceptance rises with T; and an under-confident draft, draft = 0.7 target +
N(0, 0.2^2), which reproduces the pages' falling trend."""

import numpy as np
import pytest

from tests.conftest import gpu_available
from oracle import verify as ov
from speculative_decoding_verification_47_gb300 import workloads as wl

TEMPS = (0.1, 0.7, 1.0)
RECIPES = {"plain sigma=1": (1.0, 1.0), "under-confident 0.7, sigma=0.2": (0.7, 0.2)}
K, V = 8, 32000


def make(B, T, recipe, seed=5000):
    scale, sigma = RECIPES[recipe]
    return wl.synth_verify("sweep", B, K, V, wl.BF16, K, T, sigma, ov.SAMPLED,
                           seeds=(seed, seed + 100, seed + 200), draft_scale=scale)


def betas(w):
    """beta[b, i] = sum_v min(p'_i, q'_i) for the row pairs i < k_b."""
    out = np.zeros((w.B, w.K))
    for b in range(w.B):
        T = float(w.temperature[b])
        for i in range(int(w.k_per_row[b])):
            p = ov.process_row(ov.stored_to_f64(w.target[b, i], w.dtype), T, w.top_p).p
            q = ov.process_row(ov.stored_to_f64(w.draft[b, i], w.dtype), T, w.top_p).p
            out[b, i] = np.minimum(p, q).sum()
    return out


def exact_mean_len(beta_row):
    """E[n+1] for one sequence: sum over i = 0..k of prod_{j<i} beta_j."""
    return float(np.sum(np.concatenate([[1.0], np.cumprod(beta_row)])))


def check_accepts(n, k, beta):
    """Realised accepts minus their expectation, over every tested position,
    within 4 standard deviations."""
    acc = dev = var = 0.0
    for b in range(len(n)):
        tested = int(n[b]) + (1 if n[b] < k[b] else 0)
        acc += int(n[b])
        dev += beta[b, :tested].sum()
        var += (beta[b, :tested] * (1 - beta[b, :tested])).sum()
    assert abs(acc - dev) <= 4 * np.sqrt(var) + 1, (acc, dev, var)
    return acc / max(1.0, sum(int(x) + (1 if x < kk else 0) for x, kk in zip(n, k)))


def test_oracle_acceptance_matches_beta():
    for recipe in RECIPES:
        for T in TEMPS:
            w = make(48, T, recipe)
            o = ov.spec_verify(w.target, w.draft, w.dtype, w.B, w.K, w.V, w.draft_tokens,
                               w.k_per_row, w.temperature, w.top_p, w.uniforms, w.mode)
            assert o.flags == 0
            check_accepts(o.n_accepted, w.k_per_row, betas(w))


def test_under_confident_draft_falls_with_temperature():
    """The recipe chosen to mirror the pages' trend does: mean beta falls as T
    rises, while the plain recipe's rises."""
    m = {r: [betas(make(16, T, r)).mean() for T in TEMPS] for r in RECIPES}
    a, b_ = m["under-confident 0.7, sigma=0.2"], m["plain sigma=1"]
    assert a[0] > a[1] > a[2] and b_[0] < b_[2]


@pytest.mark.gpu
@pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")
def test_gpu_acceptance_against_temperature():
    from speculative_decoding_verification_47_gb300 import build
    from tests import verify_harness as vh
    build.build()
    for recipe in RECIPES:
        for T in TEMPS:
            w = make(128, T, recipe, seed=5300)
            g = vh.run_gpu(w, diag=False)
            assert g.flags == 0
            check_accepts(g.n, w.k_per_row, betas(w))


if __name__ == "__main__":
    for recipe in RECIPES:
        for T in TEMPS:
            w = make(128, T, recipe)
            be = betas(w)
            print(f"{recipe:32s} T={T}: mean beta {be.mean():.3f}, "
                  f"E[n+1] {np.mean([exact_mean_len(r) for r in be]):.2f}")

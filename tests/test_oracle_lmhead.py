"""Pins of the RMSNorm + LM-head oracle [SSD §3.1, §4.2]."""

import math

import numpy as np

from oracle import lmhead as ol
from oracle import verify as ov
from speculative_decoding_verification_47_gb300 import workloads as wl


def test_lmhead_matches_triple_loop():
    """Pure-Python triple loop on a tiny shape (M=4, H=64, V=96)."""
    x = wl.lmhead_inputs(M=4, H=64, V=96, seed=5)
    got = ol.lmhead_rmsnorm(x.hidden, x.norm_w, x.eps, x.W)
    h = ov.bf16_bits_to_f64(x.hidden).tolist()
    w = ov.bf16_bits_to_f64(x.norm_w).tolist()
    W = ov.bf16_bits_to_f64(x.W).tolist()
    for m in range(4):
        ms = math.fsum(v * v for v in h[m]) / 64
        r = 1.0 / math.sqrt(ms + x.eps)
        y = [h[m][k] * r * w[k] for k in range(64)]
        for n in range(96):
            ref = math.fsum(y[k] * W[k][n] for k in range(64))
            assert math.isclose(got[m, n], ref, rel_tol=1e-12, abs_tol=1e-14)


def test_rmsnorm_scale_invariance_and_norm_pitfall():
    """RMSNorm removes the hidden-state scale (up to eps); leaving it out
    [SSD §3.1 pitfall] scales the logits with the hidden state, which
    sharpens the draft softmax and collapses acceptance."""
    x = wl.lmhead_inputs(M=8, H=256, V=512, seed=6)
    h8 = wl.f64_to_bf16_bits(8.0 * ov.bf16_bits_to_f64(x.hidden))  # exact x8
    a = ol.lmhead_rmsnorm(x.hidden, x.norm_w, x.eps, x.W)
    b = ol.lmhead_rmsnorm(h8, x.norm_w, x.eps, x.W)
    np.testing.assert_allclose(a, b, rtol=1e-4, atol=1e-6)
    # Without the norm: logits = h @ W scale by 8 with h.
    W = ov.bf16_bits_to_f64(x.W)
    raw8 = ov.bf16_bits_to_f64(h8) @ W
    tgt = ol.lmhead_rmsnorm(x.hidden, x.norm_w, x.eps, x.W)
    beta_norm, beta_raw = [], []
    for m in range(8):
        p = ov.temperature_softmax(tgt[m], 1.0)[0]
        q_ok = ov.temperature_softmax(b[m], 1.0)[0]
        q_bad = ov.temperature_softmax(raw8[m], 1.0)[0]
        beta_norm.append(np.minimum(p, q_ok).sum())
        beta_raw.append(np.minimum(p, q_bad).sum())
    assert min(beta_norm) > 0.99
    assert max(beta_raw) < 0.5 * min(beta_norm)

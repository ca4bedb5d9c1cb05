"""Float64 CPU oracle of the fused final-RMSNorm + LM-head contraction that
turns layer-L hidden states into draft logits.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see ``oracle/__init__.py``).

[SSD §3.1, §4.2] ("Self-speculative decoding with layer skip and KV reuse",
xdnf.cn): the draft is the first L layers of the target, followed by the
model's final normalisation and its output head; skipping that norm when
leaving at an intermediate layer gives logits of the wrong magnitude.  The
norm is RMSNorm with weight w and epsilon eps:

    y = w * h / sqrt(mean(h^2) + eps),      logits = y @ W

with h [M, H], w [H], W [H, V] (V contiguous).
"""

from __future__ import annotations

import numpy as np

from .verify import bf16_bits_to_f64


def rmsnorm(h: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of each row of h (float64)."""
    ms = np.mean(h * h, axis=1, keepdims=True)
    return h / np.sqrt(ms + eps) * w[None, :]


def lmhead_rmsnorm(hidden_bits, norm_w_bits, eps: float, W_bits) -> np.ndarray:
    """logits = rmsnorm(h) @ W in float64 from bf16 bit patterns."""
    h = bf16_bits_to_f64(hidden_bits)
    w = bf16_bits_to_f64(norm_w_bits)
    W = bf16_bits_to_f64(W_bits)
    return rmsnorm(h, w, eps) @ W


def lmhead_abs_product(hidden_bits, norm_w_bits, eps: float, W_bits) -> np.ndarray:
    """sum_k |y_k W_kn| for every output, the scale of the rounding bound."""
    h = bf16_bits_to_f64(hidden_bits)
    w = bf16_bits_to_f64(norm_w_bits)
    W = bf16_bits_to_f64(W_bits)
    return np.abs(rmsnorm(h, w, eps)) @ np.abs(W)


def lmhead_rows(hidden_bits, norm_w_bits, eps: float, W_bits, rows, cols=None):
    """A few outputs of a large problem, computed one row at a time (for
    sampled checks at full size).  Returns [len(rows), len(cols)]."""
    w = bf16_bits_to_f64(norm_w_bits)
    h = bf16_bits_to_f64(hidden_bits[rows])
    y = rmsnorm(h, w, eps)
    Wc = W_bits if cols is None else W_bits[:, cols]
    Wf = bf16_bits_to_f64(Wc)
    return y @ Wf, np.abs(y) @ np.abs(Wf)

"""Pins of the draft-side sampler oracle against what the pages and the
mathematics fix, independent of the oracle's own formulas:

  * on a uniform grid of u, the frequency of each token equals the processed
    probability p'(v) within one grid step (softmax at temperature T, then
    top-p truncation and renormalisation [FS §3.2]): exact enumeration;
  * tokens outside the nucleus are never drawn;
  * greedy rows give the argmax, lowest index on ties;
  * padding, and the flags of bad knobs, rows and uniforms.
"""

import math

import numpy as np
import pytest

from oracle import sample as osm
from oracle import verify as ov


def _grid(N):
    return (np.arange(N) + 0.5) / N


def _closed_form_probs(z, T, top_p):
    """p'(v) computed without the oracle: exp of the tempered logits (plain
    math.exp per token), normalised by a plain loop; the nucleus by sorting
    (probability desc, index asc) and keeping a token while the mass before it
    is <= top_p."""
    V = len(z)
    e = [math.exp(float(v) / T) for v in z]
    S = sum(e)
    p = [x / S for x in e]
    if top_p >= 1.0:
        return np.array(p)
    order = sorted(range(V), key=lambda v: (-p[v], v))
    kept, before = [], 0.0
    for v in order:
        if before <= top_p:
            kept.append(v)
        before += p[v]
    M = sum(p[v] for v in kept)
    out = np.zeros(V)
    for v in kept:
        out[v] = p[v] / M
    return out


@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (0.7, 1.0), (1.6, 1.0), (1.0, 0.8), (0.5, 0.6)])
def test_grid_frequencies_equal_processed_probabilities(T, top_p):
    z = np.array([0.3, -1.2, 2.0, 0.9, -0.4, 1.5, 0.0, -2.5])
    N = 4000
    counts = np.zeros(len(z))
    for u in _grid(N):
        y, _, f = osm.sample_row(z, T, top_p, float(u), False)
        assert f == 0
        counts[y] += 1
    ref = _closed_form_probs(z, T, top_p)
    assert np.all(np.abs(counts / N - ref) <= 1.0 / N + 1e-12), (counts / N, ref)
    if top_p < 1.0:
        assert np.all(counts[ref == 0.0] == 0)


def test_inverse_cdf_is_in_index_order():
    """With equal probabilities the grid walks the tokens in index order."""
    z = np.zeros(4)
    toks = [osm.sample_row(z, 1.0, 1.0, float(u), False)[0] for u in (0.1, 0.3, 0.6, 0.9)]
    assert toks == [0, 1, 2, 3]


def test_greedy_is_argmax_lowest_index():
    z = np.array([1.0, 3.0, -2.0, 3.0, 0.5])
    assert osm.sample_row(z, 1.0, 1.0, 0.99, True)[0] == 1
    assert osm.sample_row(z, 0.3, 0.5, 0.0, True)[0] == 1


def test_padding_and_flags():
    V, K = 6, 3
    r = np.random.default_rng(3)
    logits = r.normal(size=(4, K, V)).astype(np.float32)
    logits[2, 1, 3] = np.nan
    u = r.uniform(size=(4, K)).astype(np.float32)
    u[3, 0] = 1.0
    k = np.array([2, 0, 3, 3], np.int32)
    T = np.array([1.0, 1.0, 1.0, 1.0], np.float32)
    mode = np.zeros(4, np.uint8)
    tok, _, flags = osm.sample_tokens(logits, "f32", 4, K, V, k, T, 1.0, u, mode)
    assert tok[0, 2] == -1 and np.all(tok[1] == -1)
    assert tok[2, 1] == -1 and tok[2, 0] >= 0 and tok[2, 2] >= 0
    assert tok[3, 0] == -1 and tok[3, 1] >= 0
    assert flags == ov.FLAG_NONFINITE | ov.FLAG_BAD_UNIFORM
    bad = osm.sample_tokens(logits, "f32", 4, K, V, np.array([4, 1, 1, 1]), T, 1.0, u, mode)
    assert np.all(bad[0][0] == -1) and bad[2] & ov.FLAG_BAD_K
    badT = osm.sample_tokens(logits, "f32", 4, K, V, k, np.array([0.0, 1, 1, 1], np.float32), 1.0,
                             u, mode)
    assert np.all(badT[0][0] == -1) and badT[2] & ov.FLAG_BAD_TEMPERATURE


def test_bf16_rows_decode_exactly():
    """bf16 storage: the row is widened bit-exactly before the softmax."""
    z = np.array([0.5, 1.25, -3.0, 2.0], np.float32)
    bits = (z.view(np.uint32) >> 16).astype(np.uint16)
    for u in (0.05, 0.5, 0.95):
        assert osm.sample_row(ov.stored_to_f64(bits, "bf16"), 1.0, 1.0, u, False)[0] == \
            osm.sample_row(z.astype(np.float64), 1.0, 1.0, u, False)[0]

"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formulas: each compares it with an
independent route to the same fact (a library softmax, a brute-force
definition, exact enumeration of the random draws, a chi-square law, a closed
form the pages print, or the pages' printed numbers).
"""

import itertools
import json
import math
import os
import zlib

import numpy as np
import pytest
from scipy import special, stats

from oracle import analytics
from oracle import verify as ov

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# Independent textbook pieces (not the oracle's code paths)
# ----------------------------------------------------------------------------

def textbook_probs(z, T=1.0, top_p=1.0):
    """softmax(z/T) from scipy; top-p by its O(V^2) definition: keep v iff the
    mass of every token ranked before v (greater p, or equal p and smaller
    index) is at most top_p, then renormalise."""
    p = special.softmax(np.asarray(z, np.float64) / T)
    if top_p >= 1.0:
        return p
    V = len(p)
    keep = np.zeros(V, bool)
    for v in range(V):
        before = math.fsum(p[u] for u in range(V)
                           if p[u] > p[v] or (p[u] == p[v] and u < v))
        keep[v] = before <= top_p
    M = math.fsum(p[keep])
    return np.where(keep, p / M, 0.0)


def textbook_residual(p, q):
    w = np.maximum(0.0, p - q)
    s = math.fsum(w)
    return (p / math.fsum(p)) if s <= 0 else w / s


def cdf_breaks(w):
    """Points in [0,1] where inverse-CDF sampling from w changes its output."""
    c = np.cumsum(w) / math.fsum(w)
    return [float(t) for t in c[:-1]]


def cells(breaks):
    """Partition [0,1) at the given points: (midpoint, length) per piece."""
    pts = sorted(set([0.0] + [b for b in breaks if 0.0 < b < 1.0] + [1.0]))
    return [((a + b) / 2.0, b - a) for a, b in zip(pts[:-1], pts[1:]) if b > a]


def enumerate_sequence(zt, zd, k, T=1.0, top_p=1.0, topp_draft=True):
    """Exact output law of oracle.verify_sequence for one sequence with k
    drafts, by enumeration: draft tokens x_i over their law q_i, each accept
    uniform over its two pieces [0, r_i) / [r_i, 1), and the resample/bonus
    uniform over the pieces cut by every candidate distribution's CDF.  The
    pieces come from textbook p, q; the oracle is only evaluated at piece
    midpoints.  Returns {(n, out tuple): probability}."""
    V = len(zt[0])
    K = k
    P = [textbook_probs(zt[i], T, top_p) for i in range(k + 1)]
    Q = [textbook_probs(zd[i], T, top_p if topp_draft else 1.0) for i in range(k)]
    ubreaks = set(cdf_breaks(P[k]))
    for i in range(k):
        ubreaks |= set(cdf_breaks(textbook_residual(P[i], Q[i])))
    ucells = cells(ubreaks)
    law = {}
    support = [np.nonzero(Q[i] > 0)[0] for i in range(k)]
    for xs in itertools.product(*support):
        wx = math.prod(Q[i][xs[i]] for i in range(k))
        acc_cells = []
        for i in range(k):
            r = P[i][xs[i]] / Q[i][xs[i]]
            acc_cells.append(cells([min(1.0, r)]))
        for combo in itertools.product(*acc_cells):
            wu = math.prod(c[1] for c in combo)
            for um, ul in ucells:
                u = np.array([c[0] for c in combo] + [um])
                res = ov.verify_sequence(zt, zd, np.array(xs), k, K, V, T, top_p,
                                         u, ov.SAMPLED, topp_draft=topp_draft)
                key = (res.n, tuple(res.out))
                law[key] = law.get(key, 0.0) + wx * wu * ul
    return law, P, Q


def marginal(law, pos, V, cond_min_n=0):
    m = np.zeros(V)
    tot = 0.0
    for (n, out), pr in law.items():
        if n < cond_min_n:
            continue
        tot += pr
        m[out[pos]] += pr
    return (m / tot if tot > 0 else m), tot


def rand_logits(rng, V, scale=1.5):
    return rng.standard_normal(V) * scale


# ----------------------------------------------------------------------------
# (a) exact enumeration: the emitted-token marginal equals p  [SD §2.1-2.2]
# ----------------------------------------------------------------------------

ENUM_CASES = {
    "random": dict(T=1.0, top_p=1.0, kind="random"),
    "temperature": dict(T=0.6, top_p=1.0, kind="random"),
    "p_equals_q": dict(T=1.0, top_p=1.0, kind="equal"),
    "disjoint": dict(T=1.0, top_p=1.0, kind="disjoint"),
    "top_p": dict(T=0.8, top_p=0.7, kind="random"),
    "top_p_ties": dict(T=1.0, top_p=0.3, kind="ties"),
}


def _case_logits(kind, rng, V, k):
    zt = [rand_logits(rng, V) for _ in range(k + 1)]
    if kind == "equal":
        zd = [z.copy() for z in zt[:k]]
    elif kind == "disjoint":
        zt = [np.where(np.arange(V) < V // 2, z, -np.inf) for z in zt]
        zd = [np.where(np.arange(V) >= V // 2, rand_logits(rng, V), -np.inf)
              for _ in range(k)]
    elif kind == "ties":
        base = np.array([1.0, 1.0, 1.0, 0.5, 0.5, 0.0, -1.0, -1.0])[:V]
        zt = [base + 0.0 for _ in range(k + 1)]
        # a tie group of three 1.0s in both; the cut at 0.3 falls inside it
        zd = [np.array([1.0, 0.5, 1.0, 1.0, 0.5, 0.0, -1.0, -1.0])[:V] for _ in range(k)]
    else:
        zd = [z + 0.8 * rng.standard_normal(V) for z in zt[:k]]
    return zt, zd


@pytest.mark.parametrize("case", sorted(ENUM_CASES))
@pytest.mark.parametrize("k", [1, 2])
def test_enumeration_marginal_equals_p(case, k):
    V = 8
    cfg = ENUM_CASES[case]
    rng = np.random.default_rng(zlib.crc32(f"{case}/{k}".encode()))
    zt, zd = _case_logits(cfg["kind"], rng, V, k)
    law, P, Q = enumerate_sequence(zt, zd, k, cfg["T"], cfg["top_p"])
    assert math.isclose(sum(law.values()), 1.0, abs_tol=1e-12)
    # out_0 ~ p_0 exactly
    m0, _ = marginal(law, 0, V)
    np.testing.assert_allclose(m0, P[0], atol=1e-12, rtol=0)
    # given x_0 accepted, out_1 ~ p_1
    m1, tot = marginal(law, 1, V, cond_min_n=1)
    beta0 = math.fsum(np.minimum(P[0], Q[0]))
    assert math.isclose(tot, beta0, abs_tol=1e-12)
    if tot > 0:
        np.testing.assert_allclose(m1, P[1], atol=1e-12, rtol=0)
    if cfg["kind"] == "equal":
        assert all(n == k for (n, _), pr in law.items() if pr > 0)
    if cfg["kind"] == "disjoint":
        assert all(n == 0 for (n, _), pr in law.items() if pr > 0)


def test_enumeration_inverse_cdf_exact():
    """P(inverse_cdf(w, u) = v) over u ~ U[0,1) equals w_v / sum(w), and a
    zero-weight token is never drawn."""
    w = np.array([0.0, 3.0, 1.0, 0.0, 2.0, 2.0, 0.0, 0.5])
    law = np.zeros(len(w))
    for um, ul in cells(cdf_breaks(w)):
        y, _ = ov.inverse_cdf(w, um)
        law[y] += ul
    np.testing.assert_allclose(law, w / w.sum(), atol=1e-15)
    # boundaries: u exactly at C(v)/S moves to the next token (strict '>')
    C = np.cumsum(w) / w.sum()
    for v in range(len(w) - 1):
        if w[v] > 0 and C[v] < 1:
            y, _ = ov.inverse_cdf(w, float(C[v]))
            assert y > v and w[y] > 0


def test_residual_fallback_draws_from_p():
    """sum(max(0, p - q)) == 0 falls back to p [SSD §4.3]."""
    p = textbook_probs(np.array([0.3, -1.0, 2.0, 0.0]))
    w, s, fb = ov.residual_weights(p, p.copy())
    assert fb and s == 0.0
    np.testing.assert_array_equal(w, p)
    law = np.zeros(4)
    for um, ul in cells(cdf_breaks(p)):
        law[ov.inverse_cdf(w, um)[0]] += ul
    np.testing.assert_allclose(law, p, atol=1e-15)


# ----------------------------------------------------------------------------
# (b) chi-square over 10^6 seeded trials
# ----------------------------------------------------------------------------

def _chi2(counts, expected):
    keep = expected >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(expected[keep], expected[~keep].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    exp = exp * obs.sum() / exp.sum()
    return stats.chisquare(obs, exp).pvalue


@pytest.mark.parametrize("V", [8, 64])
def test_chi_square_million_trials(V):
    k = 3
    trials = 1_000_000
    rng = np.random.default_rng(1234 + V)
    zt = [rand_logits(rng, V) for _ in range(k + 1)]
    zd = [z + 0.7 * rng.standard_normal(V) for z in zt[:k]]
    T = 0.9
    P = [ov.process_row(z, T, 1.0).p for z in zt]
    Q = [ov.process_row(z, T, 1.0).p for z in zd]
    # draft tokens from q_i, uniforms on the 2^-24 grid
    X = np.stack([rng.choice(V, size=trials, p=Q[i] / Q[i].sum()) for i in range(k)], 1)
    U = rng.integers(0, 1 << 24, size=(trials, k + 1)) * 2.0 ** -24
    out0 = np.zeros(V, np.int64)
    ncount = np.zeros(k + 1, np.int64)
    Pl = [p for p in P]
    Ql = [q for q in Q]
    for t in range(trials):
        n, y, _ = ov.verify_from_distributions(Pl, Ql, X[t], k, U[t], k)
        out0[X[t, 0] if n > 0 else y] += 1
        ncount[n] += 1
    p0 = textbook_probs(zt[0], T)
    assert _chi2(out0, p0 * trials) > 1e-3
    betas = [math.fsum(np.minimum(textbook_probs(zt[i], T), textbook_probs(zd[i], T)))
             for i in range(k)]
    ge = analytics.acceptance_law(betas)
    pn = np.array([ge[i] - (ge[i + 1] if i < k else 0.0) for i in range(k + 1)])
    assert _chi2(ncount, pn * trials) > 1e-3


# ----------------------------------------------------------------------------
# (c) E(k) = (1 - a^(k+1)) / (1 - a) under i.i.d. acceptance  [SSD §3.2]
# ----------------------------------------------------------------------------

def _alpha_rows(alpha, k):
    """Every position: p = (a, 1-a), q = (1, 0), so sum min(p, q) = a."""
    zt = [np.log(np.array([alpha, 1.0 - alpha])) for _ in range(k + 1)]
    zd = [np.array([0.0, -np.inf]) for _ in range(k)]
    return zt, zd


@pytest.mark.parametrize("alpha", [0.6, 0.7, 0.8, 0.9])
def test_expected_tokens_exact(alpha):
    for k in range(1, 9):
        zt, zd = _alpha_rows(alpha, k)
        x = np.zeros(k, np.int64)
        mean = 0.0
        # enumerate the accept pieces of every position
        for pattern in itertools.product([0, 1], repeat=k):
            u = np.array([alpha / 2 if a else (1 + alpha) / 2 for a in pattern] + [0.5])
            w = math.prod(alpha if a else 1 - alpha for a in pattern)
            res = ov.verify_sequence(zt, zd, x, k, k, 2, 1.0, 1.0, u, ov.SAMPLED)
            mean += w * (res.n + 1)
        closed = (1 - alpha ** (k + 1)) / (1 - alpha)
        assert math.isclose(mean, closed, rel_tol=1e-12)
        assert math.isclose(analytics.expected_tokens(alpha, k), closed, rel_tol=1e-15)


@pytest.mark.parametrize("alpha,k", [(0.6, 3), (0.8, 5), (0.9, 8)])
def test_expected_tokens_monte_carlo(alpha, k):
    rng = np.random.default_rng(7)
    zt, zd = _alpha_rows(alpha, k)
    x = np.zeros(k, np.int64)
    trials = 20000
    tot = 0.0
    tot2 = 0.0
    for _ in range(trials):
        u = rng.integers(0, 1 << 24, size=k + 1) * 2.0 ** -24
        n = ov.verify_sequence(zt, zd, x, k, k, 2, 1.0, 1.0, u, ov.SAMPLED).n + 1
        tot += n
        tot2 += n * n
    mean = tot / trials
    sd = math.sqrt(max(tot2 / trials - mean * mean, 1e-30) / trials)
    assert abs(mean - analytics.expected_tokens(alpha, k)) < 4 * sd


# ----------------------------------------------------------------------------
# (d) the pages' speedup table and worked examples
# ----------------------------------------------------------------------------

def test_speedup_table_printed():
    g = json.load(open(os.path.join(GOLDEN, "speedup_table.json")))
    c = g["c"]
    off = 0
    for k, row in g["rows"].items():
        for a, printed in zip(g["alphas"], row):
            s = analytics.speedup(a, int(k), c)
            assert abs(s - printed) <= 0.03 + 1e-12, (k, a, s, printed)
            off += abs(round(s, 2) - printed) > 1e-9
    assert off == 7  # the seven printed entries that deviate from the formula


def test_worked_examples():
    g = json.load(open(os.path.join(GOLDEN, "worked_examples.json")))["examples"]
    for ex in g[:2]:
        s = analytics.round_speedup(ex["tokens_per_round"], *ex["costs"])
        assert round(s, ex["printed_decimals"]) == ex["printed"]
    for a, k, c, printed in g[2]["cases"]:
        assert round(analytics.speedup(a, k, c), 2) == printed


# ----------------------------------------------------------------------------
# (e) greedy reduces to an argmax match  [SSD §2.4, §5.2]
# ----------------------------------------------------------------------------

def _py_argmax(z):
    best, idx = -math.inf, -1
    for v, val in enumerate(z):
        if val > best:
            best, idx = val, v
    return idx


def test_greedy_is_longest_argmax_prefix():
    rng = np.random.default_rng(11)
    V, K = 16, 5
    for trial in range(300):
        k = int(rng.integers(0, K + 1))
        zt = [np.round(rng.standard_normal(V), 1) for _ in range(K + 1)]  # ties
        a = [_py_argmax(z) for z in zt]
        x = np.array([a[i] if rng.random() < 0.7 else int(rng.integers(V))
                      for i in range(K)])
        res = ov.verify_sequence(zt, None, x, k, K, V, 1.0, 1.0, np.zeros(K + 1),
                                 ov.GREEDY)
        n = 0
        while n < k and x[n] == a[n]:
            n += 1
        assert res.n == n
        assert res.out == [int(v) for v in x[:n]] + [a[n]] + [-1] * (K - n)


def test_sampled_with_tiny_top_p_equals_greedy():
    """top_p -> 0 keeps only the argmax on both sides; with drafts equal to the
    draft argmax, sampled mode must reproduce greedy mode (no ties)."""
    rng = np.random.default_rng(12)
    V, K = 32, 4
    for trial in range(100):
        zt = [rng.standard_normal(V) for _ in range(K + 1)]
        zd = [z + (0.0 if rng.random() < 0.6 else 2.0) * rng.standard_normal(V)
              for z in zt[:K]]
        x = np.array([int(np.argmax(z)) for z in zd])
        u = rng.random(K + 1)
        s = ov.verify_sequence(zt, zd, x, K, K, V, 0.7, 1e-9, u, ov.SAMPLED)
        g = ov.verify_sequence(zt, None, x, K, K, V, 0.7, 1.0, u, ov.GREEDY)
        assert (s.n, s.out) == (g.n, g.out)


# ----------------------------------------------------------------------------
# softmax, top-p and special cases
# ----------------------------------------------------------------------------

def test_temperature_softmax_matches_library_and_shift_invariance():
    rng = np.random.default_rng(3)
    for T in (0.1, 0.7, 1.0, 2.5):
        z = rng.standard_normal(1000) * 3
        p, m, S = ov.temperature_softmax(z, T)
        np.testing.assert_allclose(p, special.softmax(z / T), rtol=1e-12, atol=1e-300)
        p2, _, S2 = ov.temperature_softmax(z + 17.25, T)
        np.testing.assert_allclose(p2, p, rtol=1e-12, atol=1e-300)
        assert math.isclose(S, S2, rel_tol=1e-12)
        assert m == z.max()
        assert math.isclose(math.log(S), special.logsumexp((z - m) / T), rel_tol=1e-12)


@pytest.mark.parametrize("top_p", [0.05, 0.3, 0.5, 0.62, 0.9, 0.999])
def test_top_p_matches_bruteforce_definition(top_p):
    rng = np.random.default_rng(int(top_p * 1000))
    for trial in range(20):
        # coarse values produce many ties
        z = np.round(rng.standard_normal(60) * 2, 0 if trial % 2 else 1)
        p = special.softmax(z)
        kept, M, _ = ov.top_p_mask(p, top_p)
        ref = textbook_probs(z, 1.0, top_p)
        np.testing.assert_array_equal(kept, ref > 0)
        assert math.isclose(M, math.fsum(p[kept]), rel_tol=1e-14)


def test_top_p_cut_inside_tie_group_exact():
    """Dyadic masses make every running sum exact: eight tokens of 1/16 after
    one of 1/2.  top_p = 0.7 keeps the 1/2 token and the first four tied
    tokens by index (mass before them 1/2, 9/16, 10/16, 11/16 <= 0.7)."""
    p = np.array([1 / 16] * 4 + [1 / 2] + [1 / 16] * 4)
    kept, M, margin = ov.top_p_mask(p, 0.7)
    assert kept.tolist() == [True, True, True, True, True, False, False, False, False]
    assert M == 0.5 + 4 / 16
    assert math.isclose(margin, min(0.7 - 11 / 16, 12 / 16 - 0.7))


def test_p_equals_q_accepts_everything():
    rng = np.random.default_rng(5)
    V, K = 50, 6
    for _ in range(50):
        zt = [rng.standard_normal(V) for _ in range(K + 1)]
        x = rng.integers(0, V, size=K)
        u = rng.random(K + 1) * (1 - 1e-9)
        r = ov.verify_sequence(zt, zt[:K], x, K, K, V, 0.8, 1.0, u, ov.SAMPLED)
        assert r.n == K


def test_error_rows_and_laziness():
    V, K = 10, 3
    z = [np.linspace(-1, 1, V) for _ in range(K + 1)]
    x = np.array([9, 9, 9])
    u = np.zeros(K + 1)
    bad = [r.copy() for r in z]
    bad[1][3] = np.nan
    # NaN at position 1 is reached (position 0 accepts with u = 0)
    r = ov.verify_sequence(bad, z[:K], x, K, K, V, 1.0, 1.0, u, ov.SAMPLED)
    assert r.flags == ov.FLAG_NONFINITE and r.n == 0 and r.out == [-1] * (K + 1)
    # ...but not when position 0 rejects first (u = 0.999 > r = 1 is false;
    # make the draft disagree instead)
    zd = [np.where(np.arange(V) == 9, -np.inf, 0.0) for _ in range(K)]
    x0 = np.array([0, 0, 0])
    zt0 = [np.where(np.arange(V) == 0, -np.inf, 0.0)] + bad[1:]
    r = ov.verify_sequence(zt0, zd, x0, K, K, V, 1.0, 1.0, u, ov.SAMPLED)
    assert r.flags == 0 and r.n == 0
    # bad token, bad k, bad temperature, bad uniform, bad mode
    assert ov.verify_sequence(z, z[:K], np.array([V, 0, 0]), K, K, V, 1.0, 1.0, u,
                              ov.SAMPLED).flags == ov.FLAG_BAD_TOKEN
    assert ov.verify_sequence(z, z[:K], x, K + 1, K, V, 1.0, 1.0, u,
                              ov.SAMPLED).flags == ov.FLAG_BAD_K
    assert ov.verify_sequence(z, z[:K], x, K, K, V, 0.0, 1.0, u,
                              ov.SAMPLED).flags == ov.FLAG_BAD_TEMPERATURE
    assert ov.verify_sequence(z, z[:K], x, K, K, V, 1.0, 1.0, np.array([1.0, 0, 0, 0]),
                              ov.SAMPLED).flags == ov.FLAG_BAD_UNIFORM
    assert ov.verify_sequence(z, z[:K], x, K, K, V, 1.0, 1.0, u, 7).flags == ov.FLAG_BAD_MODE


def test_kv_commit_invariant():
    """After the rollback the pointer equals round-start length + accepted
    tokens, never more than k_b beyond it [SSD §3.3]."""
    rng = np.random.default_rng(9)
    B, K = 200, 8
    s0 = rng.integers(128, 4097, size=B).astype(np.int32)
    k = rng.integers(0, K + 1, size=B)
    n = np.array([rng.integers(0, kb + 1) for kb in k], np.int32)
    s1, flags = ov.kv_commit(s0, n, None, K)
    assert flags == 0
    assert np.all(s1 - s0 == n) and np.all(s1 - s0 <= k)
    cap = s0 + 2
    s2, flags = ov.kv_commit(s0, n, cap, K)
    over = s0 + n > cap
    assert (flags == ov.FLAG_CAPACITY) == bool(over.any())
    assert np.all(s2[over] == s0[over]) and np.all(s2[~over] == s1[~over])
    bad = n.copy()
    bad[0] = -1
    bad[1] = K + 1
    s3, flags = ov.kv_commit(s0, bad, None, K)
    assert flags == ov.FLAG_BAD_N and s3[0] == s0[0] and s3[1] == s0[1]
    # with the round's k_b: one more accepted than drafted is refused, even
    # below K; exactly k_b is fine
    kb = np.minimum(k, K - 1)
    more = np.minimum(kb + 1, K).astype(np.int32)
    s4, flags = ov.kv_commit(s0, more, None, K, kb)
    assert flags == ov.FLAG_BAD_N and np.all(s4 == s0)
    s5, flags = ov.kv_commit(s0, kb.astype(np.int32), None, K, kb)
    assert flags == 0 and np.all(s5 - s0 == kb)


@pytest.mark.parametrize("case", ["top_p", "top_p_ties"])
@pytest.mark.parametrize("k", [1, 2])
def test_enumeration_target_only_top_p(case, k):
    """Target-only truncation (the draft untruncated): the output law is still
    exactly the truncated target p' at every position, whatever q is."""
    V = 8
    cfg = ENUM_CASES[case]
    rng = np.random.default_rng(zlib.crc32(f"target-only/{case}/{k}".encode()))
    zt, zd = _case_logits(cfg["kind"], rng, V, k)
    law, P, Q = enumerate_sequence(zt, zd, k, cfg["T"], cfg["top_p"], topp_draft=False)
    assert math.isclose(sum(law.values()), 1.0, abs_tol=1e-12)
    assert np.count_nonzero(Q[0]) == V  # the draft really is untruncated
    m0, _ = marginal(law, 0, V)
    np.testing.assert_allclose(m0, P[0], atol=1e-12, rtol=0)
    m1, tot = marginal(law, 1, V, cond_min_n=1)
    assert math.isclose(tot, math.fsum(np.minimum(P[0], Q[0])), abs_tol=1e-12)
    if tot > 0:
        np.testing.assert_allclose(m1, P[1], atol=1e-12, rtol=0)

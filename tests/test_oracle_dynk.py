"""Pins of the dynamic-k controller oracle against the rule as the pages state
it (sliding 64-round window, +1 on an upward crossing of 0.85, -1 on a
downward crossing of 0.7, k in [2, 8], speculation off below 2), checked on
scripted histories whose window averages are computed here by hand."""

import numpy as np

from oracle import dynk


def test_steady_high_acceptance_steps_up_once():
    """alpha 0.9 from the first round: the window starts above 0.85, so no
    crossing is seen; k stays put."""
    c = dynk.DynK(4)
    ks = [c.update(9, 10) for _ in range(100)]
    assert ks == [4] * 100


def test_upward_crossing_adds_one_once():
    c = dynk.DynK(4)
    ks = [c.update(5, 10) for _ in range(3)]          # alpha 0.5 (below 0.7 from the start)
    assert ks == [4, 4, 4]
    # alpha rises: window (acc, prop) after each round
    seq = [(10, 10)] * 40
    out = [c.update(a, p) for a, p in seq]
    acc, prop = 15, 30
    expect, k, prev_above = [], 4, False
    for a, p in seq:
        acc, prop = acc + a, prop + p
        above = 20 * acc > 17 * prop
        if above and not prev_above:
            k += 1
        prev_above = above
        expect.append(k)
    assert out == expect and out[-1] == 5 and out.count(5) > 0


def test_downward_crossing_and_clamps():
    c = dynk.DynK(3)
    # start high, cross down, stay low: one step down, never below 2
    for _ in range(10):
        c.update(10, 10)
    ks = [c.update(0, 10) for _ in range(200)]
    assert min(ks) == 2 and ks[-1] == 2
    assert ks.count(3) + ks.count(2) == 200
    c2 = dynk.DynK(8)
    c2.update(1, 10)
    ks = [c2.update(10, 10) for _ in range(300)]
    assert max(ks) == 8


def test_window_forgets_after_64_rounds():
    """Only the last 64 proposing rounds count: 64 rounds of full acceptance
    after 64 of none bring alpha to exactly 1."""
    c = dynk.DynK(5)
    for _ in range(64):
        c.update(0, 8)
    for _ in range(64):
        c.update(8, 8)
    assert c.prev == (512, 512)
    assert len(c.hist) == 64


def test_rounds_without_proposal_are_skipped_and_cap():
    c = dynk.DynK(6)
    c.update(3, 4)
    before = (list(c.hist), c.prev)
    assert c.update(0, 0) == 6
    assert (list(c.hist), c.prev) == before
    assert c.update(2, 4, cap=5) == 5
    assert c.update(2, 4, cap=1) == 0      # below 2: no speculation
    assert c.k in (5, 6)                   # the cap does not change the controller's k


def test_exact_threshold_is_not_a_crossing():
    """alpha exactly 0.85 (17/20) is not above it; exactly 0.7 is not below."""
    c = dynk.DynK(4)
    c.update(7, 10)                        # first round: no previous value
    assert c.update(10, 10) == 4           # 17/20 = 0.85 exactly: not above
    assert c.update(10, 10) == 5           # 27/30 = 0.9: crosses from 0.85
    c = dynk.DynK(4)
    c.update(10, 10)
    assert c.update(4, 10) == 4            # 14/20 = 0.7 exactly: not below
    assert c.update(0, 10) == 3            # 14/30: crosses from 0.7


def test_random_histories_match_direct_window_sums():
    rng = np.random.default_rng(11)
    for trial in range(20):
        k0 = int(rng.integers(1, 10))
        c = dynk.DynK(k0)
        hist, k, prev = [], min(max(k0, 2), 8), None
        for r in range(300):
            ku = int(rng.integers(0, 9))
            a = int(rng.binomial(ku, rng.uniform(0.4, 1.0))) if ku else 0
            got = c.update(a, ku)
            if ku:
                hist.append((a, ku))
                w = hist[-64:]
                acc, prop = sum(x for x, _ in w), sum(y for _, y in w)
                if prev is not None:
                    up = acc / prop > 0.85 and not prev[0] / prev[1] > 0.85
                    dn = acc / prop < 0.7 and not prev[0] / prev[1] < 0.7
                    if up:
                        k = min(k + 1, 8)
                    elif dn:
                        k = max(k - 1, 2)
                prev = (acc, prop)
            assert got == k, (trial, r)


def test_invalid_round_is_not_recorded():
    c = dynk.DynK(5)
    c.update(3, 4)
    before = (list(c.hist), c.prev)
    assert c.update(5, 4) == 5 and c.flags == 256
    assert (list(c.hist), c.prev) == before

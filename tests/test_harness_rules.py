"""CPU checks of the parity harness's excuse rule: a GPU/oracle difference is
excused only by the oracle's decision at the first output position where
the two differ (the accept test there when the accepted lengths differ,
else the draw there, and the top-p cuts of that position), never by an
earlier decision that both sides agreed on, and never for an error."""

import math

import numpy as np

from oracle import verify as ov
from tests import verify_harness as vh


def _seq(n, out, decisions, flags=0):
    r = ov.SeqResult(n=n, out=list(out), flags=flags)
    r.decisions = [ov.Decision(k, p, m) for k, p, m in decisions]
    return r


def _excused(g_out, g_n, r):
    _, deciding = vh.first_difference(np.asarray(g_out, np.int32), g_n, r)
    return any(d.margin < vh.MARGIN for d in deciding)


def test_draw_difference_needs_a_low_margin_draw():
    # both accept x0 = 5 (with a low-margin accept test), reject at 1; the
    # draw at 1 has a large margin: a different drawn token is a failure
    r = _seq(1, [5, 7, -1], [("accept", 0, 1e-9), ("accept", 1, 0.3), ("resample", 1, 0.2)])
    assert not _excused([5, 8, -1], 1, r)
    r.decisions[2].margin = 1e-8
    assert _excused([5, 8, -1], 1, r)


def test_length_difference_needs_a_low_margin_accept_test_at_the_cut():
    # oracle rejects at 1 (low-margin draw there), GPU accepted position 1:
    # only the accept test at 1 can excuse it
    r = _seq(1, [5, 7, -1], [("accept", 0, 1e-9), ("accept", 1, 0.4), ("resample", 1, 1e-9)])
    assert not _excused([5, 6, 3], 2, r)
    r.decisions[1].margin = 5e-7
    assert _excused([5, 6, 3], 2, r)


def test_topp_cut_at_the_position_counts():
    r = _seq(0, [9, -1], [("topp", 0, 1e-8), ("accept", 0, 0.5), ("resample", 0, 0.3)])
    assert _excused([4, -1], 0, r)
    r = _seq(1, [2, 9, -1], [("topp", 0, 1e-8), ("accept", 0, 0.5), ("topp", 1, 0.2),
                            ("accept", 1, 0.5), ("resample", 1, 0.3)])
    assert not _excused([2, 4, -1], 1, r)  # the low-margin cut is at an earlier position


def test_errors_are_never_excused():
    r = _seq(0, [-1, -1], [("accept", 0, 1e-12)], flags=ov.FLAG_NONFINITE)
    assert not _excused([3, -1], 0, r)
    r = _seq(0, [3, -1], [("accept", 0, 1e-12), ("resample", 0, 1e-12)])
    assert not _excused([-1, -1], 0, r)


def test_greedy_differences_are_never_excused():
    r = _seq(0, [4, -1], [("greedy", 0, math.inf)])
    assert not _excused([5, -1], 0, r)


def test_per_call_share():
    saved = {k: (dict(v) if isinstance(v, dict) else v) for k, v in vh.BUDGET.items()}
    try:
        vh.record_call("x", 100, 1, 3)  # one disagreement is always allowed per call
        try:
            vh.record_call("y", 100, 2, 3)
        except AssertionError:
            pass
        else:
            raise AssertionError("two disagreements in 100 decisions passed")
    finally:
        vh.BUDGET.clear()
        vh.BUDGET.update(saved)

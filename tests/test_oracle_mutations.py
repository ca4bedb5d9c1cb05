"""The pins must be able to fail: plant plausible mistakes in the oracle (on
the CPU, by monkeypatching) and check that at least one pin catches each."""

import numpy as np
import pytest

from oracle import verify as ov
from tests import test_oracle_pins as pins


def _residual_unclamped(p, q):
    w = p - q
    s = float(np.sum(w))
    return (p, s, True) if s <= 0 else (w, s, False)


def _inverse_cdf_left(w, u):
    C = np.cumsum(w)
    t = u * float(C[-1])
    y = min(int(np.searchsorted(C, t, side="left")), w.shape[0] - 1)
    return y, 1.0


def _top_p_inclusive(p, top_p):
    V = p.shape[0]
    order = np.lexsort((np.arange(V), -p))
    c = np.cumsum(p[order])
    keep_sorted = c <= top_p
    keep_sorted[0] = True
    kept = np.zeros(V, bool)
    kept[order[keep_sorted]] = True
    return kept, float(p[kept].sum()), 1.0


def _top_p_ties_descending(p, top_p):
    V = p.shape[0]
    order = np.lexsort((-np.arange(V), -p))
    ps = p[order]
    c_excl = np.cumsum(ps) - ps
    keep_sorted = c_excl <= top_p
    kept = np.zeros(V, bool)
    kept[order[keep_sorted]] = True
    return kept, float(ps[keep_sorted].sum()), 1.0


def _softmax_no_temperature(z, T):
    return ov.__dict__["_orig_softmax"](z, 1.0)


MUTATIONS = {
    "residual_without_clamp": ("residual_weights", _residual_unclamped),
    "cdf_non_strict": ("inverse_cdf", _inverse_cdf_left),
    "top_p_inclusive_mass": ("top_p_mask", _top_p_inclusive),
    "top_p_ties_by_index_desc": ("top_p_mask", _top_p_ties_descending),
    "temperature_ignored": ("temperature_softmax", _softmax_no_temperature),
}

CHECKS = [
    lambda: pins.test_enumeration_marginal_equals_p("random", 2),
    lambda: pins.test_enumeration_marginal_equals_p("temperature", 1),
    lambda: pins.test_enumeration_marginal_equals_p("top_p_ties", 1),
    pins.test_enumeration_inverse_cdf_exact,
    pins.test_temperature_softmax_matches_library_and_shift_invariance,
    lambda: pins.test_top_p_matches_bruteforce_definition(0.62),
    pins.test_top_p_cut_inside_tie_group_exact,
]


def _caught():
    for check in CHECKS:
        try:
            check()
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setitem(ov.__dict__, "_orig_softmax", ov.temperature_softmax)
    monkeypatch.setattr(ov, attr, fn)
    assert _caught(), f"no pin caught the planted mistake {name!r}"


def test_pins_pass_unmutated():
    assert not _caught()


def test_strict_accept_comparison_is_pinned(monkeypatch):
    """Accepting on u <= r instead of u < r only differs on a boundary of
    measure zero; the laziness test puts u = r = 0 on it."""
    orig = ov.verify_sequence

    def le_verify(zt, zd, x, k, K, V, T, top_p, u, mode):
        u = np.asarray(u, np.float64).copy()
        u[:K] = np.where(u[:K] == 0.0, -1e-300, u[:K])  # u <= r == u' < r
        return orig(zt, zd, x, k, K, V, T, top_p, u, mode)

    monkeypatch.setattr(ov, "verify_sequence", le_verify)
    monkeypatch.setattr(ov, "_uniform_ok", lambda u: u < 1.0)
    with pytest.raises(AssertionError):
        pins.test_error_rows_and_laziness()


def test_target_only_flag_is_pinned(monkeypatch):
    """Target-only top-p leaves the output law at p' whatever q is, so only
    the acceptance law can show a draft that was truncated after all: an
    oracle that ignores topp_draft=False must fail the target-only pin."""
    orig = ov.verify_sequence

    def always_both(*args, topp_draft=True, **kw):
        return orig(*args, topp_draft=True, **kw)

    pins.test_enumeration_target_only_top_p("top_p", 1)  # passes unmutated
    monkeypatch.setattr(ov, "verify_sequence", always_both)
    with pytest.raises(AssertionError):
        for case in ("top_p", "top_p_ties"):
            for k in (1, 2):
                pins.test_enumeration_target_only_top_p(case, k)

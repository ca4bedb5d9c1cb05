"""The pins of the draft sampler, dynamic-k and paged-KV oracles must be able
to fail: plant plausible mistakes in each oracle (on the CPU, by
monkeypatching a mutated copy in) and check that at least one of that
oracle's pins catches every one."""

import inspect

import numpy as np
import pytest

from oracle import dynk as odk
from oracle import paged as opg
from oracle import sample as osm
from oracle import verify as ov
from tests import test_oracle_dynk as pins_dynk
from tests import test_oracle_paged as pins_paged
from tests import test_oracle_sample as pins_sample


def _run_pins(module, param_sets=None):
    """True if some pin of ``module`` fails with an AssertionError."""
    for name, fn in inspect.getmembers(module, inspect.isfunction):
        if not name.startswith("test_") or fn.__module__ != module.__name__:
            continue
        calls = (param_sets or {}).get(name, [()])
        for args in calls:
            try:
                fn(*args)
            except AssertionError:
                return True
    return False


SAMPLE_PARAMS = {"test_grid_frequencies_equal_processed_probabilities":
                 [(1.0, 1.0), (0.7, 1.0), (1.0, 0.8), (0.5, 0.6)]}


# ---- draft sampler --------------------------------------------------------

def _sample_row(kind):
    def f(z, T, top_p, u, greedy):
        if not ov._finite_row(z):
            return -1, np.inf, ov.FLAG_NONFINITE
        if greedy:
            y = len(z) - 1 - int(np.argmax(z[::-1])) if kind == "greedy_last_max" else int(np.argmax(z))
            return y, np.inf, 0
        if not (0.0 <= u < 1.0):
            return -1, np.inf, ov.FLAG_BAD_UNIFORM
        pr = ov.process_row(z, 1.0 if kind == "temperature_ignored" else T,
                            1.0 if kind == "top_p_ignored" else top_p)
        y, margin = ov.inverse_cdf(pr.p, u)
        return y, margin, 0
    return f


def _sample_tokens_shifted_uniform(logits, dtype, B, K, V, k_per_row, temperature, top_p,
                                   uniforms, mode):
    u = np.roll(np.asarray(uniforms), -1, axis=1)
    return _ORIG_SAMPLE_TOKENS(logits, dtype, B, K, V, k_per_row, temperature, top_p, u, mode)


_ORIG_SAMPLE_TOKENS = osm.sample_tokens


@pytest.mark.parametrize("kind", ["greedy_last_max", "temperature_ignored", "top_p_ignored"])
def test_sampler_pins_catch(kind, monkeypatch):
    monkeypatch.setattr(osm, "sample_row", _sample_row(kind))
    assert _run_pins(pins_sample, SAMPLE_PARAMS), kind


def test_sampler_pins_catch_wrong_uniform_column(monkeypatch):
    monkeypatch.setattr(osm, "sample_tokens", _sample_tokens_shifted_uniform)
    assert _run_pins(pins_sample, SAMPLE_PARAMS)


def test_sampler_pins_pass_unmutated():
    assert not _run_pins(pins_sample, SAMPLE_PARAMS)


# ---- dynamic k ------------------------------------------------------------

def _update(kind):
    def update(self, n_accepted, k_used, cap=None):
        if not (0 <= k_used <= 255 and 0 <= n_accepted <= k_used):
            self.flags |= 256
        elif k_used > 0 or kind == "idle_rounds_recorded":
            self.hist.append((int(n_accepted), int(k_used)))
            if len(self.hist) > (63 if kind == "window_63" else odk.WINDOW):
                self.hist.popleft()
            acc = sum(a for a, _ in self.hist)
            prop = sum(p for _, p in self.hist)
            if self.prev is not None or kind == "first_round_steps":
                pa, pp = self.prev if self.prev is not None else (0, 0)
                edge = kind != "level_triggered"
                if self._above(acc, prop) and not (edge and self._above(pa, pp)):
                    self.k = min(self.k + 1, odk.K_MAX)
                elif self._below(acc, prop) and not (edge and self._below(pa, pp)):
                    self.k = max(self.k - 1, odk.K_MIN if kind != "floor_1" else 1)
            self.prev = (acc, prop)
        k = self.k if cap is None else min(self.k, int(cap))
        if kind == "cap_keeps_one":
            return k
        return k if k >= odk.K_MIN else 0
    return update


@pytest.mark.parametrize("kind", ["window_63", "level_triggered", "idle_rounds_recorded",
                                  "floor_1", "cap_keeps_one", "first_round_steps"])
def test_dynk_pins_catch(kind, monkeypatch):
    monkeypatch.setattr(odk.DynK, "update", _update(kind))
    assert _run_pins(pins_dynk), kind


@pytest.mark.parametrize("side", ["above_inclusive", "below_inclusive"])
def test_dynk_pins_catch_inclusive_threshold(side, monkeypatch):
    if side == "above_inclusive":
        monkeypatch.setattr(odk.DynK, "_above",
                            staticmethod(lambda a, p: p > 0 and 20 * a >= 17 * p))
    else:
        monkeypatch.setattr(odk.DynK, "_below",
                            staticmethod(lambda a, p: p > 0 and 10 * a <= 7 * p))
    assert _run_pins(pins_dynk), side


def test_dynk_pins_pass_unmutated(monkeypatch):
    """The pins pass on the oracle, and on the scaffold with no mutation."""
    assert not _run_pins(pins_dynk)
    monkeypatch.setattr(odk.DynK, "update", _update("none"))
    assert not _run_pins(pins_dynk)


# ---- paged KV commit ------------------------------------------------------

def _paged(kind):
    def f(seq_lens, n_accepted, k_per_row, block_table, page_size, free_top, free_capacity):
        P = int(page_size)
        lens = [int(v) for v in seq_lens]
        table = [list(map(int, row)) for row in block_table]
        max_pages = len(table[0]) if table else 0
        released, flags, top, plan = [], 0, int(free_top), []
        for b in range(len(lens)):
            L, n, k = lens[b], int(n_accepted[b]), int(k_per_row[b])
            ok_n = (0 <= n < k) if kind == "n_equal_k_bad" else (0 <= n <= k)
            if not (0 <= k <= max_pages * P - L and ok_n):
                flags |= opg.FLAG_BAD_N
                continue
            Ln = L + (k if kind == "drafts_kept" else n)
            keep = Ln // P if kind == "floor" else -(-Ln // P)
            plan.append((b, L + n, keep, [table[b][j] for j in range(keep, max_pages)
                                          if table[b][j] >= 0]))
        if kind != "partial_capacity":
            if top + sum(len(r) for *_, r in plan) > free_capacity:
                return lens, table, [], top, flags | opg.FLAG_CAPACITY
        for b, Ln, keep, rel in plan:
            if kind == "partial_capacity" and top + len(rel) > free_capacity:
                flags |= opg.FLAG_CAPACITY
                continue
            if kind != "table_not_cleared":
                for j in range(keep, max_pages):
                    table[b][j] = -1
            released.extend(rel)
            top += len(rel)
            lens[b] = Ln
        return lens, table, released, top, flags
    return f


@pytest.mark.parametrize("kind", ["floor", "drafts_kept", "partial_capacity", "table_not_cleared",
                                  "n_equal_k_bad"])
def test_paged_pins_catch(kind, monkeypatch):
    monkeypatch.setattr(opg, "kv_commit_paged", _paged(kind))
    assert _run_pins(pins_paged), kind


def test_paged_pins_pass_unmutated(monkeypatch):
    assert not _run_pins(pins_paged)
    monkeypatch.setattr(opg, "kv_commit_paged", _paged("none"))
    assert not _run_pins(pins_paged)

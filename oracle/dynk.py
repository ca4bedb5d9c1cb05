"""Plain CPU oracle of the dynamic-k controller that feeds k_per_row.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests may import this.  It
shares no code with the CUDA path.

Source: "Self-speculative decoding with layer skip and KV reuse" (xdnf.cn),
§3.2 (the deployed controller) and §5.3 (long contexts): the draft length k
follows the acceptance rate alpha measured over a sliding window of the last
64 steps; when alpha crosses above 0.85, k grows by one; when it crosses below
0.7, k shrinks by one; k stays within [2, 8]; with long contexts k is
shortened further, and below 2 speculation is switched off.

Readings (the points the pages leave open, and the reading taken):
  R24 alpha over the window = tokens accepted / tokens proposed over the last
      64 rounds in which the sequence proposed (k_b > 0); rounds without a
      proposal do not enter the window.
  R25 "crosses" is edge-triggered: k changes only in the round where alpha
      goes from <= 0.85 to > 0.85 (up) or from >= 0.7 to < 0.7 (down); the
      comparisons are exact (integers: 20*acc > 17*prop, 10*acc < 7*prop).
      The first round with data compares against no previous value (no step).
  R26 an optional per-sequence cap (e.g. from the context length) bounds the
      k handed to the next round: k_next = min(k, cap); if that is below 2
      the round does not speculate (k_next = 0).  The controller's own k is
      unchanged by the cap.
  R27 a round with k_used outside [0, 255] or n_accepted outside [0, k_used]
      is not recorded and raises the bad-n flag (bit value 256).
"""

from __future__ import annotations

from collections import deque

WINDOW = 64
K_MIN, K_MAX = 2, 8


class DynK:
    """State of one sequence."""

    def __init__(self, k0: int):
        self.k = min(max(int(k0), K_MIN), K_MAX)
        self.hist = deque()      # (accepted, proposed) of the last WINDOW proposing rounds
        self.prev = None         # (acc, prop) sums of the window after the previous update
        self.flags = 0

    @staticmethod
    def _above(acc: int, prop: int) -> bool:   # alpha > 0.85
        return prop > 0 and 20 * acc > 17 * prop

    @staticmethod
    def _below(acc: int, prop: int) -> bool:   # alpha < 0.7
        return prop > 0 and 10 * acc < 7 * prop

    def update(self, n_accepted: int, k_used: int, cap: int | None = None) -> int:
        """Record one round (n_accepted of k_used drafts accepted) and return
        the k for the next round."""
        if not (0 <= k_used <= 255 and 0 <= n_accepted <= k_used):
            self.flags |= 256
        elif k_used > 0:
            self.hist.append((int(n_accepted), int(k_used)))
            if len(self.hist) > WINDOW:
                self.hist.popleft()
            acc = sum(a for a, _ in self.hist)
            prop = sum(p for _, p in self.hist)
            if self.prev is not None:
                pa, pp = self.prev
                if self._above(acc, prop) and not self._above(pa, pp):
                    self.k = min(self.k + 1, K_MAX)
                elif self._below(acc, prop) and not self._below(pa, pp):
                    self.k = max(self.k - 1, K_MIN)
            self.prev = (acc, prop)
        k = self.k if cap is None else min(self.k, int(cap))
        return k if k >= K_MIN else 0


def run(k0, rounds, caps=None):
    """Controllers for B sequences over a list of rounds; each round is a list
    of (n_accepted, k_used) per sequence.  Returns the k_next of every round."""
    ctl = [DynK(k) for k in k0]
    out = []
    for r, rnd in enumerate(rounds):
        out.append([c.update(a, ku, None if caps is None else caps[r][b])
                    for b, (c, (a, ku)) in enumerate(zip(ctl, rnd))])
    return out

"""Pins of the paged-KV commit oracle: the page-granular rollback of
"Self-speculative decoding with layer skip and KV reuse" §3.3/§4.5 checked on
hand-worked cases (including lengths that land exactly on and just past a
page boundary) and on random cases against a per-token ownership count."""

import numpy as np

from oracle import paged as opg


def test_hand_worked_boundaries():
    P = 4
    # b0: L=6 (pages 0,1), 3 drafts -> 9 tokens (pages 0..2); n=2 -> L'=8 -> keep 2 pages
    # b1: L=8 (pages 0,1), 4 drafts -> 12 (pages 0..2); n=0 -> L'=8 -> keep 2
    # b2: L=7, 1 draft -> 8; n=1 -> L'=8 -> keep 2 (no page past the boundary)
    # b3: L=3, 6 drafts -> 9 (pages 0..2); n=6 -> L'=9 -> keep 3
    table = [[10, 11, 12, -1], [20, 21, 22, -1], [30, 31, -1, -1], [40, 41, 42, -1]]
    lens, tab, rel, top, flags = opg.kv_commit_paged([6, 8, 7, 3], [2, 0, 1, 6], [3, 4, 1, 6], table,
                                                     P, free_top=5, free_capacity=100)
    assert lens == [8, 8, 8, 9] and flags == 0
    assert tab == [[10, 11, -1, -1], [20, 21, -1, -1], [30, 31, -1, -1], [40, 41, 42, -1]]
    assert rel == [12, 22] and top == 7


def test_bad_rounds_and_capacity():
    table = [[1, 2, -1], [3, 4, 5]]
    # b0: n > k (bad, unchanged); b1: L=4, 2 drafts -> 6 tokens, n=0 -> keep 2 pages, release 5
    lens, tab, rel, top, flags = opg.kv_commit_paged([2, 4], [3, 0], [2, 2], table, 2, 0, 10)
    assert lens == [2, 4] and flags == opg.FLAG_BAD_N
    assert tab == [[1, 2, -1], [3, 4, -1]] and rel == [5] and top == 1
    # a full free stack: nothing released, nothing changed
    lens, tab, rel, top, flags = opg.kv_commit_paged([2, 4], [0, 0], [2, 2], table, 2, 10, 10)
    assert flags == opg.FLAG_CAPACITY and lens == [2, 4] and rel == [] and top == 10
    # 5 + 2 tokens do not fit 3 pages of 2
    lens, tab, rel, top, flags = opg.kv_commit_paged([5], [0], [2], [[1, 2, 3]], 2, 0, 10)
    assert flags == opg.FLAG_BAD_N and lens == [5]


def test_random_against_token_ownership():
    """Every kept page holds at least one committed token and every released
    page none; pages are never lost or duplicated."""
    rng = np.random.default_rng(5)
    for trial in range(200):
        P = int(rng.integers(1, 9))
        B, maxp = 6, 12
        L = rng.integers(0, maxp * P // 2, size=B)
        k = np.array([int(rng.integers(0, min(9, maxp * P - l) + 1)) for l in L])
        n = np.array([int(rng.integers(0, kk + 1)) for kk in k])
        ids = rng.permutation(10 * B * maxp)[: B * maxp].reshape(B, maxp)
        table = [[int(ids[b, j]) if j < -(-(L[b] + k[b]) // P) else -1 for j in range(maxp)]
                 for b in range(B)]
        lens, tab, rel, top, flags = opg.kv_commit_paged(L, n, k, table, P, 0, 10**6)
        assert flags == 0 and top == len(rel)
        for b in range(B):
            assert lens[b] == L[b] + n[b]
            for j in range(maxp):
                holds = j * P < lens[b]
                if table[b][j] >= 0:
                    assert (tab[b][j] == table[b][j]) == holds
                    assert (table[b][j] in rel) == (not holds)
        before = {x for row in table for x in row if x >= 0}
        after = {x for row in tab for x in row if x >= 0}
        assert before == after | set(rel) and not (after & set(rel))


def test_capacity_is_all_or_nothing():
    """Room for one of two releases: neither happens."""
    table = [[1, 2], [3, 4]]
    lens, tab, rel, top, flags = opg.kv_commit_paged([1, 1], [0, 0], [2, 2], table, 2, 0, 1)
    assert flags == opg.FLAG_CAPACITY and rel == [] and tab == table and lens == [1, 1]
    lens, tab, rel, top, flags = opg.kv_commit_paged([1, 1], [0, 0], [2, 2], table, 2, 0, 2)
    assert flags == 0 and sorted(rel) == [2, 4] and lens == [1, 1] and top == 2

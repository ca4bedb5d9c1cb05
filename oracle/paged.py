"""Plain CPU oracle of the paged-KV commit: the KV write pointer rolls back to
the accepted length, and the pages that then hold no committed token go back
to the free pool.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests may import this.  It
shares no code with the CUDA path.

Sources: "Self-speculative decoding with layer skip and KV reuse" (xdnf.cn),
§3.3 (roll the write pointer back to the accepted prefix) and §4.5 (with a
paged KV cache the rollback is page-granular, and positions that straddle a
page boundary are the usual source of bugs).

Readings (the points the pages leave open, and the reading taken):
  R29 the cache of sequence b is a list of pages of P tokens (block_table[b],
      page ids, -1 = none).  At the start of the round it holds L_b tokens;
      the drafts were written at L_b .. L_b + k_b - 1.  After verification the
      length is L' = L_b + n_b, pages 0 .. ceil(L'/P) - 1 stay, and every
      allocated page from index ceil(L'/P) on is released: its id is pushed
      on the free stack and its table entry set to -1.  The free stack's
      order is not part of the result (only the set of released ids is).
  R30 n_b outside [0, k_b], or k_b outside [0, max_pages * P - L_b], leaves
      the sequence unchanged and raises the bad-n flag (bit value 256).  If
      the call's releases together would overflow the free stack, no
      sequence changes at all and the capacity flag (bit value 64) is raised:
      all or nothing, so the result does not depend on the order in which
      sequences are handled.
"""

from __future__ import annotations

FLAG_CAPACITY = 64
FLAG_BAD_N = 256


def kv_commit_paged(seq_lens, n_accepted, k_per_row, block_table, page_size: int,
                    free_top: int, free_capacity: int):
    """Returns (new seq_lens, new block table, released page ids as a list in
    sequence order, new free_top, flags)."""
    P = int(page_size)
    lens = [int(v) for v in seq_lens]
    table = [list(map(int, row)) for row in block_table]
    max_pages = len(table[0]) if table else 0
    released, flags, top = [], 0, int(free_top)
    plan = []  # (b, L + n, first page to release, released ids)
    for b in range(len(lens)):
        L, n, k = lens[b], int(n_accepted[b]), int(k_per_row[b])
        if not (0 <= k <= max_pages * P - L and 0 <= n <= k):
            flags |= FLAG_BAD_N
            continue
        Ln = L + n
        keep = -(-Ln // P)  # ceil(Ln / P)
        plan.append((b, Ln, keep, [table[b][j] for j in range(keep, max_pages) if table[b][j] >= 0]))
    if top + sum(len(r) for *_, r in plan) > free_capacity:
        return lens, table, [], top, flags | FLAG_CAPACITY
    for b, Ln, keep, rel in plan:
        for j in range(keep, max_pages):
            table[b][j] = -1
        released.extend(rel)
        top += len(rel)
        lens[b] = Ln
    return lens, table, released, top, flags

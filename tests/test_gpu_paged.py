"""GPU parity of the paged-KV commit (sv_kv_commit_paged) against the oracle:
lengths and block tables exactly, the released page ids as a set (their order
on the free stack is not part of the result), the free stack's new size and
the flags.  Random batches with lengths on and around page boundaries, bad
rounds, and the all-or-nothing free-stack overflow."""

import numpy as np
import pytest

from tests.conftest import gpu_available
from oracle import paged as opg
from speculative_decoding_verification_47_gb300 import binding as sb

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_verification_47_gb300 import build
    build.build()
    sb.lib()


def _batch(rng, B, maxp, P, bad_frac=0.0):
    L = rng.integers(0, maxp * P // 2 + 1, size=B).astype(np.int32)
    L[: B // 4] = (rng.integers(1, maxp // 2, size=B // 4) * P).astype(np.int32)  # on a boundary
    k = np.array([int(rng.integers(0, min(9, maxp * P - l) + 1)) for l in L], np.int32)
    n = np.array([int(rng.integers(0, kk + 1)) for kk in k], np.int32)
    bad = rng.uniform(size=B) < bad_frac
    n[bad] = k[bad] + 1
    ids = rng.permutation(4 * B * maxp)[: B * maxp].reshape(B, maxp).astype(np.int32)
    used = np.array([-(-(L[b] + k[b]) // P) for b in range(B)])
    table = np.where(np.arange(maxp)[None, :] < used[:, None], ids, -1).astype(np.int32)
    return L, n, k, table


def _run(L, n, k, table, P, top0, cap):
    import torch
    B, maxp = table.shape
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    dl, dn, dk, dt = d(L), d(n), d(k), d(table)
    free = torch.full((max(cap, 1),), -7, dtype=torch.int32, device="cuda")
    top = torch.tensor([top0], dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    sb.sv_kv_commit_paged(dl, dn, dk, dt, maxp, P, free, top, cap, B, ws, 256, None)
    flags = sb.sv_read_device_flags(ws)
    t = int(top.item())
    return dl.cpu().numpy(), dt.cpu().numpy(), free.cpu().numpy()[top0:t], t, flags


@pytest.mark.parametrize("P", [1, 3, 16, 64])
def test_paged_commit_matches_oracle(P):
    rng = np.random.default_rng(100 + P)
    B, maxp = 1000, 40
    L, n, k, table = _batch(rng, B, maxp, P, bad_frac=0.01)
    lens, tab, rel, top, flags = _run(L, n, k, table, P, 5, 10**6)
    rl, rt, rr, rtop, rflags = opg.kv_commit_paged(L, n, k, table, P, 5, 10**6)
    assert np.array_equal(lens, np.array(rl)) and np.array_equal(tab, np.array(rt))
    assert sorted(rel.tolist()) == sorted(rr) and top == rtop and flags == rflags
    assert flags == opg.FLAG_BAD_N  # some rounds were bad


def test_paged_commit_capacity_all_or_nothing():
    rng = np.random.default_rng(9)
    B, maxp, P = 200, 20, 8
    L, n, k, table = _batch(rng, B, maxp, P)
    _, _, rr, _, _ = opg.kv_commit_paged(L, n, k, table, P, 0, 10**6)
    need = len(rr)
    assert need > 1
    lens, tab, rel, top, flags = _run(L, n, k, table, P, 3, 3 + need - 1)
    assert flags == opg.FLAG_CAPACITY and top == 3 and len(rel) == 0
    assert np.array_equal(lens, L) and np.array_equal(tab, table)
    lens, tab, rel, top, flags = _run(L, n, k, table, P, 3, 3 + need)
    assert flags == 0 and top == 3 + need and sorted(rel.tolist()) == sorted(rr)


def test_paged_commit_bench_workload():
    """The round bench.py times (--workload kvp): B=1024 sequences, 64 pages
    of 16 tokens, lengths ~U[100, 512), k_b ~U{2..8}."""
    from speculative_decoding_verification_47_gb300 import workloads as wl
    r = wl.paged_round()
    args = (r.seq_lens, r.n_accepted, r.k_per_row, r.block_table, r.page_size, 0, r.pool_pages)
    lens, tab, rel, top, flags = _run(*args)
    rl, rt, rr, rtop, rflags = opg.kv_commit_paged(*args)
    assert flags == rflags == 0
    assert np.array_equal(lens, np.array(rl)) and np.array_equal(tab, np.array(rt))
    assert sorted(rel.tolist()) == sorted(rr) and top == rtop == len(rr) > 0

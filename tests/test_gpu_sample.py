"""GPU parity of sv_draft_sample (the draft-side sampler) against the float64
oracle, through the C ABI.  Tokens must match bit for bit, except at a
position whose inverse-CDF (or top-p cut) margin is below 1e-6.  Such
disagreements have their own budget (reading R22): at most 5e-4 of the
sampled tokens of the session.  Over a 128K vocabulary at T = 1 about 2% of
draws land within 1e-6 of a CDF boundary; the per-token weights are float32
(an exponential of an argument rounded to float), whose summed error reaches
a few 1e-9 of the row mass, and a draw flips when its margin is smaller than
that.  The headline batch's draft rows are drawn under ten uniform seeds
(12830 draws, the oracle in a spawn pool): 5 flips were measured there
(3.9e-4), each at an oracle margin below 1e-6 (the excuse this file checks).

Cases: the headline batch's draft rows at full size (B=256, K=8, V=128256
bf16, ragged k_b, per-row temperature), both dtypes with and without top-p,
greedy and sampled rows mixed, ragged vocabularies, one row per call (K=1),
padded layouts, and the error paths (non-finite rows, bad uniforms, bad
knobs)."""

import numpy as np
import pytest

from tests.conftest import gpu_available
from tests import verify_harness as vh
from oracle import sample as osm
from oracle import verify as ov
from speculative_decoding_verification_47_gb300 import binding as sb
from speculative_decoding_verification_47_gb300 import workloads as wl

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]

MARGIN = 1e-6
RATE = vh.SAMPLE_RATE
SAMPLE_BUDGET = vh.SAMPLE_BUDGET


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_verification_47_gb300 import build
    build.build()
    sb.lib()


def _uniforms(B, K, seed):
    return np.random.default_rng(seed).uniform(size=(B, K)).astype(np.float32)


def _run(logits, dtype, B, K, V, kpr, temp, top_p, unif, mode, strides=(0, 0), dev_logits=None):
    import torch
    if dev_logits is None:
        dev_logits = torch.from_numpy(logits.view(np.int16) if dtype == wl.BF16 else logits).cuda()
    d = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(sb.sv_draft_sample_workspace_size(), dtype=torch.uint8, device="cuda")
    sb.sv_draft_sample(dev_logits, strides[0], strides[1],
                       sb.SV_BF16 if dtype == wl.BF16 else sb.SV_F32, B, K, V, d(kpr), d(temp),
                       top_p, d(unif), d(mode), out, ws, ws.numel())
    return out.cpu().numpy(), sb.sv_read_device_flags(ws)


def _compare(got, flags, logits, dtype, B, K, V, kpr, temp, top_p, unif, mode, rows=None):
    tok, margins, oflags = osm.sample_tokens(logits, dtype, B, K, V, kpr, temp, top_p, unif, mode)
    sel = np.arange(B) if rows is None else np.asarray(rows)
    diff = (got[sel] != tok[sel])
    low = margins[sel] < MARGIN
    assert not np.any(diff & ~low), np.argwhere(diff & ~low)[:10]
    SAMPLE_BUDGET["draws"] += int(np.sum(tok[sel] >= 0))
    SAMPLE_BUDGET["disagreements"] += int(np.sum(diff))
    SAMPLE_BUDGET["low_margin"] += int(np.sum(low & (tok[sel] >= 0)))
    for b, i in np.argwhere(diff):
        SAMPLE_BUDGET["log"].append((int(sel[b]), int(i), float(margins[sel[b], i])))
    if rows is None:
        assert flags == oflags, (flags, oflags)
    return tok


def _oracle_rows(args):
    """Oracle tokens of some sequences of the headline batch (a spawn worker)."""
    import sys, os
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from speculative_decoding_verification_47_gb300 import workloads as wl_
    from oracle import sample as osm_
    seqs, unif = args
    w = wl_.config_by_name("c2")
    out = []
    for b in seqs:
        tok, mg, _ = osm_.sample_tokens(w.draft[b:b + 1], w.dtype, 1, w.K, w.V, w.k_per_row[b:b + 1],
                                        w.temperature[b:b + 1], 1.0, unif[b:b + 1], w.mode[b:b + 1])
        out.append((b, tok[0], mg[0]))
    return out


def test_headline_draft_rows_full_size():
    """B=256, K=8, V=128256 bf16: the draft rows of the headline verify batch,
    sampled with its ragged k_b and per-row temperatures under ten uniform
    seeds; all 12830 tokens checked against the oracle."""
    import multiprocessing as mp
    w = wl.config_by_name("c2")
    seeds = [5150 + s for s in range(10)]
    unifs = [_uniforms(w.B, w.K, s) for s in seeds]
    nproc = max(1, min(16, (mp.cpu_count() or 1)))
    with mp.get_context("spawn").Pool(nproc) as pool:  # (spawn: this process already uses CUDA)
        jobs = [pool.map_async(_oracle_rows, [(list(range(i, w.B, nproc)), u) for i in range(nproc)])
                for u in unifs]
        results = [sum(j.get(), []) for j in jobs]
    for unif, res in zip(unifs, results):
        got, flags = _run(w.draft, w.dtype, w.B, w.K, w.V, w.k_per_row, w.temperature, 1.0, unif, w.mode)
        assert flags == 0
        for b in range(w.B):
            assert np.all(got[b, w.k_per_row[b]:] == -1) and np.all(got[b, :w.k_per_row[b]] >= 0)
        tok = np.full((w.B, w.K), -1, np.int32)
        margins = np.full((w.B, w.K), np.inf)
        for b, t, m in res:
            tok[b], margins[b] = t, m
        diff = got != tok
        low = margins < MARGIN
        assert not np.any(diff & ~low), np.argwhere(diff & ~low)[:10]
        SAMPLE_BUDGET["draws"] += int(np.sum(tok >= 0))
        SAMPLE_BUDGET["disagreements"] += int(np.sum(diff))
        SAMPLE_BUDGET["low_margin"] += int(np.sum(low & (tok >= 0)))
        for b, i in np.argwhere(diff):
            SAMPLE_BUDGET["log"].append((int(b), int(i), float(margins[b, i])))


CASES = [
    # id, B, K, V, dtype, T, top_p, mode
    ("bf16", 6, 4, 1000, wl.BF16, [0.7, 1.0, 1.6], 1.0, 0),
    ("f32", 6, 4, 1000, wl.F32, [0.7, 1.0, 1.6], 1.0, 0),
    ("bf16_topp", 5, 3, 4099, wl.BF16, [0.5, 1.0], 0.8, 0),
    ("f32_topp", 5, 3, 4099, wl.F32, [0.5, 1.0], 0.8, 0),
    ("bf16_mixed_greedy", 6, 5, 32003, wl.BF16, 0.9, 0.95, [0, 1, 0, 1, 0, 0]),
    ("bf16_large_v", 3, 2, 200003, wl.BF16, 1.0, 1.0, 0),
    ("f32_tiny_v", 8, 3, 7, wl.F32, 1.0, 0.5, 0),
    ("bf16_one_per_call", 16, 1, 50021, wl.BF16, 0.8, 0.9, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_sample_cases(case):
    _, B, K, V, dt, T, p, m = case
    T = np.resize(np.asarray(T, np.float32), B)
    kpr = np.random.default_rng(V + B).integers(0, K + 1, size=B).astype(np.int32)
    w = wl.synth_verify("sample", B, K, V, dt, kpr, T, 1.0, m, top_p=p,
                        seeds=(9000 + V, 9100 + B, 9200 + K))
    unif = _uniforms(B, K, 9300 + V)
    got, flags = _run(w.draft, dt, B, K, V, kpr, T, w.top_p, unif, w.mode)
    _compare(got, flags, w.draft, dt, B, K, V, kpr, T, w.top_p, unif, w.mode)


def test_padded_layout_and_null_knobs():
    """Rows padded to a larger stride; k_per_row, temperature and mode NULL
    (every row sampled at T = 1 over all K positions)."""
    import torch
    B, K, V, pad = 4, 3, 3001, 7
    w = wl.synth_verify("pad", B, K, V, wl.BF16, K, 1.0, 1.0, 0, seeds=(9400, 9401, 9402))
    buf = np.zeros((B, K, V + pad), np.uint16)
    buf[:, :, :V] = w.draft
    dev = torch.from_numpy(buf.view(np.int16)).cuda()
    unif = _uniforms(B, K, 9403)
    got, flags = _run(None, wl.BF16, B, K, V, None, None, 1.0, unif, None,
                      strides=(K * (V + pad), V + pad), dev_logits=dev)
    _compare(got, flags, w.draft, wl.BF16, B, K, V, np.full(B, K, np.int32), np.ones(B, np.float32),
             1.0, unif, np.zeros(B, np.uint8))


def test_error_paths():
    """A NaN row and a bad uniform fail only their own position; a bad
    temperature or k_b fails the whole sequence; the flag word says which."""
    B, K, V = 5, 3, 2003
    w = wl.synth_verify("err", B, K, V, wl.F32, K, 1.0, 1.0, 0, seeds=(9500, 9501, 9502))
    logits = w.draft.copy()
    logits[0, 1, 17] = np.nan
    unif = _uniforms(B, K, 9503)
    unif[1, 2] = 1.0
    T = np.ones(B, np.float32)
    T[2] = 0.0
    kpr = np.full(B, K, np.int32)
    kpr[3] = K + 1
    mode = np.zeros(B, np.uint8)
    got, flags = _run(logits, wl.F32, B, K, V, kpr, T, 1.0, unif, mode)
    assert got[0, 1] == -1 and got[0, 0] >= 0 and got[0, 2] >= 0
    assert got[1, 2] == -1 and got[1, 1] >= 0
    assert np.all(got[2] == -1) and np.all(got[3] == -1) and np.all(got[4] >= 0)
    assert flags == (ov.FLAG_NONFINITE | ov.FLAG_BAD_UNIFORM | ov.FLAG_BAD_TEMPERATURE |
                     ov.FLAG_BAD_K)
    _compare(got, flags, logits, wl.F32, B, K, V, kpr, T, 1.0, unif, mode)


def test_zz_sample_disagreement_budget():
    """Low-margin disagreements over this module's draws stay under RATE (the
    session summary prints the counts)."""
    n, x = SAMPLE_BUDGET["draws"], SAMPLE_BUDGET["disagreements"]
    if n == 0:
        pytest.skip("no sampler parity test ran before this one in the session")
    assert x <= RATE * n, (x, n, SAMPLE_BUDGET["log"])

"""GPU parity of the top-p path of sv_spec_verify (nucleus truncation of both
the target and the draft distributions before the accept test, the
residual and the bonus draw) against the float64 oracle, through the C ABI.

Cases: the mixed greedy / sampled workload at full size (V=151936, top_p=0.9),
both logit types over a range of top_p, cuts that fall inside groups of equal
logits (ties broken by index), a completely flat row, near-degenerate top_p
(a single kept token; almost everything kept), windows wide enough to need
the fixed-point mass pass on bf16, a tie of 300 top tokens that the candidates'
ranking resolves by index, and rows whose target and draft copies sit at
different 16-byte phases."""

import numpy as np
import pytest

from tests.conftest import gpu_available
from tests import verify_harness as vh
from speculative_decoding_verification_47_gb300 import binding as sb
from speculative_decoding_verification_47_gb300 import workloads as wl

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_verification_47_gb300 import build
    build.build()
    sb.lib()


def _check(w, **kw):
    g = vh.run_gpu(w, **kw)
    o = vh.run_oracle(w)
    return vh.compare(w, g, o), g, o


def _logits(w, a):
    return wl.bf16_bits_to_f32(a).astype(np.float64) if w.dtype == wl.BF16 else a.astype(np.float64)


def _store(w, z):
    return wl.f64_to_bf16_bits(z) if w.dtype == wl.BF16 else z.astype(np.float32)


def test_c3_full_size_top_p():
    """B=128, k=6, V=151936 bf16, T=0.7, top_p=0.9, half the rows greedy."""
    w = wl.config_c3()
    assert w.top_p == float(np.float32(0.9))
    (dec, dis), g, o = _check(w)
    assert dec > 0


CASES = [
    # id, B, K, V, dtype, T, sigma, top_p, mode
    ("bf16_p0.9", 6, 4, 1000, wl.BF16, [0.7, 1.0], 1.0, 0.9, 0),
    ("f32_p0.9", 6, 4, 1000, wl.F32, [0.7, 1.0], 1.0, 0.9, 0),
    ("bf16_p0.5", 5, 3, 4099, wl.BF16, 1.0, 0.5, 0.5, 0),
    ("f32_p0.5", 5, 3, 4099, wl.F32, 1.0, 0.5, 0.5, 0),
    ("bf16_p0.99", 4, 5, 32003, wl.BF16, [0.1, 0.7, 1.0, 1.7], 2.0, 0.99, 0),
    ("f32_p0.99", 4, 5, 32003, wl.F32, [0.1, 0.7, 1.0, 1.7], 2.0, 0.99, 0),
    ("bf16_mix_large", 3, 2, 200003, wl.BF16, 0.8, 1.0, 0.9, [0, 1, 0]),
    ("f32_tiny_vocab", 8, 3, 7, wl.F32, 1.0, 1.0, 0.3, 0),
    ("bf16_one_token", 8, 3, 5003, wl.BF16, 1.0, 1.0, 0.001, 0),
    ("bf16_almost_all", 4, 2, 5003, wl.BF16, 1.0, 1.0, 0.999999, 0),
    ("bf16_hot_wide_window", 4, 3, 20011, wl.BF16, 20.0, 1.0, 0.9, 0),
    ("f32_hot_wide_window", 4, 3, 20011, wl.F32, 20.0, 1.0, 0.9, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_top_p_cases(case):
    _, B, K, V, dt, T, s, p, m = case
    T = np.resize(np.asarray(T, np.float32), B)  # per-row temperatures, cycled
    w = wl.synth_verify("topp", B, K, V, dt, K, T, s, m, top_p=p,
                        seeds=(8000 + V, 8100 + B, 8200 + K))
    _check(w)


@pytest.mark.parametrize("dt", [wl.BF16, wl.F32])
@pytest.mark.parametrize("top_p", [0.3, 0.75, 0.9])
def test_cut_inside_groups_of_equal_logits(dt, top_p):
    """Logits rounded to a coarse grid: every value is shared by many tokens,
    so the cut nearly always falls inside a group and the index order of the
    tied tokens decides which of them are kept."""
    B, K, V = 6, 4, 6007
    w = wl.synth_verify("ties", B, K, V, dt, K, 1.0, 1.0, 0, top_p=top_p,
                        seeds=(8300, 8301, int(top_p * 100)))
    w.target = _store(w, np.round(_logits(w, w.target) * 2.0) / 2.0)
    w.draft = _store(w, np.round(_logits(w, w.draft) * 2.0) / 2.0)
    _check(w)


@pytest.mark.parametrize("dt", [wl.BF16, wl.F32])
def test_large_tie_group_among_candidates(dt):
    """300 tokens at the row's top logit, scattered over a row of N(0,1)
    logits (131072 bf16 or 32768 fp32 tokens): the cluster's list floor
    mostly stays far below them, so the cut is taken from a few hundred
    candidates, and all 300 tied tokens fall into one value bin (more than
    the local ranking takes), so they are ranked by the distributed count;
    a row whose floor reaches the tie takes the passes.  top_p = 0.5 cuts
    inside the tie: which tied tokens are kept is decided by index order."""
    B, K = 2, 2
    V = 131072 if dt == wl.BF16 else 32768
    w = wl.synth_verify("bigtie", B, K, V, dt, K, 1.0, 1.0, 0, top_p=0.5, seeds=(8500, 8501, 8502))
    r = np.random.default_rng(8503)
    for a in (w.target, w.draft):
        z = r.standard_normal(a.shape)
        for b in range(B):
            for i in range(a.shape[1]):
                z[b, i, r.choice(V, size=300, replace=False)] = 10.0
        a[...] = _store(w, z)
    (dec, dis), g, o = _check(w)
    assert dec > 0


@pytest.mark.parametrize("dt", [wl.BF16, wl.F32])
def test_flat_rows(dt):
    """Every logit equal: one group of V tied tokens; top_p=0.5 keeps the
    first floor(V/2)+1 of them by index (V odd, so no token sits exactly on
    the threshold).  Draft tokens in the dropped half are rejected."""
    B, K, V = 4, 3, 1001
    w = wl.synth_verify("flat", B, K, V, dt, K, 1.0, 1.0, 0, top_p=0.5, seeds=(8400, 8401, 8402))
    w.target = _store(w, np.zeros_like(_logits(w, w.target)))
    w.draft = _store(w, np.zeros_like(_logits(w, w.draft)))
    r = np.random.default_rng(8403)
    w.draft_tokens[:] = r.integers(0, V, size=(B, K))
    (dec, dis), g, o = _check(w)
    for b in range(B):
        kept = V // 2 + 1
        # a token of the dropped half is rejected at once; the resample is kept
        if w.draft_tokens[b, 0] >= kept:
            assert g.n[b] == 0
        assert 0 <= g.out[b, g.n[b]] < kept


def test_mixed_phase_rows():
    """Padded layouts whose target and draft rows start at different 16-byte
    phases (element-wise paths of the count, tie and residual passes)."""
    import torch
    B, K, V = 4, 3, 3001
    w = wl.synth_verify("phase", B, K, V, wl.BF16, K, 0.7, 1.0, 0, top_p=0.8,
                        seeds=(8500, 8501, 8502))
    w.target = _store(w, np.round(_logits(w, w.target) * 4.0) / 4.0)
    w.draft = _store(w, np.round(_logits(w, w.draft) * 4.0) / 4.0)
    pt, pd = 5, 2
    tgt = np.zeros((B, K + 1, V + pt), np.uint16)
    tgt[:, :, :V] = w.target
    drf = np.zeros((B, K, V + pd), np.uint16)
    drf[:, :, :V] = w.draft
    dev = vh.to_device(w)
    dev["target"] = torch.from_numpy(tgt.view(np.int16)).cuda()
    dev["draft"] = torch.from_numpy(drf.view(np.int16)).cuda()
    strides = ((K + 1) * (V + pt), V + pt, K * (V + pd), V + pd)
    g = vh.run_gpu(w, dev=dev, strides=strides)
    vh.compare(w, g, vh.run_oracle(w))


def test_top_p_one_and_just_below_one():
    """top_p = 1 takes the untruncated kernel, the largest float below 1 the
    truncating one (a full-width key window: mass pass, then count pass);
    both agree with the oracle on the same rows."""
    B, K, V = 6, 4, 8009
    w = wl.synth_verify("p1", B, K, V, wl.BF16, K, 1.0, 1.0, 0, top_p=1.0, seeds=(8600, 8601, 8602))
    g1 = vh.run_gpu(w)
    vh.compare(w, g1, vh.run_oracle(w))
    w.top_p = float(np.float32(1.0 - 2.0 ** -24))
    g2 = vh.run_gpu(w)
    vh.compare(w, g2, vh.run_oracle(w))


TARGET_ONLY = [
    # id, B, K, V, dtype, T, top_p, mode
    ("bf16_p0.9", 6, 4, 1000, wl.BF16, [0.7, 1.0], 0.9, 0),
    ("f32_p0.5", 5, 3, 4099, wl.F32, 1.0, 0.5, 0),
    ("bf16_p0.99_mix", 6, 5, 32003, wl.BF16, [0.1, 0.7, 1.7], 0.99, [0, 1, 0, 0, 1, 0]),
    ("bf16_one_token", 8, 3, 5003, wl.BF16, 1.0, 0.001, 0),
]


@pytest.mark.parametrize("case", TARGET_ONLY, ids=[c[0] for c in TARGET_ONLY])
def test_target_only_top_p(case):
    """sv_spec_verify_target_topp: the draft keeps its untruncated softmax
    (draft tokens outside the target nucleus are rejected by p' = 0)."""
    _, B, K, V, dt, T, p, m = case
    T = np.resize(np.asarray(T, np.float32), B)
    w = wl.synth_verify("tonly", B, K, V, dt, K, T, 1.0, m, top_p=p,
                        seeds=(8700 + V, 8800 + B, 8900 + K))
    g = vh.run_gpu(w, target_topp=True)
    vh.compare(w, g, vh.run_oracle(w, topp_draft=False))


def test_c3_full_size_target_only_top_p():
    """The mixed top-p batch at full size with the draft untruncated."""
    w = wl.config_c3()
    g = vh.run_gpu(w, target_topp=True)
    dec, _ = vh.compare(w, g, vh.run_oracle(w, topp_draft=False))
    assert dec > 0


def test_target_only_equals_both_at_top_p_one():
    B, K, V = 4, 3, 3001
    w = wl.synth_verify("t1", B, K, V, wl.BF16, K, 1.0, 1.0, 0, top_p=1.0, seeds=(8950, 8951, 8952))
    a = vh.run_gpu(w)
    b = vh.run_gpu(w, target_topp=True)
    assert np.array_equal(a.out, b.out) and np.array_equal(a.n, b.n)

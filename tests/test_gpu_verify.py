"""GPU parity of sv_spec_verify / sv_kv_commit against the float64 oracle,
through the C ABI, on the seeded workloads and on edge cases."""

import numpy as np
import pytest

from tests.conftest import gpu_available
from tests import verify_harness as vh
from oracle import verify as ov
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


# ---------------------------------------------------------------- workloads

def test_c0_single_rounds():
    for r in range(8):
        _check(wl.config_c0(r))


def test_c0_64_rounds_batched():
    _check(wl.config_c0_batched(64))


def test_c1_verify_and_commit():
    import torch
    w = wl.config_c1()
    (dec, dis), g, o = _check(w)
    seq = torch.from_numpy(w.seq_lens).cuda()
    cap = torch.from_numpy(w.capacity).cuda()
    n = torch.from_numpy(g.n).cuda()
    ws = torch.zeros(sb.sv_workspace_size(w.B, w.K, w.V, sb.SV_BF16), dtype=torch.uint8, device="cuda")
    sb.sv_kv_commit(seq, n, cap, torch.from_numpy(w.k_per_row).cuda(), w.B, w.K, ws, ws.numel())
    ref, rflags = ov.kv_commit(w.seq_lens, o.n_accepted, w.capacity, w.K, w.k_per_row)
    np.testing.assert_array_equal(seq.cpu().numpy(), ref)
    assert sb.sv_read_device_flags(ws) == rflags == 0
    assert np.all(seq.cpu().numpy() - w.seq_lens == g.n)


def test_c2_full_size():
    _check(wl.config_c2())


def test_c3_greedy_half_full_size():
    w = wl.config_c3()
    w.top_p = 1.0  # greedy rows ignore top-p; sampled rows run untruncated here
    _check(w)


# ---------------------------------------------------------------- shapes

SHAPES = [
    # B, K, V, dtype, k spec, modes
    (1, 0, 1, wl.F32, 0, 0),
    (3, 1, 7, wl.BF16, [1, 0, 1], [0, 1, 0]),
    (4, 3, 8, wl.F32, [3, 2, 1, 0], 0),
    (5, 4, 33, wl.BF16, [4, 0, 2, 3, 1], [0, 0, 1, 1, 0]),
    (9, 5, 257, wl.BF16, "rand", "mix"),
    (6, 6, 1000, wl.F32, "rand", "mix"),
    (7, 8, 4099, wl.BF16, "rand", "mix"),
    (8, 2, 65537, wl.F32, "rand", 0),
    (16, 7, 200003, wl.BF16, "rand", "mix"),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}K{s[1]}V{s[2]}{s[3]}" for s in SHAPES])
def test_shapes(shape):
    B, K, V, dt, kspec, mspec = shape
    r = np.random.default_rng(B * 1000 + V)
    k = r.integers(0, K + 1, size=B) if isinstance(kspec, str) else kspec
    m = (r.integers(0, 2, size=B) if mspec == "mix" else mspec)
    T = r.choice([0.1, 0.7, 1.0, 1.7], size=B).astype(np.float32)
    s = r.choice([0.3, 1.0, 2.0], size=B)
    w = wl.synth_verify("shape", B, K, V, dt, k, T, s, m, seeds=(7000 + V, 7100 + V, 7200 + V))
    _check(w)


def test_strided_layout_and_null_optionals():
    """Non-packed layouts (row padding, sequence padding) and NULL k/T/mode."""
    import torch
    B, K, V = 4, 3, 1001
    w = wl.synth_verify("stride", B, K, V, wl.BF16, K, 1.0, 1.0, 0, seeds=(11, 12, 13))
    pad_v, pad_s = 6, 3  # 2014-byte rows: not 16-byte aligned
    tgt = np.zeros((B, K + 1 + pad_s, V + pad_v), np.uint16)
    tgt[:, :K + 1, :V] = w.target
    drf = np.zeros((B, K + pad_s, V + pad_v), np.uint16)
    drf[:, :K, :V] = w.draft
    dev = vh.to_device(w)
    dev["target"] = torch.from_numpy(tgt.view(np.int16)).cuda()
    dev["draft"] = torch.from_numpy(drf.view(np.int16)).cuda()
    strides = ((K + 1 + pad_s) * (V + pad_v), V + pad_v, (K + pad_s) * (V + pad_v), V + pad_v)
    g = vh.run_gpu(w, dev=dev, strides=strides, pass_kpr=False, pass_mode=False, pass_temp=False)
    vh.compare(w, g, vh.run_oracle(w))


def test_all_greedy_without_draft_logits():
    w = wl.synth_verify("greedy", 5, 4, 3001, wl.BF16, [4, 3, 0, 4, 2], 0.7, 1.0, 1,
                        seeds=(21, 22, 23))
    g = vh.run_gpu(w, draft=False)
    vh.compare(w, g, vh.run_oracle(w))


def test_p_equals_q_accepts_all_and_disjoint_rejects_first():
    B, K, V = 6, 5, 5003
    w = wl.synth_verify("pq", B, K, V, wl.F32, K, 0.9, 0.0, 0, seeds=(31, 32, 33))
    w.draft = w.target[:, :K].copy()
    (d, x), g, o = _check(w)
    assert np.all(g.n == K)
    w2 = wl.synth_verify("disj", B, K, V, wl.F32, K, 1.0, 1.0, 0, seeds=(34, 35, 36))
    half = np.arange(V) < V // 2
    w2.target[:, :, ~half] = -np.inf
    w2.draft[:, :, half] = -np.inf
    rr = np.random.default_rng(0)
    w2.draft_tokens[:] = rr.integers(V // 2, V, size=(B, K))
    (d, x), g, o = _check(w2)
    assert np.all(g.n == 0) and np.all(g.out[:, 0] < V // 2)


# ---------------------------------------------------------------- errors

def _fault_case():
    return wl.synth_verify("fault", 6, 4, 2049, wl.BF16, 4, 1.0, 0.3, 0, seeds=(41, 42, 43))


@pytest.mark.parametrize("fault", ["nan_pos0", "inf_pos0", "bad_token", "bad_k", "bad_T",
                                   "bad_u", "bad_uK", "bad_mode", "allneginf", "nan_past_cut"])
def test_device_faults(fault):
    w = _fault_case()
    b = 2
    if fault == "nan_pos0":
        w.target[b, 0, 100] = wl.BF16_NAN
    elif fault == "inf_pos0":
        w.draft[b, 0, 5] = 0x7F80
    elif fault == "bad_token":
        w.draft_tokens[b, 0] = w.V
    elif fault == "bad_k":
        w.k_per_row[b] = w.K + 1
    elif fault == "bad_T":
        w.temperature[b] = 0.0
    elif fault == "bad_u":
        w.uniforms[b, 0] = 1.0
    elif fault == "bad_uK":
        w.uniforms[b, w.K] = -0.5
    elif fault == "bad_mode":
        w.mode[b] = 3
    elif fault == "allneginf":
        w.target[b, 0, :] = 0xFF80
    elif fault == "nan_past_cut":
        # make position 0 reject for sure, then poison position 2
        w.target[b, 0, w.draft_tokens[b, 0]] = 0xFF80  # p(x0) = 0
        w.target[b, 2, 7] = wl.BF16_NAN
    g = vh.run_gpu(w)
    o = vh.run_oracle(w)
    vh.compare(w, g, o)
    if fault == "nan_past_cut":
        assert g.flags == 0 and g.n[b] == 0 and g.out[b, 0] >= 0
    else:
        assert g.flags != 0 and g.n[b] == 0 and np.all(g.out[b] == -1)


def test_kv_commit_faults():
    import torch
    B, K = 300, 8
    r = np.random.default_rng(3)
    s0 = r.integers(0, 5000, size=B).astype(np.int32)
    n = r.integers(0, K + 1, size=B).astype(np.int32)
    n[5], n[6] = -1, K + 1
    cap = (s0 + r.integers(0, 10, size=B)).astype(np.int32)
    seq = torch.from_numpy(s0).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    sb.sv_kv_commit(seq, torch.from_numpy(n).cuda(), torch.from_numpy(cap).cuda(), None, B, K, ws, 256)
    ref, rf = ov.kv_commit(s0, n, cap, K)
    np.testing.assert_array_equal(seq.cpu().numpy(), ref)
    assert sb.sv_read_device_flags(ws) == rf
    assert rf & ov.FLAG_BAD_N and rf & ov.FLAG_CAPACITY


def test_kv_commit_ragged_k_rejects_more_than_drafted():
    """With the round's k_per_row, a sequence whose n exceeds its own k_b (but
    not K) is left unchanged and flagged; the others move by n."""
    import torch
    B, K = 500, 8
    r = np.random.default_rng(5)
    s0 = r.integers(0, 5000, size=B).astype(np.int32)
    kb = r.integers(0, K + 1, size=B).astype(np.int32)
    n = np.array([r.integers(0, k + 1) for k in kb], np.int32)
    over = np.nonzero(kb < K)[0][:7]
    n[over] = kb[over] + 1  # in (k_b, K]
    seq = torch.from_numpy(s0).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    sb.sv_kv_commit(seq, torch.from_numpy(n).cuda(), None, torch.from_numpy(kb).cuda(), B, K, ws, 256)
    ref, rf = ov.kv_commit(s0, n, None, K, kb)
    got = seq.cpu().numpy()
    np.testing.assert_array_equal(got, ref)
    assert sb.sv_read_device_flags(ws) == rf == ov.FLAG_BAD_N
    assert np.all(got[over] == s0[over])


# ---------------------------------------------------------------- reuse

def test_workspace_reuse_and_determinism():
    import torch
    w = wl.config_c1(B=16)
    ws = torch.empty(sb.sv_workspace_size(w.B, w.K, w.V, sb.SV_BF16), dtype=torch.uint8,
                     device="cuda")
    dev = vh.to_device(w)
    a = vh.run_gpu(w, dev=dev, workspace=ws)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = vh.run_gpu(w, dev=dev, workspace=ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(a.out, b.out)
    np.testing.assert_array_equal(a.n, b.n)
    vh.compare(w, a, vh.run_oracle(w))


def test_zz_disagreement_budget():
    """Low-margin disagreements over every verify parity comparison of this
    session stay under 1e-4 of the decisions taken (each comparison also
    checks its own share; the session summary prints the counts)."""
    d, x = vh.BUDGET["decisions"], vh.BUDGET["disagreements"]
    if d == 0:
        pytest.skip("no verify parity comparison ran before this one in the session")
    assert x <= vh.RATE * d, (x, d, vh.BUDGET_LOG)

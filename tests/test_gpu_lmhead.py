"""GPU parity of sv_lmhead_rmsnorm (final RMSNorm + LM head on tcgen05) against
the float64 oracle, and of the layer-skip draft-logit producer feeding
sv_spec_verify end to end.

Tolerances (per output, derived from the arithmetic):
  * against the float64 oracle: |d| <= 2^-7 * sum_k |y_k W_kn| + 2^-8 * |ref|
    (bf16 rounding of the normalised row y, fp32 accumulation, and the bf16
    rounding of the output);
  * against the bf16-mimic oracle (y rounded to bf16 first, exact products):
    |d| <= 2^-11 * sum_k |y_k W_kn| (+ 2^-8 |ref| for bf16 output), which
    leaves room only for fp32 summation error and the rare element whose
    float32 y rounds to the other neighbouring bf16 value.
"""

import numpy as np
import pytest

from tests.conftest import gpu_available
from tests import verify_harness as vh
from oracle import lmhead as ol
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


def _run(x: wl.LMHeadInputs, out_dt=sb.SV_BF16, hidden=None):
    import torch
    h = x.hidden if hidden is None else hidden
    dh = torch.from_numpy(h.view(np.int16)).cuda()
    dw = torch.from_numpy(x.norm_w.view(np.int16)).cuda()
    dW = torch.from_numpy(x.W.view(np.int16)).cuda()
    tdt = torch.float32 if out_dt == sb.SV_F32 else torch.bfloat16
    out = torch.full((x.M, x.V), float("nan"), dtype=tdt, device="cuda")
    ws = torch.zeros(sb.sv_lmhead_workspace_size(x.M, x.H), dtype=torch.uint8, device="cuda")
    sb.sv_lmhead_rmsnorm(dh, dw, x.eps, dW, out, out_dt, x.M, x.H, x.V, ws, ws.numel())
    flags = sb.sv_read_device_flags(ws)
    return out, flags


def _mimic(x, rows=None):
    """float64 product of the bf16-rounded normalised rows."""
    h = ov.bf16_bits_to_f64(x.hidden if rows is None else x.hidden[rows])
    w = ov.bf16_bits_to_f64(x.norm_w)
    y = ov.bf16_bits_to_f64(wl.f64_to_bf16_bits(ol.rmsnorm(h, w, x.eps)))
    W = ov.bf16_bits_to_f64(x.W)
    return y @ W


def _check(x, got, out_dt, rows=None):
    if rows is None:
        ref = ol.lmhead_rmsnorm(x.hidden, x.norm_w, x.eps, x.W)
        absp = ol.lmhead_abs_product(x.hidden, x.norm_w, x.eps, x.W)
    else:
        ref, absp = ol.lmhead_rows(x.hidden, x.norm_w, x.eps, x.W, rows)
        got = got[rows]
    out_round = 2.0 ** -8 * np.abs(ref) if out_dt == sb.SV_BF16 else 0.0
    bound = 2.0 ** -7 * absp + 2.0 ** -8 * np.abs(ref)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))
    mim = _mimic(x, rows)
    tight = 2.0 ** -11 * absp + out_round
    assert np.all(np.abs(got - mim) <= tight), float(np.max(np.abs(got - mim) / tight))


SHAPES = [
    # M, H, V: one tile; several k blocks; row and column tails; many tiles
    (128, 64, 256),
    (128, 1024, 256),
    (130, 192, 272),
    (1, 64, 16),
    (257, 512, 1040),
    (512, 256, 4096),
]


@pytest.mark.parametrize("out_dt", [sb.SV_BF16, sb.SV_F32], ids=["bf16", "f32"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"M{s[0]}H{s[1]}V{s[2]}" for s in SHAPES])
def test_lmhead_shapes(shape, out_dt):
    M, H, V = shape
    x = wl.lmhead_inputs(M=M, H=H, V=V, seed=M * 7 + H + V)
    out, flags = _run(x, out_dt)
    assert flags == 0
    _check(x, out.float().cpu().numpy().astype(np.float64), out_dt)


def test_lmhead_norm_is_applied():
    """Scaling the hidden states by 16 leaves the logits unchanged (the
    RMSNorm the layer-skip draft must not skip); with eps = 0 the scaling is
    exact at every step, so the outputs are identical."""
    x = wl.lmhead_inputs(M=128, H=256, V=512, seed=11)
    x.eps = 0.0
    h16 = wl.f64_to_bf16_bits(ov.bf16_bits_to_f64(x.hidden) * 16.0)
    a, _ = _run(x, sb.SV_F32)
    b, _ = _run(x, sb.SV_F32, hidden=h16)
    a = a.cpu().numpy()
    b = b.cpu().numpy()
    np.testing.assert_array_equal(a, b)


def test_lmhead_c4_full_size_every_row():
    """M=512, H=4096, V=32000 (the layer-skip workload, on the persistent
    BN=224 cluster schedule that only this size takes): every one of the
    512 x 32000 outputs checked against the float64 oracle and the
    bf16-mimic bound."""
    x = wl.lmhead_inputs()
    out, flags = _run(x, sb.SV_BF16)
    assert flags == 0
    _check(x, out.float().cpu().numpy().astype(np.float64), sb.SV_BF16)


def test_c4_layer_skip_draft_then_verify():
    """Draft logits from layer-L hidden states and target logits from the
    perturbed ones, both through sv_lmhead_rmsnorm, fed straight into
    sv_spec_verify (B=64, k=7, T=1); the oracle verifies the same logits."""
    import torch
    x = wl.lmhead_inputs()
    B, K, V = 64, 7, x.V
    dl, f1 = _run(x, sb.SV_BF16)
    tl, f2 = _run(x, sb.SV_BF16, hidden=x.hidden_t)
    assert f1 == 0 and f2 == 0
    knobs = wl.c4_verify_knobs(B, K)
    d_bits = dl.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B, K + 1, V)
    t_bits = tl.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B, K + 1, V)
    tokens = wl.draw_draft_tokens(d_bits[:, :K], wl.BF16, knobs["k_per_row"],
                                  knobs["temperature"], knobs["mode"], seed=4004)
    w = wl.VerifyInputs(name="c4", dtype=wl.BF16, B=B, K=K, V=V, target=t_bits,
                        draft=np.ascontiguousarray(d_bits[:, :K]), draft_tokens=tokens,
                        k_per_row=knobs["k_per_row"], temperature=knobs["temperature"],
                        top_p=1.0, uniforms=knobs["uniforms"], mode=knobs["mode"],
                        sigma=np.zeros(B))
    dev = vh.to_device(w)
    dev["target"] = tl.view(torch.int16).reshape(B, K + 1, V)
    dev["draft"] = dl.view(torch.int16).reshape(B, K + 1, V)  # position K unused
    g = vh.run_gpu(w, dev=dev, strides=(0, 0, (K + 1) * V, V))
    dec, dis = vh.compare(w, g, vh.run_oracle(w))
    assert dec > B


def test_lmhead_norm_weight_two_byte_aligned():
    """The RMSNorm weight needs only 2-byte alignment: a weight vector that
    starts one element into its buffer gives the same bits as an aligned one."""
    import torch
    x = wl.lmhead_inputs(M=130, H=512, V=272, seed=21)
    a, _ = _run(x, sb.SV_F32)
    dh = torch.from_numpy(x.hidden.view(np.int16)).cuda()
    buf = torch.zeros(x.H + 8, dtype=torch.int16, device="cuda")
    buf[1:1 + x.H] = torch.from_numpy(x.norm_w.view(np.int16)).cuda()
    dw = buf[1:1 + x.H]
    assert dw.data_ptr() % 16 != 0
    dW = torch.from_numpy(x.W.view(np.int16)).cuda()
    out = torch.full((x.M, x.V), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(sb.sv_lmhead_workspace_size(x.M, x.H), dtype=torch.uint8, device="cuda")
    sb.sv_lmhead_rmsnorm(dh, dw, x.eps, dW, out, sb.SV_F32, x.M, x.H, x.V, ws, ws.numel())
    assert sb.sv_read_device_flags(ws) == 0
    np.testing.assert_array_equal(a.cpu().numpy(), out.cpu().numpy())

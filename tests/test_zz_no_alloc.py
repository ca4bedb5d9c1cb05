"""The allocation-free verify entry point, for callers with no device
allocator of their own (plugins whose memory the host framework owns,
real-time loops that cannot afford a cudaMalloc): same results as
sv_spec_verify with a workspace, two calls in a row sharing the library's
built-in scratch, and a clear refusal above its size limit.

Kept in a file that pytest collects last, so a run that stops at the first
failure has already run every other test."""

import numpy as np
import pytest

from tests.conftest import gpu_available
from speculative_decoding_verification_47_gb300 import binding as sb
from speculative_decoding_verification_47_gb300 import workloads as wl

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_verification_47_gb300 import build
    build.build()
    sb.lib()


def _inputs(seed):
    k = np.random.default_rng(seed).integers(0, 6, size=24)
    return wl.synth_verify("noalloc", 24, 5, 50021, wl.BF16, k, [0.1, 0.7, 1.0] * 8,
                           [0.3, 1.0, 2.0] * 8, [0, 0, 1] * 8, seeds=(seed, seed + 1, seed + 2))


def _run(w, noalloc):
    import torch
    d = lambda a: torch.from_numpy(a).cuda()
    args = [d(w.target.view(np.int16)), 0, 0, d(w.draft.view(np.int16)), 0, 0, sb.SV_BF16,
            w.B, w.K, w.V, d(w.draft_tokens), d(w.k_per_row), d(w.temperature), w.top_p,
            d(w.uniforms), d(w.mode)]
    out = torch.full((w.B, w.K + 1), -7, dtype=torch.int32, device="cuda")
    n = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    dg = torch.full((w.B, w.K + 1, sb.SV_DIAG_FIELDS), float("nan"), device="cuda")
    if noalloc:
        sb.sv_spec_verify_noalloc(*args, out, n, dg)
    else:
        wsb = sb.sv_workspace_size(w.B, w.K, w.V, sb.SV_BF16)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        sb.sv_spec_verify(*args, out, n, dg, ws, wsb)
    torch.cuda.synchronize()
    return out.cpu().numpy(), n.cpu().numpy(), dg.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_twice():
    for seed in (101, 202):  # two calls in a row share the built-in scratch
        w = _inputs(seed)
        o_ref, n_ref, d_ref = _run(w, noalloc=False)
        o, n, d = _run(w, noalloc=True)
        np.testing.assert_array_equal(o, o_ref)
        np.testing.assert_array_equal(n, n_ref)
        # diagnostics of positions up to the cut (later rows may or may not
        # be read, depending on when the earlier rejection became visible)
        for b in range(w.B):
            np.testing.assert_allclose(d[b, : n[b] + 1], d_ref[b, : n[b] + 1], rtol=1e-5,
                                       atol=0, equal_nan=True)
        assert (n >= 0).all() and (o[:, 0] >= 0).all()


def test_noalloc_refuses_batches_above_its_scratch():
    with pytest.raises(sb.SVError) as e:
        sb.sv_spec_verify_noalloc(1 << 20, 0, 0, 1 << 20, 0, 0, sb.SV_BF16, 8192, 20, 32000,
                                  1 << 20, None, None, 1.0, 1 << 20, None, 1 << 20, 1 << 20,
                                  None)
    assert e.value.status == sb.SV_ERR_WORKSPACE
    assert "scratch" in str(e.value)

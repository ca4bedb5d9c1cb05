"""GPU parity of the dynamic-k controller (sv_dynk_init / sv_dynk_update)
against the oracle: integer logic, so k_next must match exactly in every
round.  Random acceptance histories over more than one window (300 rounds),
rounds without speculation, per-sequence caps, invalid rounds."""

import numpy as np
import pytest

from tests.conftest import gpu_available
from oracle import dynk
from speculative_decoding_verification_47_gb300 import binding as sb

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_verification_47_gb300 import build
    build.build()
    sb.lib()


@pytest.mark.parametrize("with_cap", [False, True], ids=["no_cap", "cap"])
def test_dynk_matches_oracle_over_300_rounds(with_cap):
    import torch
    B, R = 300, 300
    rng = np.random.default_rng(77 + with_cap)
    alpha = rng.uniform(0.3, 1.0, size=B)
    state = torch.zeros(sb.sv_dynk_state_size(B), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    sb.sv_dynk_init(state, B, 4, None)
    ctl = [dynk.DynK(4) for _ in range(B)]
    k_cur = np.array([c.k for c in ctl], np.int32)
    for r in range(R):
        # the k of this round: the controller's previous answer, sometimes 0
        ku = np.where(rng.uniform(size=B) < 0.05, 0, np.maximum(k_cur, 0)).astype(np.int32)
        drift = np.clip(alpha + 0.3 * np.sin(r / 25.0 + np.arange(B)), 0.0, 1.0)
        n = rng.binomial(ku, drift).astype(np.int32)
        bad = rng.uniform(size=B) < 0.01
        n[bad] = ku[bad] + 1
        cap = rng.integers(0, 9, size=B).astype(np.int32) if with_cap else None
        dn = torch.from_numpy(n).cuda()
        dk = torch.from_numpy(ku).cuda()
        dc = torch.from_numpy(cap).cuda() if with_cap else None
        out = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        sb.sv_dynk_update(state, B, dn, dk, dc, out, ws, 256, None)
        got = out.cpu().numpy()
        ref = np.array([c.update(int(n[b]), int(ku[b]), None if cap is None else int(cap[b]))
                        for b, c in enumerate(ctl)], np.int32)
        assert np.array_equal(got, ref), (r, np.argwhere(got != ref)[:5])
        k_cur = ref
    flags = sb.sv_read_device_flags(ws)
    assert flags == (256 if any(c.flags for c in ctl) else 0)
    assert len({int(c.k) for c in ctl}) > 1  # the controllers moved


def test_dynk_init_clamps():
    import torch
    B = 5
    state = torch.zeros(sb.sv_dynk_state_size(B), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    for k0, want in [(0, 2), (5, 5), (12, 8)]:
        sb.sv_dynk_init(state, B, k0, None)
        z = torch.zeros(B, dtype=torch.int32, device="cuda")
        out = torch.empty(B, dtype=torch.int32, device="cuda")
        sb.sv_dynk_update(state, B, z, z, None, out, ws, 256, None)
        assert out.cpu().numpy().tolist() == [want] * B


def test_dynk_bench_workload():
    """The history bench.py times at its defaults (--workload dynk: 20 warm-up
    rounds, 2000 timed rounds and one more): B=256 controllers, k_used ~U{2..8},
    n ~U{0..k_used}; k_next identical to the oracle in every round."""
    import torch
    from speculative_decoding_verification_47_gb300 import workloads as wl
    B, R = 256, 2021
    nh, kh = wl.dynk_history(B, R)
    state = torch.zeros(sb.sv_dynk_state_size(B), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    sb.sv_dynk_init(state, B, 4, None)
    dn = torch.from_numpy(nh).cuda()
    dk = torch.from_numpy(kh).cuda()
    outs = torch.full((R, B), -7, dtype=torch.int32, device="cuda")
    for r in range(R):
        sb.sv_dynk_update(state, B, dn[r], dk[r], None, outs[r], ws, 256, None)
    got = outs.cpu().numpy()
    ctl = [dynk.DynK(4) for _ in range(B)]
    ref = np.array([[c.update(int(nh[r, b]), int(kh[r, b])) for b, c in enumerate(ctl)]
                    for r in range(R)], np.int32)
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]
    assert sb.sv_read_device_flags(ws) == 0

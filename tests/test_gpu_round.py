"""A speculative round chained on the GPU, four rounds in a row: the draft
length comes from the dynamic-k controller, the draft tokens from the draft
sampler, then verify, the paged-KV commit and the controller update.  Every
stage is checked against its oracle, fed with the GPU's own results of the
previous stage (so a low-margin draw that legitimately differs does not
derail the rest of the chain)."""

import numpy as np
import pytest

from tests.conftest import gpu_available
from tests import verify_harness as vh
from oracle import dynk as odk
from oracle import paged as opg
from oracle import sample as osm
from speculative_decoding_verification_47_gb300 import binding as sb
from speculative_decoding_verification_47_gb300 import workloads as wl

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_verification_47_gb300 import build
    build.build()
    sb.lib()


def test_four_chained_rounds():
    import torch
    B, K, V, P, maxp = 32, 8, 4099, 16, 64
    rng = np.random.default_rng(2024)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    T = rng.choice([0.7, 1.0], size=B).astype(np.float32)
    mode = (rng.uniform(size=B) < 0.25).astype(np.uint8)
    # KV cache: pages of P tokens, a free stack of page ids
    lens = rng.integers(100, 400, size=B).astype(np.int32)
    free = list(range(B * maxp))[::-1]
    table = np.full((B, maxp), -1, np.int32)
    for b in range(B):
        for j in range(-(-int(lens[b]) // P)):
            table[b, j] = free.pop()
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    state = torch.zeros(sb.sv_dynk_state_size(B), dtype=torch.uint8, device="cuda")
    sb.sv_dynk_init(state, B, 4, None)
    ctl = [odk.DynK(4) for _ in range(B)]
    k_used = np.array([c.k for c in ctl], np.int32)
    for r in range(4):
        # drafts write their KV: pages for L + k_b tokens
        for b in range(B):
            for j in range(-(-int(lens[b] + k_used[b]) // P)):
                if table[b, j] < 0:
                    table[b, j] = free.pop()
        w = wl.synth_verify("round", B, K, V, wl.BF16, k_used, T, 1.0, mode,
                            seeds=(3000 + r, 3100 + r, 3200 + r))
        # draft sampler
        su = rng.uniform(size=(B, K)).astype(np.float32)
        tok = torch.empty((B, K), dtype=torch.int32, device="cuda")
        dv = d(w.draft.view(np.int16))
        sb.sv_draft_sample(dv, 0, 0, sb.SV_BF16, B, K, V, d(k_used), d(T), 1.0, d(su), d(mode), tok,
                           ws, ws.numel())
        assert sb.sv_read_device_flags(ws) == 0
        got_tok = tok.cpu().numpy()
        ref_tok, margins, _ = osm.sample_tokens(w.draft, wl.BF16, B, K, V, k_used, T, 1.0, su, mode)
        assert np.all((got_tok == ref_tok) | (margins < 1e-6))
        # verify the GPU's draft tokens
        w.draft_tokens = np.where(got_tok >= 0, got_tok, 0).astype(np.int32)
        g = vh.run_gpu(w)
        vh.compare(w, g, vh.run_oracle(w))
        n = g.n.astype(np.int32)
        # paged KV commit
        dl, dn, dk, dt = d(lens), d(n), d(k_used), d(table)
        dfree = torch.full((B * maxp,), -1, dtype=torch.int32, device="cuda")
        top = torch.tensor([0], dtype=torch.int32, device="cuda")
        sb.sv_kv_commit_paged(dl, dn, dk, dt, maxp, P, dfree, top, B * maxp, B, ws, ws.numel(), None)
        rl, rt, rr, rtop, rflags = opg.kv_commit_paged(lens, n, k_used, table, P, 0, B * maxp)
        assert rflags == 0 and sb.sv_read_device_flags(ws) == 0
        assert np.array_equal(dl.cpu().numpy(), rl) and np.array_equal(dt.cpu().numpy(), rt)
        t = int(top.item())
        assert t == rtop and sorted(dfree.cpu().numpy()[:t].tolist()) == sorted(rr)
        lens, table = dl.cpu().numpy(), dt.cpu().numpy()
        free.extend(dfree.cpu().numpy()[:t].tolist())
        # dynamic k for the next round
        kn = torch.empty(B, dtype=torch.int32, device="cuda")
        sb.sv_dynk_update(state, B, dn, dk, None, kn, ws, ws.numel(), None)
        ref_k = np.array([c.update(int(n[b]), int(k_used[b])) for b, c in enumerate(ctl)], np.int32)
        assert np.array_equal(kn.cpu().numpy(), ref_k)
        k_used = ref_k

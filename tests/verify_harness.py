"""Shared helpers for the verify parity tests: run the CUDA library through its
C ABI and the float64 oracle on the same seeded inputs, and compare.

Comparison rule (per sequence):
  * out_tokens and n_accepted must be bit-exact, except where the oracle's own
    decision on the path up to the point of divergence had a margin below
    1e-6 (|u - p/q| for an accept test, distance of u*sum(w) from the
    nearest CDF boundary relative to sum(w) for a draw, distance of the
    kept-mass boundary from top_p for a top-p cut).  Such disagreements are
    counted; across a test session they must stay under 1e-4 of all decisions.
  * probabilities (S, p'(x), q'(x), ratio, residual mass) within 1e-5
    relative where the oracle's value is >= 1e-30; row maxima and greedy
    argmaxes exactly.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from oracle import verify as ov
from speculative_decoding_verification_47_gb300 import binding as sb
from speculative_decoding_verification_47_gb300 import workloads as wl

MARGIN = 1e-6
PROB_RTOL = 1e-5

# session-wide disagreement budget
BUDGET = {"decisions": 0, "disagreements": 0}
BUDGET_LOG = []  # (where, sequence, smallest margin on the path) of each disagreement


@dataclass
class GpuResult:
    out: np.ndarray
    n: np.ndarray
    diag: np.ndarray
    flags: int


def to_device(w: wl.VerifyInputs, device="cuda"):
    import torch
    t = {}
    if w.dtype == wl.BF16:
        t["target"] = torch.from_numpy(w.target.view(np.int16)).to(device)
        t["draft"] = torch.from_numpy(w.draft.view(np.int16)).to(device)
    else:
        t["target"] = torch.from_numpy(w.target).to(device)
        t["draft"] = torch.from_numpy(w.draft).to(device)
    t["tokens"] = torch.from_numpy(w.draft_tokens).to(device)
    t["kpr"] = torch.from_numpy(w.k_per_row).to(device)
    t["temp"] = torch.from_numpy(w.temperature).to(device)
    t["unif"] = torch.from_numpy(w.uniforms).to(device)
    t["mode"] = torch.from_numpy(w.mode).to(device)
    return t


def run_gpu(w: wl.VerifyInputs, dev=None, diag=True, strides=(0, 0, 0, 0), draft=True,
            workspace=None, pass_kpr=True, pass_mode=True, pass_temp=True,
            target_topp=False) -> GpuResult:
    """target_topp: call sv_spec_verify_target_topp (top-p on the target rows only)."""
    import torch
    dev = dev or to_device(w)
    B, K, V = w.B, w.K, w.V
    out = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    dg = (torch.full((B, K + 1, sb.SV_DIAG_FIELDS), float("nan"), device="cuda")
          if diag else None)
    dt = sb.SV_BF16 if w.dtype == wl.BF16 else sb.SV_F32
    wsb = sb.sv_workspace_size(B, K, V, dt)
    ws = workspace if workspace is not None else torch.empty(wsb, dtype=torch.uint8, device="cuda")
    fn = sb.sv_spec_verify_target_topp if target_topp else sb.sv_spec_verify
    fn(dev["target"], strides[0], strides[1], dev["draft"] if draft else None,
       strides[2], strides[3], dt, B, K, V, dev["tokens"],
       dev["kpr"] if pass_kpr else None, dev["temp"] if pass_temp else None,
       w.top_p, dev["unif"], dev["mode"] if pass_mode else None, out, n, dg, ws,
       ws.numel())
    flags = sb.sv_read_device_flags(ws)
    return GpuResult(out=out.cpu().numpy(), n=n.cpu().numpy(),
                     diag=dg.cpu().numpy() if diag else None, flags=flags)


def run_oracle(w: wl.VerifyInputs, rows=None, topp_draft=True) -> ov.BatchResult:
    return ov.spec_verify(w.target, w.draft, w.dtype, w.B, w.K, w.V, w.draft_tokens,
                          w.k_per_row, w.temperature, w.top_p, w.uniforms, w.mode, rows=rows,
                          topp_draft=topp_draft)


def _rel(a, b):
    return abs(a - b) / max(abs(b), 1e-300)


def compare(w: wl.VerifyInputs, g: GpuResult, o: ov.BatchResult, check_flags=True,
            check_probs=True):
    """Assert parity; return (decisions, disagreements) and add them to the
    session budget."""
    decisions = 0
    disagreements = 0
    problems = []
    for b, r in o.seqs:
        decisions += len(r.decisions)
        same = (g.n[b] == r.n) and np.array_equal(g.out[b], np.asarray(r.out, np.int32))
        if not same:
            div = min(int(g.n[b]), r.n)
            low = [d for d in r.decisions
                   if d.position <= div and d.margin < MARGIN]
            if low:
                disagreements += 1
                BUDGET_LOG.append((w.name, int(b), min(d.margin for d in low)))
            else:
                problems.append(f"seq {b}: gpu n={g.n[b]} out={g.out[b].tolist()} vs oracle "
                                f"n={r.n} out={r.out} (min margin "
                                f"{min((d.margin for d in r.decisions), default=math.inf):.3g})")
            continue
        if check_probs and g.diag is not None:
            problems.extend(_compare_diag(w, b, g.diag[b], r))
    assert not problems, "\n".join(problems[:20])
    if check_flags:
        assert g.flags == o.flags, (g.flags, o.flags)
    BUDGET["decisions"] += decisions
    BUDGET["disagreements"] += disagreements
    return decisions, disagreements


def _compare_diag(w, b, dg, r: ov.SeqResult):
    out = []

    def chk(name, got, ref, tol=PROB_RTOL, floor=1e-30):
        if abs(ref) < floor:
            return
        if not (_rel(float(got), float(ref)) <= tol):
            out.append(f"seq {b} {name}: gpu {got!r} oracle {ref!r} rel {_rel(float(got), float(ref)):.3g}")

    for i, a in r.argmax.items():
        if int(dg[i, sb.SV_DIAG_ARGMAX]) != a:
            out.append(f"seq {b} pos {i} argmax gpu {dg[i, sb.SV_DIAG_ARGMAX]} oracle {a}")
    for i, m in r.m_t.items():
        if not np.isnan(dg[i, sb.SV_DIAG_M_T]) and dg[i, sb.SV_DIAG_M_T] != np.float32(m):
            out.append(f"seq {b} pos {i} m_t gpu {dg[i, sb.SV_DIAG_M_T]} oracle {m}")
    for i, S in r.S_t.items():
        if not np.isnan(dg[i, sb.SV_DIAG_S_T]):
            chk(f"pos {i} S_t", dg[i, sb.SV_DIAG_S_T], S)
            chk(f"pos {i} M_t", dg[i, sb.SV_DIAG_MASS_T], r.M_t[i])
    for i, S in r.S_d.items():
        if not np.isnan(dg[i, sb.SV_DIAG_S_D]):
            chk(f"pos {i} S_d", dg[i, sb.SV_DIAG_S_D], S)
            chk(f"pos {i} M_d", dg[i, sb.SV_DIAG_MASS_D], r.M_d[i])
    for i, px in r.px.items():
        if not np.isnan(dg[i, sb.SV_DIAG_P_X]):
            chk(f"pos {i} p(x)", dg[i, sb.SV_DIAG_P_X], px)
            chk(f"pos {i} q(x)", dg[i, sb.SV_DIAG_Q_X], r.qx[i])
            chk(f"pos {i} ratio", dg[i, sb.SV_DIAG_RATIO], r.ratio[i])
    if not math.isnan(r.S_w) and not r.fallback:
        got = dg[r.n, sb.SV_DIAG_S_W]
        if not np.isnan(got):
            chk(f"pos {r.n} S_w", got, r.S_w)
    return out

"""Shared helpers for the verify parity tests: run the CUDA library through its
C ABI and the float64 oracle on the same seeded inputs, and compare.

Comparison rule (per sequence):
  * out_tokens and n_accepted must be bit-exact.  A difference is excused
    only by the oracle's own decision at the FIRST output position t where
    the two outputs differ, when that decision's margin is below 1e-6: the
    accept test at t when the accepted lengths differ (t = the smaller one),
    else the resample or bonus draw at t (distance of u*sum(w) from the
    nearest CDF boundary, relative to sum(w)); the top-p cuts of the rows at
    t (distance of the kept-mass boundary from top_p) count as well, since
    they decide both.  Earlier decisions agreed, so their margins excuse
    nothing.  Excused disagreements are counted: across a test session they
    must stay under 1e-4 of all decisions, and no single call may hold more
    than its 1e-4 share plus one.
  * probabilities (S, p'(x), q'(x), ratio, kept mass, residual mass) within
    1e-5 relative where the oracle's value is >= 1e-30; row maxima and greedy
    argmaxes exactly.  Every row the oracle evaluated (positions 0..n of a
    sequence) must have its diagnostics written: the kernel never drops an
    item at or before the cut, so a NaN there (the buffer's pre-fill) fails.
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

# session-wide disagreement budgets: verify decisions (accept tests, draws,
# top-p cuts) and draft-sampler draws; per call name as well
BUDGET = {"decisions": 0, "disagreements": 0, "low_margin": 0, "per_call": {}}
BUDGET_LOG = []  # (where, sequence, position, kinds, margin) of each disagreement
SAMPLE_BUDGET = {"draws": 0, "disagreements": 0, "low_margin": 0, "log": []}
RATE = 1e-4  # allowed share of excused (low-margin) disagreements of verify decisions
SAMPLE_RATE = 5e-4  # ... of draft-sampler draws (every one of them a draw: reading R22)


def record_call(name, decisions, disagreements, low):
    """Add one call's counts to the session budget and check the call's own
    share (at most RATE of its decisions, plus one)."""
    BUDGET["decisions"] += decisions
    BUDGET["disagreements"] += disagreements
    BUDGET["low_margin"] += low
    pc = BUDGET["per_call"].setdefault(name, [0, 0])
    pc[0] += decisions
    pc[1] += disagreements
    assert disagreements <= RATE * decisions + 1, (name, disagreements, decisions)


def budget_lines():
    """One line per budget that saw any decision (for the session summary)."""
    out = []
    d, x, lo = BUDGET["decisions"], BUDGET["disagreements"], BUDGET["low_margin"]
    if d:
        out.append(f"verify decisions={d} disagreements={x} low-margin decisions={lo} "
                   f"rate={x / d:.2e} (limit {RATE:g})")
    n, x, lo = SAMPLE_BUDGET["draws"], SAMPLE_BUDGET["disagreements"], SAMPLE_BUDGET["low_margin"]
    if n:
        out.append(f"sampler draws={n} disagreements={x} low-margin draws={lo} "
                   f"rate={x / n:.2e} (limit {SAMPLE_RATE:g})")
    return out


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


def first_difference(g_out, g_n, r: ov.SeqResult):
    """First output position where the GPU's and the oracle's outputs differ,
    and the oracle decisions that decided it: the accept test at that
    position if the accepted lengths differ, else the draw there; plus the
    top-p cuts of the position's rows.  Returns (t, decisions)."""
    o = np.asarray(r.out, np.int32)
    diff = np.nonzero(np.asarray(g_out, np.int32) != o)[0]
    if r.flags or np.all(np.asarray(g_out) == -1):
        return (int(diff[0]) if diff.size else 0), []  # an error on either side: never excused
    t = int(diff[0]) if diff.size else min(int(g_n), r.n)
    if int(g_n) != r.n:
        t = min(int(g_n), r.n)
        kinds = ("accept", "topp")
    else:
        kinds = ("resample", "bonus", "topp")
    return t, [d for d in r.decisions if d.position == t and d.kind in kinds]


def compare(w: wl.VerifyInputs, g: GpuResult, o: ov.BatchResult, check_flags=True,
            check_probs=True):
    """Assert parity; return (decisions, disagreements) and add them to the
    session budget."""
    decisions = 0
    disagreements = 0
    low_total = 0
    problems = []
    for b, r in o.seqs:
        decisions += len(r.decisions)
        low_total += sum(1 for d in r.decisions if d.margin < MARGIN)
        same = (g.n[b] == r.n) and np.array_equal(g.out[b], np.asarray(r.out, np.int32))
        if not same:
            t, deciding = first_difference(g.out[b], g.n[b], r)
            low = [d for d in deciding if d.margin < MARGIN]
            if low:
                disagreements += 1
                BUDGET_LOG.append((w.name, int(b), t, [d.kind for d in low],
                                   min(d.margin for d in low)))
            else:
                problems.append(f"seq {b}: gpu n={g.n[b]} out={g.out[b].tolist()} vs oracle "
                                f"n={r.n} out={r.out}; first difference at {t}, deciding "
                                f"margins {[(d.kind, d.margin) for d in deciding]}")
            continue
        if check_probs and g.diag is not None:
            problems.extend(_compare_diag(w, b, g.diag[b], r))
    assert not problems, "\n".join(problems[:20])
    if check_flags:
        assert g.flags == o.flags, (g.flags, o.flags)
    record_call(w.name, decisions, disagreements, low_total)
    return decisions, disagreements


def _compare_diag(w, b, dg, r: ov.SeqResult):
    """Diagnostics of every row the oracle evaluated (positions 0..n of the
    sequence, none of which the kernel may drop) must be written and match."""
    out = []

    def chk(name, got, ref, tol=PROB_RTOL, floor=1e-30):
        if not np.isfinite(got):
            out.append(f"seq {b} {name}: not written (gpu {got!r}, oracle {ref!r})")
            return
        if abs(ref) < floor:
            return
        if not (_rel(float(got), float(ref)) <= tol):
            out.append(f"seq {b} {name}: gpu {got!r} oracle {ref!r} rel {_rel(float(got), float(ref)):.3g}")

    for i, a in r.argmax.items():
        if not np.isfinite(dg[i, sb.SV_DIAG_ARGMAX]) or int(dg[i, sb.SV_DIAG_ARGMAX]) != a:
            out.append(f"seq {b} pos {i} argmax gpu {dg[i, sb.SV_DIAG_ARGMAX]} oracle {a}")
    for i, m in r.m_t.items():
        if dg[i, sb.SV_DIAG_M_T] != np.float32(m):
            out.append(f"seq {b} pos {i} m_t gpu {dg[i, sb.SV_DIAG_M_T]} oracle {m}")
    for i, S in r.S_t.items():
        chk(f"pos {i} S_t", dg[i, sb.SV_DIAG_S_T], S)
        chk(f"pos {i} M_t", dg[i, sb.SV_DIAG_MASS_T], r.M_t[i])
    for i, m in r.m_d.items():
        if dg[i, sb.SV_DIAG_M_D] != np.float32(m):
            out.append(f"seq {b} pos {i} m_d gpu {dg[i, sb.SV_DIAG_M_D]} oracle {m}")
    for i, S in r.S_d.items():
        chk(f"pos {i} S_d", dg[i, sb.SV_DIAG_S_D], S)
        chk(f"pos {i} M_d", dg[i, sb.SV_DIAG_MASS_D], r.M_d[i])
    for i, px in r.px.items():
        chk(f"pos {i} p(x)", dg[i, sb.SV_DIAG_P_X], px)
        chk(f"pos {i} q(x)", dg[i, sb.SV_DIAG_Q_X], r.qx[i])
        chk(f"pos {i} ratio", dg[i, sb.SV_DIAG_RATIO], r.ratio[i])
    if not math.isnan(r.S_w) and not r.fallback:
        chk(f"pos {r.n} S_w", dg[r.n, sb.SV_DIAG_S_W], r.S_w)
    return out

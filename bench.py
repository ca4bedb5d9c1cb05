#!/usr/bin/env python3
"""Benchmark of the batched speculative-decoding verify step on GB300.

One step = sv_spec_verify + sv_kv_commit over one batch of the headline
workload (B=256 sequences, K=8 with ragged k_b in 2..8, V=128256 bf16 logits,
per-row temperature in {0.1, 0.7, 1.0} and draft noise in {0.3, 1, 2};
sampled mode).  Inputs are resident in HBM when timing starts and are
rotated over three identical copies (3.3 GB > the 129 MB L2) so no step
reuses data cached by the previous one.  ``--workload c1|c3`` times the
other batch workloads the same way (c3: half greedy, top_p = 0.9);
``--workload c4`` times the layer-skip step: draft and target logits from
hidden states through sv_lmhead_rmsnorm (tcgen05 GEMM), then verify + commit.
On one GPU the headline run (c2) then also times the
LM head (c4), the top-p batch (c3) and the draft sampler (s2) in the same
process and reports them under "secondary" (``--no-secondary`` skips them).

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle on bounded samples of the same workload instead.  Under torchrun each
rank runs an independent replica (weak scaling, no collective on the data
path); the timed region is bracketed by barriers and the max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified positions/s and spec_verify HBM GB/s (% of GB300 peak) at 1 GPU"
WORKLOADS = {
    "c2": ("headline verify batch: B=256, K=8, ragged k_b~U{2..8}, V=128256 bf16 logits, "
           "T_b in {0.1,0.7,1.0}, draft noise in {0.3,1,2}, sampled; + kv_commit"),
    "c1": ("verify batch: B=64, k=5, V=32000 bf16 logits, T=0.8, draft noise 1.0, sampled; "
           "+ kv_commit"),
    "c3": ("mixed verify batch: B=128, k=6, V=151936 bf16 logits, T=0.7, top_p=0.9 on both "
           "sides, rows 0..63 greedy and 64..127 sampled, draft noise 0.5; + kv_commit"),
    "c4": ("layer-skip step: hidden [512,4096] bf16 -> final RMSNorm (eps 1e-5) -> LM head "
           "W[4096,32000] bf16 for the draft and the target logits, then verify B=64, k=7, "
           "T=1, sampled; + kv_commit"),
    "s2": ("draft-side sampler on the headline batch's draft rows: B=256, K=8, ragged "
           "k_b~U{2..8}, V=128256 bf16 logits, T_b in {0.1,0.7,1.0}, one uniform per token"),
    "c3t": ("the c3 batch through the target-only top-p call: top_p=0.9 truncates the target "
            "rows only, the draft rows enter untruncated; + kv_commit"),
    "kvp": ("paged KV commit after a round: B=1024 sequences, block tables of 64 pages of 16 "
            "tokens, lengths ~U[100,512), k_b~U{2..8}, n_b~U{0..k_b}"),
    "dynk": ("dynamic-k controller update: B=256 sequences, 64-round windows, k_used~U{2..8}, "
             "n~U{0..k_used} per round"),
}
# workloads that run the c3 rows through another entry point
ROW_WORKLOAD = {"c3t": "c3"}
COPIES = 3

# DRAM bytes (read + written) per launch of each workload's dominant kernel,
# from the ncu captures summarised in profiles/; reported only while the
# kernel source still has the hash it had when the counters were taken.
MEASURED_TRAFFIC = {
    "c2": ("sv_verify.cu", "99909b10855a5162", 498.448640e6 + 5.387008e6),
    "c1": ("sv_verify.cu", "99909b10855a5162", 39.446784e6 + 0.001280e6),
    "c3": ("sv_verify.cu", "99909b10855a5162", 246.334720e6 + 13.532160e6),
    "c3t": ("sv_verify.cu", "99909b10855a5162", 248.483840e6 + 13.175296e6),
    "c4": ("sv_lmhead.cu", "55d834ba2fbdc5ca", 271.429632e6 + 20.406272e6),
    "s2": ("sv_verify.cu", "99909b10855a5162", 329.264640e6 + 3.387392e6),
}


def traffic_for(workload: str, override):
    if override is not None:
        return override
    entry = MEASURED_TRAFFIC.get(workload)
    if entry is None:
        return None
    import hashlib
    src, digest, value = entry
    path = os.path.join(ROOT, "speculative_decoding_verification_47_gb300", "csrc", src)
    try:
        with open(path, "rb") as f:
            ok = hashlib.sha256(f.read()).hexdigest()[:16] == digest
    except OSError:
        ok = False
    return value if ok else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# CPU oracle leg (bounded sample, spawn pool, sequences regenerated per worker)
# --------------------------------------------------------------------------
def _oracle_worker(args):
    name, B, seqs = args
    topp_draft = name != "c3t"
    name = ROW_WORKLOAD.get(name, name)
    sys.path.insert(0, ROOT)
    import numpy as np
    from oracle import verify as ov
    from speculative_decoding_verification_47_gb300 import workloads as wl
    spec = wl.row_spec(name, B)
    rows = [(b,) + tuple(spec.sequence(b)) for b in seqs]
    t0 = time.perf_counter()
    pos = 0
    for b, t, d, x, u in rows:
        kb = int(spec.k_per_row[b])
        ov.verify_sequence(ov._LazyRows(t, spec.dtype), ov._LazyRows(d, spec.dtype), x, kb,
                           spec.K, spec.V, float(spec.temperature[b]), spec.top_p,
                           u.astype(np.float64), int(spec.mode[b]), topp_draft)
        pos += kb
    return pos, time.perf_counter() - t0


def cpu_oracle(name: str, B: int, sample_seqs: int, workers: int):
    """The oracle on the first ``sample_seqs`` sequences (spread over the
    batch when it mixes row modes: every (B // sample)-th sequence)."""
    import multiprocessing as mp
    sample_seqs = max(1, min(sample_seqs, B))
    stride = max(1, B // sample_seqs)
    seqs = list(range(0, B, stride))[:sample_seqs]
    chunks = [seqs[i::workers] for i in range(workers)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        res = pool.map(_oracle_worker, [(name, B, c) for c in chunks if c])
    pos = sum(r[0] for r in res)
    wall = max(r[1] for r in res)
    return pos, wall, len([c for c in chunks if c])


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------
def reduce_timing(ms: float, positions: int, pg=None, device=None):
    """Whole-job timing over the ranks of a replica run: the slowest rank's
    elapsed time and the positions all ranks verified (each rank runs its own
    batch; there is no collective on the data path)."""
    if pg is None:
        return ms, positions
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    n = torch.tensor([positions], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    pg.all_reduce(n, op=pg.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_gpu(args):
    import numpy as np
    import torch

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    from speculative_decoding_verification_47_gb300 import binding as sb
    from speculative_decoding_verification_47_gb300 import build as bld
    from speculative_decoding_verification_47_gb300 import workloads as wl
    if rank == 0 or not os.path.exists(bld.LIB):
        bld.build()
    if pg is not None:
        pg.barrier()

    # CPU baseline first (spawn pool, before any GPU work of the main loop)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        workers = min(16, len(os.sched_getaffinity(0)))
        Bw = args.B or wl.row_spec(ROW_WORKLOAD.get(args.workload, args.workload)).B
        pos, wall, used = cpu_oracle(args.workload, Bw, args.cpu_sample, workers)
        cpu = {"value": pos / wall, "unit": "positions/s", "cores": used, "kind": "oracle",
               "sample": f"{min(args.cpu_sample, Bw)} of the {Bw} sequences of the same workload "
                         f"(evenly spaced), float64 oracle, {used} spawn workers, "
                         f"wall {wall:.2f} s"}

    w = wl.config_by_name(ROW_WORKLOAD.get(args.workload, args.workload), args.B)
    B, K, V = w.B, w.K, w.V
    es = 2 if w.dtype == wl.BF16 else 4
    # c3t: top-p on the target rows only (the draft untruncated)
    verify = sb.sv_spec_verify_target_topp if args.workload == "c3t" else sb.sv_spec_verify
    svdt = sb.SV_BF16 if w.dtype == wl.BF16 else sb.SV_F32
    top_p = w.top_p
    dev = torch.device("cuda", local)
    tg = torch.from_numpy(w.target.view(np.int16) if es == 2 else w.target)
    dr = torch.from_numpy(w.draft.view(np.int16) if es == 2 else w.draft)
    tgts = [tg.to(dev) for _ in range(COPIES)]
    drfs = [dr.to(dev) for _ in range(COPIES)]
    tok = torch.from_numpy(w.draft_tokens).to(dev)
    kpr = torch.from_numpy(w.k_per_row).to(dev)
    tmp = torch.from_numpy(w.temperature).to(dev)
    uni = torch.from_numpy(w.uniforms).to(dev)
    mode = torch.from_numpy(w.mode).to(dev)
    seq0 = torch.from_numpy(w.seq_lens).to(dev)
    seq = seq0.clone()
    cap = torch.full((B,), 2**30, dtype=torch.int32, device=dev)
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    nacc = torch.empty((B,), dtype=torch.int32, device=dev)
    wsb = sb.sv_workspace_size(B, K, V, svdt)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(c):
        verify(tgts[c], 0, 0, drfs[c], 0, 0, svdt, B, K, V, tok, kpr, tmp, top_p,
                          uni, mode, out, nacc, None, ws, wsb, stream)
        sb.sv_kv_commit(seq, nacc, cap, kpr, B, K, ws, wsb, stream)

    for it in range(args.warmup):
        step(it % COPIES)
    torch.cuda.synchronize()
    flags = sb.sv_read_device_flags(ws)
    n_host = nacc.cpu().numpy()
    kb = w.k_per_row.astype(np.int64)
    positions = int(kb.sum())
    greedy = w.mode == wl.GREEDY
    # rows the rule reads: up to the cut (target + draft on sampled rows,
    # target only on greedy rows), every row when all drafts are accepted
    rows_needed = int(np.where(greedy, np.minimum(n_host, kb) + 1,
                               np.where(n_host < kb, 2 * (n_host + 1), 2 * kb + 1)).sum())
    rows_all = int(np.where(greedy, kb + 1, 2 * kb + 1).sum())
    small_bytes = B * 4 * (K + 1) * 2 + B * 16  # tokens, uniforms, outputs, per-row knobs
    bytes_needed = rows_needed * V * es + small_bytes
    bytes_all = rows_all * V * es + small_bytes

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for it in range(args.steps):
        c = it % COPIES
        ev[it][0].record(stream)
        verify(tgts[c], 0, 0, drfs[c], 0, 0, svdt, B, K, V, tok, kpr, tmp, top_p,
                          uni, mode, out, nacc, None, ws, wsb, stream)
        ev[it][1].record(stream)
        sb.sv_kv_commit(seq, nacc, cap, kpr, B, K, ws, wsb, stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if pg is not None:
        pg.barrier()
    clk = clocks.stop()
    ms, total_positions = reduce_timing(t_start.elapsed_time(t_end), positions, pg, dev)
    verify_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms_step = ms / args.steps
    value = total_positions / (ms_step * 1e-3)

    # end to end: pinned host inputs -> device, verify + commit, outputs -> host
    e2e = None
    if not args.no_e2e:
        h_t = tg.pin_memory()
        h_d = dr.pin_memory()
        h_small = [torch.from_numpy(a).pin_memory() for a in
                   (w.draft_tokens, w.k_per_row, w.temperature, w.uniforms, w.mode, w.seq_lens)]
        d_small = [tok, kpr, tmp, uni, mode, seq]
        o_out = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
        o_n = torch.empty((B,), dtype=torch.int32).pin_memory()
        o_seq = torch.empty((B,), dtype=torch.int32).pin_memory()
        steps_e2e = max(3, min(args.steps, 20))

        def e2e_step():
            tgts[0].copy_(h_t, non_blocking=True)
            drfs[0].copy_(h_d, non_blocking=True)
            for d_, h_ in zip(d_small, h_small):
                d_.copy_(h_, non_blocking=True)
            verify(tgts[0], 0, 0, drfs[0], 0, 0, svdt, B, K, V, tok, kpr, tmp,
                              top_p, uni, mode, out, nacc, None, ws, wsb, stream)
            sb.sv_kv_commit(seq, nacc, cap, kpr, B, K, ws, wsb, stream)
            o_out.copy_(out, non_blocking=True)
            o_n.copy_(nacc, non_blocking=True)
            o_seq.copy_(seq, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ems = a.elapsed_time(b)
        if pg is not None:
            t = torch.tensor([ems], device=dev, dtype=torch.float64)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            ems = float(t.item())
        h2d = (h_t.numel() + h_d.numel()) * es + sum(x.numel() * x.element_size() for x in h_small)
        d2h = (o_out.numel() + o_n.numel() + o_seq.numel()) * 4
        e2e = {"value": positions * world / (ems / steps_e2e * 1e-3), "unit": "positions/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": steps_e2e}

    peak, peak_src = peaks()
    # algorithmic bytes: every target and draft row of the call read once
    # (s*V*sum_b(2k_b+1) sampled, s*V*(k_b+1) greedy); the kernel skips the
    # rows after each sequence's first rejection, so it moves fewer
    achieved = bytes_all / (verify_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "positions/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "input_dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "name": args.workload,
                   "B": B, "K": K, "V": V, "top_p": top_p,
                   "positions_per_step": positions, "target_rows": int((kb + 1).sum()),
                   "l2": f"{COPIES} rotating input copies ({COPIES * (w.target.nbytes + w.draft.nbytes) / 1e9:.1f} GB) > 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "hbm": {"bytes_algorithmic_per_call": bytes_all,
                "bytes_rows_read_per_call": bytes_needed,
                "rows_all": rows_all, "rows_read": rows_needed,
                "gbs_algorithmic": achieved,
                "gbs_rows_read": bytes_needed / (verify_ms * 1e-3) / 1e9,
                "frac_of_peak": achieved / peak, "peak_gbs": peak, "peak_source": peak_src},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic_for(args.workload, args.traffic),
                     "kernel": f"verify_kernel<{es},{'true' if top_p < 1 else 'false'}>",
                     "launch_ms": verify_ms, "peak_source": peak_src},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "device_flags": flags,
    }
    if pg is not None:
        pg.destroy_process_group()
    return line if rank == 0 else None


# --------------------------------------------------------------------------
# c4: layer-skip draft/target logits on the tensor cores, then verify
# --------------------------------------------------------------------------
def _c4_oracle_step(x, tokens, knobs, B, K):
    """One step of the float64 oracle: both LM heads, then the verify rule."""
    import numpy as np
    from oracle import lmhead as ol
    from oracle import verify as ov
    from speculative_decoding_verification_47_gb300 import workloads as wl
    V = x.V
    dl = wl.f64_to_bf16_bits(ol.lmhead_rmsnorm(x.hidden, x.norm_w, x.eps, x.W)).reshape(B, K + 1, V)
    tl = wl.f64_to_bf16_bits(ol.lmhead_rmsnorm(x.hidden_t, x.norm_w, x.eps, x.W)).reshape(B, K + 1, V)
    ov.spec_verify(tl, np.ascontiguousarray(dl[:, :K]), wl.BF16, B, K, V, tokens,
                   knobs["k_per_row"], knobs["temperature"], 1.0, knobs["uniforms"], knobs["mode"])
    return int(knobs["k_per_row"].sum())


def run_gpu_c4(args):
    import numpy as np
    import torch

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    from speculative_decoding_verification_47_gb300 import binding as sb
    from speculative_decoding_verification_47_gb300 import build as bld
    from speculative_decoding_verification_47_gb300 import workloads as wl
    if rank == 0 or not os.path.exists(bld.LIB):
        bld.build()
    if pg is not None:
        pg.barrier()
    B, K = 64, 7
    x = wl.lmhead_inputs()
    M, H, V = x.M, x.H, x.V
    knobs = wl.c4_verify_knobs(B, K)
    dev = torch.device("cuda", local)
    d_h = torch.from_numpy(x.hidden.view(np.int16)).to(dev)
    d_ht = torch.from_numpy(x.hidden_t.view(np.int16)).to(dev)
    d_w = torch.from_numpy(x.norm_w.view(np.int16)).to(dev)
    d_W = torch.from_numpy(x.W.view(np.int16)).to(dev)  # 262 MB model weight (> L2)
    dl = torch.empty((M, V), dtype=torch.int16, device=dev)
    tl = torch.empty((M, V), dtype=torch.int16, device=dev)
    wsl = sb.sv_lmhead_workspace_size(M, H)
    ws1 = torch.zeros(wsl, dtype=torch.uint8, device=dev)
    ws2 = torch.zeros(wsl, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    # draft tokens from the first draft logits (the draft sampler precedes the path)
    sb.sv_lmhead_rmsnorm(d_h, d_w, x.eps, d_W, dl, sb.SV_BF16, M, H, V, ws1, wsl, stream)
    torch.cuda.synchronize()
    d_bits = dl.cpu().numpy().view(np.uint16).reshape(B, K + 1, V)
    tokens = wl.draw_draft_tokens(d_bits[:, :K], wl.BF16, knobs["k_per_row"], knobs["temperature"],
                                  knobs["mode"], seed=4004)
    tok = torch.from_numpy(tokens).to(dev)
    kpr = torch.from_numpy(knobs["k_per_row"]).to(dev)
    tmp = torch.from_numpy(knobs["temperature"]).to(dev)
    uni = torch.from_numpy(knobs["uniforms"]).to(dev)
    mode = torch.from_numpy(knobs["mode"]).to(dev)
    seq = torch.from_numpy(np.random.default_rng(3004).integers(128, 4097, size=B).astype(np.int32)).to(dev)
    cap = torch.full((B,), 2**30, dtype=torch.int32, device=dev)
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    nacc = torch.empty((B,), dtype=torch.int32, device=dev)
    wsb = sb.sv_workspace_size(B, K, V, sb.SV_BF16)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t0 = time.perf_counter()
        pos = _c4_oracle_step(x, tokens, knobs, B, K)
        wall = time.perf_counter() - t0
        cpu = {"value": pos / wall, "unit": "positions/s", "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle",
               "sample": f"one full step (two float64 LM heads 512x4096x32000 with NumPy BLAS, "
                         f"then the verify rule on 64 sequences), wall {wall:.2f} s"}

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(max(args.steps, 1))]

    def step(i=None):
        if i is not None:
            ev[i][0].record(stream)
        sb.sv_lmhead_rmsnorm(d_h, d_w, x.eps, d_W, dl, sb.SV_BF16, M, H, V, ws1, wsl, stream)
        if i is not None:
            ev[i][1].record(stream)
        sb.sv_lmhead_rmsnorm(d_ht, d_w, x.eps, d_W, tl, sb.SV_BF16, M, H, V, ws2, wsl, stream)
        sb.sv_spec_verify(tl, 0, 0, dl, (K + 1) * V, V, sb.SV_BF16, B, K, V, tok, kpr, tmp, 1.0,
                          uni, mode, out, nacc, None, ws, wsb, stream)
        sb.sv_kv_commit(seq, nacc, cap, kpr, B, K, ws, wsb, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flags = (sb.sv_read_device_flags(ws), sb.sv_read_device_flags(ws1))
    positions = int(knobs["k_per_row"].sum())
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for it in range(args.steps):
        step(it)
    t_end.record(stream)
    torch.cuda.synchronize()
    if pg is not None:
        pg.barrier()
    clk = clocks.stop()
    ms, total_positions = reduce_timing(t_start.elapsed_time(t_end), positions, pg, dev)
    lm_ms = statistics.mean(a.elapsed_time(b) for a, b in ev[:args.steps])
    ms_step = ms / args.steps
    value = total_positions / (ms_step * 1e-3)
    flops = 2.0 * M * H * V
    achieved = flops / (lm_ms * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        h_h = torch.from_numpy(x.hidden.view(np.int16)).pin_memory()
        h_ht = torch.from_numpy(x.hidden_t.view(np.int16)).pin_memory()
        h_small = [torch.from_numpy(a).pin_memory() for a in
                   (tokens, knobs["k_per_row"], knobs["temperature"], knobs["uniforms"], knobs["mode"])]
        d_small = [tok, kpr, tmp, uni, mode]
        o_out = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
        o_n = torch.empty((B,), dtype=torch.int32).pin_memory()
        o_seq = torch.empty((B,), dtype=torch.int32).pin_memory()
        steps_e2e = max(3, min(args.steps, 20))

        def e2e_step():
            d_h.copy_(h_h, non_blocking=True)
            d_ht.copy_(h_ht, non_blocking=True)
            for d_, h_ in zip(d_small, h_small):
                d_.copy_(h_, non_blocking=True)
            step()
            o_out.copy_(out, non_blocking=True)
            o_n.copy_(nacc, non_blocking=True)
            o_seq.copy_(seq, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ems = a.elapsed_time(b)
        if pg is not None:
            t = torch.tensor([ems], device=dev, dtype=torch.float64)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            ems = float(t.item())
        h2d = (h_h.numel() + h_ht.numel()) * 2 + sum(t_.numel() * t_.element_size() for t_ in h_small)
        d2h = (o_out.numel() + o_n.numel() + o_seq.numel()) * 4
        e2e = {"value": positions * world / (ems / steps_e2e * 1e-3), "unit": "positions/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps_e2e}

    tpeak, tsrc = tensor_peak()
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "positions/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOADS["c4"], "name": "c4", "B": B, "K": K, "V": V, "M": M, "H": H,
                   "l2": "W (262 MB) > 129 MB L2, streamed from HBM by every LM-head call",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                     "frac": achieved / tpeak, "traffic": traffic_for("c4", args.traffic),
                     "kernel": "sv_lmhead_rmsnorm (rmsnorm_kernel + lmhead_gemm_kernel), draft call",
                     "flops_per_call": flops, "launch_ms": lm_ms, "peak_source": tsrc},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 7 * args.steps,
        "clocks": clk,
        "device_flags": list(flags),
    }
    if pg is not None:
        pg.destroy_process_group()
    return line if rank == 0 else None


def run_gpu_s2(args):
    """The draft-side sampler over the headline batch's draft rows (k_b per
    sequence, per-row temperature): one sv_draft_sample call per step."""
    import numpy as np
    import torch

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    from speculative_decoding_verification_47_gb300 import binding as sb
    from speculative_decoding_verification_47_gb300 import build as bld
    from speculative_decoding_verification_47_gb300 import workloads as wl
    if rank == 0 or not os.path.exists(bld.LIB):
        bld.build()
    if pg is not None:
        pg.barrier()
    w = wl.config_by_name("c2")
    B, K, V = w.B, w.K, w.V
    unif = np.random.default_rng(5150).uniform(size=(B, K)).astype(np.float32)
    dev = torch.device("cuda", local)
    dr = torch.from_numpy(w.draft.view(np.int16))
    drfs = [dr.to(dev) for _ in range(COPIES)]
    kpr = torch.from_numpy(w.k_per_row).to(dev)
    tmp = torch.from_numpy(w.temperature).to(dev)
    uni = torch.from_numpy(unif).to(dev)
    mode = torch.from_numpy(w.mode).to(dev)
    out = torch.empty((B, K), dtype=torch.int32, device=dev)
    wsb = sb.sv_draft_sample_workspace_size()
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    tokens = int(w.k_per_row.sum())
    row_bytes = V * 2

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import sample as osm
        n = max(1, min(B, args.cpu_sample // 8))
        t0 = time.perf_counter()
        osm.sample_tokens(w.draft[:n], w.dtype, n, K, V, w.k_per_row[:n], w.temperature[:n], 1.0,
                          unif[:n], w.mode[:n])
        wall = time.perf_counter() - t0
        cpu = {"value": int(w.k_per_row[:n].sum()) / wall, "unit": "tokens/s", "cores": 1,
               "kind": "oracle",
               "sample": f"the first {n} of the {B} sequences, float64 oracle, one core, wall {wall:.2f} s"}

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(max(args.steps, 1))]

    def step(c, i=None):
        if i is not None:
            ev[i][0].record(stream)
        sb.sv_draft_sample(drfs[c], 0, 0, sb.SV_BF16, B, K, V, kpr, tmp, 1.0, uni, mode, out, ws,
                           wsb, stream)
        if i is not None:
            ev[i][1].record(stream)

    for it in range(args.warmup):
        step(it % COPIES)
    torch.cuda.synchronize()
    flags = sb.sv_read_device_flags(ws)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for it in range(args.steps):
        step(it % COPIES, it)
    t_end.record(stream)
    torch.cuda.synchronize()
    if pg is not None:
        pg.barrier()
    clk = clocks.stop()
    ms, total = reduce_timing(t_start.elapsed_time(t_end), tokens, pg, dev)
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in ev[:args.steps])
    ms_step = ms / args.steps
    value = total / (ms_step * 1e-3)
    alg_bytes = tokens * row_bytes  # every sampled row read once
    achieved = alg_bytes / (call_ms * 1e-3) / 1e9
    peak, psrc = peaks()

    e2e = None
    if not args.no_e2e:
        h_d = dr.pin_memory()
        h_small = [torch.from_numpy(a).pin_memory() for a in (w.k_per_row, w.temperature, unif, w.mode)]
        d_small = [kpr, tmp, uni, mode]
        o_out = torch.empty((B, K), dtype=torch.int32).pin_memory()
        steps_e2e = max(3, min(args.steps, 20))

        def e2e_step():
            drfs[0].copy_(h_d, non_blocking=True)
            for d_, h_ in zip(d_small, h_small):
                d_.copy_(h_, non_blocking=True)
            step(0)
            o_out.copy_(out, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ems = a.elapsed_time(b)
        if pg is not None:
            t = torch.tensor([ems], device=dev, dtype=torch.float64)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            ems = float(t.item())
        h2d = h_d.numel() * 2 + sum(t_.numel() * t_.element_size() for t_ in h_small)
        e2e = {"value": tokens * world / (ems / steps_e2e * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(o_out.numel() * 4),
               "steps": steps_e2e}

    line = {
        "metric": "draft tokens sampled/s and sampler HBM GB/s (% of GB300 peak) at 1 GPU",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "input_dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOADS["s2"], "name": "s2", "B": B, "K": K, "V": V,
                   "tokens_per_step": tokens,
                   "l2": f"{COPIES} rotating input copies ({COPIES * w.draft.nbytes / 1e9:.1f} GB) > 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "hbm": {"bytes_algorithmic_per_call": alg_bytes, "gbs_algorithmic": achieved,
                "frac_of_peak": achieved / peak, "peak_gbs": peak, "peak_source": psrc},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic_for("s2", args.traffic),
                     "kernel": "sample_kernel<2,false>", "launch_ms": call_ms, "peak_source": psrc},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "device_flags": flags,
    }
    if pg is not None:
        pg.destroy_process_group()
    return line if rank == 0 else None


# --------------------------------------------------------------------------
# Round bookkeeping: the paged-KV commit and the dynamic-k update.  Both run
# one thread per sequence and are launch-latency bound; each call is timed
# with CUDA events on its stream.
# --------------------------------------------------------------------------
def _small_call_line(args, name, metric, unit, units, call_ms, ms_step, alg_bytes, kernel, cfg,
                     cpu, e2e, launches, clk, flags, world):
    peak, psrc = peaks()
    achieved = alg_bytes / (call_ms * 1e-3) / 1e9
    return {
        "metric": metric,
        "value": units * world / (ms_step * 1e-3),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int32",
        "data": "synthetic",
        "config": dict({"workload": WORKLOADS[name], "name": name,
                        "parallelism": f"replicas x{world}"}, **cfg),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None, "kernel": kernel,
                     "launch_ms": call_ms, "peak_source": psrc,
                     "note": "one thread per sequence: launch-latency bound, far from the "
                             "HBM roof at any batch a round has"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
        "device_flags": flags,
    }


def _gpu_setup(args):
    import torch
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    from speculative_decoding_verification_47_gb300 import build as bld
    if rank == 0 or not os.path.exists(bld.LIB):
        bld.build()
    if pg is not None:
        pg.barrier()
    return world, rank, local, pg


def _timed_calls(args, stream, call, between=None, pg=None):
    """Warm-up, then args.steps calls, each bracketed by CUDA events on the
    launching stream; ``between`` (state restore) runs outside the events.
    Returns (mean call ms, clocks)."""
    import torch
    for it in range(args.warmup):
        if between:
            between(it)
        call(it)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.25)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    for it in range(args.steps):
        if between:
            between(args.warmup + it)
        ev[it][0].record(stream)
        call(args.warmup + it)
        ev[it][1].record(stream)
    torch.cuda.synchronize()
    if pg is not None:
        pg.barrier()
    clk = clocks.stop()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if pg is not None:
        t = torch.tensor([ms], dtype=torch.float64, device="cuda")
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = float(t.item())
    return ms, clk


def _e2e_time(args, stream, e2e_step, pg=None):
    import torch
    steps = max(3, min(args.steps, 20))
    e2e_step(0)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        e2e_step(i)
    b.record(stream)
    torch.cuda.synchronize()
    ems = a.elapsed_time(b)
    if pg is not None:
        t = torch.tensor([ems], dtype=torch.float64, device="cuda")
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ems = float(t.item())
    return ems / steps, steps


def run_gpu_kvp(args):
    """sv_kv_commit_paged on one round's state; the state is restored by
    device copies between calls, outside the timed events."""
    import numpy as np
    import torch
    world, rank, local, pg = _gpu_setup(args)
    from speculative_decoding_verification_47_gb300 import binding as sb
    from speculative_decoding_verification_47_gb300 import workloads as wl
    r = wl.paged_round()
    B, maxp = r.block_table.shape
    P, cap = r.page_size, r.pool_pages
    dev = torch.device("cuda", local)

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    lens0, table0, n, k = d(r.seq_lens), d(r.block_table), d(r.n_accepted), d(r.k_per_row)
    lens, table = lens0.clone(), table0.clone()
    free = torch.full((cap,), -1, dtype=torch.int32, device=dev)
    top = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import paged as opg
        calls, t0 = 0, time.perf_counter()
        while calls < 3 or time.perf_counter() - t0 < 2.0:
            opg.kv_commit_paged(r.seq_lens, r.n_accepted, r.k_per_row, r.block_table, P, 0, cap)
            calls += 1
        wall = time.perf_counter() - t0
        cpu = {"value": B * calls / wall, "unit": "sequences/s", "cores": 1, "kind": "oracle",
               "sample": f"the whole batch of {B} sequences, {calls} calls, Python oracle, "
                         f"one core, wall {wall:.2f} s"}

    def restore(_):
        lens.copy_(lens0)
        table.copy_(table0)
        top.zero_()

    def call(_):
        sb.sv_kv_commit_paged(lens, n, k, table, maxp, P, free, top, cap, B, ws, 256, stream)

    call_ms, clk = _timed_calls(args, stream, call, restore, pg)
    flags = sb.sv_read_device_flags(ws)
    released = int(top.item())
    # lengths read and written, n and k read; each table row scanned once;
    # every release writes a table entry and a free-stack slot
    alg = B * 16 + B * maxp * 4 + released * 8

    e2e = None
    if not args.no_e2e:
        h_in = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                for a in (r.seq_lens, r.n_accepted, r.k_per_row, r.block_table)]
        d_in = [lens, n, k, table]
        outs = [(torch.empty(t.shape, dtype=torch.int32).pin_memory(), t)
                for t in (lens, table, free, top)]

        def e2e_step(_):
            for d_, h_ in zip(d_in, h_in):
                d_.copy_(h_, non_blocking=True)
            top.zero_()
            call(0)
            for h_, d_ in outs:
                h_.copy_(d_, non_blocking=True)

        ems, steps = _e2e_time(args, stream, e2e_step, pg)
        e2e = {"value": B * world / (ems * 1e-3), "unit": "sequences/s",
               "h2d_bytes_per_step": int(sum(x.numel() * 4 for x in h_in)) + 4,
               "d2h_bytes_per_step": int(sum(h_.numel() * 4 for h_, _ in outs)),
               "steps": steps}

    line = _small_call_line(
        args, "kvp", "paged KV commits/s (sequences) at 1 GPU", "sequences/s", B, call_ms,
        call_ms, alg, "paged_count_kernel + paged_apply_kernel",
        {"B": B, "max_pages": int(maxp), "page_size": P, "released_pages": released,
         "bytes_algorithmic_per_call": alg,
         "l2": "state restored between calls by device copies outside the timed events; "
               "the 0.3 MB state stays in L2"},
        cpu, e2e, 2 * args.steps, clk, flags, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def run_gpu_dynk(args):
    """sv_dynk_update over a history of rounds (one update per call)."""
    import numpy as np
    import torch
    world, rank, local, pg = _gpu_setup(args)
    from speculative_decoding_verification_47_gb300 import binding as sb
    from speculative_decoding_verification_47_gb300 import workloads as wl
    B = 256
    rounds = args.warmup + args.steps + 1
    nh, kh = wl.dynk_history(B, rounds)
    dev = torch.device("cuda", local)
    dn = torch.from_numpy(nh).to(dev)
    dk = torch.from_numpy(kh).to(dev)
    state = torch.zeros(sb.sv_dynk_state_size(B), dtype=torch.uint8, device=dev)
    kn = torch.empty(B, dtype=torch.int32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sb.sv_dynk_init(state, B, 4, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import dynk as odk
        ctl = [odk.DynK(4) for _ in range(B)]
        t0 = time.perf_counter()
        for i in range(rounds):
            for b in range(B):
                ctl[b].update(int(nh[i, b]), int(kh[i, b]))
        wall = time.perf_counter() - t0
        cpu = {"value": B * rounds / wall, "unit": "sequences/s", "cores": 1, "kind": "oracle",
               "sample": f"the same {rounds} rounds of {B} controllers, Python oracle, one core, "
                         f"wall {wall:.2f} s"}

    def call(i):
        sb.sv_dynk_update(state, B, dn[i], dk[i], None, kn, ws, 256, stream)

    call_ms, clk = _timed_calls(args, stream, call, None, pg)
    flags = sb.sv_read_device_flags(ws)
    # per sequence: seven int32 state words read and written, one ring byte
    # pair read and written, n and k_used read, k_next written
    alg = B * 72

    e2e = None
    if not args.no_e2e:
        h_n = torch.from_numpy(nh[-1].copy()).pin_memory()
        h_k = torch.from_numpy(kh[-1].copy()).pin_memory()
        n1, k1 = dn[-1], dk[-1]
        o_k = torch.empty(B, dtype=torch.int32).pin_memory()

        def e2e_step(_):
            n1.copy_(h_n, non_blocking=True)
            k1.copy_(h_k, non_blocking=True)
            sb.sv_dynk_update(state, B, n1, k1, None, kn, ws, 256, stream)
            o_k.copy_(kn, non_blocking=True)

        ems, steps = _e2e_time(args, stream, e2e_step, pg)
        e2e = {"value": B * world / (ems * 1e-3), "unit": "sequences/s",
               "h2d_bytes_per_step": 2 * B * 4, "d2h_bytes_per_step": B * 4, "steps": steps}

    line = _small_call_line(
        args, "dynk", "dynamic-k controller updates/s (sequences) at 1 GPU", "sequences/s", B,
        call_ms, call_ms, alg, "dynk_update_kernel",
        {"B": B, "window": 64, "bytes_algorithmic_per_call": alg,
         "l2": f"controller state {sb.sv_dynk_state_size(B)} bytes, resident in L2"},
        cpu, e2e, args.steps, clk, flags, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def _reference_line(args, name, metric, unit, value, ms_step, cfg, sample):
    return {
        "impl": "reference",
        "metric": metric,
        "value": value,
        "unit": unit,
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int64",
        "data": "synthetic",
        "config": dict({"workload": WORKLOADS[name], "name": name, "parallelism": "host cores"},
                       **cfg),
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_kvp(args):
    """The paged-commit oracle on the whole round, one call per step."""
    from oracle import paged as opg
    from speculative_decoding_verification_47_gb300 import workloads as wl
    r = wl.paged_round()
    B, maxp = r.block_table.shape
    wall = 0.0
    for it in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        opg.kv_commit_paged(r.seq_lens, r.n_accepted, r.k_per_row, r.block_table, r.page_size, 0,
                            r.pool_pages)
        if it >= args.warmup:
            wall += time.perf_counter() - t0
    print(json.dumps(_reference_line(
        args, "kvp", "paged KV commits/s (sequences) at 1 GPU", "sequences/s",
        B * args.steps / wall, wall / args.steps * 1e3,
        {"B": B, "max_pages": int(maxp), "page_size": r.page_size},
        f"each step: the whole batch of {B} sequences, Python oracle, one core")), flush=True)


def run_reference_dynk(args):
    """The controller oracle, one round of B updates per step."""
    from oracle import dynk as odk
    from speculative_decoding_verification_47_gb300 import workloads as wl
    B = 256
    nh, kh = wl.dynk_history(B, args.warmup + args.steps)
    ctl = [odk.DynK(4) for _ in range(B)]
    wall = 0.0
    for it in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        for b in range(B):
            ctl[b].update(int(nh[it, b]), int(kh[it, b]))
        if it >= args.warmup:
            wall += time.perf_counter() - t0
    print(json.dumps(_reference_line(
        args, "dynk", "dynamic-k controller updates/s (sequences) at 1 GPU", "sequences/s",
        B * args.steps / wall, wall / args.steps * 1e3, {"B": B, "window": 64},
        f"each step: one round of {B} controllers, Python oracle, one core")), flush=True)


def secondary(args):
    """After the headline (one GPU only): the LM-head GEMM (c4), the top-p
    verify batch (c3) and the draft sampler (s2), each with its own CUDA-event
    timing of its dominant kernel, roofline and clock record."""
    import copy
    out = {}
    for name, fn in (("c4_lmhead", run_gpu_c4), ("c3", run_gpu), ("s2", run_gpu_s2)):
        a = copy.copy(args)
        a.workload = name.split("_")[0]
        a.steps = max(3, min(args.steps, args.secondary_steps))
        a.no_e2e = True
        a.no_cpu_baseline = True
        a.traffic = None
        a.B = None
        try:
            ln = fn(a)
        except Exception as exc:  # a secondary failure must not hide the headline
            out[name] = {"error": f"{type(exc).__name__}: {exc}"}
            continue
        out[name] = {k: ln.get(k) for k in ("metric", "value", "unit", "ms_per_step", "steps",
                                            "warmup", "roofline", "clocks", "device_flags")}
        out[name]["config"] = {k: ln["config"].get(k) for k in ("name", "B", "K", "V", "M", "H",
                                                                 "top_p") if k in ln["config"]}
    return out


def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except Exception:
        return 1900.0, "fallback"


def run_reference(args):
    world, rank, local = dist_setup(args)
    if rank != 0:
        return
    sys.path.insert(0, ROOT)
    from speculative_decoding_verification_47_gb300 import workloads as wl
    if args.workload == "c4":
        return run_reference_c4(args)
    if args.workload == "s2":
        return run_reference_s2(args)
    if args.workload == "kvp":
        return run_reference_kvp(args)
    if args.workload == "dynk":
        return run_reference_dynk(args)
    spec = wl.row_spec(ROW_WORKLOAD.get(args.workload, args.workload), args.B)
    workers = min(16, len(os.sched_getaffinity(0)))
    for _ in range(args.warmup):
        cpu_oracle(args.workload, spec.B, workers, workers)  # one sequence per worker
    tot_pos, tot_wall = 0, 0.0
    for _ in range(args.steps):
        pos, wall, used = cpu_oracle(args.workload, spec.B, args.ref_sample, workers)
        tot_pos += pos
        tot_wall += wall
    value = tot_pos / tot_wall
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "positions/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": tot_wall / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "name": args.workload, "B": spec.B,
                   "K": spec.K, "V": spec.V, "top_p": spec.top_p, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "positions/s", "cores": used, "kind": "oracle",
                         "sample": f"each step: {args.ref_sample} of the {spec.B} sequences "
                                   f"(evenly spaced), float64 oracle over {used} spawn workers"},
        "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_s2(args):
    """The sampler oracle on a few sequences of the headline batch per step,
    their rows regenerated from the workload's per-sequence seeds."""
    import numpy as np
    from oracle import sample as osm
    from speculative_decoding_verification_47_gb300 import workloads as wl
    spec = wl.row_spec("c2", None)
    unif = np.random.default_rng(5150).uniform(size=(spec.B, spec.K)).astype(np.float32)
    n = max(1, min(spec.B, args.ref_sample // 8))
    tot_tok, tot_wall = 0, 0.0
    for it in range(args.warmup + args.steps):
        seqs = [(it * n + j) % spec.B for j in range(n)]
        rows = [(b,) + tuple(spec.sequence(b)) for b in seqs]
        t0 = time.perf_counter()
        tok = 0
        for b, t, d, x, u in rows:
            kb = int(spec.k_per_row[b])
            osm.sample_tokens(np.asarray(d)[None], spec.dtype, 1, spec.K, spec.V, [kb],
                              [spec.temperature[b]], 1.0, unif[b:b + 1], [spec.mode[b]])
            tok += kb
        wall = time.perf_counter() - t0
        if it >= args.warmup:
            tot_tok += tok
            tot_wall += wall
    value = tot_tok / tot_wall
    line = {
        "impl": "reference",
        "metric": "draft tokens sampled/s and sampler HBM GB/s (% of GB300 peak) at 1 GPU",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": tot_wall / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOADS["s2"], "name": "s2", "B": spec.B, "K": spec.K, "V": spec.V,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: {n} of the {spec.B} sequences, float64 oracle, one core"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_c4(args):
    """The oracle on the layer-skip step; draft tokens from the oracle's own
    draft logits."""
    import numpy as np
    from oracle import lmhead as ol
    from speculative_decoding_verification_47_gb300 import workloads as wl
    B, K = 64, 7
    x = wl.lmhead_inputs()
    knobs = wl.c4_verify_knobs(B, K)
    dl = wl.f64_to_bf16_bits(ol.lmhead_rmsnorm(x.hidden, x.norm_w, x.eps, x.W)).reshape(B, K + 1, x.V)
    tokens = wl.draw_draft_tokens(dl[:, :K], wl.BF16, knobs["k_per_row"], knobs["temperature"],
                                  knobs["mode"], seed=4004)
    for _ in range(min(args.warmup, 1)):
        _c4_oracle_step(x, tokens, knobs, B, K)
    tot_pos, tot_wall = 0, 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        tot_pos += _c4_oracle_step(x, tokens, knobs, B, K)
        tot_wall += time.perf_counter() - t0
    value = tot_pos / tot_wall
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "positions/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_wall / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS["c4"], "name": "c4", "B": B, "K": K, "V": x.V,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "positions/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: both float64 LM heads and the verify rule, in full"},
        "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--workload", default="c2", choices=sorted(WORKLOADS),
                    help="c2 is the headline batch; c1 and c3 are the other batch workloads")
    ap.add_argument("--B", type=int, default=None,
                    help="sequences (the workload's own B by default; smaller only for profiling)")
    ap.add_argument("--cpu-sample", type=int, default=256)
    ap.add_argument("--ref-sample", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="c2 only: skip the LM-head (c4), top-p (c3) and sampler (s2) timings "
                         "that follow the headline in the same process")
    ap.add_argument("--secondary-steps", type=int, default=100)
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per verify launch, if measured for this kernel")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "c4":
        line = run_gpu_c4(args)
        if line is not None:
            print(json.dumps(line), flush=True)
    elif args.workload == "s2":
        line = run_gpu_s2(args)
        if line is not None:
            print(json.dumps(line), flush=True)
    elif args.workload == "kvp":
        run_gpu_kvp(args)
    elif args.workload == "dynk":
        run_gpu_dynk(args)
    else:
        line = run_gpu(args)
        if line is not None:
            world = int(os.environ.get("WORLD_SIZE", "1"))
            if args.workload == "c2" and world == 1 and args.gpus == 1 and not args.no_secondary:
                line["secondary"] = secondary(args)
            print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Throughput of the deterministic attention backward (DASH schedules) on GB300.

Default workload: full-mask attention backward, H=16, D=128, bf16 N(0,1) inputs,
B*S = 16384 tokens per batch, one step = one backward pass (prologue + tile kernel + dQ
convert) for every sequence length of the sweep S in {512, ..., 16384} (B = 16384/S).
Metric: backward TFLOP/s (algorithmic FLOPs 10*B*H*S^2*D, halved for a causal mask) of the
deterministic schedule, with the fraction of the measured dense-bf16 peak and the slowdown
against the non-deterministic atomic-dQ backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--schedule S]
    python bench.py --impl reference ...   # the fp64 CPU oracle on a bounded sample

Prints one JSON line (rank 0).  Under torchrun each rank runs the same workload on its own
GPU (independent replicas, no collective on the data path); the value is the sum of the
ranks' FLOPs over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "deterministic attn-bwd TFLOP/s, % of bf16 tensor peak, slowdown vs atomic-dQ"

WORKLOADS = {
    "full_h16_d128": dict(
        desc="full-mask attention backward, H=16, D=128, bf16 N(0,1), B*S=16384, "
             "S swept over {512,1024,2048,4096,8192,16384}",
        H=16, Hkv=16, D=128, causal=False, tokens=16384,
        seqs=[512, 1024, 2048, 4096, 8192, 16384], schedule="auto", ref_S=2048),
    "causal_h32_d128": dict(
        desc="causal-mask attention backward, H=32, D=128, bf16 N(0,1), B*S=16384, "
             "S swept over {1024,2048,4096,8192,16384}",
        H=32, Hkv=32, D=128, causal=True, tokens=16384,
        seqs=[1024, 2048, 4096, 8192, 16384], schedule="auto", ref_S=2048),
    "causal_h32_d64": dict(
        desc="causal-mask attention backward, H=32, D=64, bf16 N(0,1), B*S=16384, "
             "S swept over {1024,4096,16384}",
        H=32, Hkv=32, D=64, causal=True, tokens=16384, seqs=[1024, 4096, 16384],
        schedule="auto", ref_S=2048),
    "gqa_causal_8b": dict(
        desc="GQA causal attention backward shaped like an 8B decoder layer: 32 query heads, "
             "8 KV heads, D=128, B=2, S=8192",
        H=32, Hkv=8, D=128, causal=True, tokens=16384, seqs=[8192], schedule="auto",
        ref_S=2048),
    "small_b1_h2_s512_d64": dict(
        desc="full-mask attention backward, B=1, H=2, S=512, D=64 (4 KV blocks)",
        H=2, Hkv=2, D=64, causal=False, tokens=512, seqs=[512], schedule="auto", ref_S=512),
}
SCHEDULES = ["atomic", "serial", "descending", "shift", "shift_fill", "shift_dual"]
DETERMINISTIC = ["serial", "descending", "shift", "shift_fill", "shift_dual"]


def schedules_for(D):
    """Schedules a head dim runs (all of them)."""
    return list(SCHEDULES)
FALLBACK_PEAK_TFLOPS = 1900.0   # only if the measured-peaks file is absent
PROFILE = os.path.join(ROOT, "profiles", "bwd_tile_kernel_full_h16_d128.md")
KERNEL_SOURCES = ["bwd_kernel.cuh", "ptx.cuh", "sched.cuh", "common.cuh"]


def bwd_flops(B, S, H, D, causal):
    f = 10.0 * B * H * S * S * D
    return f / 2 if causal else f


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)) or None, "measured"
    except Exception:
        return FALLBACK_PEAK_TFLOPS, None, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for n in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "deterministic_attention_backward_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """dram bytes per tile-kernel launch, cached from the committed ncu summary (ncu cannot
    run inside the timed bench), if it was taken on the current kernel source and this
    workload; else None."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    src = re.search(r"kernel source sha256\[:16\]:\s*([0-9a-f]+)", text)
    wl = re.search(r"workload:\s*(\S+)", text)
    tr = re.search(r"dram bytes per launch[^:]*:\s*([0-9.eE+]+)", text)
    if not (src and wl and tr) or src.group(1) != kernel_source_hash() or wl.group(1) != workload:
        return None
    return float(tr.group(1))


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.out = index, None, None

    def __enter__(self):
        try:
            self.out = open(os.devnull if False else os.path.join(
                "/tmp", f"dash_clocks_{os.getpid()}.csv"), "w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.proc or not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.seek(0)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        self.out.close()
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ GPU arm
def slowest_rank_ms(elapsed_ms, world, device):
    """The timed region's length on the slowest rank (every rank gets the same value)."""
    if world <= 1:
        return elapsed_ms
    import torch
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(step_flops, steps, world, elapsed_ms):
    """Whole-job throughput: the work of every rank (each runs the full workload) over the
    slowest rank's time."""
    return step_flops * steps * world / (elapsed_ms / 1e3) / 1e12


def run_gpu(args, wl, rank, world):
    import torch
    import deterministic_attention_backward_gb300 as dash
    from deterministic_attention_backward_gb300 import _build
    from dash_inputs import make_qkv_do

    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    sched = args.schedule or wl["schedule"]
    H, Hkv, D, causal = wl["H"], wl["Hkv"], wl["D"], wl["causal"]
    seqs = [args.seq] if args.seq else wl["seqs"]

    # inputs resident in HBM, one set per sequence length of the sweep
    probs = []
    for S in seqs:
        B = max(1, wl["tokens"] // S)
        q, k, v, do = (t.to(dev) for t in make_qkv_do(B, S, H, Hkv, D, seed=0))
        o, lse = dash.fwd(q, k, v, causal=causal, check=True)
        ws = torch.empty(dash.bwd_workspace_bytes(B, S, H, D), dtype=torch.uint8, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        probs.append(dict(B=B, S=S, q=q, k=k, v=v, do=do, o=o, lse=lse, ws=ws, dq=dq, dk=dk,
                          dv=dv, flops=bwd_flops(B, S, H, D, causal)))
    step_flops = sum(p["flops"] for p in probs)

    def call(p, schedule, stages=dash.ALL_STAGES):
        dash.bwd(p["q"], p["k"], p["v"], p["o"], p["do"], p["lse"], causal=causal,
                 schedule=schedule, dq=p["dq"], dk=p["dk"], dv=p["dv"], workspace=p["ws"],
                 stages=stages)

    # correctness guard: the timed schedule must report a clean device status
    for p in probs:
        call(p, sched)
        dash.status(p["ws"])

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps * len(probs))]

    def step(record=None):
        for j, p in enumerate(probs):
            call(p, sched, dash.PROLOGUE)
            if record is not None:
                evs[record * len(probs) + j][0].record()
            call(p, sched, dash.TILES)
            if record is not None:
                evs[record * len(probs) + j][1].record()
            call(p, sched, dash.EPILOGUE)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(dev.index) as clk:
        time.sleep(0.3)
        torch.cuda.synchronize()
        t_start.record()
        for s in range(args.steps):
            step(record=s)
        t_end.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    tile_ms = sum(a.elapsed_time(b) for a, b in evs)
    for p in probs:
        dash.status(p["ws"])
    elapsed_ms = slowest_rank_ms(elapsed_ms, world, dev)

    if args.quick:  # timed loop only (profiling runs)
        return {"value_tflops": round(step_flops * args.steps / (elapsed_ms / 1e3) / 1e12, 2),
                "tile_tflops": round(step_flops * args.steps / (tile_ms / 1e3) / 1e12, 2),
                "seq_lens": seqs, "schedule": sched, "workload": args.workload}

    # per-schedule comparison (interleaved, median of reps) on the same inputs
    reps = max(3, min(10, args.steps))
    scheds = schedules_for(D)
    per = {s: [[] for _ in probs] for s in scheds}
    for _ in range(reps):
        for s in scheds:
            for j, p in enumerate(probs):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                call(p, s)
                b.record()
                per[s][j].append((a, b))
    torch.cuda.synchronize()
    sweep = []
    tot = {s: 0.0 for s in scheds}
    for j, p in enumerate(probs):
        row = {"S": p["S"], "B": p["B"]}
        for s in scheds:
            ms = statistics.median(a.elapsed_time(b) for a, b in per[s][j])
            tot[s] += ms
            row[s + "_tflops"] = round(p["flops"] / ms / 1e9, 1)
        for s in DETERMINISTIC:
            if s in scheds:
                row[s + "_slowdown_vs_atomic"] = round(row["atomic_tflops"] / row[s + "_tflops"] - 1, 4)
        row["auto_runs"] = dash.sched_resolve("auto", causal, (p["S"] + 127) // 128, D, H // Hkv)
        sweep.append(row)
    sched_summary = {s: round(step_flops / tot[s] / 1e9, 1) for s in scheds}
    # the schedule the timed step ran at each point (AUTO resolved)
    ran = [dash.sched_resolve(sched, causal, (p["S"] + 127) // 128, D, H // Hkv) for p in probs]
    ran_ms = sum(statistics.median(a.elapsed_time(b) for a, b in per[r][j])
                 for j, r in enumerate(ran))
    ran_tflops = step_flops / ran_ms / 1e9

    # end to end through the public API with host buffers (pinned), copies in the region
    e2e_val, h2d, d2h = None, 0, 0
    if not args.no_e2e:
        host = []
        for p in probs:
            hs = {n: p[n].to("cpu").pin_memory() for n in ("q", "k", "v", "o", "do", "lse")}
            outs = {n: torch.empty(p[n].shape, dtype=p[n].dtype).pin_memory()
                    for n in ("dq", "dk", "dv")}
            host.append((hs, outs))
            h2d += sum(t.numel() * t.element_size() for t in hs.values())
            d2h += sum(t.numel() * t.element_size() for t in outs.values())

        # three streams, so that the copies of one sweep point overlap the backward of the
        # previous one: inputs in, compute (the current stream), results out; a point's
        # buffers are refilled only after its previous backward and read-out are done
        comp = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        done = [None] * len(probs)   # backward of point j finished (its inputs are free)
        out_done = [None] * len(probs)  # read-out of point j finished (its outputs are free)

        def e2e_step():
            for j, (p, (hs, outs)) in enumerate(zip(probs, host)):
                with torch.cuda.stream(s_in):
                    if done[j] is not None:
                        s_in.wait_event(done[j])
                    for n, t in hs.items():
                        p[n].copy_(t, non_blocking=True)
                    ev_in = torch.cuda.Event()
                    ev_in.record(s_in)
                comp.wait_event(ev_in)
                if out_done[j] is not None:
                    comp.wait_event(out_done[j])
                call(p, sched)
                done[j] = torch.cuda.Event()
                done[j].record(comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done[j])
                    for n, t in outs.items():
                        t.copy_(p[n], non_blocking=True)
                    out_done[j] = torch.cuda.Event()
                    out_done[j].record(s_out)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(1, min(args.steps, 5))
        a.record(comp)
        s_in.wait_event(a)
        for _ in range(n_e2e):
            e2e_step()
        for ev in out_done:
            comp.wait_event(ev)
        b.record(comp)
        torch.cuda.synchronize()
        e2e_val = step_flops * n_e2e / (a.elapsed_time(b) / 1e3) / 1e12 * world

    configs = None if (args.no_configs or args.quick) else other_configs(args, dev, dash)
    block = None if (args.no_block or args.quick) else block_timing()
    varlen = None if (args.no_varlen or args.quick) else varlen_timing(dev, dash)

    peak, peak_sus, peak_kind = peaks()
    value = job_tflops(step_flops, args.steps, world, elapsed_ms)
    tile_tflops = step_flops * args.steps / (tile_ms / 1e3) / 1e12
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "description": wl["desc"], "H": H, "Hkv": Hkv,
                   "D": D, "mask": "causal" if causal else "full", "schedule": sched,
                   "seq_lens": seqs, "tokens_per_batch": wl["tokens"],
                   "l2": "inputs larger than L2 (>= 5 bf16 tensors of 16384x H x D per step "
                         "point); no flush" if wl["tokens"] * H * D * 2 * 5 > 129e6 else
                         "inputs smaller than L2; no flush (parity-size workload)",
                   "step": "prologue + tile kernel + dQ convert for every S of the sweep"},
        "pct_of_peak": round(100 * value / world / peak, 2),
        "slowdown_vs_atomic": round(sched_summary["atomic"] / ran_tflops - 1, 4),
        "schedule_ran": sorted(set(ran)),
        "schedules_tflops": sched_summary,
        "sweep": sweep,
        "roofline": {"bound": "tensor", "achieved": round(tile_tflops, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tile_tflops / peak, 4),
                     "traffic": profiled_traffic(args.workload),
                     "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum of one "
                                       "S=4096 tile-kernel launch, cached from "
                                       "profiles/bwd_tile_kernel_full_h16_d128.md (null when "
                                       "the kernel source changed since the capture)",
                     "kernel": "bwd_kernel (tile kernel, " + sched + " -> " + "/".join(sorted(set(ran))) + ")",
                     "peak_source": f"{peak_kind} dense bf16 burst"
                                    + (f"; sustained {peak_sus}" if peak_sus else "")},
        "e2e": {"value": round(e2e_val, 2) if e2e_val else None, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "clocks": clk.summary(),
        "gpu_launches": 3 * len(probs) * args.steps,
    }
    if configs is not None:
        res["configs"] = configs
    if block is not None:
        res["block"] = block
    if varlen is not None:
        res["varlen"] = varlen
    return res


def other_configs(args, dev, dash):
    """Every other workload of the benchmark, each sequence length timed for every schedule
    (whole backward call, interleaved, median of 3 after a warm-up), with the best
    deterministic schedule and its slowdown against the atomic variant.  Inputs are seeded
    N(0,1) draws made on the device (torch's CUDA generator), O and LSE from the forward."""
    import torch
    peak = peaks()[0]
    out = {}
    for name, wl in WORKLOADS.items():
        if name == args.workload:
            continue
        H, Hkv, D, causal = wl["H"], wl["Hkv"], wl["D"], wl["causal"]
        scheds = schedules_for(D)
        rows = []
        for S in wl["seqs"]:
            B = max(1, wl["tokens"] // S)
            g = torch.Generator(device=dev).manual_seed(0)
            q = torch.randn(B, S, H, D, device=dev, generator=g).to(torch.bfloat16)
            k = torch.randn(B, S, Hkv, D, device=dev, generator=g).to(torch.bfloat16)
            v = torch.randn(B, S, Hkv, D, device=dev, generator=g).to(torch.bfloat16)
            do = torch.randn(B, S, H, D, device=dev, generator=g).to(torch.bfloat16)
            o, lse = dash.fwd(q, k, v, causal=causal, check=True)
            ws = torch.empty(dash.bwd_workspace_bytes(B, S, H, D), dtype=torch.uint8, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            flops = bwd_flops(B, S, H, D, causal)

            def call(s):
                dash.bwd(q, k, v, o, do, lse, causal=causal, schedule=s, dq=dq, dk=dk, dv=dv,
                         workspace=ws)
            for s in scheds:
                call(s)
            dash.status(ws)
            ev = {s: [] for s in scheds}
            for _ in range(3):
                for s in scheds:
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    call(s)
                    b.record()
                    ev[s].append((a, b))
            torch.cuda.synchronize()
            dash.status(ws)
            row = {"S": S, "B": B}
            for s in scheds:
                row[s + "_tflops"] = round(flops / statistics.median(a.elapsed_time(b) for a, b in ev[s]) / 1e9, 1)
            best = max(DETERMINISTIC, key=lambda x: row[x + "_tflops"])
            auto = dash.sched_resolve("auto", causal, (S + 127) // 128, D, H // Hkv)
            row.update({"best_deterministic": best,
                        "best_slowdown_vs_atomic": round(row["atomic_tflops"] / row[best + "_tflops"] - 1, 4),
                        "best_pct_of_peak": round(100 * row[best + "_tflops"] / peak, 2),
                        "auto_runs": auto,
                        "auto_slowdown_vs_atomic": round(row["atomic_tflops"] / row[auto + "_tflops"] - 1, 4)})
            rows.append(row)
            del q, k, v, do, o, lse, ws, dq, dk, dv
            torch.cuda.empty_cache()
        out[name] = {"description": wl["desc"], "points": rows}
    return out


VARLEN = {"n": 64, "lo": 64, "hi": 4096, "H": 32, "Hkv": 8, "D": 128, "causal": True, "seed": 0}


def varlen_lengths(cfg=VARLEN):
    """Seeded sequence lengths of the packed batch: log-uniform in [lo, hi]."""
    import numpy as np
    rng = np.random.default_rng(cfg["seed"])
    x = rng.uniform(np.log(cfg["lo"]), np.log(cfg["hi"]), size=cfg["n"])
    return [int(round(float(np.exp(t)))) for t in x]


def varlen_timing(dev, dash, cfg=VARLEN):
    """A packed causal batch of 64 sequences (log-uniform 64..4096 tokens, GQA 32/8 heads,
    D = 128): the whole varlen backward call with every sequence's heads in one tile-kernel
    launch (packed schedules and atomic) against one B = 1 call per sequence (the same
    schedule, AUTO), median of 3 after a warm-up."""
    import numpy as np
    import torch
    lengths = varlen_lengths(cfg)
    H, Hkv, D, causal = cfg["H"], cfg["Hkv"], cfg["D"], cfg["causal"]
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    g = torch.Generator(device=dev).manual_seed(0)
    q = torch.randn(T, H, D, device=dev, generator=g).to(torch.bfloat16)
    k = torch.randn(T, Hkv, D, device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hkv, D, device=dev, generator=g).to(torch.bfloat16)
    do = torch.randn(T, H, D, device=dev, generator=g).to(torch.bfloat16)
    o, lse = dash.fwd_varlen(q, k, v, cu, causal=causal, check=True)
    ws = torch.empty(dash.bwd_varlen_workspace_bytes(cu, H, D), dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flops = sum(bwd_flops(1, S, H, D, causal) for S in lengths)
    slices = []
    for b, S in enumerate(lengths):
        s0 = int(cu[b])
        sl = lambda t: t[s0:s0 + S].unsqueeze(0)
        slices.append((sl(q), sl(k), sl(v), sl(o), sl(do),
                       lse[s0 * H:(s0 + S) * H].view(1, H, S), sl(dq), sl(dk), sl(dv)))

    def packed(s):
        dash.bwd_varlen(q, k, v, o, do, lse, cu, causal=causal, schedule=s, dq=dq, dk=dk, dv=dv,
                        workspace=ws)

    def loop(s):
        for (q1, k1, v1, o1, do1, l1, dq1, dk1, dv1) in slices:
            dash.bwd(q1, k1, v1, o1, do1, l1, causal=causal, schedule=s, dq=dq1, dk=dk1,
                     dv=dv1, workspace=ws)
    runs = {"packed_" + s: (lambda s=s: packed(s)) for s in ("atomic", "shift_fill", "shift_dual", "auto")}
    runs["per_sequence_auto"] = lambda: loop("auto")
    runs["per_sequence_atomic"] = lambda: loop("atomic")
    for f in runs.values():
        f()
    dash.status(ws)
    ev = {n: [] for n in runs}
    for _ in range(3):
        for n, f in runs.items():
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            f()
            b.record()
            ev[n].append((a, b))
    torch.cuda.synchronize()
    dash.status(ws)
    out = {"description": "packed causal batch, " + str(cfg["n"]) + " sequences of "
                          f"{min(lengths)}..{max(lengths)} tokens (log-uniform, seeded), "
                          f"{T} tokens, H={H} Hkv={Hkv} D={D}; TFLOP/s of the whole backward call",
           "tokens": T}
    for n in runs:
        out[n + "_tflops"] = round(flops / statistics.median(a.elapsed_time(b) for a, b in ev[n]) / 1e9, 1)
    auto = dash.sched_resolve("auto", causal, (max(lengths) + 127) // 128, D, H // Hkv)
    out["auto_runs"] = auto
    out["packed_speedup_vs_per_sequence"] = round(out["packed_auto_tflops"] / out["per_sequence_auto_tflops"], 3)
    out["packed_auto_slowdown_vs_atomic"] = round(out["packed_atomic_tflops"] / out["packed_auto_tflops"] - 1, 4)
    return out


def block_timing():
    """Forward + backward of the synthetic 8B-shaped decoder block (random weights) with the
    library's attention under the atomic, serialized and AUTO schedules."""
    from deterministic_attention_backward_gb300.block import time_block
    return time_block(seq=8192, batch=1, schedules=("atomic", "serial", "shift_fill", "auto"),
                      steps=5, warmup=3)


# ------------------------------------------------------------------------------ CPU oracle
class OracleSample:
    """The fp64 oracle on (batch, kv-head) groups of the workload at S = ref_S, one group
    per call; the inputs are drawn once."""

    def __init__(self, wl):
        import oracle
        from dash_inputs import make_qkv_do
        self.oracle, self.wl = oracle, wl
        self.S = wl["ref_S"]
        self.B = max(1, wl["tokens"] // self.S)
        self.G = wl["H"] // wl["Hkv"]
        self.inputs = make_qkv_do(self.B, self.S, wl["H"], wl["Hkv"], wl["D"], seed=0)
        oracle.build()
        self.n = 0

    def group(self):
        """Backward of the next group; returns (algorithmic FLOPs, seconds, threads)."""
        q, k, v, do = self.inputs
        b, g = self.n % self.B, (self.n // self.B) % self.wl["Hkv"]
        self.n += 1
        hs = slice(g * self.G, (g + 1) * self.G)
        t0 = time.perf_counter()
        _, threads = self.oracle.attn_bwd(q[b:b + 1, :, hs], k[b:b + 1, :, g:g + 1],
                                          v[b:b + 1, :, g:g + 1], do[b:b + 1, :, hs],
                                          self.wl["causal"], return_threads=True)
        secs = time.perf_counter() - t0
        return bwd_flops(1, self.S, self.G, self.wl["D"], self.wl["causal"]), secs, threads


def cpu_baseline(wl, budget_s=12.0):
    smp = OracleSample(wl)
    flops = secs = 0.0
    heads = threads = 0
    while (secs < budget_s or heads == 0) and heads < 64:
        f, s, threads = smp.group()
        flops, secs, heads = flops + f, secs + s, heads + 1
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{heads} (batch, kv-head) group(s) at S={smp.S} of this workload, fp64 "
                      f"C/OpenMP oracle, {secs:.1f} s"}


def run_reference(args, wl):
    smp = OracleSample(wl)
    for _ in range(args.warmup):
        smp.group()
    flops = secs = 0.0
    threads = 0
    for _ in range(args.steps):
        f, s, threads = smp.group()
        flops, secs = flops + f, secs + s
    value = flops / secs / 1e12
    sample = (f"one (batch, kv-head) group at S={smp.S} of this workload per step, "
              f"fp64 C/OpenMP oracle")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "description": wl["desc"]},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="full_h16_d128", choices=sorted(WORKLOADS))
    ap.add_argument("--schedule", default=None, choices=SCHEDULES + ["auto"])
    ap.add_argument("--impl", default="dash", choices=["dash", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-schedule table of the other workloads")
    ap.add_argument("--no-block", action="store_true",
                    help="skip the transformer-block timing")
    ap.add_argument("--no-varlen", action="store_true",
                    help="skip the packed variable-length batch timing")
    ap.add_argument("--seq", type=int, default=0,
                    help="run one sequence length of the workload's sweep only")
    ap.add_argument("--quick", action="store_true",
                    help="timed loop only: no schedule table, e2e or CPU baseline (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, wl)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    res = run_gpu(args, wl, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline and not args.quick:
            res["cpu_baseline"] = cpu_baseline(wl)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

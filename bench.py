#!/usr/bin/env python3
"""Benchmark: ring-chunked attention forward TFLOP/s on GB300.

One step = one ra_fwd launch over the whole headline workload (GQA causal:
B=2, H=32, Hkv=8, S=16384, D=128, P=8 chunks of 2048), inputs resident in
HBM.  FLOPs are counted exactly: 4*B*H*D*N_pairs with N_pairs = S(S+1)/2
(allowed query/key pairs; masked work the kernel still does on diagonal
tiles is not counted; softmax work is not counted).

L2 is flushed (a 256 MiB write) between timed steps; each step is timed with
CUDA events on the stream the kernel is launched on.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica of
the workload (nothing is exchanged), so scaling is weak and the value is the
sum over ranks' FLOPs divided by the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle on a bounded row sample of the
same workload (the CPU baseline) with the same metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ring_chunked_attention_gb300.inputs import HEADLINE, WORKLOADS, make_inputs, sample_rows  # noqa: E402

METRIC = "ring-chunked attention fwd TFLOP/s at 1 GB300; % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["ring_chunked_attention_gb300/csrc/ra_fwd.cu",
                  "ring_chunked_attention_gb300/csrc/ra_ptx.cuh",
                  "ring_chunked_attention_gb300/csrc/ra_umma.cuh",
                  "ring_chunked_attention_gb300/csrc/ra_internal.h",
                  "ring_chunked_attention_gb300/csrc/ra_api.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace collapsed, so that a
    comment-only edit does not count as a kernel change (string literals in
    these files hold no comment markers)."""
    import re

    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_sha() -> str:
    """Hash of the code (comments and layout ignored) of the files that make up
    the forward kernel and its launch."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def traffic_for(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernel_sha") != kernel_sha():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []  # (arrival time, csv line)
        self.t = None
        self.window = (0.0, float("inf"))

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0: float, t1: float):
        """Restrict the summary to samples that arrived inside [t0, t1]."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, power, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = self.window
        picked = [ln for t, ln in self.lines if lo <= t <= hi + 0.05]
        if not picked:  # timed region shorter than one sample period
            picked = [ln for _, ln in self.lines[-3:]]
        for ln in picked:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of ``values`` over every rank of the default
    process group (the slowest rank decides a step's time); identity when no
    group is initialised."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in values]
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def weak_scaling_value(world_size: int, units_per_rank: float, seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time, in units of 1e12 per second."""
    return world_size * units_per_rank / seconds / 1e12


# ------------------------------------------------------------- CPU oracle arm
def cpu_oracle_sample(w, budget_s: float = 15.0, seed: int = 0, inputs=None, full: bool = False):
    """Time the fp64 oracle (as it stands) on a bounded deterministic row
    sample of workload ``w`` (every row when ``full``); return (TFLOP/s,
    threads, description, seconds, rows)."""
    import numpy as np

    import oracle

    q, k, v = inputs if inputs is not None else make_inputs(w)
    threads = oracle.default_threads()
    if full:
        t0 = time.perf_counter()
        oracle.attn_direct(q, k, v, w.causal, w.scale, threads=threads)
        dt = time.perf_counter() - t0
        n = w.B * w.H * w.S
        return (w.flops / dt / 1e12, threads,
                f"every one of the {n} query rows of {w.name}, fp64 two-pass, {dt:.1f} s", dt, n)
    rows = sample_rows(w, n_random=1024, every=w.S // 4, seed=seed).numpy()
    rng = np.random.default_rng(seed)
    rows = rng.permutation(rows)
    # calibrate on a small batch, then size the sample to the budget
    s_of = rows % w.S

    def flops(rs):
        s = rs % w.S
        keys = (s + 1) if w.causal else np.full_like(s, w.S)
        return float(4 * w.D * keys.sum())

    n0 = min(len(rows), max(threads * 4, 64))
    t0 = time.perf_counter()
    oracle.attn_direct(q, k, v, w.causal, w.scale, rows=rows[:n0], threads=threads)
    dt0 = time.perf_counter() - t0
    rate = flops(rows[:n0]) / max(dt0, 1e-6)
    # grow the sample until it carries about budget_s of work
    cum = np.cumsum(4 * w.D * (((s_of + 1) if w.causal else np.full_like(s_of, w.S))).astype(np.float64))
    n = int(np.searchsorted(cum, rate * budget_s)) + 1
    n = max(n0, min(n, len(rows)))
    sample = rows[:n]
    t0 = time.perf_counter()
    oracle.attn_direct(q, k, v, w.causal, w.scale, rows=sample, threads=threads)
    dt = time.perf_counter() - t0
    tflops = flops(sample) / dt / 1e12
    desc = (f"{n} query rows (chunk boundaries, every {w.S // 4}th row and seeded random rows "
            f"of every (b,h)) of {w.name}, fp64 two-pass, {dt:.1f} s")
    return tflops, threads, desc, dt, n


def cpu_baseline_obj(w, tf, threads, desc, dt, n, full):
    """The cpu_baseline object: TFLOP/s on the sample, rows/s, and the full
    workload's time extrapolated from the sample's FLOP rate (labelled)."""
    obj = {"value": tf, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
           "rows_per_s": n / dt}
    if full:
        obj["full_s"] = dt
    else:
        obj["extrapolated_full_s"] = w.flops / (tf * 1e12)
    return obj


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    steps = []
    budget = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    inputs = make_inputs(w)
    tf, threads, desc, n = None, None, None, 0
    for i in range(args.warmup + args.steps):
        tf_i, threads, desc, dt, n = cpu_oracle_sample(w, budget_s=budget, seed=i, inputs=inputs,
                                                       full=args.full_oracle)
        if i >= args.warmup:
            steps.append((tf_i, dt))
    tf = statistics.mean(s[0] for s in steps)
    ms = statistics.mean(s[1] for s in steps) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": tf, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv,
                                            "S": w.S, "D": w.D, "P": w.P, "causal": w.causal},
            "cpu_baseline": cpu_baseline_obj(w, tf, threads, desc, ms * 1e-3, n, args.full_oracle),
            "e2e": {"value": tf, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- GPU arm
def measure_merge(ra, w, flush, stream, steps: int = 20):
    """Time ra_merge_partials (the log-sum-exp merge of per-chunk partials)
    on n = P bf16 partials of the workload's output shape.  It streams its
    inputs once, so it is measured against HBM bandwidth: algorithmic bytes =
    n*(B*S*H*D*2 + B*H*S*4) read + B*S*H*D*2 + B*H*S*4 written."""
    import torch

    n = w.P
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    o_parts = torch.randn((n, w.B, w.S, w.H, w.D), generator=g, device="cuda").to(torch.bfloat16)
    lse_parts = torch.randn((n, w.B, w.H, w.S), generator=g, device="cuda")
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    for _ in range(3):
        ra.ra_merge_partials(o_parts, lse_parts, out=out, lse=lse, stream=stream)
    ts = []
    for _ in range(steps):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ra.ra_merge_partials(o_parts, lse_parts, out=out, lse=lse, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = statistics.mean(ts)
    rows = w.B * w.S * w.H
    nbytes = n * (rows * w.D * 2 + rows * 4) + rows * w.D * 2 + rows * 4
    peaks, src = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    del o_parts, lse_parts
    return {"kernel": "merge_kernel (ra_merge_partials)", "n_partials": n, "ms": ms,
            "bytes": nbytes, "bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]),
            "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]), "peak_source": f"{src} copy"}


def measure_bwd(ra, w, flush, stream, qd, kd, vd, out, lse, steps: int = 10):
    """Time ra_bwd (row sums, dk/dv and dq kernels) on the workload, given the
    forward's out and lse and a seeded N(0,1) output gradient.  FLOPs follow
    the usual count of a backward pass, five GEMM-shaped products per allowed
    (query, key) pair (S, dP, dV, dK, dQ: 2.5x the forward's); the kernels
    execute seven (S and dP are recomputed by the dk/dv and the dq kernel),
    reported as ``executed_tflops``."""
    import torch

    g = torch.Generator(device="cuda")
    g.manual_seed(101)
    dout = torch.randn(qd.shape, generator=g, device="cuda").to(torch.bfloat16)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(ra.ra_bwd_workspace_bytes(w.B, w.H, w.S), dtype=torch.uint8, device="cuda")

    def call():
        ra.ra_bwd(qd, kd, vd, out, lse, dout, P=w.P, causal=w.causal, scale=w.scale, dq=dq, dk=dk,
                  dv=dv, workspace=ws, stream=stream)

    for _ in range(3):
        call()
    ts = []
    for _ in range(steps):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    if ra.ra_get_last_device_status() != 0:
        raise RuntimeError("device status reported a timeout in the backward")
    ms = statistics.mean(ts)
    flops = 2.5 * w.flops
    tflops = flops / (ms * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    del dout, dq, dk, dv, ws
    return {"kernels": "bwd_prep + bwd_dkdv + bwd_dq (ra_bwd)", "launches_per_step": 3,
            "ms": ms, "flops": flops, "bound": "tensor", "achieved": tflops, "peak": peak,
            "unit": "TFLOP/s", "frac": tflops / peak, "executed_tflops": 1.4 * tflops,
            "peak_source": f"{src} bf16 dense burst"}


def measure_others(ra, flush, stream, names, steps: int = 5, warmup: int = 2):
    """Device-timed ra_fwd on the other long-context workloads (the forward
    only): median of ``steps`` launches after ``warmup``, L2 flushed before
    each, CUDA events on the launch stream.  Returns {name: {...}}."""
    import torch

    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    res = {}
    for name in names:
        w = WORKLOADS[name]
        q, k, v = (t.cuda() for t in make_inputs(w))
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
        ts = []
        for i in range(warmup + steps):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ra.ra_fwd(q, k, v, P=w.P, causal=w.causal, scale=w.scale, out=out, lse=lse,
                      stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= warmup:
                ts.append(e0.elapsed_time(e1))
        if ra.ra_get_last_device_status() != 0:
            raise RuntimeError(f"device status reported a timeout on {name}")
        ms = statistics.median(ts)
        tf = w.flops / (ms * 1e-3) / 1e12
        res[name] = {"ms": ms, "tflops": tf, "frac": tf / peak, "launches": steps,
                     "config": {"B": w.B, "H": w.H, "Hkv": w.Hkv, "S": w.S, "D": w.D, "P": w.P,
                                "causal": w.causal}}
        del q, k, v, out, lse
        torch.cuda.empty_cache()
    return res


def ceilings_obj(ra, tensor_peak: float):
    """The secondary ceilings beside the tensor roofline, measured on this
    device by the library's microbenchmarks: the rate of ex2 (one per allowed
    pair) and of fp32 FMA-pipe lanes (the kernel's instruction mix spends
    three per pair at D = 128: one fma for the exponent's argument and two
    adds for the exact and the rounded row sums; two at D = 64, where the
    tensor cores take the rounded sum).  Each is converted to the forward
    TFLOP/s it would allow alone (4*D FLOP per pair)."""
    c = ra.ra_measure_ceilings()
    out = {"measured": c, "tensor_peak_tflops": tensor_peak}
    for D, lanes in ((128, 3.0), (64, 2.0)):
        out[f"d{D}"] = {
            "ex2_bound_tflops": c["ex2_per_s"] * 4 * D / 1e12,
            "fp32_lanes_per_pair": lanes,
            "fp32_bound_tflops": c["ffma2_lanes_per_s"] / lanes * 4 * D / 1e12,
        }
    return out


def measure_e2e(ra, w, q, k, v, flush, steps: int, warmup: int = 3):
    """End to end through ra_fwd with the inputs in pinned host memory: every
    step copies its q, k, v host -> device, runs the forward and reads out and
    lse back device -> host.  Steps are pipelined over two device buffer sets
    and three streams (copy in, compute, copy out), with events for every
    dependency: step i's inputs upload while step i-1 computes and step i-2's
    results download.  The same pipeline first runs `warmup` untimed steps
    (the first copies from freshly pinned buffers and the first work on new
    streams), then `steps` timed ones.  Returns (ms per step over the timed
    run, host->device bytes per step, device->host bytes per step, steps)."""
    import torch

    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    dev = []
    for _ in range(2):
        dq_, dk_, dv_ = (torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in (q, k, v))
        dev.append((dq_, dk_, dv_, torch.empty_like(dq_),
                    torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")))
    outh = [torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(2)]
    lseh = [torch.empty((w.B, w.H, w.S), dtype=torch.float32, pin_memory=True) for _ in range(2)]
    h2d = (qh.numel() + kh.numel() + vh.numel()) * 2
    d2h = outh[0].numel() * 2 + lseh[0].numel() * 4
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def pipeline(n, t0=None, t1=None):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        if t0 is not None:
            t0.record(s_in)
        for i in range(n):
            bq, bk, bv, bo, bl = dev[i % 2]
            if i >= 2:
                s_in.wait_event(ev_comp[i - 2])  # the kernel of step i-2 is done with these inputs
            with torch.cuda.stream(s_in):
                bq.copy_(qh, non_blocking=True)
                bk.copy_(kh, non_blocking=True)
                bv.copy_(vh, non_blocking=True)
            ev_in[i].record(s_in)
            s_comp.wait_event(ev_in[i])
            if i >= 2:
                s_comp.wait_event(ev_out[i - 2])  # step i-2's results were read back
            with torch.cuda.stream(s_comp):
                flush.fill_(1.0)
                ra.ra_fwd(bq, bk, bv, P=w.P, causal=w.causal, scale=w.scale, out=bo, lse=bl,
                          stream=s_comp)
            ev_comp[i].record(s_comp)
            s_out.wait_event(ev_comp[i])
            with torch.cuda.stream(s_out):
                outh[i % 2].copy_(bo, non_blocking=True)
                lseh[i % 2].copy_(bl, non_blocking=True)
            ev_out[i].record(s_out)
        if t1 is not None:
            t1.record(s_out)

    torch.cuda.synchronize()
    pipeline(warmup)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pipeline(steps, t0, t1)
    torch.cuda.synchronize()
    if ra.ra_get_last_device_status() != 0:
        raise RuntimeError("device status reported a timeout in the end-to-end steps")
    return t0.elapsed_time(t1) / steps, h2d, d2h, steps


def run_ours(args):
    import torch

    import ring_chunked_attention_gb300 as ra
    from ring_chunked_attention_gb300 import build as rab

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    if rank == 0:
        rab.build()
    if ws > 1:
        torch.distributed.barrier()
    rab.build()  # no-op once built; fails loudly if the toolchain is missing

    w = WORKLOADS[args.workload]
    ra.ra_set_mma_order(args.mma_order)
    q, k, v = make_inputs(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        ra.ra_fwd(qd, kd, vd, P=w.P, causal=w.causal, scale=w.scale, out=out, lse=lse,
                  stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    st = ra.ra_get_last_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {ra.ra_status_string(st)}")

    sampler = ClockSampler(dev)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.5)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start = time.time()
    for e0, e1 in evs:
        flush.fill_(1.0)
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(t_start, time.time())
    clocks = sampler.stop()
    kernel_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    if ra.ra_get_last_device_status() != 0:
        raise RuntimeError("device status reported a timeout in the timed region")
    ms = statistics.mean(kernel_ms)

    # end to end through the public call with host buffers (pinned), copies timed
    e2e_ms, h2d, d2h, e2e_steps = measure_e2e(ra, w, q, k, v, flush, max(10, min(args.steps, 30)),
                                              warmup=max(3, args.warmup))

    merge = None if args.no_merge else measure_merge(ra, w, flush, stream)
    others = None
    if not args.no_others:
        others = measure_others(ra, flush, stream,
                                [n for n in ("causal_s4096", "long_s65536", "d64_s32768")
                                 if n != w.name])
    ceilings = None if args.no_ceilings else ceilings_obj(ra, float(load_peaks()[0]["bf16_tflops"]))
    bwd = None if args.no_bwd else measure_bwd(ra, w, flush, stream, qd, kd, vd, out, lse)

    # slowest rank decides
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], device="cuda")

    flops = w.flops
    value = weak_scaling_value(ws, flops, ms * 1e-3)
    e2e_value = weak_scaling_value(ws, flops, e2e_ms * 1e-3)
    per_launch_tflops = flops / (ms * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    traffic = traffic_for(w.name)

    line = None
    if rank == 0:
        cpu = None
        if ws == 1 and not args.no_cpu_baseline:
            tf, threads, desc, dt, n = cpu_oracle_sample(w, budget_s=args.cpu_seconds,
                                                         inputs=(q, k, v), full=args.full_oracle)
            cpu = cpu_baseline_obj(w, tf, threads, desc, dt, n, args.full_oracle)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "S": w.S, "D": w.D,
                       "P": w.P, "causal": w.causal, "flops_per_step": flops,
                       "l2": "flushed between timed steps (256 MiB write)",
                       "parallelism": f"replicas x{ws}"},
            "roofline": {"bound": "tensor", "achieved": per_launch_tflops, "peak": peak,
                         "unit": UNIT, "frac": per_launch_tflops / peak,
                         "peak_source": f"{src} bf16 dense burst",
                         "frac_of_sustained": per_launch_tflops / float(peaks["bf16_tflops_sustained"]),
                         "traffic": traffic},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
                    "pipelining": "two device buffer sets, three streams: step i's inputs "
                                  "upload while step i-1 computes and step i-2's out/lse "
                                  "download; the time covers every copy of every timed step",
                    "warmup": max(3, args.warmup)},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "kernel_ms": {"min": min(kernel_ms), "median": statistics.median(kernel_ms),
                          "max": max(kernel_ms)},
            "kernel_sha": kernel_sha(),
            "merge": merge,
            "bwd": bwd,
            "others": others,
            "ceilings": ceilings,
            "mma_order": args.mma_order,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def run_ring(args):
    """Ring attention across ranks: the workload's sequence is sharded over the
    N ranks (one GPU each, torchrun, NCCL point-to-point for the key/value
    blocks), or over ``--virtual-ranks`` ranks emulated on one GPU.  One step
    = the whole ring forward of every rank; value = the attention FLOPs of the
    whole sequence over the slowest rank's step time (strong scaling: the
    total work is fixed as N grows)."""
    import torch

    import ring_chunked_attention_gb300 as ra
    from ring_chunked_attention_gb300 import build as rab
    from ring_chunked_attention_gb300.ring import (RingSpec, block_plan, ring_attention, shard,
                                                   virtual_ring_attention)

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    if rank == 0:
        rab.build()
    if ws > 1:
        torch.distributed.barrier()
    rab.build()
    ra.ra_set_mma_order(args.mma_order)
    w = WORKLOADS[args.workload]
    virtual = ws == 1 and args.virtual_ranks > 1
    world = args.virtual_ranks if virtual else ws
    spec = RingSpec(world, w.B, w.H, w.Hkv, w.S, w.D, w.causal, args.ring)
    q, k, v = make_inputs(w)
    mine = range(world) if virtual else [rank]
    qs = [shard(q, spec, r).cuda() for r in mine]
    ks = [shard(k, spec, r).cuda() for r in mine]
    vs = [shard(v, spec, r).cuda() for r in mine]
    del q, k, v
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    launches = 0
    for r in mine:
        steps, counts = block_plan(spec, r)
        launches += sum(len(p) for _, p in steps) + sum(1 for c in counts if c > 1)

    def step():
        if virtual:
            virtual_ring_attention(qs, ks, vs, causal=w.causal, layout=args.ring)
        else:
            ring_attention(qs[0], ks[0], vs[0], causal=w.causal, layout=args.ring, S=w.S)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if ra.ra_get_last_device_status() != 0:
        raise RuntimeError("device status after warm-up reported a timeout")
    sampler = ClockSampler(torch.cuda.current_device())
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.5)
    t_start = time.time()
    ts = []
    for _ in range(args.steps):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    sampler.mark(t_start, time.time())
    clocks = sampler.stop()
    if ra.ra_get_last_device_status() != 0:
        raise RuntimeError("device status reported a timeout in the timed region")
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ts)
    (ms,) = max_over_ranks([ms], device="cuda")
    value = w.flops / (ms * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "mode": "ring", "config": {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv,
                                       "S": w.S, "D": w.D, "causal": w.causal,
                                       "flops_per_step": w.flops, "ring_layout": args.ring,
                                       "ranks": world, "virtual_ranks": virtual,
                                       "l2": "flushed between timed steps (256 MiB write)",
                                       "parallelism": f"sequence ring x{world}"},
            "roofline": {"bound": "tensor", "achieved": value / max(1, ws), "peak": peak,
                         "unit": UNIT, "frac": value / max(1, ws) / peak,
                         "peak_source": f"{src} bf16 dense burst", "traffic": None},
            "gpu_launches": launches * args.steps, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-merge", action="store_true")
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the forward timing of the other long-context workloads")
    ap.add_argument("--no-ceilings", action="store_true",
                    help="skip the ex2 / fp32 microbenchmarks")
    ap.add_argument("--ring", choices=["contiguous", "zigzag"], default=None,
                    help="shard the sequence over the ranks (ring attention across GPUs) "
                         "instead of running one replica per rank")
    ap.add_argument("--virtual-ranks", type=int, default=0,
                    help="with --ring on one GPU: emulate this many ranks in one process")
    ap.add_argument("--mma-order", type=int, default=3, choices=[0, 1, 2, 3],
                    help="forward MMA issue order (3 bridged by a tcgen05.shift, the default; "
                         "0 strict commit wait; 1 grouped; 2 in-order)")
    ap.add_argument("--full-oracle", action="store_true",
                    help="time the CPU oracle on every row of the workload instead of a sample "
                         "(minutes at the long-context sizes)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.ring:
        return run_ring(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python
"""Benchmark of the shared-input batched linear on GB300.

Headline workload (one "step"): the single-token decode batches of a decoder
layer with bf16 weights -- the q/k/v batch (n_in 4096 -> 4096 + 1024 + 1024)
then the gate+up batch (n_in 4096 -> 12288 + 12288), t = 1, each one
``il_matmul_batch`` call over one shared x.  ``value`` is weight GB/s summed
over ranks (weight bytes as ``WeightRef::bytes`` counts them, divided by the
device time of the timed steps).  The weights rotate over several resident
copies so each step streams them from HBM, not L2.

The same JSON line carries every other workload (quantised decode, prefill,
vocab projection, tiny) as ``per_config`` entries, the roofline of the
dominant kernel, the end-to-end figure through host buffers, the clocks seen
during the timed region and the CPU oracle timed on the host as a baseline.

``--impl reference`` times the CPU oracle alone on the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

NOMINAL_HBM_GBS = 8000.0
HEADLINE = wl.DECODE_BF16
METRIC = "weight GB/s and TFLOP/s per job batch (1 GB300) as % of HBM/tensor roofline"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-per-config", action="store_true", help="headline only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", default=None, metavar="WORKLOAD:BATCH:FMT:T",
                    help="time one batch of one workload (e.g. prefill_bf16_gateup_down:gate_up:bf16:512), "
                         "or the centroid LM head (centroid_lm_head), and print its entry")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines: list[str] = []
        self.marks: list[tuple[float, float]] = []
        self.t_lines: list[float] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._reader, daemon=True).start()

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())
            self.t_lines.append(time.time())

    def mark(self, t0: float, t1: float):
        self.marks.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in zip(self.t_lines, self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            inside = any(a - 0.06 <= t <= b + 0.06 for a, b in self.marks)
            rows.append((inside, parts))
        sel = [p for inside, p in rows if inside] or [p for _, p in rows]
        if not sel:
            return None

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(p[1]) for p in sel if num(p[1]) is not None]
        mx = [num(p[2]) for p in sel if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in sel:
            for name, v in zip(names, p[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sel)}


# ---------------------------------------------------------------------------
# timed execution of a list of batches through the C ABI, as one CUDA graph
# ---------------------------------------------------------------------------
class Batch:
    """One uploaded batch: weights (several resident copies), x, y."""

    def __init__(self, sil, torch, inputs: wl.BatchInputs, copies: int):
        self.inputs = inputs
        self.t, self.n_in = inputs.t, inputs.n_in
        if inputs.fused:
            # one fused gate+up job: h = gelu(g) * u, as wide as one of the two
            (f, gate, n), (_, up, _) = inputs.jobs
            self.copies = [[sil.upload_gate_up(f, gate, up, n, inputs.n_in)] for _ in range(copies)]
            widths = [n]
        else:
            self.copies = [[sil.upload_weight(f, buf, n, inputs.n_in) for f, buf, n in inputs.jobs]
                           for _ in range(copies)]
            widths = [n for _, _, n in inputs.jobs]
        self.x = torch.from_numpy(inputs.x).cuda()
        self.ys = [torch.empty((inputs.t, n), device="cuda") for n in widths]
        self.weight_bytes = inputs.weight_bytes
        self.flops = inputs.flops
        self.io_bytes = 4 * inputs.t * inputs.n_in + sum(4 * inputs.t * n for n in widths)

    def launch(self, sil, copy: int, stream):
        sil.matmul_batch(self.x, list(zip(self.copies[copy % len(self.copies)], self.ys)),
                         stream=stream)

    def free(self):
        for c in self.copies:
            for w in c:
                w.free()


def graph_of(torch, sil, batch, steps: int, stream, copy0: int = 0):
    """Capture `steps` launches of one batch (rotating weight copies); kernels only."""
    g = torch.cuda.CUDAGraph()
    launches0 = sil.get_stats()["launches"]
    with torch.cuda.graph(g, stream=stream):
        for s in range(steps):
            batch.launch(sil, copy0 + s, stream)
    launches = sil.get_stats()["launches"] - launches0
    return g, launches


def copies_for(batch_bytes: int) -> int:
    # enough copies that a weight set is re-read only after >= ~1 GB of other weights
    return max(2, min(8, math.ceil(1.0e9 / max(batch_bytes, 1)) + 1))


def run_headline(sil, torch, args, dist, clocks: ClockSampler):
    stream = torch.cuda.Stream()
    inputs = [wl.make_workload_batch(HEADLINE, bt, 1, "bf16") for bt in HEADLINE.batches]
    step_bytes = sum(b.weight_bytes for b in inputs)
    copies = copies_for(step_bytes)
    batches = [Batch(sil, torch, b, copies) for b in inputs]
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for s in range(max(3, args.warmup)):
            for b in batches:
                b.launch(sil, s, stream)
    torch.cuda.synchronize()

    # One graph per batch holding L launches (L divides K).  The timed region
    # replays, K/L times, the q/k/v graph then the gate+up graph, with an event
    # at each graph boundary: that gives the device time of every batch kind
    # over the timed region without events between kernels.
    K = args.steps
    L = graph_steps(K)
    graphs = []
    launches_per_rep = 0
    for b in batches:
        g, n = graph_of(torch, sil, b, L, stream)
        graphs.append(g)
        launches_per_rep += n
    reps = K // L
    with torch.cuda.stream(stream):
        for g in graphs:  # upload + warm
            g.replay()
    torch.cuda.synchronize()

    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
             for _ in range(reps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        for r in range(reps):
            marks[r][0].record(stream)
            for j, g in enumerate(graphs):
                g.replay()
                marks[r][j + 1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    clocks.mark(t0, t1)
    elapsed_ms = marks[0][0].elapsed_time(marks[-1][-1])
    ms_local = elapsed_ms / K
    kern_us = [sum(marks[r][j].elapsed_time(marks[r][j + 1]) for r in range(reps)) * 1e3 / K
               for j in range(len(graphs))]
    launches_per_graph = launches_per_rep

    # e2e: host buffers, pinned, copies inside the timed region every step
    e2e = run_e2e(sil, torch, batches, args, stream)
    for b in batches:
        b.free()
    return {"ms_per_step": ms_local, "step_bytes": step_bytes,
            "step_flops": sum(b.flops for b in inputs),
            "kernel_us": kern_us, "batch_names": [bt.name for bt in HEADLINE.batches],
            "alg_bytes": [b.weight_bytes + b.io_bytes for b in batches],
            "launches": launches_per_graph * reps, "copies": copies, "e2e": e2e,
            "graph_steps": L}


def run_e2e(sil, torch, batches, args, stream):
    """End to end through the C ABI's host-buffer entry point
    (il_matmul_batch_host): every step, each batch's x goes host -> device and its
    y buffers (adjacent in one pinned buffer, so one copy) device -> host inside
    the call; the step ends when the stream has finished both batches."""
    x_sizes = [b.x.numel() for b in batches]
    y_sizes = [[y.numel() for y in b.ys] for b in batches]
    x_host = torch.from_numpy(np.concatenate([b.inputs.x.reshape(-1) for b in batches])).pin_memory()
    y_host = torch.empty(sum(sum(ys) for ys in y_sizes), pin_memory=True)
    h2d = x_host.numel() * 4
    d2h = y_host.numel() * 4
    steps = min(args.steps, 2000)
    # marshal every (batch, weight copy) job array once; x and y live in the two host buffers
    x_ptrs, prepared = [], []
    xo = yo = 0
    for b, xs, ys in zip(batches, x_sizes, y_sizes):
        x_ptrs.append(x_host.data_ptr() + 4 * xo)
        xo += xs
        y_ptrs = []
        for n in ys:
            y_ptrs.append(y_host.data_ptr() + 4 * yo)
            yo += n
        prepared.append([sil.prepare_jobs([(w, w.n_out, yp) for w, yp in zip(copy, y_ptrs)])
                         for copy in b.copies])
    sp = stream.cuda_stream

    def step(s):
        for b, xp, prep in zip(batches, x_ptrs, prepared):
            sil.matmul_batch_host_prepared(xp, b.t, b.n_in, prep[s % len(prep)], sp)
        stream.synchronize()

    for s in range(max(3, args.warmup)):
        step(s)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(steps):
        step(s)
    dt = (time.perf_counter() - t0) / steps
    step_bytes = sum(b.weight_bytes for b in batches)
    return {"value": step_bytes / dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3, "steps": steps,
            "entry": "il_matmul_batch_host"}


def run_per_config(sil, torch, pk, only=None):
    """Every workload x batch x t x format, one batch per measurement."""
    out = []
    stream = torch.cuda.Stream()
    cache = {}
    for w in wl.WORKLOADS:
        for bt in w.batches:
            for fmt in w.fmts:
                for t in w.ts:
                    if only is not None and only != (w.name, bt.name, fmt, t):
                        continue
                    # timing only: the weight draw is reused across t (fresh x per t)
                    key = (w.name, bt.name, fmt)
                    if key not in cache:
                        cache.clear()
                        cache[key] = wl.make_workload_batch(w, bt, t, fmt)
                    base = cache[key]
                    inp = wl.BatchInputs(fmt, t, bt.n_in, wl.make_x(t, bt.n_in, seed=0), base.jobs,
                                         fused=base.fused)
                    copies = copies_for(inp.weight_bytes)
                    b = Batch(sil, torch, inp, copies)
                    try:
                        with torch.cuda.stream(stream):
                            for s in range(3):
                                b.launch(sil, s, stream)
                        torch.cuda.synchronize()
                    except sil.ILError as err:
                        out.append({"workload": w.name, "batch": bt.name, "fmt": fmt, "t": t,
                                    "error": str(err)})
                        b.free()
                        continue
                    iters = max(copies, 8) if t <= 8 else max(2, min(copies, 4))
                    g, _ = graph_of(torch, sil, b, iters, stream)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    with torch.cuda.stream(stream):
                        g.replay()
                        e0.record(stream)
                        for _ in range(3):
                            g.replay()
                        e1.record(stream)
                    torch.cuda.synchronize()
                    us = e0.elapsed_time(e1) * 1e3 / (3 * iters)
                    gbs = inp.weight_bytes / (us * 1e-6) / 1e9
                    tfl = inp.flops / (us * 1e-6) / 1e12
                    e = {"workload": w.name, "batch": bt.name, "fmt": fmt, "t": t,
                         "n_in": bt.n_in, "n_outs": list(bt.n_outs), "us": round(us, 3),
                         "weight_gbs": round(gbs, 1), "tflops": round(tfl, 3),
                         "weight_bytes": inp.weight_bytes}
                    if w.fused:
                        e["fused_gelu_mul"] = True
                    if t <= 8:
                        e["bound"] = "hbm"
                        e["frac_hbm_measured"] = round(gbs / pk["hbm_gbs"], 4)
                        e["frac_hbm_nominal"] = round(gbs / NOMINAL_HBM_GBS, 4)
                    else:
                        e["bound"] = "tensor"
                        e["frac_tensor_burst"] = round(tfl / pk["bf16_tflops"], 4)
                        e["frac_tensor_sustained"] = round(tfl / pk["bf16_tflops_sustained"], 4)
                    out.append(e)
                    del g
                    b.free()
                    torch.cuda.synchronize()
    return out


def run_centroid_head(sil, torch, pk):
    """The centroid-masked LM head on the dense vocab projection's shape: time per call,
    with 8 copies of the centroids and 2 of the embedding rotating (more than L2)."""
    c = wl.CENTROID_HEAD
    inp = wl.make_head_inputs(c.h, c.vocab, c.n_cent, seed=0)
    cws = [sil.upload_weight("bf16", inp.centroids, c.n_cent, c.h) for _ in range(8)]
    ews = [sil.upload_weight("bf16", inp.embed, c.vocab, c.h) for _ in range(2)]
    x = torch.from_numpy(inp.x).cuda()
    od = torch.from_numpy(inp.ordering.view(np.int32)).cuda()
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    score = torch.zeros(1, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(8):
            sil.centroid_head(x, cws[i % 8], ews[i % 2], od, c.top_k, tok, score, stream=stream)
    torch.cuda.synchronize()
    n = 64
    launches0 = sil.get_stats()["launches"]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            sil.centroid_head(x, cws[i % 8], ews[i % 2], od, c.top_k, tok, score, stream=stream)
    launches = (sil.get_stats()["launches"] - launches0) // n
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(3):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (3 * n)
    k_rows = c.top_k * (c.vocab // c.n_cent)
    moved = c.n_cent * c.h * 2 + k_rows * (c.h * 2 + 4)
    del g
    for w in cws + ews:
        w.free()
    return {"workload": c.name, "h": c.h, "vocab": c.vocab, "n_cent": c.n_cent, "top_k": c.top_k,
            "us": round(us, 3), "launches_per_call": launches, "bytes_per_call": moved,
            "gbs": round(moved / (us * 1e-6) / 1e9, 1),
            "frac_hbm_measured": round(moved / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
            "dense_rows_bytes": c.vocab * c.h * 2}


def run_dispatch(sil, torch):
    """Fixed cost of one submission (the pages quote ~0.15 ms per dispatch on Metal):
    host time of an eager il_matmul_batch call, the same call made synchronous, the
    device time of a graph-replayed tiny batch, and a call with no jobs."""
    inp = wl.make_workload_batch(wl.TINY, wl.TINY.batches[0], 1, "bf16")
    b = Batch(sil, torch, inp, 1)
    stream = torch.cuda.Stream()
    jobs = [(w, n, y.data_ptr()) for w, (_, _, n), y in zip(b.copies[0], inp.jobs, b.ys)]
    sp = stream.cuda_stream
    xp = b.x.data_ptr()
    for _ in range(50):
        sil.matmul_batch_ptr(xp, 1, inp.n_in, jobs, sp)
    torch.cuda.synchronize()
    n = 2000
    t0 = time.perf_counter()
    for _ in range(n):
        sil.matmul_batch_ptr(xp, 1, inp.n_in, jobs, sp)
    host_us = (time.perf_counter() - t0) / n * 1e6
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        sil.matmul_batch_ptr(xp, 1, inp.n_in, jobs, sp)
        stream.synchronize()
    sync_us = (time.perf_counter() - t0) / n * 1e6
    t0 = time.perf_counter()
    for _ in range(n):
        sil.matmul_batch_ptr(xp, 1, inp.n_in, [], sp)
    empty_us = (time.perf_counter() - t0) / n * 1e6
    g, _ = graph_of(torch, sil, b, 100, stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    dev_us = e0.elapsed_time(e1) * 1e3 / 100
    del g
    b.free()
    return {"workload": "tiny_bf16 (n_in 256 -> 512 + 256, t = 1), 2 jobs",
            "host_us_per_call_async": round(host_us, 2),
            "host_us_per_call_synchronous": round(sync_us, 2),
            "host_us_per_empty_call": round(empty_us, 2),
            "device_us_per_batch_graph": round(dev_us, 2),
            "pages_metal_dispatch_us": 150.0}


# ---------------------------------------------------------------------------
# CPU oracle on the host (baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def host_threads() -> int:
    """Host cores the oracle may use (affinity-aware where the OS says)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def oracle_steps(seconds: float, min_steps: int = 1, max_steps: int | None = None, threads: int = 1):
    import oracle
    inputs = [wl.make_workload_batch(HEADLINE, bt, 1, "bf16") for bt in HEADLINE.batches]
    step_bytes = sum(b.weight_bytes for b in inputs)
    oracle.linear_threads(*inputs[0].jobs[0][:2], inputs[0].jobs[0][2], inputs[0].n_in,
                          inputs[0].x, threads)  # load + warm
    n, t0 = 0, time.perf_counter()
    while True:
        for b in inputs:
            for fmt, buf, n_out in b.jobs:
                oracle.linear_threads(fmt, buf, n_out, b.n_in, b.x, threads)
        n += 1
        el = time.perf_counter() - t0
        if (max_steps is not None and n >= max_steps) or (max_steps is None and n >= min_steps
                                                          and el >= seconds):
            break
    return {"value": step_bytes / (el / n) / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} full decode steps (q/k/v + gate/up batches, t=1, bf16 weights, "
                      f"{step_bytes} weight bytes each), C oracle with each job's rows split over "
                      f"{threads} host threads, f64 accumulate",
            "ms_per_step": el / n * 1e3, "steps": n}


def _first_rows(fmt: str, buf: np.ndarray, n_out: int, n_in: int, rows: int) -> np.ndarray:
    """The first `rows` rows of a weight in its host layout (quants, then scales)."""
    if fmt == "bf16":
        return buf[: rows * n_in * 2]
    qrow = n_in if fmt == "q8" else n_in // 2
    srow = 4 * (n_in // 32)
    return np.concatenate([buf[: rows * qrow], buf[n_out * qrow: n_out * qrow + rows * srow]])


def oracle_config_ms(inp: wl.BatchInputs, threads: int, budget_macs: float = 1.5e9):
    """The oracle's time for one whole batch on `threads` host cores, measured on a
    bounded sample: the first rows of every job (a fraction of each) and, beyond 64
    tokens, the first 64 token rows; the time is scaled by the work left out (every
    row and token costs the same)."""
    import oracle
    total = float(inp.t) * inp.n_in * sum(n for _, _, n in inp.jobs)
    x = inp.x[:64]
    tok_frac = x.shape[0] / inp.t
    row_frac = min(1.0, budget_macs / (total * tok_frac))
    done = 0.0
    t0 = time.perf_counter()
    for fmt, buf, n_out in inp.jobs:
        rows = max(1, min(n_out, math.ceil(n_out * row_frac)))
        oracle.linear_threads(fmt, _first_rows(fmt, buf, n_out, inp.n_in, rows), rows, inp.n_in, x, threads)
        done += float(x.shape[0]) * inp.n_in * rows
    el = time.perf_counter() - t0
    return el * total / done * 1e3, done / total


def add_oracle_times(entries, threads: int):
    """cpu_ms (the oracle on the host cores, per batch) and the GPU's speed-up over it,
    for every per-config entry."""
    cache = {}
    for e in entries:
        if "error" in e:
            continue
        w = wl.BY_NAME[e["workload"]]
        bt = next(b for b in w.batches if b.name == e["batch"])
        key = (w.name, bt.name, e["fmt"])
        if key not in cache:
            cache.clear()
            cache[key] = wl.make_workload_batch(w, bt, e["t"], e["fmt"])
        base = cache[key]
        inp = wl.BatchInputs(e["fmt"], e["t"], bt.n_in, wl.make_x(e["t"], bt.n_in, seed=0), base.jobs)
        ms, frac = oracle_config_ms(inp, threads)
        e["cpu_ms"] = round(ms, 3)
        e["cpu_cores"] = threads
        e["cpu_sample_fraction"] = round(frac, 6)
        e["gpu_speedup_over_cpu"] = round(ms * 1e3 / e["us"], 1)


def graph_steps(K: int) -> int:
    """Launches per captured graph: the largest divisor of K up to 200."""
    return max(d for d in range(1, min(K, 200) + 1) if K % d == 0)


def headline_config(steps: int, world: int) -> dict:
    """The headline workload's config, the same for both arms of the benchmark."""
    step_bytes = sum(2 * bt.n_in * sum(bt.n_outs) for bt in HEADLINE.batches)
    copies = copies_for(step_bytes)
    return {"workload": "decode_bf16 q/k/v + gate/up batches, t=1, n_in=4096 "
                        "(n_out 4096+1024+1024 and 12288+12288)",
            "t": 1, "n_in": 4096, "formats": "bf16",
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": f"weights rotate over {copies} resident copies ({copies * step_bytes / 1e9:.2f} GB > L2)",
            "timing": f"CUDA graphs of {graph_steps(max(1, steps))} launches replayed, one graph per batch "
                      "kind, CUDA events at graph boundaries on the launching stream"}


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    config = headline_config(args.steps, world)

    if args.impl == "reference":
        if rank != 0:
            return 0
        threads = host_threads()
        # every step is one full decode step: keep K steps of the run bounded
        steps = max(1, args.steps) if args.steps <= 50 else 20
        warm = max(0, args.warmup) if args.warmup <= 50 else 3
        if warm:
            oracle_steps(0, max_steps=warm, threads=threads)
        r = oracle_steps(0, max_steps=steps, threads=threads)
        line = {"impl": "reference", "metric": METRIC, "value": round(r["value"], 3),
                "unit": "GB/s", "n_gpus": args.gpus, "steps": r["steps"], "warmup": warm,
                "ms_per_step": round(r["ms_per_step"], 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config,
                "cpu_baseline": {"value": round(r["value"], 3), "unit": "GB/s", "cores": r["cores"],
                                 "kind": "oracle", "sample": r["sample"]},
                "e2e": {"value": round(r["value"], 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    import shared_input_linear_gb300 as sil

    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    sil.build()
    sil.load()
    pk = peaks()
    if args.only == wl.CENTROID_HEAD.name:
        entry = run_centroid_head(sil, torch, pk)
        if rank == 0:
            print(json.dumps({"metric": METRIC, "only": entry}))
        return 0
    if args.only is not None:
        wname, bname, fmt, t = args.only.split(":")
        entries = run_per_config(sil, torch, pk, only=(wname, bname, fmt, int(t)))
        if not entries:
            raise SystemExit(f"--only {args.only}: no such workload entry")
        if rank == 0:
            print(json.dumps({"metric": METRIC, "only": entries[0]}))
        return 0

    clocks = ClockSampler(local)
    clocks.start()
    head = run_headline(sil, torch, args, dist, clocks)
    clk = clocks.stop()

    ms, value = aggregate(head["ms_per_step"], head["step_bytes"], world, dist, "cuda")

    per_config = None
    dispatch = None
    lm_head = None
    if rank == 0 and world == 1 and not args.no_per_config:
        per_config = run_per_config(sil, torch, pk)
        dispatch = run_dispatch(sil, torch)
        lm_head = run_centroid_head(sil, torch, pk)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = host_threads()
        r = oracle_steps(args.cpu_seconds, threads=threads)
        cpu = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()
               if k in ("value", "unit", "cores", "kind", "sample")}
        if per_config is not None:
            add_oracle_times(per_config, threads)

    if rank == 0:
        kus = head["kernel_us"]
        alg = head["alg_bytes"]
        # one decode launch per batch: average algorithmic bytes and duration per launch
        alg_avg = sum(alg) / len(alg)
        us_avg = sum(kus) / len(kus)
        achieved = alg_avg / (us_avg * 1e-6) / 1e9
        prof = read_profile_traffic()
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "traffic": prof, "peak_source": pk["source"] + " (MEASURED_PEAKS hbm_gbs)",
                "kernel": "decode_kernel<bf16> (one launch per batch: q/k/v, gate+up)",
                "alg_bytes_per_launch": round(alg_avg),
                "us_per_launch": round(us_avg, 3),
                "per_launch_us": {n: round(u, 3) for n, u in zip(head["batch_names"], kus)},
                "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4)}
        e2e = head["e2e"]
        line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded N(0,1) x, N(0,0.02) W)",
                "config": config,
                "tflops": round(head["step_flops"] * world / (ms * 1e-3) / 1e12, 4),
                "roofline": roof, "e2e": {k: (round(v, 3) if isinstance(v, float) else v)
                                          for k, v in e2e.items()},
                "gpu_launches": head["launches"], "clocks": clk, "cpu_baseline": cpu,
                "per_config": per_config, "dispatch": dispatch, "centroid_head": lm_head}
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def aggregate(ms_local: float, step_bytes: int, world: int, dist=None, device="cpu"):
    """Whole-job figures of N independent replicas: the slowest rank's time per step,
    and the weight bytes of all ranks over that time (GB/s)."""
    ms = ms_local
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, step_bytes * world / (ms * 1e-3) / 1e9


def read_profile_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it matches this kernel build."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "decode_bf16_qkv_gateup_t1.md")
    src = os.path.join(ROOT, "shared_input_linear_gb300", "csrc", "gemv.cu")
    try:
        text = open(path).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s+gemv_sha256_16:\s*([0-9a-f]+)", text)
    if m is None or m.group(2) != digest:
        return None
    return float(m.group(1))


if __name__ == "__main__":
    sys.exit(main())

"""Seeded random batches through every entry point against the f64 CPU oracle:
random n_in (the format's multiple), ragged job widths, job counts, token counts on
both sides of the decode / tensor-core thresholds, plain and fused gate+up jobs of
mixed formats in one batch."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import GUARD, lib

pytestmark = pytest.mark.gpu

FMTS = ("bf16", "q8", "q4")


def draw_case(rng):
    n_in = int(rng.choice([32, 64, 96, 256, 480, 1024, 1056, 2080]))
    t = int(rng.choice([1, 2, 3, 5, 8, 9, 12, 16, 17, 24, 40, 100]))
    jobs = []
    for _ in range(int(rng.integers(1, 5))):
        fmt = str(rng.choice(FMTS))
        fused = bool(rng.random() < 0.25)
        n_out = int(rng.integers(1, 300)) * (2 if fused else 1)
        jobs.append((fmt, fused, n_out))
    return n_in, t, jobs


def run_case(sil, seed, entry):
    import torch
    rng = np.random.default_rng(seed)
    n_in, t, jobs = draw_case(rng)
    x = wl.make_x(t, n_in, seed=seed)
    handles, refs, widths = [], [], []
    for i, (fmt, fused, n_out) in enumerate(jobs):
        if fused:
            b = wl.make_batch(n_in, (n_out // 2, n_out // 2), 1, fmt, seed=seed * 31 + i)
            gate, up = b.jobs[0][1], b.jobs[1][1]
            handles.append(sil.upload_gate_up(fmt, gate, up, n_out // 2, n_in))
            refs.append(("gate_up", fmt, gate, up, n_out // 2))
            widths.append(n_out // 2)
        else:
            b = wl.make_batch(n_in, (n_out,), 1, fmt, seed=seed * 31 + i)
            handles.append(sil.upload_weight(fmt, b.jobs[0][1], n_out, n_in))
            refs.append(("linear", fmt, b.jobs[0][1], None, n_out))
            widths.append(n_out)
    try:
        if entry == "device":
            bufs = [torch.full((2 * GUARD + t * n,), float("nan"), device="cuda") for n in widths]
            ys = [bf[GUARD:GUARD + t * n].view(t, n) for bf, n in zip(bufs, widths)]
            sil.matmul_batch(torch.from_numpy(x).cuda(), list(zip(handles, ys)))
            torch.cuda.synchronize()
            outs = [bf.cpu().numpy() for bf in bufs]
        else:
            bufs = [torch.full((2 * GUARD + t * n,), float("nan"), pin_memory=(entry == "host_pinned"))
                    for n in widths]
            ys = [bf[GUARD:GUARD + t * n].view(t, n) for bf, n in zip(bufs, widths)]
            sil.matmul_batch_host(torch.from_numpy(x), list(zip(handles, ys)))
            outs = [bf.numpy().copy() for bf in bufs]
        for j, ((kind, fmt, w0, w1, n), h, width) in enumerate(zip(refs, outs, widths)):
            guard = np.concatenate([h[:GUARD], h[GUARD + t * width:]])
            assert np.all(np.isnan(guard)), f"seed {seed} job {j}: a write outside y"
            y = h[GUARD:GUARD + t * width].reshape(t, width)
            if kind == "linear":
                y_ref, mag = oracle.linear(fmt, w0, n, n_in, x)
                ok, worst, idx = oracle.check(y, y_ref, mag)
            else:
                _, g, u, mg, mu = oracle.gate_up(fmt, w0, w1, n, n_in, x)
                ok, worst, idx = oracle.check_gate_up(y, g, u, mg, mu)
            assert ok, (f"seed {seed} ({entry}) job {j} {kind} {fmt} t={t} n_in={n_in} n_out={n}: "
                        f"element {idx} is {worst:.3g} x tolerance")
    finally:
        for hd in handles:
            hd.free()


@pytest.mark.parametrize("seed", range(64))
def test_random_batch_device_buffers(seed):
    run_case(lib(), 1000 + seed, "device")


@pytest.mark.parametrize("seed", range(16))
@pytest.mark.parametrize("entry", ["host_pinned", "host_pageable"])
def test_random_batch_host_buffers(seed, entry):
    run_case(lib(), 2000 + seed, entry)

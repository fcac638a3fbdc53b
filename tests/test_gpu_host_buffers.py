"""il_matmul_batch_host: the batch on HOST x and y (the form in which the pages'
`Backend::matmul` takes them), against the f64 CPU oracle, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest

import workloads as wl
from gpu_util import GUARD, assert_parity, lib, upload

pytestmark = pytest.mark.gpu


def host_run(sil, b, weights, pinned=True, x_offset=0, canary=float("nan"), stream=None):
    """One batch through il_matmul_batch_host with every y in its own host buffer
    between canaries; returns (ys, guards intact?)."""
    import torch
    xs = torch.zeros(b.t * b.n_in + x_offset, dtype=torch.float32, pin_memory=pinned)
    xs[x_offset:] = torch.from_numpy(b.x.reshape(-1))
    x = xs[x_offset:].view(b.t, b.n_in)
    bufs, ys = [], []
    for (_, _, n) in b.jobs:
        full = torch.full((2 * GUARD + b.t * n,), canary, dtype=torch.float32, pin_memory=pinned)
        bufs.append(full)
        ys.append(full[GUARD:GUARD + b.t * n].view(b.t, n))
    sil.matmul_batch_host(x, list(zip(weights, ys)), stream=stream)
    out, ok = [], True
    for full, (_, _, n) in zip(bufs, b.jobs):
        h = full.numpy()
        g = np.concatenate([h[:GUARD], h[GUARD + b.t * n:]])
        ok &= bool(np.all(np.isnan(g)))
        out.append(h[GUARD:GUARD + b.t * n].reshape(b.t, n).copy())
    return out, ok


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t", [1, 5, 12, 40])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffers_match_oracle(fmt, t, pinned):
    # decode (t <= 8 bf16, <= 16 Q8/Q4) and tensor-core (t = 40) paths, ragged shapes
    sil = lib()
    b = wl.make_batch(320, (200, 72, 48), t, fmt, seed=11 + t)
    ws = upload(sil, b)
    try:
        ys, ok = host_run(sil, b, ws, pinned=pinned)
        assert ok, "a write outside y"
        assert_parity(b, ys, what=f"host {fmt} pinned={pinned}")
    finally:
        for w in ws:
            w.free()


@pytest.mark.parametrize("fmt,t", [("bf16", 1), ("q4", 8), ("bf16", 40), ("q8", 40)])
def test_host_and_device_entry_points_agree_bitwise(fmt, t):
    # same kernels on the same data: the host entry point only changes where x and y live
    import torch
    sil = lib()
    b = wl.make_batch(256, (128, 96), t, fmt, seed=3)
    ws = upload(sil, b)
    try:
        ys_h, ok = host_run(sil, b, ws)
        assert ok
        x = torch.from_numpy(b.x).cuda()
        ys_d = [torch.empty(t, n, device="cuda") for _, _, n in b.jobs]
        sil.matmul_batch(x, list(zip(ws, ys_d)))
        torch.cuda.synchronize()
        for yh, yd in zip(ys_h, ys_d):
            assert np.array_equal(yh.view(np.uint32), yd.cpu().numpy().view(np.uint32))
    finally:
        for w in ws:
            w.free()


@pytest.mark.parametrize("pinned", [False, True])
def test_adjacent_ys_come_back_whole_and_gaps_stay_untouched(pinned):
    # jobs 0 and 1 share one host buffer back to back (one copied run when the
    # buffer is pageable), job 2 lies after a gap in the same buffer (its own run);
    # the gap and the ends keep their canaries (page-locked: written in place)
    import torch
    sil = lib()
    b = wl.make_batch(512, (136, 64, 200), 3, "q8", seed=5)
    ws = upload(sil, b)
    try:
        n0, n1, n2 = (n for _, _, n in b.jobs)
        t = b.t
        gap = 40
        total = GUARD + t * (n0 + n1) + gap + t * n2 + GUARD
        buf = torch.full((total,), float("nan"), dtype=torch.float32, pin_memory=pinned)
        o0 = GUARD
        o1 = o0 + t * n0
        o2 = o1 + t * n1 + gap
        ys = [buf[o0:o0 + t * n0].view(t, n0), buf[o1:o1 + t * n1].view(t, n1),
              buf[o2:o2 + t * n2].view(t, n2)]
        # jobs listed out of address order
        sil.matmul_batch_host(torch.from_numpy(b.x), [(ws[2], ys[2]), (ws[0], ys[0]), (ws[1], ys[1])])
        h = buf.numpy()
        assert np.all(np.isnan(h[:o0])) and np.all(np.isnan(h[o1 + t * n1:o2])) and np.all(np.isnan(h[o2 + t * n2:]))
        assert_parity(b, [y.numpy().copy() for y in ys], what="runs")
    finally:
        for w in ws:
            w.free()


def test_unaligned_host_x():
    # a host x needs no alignment: a page-locked x off a 16-byte boundary is copied
    # into the library's device buffer (y is still written in place)
    sil = lib()
    b = wl.make_batch(256, (64,), 2, "bf16", seed=8)
    ws = upload(sil, b)
    try:
        ys, ok = host_run(sil, b, ws, x_offset=1)
        assert ok
        assert_parity(b, ys, what="x at +4 bytes")
    finally:
        for w in ws:
            w.free()


def test_device_buffers_are_refused_with_nothing_written():
    import torch
    sil = lib()
    b = wl.make_batch(256, (64, 32), 1, "bf16", seed=9)
    ws = upload(sil, b)
    try:
        before = sil.get_stats()["batches"]
        y_host = torch.full((1, 64), 7.0, pin_memory=True)
        y_dev = torch.full((1, 32), 7.0, device="cuda")
        x_host = torch.from_numpy(b.x)
        x_dev = x_host.cuda()
        sp = torch.cuda.current_stream().cuda_stream
        jobs = sil.prepare_jobs([(ws[0], 64, y_host.data_ptr()), (ws[1], 32, y_dev.data_ptr())])
        with pytest.raises(sil.ILError) as e:
            sil.matmul_batch_host_prepared(x_host.data_ptr(), 1, 256, jobs, sp)
        assert e.value.code == -1 and "device memory" in str(e.value)
        jobs = sil.prepare_jobs([(ws[0], 64, y_host.data_ptr())])
        with pytest.raises(sil.ILError) as e:
            sil.matmul_batch_host_prepared(x_dev.data_ptr(), 1, 256, jobs, sp)
        assert e.value.code == -1 and "x is device memory" in str(e.value)
        torch.cuda.synchronize()
        assert torch.all(y_host == 7.0) and torch.all(y_dev == 7.0)
        assert sil.get_stats()["batches"] == before
    finally:
        for w in ws:
            w.free()


def test_overlapping_host_ys_are_refused():
    import torch
    sil = lib()
    b = wl.make_batch(256, (64, 64), 1, "bf16", seed=10)
    ws = upload(sil, b)
    try:
        buf = torch.zeros(100, pin_memory=True)
        with pytest.raises(sil.ILError) as e:
            sil.matmul_batch_host(torch.from_numpy(b.x), [(ws[0], buf[0:64].view(1, 64)),
                                                          (ws[1], buf[32:96].view(1, 64))])
        assert e.value.code == -1
    finally:
        for w in ws:
            w.free()


def test_graph_capture_with_pinned_buffers():
    # a call on page-locked memory (launches only, x and y used in place) can be
    # captured; replays read the host x of the moment and write the host y
    import torch
    sil = lib()
    b = wl.make_batch(256, (96, 40), 1, "q4", seed=12)
    ws = upload(sil, b)
    try:
        s = torch.cuda.Stream()
        x = torch.from_numpy(b.x).pin_memory()
        ys = [torch.empty(1, n, pin_memory=True) for _, _, n in b.jobs]
        jobs = sil.prepare_jobs([(w, n, y.data_ptr()) for w, (_, _, n), y in zip(ws, b.jobs, ys)])
        sil.matmul_batch_host_prepared(x.data_ptr(), 1, 256, jobs, s.cuda_stream)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            sil.matmul_batch_host_prepared(x.data_ptr(), 1, 256, jobs, s.cuda_stream)
        for seed in (21, 22):
            b2 = wl.BatchInputs(b.fmt, 1, 256, wl.make_x(1, 256, seed=seed), b.jobs)
            x.copy_(torch.from_numpy(b2.x))
            g.replay()
            torch.cuda.synchronize()
            assert_parity(b2, [y.numpy().copy() for y in ys], what=f"replay x seed {seed}")
    finally:
        for w in ws:
            w.free()


@pytest.mark.parametrize("t", [1, 12, 40])
@pytest.mark.parametrize("pinned", [True, False])
def test_mixed_formats_and_fused_gate_up_on_host_buffers(t, pinned):
    # a fused gate+up job next to plain jobs of every format, over one host x:
    # one launch per format, every y back in host memory
    import oracle
    import torch
    sil = lib()
    n_in = 512
    gu = wl.make_batch(n_in, (200, 200), t, "q8", seed=60 + t)
    x, gate, up = gu.x, gu.jobs[0][1], gu.jobs[1][1]
    fused = sil.upload_gate_up("q8", gate, up, 200, n_in)
    plain = [wl.make_batch(n_in, (n,), 1, f, seed=70 + i).jobs[0] for i, (f, n) in
             enumerate((("bf16", 96), ("q4", 64), ("q8", 40)))]
    pw = [sil.upload_weight(f, buf, n, n_in) for f, buf, n in plain]
    try:
        widths = [200] + [n for _, _, n in plain]
        bufs = [torch.full((2 * GUARD + t * n,), float("nan"), pin_memory=pinned) for n in widths]
        ys = [b[GUARD:GUARD + t * n].view(t, n) for b, n in zip(bufs, widths)]
        sil.matmul_batch_host(torch.from_numpy(x), list(zip([fused] + pw, ys)))
        for b, n in zip(bufs, widths):
            h = b.numpy()
            assert np.all(np.isnan(np.concatenate([h[:GUARD], h[GUARD + t * n:]])))
        h_ref, g, u, mg, mu = oracle.gate_up("q8", gate, up, 200, n_in, x)
        assert oracle.check_gate_up(ys[0].numpy(), g, u, mg, mu)[0]
        for (f, buf, n), y in zip(plain, ys[1:]):
            y_ref, mag = oracle.linear(f, buf, n, n_in, x)
            assert oracle.check(y.numpy(), y_ref, mag)[0], f
    finally:
        fused.free()
        for w in pw:
            w.free()


@pytest.mark.parametrize("x_pinned,y_pinned", [(True, False), (False, True)])
def test_pinned_and_pageable_buffers_mixed(x_pinned, y_pinned):
    # x used in place and y copied back, or x copied in and y written in place
    import torch
    sil = lib()
    for fmt, t in (("bf16", 3), ("q4", 40)):
        b = wl.make_batch(384, (136, 64), t, fmt, seed=t + 77)
        ws = upload(sil, b)
        try:
            x = torch.from_numpy(b.x)
            x = x.pin_memory() if x_pinned else x.clone()
            bufs = [torch.full((2 * GUARD + t * n,), float("nan"), pin_memory=y_pinned) for _, _, n in b.jobs]
            ys = [buf[GUARD:GUARD + t * n].view(t, n) for buf, (_, _, n) in zip(bufs, b.jobs)]
            sil.matmul_batch_host(x, list(zip(ws, ys)))
            for buf, (_, _, n) in zip(bufs, b.jobs):
                h = buf.numpy()
                assert np.all(np.isnan(np.concatenate([h[:GUARD], h[GUARD + t * n:]])))
            assert_parity(b, [y.numpy().copy() for y in ys], what=f"{fmt} x_pinned={x_pinned}")
        finally:
            for w in ws:
                w.free()

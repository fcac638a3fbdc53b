"""il_matmul_batch_noalloc: the entry point for callers that cannot let the
library allocate device memory (services whose device memory all belongs to
their own pool, latency-critical threads that must not call cudaMalloc).

It is checked through the C ABI against il_matmul_batch, on two calls in a
row, within the same per-element tolerance as every parity test.  This file
sorts last so that a run stopping at the first failure has run all others.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sil():
    import torch
    torch.cuda.set_device(0)
    return lib()


def _run(sil, entry, b, weights, x):
    import torch
    ys = [torch.full((b.t, n), float("nan"), device="cuda") for _, _, n in b.jobs]
    jobs = [(w, n, y.data_ptr()) for w, (_, _, n), y in zip(weights, b.jobs, ys)]
    stream = torch.cuda.current_stream().cuda_stream
    entry(x.data_ptr(), b.t, b.n_in, jobs, stream)
    torch.cuda.synchronize()
    return [y.cpu().numpy() for y in ys]


@pytest.mark.parametrize("fmt,t,n_in,n_outs", [
    ("bf16", 40, 1024, (300, 64)),    # tensor-core path: x's bf16 copy in the static scratch
    ("bf16", 3, 1024, (300, 64)),     # decode path
    ("q4", 20, 512, (200,)),          # decode path in token groups
])
def test_noalloc_matches_existing_entry_point(sil, fmt, t, n_in, n_outs):
    import torch
    for call in range(2):  # two calls in a row, different x
        b = wl.make_batch(n_in, n_outs, t, fmt, seed=100 + call)
        weights = [sil.upload_weight(f, buf, n, n_in) for f, buf, n in b.jobs]
        x = torch.from_numpy(b.x).cuda()
        ref = _run(sil, sil.matmul_batch_ptr, b, weights, x)
        got = _run(sil, sil.matmul_batch_noalloc_ptr, b, weights, x)
        for (f, buf, n), y_ref_gpu, y in zip(b.jobs, ref, got):
            _, mag = oracle.linear(f, buf, n, n_in, b.x)
            tol = oracle.tolerance(mag)
            assert np.all(np.abs(y.astype(np.float64) - y_ref_gpu) <= tol), (fmt, t, call)
            y_ref, _ = oracle.linear(f, buf, n, n_in, b.x)
            ok, worst, _ = oracle.check(y, y_ref, mag)
            assert ok, (fmt, t, call, worst)
        for w in weights:
            w.free()


def test_noalloc_rejects_more_than_its_scratch(sil):
    import torch
    n_in, t = 4096, 2049  # 2049 * 4096 * 2 bytes > 16 MiB
    b = wl.make_batch(n_in, (8,), 1, "bf16", seed=1)
    w = sil.upload_weight("bf16", b.jobs[0][1], 8, n_in)
    x = torch.zeros((t, n_in), device="cuda")
    y = torch.full((t, 8), 7.0, device="cuda")
    with pytest.raises(sil.ILError) as ei:
        sil.matmul_batch_noalloc_ptr(x.data_ptr(), t, n_in, [(w, 8, y.data_ptr())],
                                     torch.cuda.current_stream().cuda_stream)
    assert ei.value.code == -8
    torch.cuda.synchronize()
    assert bool(torch.all(y == 7.0))
    w.free()


def test_noalloc_allocates_no_device_memory(sil):
    # The property the entry point exists for: after one call of each path (which
    # loads the kernels and sets the device up), further calls leave the device's
    # free memory unchanged.  Only no-alloc calls run here, so no scratch of
    # il_matmul_batch can hide an allocation.
    import torch
    cases = [("bf16", 40, 1024, (300, 64)),   # tensor-core path, bf16
             ("q8", 24, 512, (136,)),         # tensor-core path, Q8 dequantised in shared memory
             ("bf16", 3, 1024, (300, 64)),    # decode kernel, bf16
             ("q4", 3, 512, (200, 24))]       # decode kernel, Q4
    calls = []
    keep = []
    for fmt, t, n_in, n_outs in cases:
        b = wl.make_batch(n_in, n_outs, t, fmt, seed=7)
        weights = [sil.upload_weight(f, buf, n, n_in) for f, buf, n in b.jobs]
        x = torch.from_numpy(b.x).cuda()
        ys = [torch.empty((t, n), device="cuda") for n in n_outs]
        keep.append((weights, x, ys))
        calls.append((x.data_ptr(), t, n_in, [(w, n, y.data_ptr()) for w, n, y in zip(weights, n_outs, ys)]))
    stream = torch.cuda.current_stream().cuda_stream
    for xp, t, n_in, jobs in calls:
        sil.matmul_batch_noalloc_ptr(xp, t, n_in, jobs, stream)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for xp, t, n_in, jobs in calls:
            sil.matmul_batch_noalloc_ptr(xp, t, n_in, jobs, stream)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    sil.check_device_status()
    for weights, _, _ in keep:
        for w in weights:
            w.free()

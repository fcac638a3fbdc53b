"""Helpers for the GPU tests: run a batch through the C ABI, compare with the oracle."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as wl

GUARD = 64  # canary floats before and after every y buffer


def lib():
    import shared_input_linear_gb300 as sil
    sil.build()
    sil.load()
    return sil


def upload(sil, b: wl.BatchInputs):
    return [sil.upload_weight(f, buf, n, b.n_in) for f, buf, n in b.jobs]


def run(sil, b: wl.BatchInputs, weights=None, x=None, canary=float("nan"), stream=None):
    """Run one batch; returns (list of y numpy [t][n_out], guard regions intact?)."""
    import torch
    own = weights is None
    if own:
        weights = upload(sil, b)
    if x is None:
        x = torch.from_numpy(b.x).cuda()
    bufs, ys = [], []
    for (_, _, n) in b.jobs:
        full = torch.full((GUARD * 2 + b.t * n,), canary, device="cuda", dtype=torch.float32)
        bufs.append(full)
        ys.append(full[GUARD:GUARD + b.t * n].view(b.t, n))
    sil.matmul_batch(x, list(zip(weights, ys)), stream=stream)
    torch.cuda.synchronize()
    out, guards_ok = [], True
    for full, (_, _, n) in zip(bufs, b.jobs):
        h = full.cpu().numpy()
        g = np.concatenate([h[:GUARD], h[GUARD + b.t * n:]])
        guards_ok &= bool(np.all(np.isnan(g)) if np.isnan(canary) else np.all(g == canary))
        out.append(h[GUARD:GUARD + b.t * n].reshape(b.t, n).copy())
    if own:
        for w in weights:
            w.free()
    return out, guards_ok


def assert_parity(b: wl.BatchInputs, ys, what=""):
    for j, ((f, buf, n), y) in enumerate(zip(b.jobs, ys)):
        y_ref, mag = oracle.linear(f, buf, n, b.n_in, b.x)
        ok, worst, idx = oracle.check(y, y_ref, mag)
        assert ok, (f"{what} job {j} ({f}, t={b.t}, n_in={b.n_in}, n_out={n}): worst element "
                    f"{idx} is {worst:.3g} x tolerance (y={y.reshape(-1)[idx]!r}, "
                    f"ref={y_ref.reshape(-1)[idx]!r}, mag={mag.reshape(-1)[idx]!r})")


def assert_parity_sampled(b: wl.BatchInputs, ys, n_samples=256, seed=0, what=""):
    rng = np.random.default_rng(seed)
    for j, ((f, buf, n), y) in enumerate(zip(b.jobs, ys)):
        tok = rng.integers(0, b.t, size=n_samples)
        row = rng.integers(0, n, size=n_samples)
        # always include the corners and the ragged tail
        tok[:4] = [0, b.t - 1, 0, b.t - 1]
        row[:4] = [0, n - 1, n - 1, 0]
        y_ref, mag = oracle.linear_sampled(f, buf, n, b.n_in, b.x, tok, row)
        got = y[tok, row]
        ok, worst, idx = oracle.check(got, y_ref, mag)
        assert ok, (f"{what} job {j} ({f}, t={b.t}, n_in={b.n_in}, n_out={n}): sample "
                    f"(t={tok[idx]}, o={row[idx]}) is {worst:.3g} x tolerance")
        assert np.all(np.isfinite(y)), f"{what} job {j}: non-finite output (unwritten element?)"

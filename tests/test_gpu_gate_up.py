"""GPU parity of the fused gate+up job: h = gelu(x Wg^T) * (x Wu^T).

The pages run gate and up as one shared-input batch and pass both results to
gelu_mul (oxinfer 0.0.1, src/drafter.rs, `Drafter::step`).  The oracle computes
the two linear results in f64 and then gelu_mul in f64; the bar for h is the
bar of g and u carried through gelu(g) * u (``oracle.gate_up_tolerance``).
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import GUARD, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sil():
    import torch
    torch.cuda.set_device(0)
    return lib()


def _draw(fmt, n_in, n_out, t, seed, x_scale=1.0):
    """x, then the gate and up weights, from one seeded generator."""
    b = wl.make_batch(n_in, (n_out, n_out), t, fmt, seed=seed, x_scale=x_scale)
    return b.x, b.jobs[0][1], b.jobs[1][1]


def _run(sil, handles, x, t, widths, stream=None):
    """One batch; handles[j] writes widths[j] columns.  Returns ([h_j], guards intact)."""
    import torch
    xd = torch.from_numpy(x).cuda()
    bufs, outs = [], []
    for n in widths:
        full = torch.full((2 * GUARD + t * n,), float("nan"), device="cuda")
        bufs.append(full)
        outs.append(full[GUARD:GUARD + t * n].view(t, n))
    sil.matmul_batch(xd, list(zip(handles, outs)), stream=stream)
    torch.cuda.synchronize()
    res, ok = [], True
    for full, n in zip(bufs, widths):
        h = full.cpu().numpy()
        ok &= bool(np.all(np.isnan(np.concatenate([h[:GUARD], h[GUARD + t * n:]]))))
        res.append(h[GUARD:GUARD + t * n].reshape(t, n).copy())
    return res, ok


def _assert_gate_up(fmt, gate, up, n_out, n_in, x, h, what=""):
    h_ref, g, u, mg, mu = oracle.gate_up(fmt, gate, up, n_out, n_in, x)
    ok, worst, idx = oracle.check_gate_up(h, g, u, mg, mu)
    assert ok, (f"{what} ({fmt}, t={x.shape[0]}, n_in={n_in}, n_out={n_out}): element {idx} is "
                f"{worst:.3g} x tolerance (h={h.reshape(-1)[idx]!r}, ref={h_ref.reshape(-1)[idx]!r})")


SHAPES = [(256, 136), (1024, 1000), (2048, 256), (96, 7)]


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t", [1, 3, 8, 12, 24, 100])
@pytest.mark.parametrize("n_in,n_out", SHAPES)
def test_gate_up_parity(sil, fmt, t, n_in, n_out):
    # decode kernel (t <= 8, and Q8/Q4 up to 16), tensor-core kernel beyond, with
    # split K at the few-tile shapes; ragged widths leave partial row groups and tiles
    if fmt != "bf16" and n_in % 32:
        pytest.skip("Q8/Q4 need n_in % 32 == 0")
    x, gate, up = _draw(fmt, n_in, n_out, t, seed=n_in + 7 * t)
    w = sil.upload_gate_up(fmt, gate, up, n_out, n_in)
    (h,), guards = _run(sil, [w], x, t, [n_out])
    w.free()
    assert guards, "a kernel wrote outside h"
    _assert_gate_up(fmt, gate, up, n_out, n_in, x, h, "gate_up")


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
def test_gate_up_tensor_core_long_k(sil, fmt):
    # a fused job with long K over 22 row tiles of interleaved gate/up rows on the
    # tensor-core kernel, element-wise
    n_in, n_out, t = 8192, 1400, 17
    x, gate, up = _draw(fmt, n_in, n_out, t, seed=29)
    w = sil.upload_gate_up(fmt, gate, up, n_out, n_in)
    (h,), guards = _run(sil, [w], x, t, [n_out])
    w.free()
    assert guards, "a kernel wrote outside h"
    _assert_gate_up(fmt, gate, up, n_out, n_in, x, h, "gate_up long K")


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
def test_gate_up_dequant_interleaves_rows(sil, fmt):
    import torch
    n_in, n_out = 256, 40
    _, gate, up = _draw(fmt, n_in, n_out, 1, seed=3)
    w = sil.upload_gate_up(fmt, gate, up, n_out, n_in)
    out = torch.empty((2 * n_out, n_in), device="cuda")
    sil.dequantize_weight(w, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    dg = oracle.dequant(fmt, gate, n_out, n_in)
    du = oracle.dequant(fmt, up, n_out, n_in)
    assert np.array_equal(got[0::2].view(np.uint32), dg.view(np.uint32))
    assert np.array_equal(got[1::2].view(np.uint32), du.view(np.uint32))
    assert w.bytes == 2 * wl.weight_bytes(fmt, n_out, n_in)
    assert sil.is_gate_up(w) == 1
    w.free()


@pytest.mark.parametrize("t", [1, 5, 24])
def test_gate_up_with_plain_jobs_in_one_batch(sil, t):
    # a fused job next to plain jobs of every format over the same x
    n_in = 512
    x, gate, up = _draw("q8", n_in, 200, t, seed=30 + t)
    fused = sil.upload_gate_up("q8", gate, up, 200, n_in)
    plain = [wl.make_batch(n_in, (n,), 1, f, seed=40 + i).jobs[0] for i, (f, n) in
             enumerate((("bf16", 96), ("q4", 64), ("q8", 33)))]
    pw = [sil.upload_weight(f, buf, n, n_in) for f, buf, n in plain]
    hs, guards = _run(sil, [fused] + pw, x, t, [200] + [n for _, _, n in plain])
    assert guards
    _assert_gate_up("q8", gate, up, 200, n_in, x, hs[0], "fused next to plain jobs")
    for (f, buf, n), y in zip(plain, hs[1:]):
        y_ref, mag = oracle.linear(f, buf, n, n_in, x)
        assert oracle.check(y, y_ref, mag)[0], f
    fused.free()
    for w in pw:
        w.free()


def test_gate_up_equals_separate_jobs(sil):
    # the fused job against gate and up run as plain jobs of one batch, then
    # gelu_mul of those results: the two must agree within the bar
    n_in, n_out, t = 1024, 300, 4
    x, gate, up = _draw("bf16", n_in, n_out, t, seed=5)
    fused = sil.upload_gate_up("bf16", gate, up, n_out, n_in)
    wg = sil.upload_weight("bf16", gate, n_out, n_in)
    wu = sil.upload_weight("bf16", up, n_out, n_in)
    (h,), _ = _run(sil, [fused], x, t, [n_out])
    (g, u), _ = _run(sil, [wg, wu], x, t, [n_out, n_out])
    _, _, _, mg, mu = oracle.gate_up("bf16", gate, up, n_out, n_in, x)
    ok, worst, idx = oracle.check_gate_up(h, g, u, mg, mu)
    assert ok, (worst, idx)
    for w in (fused, wg, wu):
        w.free()


def test_gate_up_noalloc(sil):
    # the allocation-free entry point takes the fused job too (decode and tensor-core paths)
    import torch
    n_in, n_out = 512, 136
    for fmt, t in (("bf16", 3), ("bf16", 40), ("q4", 20)):
        x, gate, up = _draw(fmt, n_in, n_out, t, seed=60 + t)
        w = sil.upload_gate_up(fmt, gate, up, n_out, n_in)
        xd = torch.from_numpy(x).cuda()
        h = torch.full((t, n_out), float("nan"), device="cuda")
        sil.matmul_batch_noalloc_ptr(xd.data_ptr(), t, n_in, [(w, n_out, h.data_ptr())],
                                     torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        _assert_gate_up(fmt, gate, up, n_out, n_in, x, h.cpu().numpy(), "noalloc")
        w.free()


def test_gate_up_extreme_inputs(sil):
    # large gate results (gelu(g) ~ g, or ~0 for g << 0), tiny and zero tokens
    n_in, n_out, t = 256, 64, 8
    for fmt in ("bf16", "q8", "q4"):
        x, gate, up = _draw(fmt, n_in, n_out, t, seed=70)
        scales = np.array([1e3, 1.0, 1e-3, 0.0, 30.0, 1e-20, 3e5, 0.1])
        x = (x * scales[:, None]).astype(np.float32)
        w = sil.upload_gate_up(fmt, gate, up, n_out, n_in)
        (h,), guards = _run(sil, [w], x, t, [n_out])
        w.free()
        assert guards and np.all(np.isfinite(h))
        _assert_gate_up(fmt, gate, up, n_out, n_in, x, h, "extreme")


FULL = [(fmt, t) for fmt in wl.GATE_UP_FUSED.fmts for t in wl.GATE_UP_FUSED.ts]


@pytest.mark.parametrize("fmt,t", FULL)
def test_gate_up_full_size_sampled(sil, fmt, t):
    # the benchmark's fused gate+up workload (n_in 4096 -> 12288 + 12288), checked on
    # sampled elements that the oracle computes one by one
    bt = wl.GATE_UP_FUSED.batches[0]
    b = wl.make_workload_batch(wl.GATE_UP_FUSED, bt, t, fmt)
    n_in, n_out = bt.n_in, bt.n_outs[0]
    gate, up = b.jobs[0][1], b.jobs[1][1]
    w = sil.upload_gate_up(fmt, gate, up, n_out, n_in)
    (h,), guards = _run(sil, [w], b.x, t, [n_out])
    w.free()
    assert guards
    rng = np.random.default_rng(t)
    tok = rng.integers(0, t, 256)
    row = rng.integers(0, n_out, 256)
    tok[:2], row[:2] = t - 1, n_out - 1
    g, mg = oracle.linear_sampled(fmt, gate, n_out, n_in, b.x, tok, row)
    u, mu = oracle.linear_sampled(fmt, up, n_out, n_in, b.x, tok, row)
    ok, worst, idx = oracle.check_gate_up(h[tok, row], g, u, mg, mu)
    assert ok, (worst, idx)


def test_gate_up_rejects(sil):
    q8 = wl.make_batch(64, (4,), 1, "q8").jobs[0][1]
    for args, code in [((7, q8, q8, 4, 64), -3),
                       (("q8", q8, q8, 4, 48), -2),
                       (("q8", q8, q8, 0, 64), -2),
                       (("q8", q8, q8, 2 ** 30, 64), -2)]:
        with pytest.raises(sil.ILError) as ei:
            sil.upload_gate_up(*args)
        assert ei.value.code == code, args
    lib_ = sil.load()
    assert lib_.il_upload_gate_up(1, q8.ctypes.data, None, 4, 64) is None
    assert lib_.il_last_status() == -1
    assert sil.is_gate_up(0) == -1
    # a job must give the width of h as n_out (not the 2*n_out packed rows)
    import torch
    w = sil.upload_gate_up("q8", q8, q8, 4, 64)
    x = torch.zeros(1, 64, device="cuda")
    y = torch.zeros(1, 8, device="cuda")
    with pytest.raises(sil.ILError) as ei:
        sil.matmul_batch_ptr(x.data_ptr(), 1, 64, [(w, 8, y.data_ptr())], 0)
    assert ei.value.code == -2
    w.free()

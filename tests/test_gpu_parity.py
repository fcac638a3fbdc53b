"""GPU parity: the C-ABI path against the CPU oracle, element by element.

Bar (per element): |y - y_ref| <= 8e-3 * sum_i |x_i w_i| + 1e-6; dequantised
weights bit-exact; one-hot and integer-valued cases exact.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import GUARD, assert_parity, assert_parity_sampled, lib, run, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sil():
    import torch
    torch.cuda.set_device(0)
    return lib()


# ---------------------------------------------------------------------------
# small and ragged shapes: the oracle computes every element
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("t", [1, 4])
def test_tiny_workload(sil, t):
    b = wl.make_workload_batch(wl.TINY, wl.TINY.batches[0], t, "bf16")
    ys, guards = run(sil, b)
    assert guards
    assert_parity(b, ys, "tiny")


SHAPES = [  # (n_in, n_outs) -- several tiles, ragged row tails, ragged K for the 128 padding
    (32, (1, 7)),
    (96, (129, 8, 3)),
    (256, (1000,)),
    (1056, (40, 17)),
    (4128, (264, 9)),
]


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("n_in,n_outs", SHAPES)
def test_small_shapes(sil, fmt, t, n_in, n_outs):
    b = wl.make_batch(n_in, n_outs, t, fmt, seed=n_in + t)
    ys, guards = run(sil, b)
    assert guards, "a kernel wrote outside y"
    assert_parity(b, ys, "small")


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t", [1, 3, 8])
@pytest.mark.parametrize("n_in,n_outs", [(512, (1217, 7)), (1024, (2400, 130, 64)),
                                         (256, (9000,)), (4096, (1000, 24))])
def test_uneven_row_blocks(sil, fmt, t, n_in, n_outs):
    # more row groups than SMs and not a multiple of the row block: partial row
    # blocks, K split over clusters, and job boundaries inside row blocks
    b = wl.make_batch(n_in, n_outs, t, fmt, seed=n_in * 7 + t)
    ys, guards = run(sil, b)
    assert guards
    assert_parity(b, ys, "cut groups")


@pytest.mark.parametrize("fmt", ["bf16", "q4"])
def test_repeatable_bits(sil, fmt):
    # partial sums over K slices are combined in a fixed order: repeated calls give identical bits
    b = wl.make_batch(2048, (3000, 1000), 5, fmt, seed=99)
    ws = upload(sil, b)
    first, _ = run(sil, b, weights=ws)
    for _ in range(3):
        again, _ = run(sil, b, weights=ws)
        for y0, y1 in zip(first, again):
            assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))
    for w in ws:
        w.free()


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t", [9, 16, 17, 64, 129])
def test_many_tokens(sil, fmt, t):
    b = wl.make_batch(256, (136, 72, 5), t, fmt, seed=t)
    ys, guards = run(sil, b)
    assert guards
    assert_parity(b, ys, "many tokens")


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t,n_in,n_outs", [(17, 96, (1000, 136, 8)), (100, 1056, (300, 7)),
                                           (300, 4128, (264,)), (64, 8192, (200,)),
                                           (40, 12288, (128, 72))])
def test_tensor_core_shapes(sil, fmt, t, n_in, n_outs):
    # the tensor-core kernel (t >= 17 for every format; Q8/Q4 dequantised in shared
    # memory): padded K, ragged row tiles, several jobs, split K at the few-tile shapes
    b = wl.make_batch(n_in, n_outs, t, fmt, seed=n_in + t)
    ys, guards = run(sil, b)
    assert guards
    assert_parity(b, ys, "tensor-core shapes")


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t,n_in,n_outs", [(17, 8192, (1500, 1100)), (260, 4096, (2600,))])
def test_tensor_core_long_k(sil, fmt, t, n_in, n_outs):
    # long K over many row tiles, element-wise: t = 17 on 128-token tiles (t fits
    # one), t = 260 on two or three token tiles with a ragged last one
    b = wl.make_batch(n_in, n_outs, t, fmt, seed=t + len(n_outs))
    ys, guards = run(sil, b)
    assert guards
    assert_parity(b, ys, "long K")


def test_split_k_growing_tile_counts(sil):
    # consecutive tensor-core batches on one stream whose tile counts grow (split K as
    # CTA pairs at the few-tile ones): the per-tile arrival counters of split tiles
    # must start at zero every time (IL_TEST_SPLIT_WORKSPACE covers that form)
    import torch
    s = torch.cuda.Stream()
    for fmt, t, n_in, n_out in (("bf16", 300, 4096, 128), ("q4", 600, 4096, 1024), ("bf16", 1000, 4096, 4096),
                                ("q8", 700, 12288, 2048), ("bf16", 64, 8192, 256)):
        b = wl.make_batch(n_in, (n_out,), t, fmt, seed=t)
        with torch.cuda.stream(s):
            ys, guards = run(sil, b, stream=s)
        assert guards
        assert_parity_sampled(b, ys, n_samples=128, what=f"{fmt} t={t} n_out={n_out}")


def test_decode_back_to_back_launches(sil):
    # Q8/Q4 decode launches of varied size and K split queued on one stream without a
    # sync in between (each may start behind the previous one): the per-tile counters
    # of split tiles are back at zero for every launch, and every output is written
    import torch
    s = torch.cuda.Stream()
    cases = []
    for fmt, t, n_in, n_out in (("q8", 1, 4096, 24576), ("q4", 3, 4096, 24576), ("q8", 8, 2560, 40000),
                                ("q4", 1, 2560, 65536), ("q8", 5, 4096, 24576), ("q4", 8, 12288, 8192)):
        b = wl.make_batch(n_in, (n_out,), t, fmt, seed=t + n_out)
        w = upload(sil, b)
        x = torch.from_numpy(b.x).cuda()
        ys = [torch.full((t, n_out), float("nan"), device="cuda") for _ in range(2)]
        cases.append((b, w, x, ys))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for rep in range(2):
            for b, w, x, ys in cases:
                sil.matmul_batch(x, [(w[0], ys[rep])], stream=s)
    torch.cuda.synchronize()
    for b, w, x, ys in cases:
        for y in ys:
            # every output written (a tile no warp took would keep its NaNs), then sampled parity
            assert not bool(torch.isnan(y).any()), f"{b.fmt} t={b.t}: outputs left unwritten"
            assert_parity_sampled(b, [y.cpu().numpy()], n_samples=256, what=f"{b.fmt} t={b.t}")
        for wi in w:
            wi.free()


def test_bf16_odd_k(sil):
    # bf16 allows any n_in that is a multiple of 8
    for n_in in (8, 40, 264):
        b = wl.make_batch(n_in, (33, 16), 3, "bf16", seed=n_in)
        ys, guards = run(sil, b)
        assert guards
        assert_parity(b, ys, "odd k")


def test_mixed_formats_one_batch(sil):
    import torch
    n_in, t = 512, 4
    b16 = wl.make_batch(n_in, (100,), t, "bf16", seed=1)
    b8 = wl.make_batch(n_in, (64,), t, "q8", seed=1)
    b4 = wl.make_batch(n_in, (48,), t, "q4", seed=1)
    b = wl.BatchInputs("mixed", t, n_in, b16.x, b16.jobs + b8.jobs + b4.jobs)
    ys, guards = run(sil, b)
    assert guards
    assert_parity(b, ys, "mixed")


# ---------------------------------------------------------------------------
# exact cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
def test_dequant_bit_exact(sil, fmt):
    import torch
    for n_out, n_in in ((13, 160), (256, 4096)):
        b = wl.make_batch(n_in, (n_out,), 1, fmt, seed=7)
        _, buf, _ = b.jobs[0]
        w = sil.upload_weight(fmt, buf, n_out, n_in)
        out = torch.full((n_out, n_in), float("nan"), device="cuda")
        sil.dequantize_weight(w, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        ref = oracle.dequant(fmt, buf, n_out, n_in)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), fmt
        w.free()


@pytest.mark.parametrize("fmt", ["q8", "q4"])
def test_dequant_special_scales(sil, fmt):
    import torch
    # zero, subnormal, negative and huge scales must decode bit-exactly
    n_out, n_in = 8, 192
    rng = np.random.default_rng(5)
    qmax = 127 if fmt == "q8" else 7
    q = rng.integers(-qmax - 1, qmax + 1, size=(n_out, n_in))
    d = np.array([0.0, 2.0 ** -130, -3.5, 1e30, 2.0 ** -149, 0.02 / 127] * 8,
                 dtype=np.float32)[:n_out * (n_in // 32)].reshape(n_out, n_in // 32)
    buf = wl.encode_q8(q, d) if fmt == "q8" else wl.encode_q4(q, d)
    w = sil.upload_weight(fmt, buf, n_out, n_in)
    out = torch.empty((n_out, n_in), device="cuda")
    sil.dequantize_weight(w, out)
    torch.cuda.synchronize()
    ref = oracle.dequant(fmt, buf, n_out, n_in)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    w.free()


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t_total", [8, 24])
def test_one_hot_exact(sil, fmt, t_total):
    # x rows are unit vectors: y[t] must equal column k_t of the dequantised weight exactly
    n_out, n_in = 200, 1024 if fmt != "bf16" else 1000
    b = wl.make_batch(n_in, (n_out, 24), 1, fmt, seed=3)
    ks = np.linspace(0, n_in - 1, t_total).astype(int)
    x = np.zeros((t_total, n_in), dtype=np.float32)
    x[np.arange(t_total), ks] = 1.0
    bb = wl.BatchInputs(fmt, t_total, n_in, x, b.jobs)
    ys, _ = run(sil, bb)
    for (f, buf, n), y in zip(b.jobs, ys):
        deq = oracle.dequant(f, buf, n, n_in)
        if f != "bf16" and t_total >= 17:
            # tensor-core path for Q8/Q4: the weight enters as bf16(fp32(d*q)), round to nearest even
            import torch
            deq = torch.from_numpy(deq).to(torch.bfloat16).float().numpy()
        assert np.array_equal(y, deq[:, ks].T.astype(np.float32)), f


TOKEN_SCALES = (1e36, 1.0, 1e-30, 0.0, 1e-42, 3e-5, 2e20, 1e-12)


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t", [4, 8, 24])
def test_extreme_token_magnitudes(sil, fmt, t):
    # tokens of one batch whose magnitudes differ by up to 10^78 (plus an all-zero token
    # and a subnormal one): each token must meet the bar on its own, so no token's
    # precision may depend on the others' range
    n_in, n_outs = 512, (136, 40)
    b = wl.make_batch(n_in, n_outs, t, fmt, seed=21)
    scales = np.array([TOKEN_SCALES[i % len(TOKEN_SCALES)] for i in range(t)], dtype=np.float64)
    x = (b.x.astype(np.float64) * scales[:, None]).astype(np.float32)
    bb = wl.BatchInputs(fmt, t, n_in, x, b.jobs)
    ys, guards = run(sil, bb)
    assert guards
    for y in ys:
        assert np.all(np.isfinite(y))
    assert_parity(bb, ys, "extreme tokens")


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t", [1, 8, 40])
def test_integer_exact(sil, fmt, t):
    # integer weights (scale 1) and small integer x: every partial sum is an exact integer
    rng = np.random.default_rng(t)
    n_in, n_outs = 512, (77, 8)
    x = rng.integers(-4, 5, size=(t, n_in)).astype(np.float32)
    jobs = []
    for n in n_outs:
        if fmt == "bf16":
            import torch
            wint = rng.integers(-8, 9, size=(n, n_in)).astype(np.float32)
            jobs.append((fmt, wl.encode_bf16(wl.bf16_bits(torch.from_numpy(wint))), n))
        else:
            lo, hi = (-128, 128) if fmt == "q8" else (-8, 8)
            q = rng.integers(lo, hi, size=(n, n_in))
            d = np.ones((n, n_in // 32), dtype=np.float32)
            jobs.append((fmt, wl.encode_q8(q, d) if fmt == "q8" else wl.encode_q4(q, d), n))
    b = wl.BatchInputs(fmt, t, n_in, x, jobs)
    ys, _ = run(sil, b)
    for (f, buf, n), y in zip(jobs, ys):
        y_ref, _ = oracle.linear(f, buf, n, n_in, x)
        assert np.array_equal(y.astype(np.float64), y_ref), f


def test_identity_bf16(sil):
    import torch
    n = 256
    eye = wl.encode_bf16(wl.bf16_bits(torch.eye(n)))
    for t in (1, 8):
        x = wl.make_x(t, n, seed=2)
        b = wl.BatchInputs("bf16", t, n, x, [("bf16", eye, n)])
        ys, _ = run(sil, b)
        # the decode path keeps x to ~16 bits: exact for W = I up to that split
        assert np.all(np.abs(ys[0] - x) <= np.abs(x) * 2.0 ** -16)


# ---------------------------------------------------------------------------
# structural invariants
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", ["bf16", "q4"])
@pytest.mark.parametrize("t", [1, 8, 33])
def test_job_permutation(sil, fmt, t):
    b = wl.make_batch(1024, (300, 64, 500), t, fmt, seed=11)
    ws = upload(sil, b)
    ys, _ = run(sil, b, weights=ws)
    perm = [2, 0, 1]
    bp = wl.BatchInputs(fmt, t, b.n_in, b.x, [b.jobs[i] for i in perm])
    ysp, _ = run(sil, bp, weights=[ws[i] for i in perm])
    for k, i in enumerate(perm):
        assert np.array_equal(ysp[k], ys[i])
    for w in ws:
        w.free()


@pytest.mark.parametrize("fmt", ["bf16", "q8"])
@pytest.mark.parametrize("t", [4, 20])
def test_batch_equals_single_jobs(sil, fmt, t):
    b = wl.make_batch(2048, (1024, 256), t, fmt, seed=12)
    ws = upload(sil, b)
    ys, _ = run(sil, b, weights=ws)
    for j, w in enumerate(ws):
        bj = wl.BatchInputs(fmt, t, b.n_in, b.x, [b.jobs[j]])
        yj, _ = run(sil, bj, weights=[w])
        f, buf, n = b.jobs[j]
        _, mag = oracle.linear(f, buf, n, b.n_in, b.x)
        # same arithmetic up to the split of K over cluster ranks
        assert np.all(np.abs(yj[0] - ys[j]) <= 1e-5 * mag + 1e-7)
    for w in ws:
        w.free()


@pytest.mark.parametrize("t", [4, 12])
def test_row_locality(sil, t):
    import torch
    b = wl.make_batch(1024, (256, 40), t, "q8", seed=13)
    ws = upload(sil, b)
    ys, _ = run(sil, b, weights=ws)
    x2 = b.x.copy()
    x2[1] *= -3.0
    b2 = wl.BatchInputs("q8", t, b.n_in, x2, b.jobs)
    ys2, _ = run(sil, b2, weights=ws)
    for y, y2 in zip(ys, ys2):
        keep = [i for i in range(t) if i != 1]
        assert np.array_equal(y[keep], y2[keep])
        assert not np.array_equal(y[1], y2[1])
    for w in ws:
        w.free()


def test_linearity(sil):
    b = wl.make_batch(768, (96,), 5, "q4", seed=14)
    ws = upload(sil, b)
    x1 = b.x
    x2 = wl.make_x(5, 768, seed=15)
    a = np.float32(0.75)
    ya, _ = run(sil, wl.BatchInputs("q4", 5, 768, (a * x1 + x2).astype(np.float32), b.jobs), weights=ws)
    y1, _ = run(sil, wl.BatchInputs("q4", 5, 768, x1, b.jobs), weights=ws)
    y2, _ = run(sil, wl.BatchInputs("q4", 5, 768, x2, b.jobs), weights=ws)
    _, mag1 = oracle.linear("q4", b.jobs[0][1], 96, 768, np.abs(x1))
    _, mag2 = oracle.linear("q4", b.jobs[0][1], 96, 768, np.abs(x2))
    tol = 2 * (8e-3 * (a * mag1 + mag2) + 1e-6)
    assert np.all(np.abs(ya[0] - (a * y1[0] + y2[0])) <= tol)
    for w in ws:
        w.free()


def test_alternating_launch_configurations(sil):
    # the same kernel variant launched with shrinking and growing shared-memory slices
    for n_in, n_outs in ((4096, (4096, 1024)), (256, (512, 256)), (4096, (4096, 1024)),
                         (12288, (512,)), (256, (64,)), (12288, (512,))):
        b = wl.make_batch(n_in, n_outs, 1, "bf16", seed=n_in)
        ys, guards = run(sil, b)
        assert guards
        assert_parity_sampled(b, ys, n_samples=64, what=f"n_in={n_in}")


def test_stream_ordering(sil):
    # work queued on a side stream completes in stream order and is correct
    import torch
    s = torch.cuda.Stream()
    b = wl.make_batch(512, (64, 64), 3, "bf16", seed=16)
    with torch.cuda.stream(s):
        ys, guards = run(sil, b, stream=s)
    assert guards
    assert_parity(b, ys, "side stream")


# ---------------------------------------------------------------------------
# full-size workloads (the benchmark's shapes and launch configuration)
# ---------------------------------------------------------------------------
FULL = [(w, bt, t, fmt) for w in (wl.DECODE_BF16, wl.DECODE_QUANT, wl.VOCAB, wl.PREFILL_BF16,
                                   wl.PREFILL_QUANT)
        for bt in w.batches for t in w.ts for fmt in w.fmts]


@pytest.mark.parametrize("w,bt,t,fmt", FULL,
                         ids=[f"{w.name}-{bt.name}-t{t}-{fmt}" for w, bt, t, fmt in FULL])
def test_full_size_sampled(sil, w, bt, t, fmt):
    b = wl.make_workload_batch(w, bt, t, fmt)
    ys, guards = run(sil, b)
    assert guards
    assert_parity_sampled(b, ys, what=f"{w.name}/{bt.name}")


# ---------------------------------------------------------------------------
# launch counts and size limits: batches that need more than one launch of a
# kernel, and the largest n_in
# ---------------------------------------------------------------------------
def _launches(sil, b):
    before = sil.get_stats()["launches"]
    ys, guards = run(sil, b)
    return ys, guards, sil.get_stats()["launches"] - before


def test_twelve_gemm_jobs_two_launches(sil):
    # 12 bf16 jobs at t = 64: one cast of x, then 8 + 4 jobs on the tensor-core kernel
    n_outs = tuple(40 + 24 * j for j in range(12))
    b = wl.make_batch(512, n_outs, 64, "bf16", seed=31)
    ys, guards, launches = _launches(sil, b)
    assert guards
    assert launches == 3
    assert_parity(b, ys, "12 GEMM jobs")


@pytest.mark.parametrize("fmt", ["q8", "q4"])
@pytest.mark.parametrize("t", [9, 12, 16])
def test_quant_decode_sixteen_tokens_one_launch(sil, fmt, t):
    # Q8/Q4 at 9 <= t <= 16: one decode launch streams each weight once for two
    # groups of 8 token columns; ragged rows and a K split over CTAs (n_in 12288)
    for n_in, n_outs in ((1024, (300, 72)), (12288, (136,))):
        b = wl.make_batch(n_in, n_outs, t, fmt, seed=t + n_in)
        ys, guards, launches = _launches(sil, b)
        assert guards
        assert launches == 1
        assert_parity(b, ys, f"{fmt} t={t}")


def test_forty_decode_jobs_two_launches(sil):
    # 40 bf16 jobs at t = 1: 32 + 8 jobs on the decode kernel
    n_outs = tuple(8 + 16 * (j % 7) for j in range(40))
    b = wl.make_batch(256, n_outs, 1, "bf16", seed=32)
    ys, guards, launches = _launches(sil, b)
    assert guards
    assert launches == 2
    assert_parity(b, ys, "40 decode jobs")


def test_mixed_quant_formats_tensor_core(sil):
    # one Q4 job and ten Q8 jobs at t = 24: one cast, 8 + 2 Q8 jobs and 1 Q4 job on the
    # tensor-core kernel (Q8/Q4 dequantised in shared memory)
    t, n_in = 24, 512
    b4 = wl.make_batch(n_in, (200,), t, "q4", seed=33)
    b8 = wl.make_batch(n_in, tuple(16 + 40 * j for j in range(10)), t, "q8", seed=34)
    b = wl.BatchInputs("mixed", t, n_in, b4.x, b4.jobs + b8.jobs)
    ys, guards, launches = _launches(sil, b)
    assert guards
    assert launches == 4
    assert_parity(b, ys, "Q4 + 10 Q8")


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("t", [1, 8, 40])
def test_largest_n_in(sil, fmt, t):
    # n_in = 32768, the documented limit: the decode kernel splits K over a cluster
    # of 8 CTAs, the tensor-core kernel walks 512 k-blocks
    b = wl.make_batch(32768, (72, 24), t, fmt, seed=35 + t)
    ys, guards = run(sil, b)
    assert guards
    assert_parity(b, ys, "n_in 32768")


def test_split_k_pair_and_workspace_forms(sil, monkeypatch):
    # tile counts that split K in two: as CTA pairs exchanging partial sums through
    # distributed shared memory, then (IL_TEST_SPLIT_WORKSPACE=1) through the global
    # workspace, the form taken when the pairs do not fit; both against the oracle,
    # and bitwise equal (both add the same two slices)
    outs = {}
    for form in ("0", "1"):
        monkeypatch.setenv("IL_TEST_SPLIT_WORKSPACE", form)
        for fmt, t, n_in, n_out in (("bf16", 40, 1024, 1000), ("q8", 300, 2048, 520), ("q4", 512, 12288, 4096)):
            b = wl.make_batch(n_in, (n_out,), t, fmt, seed=n_out + t)
            ys, guards = run(sil, b)
            assert guards
            assert_parity_sampled(b, ys, n_samples=128, what=f"{fmt} t={t} form={form}")
            outs.setdefault((fmt, t), []).append(ys[0])
    for k, v in outs.items():
        assert np.array_equal(v[0].view(np.uint32), v[1].view(np.uint32)), k

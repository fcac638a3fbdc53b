"""Pins for the CPU oracle against what the definitions and mathematics fix.

Nothing here compares the oracle with itself: every expected value comes from
a hand derivation, a closed form, an exhaustive enumeration checked against an
independent routine (torch / numpy IEEE single arithmetic), or brute force in
Python integers.  The last test plants mistakes in a copy of the oracle source
and checks that at least one pin catches each of them.

Definitions pinned (oxinfer 0.0.0, src/gpu.rs): struct ``Job``
``y[t][n_out] = x[t][n_in] * W^T``; enum ``WeightRef`` formats Bf16 / Q8 / Q4
and ``WeightRef::bytes``; Q8 = int8 with one fp32 scale per 32-block along
n_in, Q4 = two's-complement nibbles, low nibble first, one fp32 scale per
32-block, both dequantised as ``fp32(d * q)``.
"""
import math
import os
import shutil

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

SCALES = np.array([0.0, 1.0, 2.0 ** -130, 0.02 / 127, -3.5, 1e30, 7.0e-3, 2.0 ** -149],
                  dtype=np.float32)


def _bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def _same_values(a, b):
    """Equal as values (+0 == -0), NaN positions equal."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return bool(np.all((a == b) | (np.isnan(a) & np.isnan(b))))


# ---------------------------------------------------------------------------
# pins, written as functions of an oracle so they can also run on mutants
# ---------------------------------------------------------------------------
def pin_weight_bytes(orc):
    # WeightRef::bytes: bf16 is len*2; Q8 1 + 4/32 and Q4 1/2 + 4/32 bytes per element.
    for n_out, n_in in [(1, 32), (7, 64), (4096, 4096), (262144, 2560)]:
        n = n_out * n_in
        assert orc.weight_bytes("bf16", n_out, n_in) == 2 * n
        assert orc.weight_bytes("q8", n_out, n_in) * 8 == 9 * n
        assert orc.weight_bytes("q4", n_out, n_in) * 8 == 5 * n


def pin_bf16_exhaustive(orc):
    # Every u16 pattern widens exactly; the independent routine is torch's bf16 -> fp32.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    got = orc.dequant("bf16", wl.encode_bf16(bits), 256, 256)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(_bits(got)[~nan], _bits(ref)[~nan])
    # NaN payloads pass through as the plain bit shift.
    assert np.array_equal(_bits(got)[nan], bits.astype(np.uint32)[nan] << 16)


def pin_q8_exhaustive(orc):
    # q in [-128, 127] against IEEE single multiply d*q (numpy float32), bit for bit.
    q = np.arange(-128, 128, dtype=np.int16)
    for d in SCALES:
        qq = np.tile(q, (1, 1)).reshape(8, 32)                     # 8 rows x one block
        dd = np.full((8, 1), d, dtype=np.float32)
        got = orc.dequant("q8", wl.encode_q8(qq, dd), 8, 32)
        ref = np.float32(d) * qq.astype(np.float32)
        assert np.array_equal(_bits(got), _bits(ref)), f"d={d}"


def _nibble_ref(byte_vals):
    """Independent nibble decode: arithmetic shifts of int8 (sign extension)."""
    b = np.asarray(byte_vals, dtype=np.uint8)
    lo = (b << 4).astype(np.uint8).view(np.int8) >> 4              # low nibble, sign-extended
    hi = b.view(np.int8) >> 4                                       # high nibble, sign-extended
    out = np.empty(b.size * 2, dtype=np.int8)
    out[0::2] = lo
    out[1::2] = hi
    return out


def pin_q4_exhaustive(orc):
    # All 256 bytes x every scale: element 2k is the low nibble of byte k.
    allbytes = np.arange(256, dtype=np.uint8).reshape(8, 32)        # 8 rows x 64 elements
    qref = _nibble_ref(allbytes.reshape(-1)).reshape(8, 64).astype(np.float32)
    for d in SCALES:
        dd = np.full((8, 2), d, dtype=np.float32)
        buf = np.concatenate([allbytes.reshape(-1), dd.reshape(-1).view(np.uint8)])
        got = orc.dequant("q4", buf, 8, 64)
        ref = np.float32(d) * qref
        assert np.array_equal(_bits(got), _bits(ref)), f"d={d}"


def pin_block_scale_index(orc):
    # Each 32-block along n_in uses its own scale; rows use their own scales.
    n_out, n_in = 3, 128
    q = np.ones((n_out, n_in), dtype=np.int8)
    d = np.arange(1, n_out * 4 + 1, dtype=np.float32).reshape(n_out, 4)
    got = orc.dequant("q8", wl.encode_q8(q, d), n_out, n_in)
    assert np.array_equal(got, np.repeat(d, 32, axis=1))
    p = np.full((n_out, n_in), 1, dtype=np.int8)
    got4 = orc.dequant("q4", wl.encode_q4(p, d), n_out, n_in)
    assert np.array_equal(got4, np.repeat(d, 32, axis=1))


def pin_brute_force_small(orc):
    # Hand-written dot products (bf16 values exactly representable).
    W = np.array([[1.0, 2.0, -1.0], [0.5, -3.0, 4.0]], dtype=np.float32)
    x = np.array([[1.0, 1.0, 1.0], [2.0, 0.0, -1.0]], dtype=np.float32)
    y, mag = orc.linear("bf16", wl.encode_bf16(wl.bf16_bits(torch.from_numpy(W))), 2, 3, x)
    assert np.array_equal(y, [[2.0, 1.5], [3.0, -3.0]])
    assert np.array_equal(mag, [[4.0, 7.5], [3.0, 5.0]])
    # 3x5 with fractional x: y_o = sum_i x_i w_oi worked out by hand.
    W = np.array([[1, 0, 0, 0, 2], [0, -1, 0, 0.25, 0], [1, 1, 1, 1, 1]], dtype=np.float32)
    x = np.array([[0.5, 2.0, -4.0, 8.0, 1.5]], dtype=np.float32)
    y, mag = orc.linear("bf16", wl.encode_bf16(wl.bf16_bits(torch.from_numpy(W))), 3, 5, x)
    assert np.array_equal(y, [[0.5 + 3.0, -2.0 + 2.0, 0.5 + 2.0 - 4.0 + 8.0 + 1.5]])
    assert np.array_equal(mag, [[3.5, 4.0, 16.0]])


def pin_golden_files(orc):
    for name in ("q4_worked_example.txt", "q8_worked_example.txt"):
        g = _read_golden(os.path.join(GOLDEN, name))
        n_out, n_in = int(g["n_out"]), int(g["n_in"])
        x = np.ones((2, n_in), dtype=np.float32)
        x[1, n_in // 2:] = -1.0
        scales = np.array([[float(v) for v in g[f"row{r}_scales"].split()] for r in range(n_out)],
                          dtype=np.float32)
        if g["format"] == "q4":
            rows = [np.full(n_in // 2, int(g[f"row{r}_byte"], 16), dtype=np.uint8)
                    for r in range(n_out)]
            buf = np.concatenate([np.concatenate(rows), scales.reshape(-1).view(np.uint8)])
        else:
            rows = []
            for r in range(n_out):
                b = [int(v, 16) for v in g[f"row{r}_bytes"].split()]
                rows.append(np.repeat(np.array(b, dtype=np.uint8), 32))
            buf = np.concatenate([np.concatenate(rows), scales.reshape(-1).view(np.uint8)])
        y, mag = orc.linear(g["format"], buf, n_out, n_in, x)
        assert np.array_equal(y.reshape(-1), [float(v) for v in g["y"].split()]), name
        assert np.array_equal(mag.reshape(-1), [float(v) for v in g["mag"].split()]), name


def pin_identity(orc):
    # W = I (bf16): y = x exactly, mag = |x|.
    n = 256
    x = wl.make_x(3, n, seed=5)
    eye = wl.encode_bf16(wl.bf16_bits(torch.eye(n)))
    y, mag = orc.linear("bf16", eye, n, n, x)
    assert np.array_equal(y, x.astype(np.float64))
    assert np.array_equal(mag, np.abs(x).astype(np.float64))


def pin_one_hot(orc):
    # x = e_k picks column k of the dequantised weight exactly, in every format.
    n_out, n_in = 40, 96
    g = torch.Generator().manual_seed(11)
    w = torch.randn(n_out, n_in, generator=g) * 0.02
    for fmt in ("bf16", "q8", "q4"):
        buf = wl.encode_weight(fmt, w)
        deq = orc.dequant(fmt, buf, n_out, n_in)
        for k in (0, 1, 31, 32, 63, 95):
            x = np.zeros((1, n_in), dtype=np.float32)
            x[0, k] = 1.0
            y, mag = orc.linear(fmt, buf, n_out, n_in, x)
            assert _same_values(y[0], deq[:, k]), (fmt, k)
            assert _same_values(mag[0], np.abs(deq[:, k])), (fmt, k)


def pin_integer_exact(orc):
    # Integer weights (d = 1) and integer x: every partial sum is an exact integer,
    # so y equals the brute-force Python-integer sum.
    rng = np.random.default_rng(3)
    n_out, n_in, t = 9, 64, 3
    x = rng.integers(-4, 5, size=(t, n_in)).astype(np.float32)
    for fmt, lo, hi in (("q8", -128, 128), ("q4", -8, 8)):
        q = rng.integers(lo, hi, size=(n_out, n_in))
        d = np.ones((n_out, n_in // 32), dtype=np.float32)
        buf = wl.encode_q8(q, d) if fmt == "q8" else wl.encode_q4(q, d)
        y, mag = orc.linear(fmt, buf, n_out, n_in, x)
        xi = x.astype(np.int64)
        for tt in range(t):
            for o in range(n_out):
                assert y[tt, o] == sum(int(xi[tt, i]) * int(q[o, i]) for i in range(n_in))
                assert mag[tt, o] == sum(abs(int(xi[tt, i]) * int(q[o, i])) for i in range(n_in))
    # bf16 with integer W in [-8, 8]
    wint = rng.integers(-8, 9, size=(n_out, n_in)).astype(np.float32)
    y, _ = orc.linear("bf16", wl.encode_bf16(wl.bf16_bits(torch.from_numpy(wint))), n_out, n_in, x)
    assert np.array_equal(y, (x.astype(np.int64) @ wint.astype(np.int64).T).astype(np.float64))


def pin_library_crosscheck(orc):
    # torch float64 CPU matmul of x and the dequantised weight (dequant pinned above).
    for fmt, n_out, n_in, t in (("bf16", 64, 96, 5), ("q8", 70, 128, 4), ("q4", 33, 256, 7)):
        b = wl.make_batch(n_in, (n_out,), t, fmt, seed=21)
        _, buf, _ = b.jobs[0]
        y, mag = orc.linear(fmt, buf, n_out, n_in, b.x)
        W = torch.from_numpy(orc.dequant(fmt, buf, n_out, n_in)).double()
        X = torch.from_numpy(b.x).double()
        ref = (X @ W.T).numpy()
        refmag = (X.abs() @ W.abs().T).numpy()
        assert np.all(np.abs(y - ref) <= 1e-12 * refmag + 1e-300), fmt
        assert np.allclose(mag, refmag, rtol=1e-12, atol=0), fmt


def pin_sampled_matches_definition(orc):
    # A sampled element equals the plain sum over i for that (token, row).
    b = wl.make_batch(64, (50,), 6, "q4", seed=9)
    _, buf, _ = b.jobs[0]
    deq = orc.dequant("q4", buf, 50, 64).astype(np.float64)
    tok = np.array([0, 5, 3, 3])
    row = np.array([0, 49, 17, 18])
    y, mag = orc.linear_sampled("q4", buf, 50, 64, b.x, tok, row)
    for s in range(4):
        prods = b.x[tok[s]].astype(np.float64) * deq[row[s]]
        assert abs(y[s] - prods.sum()) <= 1e-15 * np.abs(prods).sum()
        assert abs(mag[s] - np.abs(prods).sum()) <= 1e-15 * np.abs(prods).sum()


# ---------------------------------------------------------------------------
# gelu_mul after the gate+up batch (oxinfer 0.0.1, src/drafter.rs, Drafter::step;
# gelu read as the tanh form of the Gemma family)
# ---------------------------------------------------------------------------
def _gelu_erf(v):
    # the exact GELU, v * Phi(v), through the C library's erf (an independent routine)
    return 0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0)))


def pin_gelu_against_erf(orc):
    # the tanh form stays within 5e-4 of the exact GELU everywhere (max gap ~4.7e-4);
    # a dropped cubic term (gap 0.033 at 2) or a wrong constant is far outside it
    for v in np.concatenate([np.linspace(-10.0, 10.0, 2001), [0.5, 1.0, 2.0, -1.0, -3.0]]):
        assert abs(orc.gelu(float(v)) - _gelu_erf(float(v))) <= 5e-4, v


def pin_gelu_identities(orc):
    # gelu(v) - gelu(-v) = v for the tanh form (tanh is odd); gelu(0) = 0;
    # gelu(v) -> v for large v and -> 0 for large negative v
    for v in (0.1, 0.7, 1.5, 3.0, 9.0):
        assert abs(orc.gelu(v) - orc.gelu(-v) - v) <= 1e-14 * max(1.0, v), v
    assert orc.gelu(0.0) == 0.0
    assert orc.gelu(40.0) == 40.0
    assert orc.gelu(-40.0) == 0.0
    assert orc.gelu(1.0) > orc.gelu(0.5) > 0.0 > orc.gelu(-0.5)


def pin_gelu_lipschitz(orc):
    # the tolerance of gate+up results assumes sup |gelu'| <= GELU_LIPSCHITZ; the
    # supremum (about 1.12899 near |v| = 1.4185) must also be close to the constant
    xs = np.linspace(-6.0, 6.0, 120001)
    gs = np.array([orc.gelu(float(v)) for v in xs])
    d = np.diff(gs) / np.diff(xs)
    assert np.max(np.abs(d)) <= oracle.GELU_LIPSCHITZ
    assert np.max(np.abs(d)) >= oracle.GELU_LIPSCHITZ - 0.002


def pin_gelu_mul_roles(orc):
    # h = gelu(g) * u: the activation goes on the gate, not on the up result
    g = np.array([1.0, -3.0, 2.0, 0.0])
    u = np.array([2.0, 0.5, -3.0, 7.0])
    h = orc.gelu_mul(g, u)
    for i in range(4):
        assert abs(h[i] - _gelu_erf(g[i]) * u[i]) <= 5e-4 * abs(u[i]) + 1e-15, i


def pin_gate_up_one_hot(orc):
    # x = e_k: g and u are column k of the dequantised gate and up weights exactly,
    # and h = gelu(g) * u
    n_out, n_in = 24, 64
    gen = torch.Generator().manual_seed(12)
    wg = torch.randn(n_out, n_in, generator=gen) * 0.5
    wu = torch.randn(n_out, n_in, generator=gen) * 0.5
    for fmt in ("bf16", "q8"):
        bg, bu = wl.encode_weight(fmt, wg), wl.encode_weight(fmt, wu)
        dg, du = orc.dequant(fmt, bg, n_out, n_in), orc.dequant(fmt, bu, n_out, n_in)
        for k in (0, 33, 63):
            x = np.zeros((1, n_in), dtype=np.float32)
            x[0, k] = 1.0
            h, g, u, _, _ = orc.gate_up(fmt, bg, bu, n_out, n_in, x)
            assert _same_values(g[0], dg[:, k]) and _same_values(u[0], du[:, k]), (fmt, k)
            ref = np.array([_gelu_erf(float(a)) * float(b) for a, b in zip(dg[:, k], du[:, k])])
            assert np.all(np.abs(h[0] - ref) <= 5e-4 * np.abs(du[:, k]) + 1e-15), (fmt, k)


# ---------------------------------------------------------------------------
# centroid-masked LM head (oxinfer 0.0.1, src/drafter.rs, end of Drafter::step)
# ---------------------------------------------------------------------------
def _rows_bf16(rows, h=8):
    w = np.zeros((len(rows), h), dtype=np.float32)
    for r, vals in enumerate(rows):
        w[r, :len(vals)] = vals
    return wl.encode_bf16(wl.bf16_bits(torch.from_numpy(w)))


def _head_example():
    # hand-built: x = (1, 2, 0, ...), so a row (a, b, ...) scores a + 2b
    x = np.zeros(8, dtype=np.float32)
    x[:2] = (1.0, 2.0)
    centroids = _rows_bf16([(1, 0), (0, 1), (3, 0), (1, 0)])       # logits 1, 2, 3, 1
    ordering = np.array([5, 1, 7, 0, 3, 6, 2, 4], dtype=np.uint32)   # c0 {5,1} c1 {7,0} c2 {3,6} c3 {2,4}
    embed = _rows_bf16([(0, 0), (-1, 0), (10, 0), (1, 1), (10, 0), (4, 0), (2, 0.5), (0, 1.5)])
    return x, centroids, embed, ordering


def pin_centroid_head_worked_example(orc):
    # logits 1, 2, 3, 1: rank c2, c1, then the tie c0 / c3 goes to the lower index
    x, cen, emb, order = _head_example()
    r = orc.centroid_head(cen, 4, emb, 8, 8, order, x, 3)
    assert list(r["cl"]) == [1.0, 2.0, 3.0, 1.0]
    assert list(r["sel"]) == [2, 1, 0]
    # clusters in rank order: c2 {3, 6}, c1 {7, 0}, c0 {5, 1}
    assert list(r["scores"]) == [3.0, 3.0, 3.0, 0.0, 4.0, -1.0]
    assert (r["position"], r["token"], r["score"]) == (4, 5, 4.0)
    # k = 2: the three tied 3s, the first (token 3 at rank 0, position 0) wins
    r = orc.centroid_head(cen, 4, emb, 8, 8, order, x, 2)
    assert list(r["sel"]) == [2, 1] and (r["position"], r["token"]) == (0, 3)
    # k = 4 reaches c3 {2, 4}, two tied 10s: the first, token 2
    r = orc.centroid_head(cen, 4, emb, 8, 8, order, x, 4)
    assert list(r["sel"]) == [2, 1, 0, 3] and (r["position"], r["token"], r["score"]) == (6, 2, 10.0)
    # top_k above the centroid count is clamped
    assert list(orc.centroid_head(cen, 4, emb, 8, 8, order, x, 9)["sel"]) == [2, 1, 0, 3]


def pin_centroid_head_nan_and_empty(orc):
    # a NaN centroid logit ranks below every number; NaN and -inf scores never win,
    # and with no winner the token is 0 (the scan starts from (-inf, 0))
    x, _, emb, order = _head_example()
    cen = _rows_bf16([(1, 0), (float("nan"), 0), (3, 0), (-5, 0)])   # logits 1, NaN, 3, -5
    r = orc.centroid_head(cen, 4, emb, 8, 8, order, x, 3)
    assert list(r["sel"]) == [2, 0, 3]
    assert orc.first_max(np.array([np.nan, -np.inf, np.nan])) == -1
    assert orc.first_max(np.array([np.nan, 2.0, np.nan, 2.0, 1.0])) == 1
    assert orc.first_max(np.array([-np.inf, -1e300])) == 1


def pin_centroid_head_against_library(orc):
    # random data with ties: the selection equals a lexicographic sort by (-logit,
    # index) from numpy, the scores a float64 matmul of the gathered rows, and the
    # winner numpy's argmax (which also returns the first maximum)
    rng = np.random.default_rng(4)
    n_cent, per, h = 16, 4, 24
    vocab = n_cent * per
    x = rng.integers(-3, 4, size=h).astype(np.float32)
    cw = rng.integers(-2, 3, size=(n_cent, h)).astype(np.float32)
    cw[5] = cw[3]                                   # a tie between two centroids
    ew = rng.integers(-2, 3, size=(vocab, h)).astype(np.float32)
    order = rng.permutation(vocab).astype(np.uint32)
    cen = wl.encode_bf16(wl.bf16_bits(torch.from_numpy(cw)))
    emb = wl.encode_bf16(wl.bf16_bits(torch.from_numpy(ew)))
    for k in (1, 5, 16):
        r = orc.centroid_head(cen, n_cent, emb, vocab, h, order, x, k)
        cl = cw.astype(np.float64) @ x.astype(np.float64)
        assert np.array_equal(r["cl"], cl)
        want = np.lexsort((np.arange(n_cent), -cl))[:k]
        assert list(r["sel"]) == list(want), k
        rows = order[(want[:, None] * per + np.arange(per)[None, :]).reshape(-1)]
        sc = ew[rows].astype(np.float64) @ x.astype(np.float64)
        assert np.array_equal(r["scores"], sc)
        pos = int(np.argmax(sc))
        assert r["position"] == pos and r["token"] == int(rows[pos])


ALL_PINS = [pin_weight_bytes, pin_bf16_exhaustive, pin_q8_exhaustive, pin_q4_exhaustive,
            pin_block_scale_index, pin_brute_force_small, pin_golden_files, pin_identity,
            pin_one_hot, pin_integer_exact, pin_library_crosscheck,
            pin_sampled_matches_definition, pin_gelu_against_erf, pin_gelu_identities,
            pin_gelu_lipschitz, pin_gelu_mul_roles, pin_gate_up_one_hot,
            pin_centroid_head_worked_example, pin_centroid_head_nan_and_empty,
            pin_centroid_head_against_library]


def _read_golden(path):
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split("=", 1)
            out[k.strip()] = v.strip()
    return out


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


# ---------------------------------------------------------------------------
# quantiser / encoding invariants (the input side that both paths read)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt,qmax", [("q8", 127), ("q4", 7)])
def test_quantise_roundtrip(orc, fmt, qmax):
    # quant(deq(q, d)) == q when each block holds a +-qmax element and d > 0 is normal.
    rng = np.random.default_rng(1)
    n_out, n_in = 16, 128
    q = rng.integers(-qmax, qmax + 1, size=(n_out, n_in))
    q[:, ::32] = qmax * rng.choice([-1, 1], size=(n_out, n_in // 32))
    d = rng.uniform(1e-4, 1e-1, size=(n_out, n_in // 32)).astype(np.float32)
    enc = wl.encode_q8 if fmt == "q8" else wl.encode_q4
    w = orc.dequant(fmt, enc(q, d), n_out, n_in)
    q2, d2 = wl.quantize(torch.from_numpy(w), qmax)
    assert np.array_equal(q2, q)
    assert np.allclose(d2, d, rtol=2 ** -22, atol=0)


@pytest.mark.parametrize("fmt,qmax", [("q8", 127), ("q4", 7)])
def test_quantise_error_bound(orc, fmt, qmax):
    # |w - deq(quant(w))| <= d/2 (1 + 2^-23) + one fp32 rounding of the product.
    g = torch.Generator().manual_seed(4)
    w = torch.randn(32, 256, generator=g) * 0.02
    buf = wl.encode_weight(fmt, w)
    deq = orc.dequant(fmt, buf, 32, 256).astype(np.float64)
    _, d = wl.quantize(w, qmax)
    dd = np.repeat(d.astype(np.float64), 32, axis=1)
    err = np.abs(w.double().numpy() - deq)
    assert np.all(err <= dd / 2 * (1 + 2 ** -23) + np.abs(deq) * 2 ** -24 + 1e-30)


def test_nibble_pack_identity():
    # Unpack every byte (independent arithmetic-shift decode), repack, get the byte back.
    allbytes = np.arange(256, dtype=np.uint8)
    q = _nibble_ref(allbytes).reshape(1, 512)
    assert np.array_equal(wl.pack_nibbles(q).reshape(-1), allbytes)


def test_weight_bytes_agree_with_workloads(orc):
    for fmt in ("bf16", "q8", "q4"):
        for n_out, n_in in [(3, 64), (4096, 12288)]:
            assert orc.weight_bytes(fmt, n_out, n_in) == wl.weight_bytes(fmt, n_out, n_in)


def test_check_rule():
    y_ref = np.array([1.0, 0.0, -2.0])
    mag = np.array([10.0, 0.0, 2.0])
    ok, _, _ = oracle.check([1.0 + 0.08, -0.0, -2.0 - 0.016], y_ref, mag)
    assert ok
    ok, _, worst = oracle.check([1.0 + 0.0801, 0.0, -2.0], y_ref, mag)
    assert not ok and worst == 0
    ok, _, _ = oracle.check([np.nan, 0.0, -2.0], y_ref, mag)
    assert not ok
    ok, _, _ = oracle.check([1.0, 2e-6, -2.0], y_ref, mag)
    assert not ok


def test_gate_up_check_rule():
    # the derived bound: g and u each off by their full tolerance still pass ...
    g = np.array([1.4, -2.0, 0.3])
    u = np.array([2.0, -1.0, 0.0])
    mag_g = np.array([5.0, 3.0, 1.0])
    mag_u = np.array([4.0, 2.0, 1.0])
    eg, eu = oracle.tolerance(mag_g), oracle.tolerance(mag_u)
    h_worst = oracle.gelu_mul(g + eg, u + eu)
    assert oracle.check_gate_up(h_worst, g, u, mag_g, mag_u)[0]
    # ... an error twice the allowance does not, nor does a NaN
    tol = oracle.gate_up_tolerance(g, u, mag_g, mag_u)
    ok, _, worst = oracle.check_gate_up(oracle.gelu_mul(g, u) + 2 * tol * np.array([0, 1, 0]), g, u, mag_g, mag_u)
    assert not ok and worst == 1
    assert not oracle.check_gate_up([np.nan, 0.0, 0.0], g, u, mag_g, mag_u)[0]


def test_gate_up_bound_holds_under_sampled_errors():
    # the derived bar is an upper bound: g and u moved anywhere inside their own bars
    # (corners included) never move gelu(g)*u by more than gate_up_tolerance
    rng = np.random.default_rng(7)
    g = np.concatenate([rng.normal(0, 3, 4000), [0.0, -1.4185, 1.4185, -30.0, 30.0]])
    u = rng.normal(0, 2, g.size)
    mag_g = np.abs(g) * rng.uniform(1.0, 5.0, g.size)
    mag_u = np.abs(u) * rng.uniform(1.0, 5.0, g.size)
    tol = oracle.gate_up_tolerance(g, u, mag_g, mag_u)
    h = oracle.gelu_mul(g, u)
    eg, eu = oracle.tolerance(mag_g), oracle.tolerance(mag_u)
    for sg, su in [(1, 1), (1, -1), (-1, 1), (-1, -1)] + [(None, None)] * 8:
        dg = eg * (sg if sg is not None else rng.uniform(-1, 1, g.size))
        du = eu * (su if su is not None else rng.uniform(-1, 1, g.size))
        assert np.all(np.abs(oracle.gelu_mul(g + dg, u + du) - h) <= tol)


def test_oracle_rejects_bad_format(orc):
    with pytest.raises((ValueError, KeyError)):
        orc.dequant(7, np.zeros(64, np.uint8), 1, 32)
    with pytest.raises(ValueError):
        orc.linear("q8", np.zeros(10, np.uint8), 1, 32, np.zeros((1, 32), np.float32))


# ---------------------------------------------------------------------------
# planted mistakes: each mutant of the oracle must fail at least one pin
# ---------------------------------------------------------------------------
MUTANTS = {
    "nibble_order_swapped": ("(byte & 0x0F) : (byte >> 4)", "(byte >> 4) : (byte & 0x0F)"),
    "nibble_unsigned": ("(v >= 8) ? v - 16 : v", "v"),
    "q8_unsigned": ("int q = (int)(int8_t)w[o * n_in + i];", "int q = (int)w[o * n_in + i];"),
    "scale_block_off_by_one": ("4 * (o * n_blocks + i / 32), 4);\n    int q",
                               "4 * (o * n_blocks + (i + 1) / 32 % n_blocks), 4);\n    int q"),
    "dropped_last_term": ("for (int64_t i = 0; i < n_in; ++i) {\n        double p",
                          "for (int64_t i = 0; i + 1 < n_in; ++i) {\n        double p"),
    "sign_flip": ("acc += p;\n        m += fabs(p);\n      }\n      y_ref",
                  "acc -= p;\n        m += fabs(p);\n      }\n      y_ref"),
    "transposed_weight": ("out[o * n_in + i] = weight_at(format, (const uint8_t*)w, n_out, n_in, o, i);",
                          "out[o * n_in + i] = weight_at(format, (const uint8_t*)w, n_out, n_in, i % n_out, o % n_in);"),
    "mag_signed": ("m += fabs(p);\n      }\n      y_ref", "m += p;\n      }\n      y_ref"),
    "bf16_low_half": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b;"),
    "scale_rounded_twice": ("return (float)((double)d * (double)q);",
                            "return (float)(double)(float)((double)(float)d * 1.0000001 * (double)q);"),
    "gelu_no_cubic": ("(g + 0.044715 * g * g * g)", "(g + 0.0 * g * g * g)"),
    "gelu_wrong_constant": ("sqrt(2.0 / pi)", "sqrt(pi / 2.0)"),
    "gelu_sign": ("0.5 * g * (1.0 + tanh(inner))", "0.5 * g * (1.0 - tanh(inner))"),
    "gelu_mul_roles_swapped": ("h[i] = oracle_gelu(g[i]) * u[i];", "h[i] = oracle_gelu(u[i]) * g[i];"),
    "centroid_tie_to_higher_index": ("  return a < b;\n}", "  return a > b;\n}"),
    "centroid_nan_first": ("if (na != nb) return nb;", "if (na != nb) return na;"),
    "first_max_takes_last": ("if (scores[p] > best) {", "if (scores[p] >= best) {"),
    "cluster_offset_wrong": ("ordering[sel[i] * per + j]", "ordering[sel[i] + j]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mut = tmp_path / f"oracle_{name}.c"
    mut.write_text(src.replace(old, new))
    so = oracle.compile_source(str(mut), str(tmp_path / f"lib_{name}.so"))
    orc = oracle.Oracle(so)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
        except ValueError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
    shutil.rmtree(tmp_path, ignore_errors=True)


@pytest.mark.parametrize("fmt", ["bf16", "q8", "q4"])
@pytest.mark.parametrize("threads", [1, 3, 8])
def test_threaded_leg_is_the_same_computation(orc, fmt, threads):
    # The timing leg splits each job's rows over host threads; every element must
    # come out bit for bit as in the single-threaded oracle (same dequantisation,
    # same summation order), including a row count that does not divide evenly.
    b = wl.make_batch(256, (37,), 3, fmt, seed=threads)
    f, buf, n = b.jobs[0]
    y1, m1 = orc.linear(f, buf, n, 256, b.x)
    y2, m2 = orc.linear_threads(f, buf, n, 256, b.x, threads)
    assert np.array_equal(y1, y2) and np.array_equal(m1, m2)

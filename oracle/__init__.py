"""Plain CPU oracle for the shared-input batched linear -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it; the C source (``oracle.c``) is compiled here with gcc.

What it computes follows oxinfer 0.0.0 ``src/gpu.rs``: struct ``Job`` (one
matmul of a batch, ``y[t][n_out] = x[t][n_in] * W^T``), ``Backend::matmul``
(all jobs share one ``x``, ``t`` and ``n_in``) and enum ``WeightRef`` (Bf16 /
Q8 / Q4 storage).  Dequantisation is exact (bf16 bit shift, ``fp32(d*q)`` for
Q8/Q4) and the dot products accumulate in f64 with ``i`` ascending.

The acceptance rule for a GPU result ``y`` is per element
``|y - y_ref| <= 8e-3 * mag + 1e-6`` with ``mag = sum_i |x_i * w_i|``.

A fused gate+up job (oxinfer 0.0.1 ``src/drafter.rs``, ``Drafter::step``: the
gate+up batch followed by ``gelu_mul``) is the two linear results followed by
``h = gelu(g) * u`` in f64, gelu in the tanh form; its bar (``gate_up_tolerance``)
propagates the bar of g and u through that product.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BF16, Q8, Q4 = 0, 1, 2
FORMATS = {"bf16": BF16, "q8": Q8, "q4": Q4}

REL_TOL = 8e-3
ABS_TOL = 1e-6

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def compile_source(src: str, out: str) -> str:
    """Compile one C source of the oracle into a shared library at ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *GCC_FLAGS, "-o", tmp, src, "-lm", "-lpthread"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (plain gcc, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


class Oracle:
    """ctypes view of one compiled copy of ``oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_weight_bytes.argtypes = [ctypes.c_int, i64, i64]
        lib.oracle_weight_bytes.restype = i64
        lib.oracle_dequant.argtypes = [ctypes.c_int, vp, i64, i64, vp]
        lib.oracle_dequant.restype = ctypes.c_int
        lib.oracle_linear.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, vp, vp]
        lib.oracle_linear.restype = ctypes.c_int
        lib.oracle_linear_threads.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, vp, ctypes.c_int]
        lib.oracle_linear_threads.restype = ctypes.c_int
        lib.oracle_linear_sampled.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, i64,
                                              vp, vp, vp, vp]
        lib.oracle_linear_sampled.restype = ctypes.c_int
        lib.oracle_gelu.argtypes = [ctypes.c_double]
        lib.oracle_gelu.restype = ctypes.c_double
        lib.oracle_gelu_mul.argtypes = [vp, vp, i64, vp]
        lib.oracle_gelu_mul.restype = None
        lib.oracle_centroid_select.argtypes = [vp, i64, i64, vp, i64, vp, vp]
        lib.oracle_centroid_select.restype = ctypes.c_int
        lib.oracle_cluster_scores.argtypes = [vp, i64, i64, vp, i64, vp, i64, vp, vp, vp]
        lib.oracle_cluster_scores.restype = ctypes.c_int
        lib.oracle_first_max.argtypes = [vp, i64]
        lib.oracle_first_max.restype = i64
        self.lib = lib

    def weight_bytes(self, fmt, n_out: int, n_in: int) -> int:
        """Bytes of one weight in the host layout (``WeightRef::bytes``)."""
        return int(self.lib.oracle_weight_bytes(_fmt(fmt), n_out, n_in))

    def _check_w(self, fmt, w: np.ndarray, n_out: int, n_in: int) -> np.ndarray:
        w = np.ascontiguousarray(w).view(np.uint8).reshape(-1)
        if w.size != self.weight_bytes(fmt, n_out, n_in):
            raise ValueError(f"weight buffer has {w.size} bytes, expected "
                             f"{self.weight_bytes(fmt, n_out, n_in)}")
        return w

    def dequant(self, fmt, w: np.ndarray, n_out: int, n_in: int) -> np.ndarray:
        """Every weight element as fp32, ``[n_out][n_in]``."""
        f = _fmt(fmt)
        w = self._check_w(f, w, n_out, n_in)
        out = np.empty((n_out, n_in), dtype=np.float32)
        rc = self.lib.oracle_dequant(f, _ptr(w), n_out, n_in, _ptr(out))
        if rc != 0:
            raise ValueError(f"oracle_dequant rejected the weight (code {rc})")
        return out

    def linear(self, fmt, w: np.ndarray, n_out: int, n_in: int, x: np.ndarray):
        """One job: returns ``(y_ref, mag)``, both f64 ``[t][n_out]``."""
        f = _fmt(fmt)
        w = self._check_w(f, w, n_out, n_in)
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim != 2 or x.shape[1] != n_in:
            raise ValueError("x must be [t][n_in] fp32")
        t = x.shape[0]
        y = np.empty((t, n_out), dtype=np.float64)
        mag = np.empty((t, n_out), dtype=np.float64)
        row = np.empty(n_in, dtype=np.float32)
        rc = self.lib.oracle_linear(f, _ptr(w), n_out, n_in, _ptr(x), t, _ptr(y), _ptr(mag),
                                    _ptr(row))
        if rc != 0:
            raise ValueError(f"oracle_linear rejected the weight (code {rc})")
        return y, mag

    def linear_threads(self, fmt, w: np.ndarray, n_out: int, n_in: int, x: np.ndarray, threads: int):
        """``linear`` with the rows split over ``threads`` host threads: the same
        arithmetic element by element, so the same results, in less wall time."""
        f = _fmt(fmt)
        w = self._check_w(f, w, n_out, n_in)
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim != 2 or x.shape[1] != n_in:
            raise ValueError("x must be [t][n_in] fp32")
        t = x.shape[0]
        y = np.empty((t, n_out), dtype=np.float64)
        mag = np.empty((t, n_out), dtype=np.float64)
        rc = self.lib.oracle_linear_threads(f, _ptr(w), n_out, n_in, _ptr(x), t, _ptr(y), _ptr(mag), int(threads))
        if rc != 0:
            raise ValueError(f"oracle_linear_threads failed (code {rc})")
        return y, mag

    def linear_sampled(self, fmt, w: np.ndarray, n_out: int, n_in: int, x: np.ndarray,
                       tok: np.ndarray, row: np.ndarray):
        """Selected outputs ``(tok[s], row[s])`` of one job: ``(y_ref, mag)`` f64 ``[S]``."""
        f = _fmt(fmt)
        w = self._check_w(f, w, n_out, n_in)
        x = np.ascontiguousarray(x, dtype=np.float32)
        tok = np.ascontiguousarray(tok, dtype=np.int64)
        row = np.ascontiguousarray(row, dtype=np.int64)
        if tok.shape != row.shape or tok.ndim != 1:
            raise ValueError("tok and row must be 1-D and the same length")
        y = np.empty(tok.size, dtype=np.float64)
        mag = np.empty(tok.size, dtype=np.float64)
        rc = self.lib.oracle_linear_sampled(f, _ptr(w), n_out, n_in, _ptr(x), x.shape[0],
                                            tok.size, _ptr(tok), _ptr(row), _ptr(y), _ptr(mag))
        if rc != 0:
            raise ValueError(f"oracle_linear_sampled failed (code {rc})")
        return y, mag


    def gelu(self, g: float) -> float:
        """gelu in the tanh form, in double."""
        return float(self.lib.oracle_gelu(float(g)))

    def gelu_mul(self, g: np.ndarray, u: np.ndarray) -> np.ndarray:
        """``gelu(g) * u`` elementwise, f64 (the drafter's ``gelu_mul(&mut g, &u)``)."""
        g = np.ascontiguousarray(g, dtype=np.float64)
        u = np.ascontiguousarray(u, dtype=np.float64)
        if g.shape != u.shape:
            raise ValueError("g and u must have one shape")
        h = np.empty_like(g)
        self.lib.oracle_gelu_mul(_ptr(g), _ptr(u), g.size, _ptr(h))
        return h

    def gate_up(self, fmt, gate: np.ndarray, up: np.ndarray, n_out: int, n_in: int, x: np.ndarray):
        """A gate+up job: the two linear results over one x, then ``gelu_mul``.

        Returns ``(h, g, u, mag_g, mag_u)``, all f64 ``[t][n_out]``.
        """
        g, mag_g = self.linear(fmt, gate, n_out, n_in, x)
        u, mag_u = self.linear(fmt, up, n_out, n_in, x)
        return self.gelu_mul(g, u), g, u, mag_g, mag_u


    # -- centroid-masked LM head (oxinfer 0.0.1, src/drafter.rs, end of Drafter::step)
    def centroid_select(self, centroids: np.ndarray, n_cent: int, h: int, x: np.ndarray, k: int):
        """Centroid logits (f64 ``[n_cent]``) and the ``k`` selected centroids in rank order."""
        c = self._check_w(BF16, centroids, n_cent, h)
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
        if x.size != h:
            raise ValueError("x must hold h values")
        cl = np.empty(n_cent, dtype=np.float64)
        sel = np.empty(k, dtype=np.int64)
        if self.lib.oracle_centroid_select(_ptr(c), n_cent, h, _ptr(x), k, _ptr(cl), _ptr(sel)) != 0:
            raise ValueError("oracle_centroid_select rejected its arguments")
        return cl, sel

    def cluster_scores(self, embed: np.ndarray, vocab: int, h: int, ordering: np.ndarray, per: int,
                       sel: np.ndarray, x: np.ndarray):
        """Exact logits (and ``mag``) of the tokens of the clusters ``sel``, (rank, position) order."""
        e = self._check_w(BF16, embed, vocab, h)
        ordering = np.ascontiguousarray(ordering, dtype=np.uint32)
        sel = np.ascontiguousarray(sel, dtype=np.int64)
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
        k = sel.size
        scores = np.empty(k * per, dtype=np.float64)
        mag = np.empty(k * per, dtype=np.float64)
        rc = self.lib.oracle_cluster_scores(_ptr(e), vocab, h, _ptr(ordering), per, _ptr(sel), k, _ptr(x),
                                            _ptr(scores), _ptr(mag))
        if rc != 0:
            raise ValueError("oracle_cluster_scores: an ordering entry is out of range")
        return scores, mag

    def first_max(self, scores: np.ndarray) -> int:
        """Position of the first strict maximum above -inf, or -1."""
        s = np.ascontiguousarray(scores, dtype=np.float64)
        return int(self.lib.oracle_first_max(_ptr(s), s.size))

    def centroid_head(self, centroids, n_cent, embed, vocab, h, ordering, x, top_k):
        """The whole head: returns a dict with cl, sel, scores, mag, position, token, score."""
        k = min(int(top_k), int(n_cent))
        per = vocab // n_cent
        cl, sel = self.centroid_select(centroids, n_cent, h, x, k)
        scores, mag = self.cluster_scores(embed, vocab, h, ordering, per, sel, x)
        pos = self.first_max(scores)
        ordering = np.asarray(ordering, dtype=np.uint32)
        token = 0 if pos < 0 else int(ordering[sel[pos // per] * per + pos % per])
        score = -np.inf if pos < 0 else float(scores[pos])
        return {"cl": cl, "sel": sel, "scores": scores, "mag": mag, "position": pos, "token": token,
                "score": score, "per": per}


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def default() -> Oracle:
    """The oracle compiled from ``oracle.c`` in this directory."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def weight_bytes(fmt, n_out: int, n_in: int) -> int:
    return default().weight_bytes(fmt, n_out, n_in)


def dequant(fmt, w, n_out: int, n_in: int) -> np.ndarray:
    return default().dequant(fmt, w, n_out, n_in)


def linear(fmt, w, n_out: int, n_in: int, x):
    return default().linear(fmt, w, n_out, n_in, x)


def linear_sampled(fmt, w, n_out: int, n_in: int, x, tok, row):
    return default().linear_sampled(fmt, w, n_out, n_in, x, tok, row)


def linear_threads(fmt, w, n_out: int, n_in: int, x, threads: int):
    return default().linear_threads(fmt, w, n_out, n_in, x, threads)


def matmul_batch(x: np.ndarray, jobs):
    """The batch: ``jobs`` is a list of ``(fmt, host_bytes, n_out)`` over one shared ``x``.

    Returns one ``(y_ref, mag)`` pair per job (oxinfer ``Backend::matmul``).
    """
    n_in = x.shape[1]
    return [linear(fmt, w, n_out, n_in, x) for fmt, w, n_out in jobs]


def centroid_head(centroids, n_cent, embed, vocab, h, ordering, x, top_k):
    return default().centroid_head(centroids, n_cent, embed, vocab, h, ordering, x, top_k)


def gelu_mul(g, u) -> np.ndarray:
    return default().gelu_mul(g, u)


def gate_up(fmt, gate, up, n_out: int, n_in: int, x):
    return default().gate_up(fmt, gate, up, n_out, n_in, x)


# sup |gelu'(g)| over all g for the tanh form (about 1.12899, at |g| ~ 1.4185)
GELU_LIPSCHITZ = 1.13
# relative error allowed for evaluating gelu(g) * u in fp32 on top of the input errors
GELU_EVAL_REL = 1e-5


def gate_up_tolerance(g, u, mag_g, mag_u) -> np.ndarray:
    """Allowed absolute error of ``h = gelu(g) * u`` when g and u each meet the bar.

    With |g^ - g| <= eg = tol(mag_g) and |u^ - u| <= eu = tol(mag_u):
    |gelu(g^) u^ - gelu(g) u| <= L eg (|u| + eu) + |gelu(g)| eu, L = sup |gelu'|,
    plus a relative allowance for the fp32 evaluation of the product.
    """
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    eg = tolerance(mag_g)
    eu = tolerance(mag_u)
    gl = np.abs(default().gelu_mul(g, np.ones_like(g)))
    prop = GELU_LIPSCHITZ * eg * (np.abs(u) + eu) + gl * eu
    return prop + GELU_EVAL_REL * (gl + GELU_LIPSCHITZ * eg) * (np.abs(u) + eu) + ABS_TOL


def check_gate_up(h, g, u, mag_g, mag_u) -> tuple[bool, float, int]:
    """Accept a gate+up result ``h`` against the oracle's (h_ref = gelu_mul(g, u))."""
    h = np.asarray(h, dtype=np.float64).reshape(-1)
    h_ref = default().gelu_mul(g, u).reshape(-1)
    tol = gate_up_tolerance(g, u, mag_g, mag_u).reshape(-1)
    if h.size == 0:
        return True, 0.0, -1
    err = np.abs(h - h_ref)
    err = np.where(np.isnan(err), np.inf, err)
    ratio = err / tol
    worst = int(np.argmax(ratio))
    return bool(np.all(err <= tol)), float(ratio[worst]), worst


def tolerance(mag: np.ndarray) -> np.ndarray:
    """Allowed absolute error per element."""
    return REL_TOL * np.asarray(mag, dtype=np.float64) + ABS_TOL


def check(y, y_ref, mag) -> tuple[bool, float, int]:
    """Accept ``y`` iff every element is within tolerance (f64 compare, +0 == -0).

    Returns ``(ok, worst ratio err/tol, index of the worst element)``.
    """
    y = np.asarray(y, dtype=np.float64).reshape(-1)
    y_ref = np.asarray(y_ref, dtype=np.float64).reshape(-1)
    tol = tolerance(mag).reshape(-1)
    if y.size == 0:
        return True, 0.0, -1
    err = np.abs(y - y_ref)
    err = np.where(np.isnan(err), np.inf, err)
    ratio = err / tol
    worst = int(np.argmax(ratio))
    return bool(np.all(err <= tol)), float(ratio[worst]), worst

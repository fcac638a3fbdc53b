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


GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def compile_source(src: str, out: str) -> str:
    """Compile one C source of the oracle into a shared library at ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *GCC_FLAGS, "-o", tmp, src, "-lm"])
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
        lib.oracle_linear_sampled.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, i64,
                                              vp, vp, vp, vp]
        lib.oracle_linear_sampled.restype = ctypes.c_int
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


def matmul_batch(x: np.ndarray, jobs):
    """The batch: ``jobs`` is a list of ``(fmt, host_bytes, n_out)`` over one shared ``x``.

    Returns one ``(y_ref, mag)`` pair per job (oxinfer ``Backend::matmul``).
    """
    n_in = x.shape[1]
    return [linear(fmt, w, n_out, n_in, x) for fmt, w, n_out in jobs]


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

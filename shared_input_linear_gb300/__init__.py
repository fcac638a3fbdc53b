"""Python binding of the ``il`` C ABI (``include/il.h``): argument marshalling only.

Every computation runs in ``libil.so``'s CUDA kernels.  There is no CPU
fallback: if the library is missing or no sm_103a device is current, the calls
raise :class:`ILError`.

The names follow the C ABI: :func:`upload_weight` (oxinfer ``Backend::upload``),
:func:`matmul_batch` (``Backend::matmul``: all jobs over one shared ``x``),
:func:`free_weight`, :func:`weight_bytes` (``WeightRef::bytes``),
:func:`dequantize_weight` (test hook), :func:`get_stats`.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

__all__ = ["ILError", "Weight", "FORMATS", "IL_BF16", "IL_Q8", "IL_Q4", "load", "build",
           "upload_weight", "matmul_batch", "matmul_batch_ptr", "matmul_batch_noalloc_ptr", "free_weight", "weight_bytes",
           "dequantize_weight", "check_device_status", "release_scratch", "get_stats", "reset_stats", "last_error",
           "version", "LIB_PATH", "STATUS"]

IL_BF16, IL_Q8, IL_Q4 = 0, 1, 2
FORMATS = {"bf16": IL_BF16, "q8": IL_Q8, "q4": IL_Q4}
STATUS = {0: "IL_OK", -1: "IL_ERR_ARG", -2: "IL_ERR_SHAPE", -3: "IL_ERR_FORMAT",
          -4: "IL_ERR_HANDLE", -5: "IL_ERR_OOM", -6: "IL_ERR_CUDA",
          -7: "IL_ERR_DEVICE_TIMEOUT", -8: "IL_ERR_UNSUPPORTED"}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libil.so")


class ILError(RuntimeError):
    """An ``il_*`` call failed; ``code`` is the negative ``il_status``."""

    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class _Job(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("n_out", ctypes.c_int64), ("y", ctypes.c_void_p)]


class _Stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("uploads", "upload_bytes", "batches", "jobs", "launches", "weight_bytes",
                 "flops", "errors", "profiled_batches", "device_ns")]


_lib = None
_lock = threading.Lock()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``libil.so`` in-tree with nvcc (sm_103a)."""
    from . import _build
    return _build.build(force=force, verbose=verbose)


def load() -> ctypes.CDLL:
    """Load ``libil.so``; raises :class:`ILError` when it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ILError(-8, f"{LIB_PATH} is missing: build it with "
                              "shared_input_linear_gb300.build() (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.il_upload_weight.argtypes = [ci, vp, i64, i64]
        lib.il_upload_weight.restype = vp
        lib.il_matmul_batch.argtypes = [vp, i64, i64, ctypes.POINTER(_Job), ci, vp]
        lib.il_matmul_batch.restype = ci
        lib.il_matmul_batch_noalloc.argtypes = [vp, i64, i64, ctypes.POINTER(_Job), ci, vp]
        lib.il_matmul_batch_noalloc.restype = ci
        lib.il_matmul_batch_host.argtypes = [vp, i64, i64, ctypes.POINTER(_Job), ci, vp]
        lib.il_matmul_batch_host.restype = ci
        lib.il_upload_gate_up.argtypes = [ci, vp, vp, i64, i64]
        lib.il_upload_gate_up.restype = vp
        lib.il_centroid_head.argtypes = [vp, i64, vp, vp, vp, i64, vp, vp, vp, vp, vp]
        lib.il_centroid_head.restype = ci
        lib.il_weight_is_gate_up.argtypes = [vp]
        lib.il_weight_is_gate_up.restype = ci
        lib.il_free_weight.argtypes = [vp]
        lib.il_free_weight.restype = None
        lib.il_weight_bytes.argtypes = [vp]
        lib.il_weight_bytes.restype = i64
        lib.il_weight_info.argtypes = [vp, ctypes.POINTER(ci), ctypes.POINTER(i64),
                                       ctypes.POINTER(i64)]
        lib.il_weight_info.restype = ci
        lib.il_dequantize_weight.argtypes = [vp, vp, vp]
        lib.il_dequantize_weight.restype = ci
        lib.il_check_device_status.argtypes = [vp]
        lib.il_check_device_status.restype = ci
        lib.il_release_scratch.argtypes = [vp]
        lib.il_release_scratch.restype = ci
        lib.il_last_error.argtypes = []
        lib.il_last_error.restype = ctypes.c_char_p
        lib.il_last_status.argtypes = []
        lib.il_last_status.restype = ci
        lib.il_get_stats.argtypes = [ctypes.POINTER(_Stats)]
        lib.il_get_stats.restype = ci
        lib.il_reset_stats.argtypes = []
        lib.il_reset_stats.restype = None
        lib.il_version.argtypes = []
        lib.il_version.restype = ci
        _lib = lib
        return lib


def last_error() -> str:
    return load().il_last_error().decode()


def _check(rc: int) -> int:
    if rc != 0:
        raise ILError(rc, last_error())
    return rc


def version() -> int:
    return load().il_version()


class Weight:
    """Owner of one device weight handle (freed on :meth:`free` or garbage collection)."""

    def __init__(self, handle: int, fmt: int, n_out: int, n_in: int, gate_up: bool = False):
        self.handle = handle
        self.fmt = fmt
        self.n_out = n_out      # columns of a job's output (the width of h for gate+up)
        self.n_in = n_in
        self.gate_up = gate_up

    @property
    def bytes(self) -> int:
        return weight_bytes(self)

    def free(self) -> None:
        if self.handle:
            load().il_free_weight(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def upload_weight(fmt, host, n_out: int, n_in: int) -> Weight:
    """``il_upload_weight``: ``host`` is a host buffer (numpy) in the documented layout."""
    buf = np.ascontiguousarray(host)
    lib = load()
    h = lib.il_upload_weight(_fmt(fmt), buf.ctypes.data, int(n_out), int(n_in))
    if not h:
        raise ILError(lib.il_last_status(), last_error())
    return Weight(h, _fmt(fmt), int(n_out), int(n_in))


def upload_gate_up(fmt, gate, up, n_out: int, n_in: int) -> Weight:
    """``il_upload_gate_up``: ``gate`` and ``up`` are host buffers of one shape in the
    layout of :func:`upload_weight`; a job of the result writes ``h = gelu(g) * u``,
    ``[t][n_out]``."""
    g = np.ascontiguousarray(gate)
    u = np.ascontiguousarray(up)
    lib = load()
    h = lib.il_upload_gate_up(_fmt(fmt), g.ctypes.data, u.ctypes.data, int(n_out), int(n_in))
    if not h:
        raise ILError(lib.il_last_status(), last_error())
    return Weight(h, _fmt(fmt), int(n_out), int(n_in), gate_up=True)


def is_gate_up(w) -> int:
    """``il_weight_is_gate_up``: 1, 0, or -1 for an invalid handle."""
    return int(load().il_weight_is_gate_up(w.handle if isinstance(w, Weight) else w))


def centroid_head(x, centroids: Weight, embed: Weight, ordering, top_k: int, token_out, score_out=None,
                  selected_out=None, scores_out=None, stream=None) -> None:
    """``il_centroid_head`` on torch CUDA tensors: ``x`` fp32 ``[h]``, ``ordering`` int32/uint32
    ``[vocab]``, ``token_out`` 32-bit ``[1]``; the optional outputs as documented in
    ``include/il.h``.  Enqueued on ``stream`` (default: the current torch stream)."""
    def ptr(t):
        return 0 if t is None else t.data_ptr()
    if not x.is_contiguous() or not ordering.is_contiguous():
        raise ILError(-1, "x and ordering must be contiguous")
    _check(load().il_centroid_head(ptr(x), int(x.numel()), centroids.handle, embed.handle, ptr(ordering),
                                   int(top_k), ptr(token_out), ptr(score_out), ptr(selected_out),
                                   ptr(scores_out), _stream_ptr(stream)))


def free_weight(w: Weight) -> None:
    w.free()


def weight_bytes(w: Weight) -> int:
    return int(load().il_weight_bytes(w.handle))


def _stream_ptr(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def matmul_batch_ptr(x_ptr: int, t: int, n_in: int, jobs, stream_ptr: int) -> int:
    """``il_matmul_batch`` on raw device pointers; ``jobs`` is ``[(Weight|handle, n_out, y_ptr)]``."""
    arr = (_Job * max(1, len(jobs)))()
    for i, (w, n_out, y) in enumerate(jobs):
        arr[i].w = w.handle if isinstance(w, Weight) else w
        arr[i].n_out = int(n_out)
        arr[i].y = int(y)
    return _check(load().il_matmul_batch(x_ptr, int(t), int(n_in), arr, len(jobs), stream_ptr))


def prepare_jobs(jobs):
    """A reusable ``il_job`` array for ``[(Weight|handle, n_out, y_ptr)]``: marshal once,
    call :func:`matmul_batch_prepared` many times."""
    arr = (_Job * max(1, len(jobs)))()
    for i, (w, n_out, y) in enumerate(jobs):
        arr[i].w = w.handle if isinstance(w, Weight) else w
        arr[i].n_out = int(n_out)
        arr[i].y = int(y)
    return arr, len(jobs)


def matmul_batch_prepared(x_ptr: int, t: int, n_in: int, prepared, stream_ptr: int) -> int:
    """``il_matmul_batch`` with a job array from :func:`prepare_jobs`."""
    arr, n = prepared
    return _check(load().il_matmul_batch(x_ptr, int(t), int(n_in), arr, n, stream_ptr))


def matmul_batch_noalloc_ptr(x_ptr: int, t: int, n_in: int, jobs, stream_ptr: int) -> int:
    """``il_matmul_batch_noalloc`` on raw device pointers (same ``jobs`` form as
    :func:`matmul_batch_ptr`).  The library allocates no device memory for it;
    see ``include/il.h`` for the fixed scratch limit."""
    arr = (_Job * max(1, len(jobs)))()
    for i, (w, n_out, y) in enumerate(jobs):
        arr[i].w = w.handle if isinstance(w, Weight) else w
        arr[i].n_out = int(n_out)
        arr[i].y = int(y)
    return _check(load().il_matmul_batch_noalloc(x_ptr, int(t), int(n_in), arr, len(jobs), stream_ptr))


def matmul_batch(x, jobs, stream=None) -> None:
    """``il_matmul_batch`` on torch CUDA tensors.

    ``x``: fp32 ``[t][n_in]`` contiguous; ``jobs``: ``[(Weight, y)]`` with ``y``
    fp32 ``[t][n_out]`` contiguous, overwritten.  Enqueued on ``stream`` (default:
    the current torch stream).
    """
    if x.dim() != 2 or not x.is_contiguous():
        raise ILError(-1, "x must be a contiguous [t][n_in] tensor")
    t, n_in = x.shape
    lst = []
    for w, y in jobs:
        if not y.is_contiguous():
            raise ILError(-1, "y must be contiguous")
        lst.append((w, w.n_out, y.data_ptr()))
    matmul_batch_ptr(x.data_ptr(), t, n_in, lst, _stream_ptr(stream))


def matmul_batch_host_prepared(x_ptr: int, t: int, n_in: int, prepared, stream_ptr: int) -> int:
    """``il_matmul_batch_host`` with a job array from :func:`prepare_jobs` whose y
    pointers are host addresses; ``x_ptr`` is a host address too."""
    arr, n = prepared
    return _check(load().il_matmul_batch_host(x_ptr, int(t), int(n_in), arr, n, stream_ptr))


def matmul_batch_host(x, jobs, stream=None, sync: bool = True) -> None:
    """``il_matmul_batch_host`` on CPU torch tensors (pinned or not).

    ``x``: fp32 ``[t][n_in]`` contiguous; ``jobs``: ``[(Weight, y)]`` with ``y``
    fp32 ``[t][n_out]`` contiguous on the CPU, overwritten.  Enqueued on
    ``stream`` (default: the current torch stream); with ``sync`` the call waits
    for the stream, so ``y`` holds the results when it returns.
    """
    if x.device.type != "cpu" or x.dim() != 2 or not x.is_contiguous():
        raise ILError(-1, "x must be a contiguous [t][n_in] CPU tensor")
    t, n_in = x.shape
    lst = []
    for w, y in jobs:
        if y.device.type != "cpu" or not y.is_contiguous():
            raise ILError(-1, "y must be a contiguous CPU tensor")
        lst.append((w, w.n_out, y.data_ptr()))
    sp = _stream_ptr(stream)
    arr = (_Job * max(1, len(lst)))()
    for i, (w, n_out, y) in enumerate(lst):
        arr[i].w = w.handle if isinstance(w, Weight) else w
        arr[i].n_out = int(n_out)
        arr[i].y = int(y)
    _check(load().il_matmul_batch_host(x.data_ptr(), int(t), int(n_in), arr, len(lst), sp))
    if sync:
        import torch
        if sp:
            torch.cuda.ExternalStream(sp).synchronize()
        else:
            torch.cuda.synchronize()


def dequantize_weight(w: Weight, out, stream=None) -> None:
    """Test hook: every element of ``w`` as fp32 into ``out`` ([n_out][n_in], CUDA;
    [2*n_out][n_in] with gate/up rows interleaved for a gate+up weight)."""
    _check(load().il_dequantize_weight(w.handle, out.data_ptr(), _stream_ptr(stream)))


def check_device_status(stream=None) -> None:
    _check(load().il_check_device_status(_stream_ptr(stream)))


def release_scratch(stream=None) -> None:
    """``il_release_scratch``: frees the library's scratch for ``stream`` (stream-ordered)."""
    _check(load().il_release_scratch(_stream_ptr(stream)))


def get_stats() -> dict:
    s = _Stats()
    _check(load().il_get_stats(ctypes.byref(s)))
    return {name: getattr(s, name) for name, _ in _Stats._fields_}


def reset_stats() -> None:
    load().il_reset_stats()

"""Boundary behaviour of the C ABI on a GPU: every bad call returns its documented
status, launches nothing and leaves every output untouched (oxinfer src/gpu.rs,
`Backend::matmul`: an unsuccessful call computes nothing)."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import workloads as wl
from gpu_util import lib

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sil():
    import torch
    torch.cuda.set_device(0)
    return lib()


@pytest.fixture(scope="module")
def setup(sil):
    import torch
    b = wl.make_batch(256, (64, 32), 2, "q8", seed=0)
    ws = [sil.upload_weight(f, buf, n, 256) for f, buf, n in b.jobs]
    x = torch.from_numpy(b.x).cuda()
    yield b, ws, x
    for w in ws:
        w.free()


def _canaries(b, value=123.5):
    import torch
    return [torch.full((b.t, n), value, device="cuda") for _, _, n in b.jobs]


def _expect(sil, code, fn):
    before = sil.get_stats()
    with pytest.raises(sil.ILError) as ei:
        fn()
    assert ei.value.code == code, str(ei.value)
    after = sil.get_stats()
    assert after["launches"] == before["launches"]
    assert after["errors"] == before["errors"] + 1
    return ei.value


def _untouched(ys, value=123.5):
    import torch
    torch.cuda.synchronize()
    return all(bool(torch.all(y == value)) for y in ys)


def test_upload_rejects(sil):
    q8 = wl.make_batch(64, (4,), 1, "q8").jobs[0][1]
    ILError = sil.ILError
    for fmt, buf, n_out, n_in, code in [
        (7, q8, 4, 64, -3),                       # unknown format
        ("q8", q8, 4, 48, -2),                    # Q needs n_in % 32 == 0
        ("bf16", np.zeros(2 * 4 * 12, np.uint8), 4, 12, -2),   # bf16 needs n_in % 8 == 0
        ("q8", q8, 0, 64, -2),                    # n_out >= 1
        ("q8", q8, 4, 0, -2),
        ("bf16", np.zeros(16, np.uint8), 1, 65536, -2),       # n_in limit
    ]:
        with pytest.raises(ILError) as ei:
            sil.upload_weight(fmt, buf, n_out, n_in)
        assert ei.value.code == code, (fmt, n_out, n_in, str(ei.value))
    lib_ = sil.load()
    assert lib_.il_upload_weight(0, None, 4, 64) is None
    assert lib_.il_last_status() == -1


def test_bad_batches_compute_nothing(sil, setup):
    import torch
    b, ws, x = setup
    ys = _canaries(b)
    jobs = list(zip(ws, ys))

    # n_in mismatch: a weight of another width
    other = sil.upload_weight("q8", wl.make_batch(128, (64,), 1, "q8").jobs[0][1], 64, 128)
    _expect(sil, -2, lambda: sil.matmul_batch(x, [(other, ys[0]), (ws[1], ys[1])]))
    other.free()
    # n_out mismatch
    _expect(sil, -2, lambda: sil.matmul_batch_ptr(x.data_ptr(), b.t, 256,
                                                  [(ws[0], 63, ys[0].data_ptr())], 0))
    # freed handle
    dead = sil.upload_weight("q8", b.jobs[0][1], 64, 256)
    h = dead.handle
    dead.free()
    _expect(sil, -4, lambda: sil.matmul_batch_ptr(x.data_ptr(), b.t, 256,
                                                  [(h, 64, ys[0].data_ptr())], 0))
    # forged handle
    fake = ctypes.create_string_buffer(256)
    _expect(sil, -4, lambda: sil.matmul_batch_ptr(x.data_ptr(), b.t, 256,
                                                  [(ctypes.addressof(fake), 64, ys[0].data_ptr())], 0))
    # null y / null x / misaligned x / misaligned y
    _expect(sil, -1, lambda: sil.matmul_batch_ptr(x.data_ptr(), b.t, 256, [(ws[0], 64, 0)], 0))
    _expect(sil, -1, lambda: sil.matmul_batch_ptr(0, b.t, 256, [(ws[0], 64, ys[0].data_ptr())], 0))
    xb = torch.zeros(b.t * 256 + 4, device="cuda")
    _expect(sil, -1, lambda: sil.matmul_batch_ptr(xb.data_ptr() + 4, b.t, 256,
                                                  [(ws[0], 64, ys[0].data_ptr())], 0))
    _expect(sil, -1, lambda: sil.matmul_batch_ptr(x.data_ptr(), b.t, 256,
                                                  [(ws[0], 64, ys[0].data_ptr() + 2)], 0))
    # overlapping outputs, and y overlapping x
    _expect(sil, -1, lambda: sil.matmul_batch_ptr(x.data_ptr(), b.t, 256,
                                                  [(ws[0], 64, ys[0].data_ptr()),
                                                   (ws[1], 32, ys[0].data_ptr() + 64)], 0))
    _expect(sil, -1, lambda: sil.matmul_batch_ptr(x.data_ptr(), b.t, 256,
                                                  [(ws[0], 64, x.data_ptr())], 0))
    # negative sizes
    _expect(sil, -1, lambda: sil.matmul_batch_ptr(x.data_ptr(), -1, 256,
                                                  [(ws[0], 64, ys[0].data_ptr())], 0))
    # one bad job among good ones: nothing at all is computed
    _expect(sil, -2, lambda: sil.matmul_batch_ptr(x.data_ptr(), b.t, 256,
                                                  [(ws[0], 64, ys[0].data_ptr()),
                                                   (ws[1], 31, ys[1].data_ptr())], 0))
    assert _untouched(ys)


def test_noops(sil, setup):
    b, ws, x = setup
    ys = _canaries(b)
    before = sil.get_stats()
    sil.matmul_batch_ptr(x.data_ptr(), 0, 256, [(ws[0], 64, ys[0].data_ptr())], 0)
    sil.matmul_batch_ptr(x.data_ptr(), b.t, 256, [], 0)
    assert sil.get_stats()["launches"] == before["launches"]
    assert _untouched(ys)


def test_weight_bytes_and_info(sil):
    for fmt, n_out, n_in in (("bf16", 24, 64), ("q8", 24, 64), ("q4", 24, 64)):
        buf = wl.make_batch(n_in, (n_out,), 1, fmt).jobs[0][1]
        w = sil.upload_weight(fmt, buf, n_out, n_in)
        assert w.bytes == buf.size == wl.weight_bytes(fmt, n_out, n_in)
        f, o, i = ctypes.c_int(), ctypes.c_int64(), ctypes.c_int64()
        assert sil.load().il_weight_info(w.handle, ctypes.byref(f), ctypes.byref(o),
                                         ctypes.byref(i)) == 0
        assert (f.value, o.value, i.value) == (sil.FORMATS[fmt], n_out, n_in)
        w.free()
    assert sil.load().il_weight_bytes(None) == -1


def test_stats_count_work(sil, setup):
    b, ws, x = setup
    ys = _canaries(b)
    sil.reset_stats()
    sil.matmul_batch(x, list(zip(ws, ys)))
    s = sil.get_stats()
    assert s["batches"] == 1 and s["jobs"] == 2 and s["launches"] >= 1
    assert s["weight_bytes"] == sum(w.bytes for w in ws)
    assert s["flops"] == 2 * b.t * 256 * (64 + 32)


def test_device_status_clean(sil):
    sil.check_device_status()


_ALLOC_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
import torch
torch.cuda.set_device(0)
import shared_input_linear_gb300 as sil
import workloads as wl
buf = wl.make_batch(64, (16,), 1, "q4").jobs[0][1]
try:
    sil.upload_weight("q4", buf, 16, 64)
except sil.ILError as e:
    print("CODE", e.code)
    # a later upload also fails (the injected limit stays), and the process stays healthy
    x = torch.ones(4, device="cuda")
    torch.cuda.synchronize()
    print("HEALTHY", float(x.sum()))
"""


def test_allocation_failure_injected(sil):
    # IL_FAULT_ALLOC_FAIL_AFTER=1: the status word allocates, the weight's allocation fails
    env = dict(os.environ, IL_FAULT_ALLOC_FAIL_AFTER="1")
    out = subprocess.run([sys.executable, "-c", _ALLOC_SCRIPT.format(root=ROOT)], env=env,
                         capture_output=True, text=True, timeout=300)
    assert "CODE -5" in out.stdout, out.stdout + out.stderr
    assert "HEALTHY 4.0" in out.stdout, out.stdout + out.stderr


_TIMEOUT_SCRIPT = r"""
import os, sys
sys.path.insert(0, {root!r})
import numpy as np
import torch
torch.cuda.set_device(0)
import shared_input_linear_gb300 as sil
import workloads as wl
import oracle
b = wl.make_batch(256, (128,), 16, "bf16", seed=3)
w = sil.upload_weight("bf16", b.jobs[0][1], 128, 256)
x = torch.from_numpy(b.x).cuda()
y = torch.zeros(16, 128, device="cuda")
os.environ["IL_TEST_STALL_TMA_PRODUCER"] = "1"
sil.matmul_batch(x, [(w, y)])          # enqueues; the kernel's wait gives up after ~1 s
try:
    sil.check_device_status()
    print("NO_TIMEOUT")
except sil.ILError as e:
    print("CODE", e.code)
del os.environ["IL_TEST_STALL_TMA_PRODUCER"]
sil.matmul_batch(x, [(w, y)])          # the context is still usable
torch.cuda.synchronize()
sil.check_device_status()
y_ref, mag = oracle.linear("bf16", b.jobs[0][1], 128, 256, b.x)
ok, worst, _ = oracle.check(y.cpu().numpy(), y_ref, mag)
print("AFTER", ok)
"""


def test_bounded_wait_reports_timeout():
    # A wait that nothing will satisfy (the TMA producer is told to issue nothing):
    # the tensor-core kernel gives up after about a second, records the timeout in
    # the device status word, and the next call on the same context is correct.
    out = subprocess.run([sys.executable, "-c", _TIMEOUT_SCRIPT.format(root=ROOT)],
                         capture_output=True, text=True, timeout=300)
    assert "CODE -7" in out.stdout, out.stdout + out.stderr
    assert "AFTER True" in out.stdout, out.stdout + out.stderr


_STALL_SCRIPT = r"""
import os, sys
sys.path.insert(0, {root!r})
import numpy as np
import torch
torch.cuda.set_device(0)
import shared_input_linear_gb300 as sil
import workloads as wl
import oracle
fmt, t, entry = {fmt!r}, {t!r}, {entry!r}
if entry == "batch_ws":                  # split K through the global workspace, not CTA pairs
    os.environ["IL_TEST_SPLIT_WORKSPACE"] = "1"
b = wl.make_batch(512, (96, 40), t, fmt, seed=4)
ws = [sil.upload_weight(f, buf, n, 512) for f, buf, n in b.jobs]
x = torch.from_numpy(b.x).cuda()
ys = [torch.zeros(t, n, device="cuda") for _, _, n in b.jobs]
jobs = [(w, n, y.data_ptr()) for w, (_, _, n), y in zip(ws, b.jobs, ys)]
call = sil.matmul_batch_noalloc_ptr if entry == "noalloc" else sil.matmul_batch_ptr
s = torch.cuda.current_stream().cuda_stream
call(x.data_ptr(), t, 512, jobs, s)      # a warm call: the entry point is set up
torch.cuda.synchronize()
os.environ["IL_TEST_STALL_TMA_PRODUCER"] = "1"
call(x.data_ptr(), t, 512, jobs, s)      # the kernel's waits give up after ~1 s
try:
    sil.check_device_status()
    print("NO_TIMEOUT")
except sil.ILError as e:
    print("CODE", e.code)
del os.environ["IL_TEST_STALL_TMA_PRODUCER"]
for y in ys:
    y.fill_(float("nan"))
call(x.data_ptr(), t, 512, jobs, s)      # the context is still usable
torch.cuda.synchronize()
sil.check_device_status()
ok = True
for (f, buf, n), y in zip(b.jobs, ys):
    y_ref, mag = oracle.linear(f, buf, n, 512, b.x)
    ok &= oracle.check(y.cpu().numpy(), y_ref, mag)[0]
print("AFTER", ok)
"""


@pytest.mark.parametrize("fmt,t,entry", [
    ("q4", 1, "batch"),      # Q8/Q4 decode kernel: its bulk-copy waits
    ("q8", 6, "batch"),
    ("bf16", 16, "noalloc"),  # tensor-core kernel through the no-alloc entry point
    ("bf16", 24, "batch"),    # tensor-core kernel, split K as CTA pairs (cluster barriers)
    ("q8", 24, "batch_ws"),   # tensor-core kernel, split K through the global workspace
    ("q4", 3, "noalloc"),     # decode kernel through the no-alloc entry point
])
def test_stalled_copies_report_timeout(fmt, t, entry):
    # The copies a kernel waits for are never issued (a test switch read on the
    # host): its bounded waits give up after about a second, the code lands in
    # the status word of that entry point, il_check_device_status reports it, and
    # the next call on the same context is correct.
    out = subprocess.run([sys.executable, "-c", _STALL_SCRIPT.format(root=ROOT, fmt=fmt, t=t, entry=entry)],
                         capture_output=True, text=True, timeout=300)
    assert "CODE -7" in out.stdout, out.stdout + out.stderr
    assert "AFTER True" in out.stdout, out.stdout + out.stderr


_MAPFAIL_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
import numpy as np
import torch
torch.cuda.set_device(0)
import shared_input_linear_gb300 as sil
import workloads as wl
t, n_in = 64, 512
b16 = wl.make_batch(n_in, (200, 72), t, "bf16", seed=5)
b8 = wl.make_batch(n_in, (136,), t, "q8", seed=6)
jobs = b16.jobs + b8.jobs
ws = [sil.upload_weight(f, buf, n, n_in) for f, buf, n in jobs]
x = torch.from_numpy(b16.x).cuda()
ys = [torch.full((t, n), 7.0, device="cuda") for _, _, n in jobs]
before = sil.get_stats()["launches"]
try:
    # tensor maps: x and two weights for the bf16 launch, then x, quants and scales
    # for the Q8 launch; the 4th encoding fails, after the bf16 launch was prepared
    sil.matmul_batch(x, list(zip(ws, ys)))
    print("NO_ERROR")
except sil.ILError as e:
    print("CODE", e.code)
torch.cuda.synchronize()
print("LAUNCHES", sil.get_stats()["launches"] - before)
print("UNTOUCHED", all(bool(torch.all(y == 7.0)) for y in ys))
"""


def test_failed_preparation_enqueues_nothing():
    # A mixed bf16 + Q8 batch on the tensor-core path whose second launch cannot be
    # prepared (the 4th tensor-map encoding of the process is made to fail): the
    # call returns an error, launched no kernel (not even the cast of x or the bf16
    # launch that was ready) and wrote no y.
    env = dict(os.environ, IL_FAULT_TENSOR_MAP_FAIL_AFTER="3")
    out = subprocess.run([sys.executable, "-c", _MAPFAIL_SCRIPT.format(root=ROOT)], env=env,
                         capture_output=True, text=True, timeout=300)
    assert "CODE -6" in out.stdout, out.stdout + out.stderr
    assert "LAUNCHES 0" in out.stdout, out.stdout + out.stderr
    assert "UNTOUCHED True" in out.stdout, out.stdout + out.stderr


def test_release_scratch(sil):
    import torch
    import oracle
    import workloads as wl
    s = torch.cuda.Stream()
    b = wl.make_batch(1024, (300, 40), 64, "bf16", seed=8)
    ws = [sil.upload_weight(f, buf, n, 1024) for f, buf, n in b.jobs]
    x = torch.from_numpy(b.x).cuda()
    for _ in range(2):
        ys = [torch.full((64, n), float("nan"), device="cuda") for _, _, n in b.jobs]
        with torch.cuda.stream(s):
            sil.matmul_batch(x, list(zip(ws, ys)), stream=s)
            sil.release_scratch(s)  # freed in stream order, after the batch that reads it
        s.synchronize()
        for (f, buf, n), y in zip(b.jobs, ys):
            y_ref, mag = oracle.linear(f, buf, n, 1024, b.x)
            assert oracle.check(y.cpu().numpy(), y_ref, mag)[0]
    for w in ws:
        w.free()


_PROFILE_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
import torch
torch.cuda.set_device(0)
import shared_input_linear_gb300 as sil
import workloads as wl
b = wl.make_batch(1024, (512, 256), 4, "q8", seed=8)
ws = [sil.upload_weight(f, buf, n, 1024) for f, buf, n in b.jobs]
x = torch.from_numpy(b.x).cuda()
ys = [torch.empty(4, n, device="cuda") for _, _, n in b.jobs]
sil.reset_stats()
for _ in range(3):
    sil.matmul_batch(x, list(zip(ws, ys)))
st = sil.get_stats()
print("STATS", st["batches"], st["profiled_batches"], st["device_ns"])
"""


@pytest.mark.parametrize("profile", ["1", "0"])
def test_profile_timing(profile):
    # IL_PROFILE=1: every batch is timed with CUDA events and il_get_stats adds the
    # device time; without it nothing is timed
    import os
    env = dict(os.environ, IL_PROFILE=profile)
    out = subprocess.run([sys.executable, "-c", _PROFILE_SCRIPT.format(root=ROOT)], capture_output=True,
                         text=True, timeout=300, env=env)
    line = [l for l in out.stdout.splitlines() if l.startswith("STATS")]
    assert line, out.stdout + out.stderr
    batches, profiled, ns = (int(v) for v in line[0].split()[1:])
    assert batches == 3
    if profile == "1":
        assert profiled == 3 and 0 < ns < 3_000_000_000
    else:
        assert profiled == 0 and ns == 0

"""Host-side checks of the C-ABI library (no GPU needed): it builds for sm_103a,
loads, and exports every function ``include/il.h`` declares.  No compute call
is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "il.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(il_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libil():
    import shared_input_linear_gb300 as sil
    sil.build()
    return ctypes.CDLL(sil.LIB_PATH)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("il_upload_weight", "il_matmul_batch", "il_free_weight", "il_weight_bytes",
                 "il_dequantize_weight", "il_last_error", "il_get_stats"):
        assert must in names


def test_every_declared_symbol_is_exported(libil):
    missing = [n for n in declared_functions() if not hasattr(libil, n)]
    assert not missing, f"declared in il.h but not exported: {missing}"


def test_version_needs_no_device(libil):
    libil.il_version.restype = ctypes.c_int
    assert libil.il_version() == 3


def test_binding_names_match_abi():
    import shared_input_linear_gb300 as sil
    for name in ("upload_weight", "matmul_batch", "matmul_batch_host", "free_weight", "weight_bytes",
                 "dequantize_weight", "get_stats", "last_error", "check_device_status"):
        assert callable(getattr(sil, name))


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "shared_input_linear_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.lower(), f"{f} mentions the oracle"


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import shared_input_linear_gb300 as sil
    monkeypatch.setattr(sil, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(sil, "_lib", None)
    with pytest.raises(sil.ILError):
        sil.load()


def test_stats_layout_matches_header(libil):
    # the binding's il_stats mirror has the header's fields in the header's order,
    # and il_get_stats fills it without a device (nothing is timed unless IL_PROFILE=1)
    import shared_input_linear_gb300 as sil
    text = open(HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} il_stats;", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"uint64_t\s+(\w+)\s*;", body)
    assert [f for f, _ in sil._Stats._fields_] == fields
    st = sil._Stats()
    libil.il_get_stats.argtypes = [ctypes.c_void_p]
    libil.il_get_stats.restype = ctypes.c_int
    assert libil.il_get_stats(ctypes.byref(st)) == 0


def test_host_entry_checks_arguments_before_the_device(libil):
    # il_matmul_batch_host: sizes and NULL pointers are refused before any device
    # is touched, and t == 0 / n_jobs == 0 are successful no-ops (as il_matmul_batch)
    f = libil.il_matmul_batch_host
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_void_p]
    f.restype = ctypes.c_int
    job = (ctypes.c_char * 24)()
    x = (ctypes.c_float * 8)()
    assert f(None, 0, 8, None, 0, None) == 0
    assert f(ctypes.addressof(x), 1, 8, ctypes.addressof(job), 0, None) == 0
    assert f(None, 1, 8, ctypes.addressof(job), 1, None) == -1        # IL_ERR_ARG: x is NULL
    assert f(ctypes.addressof(x), -1, 8, ctypes.addressof(job), 1, None) == -1
    assert f(ctypes.addressof(x), 1, 8, None, 1, None) == -1          # jobs is NULL
    assert f(ctypes.addressof(x), 1, 0, ctypes.addressof(job), 1, None) == -2   # IL_ERR_SHAPE: n_in
    # a host x needs no 16-byte alignment (it is copied): an odd address passes
    # the argument checks and fails later, at the first device step, not with IL_ERR_ARG
    libil.il_last_error.restype = ctypes.c_char_p
    rc = f(ctypes.addressof(x) + 4, 1, 8, None, 1, None)
    assert rc == -1 and b"jobs" in libil.il_last_error()

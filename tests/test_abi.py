"""The C ABI library: loads, exports every declared symbol, host-side behaviour (no GPU)."""
import ctypes
import os
import re

import pytest

import csr_spmm_gb300 as cs
from csr_spmm_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    return _lib.library()


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(spmm_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_symbols()
    assert {"spmm_create", "spmm_destroy", "spmm_csr_f32", "spmm_csr_f64",
            "spmm_csr_check", "spmm_status_string"} <= declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert declared == set(_lib.EXPORTED)


def test_status_strings(lib):
    for code in range(9):
        s = cs.status_string(code)
        assert s.startswith("SPMM_")
    assert "unknown" in cs.status_string(99)


def test_null_handle_is_rejected_before_any_device_work(lib):
    vp = ctypes.c_void_p
    assert lib.spmm_csr_f32(None, 1.0, None, None, None, 4, 4, None, 4, 4, 0.0, None, 4,
                            None) == cs.SPMM_ERR_INVALID_ARGUMENT
    assert lib.spmm_csr_f64(None, 1.0, None, None, None, 4, 4, None, 4, 4, 0.0, None, 4,
                            None) == cs.SPMM_ERR_INVALID_ARGUMENT
    assert lib.spmm_reserve(None, 4, 4, 4) == cs.SPMM_ERR_INVALID_ARGUMENT
    st = ctypes.c_int32(0)
    assert lib.spmm_csr_check(None, None, None, 1, 1, 0, None,
                              ctypes.byref(st)) == cs.SPMM_ERR_INVALID_ARGUMENT
    assert lib.spmm_create(None, 0) == cs.SPMM_ERR_NULL_POINTER
    assert lib.spmm_destroy(None) == cs.SPMM_OK
    del vp


def test_every_entry_point_rejects_a_null_handle_or_plan_on_the_host(lib):
    """Every call that takes a handle or a plan returns SPMM_ERR_INVALID_ARGUMENT
    for a NULL one before it touches a device (the header's error rules); the
    plan calls clear their outputs first.  All other pointers are NULL too, so
    nothing here can reach a device on any machine."""
    inv, null = cs.SPMM_ERR_INVALID_ARGUMENT, cs.SPMM_ERR_NULL_POINTER
    for name in ("spmm_csr_squared_f32", "spmm_csr_squared_f64"):
        assert getattr(lib, name)(None, 1.0, None, None, None, 4, None, 4, 4, 0.0, None, 4,
                                  None) == inv, name
    for name in ("spmm_fw_argmin_f32", "spmm_fw_argmin_f64"):
        assert getattr(lib, name)(None, 4, 4, *([None] * 12), None, None, None, None) == inv, name
    for name in ("spmm_ilu0_f32", "spmm_ilu0_f64"):
        assert getattr(lib, name)(None, 4, 12, None, None, None, None, None, None) == inv, name
    assert lib.spmm_set_l2_persistence(None, 0) == inv
    assert lib.spmm_set_profiling(None, 1) == inv
    prof = _lib.SpmmProfile()
    assert lib.spmm_get_profile(None, ctypes.byref(prof)) == inv
    rate = ctypes.c_double(0.0)
    assert lib.spmm_measure_fp64_fma_rate(None, ctypes.byref(rate)) == inv
    plan = ctypes.c_void_p(1)
    assert lib.spmm_plan_create(None, ctypes.byref(plan), None, 4, 4, 4, 4, None) == inv
    assert plan.value is None
    assert lib.spmm_plan_create(None, None, None, 4, 4, 4, 4, None) == null
    assert lib.spmm_plan_destroy(None) == cs.SPMM_OK
    for name in ("spmm_plan_csr_f32", "spmm_plan_csr_f64", "spmm_plan_csr_squared_f32",
                 "spmm_plan_csr_squared_f64"):
        assert getattr(lib, name)(None, 1.0, None, None, None, None, 4, 0.0, None, 4,
                                  None) == inv, name
    assert lib.spmm_plan_order_rows(None, None, None, None) == inv
    applied = ctypes.c_int32(7)
    assert lib.spmm_plan_order_rows_auto(None, None, None, None, ctypes.byref(applied)) == inv
    assert applied.value == 0


def test_no_allocation_entry_point_checks_its_arguments_on_the_host(lib):
    """spmm_csr_f32_noalloc: dimension, size-limit and NULL checks return before
    the device is queried, in the handle path's order; an empty product is a
    no-op.  Every pointer is NULL, so no case can reach a device."""
    f = lib.spmm_csr_f32_noalloc

    def call(m, k, n, ldb, ldc, alpha=1.0):
        return f(alpha, None, None, None, m, k, None, ldb, n, 0.0, None, ldc, None)

    assert call(-1, 4, 4, 4, 4) == cs.SPMM_ERR_INVALID_ARGUMENT
    assert call(4, -1, 4, 4, 4) == cs.SPMM_ERR_INVALID_ARGUMENT
    assert call(4, 4, -1, 4, 4) == cs.SPMM_ERR_INVALID_ARGUMENT
    assert call(4, 4, 8, 4, 8) == cs.SPMM_ERR_DIMENSION_MISMATCH      # ldb < n
    assert call(4, 4, 8, 8, 4) == cs.SPMM_ERR_DIMENSION_MISMATCH      # ldc < n
    assert call(4, 4, 4, 1 << 31, 4) == cs.SPMM_ERR_INVALID_ARGUMENT  # 32-bit gather offsets
    assert call(524_289, 4, 4, 4, 4) == cs.SPMM_ERR_TOO_LARGE
    assert call(4, 4, 513, 513, 513) == cs.SPMM_ERR_TOO_LARGE
    assert call(0, 4, 4, 4, 4) == cs.SPMM_OK
    assert call(4, 4, 0, 1, 1) == cs.SPMM_OK
    assert call(4, 4, 4, 4, 4) == cs.SPMM_ERR_NULL_POINTER            # C is NULL


def test_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p(1)
    s = lib.spmm_create(ctypes.byref(h), 0)
    assert s != cs.SPMM_OK and h.value is None


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(ImportError):
        _lib.library(str(tmp_path / "nope.so"))


def test_header_is_plain_c(tmp_path):
    """include/csr_spmm.h compiles as C (C99 and C11), not only as C++, and
    every declared entry point can be referenced from C."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("gcc not available")
    names = sorted(_declared_symbols())
    src = tmp_path / "use_header.c"
    src.write_text('#include "csr_spmm.h"\n'
                   + "".join(f"void (*ref_{n})(void) = (void (*)(void))&{n};\n" for n in names))
    for std in ("c99", "c11"):
        r = subprocess.run([gcc, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-pedantic",
                            "-fsyntax-only",
                            "-I", os.path.join(ROOT, "include"), str(src)],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr

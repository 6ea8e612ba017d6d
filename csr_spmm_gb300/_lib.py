"""ctypes binding of the C ABI declared in include/csr_spmm.h.

Argument marshalling only: every step of the product runs in the CUDA
library.  Functions keep the C names; pointers are passed as Python ints
(device addresses), streams as ints (``torch.cuda.Stream.cuda_stream``) or 0.
If the library is missing, importing the functions raises at once: there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libcsrspmm.so")

SPMM_OK = 0
SPMM_ERR_INVALID_ARGUMENT = 1
SPMM_ERR_DIMENSION_MISMATCH = 2
SPMM_ERR_NULL_POINTER = 3
SPMM_ERR_UNSUPPORTED_DEVICE = 4
SPMM_ERR_ALLOC = 5
SPMM_ERR_CUDA = 6
SPMM_ERR_INVALID_CSR = 7
SPMM_ERR_TOO_LARGE = 8

# every symbol include/csr_spmm.h declares
EXPORTED = ("spmm_create", "spmm_destroy", "spmm_reserve", "spmm_csr_f32", "spmm_csr_f64",
            "spmm_csr_check", "spmm_set_profiling", "spmm_get_profile", "spmm_csr_f32_noalloc",
            "spmm_set_l2_persistence", "spmm_csr_squared_f32", "spmm_csr_squared_f64",
            "spmm_fw_argmin_f32", "spmm_fw_argmin_f64", "spmm_ilu0_f32", "spmm_ilu0_f64",
            "spmm_plan_create", "spmm_plan_destroy", "spmm_plan_csr_f32", "spmm_plan_csr_f64",
            "spmm_plan_order_rows", "spmm_row_order_bfs", "spmm_plan_csr_squared_f32",
            "spmm_plan_csr_squared_f64", "spmm_measure_fp64_fma_rate", "spmm_plan_order_rows_auto",
            "spmm_status_string")


class SpmmProfile(ctypes.Structure):
    """Mirror of spmm_profile_t."""
    _fields_ = [("prepass_ms", ctypes.c_float), ("rows_ms", ctypes.c_float),
                ("long_ms", ctypes.c_float), ("fixup_ms", ctypes.c_float),
                ("total_ms", ctypes.c_float), ("launches", ctypes.c_int32),
                ("rows_short", ctypes.c_int32), ("rows_medium", ctypes.c_int32),
                ("rows_long", ctypes.c_int32), ("long_nnz", ctypes.c_int32),
                ("panels", ctypes.c_int32), ("panel_cols", ctypes.c_int32),
                ("vec_elems", ctypes.c_int32), ("group_lanes", ctypes.c_int32),
                ("slots", ctypes.c_int32), ("short_max", ctypes.c_int32),
                ("long_min", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class SpmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None


def library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = load_library(path)
    return _lib


def load_library(path: str) -> ctypes.CDLL:
    """Load a build of the library from `path` (a variant built with other
    -D flags, for tests) with the C signatures declared; not cached."""
    if not os.path.exists(path):
        raise ImportError(
            f"CUDA library not built: {path} is missing. Run `python -m csr_spmm_gb300.build` "
            "(or __graft_entry__.build()); there is no CPU fallback.")
    lib = ctypes.CDLL(path)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    st = ctypes.c_int
    lib.spmm_create.argtypes = [ctypes.POINTER(vp), ctypes.c_int]
    lib.spmm_create.restype = st
    lib.spmm_destroy.argtypes = [vp]
    lib.spmm_destroy.restype = st
    lib.spmm_reserve.argtypes = [vp, i64, i64, ctypes.c_int]
    lib.spmm_reserve.restype = st
    lib.spmm_csr_f32.argtypes = [vp, ctypes.c_float, vp, vp, vp, i64, i64, vp, i64, i64,
                                 ctypes.c_float, vp, i64, vp]
    lib.spmm_csr_f32.restype = st
    lib.spmm_csr_f64.argtypes = [vp, ctypes.c_double, vp, vp, vp, i64, i64, vp, i64, i64,
                                 ctypes.c_double, vp, i64, vp]
    lib.spmm_csr_f64.restype = st
    lib.spmm_csr_check.argtypes = [vp, vp, vp, i64, i64, i64, vp, ctypes.POINTER(i32)]
    lib.spmm_csr_check.restype = st
    lib.spmm_set_profiling.argtypes = [vp, ctypes.c_int]
    lib.spmm_set_profiling.restype = st
    lib.spmm_get_profile.argtypes = [vp, ctypes.POINTER(SpmmProfile)]
    lib.spmm_get_profile.restype = st
    lib.spmm_csr_f32_noalloc.argtypes = [ctypes.c_float, vp, vp, vp, i64, i64, vp, i64, i64,
                                         ctypes.c_float, vp, i64, vp]
    lib.spmm_csr_f32_noalloc.restype = st
    for name, real in (("spmm_csr_squared_f32", ctypes.c_float),
                       ("spmm_csr_squared_f64", ctypes.c_double)):
        fn = getattr(lib, name)
        fn.argtypes = [vp, real, vp, vp, vp, i64, vp, i64, i64, real, vp, i64, vp]
        fn.restype = st
    for name in ("spmm_fw_argmin_f32", "spmm_fw_argmin_f64"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, i64, i64] + [vp] * 12 + [vp, vp, vp, vp]
        fn.restype = st
    for name in ("spmm_ilu0_f32", "spmm_ilu0_f64"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp, vp]
        fn.restype = st
    lib.spmm_set_l2_persistence.argtypes = [vp, i64]
    lib.spmm_set_l2_persistence.restype = st
    lib.spmm_plan_order_rows_auto.argtypes = [vp, vp, vp, vp, ctypes.POINTER(ctypes.c_int32)]
    lib.spmm_plan_order_rows_auto.restype = st
    lib.spmm_measure_fp64_fma_rate.argtypes = [vp, ctypes.POINTER(ctypes.c_double)]
    lib.spmm_measure_fp64_fma_rate.restype = st
    lib.spmm_plan_create.argtypes = [vp, ctypes.POINTER(vp), vp, i64, i64, i64, ctypes.c_int, vp]
    lib.spmm_plan_create.restype = st
    lib.spmm_plan_destroy.argtypes = [vp]
    lib.spmm_plan_destroy.restype = st
    lib.spmm_plan_csr_f32.argtypes = [vp, ctypes.c_float, vp, vp, vp, vp, i64, ctypes.c_float, vp,
                                      i64, vp]
    lib.spmm_plan_csr_f32.restype = st
    lib.spmm_plan_csr_f64.argtypes = [vp, ctypes.c_double, vp, vp, vp, vp, i64, ctypes.c_double,
                                      vp, i64, vp]
    lib.spmm_plan_csr_f64.restype = st
    lib.spmm_plan_csr_squared_f32.argtypes = [vp, ctypes.c_float, vp, vp, vp, vp, i64,
                                              ctypes.c_float, vp, i64, vp]
    lib.spmm_plan_csr_squared_f32.restype = st
    lib.spmm_plan_csr_squared_f64.argtypes = [vp, ctypes.c_double, vp, vp, vp, vp, i64,
                                              ctypes.c_double, vp, i64, vp]
    lib.spmm_plan_csr_squared_f64.restype = st
    lib.spmm_plan_order_rows.argtypes = [vp, vp, vp, vp]
    lib.spmm_plan_order_rows.restype = st
    lib.spmm_row_order_bfs.argtypes = [vp, vp, i64, vp]
    lib.spmm_row_order_bfs.restype = st
    lib.spmm_status_string.argtypes = [ctypes.c_int]
    lib.spmm_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return library().spmm_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != SPMM_OK:
        raise SpmmError(status, where)


def spmm_create(device: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(library().spmm_create(ctypes.byref(h), int(device)), "spmm_create")
    return h.value


def spmm_destroy(handle: int) -> None:
    _check(library().spmm_destroy(handle), "spmm_destroy")


def spmm_reserve(handle: int, m: int, n: int, elem_size: int) -> None:
    _check(library().spmm_reserve(handle, m, n, elem_size), "spmm_reserve")


def spmm_csr_f32(handle, alpha, row_ptr, col_idx, values, m, k, B, ldb, n, beta, C, ldc,
                 stream=0, check=True) -> int:
    s = library().spmm_csr_f32(handle, float(alpha), row_ptr, col_idx, values, m, k, B, ldb, n,
                               float(beta), C, ldc, stream or None)
    if check:
        _check(s, "spmm_csr_f32")
    return s


def spmm_csr_f64(handle, alpha, row_ptr, col_idx, values, m, k, B, ldb, n, beta, C, ldc,
                 stream=0, check=True) -> int:
    s = library().spmm_csr_f64(handle, float(alpha), row_ptr, col_idx, values, m, k, B, ldb, n,
                               float(beta), C, ldc, stream or None)
    if check:
        _check(s, "spmm_csr_f64")
    return s


def spmm_csr_check(handle, row_ptr, col_idx, m, k, nnz, stream=0):
    """Returns (status, mask); mask 0 means the CSR structure is valid."""
    mask = ctypes.c_int32(-1)
    s = library().spmm_csr_check(handle, row_ptr, col_idx, m, k, nnz, stream or None,
                                 ctypes.byref(mask))
    return s, mask.value


def spmm_set_profiling(handle, enable: bool) -> None:
    _check(library().spmm_set_profiling(handle, 1 if enable else 0), "spmm_set_profiling")


def spmm_get_profile(handle) -> dict:
    prof = SpmmProfile()
    _check(library().spmm_get_profile(handle, ctypes.byref(prof)), "spmm_get_profile")
    return prof.as_dict()


def spmm_csr_f32_noalloc(alpha, row_ptr, col_idx, values, m, k, B, ldb, n, beta, C, ldc,
                         stream=0, check=True) -> int:
    """The handle-free binary32 product whose scratch is a fixed device array
    inside the library (for callers that cannot allocate device memory)."""
    s = library().spmm_csr_f32_noalloc(float(alpha), row_ptr, col_idx, values, m, k, B, ldb, n,
                                       float(beta), C, ldc, stream or None)
    if check:
        _check(s, "spmm_csr_f32_noalloc")
    return s


def spmm_plan_csr_squared_f32(plan, alpha, row_ptr, col_idx, values, B, ldb, beta, C, ldc,
                              stream=0, check=True) -> int:
    s = library().spmm_plan_csr_squared_f32(plan, float(alpha), row_ptr, col_idx, values, B, ldb,
                                            float(beta), C, ldc, stream or None)
    if check:
        _check(s, "spmm_plan_csr_squared_f32")
    return s


def spmm_plan_csr_squared_f64(plan, alpha, row_ptr, col_idx, values, B, ldb, beta, C, ldc,
                              stream=0, check=True) -> int:
    s = library().spmm_plan_csr_squared_f64(plan, float(alpha), row_ptr, col_idx, values, B, ldb,
                                            float(beta), C, ldc, stream or None)
    if check:
        _check(s, "spmm_plan_csr_squared_f64")
    return s


def spmm_plan_order_rows(plan, row_ptr, col_idx, stream=0) -> None:
    """Process the plan's rows in breadth-first order of A's pattern (device arrays)."""
    _check(library().spmm_plan_order_rows(plan, row_ptr, col_idx, stream or None),
           "spmm_plan_order_rows")


def spmm_row_order_bfs(row_ptr, col_idx):
    """Breadth-first row order of a CSR pattern given as host (numpy) arrays;
    returns an int32 numpy permutation of the m rows."""
    import numpy as np
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    m = rp.size - 1
    order = np.empty(max(m, 0), dtype=np.int32)
    _check(library().spmm_row_order_bfs(rp.ctypes.data, ci.ctypes.data if ci.size else None, m,
                                        order.ctypes.data if m > 0 else None),
           "spmm_row_order_bfs")
    return order


def spmm_plan_create(handle, row_ptr, m, k, n, elem_size, stream=0) -> int:
    """Analyse a sparsity structure once; returns the plan pointer."""
    plan = ctypes.c_void_p()
    _check(library().spmm_plan_create(handle, ctypes.byref(plan), row_ptr, m, k, n, elem_size,
                                      stream or None), "spmm_plan_create")
    return plan.value


def spmm_plan_destroy(plan) -> None:
    _check(library().spmm_plan_destroy(plan), "spmm_plan_destroy")


def spmm_plan_csr_f32(plan, alpha, row_ptr, col_idx, values, B, ldb, beta, C, ldc, stream=0,
                      check=True) -> int:
    s = library().spmm_plan_csr_f32(plan, float(alpha), row_ptr, col_idx, values, B, ldb,
                                    float(beta), C, ldc, stream or None)
    if check:
        _check(s, "spmm_plan_csr_f32")
    return s


def spmm_plan_csr_f64(plan, alpha, row_ptr, col_idx, values, B, ldb, beta, C, ldc, stream=0,
                      check=True) -> int:
    s = library().spmm_plan_csr_f64(plan, float(alpha), row_ptr, col_idx, values, B, ldb,
                                    float(beta), C, ldc, stream or None)
    if check:
        _check(s, "spmm_plan_csr_f64")
    return s


def spmm_plan_order_rows_auto(plan, row_ptr, col_idx, stream=0) -> bool:
    """Breadth-first row order for the plan where it raises B-row reuse;
    returns whether the order was changed."""
    out = ctypes.c_int32(0)
    _check(library().spmm_plan_order_rows_auto(plan, row_ptr, col_idx, stream or None,
                                               ctypes.byref(out)), "spmm_plan_order_rows_auto")
    return bool(out.value)


def spmm_measure_fp64_fma_rate(handle) -> float:
    """The device's binary64 FMA instructions per second (a measurement aid;
    synchronises)."""
    out = ctypes.c_double(0.0)
    _check(library().spmm_measure_fp64_fma_rate(handle, ctypes.byref(out)),
           "spmm_measure_fp64_fma_rate")
    return out.value


def spmm_set_l2_persistence(handle, nbytes) -> None:
    """Persisting L2 set-aside for B (0: off, < 0: device maximum)."""
    _check(library().spmm_set_l2_persistence(handle, int(nbytes)), "spmm_set_l2_persistence")


def spmm_csr_squared_f32(handle, alpha, row_ptr, col_idx, values, m, B, ldb, n, beta, C, ldc,
                         stream=0, check=True) -> int:
    """C = alpha * A (A B) + beta * C for a square m x m CSR A (binary32)."""
    s = library().spmm_csr_squared_f32(handle, float(alpha), row_ptr, col_idx, values, m, B, ldb,
                                       n, float(beta), C, ldc, stream or None)
    if check:
        _check(s, "spmm_csr_squared_f32")
    return s


def spmm_csr_squared_f64(handle, alpha, row_ptr, col_idx, values, m, B, ldb, n, beta, C, ldc,
                         stream=0, check=True) -> int:
    """C = alpha * A (A B) + beta * C for a square m x m CSR A (binary64)."""
    s = library().spmm_csr_squared_f64(handle, float(alpha), row_ptr, col_idx, values, m, B, ldb,
                                       n, float(beta), C, ldc, stream or None)
    if check:
        _check(s, "spmm_csr_squared_f64")
    return s


def spmm_fw_argmin(handle, n, k, k2b, t1, t2, bmat, min_val, min_idx, gap, f64=False, stream=0,
                   check=True) -> int:
    """Frank-Wolfe gradient scan; each matrix a (row_ptr, col_idx, values)
    triple of device pointers, outputs device pointers."""
    fn = library().spmm_fw_argmin_f64 if f64 else library().spmm_fw_argmin_f32
    s = fn(handle, n, k, *k2b, *t1, *t2, *bmat, min_val, min_idx, gap, stream or None)
    if check:
        _check(s, "spmm_fw_argmin_f64" if f64 else "spmm_fw_argmin_f32")
    return s


ILU0_SINGULAR = 1
ILU0_WAIT_TIMEOUT = 2


def spmm_ilu0(handle, n, nnz, row_ptr, col_idx, values, depth, status, f64=False, stream=0,
              check=True) -> int:
    """ILU(0) in place on the device values (pointers); status is a device int32."""
    fn = library().spmm_ilu0_f64 if f64 else library().spmm_ilu0_f32
    s = fn(handle, n, nnz, row_ptr, col_idx, values, depth, status, stream or None)
    if check:
        _check(s, "spmm_ilu0_f64" if f64 else "spmm_ilu0_f32")
    return s

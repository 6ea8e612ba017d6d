"""CPU oracle for CSR SpMM (C = alpha * A * B + beta * C0), the squared
chain (C = alpha * A (A B) + beta * C0) and the Frank-Wolfe gradient scan
(per-column argmin of G = K2B t1 - T2 and the gap sum), fp64 accumulation.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it; the product path never does.  The
arithmetic lives in ``spmm_oracle.c`` (plain C, compiled here with gcc, with
floating-point contraction off so results are identical on every host); this
module only builds it and marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spmm_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

OK, BAD_ARGS, BAD_CSR, NO_MEMORY, SINGULAR = 0, -1, -2, -3, -4

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (if stale) and return its path."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str):
    """ctypes handle on a build of spmm_oracle.c, with argument types declared."""
    lib = ctypes.CDLL(path)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_spmm.restype = ctypes.c_int
    lib.oracle_spmm.argtypes = [ctypes.c_int, i64, i64, i64, ctypes.c_double, p, p, p, p,
                                i64, ctypes.c_double, p, i64, p, i64, p, p, i64]
    lib.oracle_spmm_squared.restype = ctypes.c_int
    lib.oracle_spmm_squared.argtypes = [ctypes.c_int, i64, i64, ctypes.c_double, p, p, p, p, i64,
                                        ctypes.c_double, p, i64, p, i64, p, p, i64]
    lib.oracle_fw_gradient.restype = ctypes.c_int
    lib.oracle_fw_gradient.argtypes = [ctypes.c_int, i64, i64] + [p] * 9 + [p, i64, p, p]
    lib.oracle_fw_argmin.restype = ctypes.c_int
    lib.oracle_fw_argmin.argtypes = [ctypes.c_int, i64, i64] + [p] * 12 + [p] * 5
    lib.oracle_ilu0.restype = ctypes.c_int
    lib.oracle_ilu0.argtypes = [ctypes.c_int, i64, p, p, p, p]
    lib.oracle_ilu0_levels.restype = i64
    lib.oracle_ilu0_levels.argtypes = [i64, p, p, p]
    lib.oracle_csr_check.restype = ctypes.c_int
    lib.oracle_csr_check.argtypes = [i64, i64, i64, p, p]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def csr_check(m: int, k: int, row_ptr: np.ndarray, col_idx: np.ndarray) -> int:
    """0 when (row_ptr, col_idx) is a valid m x k CSR structure, else BAD_CSR."""
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int32)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    nnz = int(row_ptr[m]) if row_ptr.size > m else -1
    if nnz < 0 or col_idx.size < nnz:
        return BAD_CSR
    return _load().oracle_csr_check(m, k, nnz, _ptr(row_ptr), _ptr(col_idx))


def spmm(m: int, k: int, n: int, alpha: float, row_ptr, col_idx, values, B, ldb: int,
         beta: float, C0=None, ldc: int = 0, rows: Optional[np.ndarray] = None, _lib=None):
    """Evaluate alpha * A * B + beta * C0 in fp64 for all rows (or ``rows``).

    ``values``, ``B`` and ``C0`` must share one dtype, float32 or float64;
    B is addressed as B.flat[col * ldb + c] and C0 as C0.flat[i * ldc + c].
    Returns ``(out, bound)``, both float64 of shape [len(rows) or m, n]:
    the result and the error-bound scale |alpha| sum|a||b| + |beta||C0|.
    ``_lib`` substitutes another build of ``spmm_oracle.c`` (the tests use it
    to show that deliberately broken copies fail the pins).
    """
    values = np.ascontiguousarray(values)
    dt = values.dtype
    if dt not in (np.float32, np.float64):
        raise TypeError("values must be float32 or float64")
    B = np.ascontiguousarray(B, dtype=dt)
    C0 = None if C0 is None else np.ascontiguousarray(C0, dtype=dt)
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int32)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    rsel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = m if rsel is None else int(rsel.size)
    out = np.zeros((nrows, n), dtype=np.float64)
    bound = np.zeros((nrows, n), dtype=np.float64)
    lib = _load() if _lib is None else _lib
    rc = lib.oracle_spmm(dt.itemsize, m, k, n, float(alpha), _ptr(row_ptr), _ptr(col_idx),
                         _ptr(values), _ptr(B), ldb, float(beta), _ptr(C0), ldc,
                         _ptr(rsel), nrows, _ptr(out), _ptr(bound), n)
    if rc != OK:
        raise ValueError(f"oracle_spmm rejected its inputs (status {rc})")
    return out, bound


def spmm_squared(m: int, n: int, alpha: float, row_ptr, col_idx, values, B, ldb: int,
                 beta: float, C0=None, ldc: int = 0, rows: Optional[np.ndarray] = None,
                 _lib=None):
    """Evaluate alpha * A (A B) + beta * C0 in fp64 for a square m x m CSR A.

    Same conventions and return value as :func:`spmm`; the bound is
    |alpha| |A| |A| |B| + |beta| |C0|.  The intermediate A B stays in fp64.
    """
    values = np.ascontiguousarray(values)
    dt = values.dtype
    if dt not in (np.float32, np.float64):
        raise TypeError("values must be float32 or float64")
    B = np.ascontiguousarray(B, dtype=dt)
    C0 = None if C0 is None else np.ascontiguousarray(C0, dtype=dt)
    # A may be absent when alpha == 0 (it is not read then)
    row_ptr = None if row_ptr is None else np.ascontiguousarray(row_ptr, dtype=np.int32)
    col_idx = None if col_idx is None else np.ascontiguousarray(col_idx, dtype=np.int32)
    rsel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = m if rsel is None else int(rsel.size)
    out = np.zeros((nrows, n), dtype=np.float64)
    bound = np.zeros((nrows, n), dtype=np.float64)
    lib = _load() if _lib is None else _lib
    rc = lib.oracle_spmm_squared(dt.itemsize, m, n, float(alpha), _ptr(row_ptr), _ptr(col_idx),
                                 _ptr(values), _ptr(B), ldb, float(beta), _ptr(C0), ldc,
                                 _ptr(rsel), nrows, _ptr(out), _ptr(bound), n)
    if rc != OK:
        raise ValueError(f"oracle_spmm_squared rejected its inputs (status {rc})")
    return out, bound


def spmm_problem(p, rows: Optional[np.ndarray] = None):
    """Oracle on a :class:`synth.Problem`."""
    return spmm(p.m, p.k, p.n, p.alpha, p.row_ptr, p.col_idx, p.values, p.B, p.ldb,
                p.beta, p.C0, p.ldc, rows)


def _csr(mat, dt):
    rp, ci, v = mat
    return (np.ascontiguousarray(rp, dtype=np.int32), np.ascontiguousarray(ci, dtype=np.int32),
            np.ascontiguousarray(v, dtype=dt))


def fw_gradient(n: int, k: int, k2b, t1, t2, rows: Optional[np.ndarray] = None, _lib=None):
    """Rows of G = K2B t1 - T2 (each argument a CSR triple (row_ptr, col_idx,
    values), K2B and T2 n x k, t1 k x k) in fp64, with their bound scale.
    Returns (G, gbound), float64 [len(rows) or n, k]."""
    dt = np.asarray(k2b[2]).dtype
    if dt not in (np.float32, np.float64):
        raise TypeError("values must be float32 or float64")
    a, b, c = _csr(k2b, dt), _csr(t1, dt), _csr(t2, dt)
    rsel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = n if rsel is None else int(rsel.size)
    g = np.zeros((nrows, k))
    gb = np.zeros((nrows, k))
    lib = _load() if _lib is None else _lib
    rc = lib.oracle_fw_gradient(dt.itemsize, n, k, *(_ptr(x) for x in a + b + c), _ptr(rsel),
                                nrows, _ptr(g), _ptr(gb))
    if rc != OK:
        raise ValueError(f"oracle_fw_gradient rejected its inputs (status {rc})")
    return g, gb


def fw_argmin(n: int, k: int, k2b, t1, t2, bmat, _lib=None):
    """The Frank-Wolfe B-update scan: per column the minimum of G = K2B t1 - T2
    over rows (lowest row on ties), and gap = sum of B * G over B's entries.

    Returns a dict: min_val [k], min_idx [k] (int64), col_scale [k], gap,
    gap_bound.
    """
    dt = np.asarray(k2b[2]).dtype
    if dt not in (np.float32, np.float64):
        raise TypeError("values must be float32 or float64")
    a, b, c, d = _csr(k2b, dt), _csr(t1, dt), _csr(t2, dt), _csr(bmat, dt)
    mv = np.zeros(max(k, 1))
    mi = np.zeros(max(k, 1), np.int64)
    cs = np.zeros(max(k, 1))
    gap = np.zeros(1)
    gbd = np.zeros(1)
    lib = _load() if _lib is None else _lib
    rc = lib.oracle_fw_argmin(dt.itemsize, n, k, *(_ptr(x) for x in a + b + c + d), _ptr(mv),
                              _ptr(mi), _ptr(cs), _ptr(gap), _ptr(gbd))
    if rc != OK:
        raise ValueError(f"oracle_fw_argmin rejected its inputs (status {rc})")
    return {"min_val": mv[:k], "min_idx": mi[:k], "col_scale": cs[:k], "gap": float(gap[0]),
            "gap_bound": float(gbd[0])}


class SingularMatrix(ValueError):
    """ILU(0) met a zero or missing pivot."""


def ilu0(row_ptr, col_idx, values, _lib=None):
    """ILU(0) of a square CSR matrix (columns ascending within rows), in the
    element type of ``values`` (float32 or float64), as the oxicuda page
    computes it.  Returns (factored values in A's pattern, depth per row).
    Raises SingularMatrix on a zero or missing pivot."""
    values = np.array(values, copy=True)
    dt = values.dtype
    if dt not in (np.float32, np.float64):
        raise TypeError("values must be float32 or float64")
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int32)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    n = row_ptr.size - 1
    depth = np.zeros(max(n, 1), np.int64)
    lib = _load() if _lib is None else _lib
    rc = lib.oracle_ilu0(dt.itemsize, n, _ptr(row_ptr), _ptr(col_idx), _ptr(values), _ptr(depth))
    if rc == SINGULAR:
        raise SingularMatrix("zero or missing pivot")
    if rc != OK:
        raise ValueError(f"oracle_ilu0 rejected its inputs (status {rc})")
    return values, depth[:n]


def ilu0_split(row_ptr, col_idx, factored):
    """(L, U) as dense arrays from factors stored in A's pattern: L the
    strictly lower part plus a unit diagonal, U the diagonal and above."""
    row_ptr = np.asarray(row_ptr)
    n = row_ptr.size - 1
    L = np.eye(n)
    U = np.zeros((n, n))
    for i in range(n):
        for p in range(row_ptr[i], row_ptr[i + 1]):
            j = int(col_idx[p])
            (L if j < i else U)[i, j] = factored[p]
    return L, U

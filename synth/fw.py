"""Seeded inputs of the Frank-Wolfe gradient scan (SEACells B update):
K2B and T2 (n x k), t1 (k x k) and B (n x k), all CSR.

This module holds no arithmetic of the scan; it only draws matrices.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import rng
from .workloads import distinct_sorted_columns

S_K2B_COLS, S_K2B_VALS, S_T1, S_T2_COLS, S_T2_VALS, S_B_SUP, S_B_W = 301, 302, 303, 304, 305, 306, 307


@dataclass
class FwProblem:
    name: str
    n: int
    k: int
    k2b: tuple          # (row_ptr int32 [n+1], col_idx int32, values)
    t1: tuple           # k x k
    t2: tuple           # n x k
    b: tuple            # n x k
    meta: dict = field(default_factory=dict)

    @property
    def dtype(self):
        return self.k2b[2].dtype

    def flops(self) -> int:
        """2 * nnz(K2B) * k: one multiply-add per K2B entry and column."""
        return 2 * int(self.k2b[0][-1]) * self.k

    def algorithmic_bytes(self) -> int:
        """Every CSR array once, t1 once, the outputs once."""
        es = self.dtype.itemsize
        total = 0
        for rp, ci, v in (self.k2b, self.t1, self.t2, self.b):
            total += 4 * rp.size + 4 * ci.size + es * v.size
        return total + (es + 4) * self.k + es


def _csr(rp, ci, vals, dtype):
    return (np.asarray(rp, np.int32), np.asarray(ci, np.int32), np.asarray(vals, dtype))


def fw_random(n: int, k: int, per_row: int, seed: int, *, dtype=np.float32,
              t1_density: float = 1.0, b_support: int = 50, name: str = "fw") -> FwProblem:
    """K2B and T2: ``per_row`` distinct sorted uniform columns per row, values
    U[0, 1).  t1: each entry kept with probability ``t1_density``, values
    U[0, 1) (diagonal always kept).  B: every column c has a random support of
    ``b_support`` distinct rows with Dirichlet(1) weights (normalised Exp(1)),
    stored row-wise."""
    lens = np.full(n, min(per_row, k), np.int64)
    rp, ci = distinct_sorted_columns(lens, k, seed, S_K2B_COLS)
    k2b = _csr(rp, ci, rng.uniform(seed, S_K2B_VALS, int(rp[-1])), dtype)
    rp2, ci2 = distinct_sorted_columns(lens, k, seed, S_T2_COLS)
    t2 = _csr(rp2, ci2, rng.uniform(seed, S_T2_VALS, int(rp2[-1])), dtype)
    u = rng.uniform(seed, S_T1, 2 * k * k).reshape(2, k, k)
    keep = (u[0] < t1_density) | np.eye(k, dtype=bool)
    rows, cols = np.nonzero(keep)
    t1rp = np.zeros(k + 1, np.int64)
    np.cumsum(keep.sum(axis=1), out=t1rp[1:])
    t1 = _csr(t1rp, cols, u[1][rows, cols], dtype)
    sup = min(b_support, n)
    sp, srow = distinct_sorted_columns(np.full(k, sup, np.int64), n, seed, S_B_SUP)
    w = rng.exponential(seed, S_B_W, int(sp[-1]))
    col_of = np.repeat(np.arange(k, dtype=np.int64), sup)
    w = w / np.bincount(col_of, weights=w, minlength=k)[col_of]
    order = np.lexsort((col_of, srow))                 # row-major: by row, then column
    brow, bcol, bval = srow[order], col_of[order], w[order]
    brp = np.zeros(n + 1, np.int64)
    np.cumsum(np.bincount(brow, minlength=n), out=brp[1:])
    b = _csr(brp, bcol, bval, dtype)
    return FwProblem(name, n, k, k2b, t1, t2, b,
                     meta={"seed": seed, "per_row": per_row, "t1_density": t1_density,
                           "b_support": sup})


def seacells_fw(seed: int = 1) -> FwProblem:
    """SEACells-shaped B-update scan: 200,000 cells, 100 archetypes (the
    columns of the SEACells-shaped product), 32 stored entries per row of K2B
    and K2At, dense t1, 50-cell Dirichlet supports per column of B, fp32."""
    return fw_random(200_000, 100, 32, seed, name="seacells_fw")

"""Seeded synthetic CSR SpMM problems: ``C = alpha * A @ B + beta * C0``.

Each generator returns a :class:`Problem` whose arrays are plain numpy arrays
(int32 CSR indices, float32/float64 values).  The five named workloads follow
the shapes, sizes, value distributions and sparsity structure stated for the
benchmark (tiny uniform, SEACells-shaped kNN kernel product, Zipf power-law
rows, 2-D 5-point Laplacian, wide-N exact integers); the same generators take
smaller sizes for the parity tests.  All randomness comes from the
counter-based SplitMix64 streams in :mod:`synth.rng`.

This module builds inputs only.  It contains no part of the product
arithmetic, and is shared by the CPU oracle tests and the CUDA path alike.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from . import rng

# stream ids (any distinct integers)
S_COLS, S_VALS, S_B, S_C0, S_PTS, S_PAIR, S_SUPPORT, S_WEIGHT, S_ZIPF, S_DIAG = range(10, 20)


@dataclass
class Problem:
    name: str
    m: int
    k: int
    n: int
    row_ptr: np.ndarray          # int32 [m+1]
    col_idx: np.ndarray          # int32 [nnz]
    values: np.ndarray           # float32/float64 [nnz]
    B: np.ndarray                # [k, ldb] row-major (only the first n columns are operands)
    C0: Optional[np.ndarray]     # [m, ldc] or None when beta == 0
    alpha: float
    beta: float
    ldb: int = 0
    ldc: int = 0
    meta: dict = field(default_factory=dict)

    def __post_init__(self):
        if not self.ldb:
            self.ldb = self.B.shape[1] if self.B.ndim == 2 else self.n
        if not self.ldc:
            self.ldc = self.C0.shape[1] if self.C0 is not None else self.n

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1]) if self.m > 0 else 0

    @property
    def dtype(self):
        return self.values.dtype

    def flops(self) -> int:
        """2 * nnz * n."""
        return 2 * self.nnz * self.n

    def algorithmic_bytes(self) -> int:
        """CSR arrays + B once + C read (beta != 0) + C write."""
        es = self.values.dtype.itemsize
        b = 4 * (self.m + 1) + 4 * self.nnz + es * self.nnz + es * self.k * self.n
        b += es * self.m * self.n * (2 if self.beta != 0.0 else 1)
        return b


# ---------------------------------------------------------------------------
# building blocks
# ---------------------------------------------------------------------------

def distinct_sorted_columns(lengths: np.ndarray, k: int, seed: int, stream: int):
    """For row i draw ``lengths[i]`` distinct column indices uniform on [0, k),
    returned row by row in ascending order.

    Duplicates are removed and re-drawn from later counters of the same
    stream until every row is full, so the result is a deterministic function
    of (lengths, k, seed, stream).
    Returns (row_ptr int64 [m+1], col_idx int64 [nnz]).
    """
    lengths = np.asarray(lengths, dtype=np.int64)
    m = lengths.shape[0]
    if m and int(lengths.max(initial=0)) > k:
        raise ValueError("row length exceeds k")
    total = int(lengths.sum())
    rows = np.repeat(np.arange(m, dtype=np.int64), lengths)
    draws = np.floor(rng.to_unit(rng.raw_u64(seed, stream, total)) * k).astype(np.int64)
    keys = sorted_unique(rows * k + draws)
    offset = total
    while True:
        counts = np.bincount(keys // k, minlength=m) if m else np.zeros(0, np.int64)
        deficit = lengths - counts
        need = int(deficit.sum())
        if need == 0:
            break
        rows2 = np.repeat(np.arange(m, dtype=np.int64), deficit)
        d2 = np.floor(rng.to_unit(rng.raw_u64(seed, stream, need, offset)) * k).astype(np.int64)
        offset += need
        keys = sorted_unique(np.concatenate([keys, rows2 * k + d2]))
    row_ptr = np.zeros(m + 1, dtype=np.int64)
    np.cumsum(lengths, out=row_ptr[1:])
    return row_ptr, keys % k if k else keys


def sorted_unique(a: np.ndarray) -> np.ndarray:
    """Ascending distinct values of an integer array (sort, then drop repeats)."""
    s = np.sort(np.asarray(a), kind="stable")
    if s.size == 0:
        return s
    keep = np.empty(s.size, dtype=bool)
    keep[0] = True
    np.not_equal(s[1:], s[:-1], out=keep[1:])
    return s[keep]


def _as_csr(row_ptr, col_idx, values, dtype):
    if int(row_ptr[-1]) > np.iinfo(np.int32).max:
        raise ValueError("nnz exceeds int32 CSR indexing")
    return (np.ascontiguousarray(row_ptr, dtype=np.int32),
            np.ascontiguousarray(col_idx, dtype=np.int32),
            np.ascontiguousarray(values, dtype=dtype))


def _pad(mat: np.ndarray, ld: int) -> np.ndarray:
    rows, cols = mat.shape
    if ld == cols:
        return np.ascontiguousarray(mat)
    out = np.zeros((rows, ld), dtype=mat.dtype)
    out[:, :cols] = mat
    return out


# ---------------------------------------------------------------------------
# generic families (also used at small sizes by the tests)
# ---------------------------------------------------------------------------

def uniform_rows(m: int, k: int, n: int, per_row: int, seed: int, *, dtype=np.float32,
                 alpha=1.5, beta=0.5, integer_range: Optional[int] = None,
                 ldb: int = 0, ldc: int = 0, name: str = "uniform") -> Problem:
    """Every row holds ``per_row`` distinct sorted uniform-random columns.

    Values, B and C0 are U[-1, 1], or integers uniform on
    [-integer_range, integer_range] when ``integer_range`` is given.
    """
    lengths = np.full(m, min(per_row, k), dtype=np.int64)
    rp, ci = distinct_sorted_columns(lengths, k, seed, S_COLS)
    nnz = int(rp[-1])
    if integer_range is None:
        vals = rng.uniform(seed, S_VALS, nnz, -1.0, 1.0)
        B = rng.uniform(seed, S_B, k * n, -1.0, 1.0).reshape(k, n)
        C0 = rng.uniform(seed, S_C0, m * n, -1.0, 1.0).reshape(m, n)
    else:
        r = integer_range
        vals = rng.integers(seed, S_VALS, nnz, -r, r).astype(np.float64)
        B = rng.integers(seed, S_B, k * n, -r, r).astype(np.float64).reshape(k, n)
        C0 = rng.integers(seed, S_C0, m * n, -r, r).astype(np.float64).reshape(m, n)
    rp32, ci32, v = _as_csr(rp, ci, vals, dtype)
    return Problem(name, m, k, n, rp32, ci32, v,
                   _pad(B.astype(dtype), ldb or n),
                   None if beta == 0.0 else _pad(C0.astype(dtype), ldc or n),
                   alpha, beta, ldb or n, ldc or n,
                   meta={"seed": seed, "per_row": per_row})


def knn_kernel_graph(cells: int, knn: int, n: int, support: int, seed: int, *,
                     dtype=np.float32, alpha=1.0, beta=0.0, sigma=1.0,
                     name: str = "seacells_knn") -> Problem:
    """SEACells-shaped kernel product.

    A: points iid uniform in [0,1]^3; the exact ``knn`` nearest neighbours of
    every point, the point itself included; symmetrised by union (so rows hold
    knn..2*knn entries).  Each unordered off-diagonal pair {i, j} gets one
    draw d ~ U[0, 2] and the value exp(-d^2 / sigma^2); the diagonal is 1.
    B: cells x n, column c has a random support of ``support`` distinct cells
    with Dirichlet(1) weights (normalised Exp(1) draws), zeros elsewhere.
    """
    from scipy.spatial import cKDTree

    pts = rng.uniform(seed, S_PTS, cells * 3).reshape(cells, 3)
    kk = min(knn, cells)
    _, idx = cKDTree(pts).query(pts, k=kk, workers=-1)
    idx = np.asarray(idx, dtype=np.int64).reshape(cells, kk)
    rows = np.repeat(np.arange(cells, dtype=np.int64), kk)
    cols = idx.ravel()
    # the query returns the point itself first; make sure the diagonal is present
    keys = sorted_unique(np.concatenate([rows * cells + cols, cols * cells + rows,
                                     np.arange(cells, dtype=np.int64) * (cells + 1)]))
    r = keys // cells
    c = keys % cells
    lo = np.minimum(r, c)
    hi = np.maximum(r, c)
    d = 2.0 * rng.to_unit(rng.raw_at(seed, S_PAIR, lo * cells + hi))
    vals = np.exp(-(d * d) / (sigma * sigma))
    vals[r == c] = 1.0
    counts = np.bincount(r, minlength=cells)
    rp = np.zeros(cells + 1, dtype=np.int64)
    np.cumsum(counts, out=rp[1:])

    sup_len = np.full(n, min(support, cells), dtype=np.int64)
    sp, srow = distinct_sorted_columns(sup_len, cells, seed, S_SUPPORT)
    w = rng.exponential(seed, S_WEIGHT, int(sp[-1]))
    col_of = np.repeat(np.arange(n, dtype=np.int64), sup_len)
    sums = np.bincount(col_of, weights=w, minlength=n)
    B = np.zeros((cells, n), dtype=np.float64)
    B[srow, col_of] = w / sums[col_of]

    rp32, ci32, v = _as_csr(rp, c, vals, dtype)
    C0 = None
    if beta != 0.0:
        C0 = rng.uniform(seed, S_C0, cells * n, -1.0, 1.0).reshape(cells, n).astype(dtype)
    lens = np.diff(rp)
    return Problem(name, cells, cells, n, rp32, ci32, v, B.astype(dtype), C0, alpha, beta,
                   meta={"seed": seed, "knn": knn, "support": support,
                         "row_len_min": int(lens.min()), "row_len_mean": float(lens.mean()),
                         "row_len_max": int(lens.max())})


def zipf_lengths(m: int, total: int, cap: int, seed: int, exponent: float = 2.0,
                 support: Optional[int] = None):
    """Row lengths L_i = min(cap, max(1, floor(s * raw_i + 1/2))), raw_i ~ Zipf(exponent)
    on 1..support (inverse-CDF table), with the scale s found by bisection as
    the smallest value giving sum(L) >= total.  Returns (lengths, s)."""
    support = support or m
    r = np.arange(1, support + 1, dtype=np.float64)
    cdf = np.cumsum(r ** (-exponent))
    cdf /= cdf[-1]
    u = rng.to_unit(rng.raw_u64(seed, S_ZIPF, m))
    raw = np.minimum(np.searchsorted(cdf, u, side="right"), support - 1).astype(np.float64) + 1.0

    def lengths_at(s):
        return np.minimum(cap, np.maximum(1, np.floor(s * raw + 0.5))).astype(np.int64)

    if int(lengths_at(1e-9).sum()) >= total:
        return lengths_at(1e-9), 1e-9
    lo, hi = 1e-9, 1.0
    while int(lengths_at(hi).sum()) < total:
        hi *= 2.0
        if hi > 1e12:
            break
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if int(lengths_at(mid).sum()) >= total:
            hi = mid
        else:
            lo = mid
    return lengths_at(hi), hi


def power_law(m: int, k: int, n: int, total_nnz: int, cap: int, seed: int, *,
              dtype=np.float32, alpha=1.0, beta=1.0, name: str = "power_law") -> Problem:
    """Zipf(2) row lengths scaled to ~total_nnz with the longest row capped;
    distinct sorted uniform columns; values, B and C0 N(0, 1)."""
    cap = min(cap, k)
    lengths, s = zipf_lengths(m, total_nnz, cap, seed)
    rp, ci = distinct_sorted_columns(lengths, k, seed, S_COLS)
    nnz = int(rp[-1])
    vals = rng.normal(seed, S_VALS, nnz)
    B = rng.normal(seed, S_B, k * n).reshape(k, n)
    C0 = rng.normal(seed, S_C0, m * n).reshape(m, n) if beta != 0.0 else None
    rp32, ci32, v = _as_csr(rp, ci, vals, dtype)
    return Problem(name, m, k, n, rp32, ci32, v, B.astype(dtype),
                   None if C0 is None else C0.astype(dtype), alpha, beta,
                   meta={"seed": seed, "zipf_scale": s, "cap": cap,
                         "rows_at_cap": int((lengths == cap).sum()),
                         "row_len_max": int(lengths.max(initial=0))})


def laplacian_2d(side: int, n: int, seed: int, *, dtype=np.float64, alpha=2.0, beta=-1.0,
                 perturb: float = 0.1, name: str = "laplacian5") -> Problem:
    """5-point Laplacian on a side x side grid, nodes in row-major grid order,
    neighbours outside the grid dropped.  Diagonal 4 + U[0, perturb],
    off-diagonals -1.  B and C0 U[-1, 1]."""
    N = side * side
    y, x = np.divmod(np.arange(N, dtype=np.int64), side)
    cand = [(y > 0, -side), (x > 0, -1), (np.ones(N, bool), 0), (x < side - 1, 1),
            (y < side - 1, side)]
    mask = np.stack([c for c, _ in cand], axis=1)          # [N, 5], ascending column order
    offs = np.array([o for _, o in cand], dtype=np.int64)
    cols_full = np.arange(N, dtype=np.int64)[:, None] + offs[None, :]
    ci = cols_full[mask]
    diag = 4.0 + rng.uniform(seed, S_DIAG, N, 0.0, perturb)
    vals_full = np.where(offs[None, :] == 0, diag[:, None], -1.0)
    vals = vals_full[mask]
    rp = np.zeros(N + 1, dtype=np.int64)
    np.cumsum(mask.sum(axis=1), out=rp[1:])
    B = rng.uniform(seed, S_B, N * n, -1.0, 1.0).reshape(N, n)
    C0 = rng.uniform(seed, S_C0, N * n, -1.0, 1.0).reshape(N, n) if beta != 0.0 else None
    rp32, ci32, v = _as_csr(rp, ci, vals, dtype)
    return Problem(name, N, N, n, rp32, ci32, v, B.astype(dtype),
                   None if C0 is None else C0.astype(dtype), alpha, beta,
                   meta={"seed": seed, "side": side})


# ---------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------

def tiny_uniform(seed: int = 0) -> Problem:
    """m=k=1024, 8 distinct sorted uniform columns per row, U[-1,1] values,
    B 1024x16, C0 U[-1,1], alpha=1.5, beta=0.5, fp32."""
    return uniform_rows(1024, 1024, 16, 8, seed, alpha=1.5, beta=0.5, name="tiny_uniform")


def seacells_knn(seed: int = 1) -> Problem:
    """Symmetrised 30-NN kernel graph over 200,000 cells, B 200,000x100
    column-stochastic with 50-cell supports, alpha=1, beta=0, fp32."""
    return knn_kernel_graph(200_000, 30, 100, 50, seed, name="seacells_knn")


def power_law_1m(seed: int = 2) -> Problem:
    """m=k=1,000,000, Zipf(2) row lengths scaled to ~20M nnz, cap 100,000,
    N(0,1) values, B 1e6x64 N(0,1), C0 N(0,1), alpha=1, beta=1, fp32."""
    return power_law(1_000_000, 1_000_000, 64, 20_000_000, 100_000, seed, name="power_law_1m")


def laplacian_707(seed: int = 3) -> Problem:
    """707x707 5-point Laplacian, B 499,849x32 U[-1,1], C0 U[-1,1],
    alpha=2, beta=-1, fp64."""
    return laplacian_2d(707, 32, seed, name="laplacian_707")


def wide_n_integer(seed: int = 4) -> Problem:
    """m=k=262,144, 16 distinct sorted uniform columns per row, integers in
    [-3,3] for A and B, B 262,144x512, alpha=1, beta=0, fp32 (exact)."""
    return uniform_rows(262_144, 262_144, 512, 16, seed, alpha=1.0, beta=0.0, integer_range=3,
                        name="wide_n_integer")


def seacells_k2b(seed: int = 1) -> Problem:
    """The SEACells-shaped product applied twice: C = K (K B) with the kNN
    kernel matrix K and the column-stochastic B of seacells_knn (the K^2 B
    operand of the bixverse page's Frank-Wolfe kernels), alpha=1, beta=0."""
    p = knn_kernel_graph(200_000, 30, 100, 50, seed, name="seacells_k2b")
    p.meta["chain"] = "squared"
    return p


WORKLOADS = {
    "tiny_uniform": tiny_uniform,
    "seacells_knn": seacells_knn,
    "power_law_1m": power_law_1m,
    "laplacian_707": laplacian_707,
    "wide_n_integer": wide_n_integer,
    "seacells_k2b": seacells_k2b,
}

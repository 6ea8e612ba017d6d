"""GPU ILU(0) (the oxicuda preconditioner page's factorisation) against the
CPU oracle.  Both take the page's steps with single rounded operations in
the element type, so the factors must agree bit for bit, and the per-row
levels exactly."""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
import oracle
from synth import laplacian_2d
from test_oracle_ilu0 import random_dd, tridiag

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()
    h = cs.Handle(0)
    yield h
    h.close()


def gpu_ilu0(handle, rp, ci, v):
    import torch
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).cuda()  # noqa: E731
    vals = t(v, v.dtype)
    depth = cs.ilu0(handle, t(rp, np.int32), t(ci, np.int32), vals, with_depth=True)
    return vals.cpu().numpy(), depth.cpu().numpy().astype(np.int64)


def check(handle, rp, ci, v, what):
    want, wdepth = oracle.ilu0(rp, ci, v)
    got, depth = gpu_ilu0(handle, rp, ci, v)
    bits = np.uint32 if v.dtype == np.float32 else np.uint64
    bad = np.nonzero(got.view(bits) != want.view(bits))[0]
    assert bad.size == 0, f"{what}: {bad.size} factors differ, first at {bad[:3]}"
    assert np.array_equal(depth, wdepth), what


PAGE = {
    "dense_2x2": ([0, 2, 4], [0, 1, 0, 1], [4.0, 2.0, 1.0, 3.0]),
    "dense_3x3": ([0, 3, 6, 9], [0, 1, 2, 0, 1, 2, 0, 1, 2],
                  [4.0, 1.0, 2.0, 1.0, 5.0, 1.0, 2.0, 1.0, 6.0]),
    "identity_4": ([0, 1, 2, 3, 4], [0, 1, 2, 3], [1.0, 1.0, 1.0, 1.0]),
}


@pytest.mark.parametrize("name", sorted(PAGE))
def test_page_matrices(handle, name):
    rp, ci, v = PAGE[name]
    check(handle, np.array(rp), np.array(ci), np.array(v), name)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_tridiagonal(handle, dtype):
    rp, ci, v = tridiag(5, dtype=dtype)
    check(handle, rp, ci, v, "tridiagonal 5")
    rp, ci, v = tridiag(3000, dtype=dtype)          # one long dependency chain
    check(handle, rp, ci, v, "tridiagonal 3000")


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_random_sparse(handle, dtype):
    for n, per, seed in ((500, 5, 1), (20_000, 9, 2)):
        rp, ci, v = random_dd(n, per, seed, dtype=dtype)
        check(handle, rp, ci, v, f"random {n}")


def mixed_lengths(n, seed, dtype=np.float64):
    """Rows of about 12 entries, every 7th row about 60 (past one warp), so
    both the register path and the long-row path run, and short rows pivot
    on long ones."""
    from synth import distinct_sorted_columns, rng
    lens = np.where(np.arange(n) % 7 == 0, 60, 12).astype(np.int64)
    rp, ci = distinct_sorted_columns(lens, n, seed, 21)
    rows = np.repeat(np.arange(n), np.diff(rp))
    keys = np.unique(np.concatenate([rows * n + ci, np.arange(n) * (n + 1)]))
    r, c = keys // n, keys % n
    vals = rng.uniform(seed, 22, keys.size, -1.0, 1.0)
    vals[r == c] = 70.0 + rng.uniform(seed, 23, n)
    rp2 = np.zeros(n + 1, np.int64)
    np.cumsum(np.bincount(r, minlength=n), out=rp2[1:])
    return rp2, c, vals.astype(dtype)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_long_rows(handle, dtype):
    rp, ci, v = mixed_lengths(4000, 3, dtype)
    check(handle, rp, ci, v, "mixed row lengths")
    rp, ci, v = random_dd(1500, 45, 4, dtype=dtype)          # every row past one warp
    check(handle, rp, ci, v, "long rows")


def test_laplacian_grid(handle):
    p = laplacian_2d(60, 1, seed=3)
    check(handle, p.row_ptr, p.col_idx, p.values.astype(np.float64), "laplacian 60")


def test_laplacian_707_full(handle):
    """The 707 x 707 5-point Laplacian of the preconditioner-shaped workload
    (499,849 rows, 1413 levels), in binary64 and binary32."""
    p = laplacian_2d(707, 1, seed=3)
    check(handle, p.row_ptr, p.col_idx, p.values.astype(np.float64), "laplacian 707 f64")
    check(handle, p.row_ptr, p.col_idx, p.values.astype(np.float32), "laplacian 707 f32")


def test_singular_pivot_reported(handle):
    # the page's singular case: zero diagonal in row 0, row 1 pivots on it
    with pytest.raises(cs.Ilu0Error, match="pivot"):
        gpu_ilu0(handle, np.array([0, 2, 4]), np.array([0, 1, 0, 1]),
                 np.array([0.0, 2.0, 1.0, 3.0]))
    # a pivot row without a stored diagonal
    with pytest.raises(cs.Ilu0Error, match="pivot"):
        gpu_ilu0(handle, np.array([0, 1, 3]), np.array([1, 0, 1]), np.array([2.0, 1.0, 3.0]))
    # the handle still works afterwards
    rp, ci, v = tridiag(50)
    check(handle, rp, ci, v, "after a failure")


def test_deterministic(handle):
    rp, ci, v = random_dd(30_000, 7, 5)
    a, _ = gpu_ilu0(handle, rp, ci, v)
    b, _ = gpu_ilu0(handle, rp, ci, v)
    assert np.array_equal(a.view(np.uint64), b.view(np.uint64))


def test_rejects_empty(handle):
    import torch
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = cs.spmm_ilu0(handle.ptr, 0, 0, z.data_ptr(), z.data_ptr(), z.data_ptr(), 0, z.data_ptr(),
                     check=False)
    assert s == 1                                     # SPMM_ERR_INVALID_ARGUMENT (as the page)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_band_pivot_rows_past_one_warp(handle, dtype):
    """Rows of 25 entries (band of half-width 12): a row's pivot rows, from
    their pivots on, hold 12 x 13 entries together, more than one warp reads
    at once, so they are read pivot row by pivot row; the narrow band below
    (half-width 2, 5 pivot entries per row at most) reads them in one batch."""
    from synth import rng
    for n, w in ((3000, 12), (3000, 2)):
        r = np.repeat(np.arange(n), 2 * w + 1)
        c = r + np.tile(np.arange(-w, w + 1), n)
        keep = (c >= 0) & (c < n)
        r, c = r[keep], c[keep]
        vals = rng.uniform(7, 1, r.size, -1.0, 1.0)
        vals[r == c] = 4.0 * w + 1.0
        rp = np.zeros(n + 1, np.int64)
        np.cumsum(np.bincount(r, minlength=n), out=rp[1:])
        check(handle, rp, c, vals.astype(dtype), f"band {w}")


# The published-value sentinels of the factorisation (signalling NaNs that no
# arithmetic returns): an input value with exactly these bits must still be
# passed on, through the kernel's done-flag path.
SENTINEL = {np.float64: np.uint64(0x7FF4C0DE5A5A5A5A), np.float32: np.uint32(0x7FA5C0DE)}


def sentinel_value(dtype):
    bits = np.uint64 if dtype == np.float64 else np.uint32
    return np.array([SENTINEL[dtype]], dtype=bits).view(dtype)[0]


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_sentinel_bits_in_an_unused_upper_entry(handle, dtype):
    """Row 0 stores the sentinel's bit pattern at (0, 2); row 1 reads row 0
    from its pivot on, so it waits on that value, but stores no column 2, so
    every factor is finite except the sentinel entry, which passes through."""
    rp = np.array([0, 2, 4, 6, 8])
    ci = np.array([0, 2, 0, 1, 1, 2, 2, 3])
    v = np.array([4.0, 0.0, 1.0, 5.0, 1.0, 6.0, 1.0, 7.0], dtype=dtype)
    v[1] = sentinel_value(dtype)
    check(handle, rp, ci, v, "sentinel in an upper entry")


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_sentinel_bits_on_the_long_row_path(handle, dtype):
    """Row 0 holds 40 entries (the long-row path) and 49 dependents (no
    structure record); its last column holds the sentinel's bits, which row 39
    uses (a NaN results) and every other row only reads past.  NaN factors
    may differ in payload between the host and the GPU, so those compare as
    NaN; the rest bit for bit."""
    n = 50
    rows = [list(range(40))] + [[0, i] for i in range(1, n)]
    rp = np.zeros(n + 1, dtype=np.int64)
    rp[1:] = np.cumsum([len(r) for r in rows])
    ci = np.concatenate([np.array(r) for r in rows])
    v = np.where(ci == np.repeat(np.arange(n), np.diff(rp)), 50.0, 1.0).astype(dtype)
    v[39] = sentinel_value(dtype)
    want, wdepth = oracle.ilu0(rp, ci, v)
    got, depth = gpu_ilu0(handle, rp, ci, v)
    bits = np.uint32 if dtype == np.float32 else np.uint64
    nan_w, nan_g = np.isnan(want), np.isnan(got)
    assert np.array_equal(nan_w, nan_g)
    assert nan_w.sum() >= 2                          # the sentinel and row 39's diagonal
    assert got.view(bits)[39] == SENTINEL[dtype]     # passed through unchanged
    ok = ~nan_w
    assert np.array_equal(got[ok].view(bits), want[ok].view(bits))
    assert np.array_equal(depth, wdepth)

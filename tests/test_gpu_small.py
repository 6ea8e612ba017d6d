"""GPU tests of the one-launch path for products of at most 2,048 rows.

Such a product runs as a single kernel in which every CTA bins the rows
itself in shared memory.  Short and medium rows are summed exactly as on the
binned path (same per-row arithmetic), so a product must equal, bit for bit,
the same rows computed on the binned path, which a copy of the problem padded
with empty rows past 2,048 takes.  Rows of 1,024 entries or more, which the
binned path splits across CTAs, are summed by one warp each here: those are
checked against the oracle, for determinism, and for equality between the
direct call, a plan and the no-allocation entry point (all three take the
one-launch path)."""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
from gpu_helpers import assert_parity, run_problem
from synth import Problem, distinct_sorted_columns, knn_kernel_graph, rng, uniform_rows

pytestmark = pytest.mark.gpu

SMALL_ROWS = 2048


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


def _bits(a):
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint64)


def _padded(p, m_total):
    """The same product with empty rows appended up to m_total rows."""
    extra = m_total - p.m
    rp = np.concatenate([p.row_ptr, np.full(extra, p.row_ptr[-1], p.row_ptr.dtype)])
    C0 = None
    if p.C0 is not None:
        C0 = np.concatenate([p.C0, np.zeros((extra, p.C0.shape[1]), p.C0.dtype)])
    return Problem(p.name + "_padded", m_total, p.k, p.n, rp, p.col_idx, p.values, p.B, C0,
                   p.alpha, p.beta, ldb=p.ldb, ldc=p.ldc)


def _ragged(m, k, n, max_len, seed, dtype=np.float32, alpha=1.25, beta=0.5, min_len=0):
    lens = min_len + np.floor(rng.uniform(seed, 1, m) * (max_len - min_len + 1)).astype(np.int64)
    lens = np.minimum(lens, k)
    rp, ci = distinct_sorted_columns(lens, k, seed, 2)
    vals = rng.uniform(seed, 3, int(rp[-1]), -1, 1).astype(dtype)
    B = rng.uniform(seed, 4, k * n, -1, 1).reshape(k, n).astype(dtype)
    C0 = rng.uniform(seed, 5, m * n, -1, 1).reshape(m, n).astype(dtype) if beta != 0 else None
    return Problem("ragged", m, k, n, rp.astype(np.int32), ci.astype(np.int32), vals, B, C0,
                   alpha, beta)


CASES = {
    "short_n16": lambda: uniform_rows(1024, 1024, 16, 8, seed=0, alpha=1.5, beta=0.5),
    "knn_n100_whole": lambda: knn_kernel_graph(2000, 20, 100, 40, seed=3),
    "ragged_medium_n64": lambda: _ragged(1500, 5000, 64, 900, seed=5),
    "ragged_n3": lambda: _ragged(2048, 3000, 3, 200, seed=6, beta=0.0),
    "f64_beta_m1": lambda: _ragged(1800, 4000, 32, 300, seed=7, dtype=np.float64, alpha=2.0,
                                   beta=-1.0),
    "f64_beta_general": lambda: _ragged(900, 2000, 10, 120, seed=8, dtype=np.float64, alpha=-0.5,
                                        beta=0.75),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("b_offset", [0, 1])
def test_small_path_equals_binned_path(handle, name, b_offset):
    p = CASES[name]()
    assert p.m <= SMALL_ROWS and np.diff(p.row_ptr).max() < 1024
    got, _ = run_problem(handle, p, b_offset=b_offset)
    q = _padded(p, SMALL_ROWS + 300)
    want, _ = run_problem(handle, q, b_offset=b_offset)
    assert np.array_equal(_bits(got[:, :p.n]), _bits(want[: p.m, : p.n])), name
    assert_parity(p, got, what=f"small path {name}")


def test_small_path_long_rows(handle):
    """Rows of 1,024-6,000 entries among short rows, m = 600: one warp per
    long row; oracle parity, determinism, and the same bits through a plan
    and through the no-allocation entry point."""
    import torch
    m, k, n = 600, 30_000, 48
    lens = np.floor(rng.uniform(21, 1, m) * 12).astype(np.int64)
    lens[::37] = 1024 + np.floor(rng.uniform(21, 2, len(lens[::37])) * 5000).astype(np.int64)
    rp, ci = distinct_sorted_columns(lens, k, 21, 3)
    vals = rng.uniform(21, 4, int(rp[-1]), -1, 1).astype(np.float32)
    B = rng.uniform(21, 5, k * n, -1, 1).reshape(k, n).astype(np.float32)
    C0 = rng.uniform(21, 6, m * n, -1, 1).reshape(m, n).astype(np.float32)
    p = Problem("small_long", m, k, n, rp.astype(np.int32), ci.astype(np.int32), vals, B, C0,
                -1.5, 0.25)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what="small path, long rows")
    again, _ = run_problem(handle, p)
    assert np.array_equal(_bits(got), _bits(again)), "not deterministic"
    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    rpd, cid, vad, Bd = t(p.row_ptr), t(p.col_idx), t(p.values), t(p.B)
    C = t(C0.copy())
    plan = cs.Plan(handle, rpd, k, n, torch.float32)
    try:
        plan(p.alpha, rpd, cid, vad, Bd, p.beta, C)
        torch.cuda.synchronize()
    finally:
        plan.close()
    assert np.array_equal(_bits(C.cpu().numpy()), _bits(got[:, :n]))
    C2 = t(C0.copy())
    cs.spmm_csr_f32_noalloc(p.alpha, rpd.data_ptr(), cid.data_ptr(), vad.data_ptr(), m, k,
                            Bd.data_ptr(), n, n, p.beta, C2.data_ptr(), n,
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(C2.cpu().numpy()), _bits(got[:, :n]))


@pytest.mark.parametrize("m", [SMALL_ROWS, SMALL_ROWS + 1])
def test_around_the_small_bound(handle, m):
    p = _ragged(m, 4000, 24, 1500, seed=31)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what=f"m = {m}")


def test_small_path_profile_counts_one_launch(handle):
    p = CASES["short_n16"]()
    cs.spmm_set_profiling(handle.ptr, True)
    try:
        run_problem(handle, p)
        prof = cs.spmm_get_profile(handle.ptr)
    finally:
        cs.spmm_set_profiling(handle.ptr, False)
    assert prof["launches"] == 1 and prof["rows_short"] == p.m and prof["rows_long"] == 0

"""GPU parity at the five full workload sizes, through the same C-ABI call and
launch configuration the benchmark times.  The oracle evaluates sampled rows
(every long row of the power-law matrix included); properties that hold at any
size check the rest."""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
from gpu_helpers import assert_parity, run_problem
from synth import rng
from synth import workloads as wl

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


def _sample_rows(m, count, seed, extra=()):
    r = np.floor(rng.uniform(seed, 77, count) * m).astype(np.int64)
    return np.unique(np.concatenate([r, [0, m - 1], np.asarray(extra, np.int64)]))


def test_full_tiny_uniform(handle):
    p = wl.tiny_uniform()
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what="tiny_uniform")


def test_full_seacells_knn(handle):
    p = wl.seacells_knn()
    got, _ = run_problem(handle, p, C_init=np.full((p.m, p.ldc), np.nan, np.float32))
    assert np.all(np.isfinite(got))
    assert_parity(p, got, rows=_sample_rows(p.m, 4000, 1), what="seacells_knn")
    # every column of B sums to 1 and A >= 0, so each column of C sums to
    # sum_ij A_ij * B_jc = (1^T A) B_c, checked for all rows at once
    colsum_A = np.bincount(p.col_idx, weights=p.values.astype(np.float64), minlength=p.k)
    want = colsum_A @ p.B.astype(np.float64)
    assert np.allclose(got.astype(np.float64).sum(axis=0), want, rtol=1e-5)


def test_full_power_law(handle):
    p = wl.power_law_1m()
    lens = np.diff(p.row_ptr)
    long_rows = np.flatnonzero(lens >= 1024)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, rows=_sample_rows(p.m, 3000, 2, extra=long_rows), what="power_law_1m")
    again, _ = run_problem(handle, p)
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32)), "not deterministic"


def test_full_laplacian(handle):
    p = wl.laplacian_707()
    got, _ = run_problem(handle, p)
    edge = np.concatenate([np.arange(707), np.arange(p.m - 707, p.m)])
    assert_parity(p, got, rows=_sample_rows(p.m, 6000, 3, extra=edge), what="laplacian_707")


def test_full_wide_n_integer(handle):
    p = wl.wide_n_integer()
    got, _ = run_problem(handle, p, C_init=np.full((p.m, p.ldc), np.nan, np.float32))
    assert_parity(p, got, rows=_sample_rows(p.m, 3000, 4), exact=True, what="wide_n_integer")
    # exact for all rows at once: column sums of C equal (1^T A) B in integers
    colsum_A = np.bincount(p.col_idx, weights=p.values.astype(np.float64),
                           minlength=p.k).astype(np.int64)
    want = colsum_A @ p.B.astype(np.int64)
    assert np.all(np.isfinite(got))
    assert np.array_equal(got.astype(np.int64).sum(axis=0), want)


def test_b_and_c_beyond_2_31_elements(handle):
    """B (k x ldb) and C (m x ldc) each hold more than 2^31 elements (8.8 GB
    apiece), so gather and store addresses need 64-bit arithmetic.  Only a
    few rows of A are non-empty; they read B rows on both sides of the 2^31
    boundary and write C rows past it.  The oracle evaluates the same sums on
    a compacted copy of the B rows that A references (same entries, same
    order); every other row of C must come out as alpha * 0 = 0."""
    import torch
    from synth import Problem
    m = k = 2_200_000
    n, ld = 1000, 1004
    assert m * ld > 2 ** 31 and k * ld > 2 ** 31
    rows = np.unique(np.concatenate([[0, 1, m // 2], np.arange(m - 100, m)]))
    per = 5
    hi_cols = (2 ** 31) // ld + np.arange(0, 50_000, 997)              # rows past element 2^31
    pool = np.unique(np.concatenate([[0, 1, k // 2, k - 2, k - 1], hi_cols]))
    pick = np.floor(rng.uniform(40, 1, rows.size * per) * pool.size).astype(np.int64)
    cols = np.sort(pool[pick].reshape(rows.size, per), axis=1)
    lens = np.zeros(m, np.int64)
    lens[rows] = per
    rp = np.zeros(m + 1, np.int64)
    np.cumsum(lens, out=rp[1:])
    ci = cols.ravel().astype(np.int32)
    vals = rng.uniform(40, 2, ci.size, -1.0, 1.0).astype(np.float32)
    used, local = np.unique(ci, return_inverse=True)
    Bused = rng.uniform(40, 3, used.size * n, -1.0, 1.0).reshape(used.size, n).astype(np.float32)

    dev = torch.device("cuda")
    Bd = torch.empty((k, ld), dtype=torch.float32, device=dev)
    Bd[torch.from_numpy(used.astype(np.int64)).to(dev), :n] = torch.from_numpy(Bused).to(dev)
    Cd = torch.full((m, ld), float("nan"), dtype=torch.float32, device=dev)
    rpd = torch.from_numpy(rp.astype(np.int32)).to(dev)
    cid = torch.from_numpy(ci).to(dev)
    vd = torch.from_numpy(vals).to(dev)
    alpha = 1.5
    cs.spmm_csr_f32(handle.ptr, alpha, rpd.data_ptr(), cid.data_ptr(), vd.data_ptr(), m, k,
                    Bd.data_ptr(), ld, n, 0.0, Cd.data_ptr(), ld,
                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    empty = np.array([2, 3, m // 2 + 1, m - 101], np.int64)
    check = np.concatenate([rows, empty])
    got = Cd[torch.from_numpy(check).to(dev), :n].cpu().numpy()
    del Bd, Cd
    torch.cuda.empty_cache()
    # the same sums on the compacted B: rows of A restricted to `rows`
    sub_rp = np.zeros(rows.size + 1, np.int64)
    np.cumsum(lens[rows], out=sub_rp[1:])
    q = Problem("beyond_2_31", rows.size, used.size, n, sub_rp.astype(np.int32),
                local.astype(np.int32), vals, Bused, None, alpha, 0.0)
    assert_parity(q, got[: rows.size], what="64-bit addressing")
    assert np.all(got[rows.size:] == 0.0)


def test_full_seacells_plan_in_breadth_first_order(handle):
    """The SEACells product through a plan whose rows were put in
    breadth-first order: bit for bit the direct product, at full size, on two
    calls with different B."""
    import copy

    import torch
    p = wl.seacells_knn()
    direct, _ = run_problem(handle, p)
    dev = torch.device("cuda")
    rp = torch.from_numpy(p.row_ptr).to(dev)
    ci = torch.from_numpy(p.col_idx).to(dev)
    va = torch.from_numpy(p.values).to(dev)
    C = torch.full((p.m, p.n), float("nan"), dtype=torch.float32, device=dev)
    plan = cs.Plan(handle, rp, p.k, p.n, torch.float32)
    try:
        assert plan.order_rows(rp, ci), "the kNN pattern should be reordered"
        for it, B in enumerate((p.B, p.B[::-1].copy())):
            plan(p.alpha, rp, ci, va, torch.from_numpy(B).to(dev), p.beta, C)
            torch.cuda.synchronize()
            got = C.cpu().numpy()
            if it == 0:
                assert np.array_equal(got.view(np.uint32), direct[:, :p.n].view(np.uint32))
            else:
                q = copy.copy(p)
                q.B = B
                want, _ = run_problem(handle, q)
                assert np.array_equal(got.view(np.uint32), want[:, :p.n].view(np.uint32))
    finally:
        plan.close()

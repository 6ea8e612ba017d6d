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

"""GPU tests of the persisting-L2 window on B: with the set-aside on, products
must be bitwise the same as without it (the window changes cache policy only),
and switching it off must leave later products unaffected."""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
from gpu_helpers import assert_parity, run_problem
from synth import knn_kernel_graph, power_law

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


def _bits(a):
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint64)


@pytest.mark.parametrize("make", [
    lambda: knn_kernel_graph(6000, 30, 100, 50, seed=1),                   # B fits: window on
    lambda: power_law(30_000, 30_000, 64, 600_000, 10_000, seed=5),        # long rows, beta != 0
])
def test_window_does_not_change_results(handle, make):
    p = make()
    off, _ = run_problem(handle, p)
    try:
        cs.spmm_set_l2_persistence(handle.ptr, -1)
        on, _ = run_problem(handle, p)
        on2, _ = run_problem(handle, p)
        cs.spmm_set_l2_persistence(handle.ptr, 8 << 20)   # a smaller set-aside
        small, _ = run_problem(handle, p)
    finally:
        cs.spmm_set_l2_persistence(handle.ptr, 0)
    after, _ = run_problem(handle, p)
    for got in (on, on2, small, after):
        assert np.array_equal(_bits(got[:, :p.n]), _bits(off[:, :p.n]))
    assert_parity(p, on, rows=np.arange(0, p.m, 11), what="persisting window")


def test_persistence_off_twice_is_harmless(handle):
    cs.spmm_set_l2_persistence(handle.ptr, 0)
    cs.spmm_set_l2_persistence(handle.ptr, 0)
    with pytest.raises(cs.SpmmError):
        cs.spmm_set_l2_persistence(0, -1)

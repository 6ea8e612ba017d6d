"""GPU parity of the squared chain C = alpha * A (A B) + beta * C (the K^2 B
product of the bixverse page's SEACells kernels) against the CPU oracle.

The GPU rounds the intermediate A B to the element type, so each output may
carry the error of two products: the tolerance is 2 * tau * bound with the
chain's bound |alpha| |A| |A| |B| + |beta| |C0| (tau = 1e-5 binary32, 1e-13
binary64).  Integer-valued inputs with small sums are checked bit for bit.
"""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
import oracle
from gpu_helpers import TAU, _dev
from synth import knn_kernel_graph, laplacian_2d, power_law, uniform_rows
from synth.workloads import seacells_knn

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


def run_squared(handle, p, b_offset=0, C_init=None, check=True):
    import torch
    dev = torch.device("cuda")
    rp, ci, va = (_dev(a, torch, dev) for a in (p.row_ptr, p.col_idx, p.values))
    Bd = _dev(np.concatenate([np.zeros(b_offset, p.B.dtype), p.B.ravel()]), torch, dev)
    if C_init is None:
        C_init = p.C0 if p.C0 is not None else np.full((p.m, p.ldc), np.nan, p.values.dtype)
    Cd = _dev(np.ascontiguousarray(C_init).copy(), torch, dev)
    fn = cs.spmm_csr_squared_f32 if p.values.dtype == np.float32 else cs.spmm_csr_squared_f64
    s = fn(handle.ptr, p.alpha, rp.data_ptr(), ci.data_ptr(), va.data_ptr(), p.m,
           Bd.data_ptr() + b_offset * p.B.itemsize, p.ldb, p.n, p.beta, Cd.data_ptr(), p.ldc,
           torch.cuda.current_stream().cuda_stream, check=check)
    torch.cuda.synchronize()
    out = Cd.cpu().numpy()[: p.m * p.ldc].reshape(p.m, p.ldc) if p.m else np.zeros((0, p.ldc))
    return out, s


def oracle_squared(p, rows=None):
    return oracle.spmm_squared(p.m, p.n, p.alpha, p.row_ptr, p.col_idx, p.values, p.B, p.ldb,
                               p.beta, p.C0, p.ldc, rows)


def assert_chain_parity(p, got, rows=None, exact=False, what=""):
    ref, bound = oracle_squared(p, rows)
    g = (got if rows is None else got[np.asarray(rows)])[:, : p.n]
    if exact:
        want = ref.astype(p.values.dtype)
        assert np.array_equal(g, want), f"{what}: {int((g != want).sum())} outputs differ"
        return
    err = np.abs(g.astype(np.float64) - ref)
    ok = err <= 2 * TAU[np.dtype(p.values.dtype)] * bound
    assert np.all(ok), (f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; worst "
                        f"ratio {np.max(err / np.maximum(bound, 1e-300)):.3g}")


def test_knn_whole_vectors(handle):
    p = knn_kernel_graph(6000, 30, 100, 50, seed=1)            # G = 32, n % 4 == 0
    got, _ = run_squared(handle, p)
    assert_chain_parity(p, got, what="knn chain")


def test_power_law_long_rows_beta(handle):
    p = power_law(30_000, 30_000, 64, 600_000, 10_000, seed=5)   # long rows, beta = 1
    got, _ = run_squared(handle, p)
    rows = np.unique(np.concatenate([np.argsort(-np.diff(p.row_ptr))[:40],
                                     np.linspace(0, p.m - 1, 300).astype(np.int64)]))
    assert_chain_parity(p, got, rows=rows, what="power-law chain")


def test_laplacian_f64(handle):
    p = laplacian_2d(60, 32, seed=3)                            # alpha 2, beta -1
    got, _ = run_squared(handle, p)
    assert_chain_parity(p, got, what="laplacian chain")


@pytest.mark.parametrize("n", [1, 3, 5, 17])
def test_ragged_columns(handle, n):
    p = uniform_rows(700, 700, n, 9, seed=20 + n, dtype=np.float32, alpha=-0.75, beta=0.5)
    got, _ = run_squared(handle, p)
    assert_chain_parity(p, got, what=f"n={n}")


def test_unaligned_b(handle):
    p = uniform_rows(900, 900, 12, 7, seed=31, dtype=np.float32)
    got, _ = run_squared(handle, p, b_offset=1)
    assert_chain_parity(p, got, what="unaligned B")


def test_integer_exact(handle):
    # |sum| <= 8 * 3 * 8 * 3 * 3 = 1728 < 2^24: every partial sum exact in binary32
    p = uniform_rows(3000, 3000, 40, 8, seed=32, dtype=np.float32, alpha=1.0, beta=0.0,
                     integer_range=3)
    got, _ = run_squared(handle, p)
    assert_chain_parity(p, got, exact=True, what="integer chain")


def test_alpha_zero_and_empty(handle):
    p = uniform_rows(300, 300, 8, 4, seed=33, dtype=np.float64, alpha=0.0, beta=-2.0)
    got, _ = run_squared(handle, p)
    assert np.array_equal(got[:, :p.n], -2.0 * p.C0[:, :p.n])
    q = uniform_rows(200, 200, 6, 0, seed=34, dtype=np.float32, alpha=1.0, beta=0.5)
    got, _ = run_squared(handle, q)                                  # every row empty
    assert_chain_parity(q, got, what="empty rows")


def test_deterministic(handle):
    p = power_law(30_000, 30_000, 64, 600_000, 10_000, seed=7)
    a, _ = run_squared(handle, p)
    b, _ = run_squared(handle, p)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_torch_wrapper(handle):
    import torch
    p = knn_kernel_graph(2000, 15, 40, 20, seed=14)
    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    C = torch.full((p.m, p.n), float("nan"), dtype=torch.float32, device=dev)
    cs.spmm_squared(handle, p.alpha, t(p.row_ptr), t(p.col_idx), t(p.values), t(p.B), p.beta, C)
    torch.cuda.synchronize()
    assert_chain_parity(p, C.cpu().numpy(), what="torch wrapper")


def test_seacells_full_size_sampled(handle):
    """The SEACells-shaped chain at full size (200,000 cells), the launch shape
    bench.py times, checked on sampled rows."""
    p = seacells_knn()
    got, _ = run_squared(handle, p)
    rows = np.unique(np.linspace(0, p.m - 1, 400).astype(np.int64))
    assert_chain_parity(p, got, rows=rows, what="seacells chain")
    # column sums: B is column-stochastic and A symmetric, so 1^T A A B = (A 1)^T (A B)
    s_got = got[:, :p.n].astype(np.float64).sum(axis=0)
    a1 = np.zeros(p.m)
    np.add.at(a1, np.repeat(np.arange(p.m), np.diff(p.row_ptr)), p.values.astype(np.float64))
    ab, _ = oracle.spmm(p.m, p.k, p.n, 1.0, p.row_ptr, p.col_idx, p.values, p.B, p.ldb, 0.0)
    want = a1 @ ab
    assert np.allclose(s_got, want, rtol=1e-4)


def run_plan_squared(handle, p, order=False, b_offset=0):
    """The chain through a plan (pre-pass once), optionally in breadth-first row order."""
    import torch
    dev = torch.device("cuda")
    rp, ci, va = (_dev(a, torch, dev) for a in (p.row_ptr, p.col_idx, p.values))
    Bd = _dev(np.concatenate([np.zeros(b_offset, p.B.dtype), p.B.ravel()]), torch, dev)
    C_init = p.C0 if p.C0 is not None else np.full((p.m, p.ldc), np.nan, p.values.dtype)
    Cd = _dev(np.ascontiguousarray(C_init).copy(), torch, dev)
    st = torch.cuda.current_stream().cuda_stream
    plan = cs.spmm_plan_create(handle.ptr, rp.data_ptr(), p.m, p.m, p.n, p.values.itemsize, st)
    try:
        if order:
            cs.spmm_plan_order_rows(plan, rp.data_ptr(), ci.data_ptr(), st)
        fn = (cs.spmm_plan_csr_squared_f32 if p.values.dtype == np.float32
              else cs.spmm_plan_csr_squared_f64)
        fn(plan, p.alpha, rp.data_ptr(), ci.data_ptr(), va.data_ptr(),
           Bd.data_ptr() + b_offset * p.B.itemsize, p.ldb, p.beta, Cd.data_ptr(), p.ldc, st)
        torch.cuda.synchronize()
    finally:
        cs.spmm_plan_destroy(plan)
    return Cd.cpu().numpy()[: p.m * p.ldc].reshape(p.m, p.ldc)


def _bits(a):
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint64)


@pytest.mark.parametrize("name", ["knn", "power_law", "laplacian_f64"])
@pytest.mark.parametrize("order", [False, True])
def test_plan_chain_equals_direct_chain(handle, name, order):
    """Through a plan, in natural or breadth-first row order, the chain gives
    the direct chain's bits (same bins, same per-row arithmetic), and so the
    oracle's parity."""
    p = {"knn": lambda: knn_kernel_graph(6000, 30, 100, 50, seed=1),
         "power_law": lambda: power_law(30_000, 30_000, 64, 600_000, 10_000, seed=5),
         "laplacian_f64": lambda: laplacian_2d(60, 32, seed=3)}[name]()
    direct, _ = run_squared(handle, p)
    got = run_plan_squared(handle, p, order=order)
    assert np.array_equal(_bits(got[:, :p.n]), _bits(direct[:, :p.n])), (name, order)
    rows = np.unique(np.linspace(0, p.m - 1, 200).astype(np.int64))
    assert_chain_parity(p, got, rows=rows, what=f"plan chain {name}")


def test_plan_chain_unaligned_b_and_errors(handle):
    import torch
    p = knn_kernel_graph(2000, 15, 40, 20, seed=14)
    direct, _ = run_squared(handle, p, b_offset=1)
    got = run_plan_squared(handle, p, b_offset=1)
    assert np.array_equal(_bits(got[:, :p.n]), _bits(direct[:, :p.n]))
    # a plan made for a non-square structure is rejected
    q = uniform_rows(100, 80, 8, 3, seed=15, dtype=np.float32)
    rp = torch.from_numpy(q.row_ptr).cuda()
    plan = cs.spmm_plan_create(handle.ptr, rp.data_ptr(), q.m, q.k, q.n, 4)
    try:
        d = torch.zeros(16, dtype=torch.float32, device="cuda")
        s = cs.spmm_plan_csr_squared_f32(plan, 1.0, d.data_ptr(), d.data_ptr(), d.data_ptr(),
                                         d.data_ptr(), q.n, 0.0, d.data_ptr(), q.n, check=False)
        assert s == cs.SPMM_ERR_INVALID_ARGUMENT
        s = cs.spmm_plan_csr_squared_f64(plan, 1.0, d.data_ptr(), d.data_ptr(), d.data_ptr(),
                                         d.data_ptr(), q.n, 0.0, d.data_ptr(), q.n, check=False)
        assert s == cs.SPMM_ERR_INVALID_ARGUMENT
    finally:
        cs.spmm_plan_destroy(plan)


def test_plan_class_squared(handle):
    """The Python Plan wrapper's chain, in breadth-first row order."""
    import torch
    p = knn_kernel_graph(3000, 15, 40, 20, seed=16)
    dev = torch.device("cuda")
    rp = torch.from_numpy(p.row_ptr).to(dev)
    ci = torch.from_numpy(p.col_idx).to(dev)
    va = torch.from_numpy(p.values).to(dev)
    B = torch.from_numpy(p.B).to(dev)
    C = torch.empty(p.m, p.n, dtype=torch.float32, device=dev)
    plan = cs.Plan(handle, rp, p.k, p.n, torch.float32)
    try:
        assert plan.order_rows(rp, ci)
        plan.squared(p.alpha, rp, ci, va, B, p.beta, C)
        torch.cuda.synchronize()
    finally:
        plan.close()
    direct, _ = run_squared(handle, p)
    assert np.array_equal(C.cpu().numpy().view(np.uint32), direct[:, :p.n].view(np.uint32))

"""GPU tests of analysis reuse: a plan bins the rows of one sparsity structure
once, and its products must equal the direct products bit for bit (both run
the same kernels on the same bins), stay in parity with the oracle, and remain
right when values, B and C change between calls on the same plan."""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
from gpu_helpers import _dev, assert_parity, run_problem
from synth import knn_kernel_graph, laplacian_2d, power_law, rng, uniform_rows
from synth.workloads import tiny_uniform

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


def _plan_run(handle, plan, p, b_offset=0):
    """One product through the plan on the problem's arrays; returns C (numpy)."""
    import torch
    dev = torch.device("cuda")
    # empty arrays get a 1-element buffer: a valid address, as for direct products
    rp, ci, va = (_dev(a, torch, dev) for a in (p.row_ptr, p.col_idx, p.values))
    Bd = _dev(np.concatenate([np.zeros(b_offset, p.B.dtype), p.B.ravel()]), torch, dev)
    C0 = p.C0 if p.C0 is not None else np.full((p.m, p.ldc), np.nan, p.values.dtype)
    Cd = torch.from_numpy(np.ascontiguousarray(C0).copy()).to(dev)
    st = torch.cuda.current_stream().cuda_stream
    fn = cs.spmm_plan_csr_f32 if p.values.dtype == np.float32 else cs.spmm_plan_csr_f64
    fn(plan, p.alpha, rp.data_ptr(), ci.data_ptr(), va.data_ptr(),
       Bd.data_ptr() + b_offset * p.B.itemsize, p.ldb, p.beta, Cd.data_ptr(), p.ldc, st)
    torch.cuda.synchronize()
    return Cd.cpu().numpy().reshape(p.m, p.ldc)


def _make_plan(handle, p):
    import torch
    rp = torch.from_numpy(p.row_ptr).cuda()
    plan = cs.spmm_plan_create(handle.ptr, rp.data_ptr(), p.m, p.k, p.n, p.values.itemsize,
                               torch.cuda.current_stream().cuda_stream)
    return plan


def _revalue(p, seed):
    """Same structure, new values, B and C0 (as an iterative solver would see)."""
    nnz = p.values.size
    p.values = (p.values * rng.uniform(seed, 901, nnz, 0.5, 1.5)).astype(p.values.dtype)
    p.B = rng.uniform(seed, 902, p.B.size, -1.0, 1.0).reshape(p.B.shape).astype(p.B.dtype)
    if p.C0 is not None:
        p.C0 = rng.uniform(seed, 903, p.C0.size, -1.0, 1.0).reshape(p.C0.shape).astype(
            p.C0.dtype)
    return p


CASES = {
    # long rows (split across CTAs with the in-launch fixup), beta != 0
    "power_law": lambda: power_law(30_000, 30_000, 64, 600_000, 10_000, seed=5),
    # short and medium rows, beta = 0
    "knn": lambda: knn_kernel_graph(6000, 30, 100, 50, seed=1),
    # binary64, beta != 0
    "laplacian": lambda: laplacian_2d(60, 32, seed=3),
    "tiny": lambda: tiny_uniform(),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_plan_matches_direct_and_oracle(handle, name):
    p = CASES[name]()
    plan = _make_plan(handle, p)
    try:
        rows = np.unique(np.linspace(0, p.m - 1, 400).astype(np.int64))
        for it in range(3):                 # repeated products on one plan
            if it:
                p = _revalue(p, 100 + it)
            direct, _ = run_problem(handle, p)
            got = _plan_run(handle, plan, p)
            assert np.array_equal(_bits(got[:, :p.n]), _bits(direct[:, :p.n])), (name, it)
            assert_parity(p, got, rows=rows, what=f"plan {name} #{it}")
    finally:
        cs.spmm_plan_destroy(plan)


def test_plan_unaligned_b(handle):
    """B at an odd element offset: the product falls back to scalar gathers
    while the plan's bins (made for 16-byte operands) stay valid."""
    p = power_law(8000, 8000, 24, 160_000, 3000, seed=9)
    plan = _make_plan(handle, p)
    try:
        direct, _ = run_problem(handle, p, b_offset=1)
        got = _plan_run(handle, plan, p, b_offset=1)
        assert np.array_equal(_bits(got[:, :p.n]), _bits(direct[:, :p.n]))
        assert_parity(p, got, rows=np.arange(0, p.m, 37), what="plan unaligned B")
    finally:
        cs.spmm_plan_destroy(plan)


def test_plan_alpha_zero_scales(handle):
    p = uniform_rows(500, 300, 20, 7, seed=11, dtype=np.float64, alpha=0.0, beta=-2.0)
    plan = _make_plan(handle, p)
    try:
        got = _plan_run(handle, plan, p)
        assert np.array_equal(got[:, :p.n], -2.0 * p.C0[:, :p.n])
    finally:
        cs.spmm_plan_destroy(plan)


def test_plan_errors(handle):
    import torch
    p = uniform_rows(100, 50, 8, 3, seed=12, dtype=np.float32)
    plan = _make_plan(handle, p)
    try:
        d = torch.zeros(16, dtype=torch.float64, device="cuda")
        # a plan made for 4-byte elements rejects a binary64 product
        s = cs.spmm_plan_csr_f64(plan, 1.0, d.data_ptr(), d.data_ptr(), d.data_ptr(),
                                 d.data_ptr(), p.n, 0.0, d.data_ptr(), p.n, check=False)
        assert s == 1          # SPMM_ERR_INVALID_ARGUMENT
        # leading dimension below n
        s = cs.spmm_plan_csr_f32(plan, 1.0, d.data_ptr(), d.data_ptr(), d.data_ptr(),
                                 d.data_ptr(), p.n - 1, 0.0, d.data_ptr(), p.n, check=False)
        assert s != 0
    finally:
        cs.spmm_plan_destroy(plan)
    cs.spmm_plan_destroy(None)               # NULL is accepted
    with pytest.raises(cs.SpmmError):
        cs.spmm_plan_create(handle.ptr, 0, 10, 10, 4, 3)     # bad element size


def test_plan_empty(handle):
    import torch
    rp = torch.zeros(1, dtype=torch.int32, device="cuda")
    plan = cs.spmm_plan_create(handle.ptr, rp.data_ptr(), 0, 5, 4, 4)
    cs.spmm_plan_destroy(plan)
    # rows with no entries at all: C = beta * C
    p = uniform_rows(64, 40, 12, 0, seed=13, dtype=np.float32, beta=0.5)
    plan = _make_plan(handle, p)
    try:
        got = _plan_run(handle, plan, p)
        assert_parity(p, got, what="plan empty rows")
    finally:
        cs.spmm_plan_destroy(plan)


def test_plan_wrapper_class(handle):
    import torch
    p = knn_kernel_graph(2000, 15, 40, 20, seed=14)
    dev = torch.device("cuda")
    rp = torch.from_numpy(p.row_ptr).to(dev)
    ci = torch.from_numpy(p.col_idx).to(dev)
    va = torch.from_numpy(p.values).to(dev)
    B = torch.from_numpy(p.B).to(dev)
    C = torch.empty(p.m, p.n, dtype=torch.float32, device=dev)
    plan = cs.Plan(handle, rp, p.k, p.n, torch.float32)
    plan(p.alpha, rp, ci, va, B, p.beta, C)
    torch.cuda.synchronize()
    plan.close()
    assert_parity(p, C.cpu().numpy(), what="Plan class")


def test_plan_outlives_its_handle():
    """Destroying a plan after its handle is allowed (the plan keeps no
    reference the destruction needs)."""
    import torch
    h = cs.Handle(0)
    p = uniform_rows(300, 200, 8, 5, seed=15, dtype=np.float32)
    rp = torch.from_numpy(p.row_ptr).cuda()
    plan = cs.spmm_plan_create(h.ptr, rp.data_ptr(), p.m, p.k, p.n, 4,
                               torch.cuda.current_stream().cuda_stream)
    h.close()
    cs.spmm_plan_destroy(plan)


def _order_plan_rows(plan, p):
    import torch
    rp = torch.from_numpy(p.row_ptr).cuda()
    ci = (torch.from_numpy(p.col_idx).cuda() if p.col_idx.size
          else torch.zeros(1, dtype=torch.int32, device="cuda"))
    cs.spmm_plan_order_rows(plan, rp.data_ptr(), ci.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", sorted(CASES))
def test_plan_row_order_keeps_results(handle, name):
    """Processing the rows in breadth-first order changes when each row is
    computed, not how: the products stay bit for bit those of the direct call,
    including short, medium and long rows, and across new values."""
    p = CASES[name]()
    plan = _make_plan(handle, p)
    try:
        _order_plan_rows(plan, p)
        rows = np.unique(np.linspace(0, p.m - 1, 300).astype(np.int64))
        for it in range(2):
            if it:
                p = _revalue(p, 200 + it)
            direct, _ = run_problem(handle, p)
            got = _plan_run(handle, plan, p)
            assert np.array_equal(_bits(got[:, :p.n]), _bits(direct[:, :p.n])), (name, it)
            assert_parity(p, got, rows=rows, what=f"ordered plan {name} #{it}")
    finally:
        cs.spmm_plan_destroy(plan)


def test_plan_row_order_medium_rows_and_unaligned(handle):
    """Medium rows (their entry prefix is rebuilt after the reorder) on a
    narrow geometry, and unaligned B through an ordered plan."""
    p = power_law(20_000, 20_000, 8, 400_000, 900, seed=21)
    plan = _make_plan(handle, p)
    try:
        _order_plan_rows(plan, p)
        for off in (0, 1):
            direct, _ = run_problem(handle, p, b_offset=off)
            got = _plan_run(handle, plan, p, b_offset=off)
            assert np.array_equal(_bits(got[:, :p.n]), _bits(direct[:, :p.n])), off
    finally:
        cs.spmm_plan_destroy(plan)


def test_plan_row_order_errors(handle):
    import torch
    p = uniform_rows(100, 100, 8, 3, seed=22, dtype=np.float32)
    plan = _make_plan(handle, p)
    try:
        bad = p.row_ptr.copy()
        bad[0] = 1
        rp = torch.from_numpy(bad).cuda()
        ci = torch.from_numpy(p.col_idx).cuda()
        st = torch.cuda.current_stream().cuda_stream
        assert cs.library().spmm_plan_order_rows(plan, rp.data_ptr(), ci.data_ptr(),
                                                 st) == cs.SPMM_ERR_INVALID_CSR
        assert cs.library().spmm_plan_order_rows(plan, None, ci.data_ptr(),
                                                 st) == cs.SPMM_ERR_NULL_POINTER
        assert cs.library().spmm_plan_order_rows(None, rp.data_ptr(), ci.data_ptr(),
                                                 st) == cs.SPMM_ERR_INVALID_ARGUMENT
        # the plan is untouched by the rejected calls
        direct, _ = run_problem(handle, p)
        got = _plan_run(handle, plan, p)
        assert np.array_equal(_bits(got[:, :p.n]), _bits(direct[:, :p.n]))
    finally:
        cs.spmm_plan_destroy(plan)


def test_plan_class_order_rows(handle):
    import torch
    p = knn_kernel_graph(3000, 15, 40, 20, seed=23)
    dev = torch.device("cuda")
    rp = torch.from_numpy(p.row_ptr).to(dev)
    ci = torch.from_numpy(p.col_idx).to(dev)
    va = torch.from_numpy(p.values).to(dev)
    B = torch.from_numpy(p.B).to(dev)
    C = torch.empty(p.m, p.n, dtype=torch.float32, device=dev)
    plan = cs.Plan(handle, rp, p.k, p.n, torch.float32)
    assert plan.order_rows(rp, ci)              # a kNN pattern: the reorder is kept
    plan(p.alpha, rp, ci, va, B, p.beta, C)
    torch.cuda.synchronize()
    plan.close()
    assert_parity(p, C.cpu().numpy(), what="Plan class, ordered rows")


@pytest.mark.parametrize("name,want", [("knn", True), ("power_law", False), ("tiny", False)])
def test_plan_row_order_auto(handle, name, want):
    """The automatic reorder keeps the breadth-first order only where it
    raises B-row reuse (a kNN kernel pattern), leaves uniformly random
    columns in their order, and either way the products equal the direct
    call's bits."""
    import torch
    p = CASES[name]()
    plan = _make_plan(handle, p)
    try:
        rp = torch.from_numpy(p.row_ptr).cuda()
        ci = torch.from_numpy(p.col_idx).cuda()
        applied = cs.spmm_plan_order_rows_auto(plan, rp.data_ptr(), ci.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
        assert applied is want, name
        direct, _ = run_problem(handle, p)
        got = _plan_run(handle, plan, p)
        assert np.array_equal(_bits(got[:, :p.n]), _bits(direct[:, :p.n])), name
    finally:
        cs.spmm_plan_destroy(plan)

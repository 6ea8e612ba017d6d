"""Products captured in CUDA graphs and replayed.  Launch-bound calls (small
products, chains of calls in an iterative solver) are meant to run this way:
the handle's scratch is sized first (spmm_reserve, or one call outside the
capture), so nothing allocates or synchronises inside the capture, and the
programmatic dependent launches between the library's kernels are captured as
graph edges."""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
import oracle
from gpu_helpers import assert_parity
from synth import knn_kernel_graph, power_law
from synth.fw import fw_random
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


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("make", [tiny_uniform,
                                  lambda: power_law(30_000, 30_000, 64, 600_000, 10_000, seed=5)])
def test_product_graph_replays(handle, make):
    import torch
    p = make()
    rp, ci, va, B = _t(p.row_ptr), _t(p.col_idx), _t(p.values), _t(p.B)
    C = _t(p.C0)
    C0 = C.clone()
    h = handle
    h.reserve(p.m, p.n, p.values.itemsize)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            cs.spmm(h, p.alpha, rp, ci, va, p.k, B, p.beta, C)
    # replays on new B and C contents (static buffers, new values)
    rng = np.random.default_rng(0)
    for it in range(3):
        newB = rng.standard_normal(p.B.shape).astype(p.B.dtype)
        B.copy_(_t(newB))
        C.copy_(C0)
        g.replay()
        torch.cuda.synchronize()
        q = type(p)(**{**p.__dict__, "B": newB})
        assert_parity(q, C.cpu().numpy(), rows=np.arange(0, p.m, 7), what=f"graph replay {it}")


def test_chain_and_scan_graph(handle):
    import torch
    p = knn_kernel_graph(3000, 20, 64, 30, seed=2)
    rp, ci, va, B = _t(p.row_ptr), _t(p.col_idx), _t(p.values), _t(p.B)
    C = torch.full((p.m, p.n), float("nan"), device="cuda")
    f = fw_random(2000, 60, 12, seed=3)
    mats = [tuple(_t(x) for x in m) for m in (f.k2b, f.t1, f.t2, f.b)]
    # one call of each outside the capture sizes the scratch
    cs.spmm_squared(handle, p.alpha, rp, ci, va, B, p.beta, C)
    cs.fw_argmin(handle, f.k, *mats)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            cs.spmm_squared(handle, p.alpha, rp, ci, va, B, p.beta, C)
            mv, mi, gap = cs.fw_argmin(handle, f.k, *mats)
    C.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    ref, bound = oracle.spmm_squared(p.m, p.n, p.alpha, p.row_ptr, p.col_idx, p.values, p.B,
                                     p.ldb, p.beta, None, p.ldc)
    err = np.abs(C.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= 2e-5 * bound)
    r = oracle.fw_argmin(f.n, f.k, f.k2b, f.t1, f.t2, f.b)
    assert np.all(np.abs(mv.cpu().numpy() - r["min_val"]) <= 1e-5 * r["col_scale"])
    assert abs(float(gap.item()) - r["gap"]) <= 1e-5 * r["gap_bound"]

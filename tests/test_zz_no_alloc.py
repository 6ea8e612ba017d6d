"""spmm_csr_f32_noalloc: the product for callers that cannot allocate device
memory (its scratch is a fixed array inside the library).  Two calls in a row
through the C ABI must match the handle-based spmm_csr_f32 on the same inputs,
within the fp32 tolerance of the other parity tests.  This file is collected
last so that a failure here never hides another test's result."""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
import oracle
from synth import knn_kernel_graph, power_law

pytestmark = pytest.mark.gpu


def _run(fn_kind, handle, p):
    import torch
    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    rp, ci, va, B = t(p.row_ptr), t(p.col_idx), t(p.values), t(p.B)
    C = t(p.C0.copy()) if p.C0 is not None else torch.full((p.m, p.ldc), float("nan"), device=dev)
    st = torch.cuda.current_stream().cuda_stream
    args = (p.alpha, rp.data_ptr(), ci.data_ptr(), va.data_ptr(), p.m, p.k, B.data_ptr(), p.ldb,
            p.n, p.beta, C.data_ptr(), p.ldc, st)
    if fn_kind == "noalloc":
        cs.spmm_csr_f32_noalloc(*args)
    else:
        cs.spmm_csr_f32(handle.ptr, *args)
    torch.cuda.synchronize()
    return C.cpu().numpy()


def test_noalloc_matches_handle_path_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()
    problems = [power_law(20_000, 20_000, 48, 400_000, 8_000, seed=31),   # long rows + fixup
                knn_kernel_graph(5_000, 30, 100, 50, seed=32)]            # beta == 0, NaN C
    h = cs.Handle(0)
    try:
        for p in problems:                       # two calls in a row, different shapes
            want = _run("handle", h, p)
            got = _run("noalloc", h, p)
            _, bound = oracle.spmm_problem(p)
            diff = np.abs(got[:, :p.n].astype(np.float64) - want[:, :p.n].astype(np.float64))
            assert np.all(np.isfinite(got[:, :p.n]))
            assert np.all(diff <= 1e-5 * bound), f"{p.name}: max diff {diff.max()}"
    finally:
        h.close()


def test_noalloc_rejects_oversize():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    C = torch.zeros(4, 4, device="cuda")
    s = cs.spmm_csr_f32_noalloc(1.0, 0, 0, 0, 600_000, 10, 0, 4, 4, 0.0, C.data_ptr(), 4,
                                check=False)
    assert s == cs._lib.SPMM_ERR_TOO_LARGE
    s = cs.spmm_csr_f32_noalloc(1.0, 0, 0, 0, 4, 10, 0, 1024, 1024, 0.0, C.data_ptr(), 1024,
                                check=False)
    assert s == cs._lib.SPMM_ERR_TOO_LARGE

"""spmm_csr_f32_noalloc: the product for callers that cannot allocate device
memory (its scratch is a fixed array inside the library).

It takes the handle path's plan and runs its kernels, so two calls in a row
through the C ABI must give the handle-based spmm_csr_f32's results bit for
bit, and both must agree with the oracle element by element within the fp32
tolerance of the other parity tests.  Cases: long rows with the fixup, beta
== 0 over a NaN C, an unaligned B (scalar geometry), and a product at the
array's limits (m = 524,288 rows, n = 512 columns, long rows present).  This
file is collected last so that a failure here never hides another test's
result."""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
from gpu_helpers import assert_parity
from synth import knn_kernel_graph, power_law, rng

pytestmark = pytest.mark.gpu


def _run(fn_kind, handle, p, b_offset=0):
    import torch
    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    rp, ci, va = t(p.row_ptr), t(p.col_idx), t(p.values)
    Bflat = np.concatenate([np.zeros(b_offset, p.B.dtype), p.B.ravel()]) if b_offset else p.B
    B = t(Bflat)
    C = t(p.C0.copy()) if p.C0 is not None else torch.full((p.m, p.ldc), float("nan"), device=dev)
    st = torch.cuda.current_stream().cuda_stream
    args = (p.alpha, rp.data_ptr(), ci.data_ptr(), va.data_ptr(), p.m, p.k,
            B.data_ptr() + 4 * b_offset, p.ldb, p.n, p.beta, C.data_ptr(), p.ldc, st)
    if fn_kind == "noalloc":
        cs.spmm_csr_f32_noalloc(*args)
    else:
        cs.spmm_csr_f32(handle.ptr, *args)
    torch.cuda.synchronize()
    return C.cpu().numpy()


def _checked_rows(p, sample, seed):
    lens = np.diff(p.row_ptr)
    big = np.flatnonzero(lens > 32)
    pick = np.floor(rng.uniform(seed, 93, sample) * p.m).astype(np.int64)
    return np.unique(np.concatenate([big, pick, [0, p.m - 1]]))


def _compare(h, p, rows=None, b_offset=0):
    want = _run("handle", h, p, b_offset)
    for call in range(2):                       # two calls in a row share the array
        got = _run("noalloc", h, p, b_offset)
        assert np.array_equal(got[:, :p.n].view(np.uint32), want[:, :p.n].view(np.uint32)), \
            f"{p.name}: call {call} differs from spmm_csr_f32"
    assert_parity(p, got, rows=rows, what=f"{p.name} (no-allocation entry point)")


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


def test_noalloc_matches_handle_path_and_oracle(handle):
    p = power_law(20_000, 20_000, 48, 400_000, 8_000, seed=31)           # long rows + fixup
    _compare(handle, p)
    q = knn_kernel_graph(5_000, 30, 100, 50, seed=32)                     # beta == 0, NaN C
    _compare(handle, q)


def test_noalloc_unaligned_b(handle):
    p = power_law(20_000, 20_000, 40, 300_000, 6_000, seed=33, beta=0.5)
    _compare(handle, p, b_offset=1)


def test_noalloc_at_its_limits(handle):
    """m = 524,288 and n = 512 (the array's limits) with long rows, k small
    so that B stays modest; beta == 0 over a NaN C."""
    p = power_law(524_288, 16_384, 512, 2_000_000, 3_000, seed=34, beta=0.0,
                  name="noalloc_limits")
    assert np.diff(p.row_ptr).max() >= 1024
    _compare(handle, p, rows=_checked_rows(p, 2_000, 5))


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

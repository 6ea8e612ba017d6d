"""The ILU(0) wait-timeout status, reached without a fault.

The factorisation's persistent kernel waits for queued rows with bounded
polls; a wait that runs out sets SPMM_ILU0_WAIT_TIMEOUT in the status word
and the kernel returns (the page's `ilu0_gpu` reads a status word back the
same way; oxicuda preconditioner, ilu0.rs).  Valid input never runs out, so
this test uses a variant of the library built with two test-only macros:
the last row is given one dependency that no row counts down (it is never
queued), and the poll limit is small.  Every other row must then be
factored exactly as the oracle factors it, the last row must be left as it
was, the status must read 2, and the GPU must go on answering: a product on
the regular library follows and is checked against the oracle."""
import ctypes
import os
import time

import numpy as np
import pytest

import csr_spmm_gb300 as cs
import oracle
from csr_spmm_gb300 import _lib
from csr_spmm_gb300 import build as csb
from gpu_helpers import assert_parity, run_problem
from synth import laplacian_2d, uniform_rows

pytestmark = pytest.mark.gpu

VARIANT = os.path.join(csb.LIB_DIR, "variants", "libcsrspmm_ilu0_withheld.so")
FLAGS = ("-DSPMM_ILU0_TEST_WITHHOLD_LAST_ROW=1", "-DSPMM_ILU0_SPIN_LIMIT=16384")


@pytest.fixture(scope="module")
def variant():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    path = csb.build(extra_flags=FLAGS, out=VARIANT, flag_units=("spmm_ilu0.cu",))
    return _lib.load_library(path)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_wait_timeout_status_and_recovery(variant, dtype):
    import torch
    dev = torch.device("cuda")
    p = laplacian_2d(40, 1, seed=3)
    n, nnz = p.m, p.nnz
    vals = p.values.astype(dtype)
    rp = torch.from_numpy(p.row_ptr).to(dev)
    ci = torch.from_numpy(p.col_idx).to(dev)
    v = torch.from_numpy(vals.copy()).to(dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    h = ctypes.c_void_p()
    assert variant.spmm_create(ctypes.byref(h), 0) == 0
    try:
        fn = variant.spmm_ilu0_f64 if dtype == np.float64 else variant.spmm_ilu0_f32
        t0 = time.perf_counter()
        s = fn(h, n, nnz, rp.data_ptr(), ci.data_ptr(), v.data_ptr(), None, status.data_ptr(),
               torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        variant.spmm_destroy(h)
    assert s == _lib.SPMM_OK
    assert int(status.item()) == 2, "the withheld row's wait should have run out"
    assert elapsed < 30.0
    got = v.cpu().numpy()
    want, _ = oracle.ilu0(p.row_ptr, p.col_idx, vals.copy())
    last = slice(int(p.row_ptr[n - 1]), int(p.row_ptr[n]))
    # rows 0 .. n-2 depend only on lower-numbered rows: all final, bit for bit
    assert np.array_equal(got[: last.start].view(np.uint8), want[: last.start].view(np.uint8))
    # the withheld row was never factored
    assert np.array_equal(got[last].view(np.uint8), vals[last].view(np.uint8))

    # the context is intact: a product on the regular library follows
    h2 = cs.Handle(0)
    try:
        q = uniform_rows(3000, 3000, 40, 9, seed=71, beta=0.5)
        out, st = run_problem(h2, q)
        assert st == _lib.SPMM_OK
        assert_parity(q, out, what="product after the timed-out factorisation")
    finally:
        h2.close()

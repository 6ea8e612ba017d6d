"""The torch binding's argument checks, on the host (no GPU).

The wrappers hand raw addresses to the C library, which takes them as device
memory of the handle's GPU.  Each wrapper must therefore refuse, before any
library call or CUDA query, a tensor that is not on the GPU, CSR arrays of
different lengths, and dense operands smaller than the product.
"""
import types

import numpy as np
import pytest

import csr_spmm_gb300 as cs

torch = pytest.importorskip("torch")

FAKE = types.SimpleNamespace(ptr=None, device=0)   # never reaches the library


def _csr(m=4, k=4, per_row=2, dtype=torch.float32):
    rp = torch.arange(0, per_row * (m + 1), per_row, dtype=torch.int32)
    ci = torch.tensor(np.tile(np.arange(per_row) % k, m), dtype=torch.int32)
    va = torch.ones(m * per_row, dtype=dtype)
    return rp, ci, va


def test_host_tensors_are_refused_by_every_wrapper():
    rp, ci, va = _csr()
    B = torch.zeros(4, 3)
    C = torch.zeros(4, 3)
    with pytest.raises(ValueError, match="CUDA tensor"):
        cs.spmm(FAKE, 1.0, rp, ci, va, 4, B, 0.0, C)
    with pytest.raises(ValueError, match="CUDA tensor"):
        cs.spmm_squared(FAKE, 1.0, rp, ci, va, B, 0.0, C)
    with pytest.raises(ValueError, match="CUDA tensor"):
        cs.fw_argmin(FAKE, 4, (rp, ci, va), (rp, ci, va), (rp, ci, va), (rp, ci, va))
    with pytest.raises(ValueError, match="CUDA tensor"):
        cs.ilu0(FAKE, rp, ci, va.clone())
    with pytest.raises(ValueError, match="CUDA tensor"):
        cs.Plan(FAKE, rp, 4, 3, torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        cs.csr_check(FAKE, rp, ci, 4)


def test_csr_arrays_of_different_lengths_are_refused():
    rp, ci, va = _csr()
    B = torch.zeros(4, 3)
    C = torch.zeros(4, 3)
    short = va[:-1].clone()
    with pytest.raises(ValueError, match="same number of entries"):
        cs.spmm(FAKE, 1.0, rp, ci, short, 4, B, 0.0, C)
    with pytest.raises(ValueError, match="same number of entries"):
        cs.spmm_squared(FAKE, 1.0, rp, ci, short, B, 0.0, C)
    with pytest.raises(ValueError, match="same number of entries"):
        cs.fw_argmin(FAKE, 4, (rp, ci, short), (rp, ci, va), (rp, ci, va), (rp, ci, va))
    with pytest.raises(ValueError, match="same number of entries"):
        cs.ilu0(FAKE, rp, ci, short)


def test_dense_operand_checks_of_the_direct_call():
    rp, ci, va = _csr()
    with pytest.raises(ValueError, match="shape mismatch"):
        cs.spmm(FAKE, 1.0, rp, ci, va, 4, torch.zeros(3, 3), 0.0, torch.zeros(4, 3))
    with pytest.raises(ValueError, match="unit column stride"):
        cs.spmm(FAKE, 1.0, rp, ci, va, 4, torch.zeros(3, 4).t(), 0.0, torch.zeros(4, 3))
    with pytest.raises(TypeError, match="one dtype"):
        cs.spmm(FAKE, 1.0, rp, ci, va, 4, torch.zeros(4, 3, dtype=torch.float64), 0.0,
                torch.zeros(4, 3))
    with pytest.raises(TypeError, match="int32"):
        cs.spmm(FAKE, 1.0, rp.long(), ci, va, 4, torch.zeros(4, 3), 0.0, torch.zeros(4, 3))


def _plan(m=4, k=4, n=3, dtype=torch.float32):
    """A Plan object with its dimensions set and no library plan behind it."""
    pl = object.__new__(cs.Plan)
    pl.handle, pl.m, pl.k, pl.n, pl.dtype, pl.ptr = FAKE, m, k, n, dtype, None
    return pl


def test_plan_checks_its_dense_operands_against_the_plan():
    rp, ci, va = _csr()
    pl = _plan()
    with pytest.raises(ValueError, match="smaller than"):
        pl(1.0, rp, ci, va, torch.zeros(3, 3), 0.0, torch.zeros(4, 3))     # B rows < k
    with pytest.raises(ValueError, match="smaller than"):
        pl(1.0, rp, ci, va, torch.zeros(4, 2), 0.0, torch.zeros(4, 3))     # B columns < n
    with pytest.raises(ValueError, match="smaller than"):
        pl(1.0, rp, ci, va, torch.zeros(4, 3), 0.0, torch.zeros(3, 3))     # C rows < m
    with pytest.raises(ValueError, match="smaller than"):
        pl.squared(1.0, rp, ci, va, torch.zeros(4, 3), 0.0, torch.zeros(4, 2))
    with pytest.raises(TypeError, match="one dtype"):
        pl(1.0, rp, ci, va, torch.zeros(4, 3, dtype=torch.float64), 0.0,
           torch.zeros(4, 3, dtype=torch.float64))
    with pytest.raises(TypeError, match="plan's dtype"):
        pl(1.0, rp, ci, va.double(), torch.zeros(4, 3), 0.0, torch.zeros(4, 3))
    # wider operands than the product (leading dimensions above n) pass the
    # dense checks and stop at the host tensors
    with pytest.raises(ValueError, match="CUDA tensor"):
        pl(1.0, rp, ci, va, torch.zeros(4, 8)[:, :5], 0.0, torch.zeros(4, 8))


def test_plan_refuses_unsupported_dtypes():
    rp, _, _ = _csr()
    with pytest.raises(TypeError, match="float32 or float64"):
        cs.Plan(FAKE, rp, 4, 3, torch.float16)
    with pytest.raises(TypeError, match="int32"):
        cs.Plan(FAKE, rp.long(), 4, 3, torch.float32)


class _AsCuda(torch.Tensor):
    """A host tensor that reports itself as on cuda:0, so that the wrappers'
    marshalling runs on the host against recorded (never executed) calls."""

    @property
    def is_cuda(self):
        return True

    @property
    def device(self):
        return torch.device("cuda", 0)


def _cuda(t):
    return torch.Tensor._make_subclass(_AsCuda, t)


@pytest.fixture
def recorded(monkeypatch):
    calls = []

    def recorder(name):
        def fn(*args, **kw):
            calls.append((name, args, kw))
            return (0, 0) if name == "spmm_csr_check" else 0
        return fn

    for name in ("spmm_csr_f32", "spmm_csr_f64", "spmm_csr_squared_f32", "spmm_csr_squared_f64",
                 "spmm_plan_csr_f32", "spmm_plan_csr_f64", "spmm_plan_csr_squared_f32",
                 "spmm_plan_csr_squared_f64", "spmm_plan_order_rows", "spmm_plan_order_rows_auto",
                 "spmm_csr_check"):
        monkeypatch.setattr(cs, name, recorder(name))
    monkeypatch.setattr(torch.cuda, "current_stream",
                        lambda *a: types.SimpleNamespace(cuda_stream=77))
    return calls


def test_direct_calls_pass_addresses_and_leading_dimensions(recorded):
    rp, ci, va = (_cuda(x) for x in _csr(m=5, k=6, per_row=3))
    B = _cuda(torch.zeros(6, 10))[:, :4]           # k x n = 6 x 4, ldb 10
    C = _cuda(torch.zeros(5, 7))[:, :4]            # m x n = 5 x 4, ldc 7
    h = types.SimpleNamespace(ptr=1234, device=0)
    cs.spmm(h, 1.5, rp, ci, va, 6, B, -0.5, C)
    name, args, _ = recorded[-1]
    assert name == "spmm_csr_f32"
    assert args == (1234, 1.5, rp.data_ptr(), ci.data_ptr(), va.data_ptr(), 5, 6, B.data_ptr(),
                    10, 4, -0.5, C.data_ptr(), 7, 77)
    rq, cq, vq = (_cuda(x) for x in _csr(m=6, k=6, per_row=2, dtype=torch.float64))
    Bq = _cuda(torch.zeros(6, 3, dtype=torch.float64))
    Cq = _cuda(torch.zeros(6, 3, dtype=torch.float64))
    cs.spmm_squared(h, 2.0, rq, cq, vq, Bq, 0.0, Cq)
    name, args, _ = recorded[-1]
    assert name == "spmm_csr_squared_f64"
    assert args == (1234, 2.0, rq.data_ptr(), cq.data_ptr(), vq.data_ptr(), 6, Bq.data_ptr(), 3,
                    3, 0.0, Cq.data_ptr(), 3, 77)
    assert cs.csr_check(h, rp, ci, 6) == 0
    name, args, _ = recorded[-1]
    assert name == "spmm_csr_check"
    assert args == (1234, rp.data_ptr(), ci.data_ptr(), 5, 6, 15, 77)


def test_plan_calls_pass_addresses_and_leading_dimensions(recorded):
    rp, ci, va = (_cuda(x) for x in _csr(m=4, k=4, per_row=2))
    pl = _plan(m=4, k=4, n=3)
    pl.ptr = 99
    B = _cuda(torch.zeros(4, 8))[:, :5]            # wider than n: ldb 8
    C = _cuda(torch.zeros(4, 3))
    pl(1.0, rp, ci, va, B, 0.25, C)
    name, args, _ = recorded[-1]
    assert name == "spmm_plan_csr_f32"
    assert args == (99, 1.0, rp.data_ptr(), ci.data_ptr(), va.data_ptr(), B.data_ptr(), 8, 0.25,
                    C.data_ptr(), 3, 77)
    pl.squared(1.0, rp, ci, va, B, 0.0, C)
    assert recorded[-1][0] == "spmm_plan_csr_squared_f32"
    assert pl.order_rows(rp, ci) == 0 and recorded[-1][0] == "spmm_plan_order_rows_auto"
    assert pl.order_rows(rp, ci, automatic=False) is True
    assert recorded[-1][1] == (99, rp.data_ptr(), ci.data_ptr(), 77)
    pl.ptr = None


def test_tensors_on_another_gpu_or_with_gaps_are_refused(recorded):
    rp, ci, va = (_cuda(x) for x in _csr())
    B = _cuda(torch.zeros(4, 3))
    C = _cuda(torch.zeros(4, 3))
    with pytest.raises(ValueError, match="handle is on cuda:1"):
        cs.spmm(types.SimpleNamespace(ptr=1, device=1), 1.0, rp, ci, va, 4, B, 0.0, C)
    gappy = _cuda(torch.ones(16)[::2])
    with pytest.raises(ValueError, match="contiguous"):
        cs.spmm(types.SimpleNamespace(ptr=1, device=0), 1.0, rp, ci, gappy, 4, B, 0.0, C)
    assert recorded == []

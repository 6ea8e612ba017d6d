"""GB300-native CSR SpMM: C = alpha * A * B + beta * C on one sm_103a GPU.

The product runs in hand-written CUDA kernels behind the C ABI of
``include/csr_spmm.h`` (library ``csr_spmm_gb300/lib/libcsrspmm.so``).  This
package is the Python face of that ABI:

* :mod:`csr_spmm_gb300._lib` -- the C entry points under their C names
  (``spmm_create``, ``spmm_csr_f32``, ...), pointers as integers;
* :class:`Handle` and :func:`spmm` -- the same call taking torch CUDA tensors
  (PyTorch supplies device memory and the current stream only).

There is no CPU path: without the built library every call raises.
"""
from __future__ import annotations

from ._lib import (EXPORTED, SPMM_ERR_ALLOC, SPMM_ERR_CUDA, SPMM_ERR_DIMENSION_MISMATCH,
                   SPMM_ERR_INVALID_ARGUMENT, SPMM_ERR_INVALID_CSR, SPMM_ERR_NULL_POINTER,
                   SPMM_ERR_TOO_LARGE, SPMM_ERR_UNSUPPORTED_DEVICE, SPMM_OK, SpmmError,
                   library, spmm_create,
                   spmm_csr_check, spmm_csr_f32, spmm_csr_f32_noalloc, spmm_csr_f64,
                   spmm_destroy, spmm_get_profile, spmm_plan_create, spmm_plan_csr_f32,
                   spmm_plan_csr_f64, spmm_plan_csr_squared_f32, spmm_plan_csr_squared_f64,
                   spmm_plan_destroy, spmm_plan_order_rows,
                   spmm_row_order_bfs, spmm_set_l2_persistence, spmm_measure_fp64_fma_rate,
                   spmm_plan_order_rows_auto,
                   spmm_csr_squared_f32, spmm_csr_squared_f64, spmm_fw_argmin,
                   spmm_ilu0, ILU0_SINGULAR, ILU0_WAIT_TIMEOUT,
                   spmm_reserve, spmm_set_profiling, status_string)

__all__ = ["Handle", "spmm", "csr_check", "SpmmError", "library", "spmm_create", "spmm_destroy",
           "spmm_reserve", "spmm_csr_f32", "spmm_csr_f64", "spmm_csr_check", "status_string",
           "spmm_set_profiling", "spmm_get_profile", "spmm_csr_f32_noalloc", "spmm_plan_create",
           "spmm_plan_destroy", "spmm_set_l2_persistence", "spmm_plan_csr_f32",
           "spmm_csr_squared_f32", "spmm_csr_squared_f64", "spmm_squared",
           "spmm_fw_argmin", "fw_argmin", "spmm_ilu0", "ilu0", "Ilu0Error",
           "spmm_plan_csr_f64", "spmm_plan_order_rows", "spmm_row_order_bfs",
           "spmm_plan_csr_squared_f32", "spmm_plan_csr_squared_f64", "Plan",
           "spmm_measure_fp64_fma_rate", "spmm_plan_order_rows_auto", "EXPORTED"]


class Handle:
    """Owns one ``spmm_handle_t`` (scratch for row bins and long-row partials)."""

    def __init__(self, device: int | None = None):
        import torch
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.ptr = spmm_create(self.device)

    def reserve(self, m: int, n: int, elem_size: int) -> None:
        spmm_reserve(self.ptr, m, n, elem_size)

    def close(self) -> None:
        if self.ptr:
            spmm_destroy(self.ptr)
            self.ptr = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _ptr(t, device: int):
    """Device address of a tensor the library reads or writes (0 for None).
    Refused here, because its address would reach a kernel as device memory
    of the call's GPU: a tensor not on CUDA, a tensor on another GPU than
    the handle's, and a 1-D array whose entries are not contiguous."""
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    if t.device.index != device:
        raise ValueError(f"tensor on {t.device}, but the handle is on cuda:{device}")
    if t.dim() <= 1 and not t.is_contiguous():
        raise ValueError("1-D arrays (row_ptr, col_idx, values) must be contiguous")
    return t.data_ptr()


def _check_dense(B, C, b_rows: int, m: int, n: int, dtype) -> None:
    """B holds at least b_rows x n and C at least m x n elements, row-major with
    unit column stride, all of the values' dtype."""
    if C.dim() != 2 or B.dim() != 2 or C.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("B and C must be 2-D with unit column stride")
    if B.shape[0] < b_rows or B.shape[1] < n or C.shape[0] < m or C.shape[1] < n:
        raise ValueError(f"B {tuple(B.shape)} or C {tuple(C.shape)} smaller than the "
                         f"product's {b_rows} x {n} and {m} x {n}")
    if not (B.dtype == C.dtype == dtype):
        raise TypeError("values, B and C must share one dtype")


def spmm(handle: Handle, alpha: float, row_ptr, col_idx, values, k: int, B, beta: float, C,
         stream=None) -> None:
    """C <- alpha * A * B + beta * C, A given by CSR tensors (int32, int32, float32/64).

    ``B`` is a [k, n] CUDA tensor and ``C`` an [m, n] CUDA tensor, each with
    unit column stride (any row stride: the leading dimension).  Enqueued on
    ``stream`` (default: torch's current stream); returns without waiting.
    """
    import torch
    m = int(row_ptr.numel()) - 1
    n = int(C.shape[1])
    if C.dim() != 2 or B.dim() != 2 or C.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("B and C must be 2-D with unit column stride")
    if B.shape[0] != k or B.shape[1] != n or C.shape[0] != m:
        raise ValueError(f"shape mismatch: A {m}x{k}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    if row_ptr.dtype != torch.int32 or col_idx.dtype != torch.int32:
        raise TypeError("row_ptr and col_idx must be int32")
    if not (values.dtype == B.dtype == C.dtype):
        raise TypeError("values, B and C must share one dtype")
    if col_idx.numel() != values.numel():
        raise ValueError("col_idx and values must hold the same number of entries")
    d = handle.device
    a_rp, a_ci, a_va, a_b, a_c = (_ptr(x, d) for x in (row_ptr, col_idx, values, B, C))
    st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
    ldb = B.stride(0) if B.shape[0] > 1 else max(1, n)
    ldc = C.stride(0) if C.shape[0] > 1 else max(1, n)
    args = (handle.ptr, alpha, a_rp, a_ci, a_va, m, k, a_b, ldb, n, beta, a_c, ldc, st)
    if values.dtype == torch.float32:
        spmm_csr_f32(*args)
    elif values.dtype == torch.float64:
        spmm_csr_f64(*args)
    else:
        raise TypeError("values must be float32 or float64")


def spmm_squared(handle: Handle, alpha: float, row_ptr, col_idx, values, B, beta: float, C,
                 stream=None) -> None:
    """C <- alpha * A (A B) + beta * C for a square CSR A (the K^2 B chain).

    ``B`` and ``C`` are [m, n] CUDA tensors with unit column stride.
    Enqueued on ``stream`` (default: torch's current stream).
    """
    import torch
    m = int(row_ptr.numel()) - 1
    n = int(C.shape[1])
    if C.dim() != 2 or B.dim() != 2 or C.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("B and C must be 2-D with unit column stride")
    if tuple(B.shape) != (m, n) or C.shape[0] != m:
        raise ValueError(f"shape mismatch: A {m}x{m}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    if row_ptr.dtype != torch.int32 or col_idx.dtype != torch.int32:
        raise TypeError("row_ptr and col_idx must be int32")
    if not (values.dtype == B.dtype == C.dtype):
        raise TypeError("values, B and C must share one dtype")
    if col_idx.numel() != values.numel():
        raise ValueError("col_idx and values must hold the same number of entries")
    d = handle.device
    a_rp, a_ci, a_va, a_b, a_c = (_ptr(x, d) for x in (row_ptr, col_idx, values, B, C))
    st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
    ldb = B.stride(0) if B.shape[0] > 1 else max(1, n)
    ldc = C.stride(0) if C.shape[0] > 1 else max(1, n)
    args = (handle.ptr, alpha, a_rp, a_ci, a_va, m, a_b, ldb, n, beta, a_c, ldc, st)
    if values.dtype == torch.float32:
        spmm_csr_squared_f32(*args)
    elif values.dtype == torch.float64:
        spmm_csr_squared_f64(*args)
    else:
        raise TypeError("values must be float32 or float64")


def fw_argmin(handle: Handle, k: int, k2b, t1, t2, bmat, stream=None):
    """Frank-Wolfe gradient scan on CUDA tensors: each matrix a (row_ptr,
    col_idx, values) triple of int32 / int32 / float tensors (K2B, T2 and B
    n x k, t1 k x k).  Returns device tensors (min_val [k], min_idx [k] int32,
    gap [1]); enqueued on ``stream``."""
    import torch
    n = int(k2b[0].numel()) - 1
    dt = k2b[2].dtype
    if dt not in (torch.float32, torch.float64):
        raise TypeError("values must be float32 or float64")
    for mat, rows in ((k2b, n), (t1, k), (t2, n), (bmat, n)):
        if int(mat[0].numel()) != rows + 1 or mat[2].dtype != dt:
            raise ValueError("CSR triples must be (row_ptr [rows+1], col_idx, values) of one dtype")
        if mat[1].numel() != mat[2].numel():
            raise ValueError("col_idx and values must hold the same number of entries")
        if mat[0].dtype != torch.int32 or mat[1].dtype != torch.int32:
            raise TypeError("row_ptr and col_idx must be int32")
    d = handle.device
    mats = [tuple(_ptr(x, d) for x in m) for m in (k2b, t1, t2, bmat)]
    dev = k2b[0].device
    min_val = torch.empty(max(k, 1), dtype=dt, device=dev)
    min_idx = torch.empty(max(k, 1), dtype=torch.int32, device=dev)
    gap = torch.empty(1, dtype=dt, device=dev)
    st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
    spmm_fw_argmin(handle.ptr, n, k, *mats, _ptr(min_val, d), _ptr(min_idx, d), _ptr(gap, d),
                   f64=dt == torch.float64, stream=st)
    return min_val[:k], min_idx[:k], gap


class Ilu0Error(RuntimeError):
    """ILU(0) stopped: a zero or missing pivot, or a dependency wait ran out."""


def ilu0(handle: Handle, row_ptr, col_idx, values, with_depth: bool = False, stream=None):
    """ILU(0) in place on ``values`` (CUDA tensors of a square CSR matrix,
    columns strictly ascending within rows).  Waits for the result and raises
    Ilu0Error on failure; returns the per-row levels when ``with_depth``."""
    import torch
    n = int(row_ptr.numel()) - 1
    if row_ptr.dtype != torch.int32 or col_idx.dtype != torch.int32:
        raise TypeError("row_ptr and col_idx must be int32")
    if values.dtype not in (torch.float32, torch.float64):
        raise TypeError("values must be float32 or float64")
    if col_idx.numel() != values.numel():
        raise ValueError("col_idx and values must hold the same number of entries")
    d = handle.device
    a_rp, a_ci, a_va = (_ptr(x, d) for x in (row_ptr, col_idx, values))
    dev = values.device
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    depth = torch.empty(max(n, 1), dtype=torch.int32, device=dev) if with_depth else None
    st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
    spmm_ilu0(handle.ptr, n, int(values.numel()), a_rp, a_ci, a_va, _ptr(depth, d),
              _ptr(status, d), f64=values.dtype == torch.float64, stream=st)
    code = int(status.item())                          # synchronises
    if code:
        why = "zero or missing pivot" if code & ILU0_SINGULAR else "a dependency wait ran out"
        raise Ilu0Error(f"ILU(0) failed: {why} (status {code})")
    return depth[:n] if with_depth else None


class Plan:
    """The row bins of one sparsity structure, reused by repeated products."""

    def __init__(self, handle: Handle, row_ptr, k: int, n: int, dtype, stream=None):
        import torch
        self.handle = handle
        self.m = int(row_ptr.numel()) - 1
        self.k, self.n = int(k), int(n)
        self.dtype = dtype
        if dtype not in (torch.float32, torch.float64):
            raise TypeError("dtype must be float32 or float64")
        if row_ptr.dtype != torch.int32:
            raise TypeError("row_ptr must be int32")
        es = 4 if dtype == torch.float32 else 8
        a_rp = _ptr(row_ptr, handle.device)
        st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        self.ptr = spmm_plan_create(handle.ptr, a_rp, self.m, self.k, self.n, es, st)

    def order_rows(self, row_ptr, col_idx, stream=None, automatic=True) -> bool:
        """Process rows in breadth-first order of A's pattern: where that raises
        B-row reuse (spmm_plan_order_rows_auto, the default), or always
        (automatic=False, spmm_plan_order_rows).  Returns whether the order
        was changed."""
        import torch
        d = self.handle.device
        a_rp, a_ci = _ptr(row_ptr, d), _ptr(col_idx, d)
        st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        if automatic:
            return spmm_plan_order_rows_auto(self.ptr, a_rp, a_ci, st)
        spmm_plan_order_rows(self.ptr, a_rp, a_ci, st)
        return True

    def __call__(self, alpha, row_ptr, col_idx, values, B, beta, C, stream=None) -> None:
        """C <- alpha * A * B + beta * C with A's structure from the plan."""
        import torch
        _check_dense(B, C, self.k, self.m, self.n, self.dtype)
        if values.dtype != self.dtype:
            raise TypeError("values must have the plan's dtype")
        d = self.handle.device
        a_rp, a_ci, a_va, a_b, a_c = (_ptr(x, d) for x in (row_ptr, col_idx, values, B, C))
        st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        ldb = B.stride(0) if B.shape[0] > 1 else max(1, self.n)
        ldc = C.stride(0) if C.shape[0] > 1 else max(1, self.n)
        fn = spmm_plan_csr_f32 if values.dtype == torch.float32 else spmm_plan_csr_f64
        fn(self.ptr, alpha, a_rp, a_ci, a_va, a_b, ldb, beta, a_c, ldc, st)

    def squared(self, alpha, row_ptr, col_idx, values, B, beta, C, stream=None) -> None:
        """C <- alpha * A (A B) + beta * C with A's structure from the plan (square A)."""
        import torch
        _check_dense(B, C, self.m, self.m, self.n, self.dtype)
        if values.dtype != self.dtype:
            raise TypeError("values must have the plan's dtype")
        d = self.handle.device
        a_rp, a_ci, a_va, a_b, a_c = (_ptr(x, d) for x in (row_ptr, col_idx, values, B, C))
        st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        ldb = B.stride(0) if B.shape[0] > 1 else max(1, self.n)
        ldc = C.stride(0) if C.shape[0] > 1 else max(1, self.n)
        fn = (spmm_plan_csr_squared_f32 if values.dtype == torch.float32
              else spmm_plan_csr_squared_f64)
        fn(self.ptr, alpha, a_rp, a_ci, a_va, a_b, ldb, beta, a_c, ldc, st)

    def close(self) -> None:
        if self.ptr:
            spmm_plan_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def csr_check(handle: Handle, row_ptr, col_idx, k: int, stream=None) -> int:
    """Device-side CSR structure check; returns the status bit mask (0 = valid)."""
    import torch
    m = int(row_ptr.numel()) - 1
    nnz = int(col_idx.numel())
    d = handle.device
    a_rp, a_ci = _ptr(row_ptr, d), _ptr(col_idx, d)
    st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
    _, mask = spmm_csr_check(handle.ptr, a_rp, a_ci, m, k, nnz, st)
    return mask

"""Shared helpers of the GPU parity tests: run the C ABI on a synth.Problem and
compare with the CPU oracle element by element."""
from __future__ import annotations

import numpy as np

import oracle

TAU = {np.dtype(np.float32): 1e-5, np.dtype(np.float64): 1e-13}


def _dev(a, torch, dev):
    """numpy -> CUDA tensor; empty arrays get a 1-element buffer (valid address)."""
    if a.size == 0:
        return torch.zeros(1, dtype=torch.from_numpy(a[:0]).dtype, device=dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def run_problem(handle, p, C_init=None, stream=None, b_offset=0, check=True):
    """Run C = alpha*A*B + beta*C0 on the GPU through the C ABI; returns (C numpy, status).

    C_init overrides the initial C (same [m, ldc] shape); b_offset shifts B by
    that many elements inside a larger buffer (to exercise unaligned bases).
    """
    import torch

    import csr_spmm_gb300 as cs
    dev = torch.device("cuda")
    rp = _dev(p.row_ptr, torch, dev)
    ci = _dev(p.col_idx, torch, dev)
    va = _dev(p.values, torch, dev)
    Bflat = np.concatenate([np.zeros(b_offset, p.B.dtype), p.B.ravel()]) if b_offset else p.B
    Bd = _dev(Bflat, torch, dev)
    if C_init is None:
        C_init = p.C0 if p.C0 is not None else np.full((p.m, p.ldc), np.nan, p.values.dtype)
    Cd = _dev(np.ascontiguousarray(C_init).copy(), torch, dev)
    st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
    fn = cs.spmm_csr_f32 if p.values.dtype == np.float32 else cs.spmm_csr_f64
    status = fn(handle.ptr, p.alpha, rp.data_ptr(), ci.data_ptr(), va.data_ptr(), p.m, p.k,
                Bd.data_ptr() + b_offset * p.B.itemsize, p.ldb, p.n, p.beta, Cd.data_ptr(),
                p.ldc, st, check=check)
    torch.cuda.synchronize()
    out = Cd.cpu().numpy()[: p.m * p.ldc].reshape(p.m, p.ldc) if p.m else np.zeros((0, p.ldc))
    return out, status


def assert_parity(p, got, rows=None, exact=False, what=""):
    """Element-wise comparison with the oracle on all rows (or `rows`).

    exact: bit-identical after rounding the fp64 oracle to the problem dtype.
    else : |C - C_ref| <= tau * (|alpha| sum|a||b| + |beta||C0|), tau 1e-5 (fp32)
           or 1e-13 (fp64); a zero bound demands exact equality.
    """
    ref, bound = oracle.spmm_problem(p, rows)
    g = got if rows is None else got[np.asarray(rows)]
    g = g[:, : p.n]
    if exact:
        want = ref.astype(p.values.dtype)
        bad = np.argwhere(g.view(np.uint32 if g.dtype == np.float32 else np.uint64)
                          != want.view(np.uint32 if want.dtype == np.float32 else np.uint64))
        assert bad.size == 0, f"{what}: {len(bad)} outputs differ bitwise, first {bad[:3].tolist()}"
        return
    tau = TAU[np.dtype(p.values.dtype)]
    err = np.abs(g.astype(np.float64) - ref)
    ok = err <= tau * bound
    if not np.all(ok):
        i = np.argwhere(~ok)[:3]
        raise AssertionError(
            f"{what}: {int((~ok).sum())} of {ok.size} outputs outside tolerance; first at "
            f"{i.tolist()}: got {[g[tuple(x)] for x in i]}, want {[ref[tuple(x)] for x in i]}, "
            f"bound {[bound[tuple(x)] for x in i]}")

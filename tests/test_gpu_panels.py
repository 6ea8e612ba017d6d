"""GPU parity of products whose B is split into column panels.

The library splits B (and C) into column panels when B is larger than three
times the L2, so that the panel being gathered stays resident.  Every bin
has its own panel loop: short rows (a lane group per row), medium rows (a
warp per row, groups combined at the row's end) and long rows (the CTA split,
whose partial sums span all n columns and are added by the last CTA to
finish the row).  These tests build B above that size with Zipf(2) row
lengths, so that all three bins are populated, and compare every medium and
long row (and a sample of short rows) with the oracle element by element,
in binary32 and binary64, directly and through a plan.  The page stresses
ragged shapes (oxicuda-sparse, ops/spmm.rs, device tests with n = 1, 3, 5
and the "tile ragged edge" note in its kernel); the panel split is the same
kind of edge along another axis."""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
from gpu_helpers import assert_parity, run_problem
from synth import power_law, rng

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


def _l2_bytes():
    import torch
    props = torch.cuda.get_device_properties(0)
    return int(getattr(props, "L2_cache_size", 0) or (128 << 20))


def _checked_rows(p, short_sample, seed):
    """Every row of 33 or more entries, the first and last rows, and a
    seeded sample of the rest."""
    lens = np.diff(p.row_ptr)
    big = np.flatnonzero(lens > 32)
    pick = np.floor(rng.uniform(seed, 91, short_sample) * p.m).astype(np.int64)
    return np.unique(np.concatenate([big, pick, [0, p.m - 1]]))


def _profiled(handle, fn):
    cs.spmm_set_profiling(handle.ptr, True)
    try:
        out = fn()
        prof = cs.spmm_get_profile(handle.ptr)
    finally:
        cs.spmm_set_profiling(handle.ptr, False)
    return out, prof


@pytest.fixture(scope="module")
def wide_f32():
    """1,000,000 x 1,000,000 with about 3 M entries; B 1,000,000 x 128
    binary32 (512 MB, above three times the L2); beta = 0.5."""
    p = power_law(1_000_000, 1_000_000, 128, 3_000_000, 20_000, seed=41, dtype=np.float32,
                  alpha=1.25, beta=0.5, name="panels_f32")
    assert p.k * p.n * 4 > 3 * _l2_bytes()
    return p


def _assert_bins_and_panels(prof, min_panels=2):
    assert prof["panels"] >= min_panels, prof
    assert prof["rows_medium"] > 0 and prof["rows_long"] > 0, prof


def test_panels_f32_every_bin(handle, wide_f32):
    p = wide_f32
    (got, _), prof = _profiled(handle, lambda: run_problem(handle, p))
    _assert_bins_and_panels(prof)
    lens = np.diff(p.row_ptr)
    # several CTAs share at least one long row, so the fixup adds partials
    assert lens.max() > 2 * 2048
    assert_parity(p, got, rows=_checked_rows(p, 20_000, 1), what="panels f32")


def test_panels_f32_deterministic_and_plan_bitwise(handle, wide_f32):
    """A second direct call and a call through a plan give the same bits."""
    import torch
    p = wide_f32
    first, _ = run_problem(handle, p)
    again, _ = run_problem(handle, p)
    assert np.array_equal(first.view(np.uint32), again.view(np.uint32)), "not deterministic"
    dev = torch.device("cuda")
    rp = torch.from_numpy(p.row_ptr).to(dev)
    ci = torch.from_numpy(p.col_idx).to(dev)
    va = torch.from_numpy(p.values).to(dev)
    B = torch.from_numpy(p.B).to(dev)
    C = torch.from_numpy(p.C0.copy()).to(dev)
    plan = cs.Plan(handle, rp, p.k, p.n, torch.float32)
    try:
        plan(p.alpha, rp, ci, va, B, p.beta, C)
        torch.cuda.synchronize()
        got = C.cpu().numpy()
    finally:
        plan.close()
    assert np.array_equal(got.view(np.uint32), first[:, :p.n].view(np.uint32))


def test_panels_f32_unaligned_b(handle, wide_f32):
    """B one element off a 16-byte boundary: the scalar geometry, still in
    panels."""
    p = wide_f32
    (got, _), prof = _profiled(handle, lambda: run_problem(handle, p, b_offset=1))
    _assert_bins_and_panels(prof)
    assert prof["vec_elems"] == 1
    assert_parity(p, got, rows=_checked_rows(p, 5_000, 2), what="panels f32, unaligned B")


def test_panels_f64_every_bin(handle):
    """400,000 x 400,000 binary64, about 1.5 M entries; B 400,000 x 160
    (512 MB); alpha = 2, beta = -1 (the binary64 beta = -1 rows kernel)."""
    p = power_law(400_000, 400_000, 160, 1_500_000, 20_000, seed=42, dtype=np.float64,
                  alpha=2.0, beta=-1.0, name="panels_f64")
    assert p.k * p.n * 8 > 3 * _l2_bytes()
    (got, _), prof = _profiled(handle, lambda: run_problem(handle, p))
    _assert_bins_and_panels(prof)
    assert_parity(p, got, rows=_checked_rows(p, 10_000, 3), what="panels f64")
    again, _ = run_problem(handle, p)
    assert np.array_equal(got.view(np.uint64), again.view(np.uint64)), "not deterministic"


def test_panels_f64_ragged_last_panel(handle):
    """n = 171 binary64 columns (not a multiple of the panel width, odd): the
    last panel is narrower and ends in a partial vector."""
    p = power_law(400_000, 400_000, 171, 1_200_000, 12_000, seed=43, dtype=np.float64,
                  alpha=-0.75, beta=0.25, name="panels_f64_ragged")
    assert p.k * p.n * 8 > 3 * _l2_bytes()
    (got, _), prof = _profiled(handle, lambda: run_problem(handle, p))
    _assert_bins_and_panels(prof)
    assert p.n % prof["panel_cols"] != 0
    assert_parity(p, got, rows=_checked_rows(p, 10_000, 4), what="panels f64, ragged")

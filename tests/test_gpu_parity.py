"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element
by element, on seeded inputs small enough for the oracle to finish in seconds.
They still span many tiles, every row bin, ragged column tails and the edge
cases of the definition."""
import json
import os

import numpy as np
import pytest

import csr_spmm_gb300 as cs
from gpu_helpers import assert_parity, run_problem
from synth import Problem, knn_kernel_graph, laplacian_2d, power_law, rng, uniform_rows
from synth.workloads import tiny_uniform

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


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


def _problem(name, m, k, n, rp, ci, vals, B, alpha, beta, C0=None, dtype=np.float64):
    return Problem(name, m, k, n, np.asarray(rp, np.int32), np.asarray(ci, np.int32),
                   np.asarray(vals, dtype), np.asarray(B, dtype).reshape(k, -1),
                   None if C0 is None else np.asarray(C0, dtype).reshape(m, -1), alpha, beta)


def _dense_fixture(k, n, base):
    idx = np.arange(k * n, dtype=np.float64)
    return (base + 0.5 * idx - 0.1 * (idx % 3)).reshape(k, n)


# ---------------------------------------------------------------------------
# the page's worked examples and device-test fixtures
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_page_known_values(handle, dtype):
    cases = json.load(open(os.path.join(HERE, "golden", "spmm_known_values.json")))["cases"]
    for c in cases:
        p = _problem(c["name"], c["m"], c["k"], c["n"], c["row_ptr"], c["col_idx"], c["values"],
                     c["B"], 1.0, 0.0, dtype=dtype)
        got, _ = run_problem(handle, p)
        assert np.array_equal(got[:, :p.n], np.array(c["expected"], dtype)), c["name"]


@pytest.mark.parametrize("n,alpha,beta,bb,cb,dtype", [
    (3, 1.75, -0.5, 1.0, 7.0, np.float64),     # spmm_f64_n3_alpha_beta
    (5, 2.0, 0.5, -2.0, 0.25, np.float64),     # spmm_f64_n5_alpha_beta
    (3, 1.25, -0.75, 0.5, 3.0, np.float32),    # spmm_f32_n3_alpha_beta
    (1, 1.0, 0.0, 1.0, None, np.float64),      # spmm_f64_single_column_beta_zero (C0 = 1e8)
])
def test_page_matrix_3x4(handle, n, alpha, beta, bb, cb, dtype):
    rp, ci, v = [0, 2, 4, 6], [0, 2, 1, 3, 0, 3], [1, 2, 3, 4, 5, 6]
    C0 = np.full((3, n), 1e8) if cb is None else _dense_fixture(3, n, cb)
    p = _problem("m3x4", 3, 4, n, rp, ci, v, _dense_fixture(4, n, bb), alpha, beta, C0,
                 dtype=dtype)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what="matrix_3x4")
    g = json.load(open(os.path.join(HERE, "golden", "spmm_matrix_3x4_hand.json")))
    for c in g["cases"]:
        if c["n"] == n and c["alpha"] == alpha and c["beta"] == beta and dtype == np.float64:
            assert np.allclose(got[:, :n], np.array(c["expected"]), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# workload families at small sizes
# ---------------------------------------------------------------------------

def test_tiny_uniform_full(handle):
    p = tiny_uniform()
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what="tiny_uniform")


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 15, 16, 17, 31, 32, 33, 64, 100, 127, 128,
                               129, 255, 256, 257, 511, 512, 513, 700])
def test_column_sweep_f32(handle, n):
    p = uniform_rows(300, 500, n, 40, seed=n, alpha=1.25, beta=-0.5)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what=f"n={n}")


@pytest.mark.parametrize("n", [1, 2, 3, 8, 31, 32, 33, 64, 65, 128, 129, 300])
def test_column_sweep_f64(handle, n):
    p = uniform_rows(200, 300, n, 24, seed=100 + n, dtype=np.float64, alpha=-0.75, beta=2.0)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what=f"f64 n={n}")


def _ragged_rows(m, k, n, max_len, seed, dtype=np.float32, alpha=1.0, beta=0.5):
    """Rows of uniform random length 0..max_len (distinct sorted columns)."""
    from synth import distinct_sorted_columns
    lens = np.floor(rng.uniform(seed, 1, m) * (max_len + 1)).astype(np.int64)
    lens = np.minimum(lens, k)
    rp, ci = distinct_sorted_columns(lens, k, seed, 2)
    vals = rng.uniform(seed, 3, int(rp[-1]), -1, 1)
    B = rng.uniform(seed, 4, k * n, -1, 1).reshape(k, n)
    C0 = rng.uniform(seed, 5, m * n, -1, 1).reshape(m, n)
    return _problem("ragged", m, k, n, rp, ci, vals, B, alpha, beta, C0, dtype=dtype)


@pytest.mark.parametrize("n", [4, 16, 64, 100, 256])
@pytest.mark.parametrize("max_len", [3, 70, 600, 3000])
def test_ragged_row_lengths(handle, n, max_len):
    p = _ragged_rows(2500 if max_len < 1000 else 400, 4000, n, max_len, seed=n * 7 + max_len)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what=f"ragged n={n} max_len={max_len}")


@pytest.mark.parametrize("n", [16, 64, 100])
def test_power_law_small(handle, n):
    p = power_law(30_000, 30_000, n, 600_000, 10_000, seed=5)
    assert p.meta["row_len_max"] >= 5_000
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what=f"power_law n={n}")


def test_laplacian_small_f64(handle):
    p = laplacian_2d(60, 32, seed=3)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what="laplacian")


def test_knn_small_beta_zero_nan_c(handle):
    p = knn_kernel_graph(6000, 30, 100, 50, seed=1)
    C_nan = np.full((p.m, p.ldc), np.nan, np.float32)
    got, _ = run_problem(handle, p, C_init=C_nan)
    assert np.all(np.isfinite(got))
    assert_parity(p, got, what="knn")


def test_integer_wide_exact(handle):
    p = uniform_rows(8192, 8192, 512, 16, seed=4, alpha=1.0, beta=0.0, integer_range=3)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, exact=True, what="integer")


@pytest.mark.parametrize("n", [1, 16, 64, 200])
@pytest.mark.parametrize("pad", [0, 2100])
def test_single_huge_row(handle, n, pad):
    # pad: empty rows appended so that m exceeds 2,048 and the row is split
    # across CTAs (pad = 0: the one-launch path, one warp for the row)
    k = 300_000
    lens = np.concatenate([np.array([3, 150_000, 0, 7]), np.zeros(pad, np.int64)])
    from synth import distinct_sorted_columns
    rp, ci = distinct_sorted_columns(lens, k, 9, 1)
    vals = rng.uniform(9, 2, int(rp[-1]), -1, 1)
    B = rng.uniform(9, 3, k * n, -1, 1).reshape(k, n)
    C0 = rng.uniform(9, 4, (4 + pad) * n, -1, 1).reshape(4 + pad, n)
    p = _problem("huge_row", 4 + pad, k, n, rp, ci, vals, B, 1.0, 1.0, C0, dtype=np.float32)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what=f"huge row n={n}")


def test_many_long_rows_across_ctas(handle):
    # 700 rows of 1000..9000 entries: rows span CTAs and CTAs span rows
    from synth import distinct_sorted_columns
    # 2,100 rows, so that the binned path (and its CTA split) takes them; the
    # last 1,400 are empty
    m, k, n = 2100, 20_000, 48
    lens = 1000 + np.floor(rng.uniform(11, 1, m) * 8000).astype(np.int64)
    lens[700:] = 0
    rp, ci = distinct_sorted_columns(lens, k, 11, 2)
    vals = rng.uniform(11, 3, int(rp[-1]), -1, 1)
    B = rng.uniform(11, 4, k * n, -1, 1).reshape(k, n)
    C0 = rng.uniform(11, 5, m * n, -1, 1).reshape(m, n)
    p = _problem("long_rows", m, k, n, rp, ci, vals, B, -1.5, 0.25, C0, dtype=np.float32)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what="long rows")
    p64 = _problem("long_rows64", m, k, n, rp, ci, vals, B, -1.5, 0.25, C0, dtype=np.float64)
    got64, _ = run_problem(handle, p64)
    assert_parity(p64, got64, what="long rows f64")


# ---------------------------------------------------------------------------
# edge cases and conventions
# ---------------------------------------------------------------------------

def test_duplicate_columns_and_explicit_zeros(handle):
    rp = [0, 4, 4, 7]
    ci = [2, 2, 0, 2, 1, 1, 1]
    vals = [1.0, 2.0, 0.0, -3.0, 0.5, 0.5, 0.25]
    B = rng.uniform(1, 1, 3 * 6, -1, 1).reshape(3, 6)
    C0 = rng.uniform(1, 2, 3 * 6, -1, 1).reshape(3, 6)
    for dt in (np.float32, np.float64):
        p = _problem("dups", 3, 3, 6, rp, ci, vals, B, 2.0, -1.0, C0, dtype=dt)
        got, _ = run_problem(handle, p)
        assert_parity(p, got, what="duplicates")


def test_empty_rows_and_all_empty(handle):
    m, k, n = 5000, 100, 24
    rp = np.zeros(m + 1, np.int32)
    p = _problem("all_empty", m, k, n, rp, [], [], rng.uniform(2, 1, k * n, -1, 1), 1.0, 0.5,
                 rng.uniform(2, 2, m * n, -1, 1), dtype=np.float32)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what="all empty")
    p.beta = 0.0
    got, _ = run_problem(handle, p, C_init=np.full((m, n), np.nan, np.float32))
    assert np.array_equal(got, np.zeros((m, n), np.float32))


def test_k_zero_and_alpha_zero(handle):
    import torch
    m, n = 700, 33
    C0 = rng.uniform(3, 1, m * n, -1, 1).reshape(m, n).astype(np.float32)
    # k == 0: C = beta * C, A and B never read (NULL pointers accepted)
    Cd = torch.from_numpy(C0.copy()).cuda()
    cs.spmm_csr_f32(handle.ptr, 1.0, 0, 0, 0, m, 0, 0, n, n, -2.0, Cd.data_ptr(), n,
                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.cpu().numpy(), (-2.0 * C0).astype(np.float32))
    # alpha == 0, beta == 0: C = 0 even when C held NaN; A and B NULL
    Cd = torch.full((m, n), float("nan"), device="cuda")
    cs.spmm_csr_f32(handle.ptr, 0.0, 0, 0, 0, m, 50, 0, n, n, 0.0, Cd.data_ptr(), n,
                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.cpu().numpy(), np.zeros((m, n), np.float32))
    # m == 0 / n == 0: nothing happens
    Cd = torch.full((4, 4), 7.0, device="cuda")
    cs.spmm_csr_f32(handle.ptr, 1.0, 0, 0, 0, 0, 5, 0, 4, 4, 0.0, Cd.data_ptr(), 4, 0)
    cs.spmm_csr_f32(handle.ptr, 1.0, 0, 0, 0, 4, 5, 0, 1, 0, 0.0, Cd.data_ptr(), 1, 0)
    torch.cuda.synchronize()
    assert torch.all(Cd == 7.0)


@pytest.mark.parametrize("n,ldb,ldc,b_offset", [(16, 17, 19, 0), (64, 64, 64, 1), (100, 101, 100, 0),
                                                  (5, 6, 5, 3), (512, 515, 512, 0)])
def test_unaligned_leading_dimensions(handle, n, ldb, ldc, b_offset):
    p = uniform_rows(400, 600, n, 20, seed=n + ldb, alpha=1.0, beta=1.0, ldb=ldb, ldc=ldc)
    got, _ = run_problem(handle, p, b_offset=b_offset)
    assert_parity(p, got, what=f"ld {ldb}/{ldc} off {b_offset}")


def test_padding_columns_of_c_untouched(handle):
    p = uniform_rows(300, 200, 20, 9, seed=8, alpha=1.0, beta=0.0, ldc=27)
    C_init = np.full((p.m, 27), 5.0, np.float32)
    got, _ = run_problem(handle, p, C_init=C_init)
    assert np.all(got[:, 20:] == 5.0)
    assert_parity(p, got, what="ldc padding")


def test_deterministic_bitwise(handle):
    p = power_law(30_000, 30_000, 64, 600_000, 10_000, seed=6)
    a, _ = run_problem(handle, p)
    b, _ = run_problem(handle, p)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_nondefault_stream(handle):
    import torch
    p = uniform_rows(1000, 1000, 64, 12, seed=12)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got, _ = run_problem(handle, p, stream=s)
    assert_parity(p, got, what="side stream")


def test_torch_convenience_api(handle):
    import torch
    p = uniform_rows(500, 400, 40, 10, seed=13, alpha=0.5, beta=1.5)
    dev = "cuda"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    C = t(p.C0.copy())
    cs.spmm(handle, p.alpha, t(p.row_ptr), t(p.col_idx), t(p.values), p.k, t(p.B), p.beta, C)
    torch.cuda.synchronize()
    assert_parity(p, C.cpu().numpy(), what="torch api")


# ---------------------------------------------------------------------------
# error paths (host validation; no kernel sees invalid input)
# ---------------------------------------------------------------------------

def test_error_paths(handle):
    import torch
    B = torch.zeros(10, 8, device="cuda")
    C = torch.zeros(10, 8, device="cuda")
    rp = torch.zeros(11, dtype=torch.int32, device="cuda")
    ci = torch.zeros(1, dtype=torch.int32, device="cuda")
    v = torch.zeros(1, device="cuda")
    f = lambda *a: cs.spmm_csr_f32(handle.ptr, *a, check=False)  # noqa: E731
    P = (rp.data_ptr(), ci.data_ptr(), v.data_ptr())
    assert f(1.0, *P, 10, 10, B.data_ptr(), 7, 8, 0.0, C.data_ptr(), 8, 0) == \
        cs.SPMM_ERR_DIMENSION_MISMATCH                                  # ldb < n
    assert f(1.0, *P, 10, 10, B.data_ptr(), 8, 8, 0.0, C.data_ptr(), 4, 0) == \
        cs.SPMM_ERR_DIMENSION_MISMATCH                                  # ldc < n
    assert f(1.0, *P, -1, 10, B.data_ptr(), 8, 8, 0.0, C.data_ptr(), 8, 0) == \
        cs.SPMM_ERR_INVALID_ARGUMENT
    assert f(1.0, *P, 10, 10, B.data_ptr(), 2**31, 8, 0.0, C.data_ptr(), 8, 0) == \
        cs.SPMM_ERR_INVALID_ARGUMENT                                    # ldb > INT32_MAX
    assert f(1.0, *P, 10, 10, B.data_ptr(), 8, 8, 0.0, 0, 8, 0) == cs.SPMM_ERR_NULL_POINTER
    assert f(1.0, 0, ci.data_ptr(), v.data_ptr(), 10, 10, B.data_ptr(), 8, 8, 0.0,
             C.data_ptr(), 8, 0) == cs.SPMM_ERR_NULL_POINTER
    assert f(1.0, *P, 10, 10, 0, 8, 8, 0.0, C.data_ptr(), 8, 0) == cs.SPMM_ERR_NULL_POINTER
    with pytest.raises(cs.SpmmError):
        cs.spmm_csr_f32(handle.ptr, 1.0, *P, 10, 10, B.data_ptr(), 7, 8, 0.0, C.data_ptr(), 8, 0)


def test_csr_check(handle):
    import torch
    t = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")  # noqa: E731
    assert cs.csr_check(handle, t([0, 2, 4]), t([0, 2, 1, 2]), 3) == 0
    assert cs.csr_check(handle, t([1, 2, 4]), t([0, 2, 1, 2]), 3) & 1
    assert cs.csr_check(handle, t([0, 3, 2]), t([0, 2]), 3) & 2
    assert cs.csr_check(handle, t([0, 2, 3]), t([0, 2, 1, 2]), 3) & 4
    assert cs.csr_check(handle, t([0, 2, 4]), t([0, 3, 1, 2]), 3) & 8
    p = tiny_uniform()
    assert cs.csr_check(handle, torch.from_numpy(p.row_ptr).cuda(),
                        torch.from_numpy(p.col_idx).cuda(), p.k) == 0


# ---------------------------------------------------------------------------
# binary64 with beta = +1 / -1: the epilogue leaves out the multiply by beta
# (exact), on the 16-byte path; other widths take the general epilogue
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [2, 6, 32, 64, 100])
@pytest.mark.parametrize("beta", [1.0, -1.0])
def test_f64_unit_beta(handle, n, beta):
    p = laplacian_2d(40, n, seed=31)
    p.beta = beta
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what=f"f64 beta={beta} n={n}")
    # beta = -1 with C0 and beta = +1 with -C0 give the same bits
    if beta == -1.0:
        q = laplacian_2d(40, n, seed=31)
        q.beta = 1.0
        q.C0 = -q.C0
        other, _ = run_problem(handle, q)
        assert np.array_equal(got[:, :n].view(np.uint64), other[:, :n].view(np.uint64))


@pytest.mark.parametrize("beta", [1.0, -1.0])
def test_f64_unit_beta_integer_exact(handle, beta):
    p = uniform_rows(3000, 2500, 32, 9, seed=32, dtype=np.float64, alpha=2.0, beta=beta,
                     integer_range=3)
    got, _ = run_problem(handle, p)
    assert_parity(p, got, exact=True, what=f"f64 integer beta={beta}")


def test_f64_unit_beta_unaligned_b(handle):
    """B at an odd element offset takes the scalar path with the general
    epilogue; the result stays in parity."""
    p = laplacian_2d(30, 32, seed=33)
    got, _ = run_problem(handle, p, b_offset=1)
    assert_parity(p, got, what="f64 beta=-1 unaligned B")


def test_mixed_tiles_of_short_rows_and_long_rows(handle):
    """Full-warp lane groups (n = 100) make every row under 1024 entries short,
    so most pre-pass tiles hold short rows only (listed by their fast path)
    while the tiles holding a long row take the ranked scatter; and one-CTA
    pre-pass sizes, with and without a long row."""
    p = power_law(40_000, 40_000, 100, 900_000, 20_000, seed=34)
    lens = np.diff(p.row_ptr)
    assert 0 < int((lens >= 1024).sum()) < 200
    got, _ = run_problem(handle, p)
    assert_parity(p, got, what="mixed tiles")
    for m, cap in ((2000, 50), (2000, 1500)):
        q = power_law(m, m, 100, 40 * m, cap, seed=35)
        got, _ = run_problem(handle, q)
        assert_parity(q, got, what=f"one-CTA pre-pass m={m} cap={cap}")


def test_prepass_beyond_one_wave_of_tiles(handle):
    """More than 2.49 M rows: the pre-pass tiles exceed one wave, and a one-CTA
    scan of the tile records runs between count and scatter (below that each
    scatter CTA reduces the records itself)."""
    p = power_law(2_600_000, 2_600_000, 8, 9_000_000, 4000, seed=36)
    lens = np.diff(p.row_ptr)
    assert int((lens >= 1024).sum()) > 0 and int(((lens > 16) & (lens < 1024)).sum()) > 0
    got, _ = run_problem(handle, p)
    rows = np.unique(np.concatenate([np.linspace(0, p.m - 1, 3000).astype(np.int64),
                                     np.flatnonzero(lens >= 1024)[:50]]))
    assert_parity(p, got, rows=rows, what="pre-pass with a scan launch")


def test_fp64_fma_rate_probe(handle):
    """The binary64 FMA-rate probe that binary64 rooflines are set against:
    positive, repeatable within a few percent, and within the range a part
    with 1-4 binary64 FMA per clock per SM at 1-2.5 GHz can reach."""
    import torch
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    r1 = cs.spmm_measure_fp64_fma_rate(handle.ptr)
    r2 = cs.spmm_measure_fp64_fma_rate(handle.ptr)
    assert r1 > 0 and r2 > 0
    assert abs(r1 - r2) <= 0.1 * max(r1, r2)
    assert sms * 1.0 * 1.0e9 * 0.5 <= r1 <= sms * 4.0 * 2.5e9

"""GPU parity of the Frank-Wolfe gradient scan (bixverse page,
seacells_kernels.rs: `fw_argmin_b` + `reduce_argmin_blocks`) against the CPU
oracle.

The GPU sums G in the element type, the oracle in binary64, so:
  - min_val[c] must lie within tau * col_scale[c] of the oracle's minimum;
  - min_idx[c] must equal the oracle's row wherever the minimum is clear
    (the runner-up lies more than 2 tau * col_scale[c] above it); where it is
    not, the row the GPU chose must itself be a minimum within that margin
    (several rows are then correct answers);
  - gap must lie within tau * gap_bound of the oracle's.
tau = 1e-5 (binary32) or 1e-13 (binary64), as for the product.
"""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
import oracle
from gpu_helpers import TAU
from synth.fw import FwProblem, fw_random, seacells_fw

pytestmark = pytest.mark.gpu
F32_MAX = float(np.finfo(np.float32).max)


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


def run_fw(handle, p: FwProblem):
    import torch
    dev = torch.device("cuda")

    def t(a):
        a = np.ascontiguousarray(a)
        if a.size == 0:                 # a valid address for an empty array
            return torch.zeros(1, dtype=torch.from_numpy(a[:0]).dtype, device=dev)
        return torch.from_numpy(a).to(dev)

    mats = [tuple(t(x) for x in m) for m in (p.k2b, p.t1, p.t2, p.b)]
    # the wrapper checks row_ptr lengths; hand the padded empties through the ABI
    dt = torch.float32 if p.dtype == np.float32 else torch.float64
    mv = torch.full((max(p.k, 1),), float("nan"), dtype=dt, device=dev)
    mi = torch.full((max(p.k, 1),), -7, dtype=torch.int32, device=dev)
    gap = torch.full((1,), float("nan"), dtype=dt, device=dev)
    ptrs = lambda m: tuple(x.data_ptr() for x in m)  # noqa: E731
    cs.spmm_fw_argmin(handle.ptr, p.n, p.k, *[ptrs(m) for m in mats], mv.data_ptr(),
                      mi.data_ptr(), gap.data_ptr(), f64=dt == torch.float64,
                      stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return mv.cpu().numpy()[:p.k], mi.cpu().numpy()[:p.k].astype(np.int64), float(gap.item())


def check(p, got, what=""):
    mv, mi, gap = got
    ref = oracle.fw_argmin(p.n, p.k, p.k2b, p.t1, p.t2, p.b)
    tau = TAU[np.dtype(p.dtype)]
    scale = ref["col_scale"]
    assert np.all(np.abs(mv - ref["min_val"]) <= tau * scale), what + " min_val"
    assert abs(gap - ref["gap"]) <= tau * ref["gap_bound"], (what, gap, ref["gap"])
    diff = np.nonzero(mi != ref["min_idx"])[0]
    if diff.size:
        G, _ = oracle.fw_gradient(p.n, p.k, p.k2b, p.t1, p.t2)
        for c in diff:
            col = G[:, c]
            order = np.sort(col)
            # a different row is only right when the minimum is not clear
            assert order[1] - order[0] <= 2 * tau * scale[c], (what, c, "clear minimum missed")
            assert 0 <= mi[c] < p.n and col[mi[c]] <= order[0] + 2 * tau * scale[c], (what, c)
    return ref


@pytest.mark.parametrize("n,k", [(40, 7), (257, 33), (1000, 130), (20_000, 100), (3000, 300)])
def test_shapes(handle, n, k):
    """k spans one to three column passes; n = 20,000 is several rows per warp."""
    p = fw_random(n, k, min(k, 24), seed=n + k)
    check(p, run_fw(handle, p), f"{n}x{k}")


def test_sparse_t1_and_wide_k(handle):
    p = fw_random(600, 1100, 40, seed=5, t1_density=0.05)
    check(p, run_fw(handle, p), "k=1100")


def test_binary64(handle):
    p = fw_random(5000, 70, 16, seed=6, dtype=np.float64)
    mv, mi, gap = run_fw(handle, p)
    ref = check(p, (mv, mi, gap), "f64")
    assert np.array_equal(mi, ref["min_idx"])


def test_tie_goes_to_lowest_row(handle):
    """The page's tie test: t1 = I, K2At = 0, every row of K2B alike, so every
    row ties; warps scan different rows, and the reduction must pick row 0."""
    n, k = 2048, 4
    vals = np.tile(-1.0 - np.arange(k), n).astype(np.float32)
    k2b = (np.arange(0, n * k + 1, k, dtype=np.int32), np.tile(np.arange(k), n).astype(np.int32),
           vals)
    eye = (np.arange(k + 1, dtype=np.int32), np.arange(k, dtype=np.int32), np.ones(k, np.float32))
    empty = (np.zeros(n + 1, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float32))
    p = FwProblem("tie", n, k, k2b, eye, empty, empty)
    mv, mi, gap = run_fw(handle, p)
    assert np.array_equal(mi, np.zeros(k)) and np.array_equal(mv, -1.0 - np.arange(k))
    assert gap == 0.0


def test_empty_rows_take_part(handle):
    p = fw_random(3000, 40, 12, seed=7)
    rp, ci, v = p.k2b
    lens = np.diff(rp)
    lens[::3] = 0                                          # blank every third row
    keep = np.repeat(lens > 0, np.diff(rp))
    rp2 = np.zeros_like(rp)
    np.cumsum(lens, out=rp2[1:])
    q = FwProblem("empty", p.n, p.k, (rp2, ci[keep], v[keep]), p.t1, p.t2, p.b)
    check(q, run_fw(handle, q), "empty rows")


def test_no_rows_and_no_columns(handle):
    e = lambda r: (np.zeros(r + 1, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float32))  # noqa
    p = FwProblem("n0", 0, 5, e(0), e(5), e(0), e(0))
    mv, mi, gap = run_fw(handle, p)
    assert np.array_equal(mv, np.full(5, F32_MAX, np.float32)) and not mi.any() and gap == 0.0
    q = FwProblem("k0", 10, 0, e(10), e(0), e(10), e(10))
    _, _, gap = run_fw(handle, q)
    assert gap == 0.0


def test_deterministic(handle):
    p = fw_random(30_000, 100, 32, seed=8)
    a = run_fw(handle, p)
    b = run_fw(handle, p)
    assert np.array_equal(a[0].view(np.uint32), b[0].view(np.uint32))
    assert np.array_equal(a[1], b[1]) and a[2] == b[2]


def test_torch_wrapper(handle):
    import torch
    p = fw_random(500, 50, 10, seed=9)
    t = lambda m: tuple(torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in m)  # noqa
    mv, mi, gap = cs.fw_argmin(handle, p.k, t(p.k2b), t(p.t1), t(p.t2), t(p.b))
    torch.cuda.synchronize()
    check(p, (mv.cpu().numpy(), mi.cpu().numpy().astype(np.int64), float(gap.item())), "wrapper")


def test_seacells_full_size(handle):
    """The SEACells-shaped scan bench.py times (200,000 cells, 100 archetypes)."""
    p = seacells_fw()
    check(p, run_fw(handle, p), "seacells_fw")


def _with_adjacent_duplicates(mat, every):
    """The same CSR matrix with every `every`-th stored entry repeated in
    place (a duplicate column right after itself, half the value each), so
    the sum of each row is unchanged but runs of equal columns appear."""
    rp, ci, v = (np.asarray(x) for x in mat)
    rows = np.repeat(np.arange(len(rp) - 1), np.diff(rp))
    dup = (np.arange(len(ci)) % every) == 0
    rep = np.where(dup, 2, 1)
    ci2 = np.repeat(ci, rep)
    v2 = np.repeat(np.where(dup, v / 2, v), rep).astype(v.dtype)
    rows2 = np.repeat(rows, rep)
    rp2 = np.zeros_like(rp)
    np.cumsum(np.bincount(rows2, minlength=len(rp) - 1), out=rp2[1:])
    return rp2.astype(rp.dtype), ci2.astype(ci.dtype), v2


def test_long_rows_and_duplicates_on_the_tensor_core_path(handle):
    """binary32, k = 100 (the tensor-core scan): K2B and T2 rows of 60
    entries (past the 32 entries each warp loads ahead), runs of duplicate
    columns in K2B, T2 and B, and a last tile of 37 rows."""
    p = fw_random(3 * 128 + 37, 100, 60, seed=11)
    q = FwProblem("dups", p.n, p.k, _with_adjacent_duplicates(p.k2b, 7), p.t1,
                  _with_adjacent_duplicates(p.t2, 5), _with_adjacent_duplicates(p.b, 3))
    assert np.diff(q.k2b[0]).max() > 64
    check(q, run_fw(handle, q), "long rows with duplicates")


@pytest.mark.parametrize("k", [1, 8, 9, 16, 17, 103, 104, 105])
def test_tensor_core_k_bounds(handle, k):
    """The tensor-core scan's k geometry (k step 8, N a multiple of 16, at most
    104 columns) at and around its edges, and the first k past it (the
    CUDA-core scan), on a ragged last tile of rows."""
    p = fw_random(300, k, min(k, 24), seed=100 + k)
    check(p, run_fw(handle, p), f"k={k}")

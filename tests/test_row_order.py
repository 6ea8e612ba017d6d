"""The breadth-first row order (host code of the library, no GPU): a
permutation of the rows, equal to scipy's breadth-first traversal on
connected patterns, and one that gathers the rows of a hidden block
structure together."""
import numpy as np
import pytest

import csr_spmm_gb300 as cs
from synth import knn_kernel_graph, rng, uniform_rows


@pytest.fixture(scope="module", autouse=True)
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    return cs.library()


def _csr(rows, cols, m):
    order = np.lexsort((cols, rows))
    rows, cols = np.asarray(rows)[order], np.asarray(cols)[order]
    rp = np.zeros(m + 1, dtype=np.int32)
    np.cumsum(np.bincount(rows, minlength=m), out=rp[1:])
    return rp, np.ascontiguousarray(cols, dtype=np.int32)


def test_order_is_a_permutation():
    for seed, (m, k, per) in enumerate([(1, 1, 1), (50, 50, 3), (300, 700, 5), (400, 90, 4),
                                         (1000, 1000, 0)]):
        p = uniform_rows(m, k, 4, per, seed=seed)
        order = cs.spmm_row_order_bfs(p.row_ptr, p.col_idx)
        assert np.array_equal(np.sort(order), np.arange(m)), (m, k, per)


def test_empty_and_duplicates_and_out_of_range_columns():
    assert cs.spmm_row_order_bfs(np.zeros(1, np.int32), np.zeros(0, np.int32)).size == 0
    # row 0 -> 2 (twice), 7 (no such row), -1 (skipped); row 2 -> 1
    rp = np.array([0, 4, 4, 5], np.int32)
    ci = np.array([2, 2, 7, -1, 1], np.int32)
    assert cs.spmm_row_order_bfs(rp, ci).tolist() == [0, 2, 1]
    # no entries at all: each row is its own component, in index order
    assert cs.spmm_row_order_bfs(np.zeros(5, np.int32), np.zeros(0, np.int32)).tolist() == \
        [0, 1, 2, 3]


def test_band_matrix_keeps_natural_order():
    m = 200
    r = np.repeat(np.arange(m), 3)
    c = r + np.tile([-1, 0, 1], m)
    keep = (c >= 0) & (c < m)
    rp, ci = _csr(r[keep], c[keep], m)
    assert np.array_equal(cs.spmm_row_order_bfs(rp, ci), np.arange(m))


def test_matches_scipy_breadth_first_order_on_connected_graph():
    sp = pytest.importorskip("scipy.sparse")
    csgraph = pytest.importorskip("scipy.sparse.csgraph")
    p = knn_kernel_graph(3000, 12, 4, 3, seed=7)
    A = sp.csr_matrix((np.ones(p.col_idx.size), p.col_idx, p.row_ptr), shape=(p.m, p.m))
    ncomp, _ = csgraph.connected_components(A, directed=False)
    assert ncomp == 1
    want = csgraph.breadth_first_order(A, 0, directed=True, return_predecessors=False)
    assert np.array_equal(cs.spmm_row_order_bfs(p.row_ptr, p.col_idx), want)


def test_hidden_blocks_come_out_contiguous():
    """A block-diagonal pattern under a random renumbering: the traversal
    lists each block's rows together."""
    nb, bs = 40, 25
    m = nb * bs
    perm = np.argsort(rng.uniform(3, 50, m))            # new index of old row i is perm[i]
    rows, cols = [], []
    for b in range(nb):
        blk = np.arange(b * bs, (b + 1) * bs)
        rr, cc = np.meshgrid(blk, blk, indexing="ij")
        rows.append(perm[rr.ravel()])
        cols.append(perm[cc.ravel()])
    rp, ci = _csr(np.concatenate(rows), np.concatenate(cols), m)
    order = cs.spmm_row_order_bfs(rp, ci)
    block_of = np.empty(m, np.int64)
    block_of[perm] = np.arange(m) // bs
    seq = block_of[order]
    assert np.all(seq.reshape(nb, bs) == seq.reshape(nb, bs)[:, :1])


def test_invalid_row_pointers_are_rejected():
    lib = cs.library()
    order = np.zeros(3, np.int32)
    ci = np.zeros(4, np.int32)
    for bad in ([1, 2, 3, 4], [0, 3, 2, 4]):
        rp = np.array(bad, np.int32)
        assert lib.spmm_row_order_bfs(rp.ctypes.data, ci.ctypes.data, 3,
                                      order.ctypes.data) == cs.SPMM_ERR_INVALID_CSR
    rp = np.array([0, 1, 2, 4], np.int32)
    assert lib.spmm_row_order_bfs(rp.ctypes.data, None, 3,
                                  order.ctypes.data) == cs.SPMM_ERR_NULL_POINTER
    assert lib.spmm_row_order_bfs(rp.ctypes.data, ci.ctypes.data, -1,
                                  order.ctypes.data) == cs.SPMM_ERR_INVALID_ARGUMENT

"""Seeded generators: determinism and the structure each workload promises (no GPU)."""
import numpy as np

from synth import (distinct_sorted_columns, knn_kernel_graph, laplacian_2d, power_law, rng,
                   uniform_rows, zipf_lengths)
from synth import workloads


def _rows_sorted_distinct(rp, ci):
    for i in range(len(rp) - 1):
        r = ci[rp[i]:rp[i + 1]]
        if r.size > 1 and not np.all(np.diff(r) > 0):
            return False
    return True


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    z = rng._mix(np.array([0x9E3779B97F4A7C15], dtype=np.uint64))
    assert int(z[0]) == 0xE220A8397B1DCDAF
    z = rng._mix(np.array([(2 * 0x9E3779B97F4A7C15) & (2**64 - 1)], dtype=np.uint64))
    assert int(z[0]) == 0x6E789E6AA1B965F4


def test_streams_are_deterministic_and_offsettable():
    a = rng.raw_u64(5, 3, 1000)
    assert np.array_equal(a, rng.raw_u64(5, 3, 1000))
    assert np.array_equal(a[400:], rng.raw_u64(5, 3, 600, offset=400))
    assert np.array_equal(a[[3, 999]], rng.raw_at(5, 3, np.array([3, 999])))
    assert not np.array_equal(a, rng.raw_u64(6, 3, 1000))
    u = rng.to_unit(a)
    assert u.min() >= 0.0 and u.max() < 1.0


def test_distinct_sorted_columns():
    lens = np.array([0, 5, 17, 17, 1])
    rp, ci = distinct_sorted_columns(lens, 17, 1, 2)
    assert np.array_equal(np.diff(rp), lens)
    assert _rows_sorted_distinct(rp, ci)
    assert np.array_equal(ci[rp[2]:rp[3]], np.arange(17))   # full row


def test_tiny_uniform_matches_stated_sizes():
    p = workloads.tiny_uniform()
    assert (p.m, p.k, p.n, p.nnz) == (1024, 1024, 16, 8192)
    assert p.algorithmic_bytes() == 266_244 and p.flops() == 262_144
    assert _rows_sorted_distinct(p.row_ptr, p.col_idx)
    assert p.values.dtype == np.float32 and np.abs(p.values).max() <= 1.0


def test_laplacian_structure():
    p = laplacian_2d(9, 4, 3)
    A = np.zeros((81, 81))
    A[np.repeat(np.arange(81), np.diff(p.row_ptr)), p.col_idx] = p.values
    assert np.allclose(A, A.T * (A != np.diag(np.diag(A))) + np.diag(np.diag(A)))
    assert np.all((np.diag(A) >= 4.0) & (np.diag(A) <= 4.1))
    assert p.nnz == 5 * 81 - 4 * 9
    assert 5 * 707 * 707 - 4 * 707 == 2_496_417


def test_knn_graph_small():
    p = knn_kernel_graph(2000, 10, 7, 20, seed=3)
    lens = np.diff(p.row_ptr)
    assert lens.min() >= 10 and lens.max() <= 20 + 20
    A = np.zeros((2000, 2000), np.float32)
    A[np.repeat(np.arange(2000), lens), p.col_idx] = p.values
    assert np.array_equal(A, A.T)                       # symmetric values
    assert np.all(np.diag(A) == 1.0)
    off = A[(A != 0) & ~np.eye(2000, dtype=bool)]
    assert off.min() >= np.exp(-4.0) - 1e-6 and off.max() <= 1.0
    assert np.allclose(p.B.sum(axis=0), 1.0, atol=1e-5)
    assert np.all((p.B > 0).sum(axis=0) == 20) and p.B.min() >= 0


def test_power_law_small():
    p = power_law(20_000, 20_000, 8, 200_000, 5_000, seed=2)
    lens = np.diff(p.row_ptr)
    assert abs(int(lens.sum()) - 200_000) < 200_000 * 0.01
    assert lens.min() >= 1 and lens.max() <= 5_000
    assert _rows_sorted_distinct(p.row_ptr, p.col_idx)
    lens2, s = zipf_lengths(20_000, 200_000, 5_000, seed=2)
    assert np.array_equal(lens, lens2) and s > 0


def test_integer_workload_values():
    p = uniform_rows(64, 64, 8, 4, seed=4, integer_range=3, alpha=1.0, beta=0.0)
    assert set(np.unique(p.values)).issubset(set(range(-3, 4)))
    assert set(np.unique(p.B)).issubset(set(range(-3, 4)))
    assert p.C0 is None

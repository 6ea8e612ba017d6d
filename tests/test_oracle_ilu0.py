"""Pins for the ILU(0) oracle (no GPU).

ILU(0) of the oxicuda preconditioner page (preconditioner/ilu0.rs): an
incomplete LU with zero fill-in, L unit lower and U upper triangular in A's
pattern, computed level by level with one rounded divide / multiply /
subtract per step in the element type.  The pins tie ``oracle.ilu0`` to the
page's own test values, to the defining property of ILU(0) ((LU)[i, j] =
A[i, j] on A's pattern), to exact LU where no fill-in is dropped (dense and
tridiagonal patterns), to the closed-form recurrence of a tridiagonal matrix
evaluated with the same rounded operations, and to the known level
structure of the identity, a tridiagonal and a 2-D 5-point grid.
"""
import json
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

import oracle
from synth import distinct_sorted_columns, laplacian_2d, rng

HERE = os.path.dirname(os.path.abspath(__file__))


def tridiag(n, d=4.0, off=-1.0, dtype=np.float64):
    rp, ci, v = [0], [], []
    for i in range(n):
        if i > 0:
            ci.append(i - 1); v.append(off)
        ci.append(i); v.append(d)
        if i < n - 1:
            ci.append(i + 1); v.append(off)
        rp.append(len(ci))
    return np.array(rp), np.array(ci), np.array(v, dtype)


def random_dd(n, per_row, seed, dtype=np.float64):
    """Random sparse pattern plus the diagonal, diagonally dominant values."""
    lens = np.full(n, per_row, np.int64)
    rp, ci = distinct_sorted_columns(lens, n, seed, 11)
    rows = np.repeat(np.arange(n), np.diff(rp))
    keys = np.unique(np.concatenate([rows * n + ci, np.arange(n) * (n + 1)]))
    r, c = keys // n, keys % n
    vals = rng.uniform(seed, 12, keys.size, -1.0, 1.0)
    vals[r == c] = per_row + 2.0 + rng.uniform(seed, 13, n)
    rp2 = np.zeros(n + 1, np.int64)
    np.cumsum(np.bincount(r, minlength=n), out=rp2[1:])
    return rp2, c, vals.astype(dtype)


def dense(rp, ci, v, n):
    A = np.zeros((n, n))
    A[np.repeat(np.arange(n), np.diff(rp)), ci] = v
    return A


def pin_page_examples(ilu):
    g = json.load(open(os.path.join(HERE, "golden", "ilu0_page_examples.json")))
    for c in g["cases"]:
        vals = np.array(c["values"], np.float64)
        if c.get("singular"):
            with pytest.raises(oracle.SingularMatrix):
                ilu(c["row_ptr"], c["col_idx"], vals)
            continue
        f, depth = ilu(c["row_ptr"], c["col_idx"], vals)
        assert np.array_equal(f, np.array(c["factored"], np.float64)), c["name"]
        assert int(depth.max()) + 1 == c["levels"], c["name"]
        if "rows_in_level_0" in c:
            assert int((depth == 0).sum()) == c["rows_in_level_0"]


def pin_pattern_property(ilu):
    """(L U)[i, j] = A[i, j] for every (i, j) stored in A."""
    for n, per, seed in ((60, 4, 1), (200, 7, 2)):
        rp, ci, v = random_dd(n, per, seed)
        f, _ = ilu(rp, ci, v)
        L, U = oracle.ilu0_split(rp, ci, f)
        LU = L @ U
        rows = np.repeat(np.arange(n), np.diff(rp))
        assert np.allclose(LU[rows, ci], v, rtol=1e-12, atol=1e-12)


def pin_dense_is_exact_lu(ilu):
    n = 9
    A = rng.uniform(3, 1, n * n, -1.0, 1.0).reshape(n, n) + n * np.eye(n)
    rp = np.arange(0, n * n + 1, n)
    ci = np.tile(np.arange(n), n)
    f, depth = ilu(rp, ci, A.ravel())
    L, U = oracle.ilu0_split(rp, ci, f)
    assert np.allclose(L @ U, A, rtol=0, atol=1e-12)
    assert np.array_equal(depth, np.arange(n))


def _tridiag_recurrence(ilu, dtype):
    n = 50
    rp, ci, v = tridiag(n, dtype=dtype)
    f, depth = ilu(rp, ci, v)
    # the same rounded operations, written out for this structure:
    # l_i = a_{i,i-1} / u_{i-1};  u_i = a_ii - l_i * a_{i-1,i}
    four, m1 = dtype(4.0), dtype(-1.0)
    u_prev = four
    assert f[0] == four                                  # u_00 (row 0 stores the diagonal first)
    for i in range(1, n):
        l = dtype(m1 / u_prev)
        u = dtype(four - dtype(l * m1))
        p_l = rp[i]                                     # (i, i-1) is the row's first entry
        assert f[p_l] == l and f[p_l + 1] == u, i
        u_prev = u
    assert np.array_equal(depth, np.arange(n))


def pin_tridiagonal_recurrence_f64(ilu):
    _tridiag_recurrence(ilu, np.float64)


def pin_tridiagonal_recurrence_f32(ilu):
    _tridiag_recurrence(ilu, np.float32)


def pin_grid_levels(ilu):
    """Natural order on a side x side 5-point grid: the level of node (x, y)
    is x + y (lower neighbours are left and below)."""
    side = 9
    p = laplacian_2d(side, 1, seed=3)
    _, depth = ilu(p.row_ptr, p.col_idx, p.values.astype(np.float64))
    y, x = np.divmod(np.arange(side * side), side)
    assert np.array_equal(depth, x + y)


def pin_missing_pivot_is_singular(ilu):
    # row 0 stores no diagonal; row 1 needs it as a pivot
    with pytest.raises(oracle.SingularMatrix):
        ilu([0, 1, 3], [1, 0, 1], np.array([2.0, 1.0, 3.0]))


PINS = [pin_page_examples, pin_pattern_property, pin_dense_is_exact_lu,
        pin_tridiagonal_recurrence_f64, pin_tridiagonal_recurrence_f32, pin_grid_levels,
        pin_missing_pivot_is_singular]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_ilu0_oracle_pin(pin):
    pin(oracle.ilu0)


def test_rejects_unsorted_rows():
    with pytest.raises(ValueError):
        oracle.ilu0([0, 2, 4], [1, 0, 0, 1], np.array([1.0, 4.0, 1.0, 3.0]))


MUTANTS = {
    "ratio_not_stored": ("                v[p] = l_ik;", "                (void)0;"),
    "update_added": ("v[t] = v[t] - prod;", "v[t] = v[t] + prod;"),
    "pivot_row_is_own_row": ("const int64_t pk = diag[k];", "const int64_t pk = slot[k];"),
    "update_includes_pivot": ("for (int64_t q = pk + 1; q < (int64_t)rp[k + 1]; ++q) {",
                              "for (int64_t q = rp[k]; q < (int64_t)rp[k + 1]; ++q) {"),
    "diagonal_eliminated": ("for (int64_t p = lo; p < hi && ci[p] < i; ++p) {",
                            "for (int64_t p = lo; p < hi && ci[p] <= i; ++p) {"),
    "level_off_by_one": ("if (j < i && depth[j] + 1 > d) d = depth[j] + 1;",
                         "if (j < i && depth[j] + 2 > d) d = depth[j] + 2;"),
    "zero_pivot_accepted": ("if (pk < 0 || v[pk] == (T)0) {", "if (pk < 0) {"),
    "positions_not_cleared": ("for (int64_t p = lo; p < hi; ++p) slot[ci[p]] = -1;",
                              "(void)0;"),
    "fill_in_added_to_diagonal": ("if (t < 0) continue;",
                                  "if (t < 0) { v[diag[i]] = v[diag[i]] - l_ik * v[q]; continue; }"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "spmm_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(so), str(mutated), "-lm"], check=True)
    code = ("import sys; sys.path[:0] = [%r, %r]\n"
            "import oracle, test_oracle_ilu0 as t\n"
            "lib = oracle.load_library(%r)\n"
            "bad = t.failing_pins(lambda *a, **k: oracle.ilu0(*a, _lib=lib, **k))\n"
            "print('FAILED:' + ','.join(bad))\n") % (os.path.dirname(HERE), HERE, str(so))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode == 0:
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED:")][-1]
        assert line != "FAILED:", f"mutant {name} passed every pin"
    else:
        assert r.returncode < 0 or "Error" in r.stderr, r.stderr


def failing_pins(ilu):
    failed = []
    for pin in PINS:
        try:
            pin(ilu)
        except (AssertionError, ValueError, pytest.fail.Exception):
            failed.append(pin.__name__)
    return failed

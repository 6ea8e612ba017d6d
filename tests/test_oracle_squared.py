"""Pins for the squared-chain oracle C = alpha * A (A B) + beta * C0 (no GPU).

The chain is the K^2 B product that the SEACells Frank-Wolfe kernels of the
bixverse page consume (module doc: the n x k output of `k_squared_matmul`).
Each check ties ``oracle.spmm_squared`` to something other than itself:
hand-derived values, a dense product computed by numpy, exact integer
arithmetic in Python, and closed forms (identity, permutation, nilpotent and
diagonal A).  ``test_planted_mistakes_are_caught`` compiles broken copies of
the oracle and shows every one fails at least one pin.
"""
import json
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

import oracle
from synth import distinct_sorted_columns, rng

HERE = os.path.dirname(os.path.abspath(__file__))


def _random_square_csr(m, seed, max_len=6, dup=False):
    lens = np.floor(rng.uniform(seed, 1, m) * (max_len + 1)).astype(np.int64)
    if dup:
        rp = np.zeros(m + 1, np.int64)
        np.cumsum(lens, out=rp[1:])
        cols = np.floor(rng.uniform(seed, 2, int(rp[-1])) * m).astype(np.int64)
    else:
        rp, cols = distinct_sorted_columns(np.minimum(lens, m), m, seed, 3)
    vals = rng.uniform(seed, 4, int(rp[-1]), -1.0, 1.0)
    return rp.astype(np.int32), cols.astype(np.int32), vals


def _dense(m, rp, ci, vals):
    A = np.zeros((m, m))
    np.add.at(A, (np.repeat(np.arange(m), np.diff(rp)), ci), vals)
    return A


def pin_hand_derived(sq):
    g = json.load(open(os.path.join(HERE, "golden", "spmm_squared_hand.json")))
    for c in g["cases"]:
        B = np.array(c["B"], np.float64)
        C0 = None if c["C0"] is None else np.array(c["C0"], np.float64)
        out, _ = sq(c["m"], c["n"], c["alpha"], c["row_ptr"], c["col_idx"],
                    np.array(c["values"], np.float64), B, c["n"], c["beta"], C0, c["n"])
        assert np.array_equal(out, np.array(c["expected"], np.float64)), c["name"]
        # the intermediate: A^2 applied to the unit vectors
        I = np.eye(c["m"])
        a2, _ = sq(c["m"], c["m"], 1.0, c["row_ptr"], c["col_idx"],
                   np.array(c["values"], np.float64), I, c["m"], 0.0)
        assert np.array_equal(a2, np.array(c["A2"], np.float64)), c["name"] + " A^2"


def pin_dense_bruteforce(sq):
    for seed, dup in ((31, False), (32, True)):
        m, n = 37, 5
        rp, ci, vals = _random_square_csr(m, seed, dup=dup)
        B = rng.uniform(seed, 5, m * n, -1, 1).reshape(m, n)
        C0 = rng.uniform(seed, 6, m * n, -1, 1).reshape(m, n)
        out, bound = sq(m, n, 1.25, rp, ci, vals, B, n, -0.5, C0, n)
        A = _dense(m, rp, ci, vals)
        want = 1.25 * (A @ (A @ B)) - 0.5 * C0
        assert np.all(np.abs(out - want) <= 1e-13 * bound + 1e-300)


def pin_identity(sq):
    m, n = 9, 3
    B = rng.uniform(40, 1, m * n, -1, 1).reshape(m, n)
    C0 = rng.uniform(40, 2, m * n, -1, 1).reshape(m, n)
    out, _ = sq(m, n, 1.0, np.arange(m + 1), np.arange(m), np.ones(m), B, n, 2.0, C0, n)
    assert np.array_equal(out, B + 2.0 * C0)


def pin_permutation(sq):
    """A = cyclic shift (row i has a one in column (i+1) mod m): A^2 B picks row i+2."""
    m, n = 7, 4
    B = rng.uniform(41, 1, m * n, -1, 1).reshape(m, n)
    cols = (np.arange(m) + 1) % m
    out, _ = sq(m, n, 1.0, np.arange(m + 1), cols, np.ones(m), B, n, 0.0)
    assert np.array_equal(out, B[(np.arange(m) + 2) % m])


def pin_nilpotent(sq):
    """A = e0 e1^T: A^2 = 0, so C = beta * C0 exactly."""
    n = 3
    B = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])
    C0 = np.array([[1.0, -1.0, 0.5], [2.0, 0.0, -3.0]])
    out, bound = sq(2, n, 3.0, [0, 1, 1], [1], [7.0], B, n, 0.5, C0, n)
    assert np.array_equal(out, 0.5 * C0)
    assert np.array_equal(bound, 0.5 * np.abs(C0))


def pin_diagonal(sq):
    m, n = 6, 2
    d = np.array([1.0, -2.0, 3.0, 0.5, -1.0, 4.0])
    B = np.arange(m * n, dtype=np.float64).reshape(m, n) - 3.0
    out, _ = sq(m, n, 1.0, np.arange(m + 1), np.arange(m), d, B, n, 0.0)
    assert np.array_equal(out, (d * d)[:, None] * B)


def pin_integer_exact(sq):
    """Small integers: every partial sum is exact in binary64; compare with
    Python integer arithmetic on dictionaries of rows."""
    m, n = 15, 4
    rp, ci, _ = _random_square_csr(m, 42, max_len=5, dup=True)
    vals = rng.integers(42, 7, ci.size, -3, 3).astype(np.float64)
    B = rng.integers(42, 8, m * n, -4, 4).astype(np.float64).reshape(m, n)
    C0 = rng.integers(42, 9, m * n, -5, 5).astype(np.float64).reshape(m, n)
    out, _ = sq(m, n, 2.0, rp, ci, vals, B, n, -3.0, C0, n)
    rows = [[(int(ci[p]), int(vals[p])) for p in range(rp[i], rp[i + 1])] for i in range(m)]
    for i in range(m):
        for c in range(n):
            s = 0
            for j, a in rows[i]:
                s += a * sum(aj * int(B[l, c]) for l, aj in rows[j])
            assert out[i, c] == 2 * s - 3 * int(C0[i, c]), (i, c)


def pin_alpha_zero(sq):
    m, n = 5, 2
    C0 = rng.uniform(43, 1, m * n, -1, 1).reshape(m, n)
    out, _ = sq(m, n, 0.0, None, None, np.zeros(0), np.zeros((0, n)), n, -2.0, C0, n)
    assert np.array_equal(out, -2.0 * C0)


def pin_beta_zero_ignores_c0(sq):
    m, n = 8, 3
    rp, ci, vals = _random_square_csr(m, 44)
    B = rng.uniform(44, 5, m * n, -1, 1).reshape(m, n)
    a, _ = sq(m, n, 1.0, rp, ci, vals, B, n, 0.0)
    b, _ = sq(m, n, 1.0, rp, ci, vals, B, n, 0.0, np.full((m, n), np.nan), n)
    assert np.array_equal(a, b) and np.all(np.isfinite(b))


def pin_bound_scale(sq):
    m, n = 20, 3
    rp, ci, vals = _random_square_csr(m, 45, dup=True)
    B = rng.uniform(45, 5, m * n, -1, 1).reshape(m, n)
    C0 = rng.uniform(45, 6, m * n, -1, 1).reshape(m, n)
    _, bound = sq(m, n, -1.5, rp, ci, vals, B, n, 0.75, C0, n)
    absA = np.abs(_dense(m, rp, ci, np.abs(vals)))
    want = 1.5 * (absA @ (absA @ np.abs(B))) + 0.75 * np.abs(C0)
    assert np.allclose(bound, want, rtol=1e-13, atol=0)


def pin_leading_dimension_and_rows(sq):
    m, n, ldb, ldc = 11, 3, 7, 5
    rp, ci, vals = _random_square_csr(m, 46)
    Bp = rng.uniform(46, 5, m * ldb, -1, 1).reshape(m, ldb)
    C0p = rng.uniform(46, 6, m * ldc, -1, 1).reshape(m, ldc)
    full, _ = sq(m, n, 1.0, rp, ci, vals, Bp, ldb, 0.25, C0p, ldc)
    A = _dense(m, rp, ci, vals)
    want = A @ (A @ Bp[:, :n]) + 0.25 * C0p[:, :n]
    assert np.allclose(full, want, rtol=1e-12, atol=1e-14)
    rows = np.array([10, 0, 4, 4])
    sub, _ = sq(m, n, 1.0, rp, ci, vals, Bp, ldb, 0.25, C0p, ldc, rows=rows)
    assert np.array_equal(sub, full[rows])


PINS = [pin_hand_derived, pin_dense_bruteforce, pin_identity, pin_permutation, pin_nilpotent,
        pin_diagonal, pin_integer_exact, pin_alpha_zero, pin_beta_zero_ignores_c0,
        pin_bound_scale, pin_leading_dimension_and_rows]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_squared_oracle_pin(pin):
    pin(oracle.spmm_squared)


def test_squared_oracle_rejects_bad_csr():
    with pytest.raises(ValueError):
        oracle.spmm_squared(2, 1, 1.0, [0, 1, 2], [0, 5], [1.0, 1.0], np.ones((2, 1)), 1, 0.0)


# (anchor, replacement, which occurrence in spmm_oracle.c)
MUTANTS = {
    "single_product": ("acc[c] += a * t[c];", "acc[c] += a * load(B, j * ldb + c, esize);", 0),
    "inner_row_is_outer_row": ("for (int64_t q = row_ptr[j]; q < (int64_t)row_ptr[j + 1]; ++q)",
                               "for (int64_t q = row_ptr[i]; q < (int64_t)row_ptr[i + 1]; ++q)", 0),
    "inner_value_from_outer": ("double aj = load(values, q, esize);",
                               "double aj = load(values, p, esize);", 0),
    "inner_column_is_outer": ("int64_t l = col_idx[q];", "int64_t l = j;", 0),
    "transposed_b": ("load(B, l * ldb + c, esize)", "load(B, c * ldb + l, esize)", 0),
    "intermediate_not_reset": ("t[c] = 0.0;\n                abst[c] = 0.0;",
                               "abst[c] = 0.0;", 0),
    "bound_without_abs": ("abst[c] += fabs(aj) * fabs(b);", "abst[c] += aj * b;", 0),
    "dropped_beta_term": ("v += beta * c0;", "v += 0.0 * c0;", 1),
    "alpha_not_applied": ("double v = alpha * acc[c];", "double v = acc[c];", 1),
    "beta_zero_reads_c0": ("if (beta != 0.0) {                   /* C0 read only when beta != 0 */",
                           "if (1) {", 1),
}


def _replace_nth(s, old, new, k):
    i = -1
    for _ in range(k + 1):
        i = s.index(old, i + 1)
    return s[:i] + new + s[i + len(old):]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "spmm_oracle.c")).read()
    old, new, k = MUTANTS[name]
    assert src.count(old) == k + 1 or (k == 0 and src.count(old) == 1), name
    mutated = tmp_path / "mut.c"
    mutated.write_text(_replace_nth(src, old, new, k))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(so), str(mutated), "-lm"], check=True)
    code = ("import sys; sys.path[:0] = [%r, %r]\n"
            "import oracle, test_oracle_squared as t\n"
            "lib = oracle.load_library(%r)\n"
            "bad = t.failing_pins(lambda *a, **k: oracle.spmm_squared(*a, _lib=lib, **k))\n"
            "print('FAILED:' + ','.join(bad))\n") % (os.path.dirname(HERE), HERE, str(so))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode == 0:
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED:")][-1]
        assert line != "FAILED:", f"mutant {name} passed every pin"
    else:
        assert r.returncode < 0 or "Error" in r.stderr, r.stderr


def failing_pins(sq):
    failed = []
    for pin in PINS:
        try:
            pin(sq)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    return failed

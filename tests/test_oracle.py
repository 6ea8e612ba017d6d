"""Pins for the CPU oracle (no GPU).

Each check ties the oracle to something other than itself: the worked
examples printed by the reference page (oxicuda-sparse, ops/spmm.rs, CPU
reference tests), values derived by hand from the page's fixtures, a dense
matrix product computed by numpy, exact integer arithmetic in Python, and
identities of the definition (identity A, alpha = 0, beta = 0, linearity in
B).  ``test_planted_mistakes_are_caught`` compiles deliberately broken copies
of the oracle and shows every one of them fails at least one pin.
"""
import json
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

import oracle
from synth import rng, uniform_rows

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden(name):
    with open(os.path.join(HERE, "golden", name)) as f:
        return json.load(f)


def _dense_fixture(k, n, base):
    """The page's dense(k, n, base): row-major, base + 0.5*idx - 0.1*(idx % 3)."""
    idx = np.arange(k * n, dtype=np.float64)
    return (base + 0.5 * idx - 0.1 * (idx % 3)).reshape(k, n)


def _random_csr(m, k, seed, max_len=None, dup=False):
    """Small random CSR with empty rows, optional duplicate columns."""
    max_len = max_len if max_len is not None else min(k, 8)
    lens = np.floor(rng.uniform(seed, 1, m) * (max_len + 1)).astype(np.int64)
    rp = np.zeros(m + 1, np.int64)
    np.cumsum(lens, out=rp[1:])
    nnz = int(rp[-1])
    cols = np.floor(rng.uniform(seed, 2, nnz) * k).astype(np.int64)
    if not dup:
        # distinct sorted within each row
        from synth import distinct_sorted_columns
        rp, cols = distinct_sorted_columns(np.minimum(lens, k), k, seed, 3)
        nnz = int(rp[-1])
    vals = rng.uniform(seed, 4, nnz, -1.0, 1.0)
    return rp.astype(np.int32), cols.astype(np.int32), vals


def _to_dense(m, k, rp, ci, vals):
    A = np.zeros((m, k), np.float64)
    rows = np.repeat(np.arange(m), np.diff(rp))
    np.add.at(A, (rows, ci), vals)          # duplicates add
    return A


# ---------------------------------------------------------------------------
# pins, written against a callable with oracle.spmm's signature
# ---------------------------------------------------------------------------

def pin_page_known_values(spmm):
    for case in _golden("spmm_known_values.json")["cases"]:
        for dt in (np.float32, np.float64):
            B = np.array(case["B"], dt).reshape(case["k"], case["n"])
            out, _ = spmm(case["m"], case["k"], case["n"], 1.0, np.array(case["row_ptr"]),
                          np.array(case["col_idx"]), np.array(case["values"], dt), B,
                          case["n"], 0.0)
            assert np.array_equal(out, np.array(case["expected"], np.float64)), case["name"]


def pin_hand_derived_3x4(spmm):
    g = _golden("spmm_matrix_3x4_hand.json")
    A = g["A"]
    for case in g["cases"]:
        n = case["n"]
        B = _dense_fixture(A["k"], n, case["b_base"])
        if "c0_fill" in case:
            C0 = np.full((A["m"], n), case["c0_fill"])
        else:
            C0 = _dense_fixture(A["m"], n, case["c_base"])
        out, _ = spmm(A["m"], A["k"], n, case["alpha"], np.array(A["row_ptr"]),
                      np.array(A["col_idx"]), np.array(A["values"], np.float64), B, n,
                      case["beta"], C0, n)
        assert np.allclose(out, np.array(case["expected"]), rtol=0, atol=1e-12), case["name"]


def pin_dense_bruteforce(spmm):
    """Against numpy's dense product of the expanded matrix (m, k <= 64)."""
    for seed, (m, k, n) in enumerate([(1, 1, 1), (7, 5, 3), (64, 64, 17), (33, 64, 64),
                                      (64, 9, 5), (20, 40, 1)]):
        for dup in (False, True):
            rp, ci, vals = _random_csr(m, k, 100 + seed, dup=dup)
            B = rng.uniform(seed, 5, k * n, -2, 2).reshape(k, n)
            C0 = rng.uniform(seed, 6, m * n, -2, 2).reshape(m, n)
            for alpha, beta in [(1.0, 0.0), (1.75, -0.5), (-2.0, 1.0)]:
                want = alpha * (_to_dense(m, k, rp, ci, vals) @ B) + beta * C0
                out, bound = spmm(m, k, n, alpha, rp, ci, vals, B, n, beta, C0, n)
                assert np.all(np.abs(out - want) <= 1e-13 * (bound + 1e-300)), (m, k, n, dup)


def pin_integer_exact(spmm):
    """Integer inputs: compare with exact Python-int arithmetic (pure loops, tiny)."""
    m, k, n = 12, 10, 7
    rp, ci, _ = _random_csr(m, k, 7, dup=True)
    vals = rng.integers(7, 8, int(rp[-1]), -3, 3)
    B = rng.integers(7, 9, k * n, -3, 3).reshape(k, n)
    C0 = rng.integers(7, 10, m * n, -5, 5).reshape(m, n)
    alpha, beta = 3, -2
    want = np.zeros((m, n), np.int64)
    for i in range(m):
        for c in range(n):
            s = 0
            for p in range(int(rp[i]), int(rp[i + 1])):
                s += int(vals[p]) * int(B[int(ci[p]), c])
            want[i, c] = alpha * s + beta * int(C0[i, c])
    for dt in (np.float32, np.float64):
        out, _ = spmm(m, k, n, float(alpha), rp, ci, vals.astype(dt), B.astype(dt), n,
                      float(beta), C0.astype(dt), n)
        assert np.array_equal(out, want.astype(np.float64))


def pin_identity(spmm):
    """Identity A gives alpha * B + beta * C0."""
    m, n = 9, 6
    rp = np.arange(m + 1)
    ci = np.arange(m)
    B = rng.uniform(3, 1, m * n, -1, 1).reshape(m, n)
    C0 = rng.uniform(3, 2, m * n, -1, 1).reshape(m, n)
    out, _ = spmm(m, m, n, 1.5, rp, ci, np.ones(m), B, n, 0.25, C0, n)
    assert np.array_equal(out, 1.5 * B + 0.25 * C0)


def pin_alpha_zero(spmm):
    """alpha = 0 gives beta * C0 and reads neither A's values nor B."""
    m, k, n = 6, 5, 4
    rp, ci, _ = _random_csr(m, k, 11)
    vals = np.full(int(rp[-1]), np.nan)
    B = np.full((k, n), np.nan)
    C0 = rng.uniform(4, 1, m * n, -1, 1).reshape(m, n)
    out, _ = spmm(m, k, n, 0.0, rp, ci, vals, B, n, -0.75, C0, n)
    assert np.array_equal(out, -0.75 * C0)
    out, _ = spmm(m, k, n, 0.0, rp, ci, vals, B, n, 0.0, np.full((m, n), np.nan), n)
    assert np.array_equal(out, np.zeros((m, n)))


def pin_beta_zero_ignores_c0(spmm):
    m, k, n = 6, 5, 4
    rp, ci, vals = _random_csr(m, k, 12)
    B = rng.uniform(5, 1, k * n, -1, 1).reshape(k, n)
    nanC = np.full((m, n), np.nan)
    out, _ = spmm(m, k, n, 2.0, rp, ci, vals, B, n, 0.0, nanC, n)
    assert np.all(np.isfinite(out))
    assert np.allclose(out, 2.0 * (_to_dense(m, k, rp, ci, vals) @ B), rtol=1e-14, atol=1e-14)


def pin_linearity_in_b(spmm):
    """C(B1 + B2) == C(B1) + C(B2), exact on small integers."""
    m, k, n = 20, 15, 9
    rp, ci, _ = _random_csr(m, k, 13, dup=True)
    vals = rng.integers(13, 1, int(rp[-1]), -4, 4).astype(np.float64)
    B1 = rng.integers(13, 2, k * n, -4, 4).reshape(k, n).astype(np.float64)
    B2 = rng.integers(13, 3, k * n, -4, 4).reshape(k, n).astype(np.float64)
    o1, _ = spmm(m, k, n, 1.0, rp, ci, vals, B1, n, 0.0)
    o2, _ = spmm(m, k, n, 1.0, rp, ci, vals, B2, n, 0.0)
    o12, _ = spmm(m, k, n, 1.0, rp, ci, vals, B1 + B2, n, 0.0)
    assert np.array_equal(o1 + o2, o12)
    assert np.any(o12 != 0)


def pin_leading_dimensions(spmm):
    """Padding columns of B and C0 (filled with NaN) are never read."""
    m, k, n, ldb, ldc = 10, 8, 5, 11, 7
    rp, ci, vals = _random_csr(m, k, 14)
    B = rng.uniform(6, 1, k * n, -1, 1).reshape(k, n)
    C0 = rng.uniform(6, 2, m * n, -1, 1).reshape(m, n)
    Bp = np.full((k, ldb), np.nan)
    Bp[:, :n] = B
    Cp = np.full((m, ldc), np.nan)
    Cp[:, :n] = C0
    o_pad, _ = spmm(m, k, n, 1.25, rp, ci, vals, Bp, ldb, -0.5, Cp, ldc)
    o_ref, _ = spmm(m, k, n, 1.25, rp, ci, vals, B, n, -0.5, C0, n)
    assert np.array_equal(o_pad, o_ref)
    want = 1.25 * (_to_dense(m, k, rp, ci, vals) @ B) - 0.5 * C0
    assert np.allclose(o_ref, want, rtol=1e-13, atol=1e-13)


def pin_row_subset(spmm):
    m, k, n = 15, 12, 3
    rp, ci, vals = _random_csr(m, k, 15)
    B = rng.uniform(7, 1, k * n, -1, 1).reshape(k, n)
    C0 = rng.uniform(7, 2, m * n, -1, 1).reshape(m, n)
    full, fb = spmm(m, k, n, 0.5, rp, ci, vals, B, n, 2.0, C0, n)
    rows = np.array([14, 0, 7, 7, 3])
    sub, sb = spmm(m, k, n, 0.5, rp, ci, vals, B, n, 2.0, C0, n, rows=rows)
    assert np.array_equal(sub, full[rows]) and np.array_equal(sb, fb[rows])


def pin_error_bound_scale(spmm):
    m, k, n = 16, 11, 4
    rp, ci, vals = _random_csr(m, k, 16, dup=True)
    B = rng.uniform(8, 1, k * n, -1, 1).reshape(k, n)
    C0 = rng.uniform(8, 2, m * n, -1, 1).reshape(m, n)
    _, bound = spmm(m, k, n, -1.5, rp, ci, vals, B, n, 0.75, C0, n)
    absA = np.zeros((m, k))
    np.add.at(absA, (np.repeat(np.arange(m), np.diff(rp)), ci), np.abs(vals))
    want = 1.5 * (absA @ np.abs(B)) + 0.75 * np.abs(C0)
    assert np.allclose(bound, want, rtol=1e-13, atol=0)


def pin_k_zero(spmm):
    """k = 0: every row is empty, the result is beta * C0."""
    m, n = 4, 3
    C0 = rng.uniform(9, 1, m * n, -1, 1).reshape(m, n)
    out, _ = spmm(m, 0, n, 1.0, np.zeros(m + 1, np.int32), np.zeros(0, np.int32),
                  np.zeros(0), np.zeros((0, n)), n, 0.5, C0, n)
    assert np.array_equal(out, 0.5 * C0)


PINS = [pin_page_known_values, pin_hand_derived_3x4, pin_dense_bruteforce, pin_integer_exact,
        pin_identity, pin_alpha_zero, pin_beta_zero_ignores_c0, pin_linearity_in_b,
        pin_leading_dimensions, pin_row_subset, pin_error_bound_scale, pin_k_zero]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.spmm)


def test_csr_check():
    assert oracle.csr_check(2, 3, np.array([0, 2, 4]), np.array([0, 2, 1, 2])) == oracle.OK
    assert oracle.csr_check(2, 3, np.array([1, 2, 4]), np.array([0, 2, 1, 2])) == oracle.BAD_CSR
    assert oracle.csr_check(2, 3, np.array([0, 3, 2]), np.array([0, 2])) == oracle.BAD_CSR
    assert oracle.csr_check(2, 3, np.array([0, 2, 4]), np.array([0, 3, 1, 2])) == oracle.BAD_CSR
    assert oracle.csr_check(2, 3, np.array([0, 2, 4]), np.array([0, -1, 1, 2])) == oracle.BAD_CSR


def test_oracle_rejects_out_of_range_columns():
    with pytest.raises(ValueError):
        oracle.spmm(1, 2, 1, 1.0, np.array([0, 1]), np.array([5]), np.ones(1), np.ones((2, 1)),
                    1, 0.0)


def test_oracle_on_generated_problem_matches_dense():
    p = uniform_rows(50, 40, 12, 6, seed=21)
    out, bound = oracle.spmm_problem(p)
    want = p.alpha * (_to_dense(p.m, p.k, p.row_ptr, p.col_idx, p.values.astype(np.float64))
                      @ p.B.astype(np.float64)) + p.beta * p.C0.astype(np.float64)
    assert np.all(np.abs(out - want) <= 1e-13 * bound)


# ---------------------------------------------------------------------------
# planted mistakes: each broken copy of the oracle must fail at least one pin
# ---------------------------------------------------------------------------

MUTANTS = {
    "dropped_beta_term": ("v += beta * c0;", "v += 0.0 * c0;"),
    "beta_coefficient_one": ("v += beta * c0;", "v += c0;"),
    "alpha_not_applied": ("double v = alpha * acc[c];", "double v = acc[c];"),
    "wrong_sign": ("acc[c] += a * b;", "acc[c] -= a * b;"),
    "ldb_ignored": ("load(B, j * ldb + c, esize)", "load(B, j * n + c, esize)"),
    "transposed_b": ("load(B, j * ldb + c, esize)", "load(B, c * ldb + j, esize)"),
    "row_index_for_column": ("int64_t j = col_idx[p];", "int64_t j = i;"),
    "ldc_ignored": ("double c0 = load(C0, i * ldc + c, esize);\n                v += beta * c0;",
                    "double c0 = load(C0, i * n + c, esize);\n                v += beta * c0;"),
    "last_entry_dropped": ("for (int64_t p = row_ptr[i]; p < (int64_t)row_ptr[i + 1]; ++p) {\n"
                           "            int64_t j",
                           "for (int64_t p = row_ptr[i]; p < (int64_t)row_ptr[i + 1] - 1; ++p) {\n"
                           "            int64_t j"),
    "accumulator_not_reset": ("acc[c] = 0.0;\n            absacc[c] = 0.0;",
                              "absacc[c] = 0.0;"),
    "beta_zero_reads_c0": ("if (beta != 0.0) {                   /* C0 read only when beta != 0 */",
                           "if (1) {"),
    "bound_without_abs": ("absacc[c] += fabs(a) * fabs(b);", "absacc[c] += a * b;"),
    "alpha_zero_reads_b": ("if (alpha == 0.0) {                      /* A and B not referenced */",
                           "if (0) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "spmm_oracle.c")).read()
    old, new = MUTANTS[name]
    # the anchor's first occurrence lies in oracle_spmm (the squared chain,
    # further down the file, has its own mutants in test_oracle_squared.py)
    assert src.count(old) >= 1 and src.index(old) < src.index("int oracle_spmm_squared("), name
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(so), str(mutated), "-lm"], check=True)
    # run the pins in a child process: a mutant that reads out of bounds may crash
    code = ("import sys; sys.path[:0] = [%r, %r]\n"
            "import oracle, test_oracle as t\n"
            "lib = oracle.load_library(%r)\n"
            "bad = t.failing_pins(lambda *a, **k: oracle.spmm(*a, _lib=lib, **k))\n"
            "print('FAILED:' + ','.join(bad))\n") % (os.path.dirname(HERE), HERE, str(so))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode == 0:
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED:")][-1]
        assert line != "FAILED:", f"mutant {name} passed every pin"
    else:
        assert r.returncode < 0 or "Error" in r.stderr, r.stderr  # crashed: caught


def failing_pins(spmm):
    failed = []
    for pin in PINS:
        try:
            pin(spmm)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    return failed

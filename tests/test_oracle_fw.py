"""Pins for the Frank-Wolfe gradient-scan oracle (no GPU).

The scan is the step after the product in SEACells (bixverse page,
seacells_kernels.rs, `fw_argmin_b` and `reduce_argmin_blocks`): with
G = K2B t1 - K2At, it returns per column the minimum of G over rows (the
lowest row on ties) and gap = sum of B * G over B's stored entries.  The
pins tie ``oracle.fw_argmin`` to hand-derived values, to numpy on dense
matrices, and to the page's own test expectations (ties go to row 0, empty
K2B rows still take part, the scan starts from the largest finite value).
"""
import json
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

import oracle
from synth import rng

HERE = os.path.dirname(os.path.abspath(__file__))
F32_MAX = float(np.finfo(np.float32).max)


def dense_to_csr(a):
    """Row-major dense -> (row_ptr, col_idx, values) of its non-zeros."""
    rows, cols = np.nonzero(a)
    rp = np.zeros(a.shape[0] + 1, np.int64)
    np.cumsum(np.bincount(rows, minlength=a.shape[0]), out=rp[1:])
    return rp, cols, a[rows, cols]


def random_dense(shape, seed, stream, zero_frac):
    v = rng.uniform(seed, stream, int(np.prod(shape)), -1.0, 1.0).reshape(shape)
    z = rng.uniform(seed, stream + 100, int(np.prod(shape))).reshape(shape) < zero_frac
    v[z] = 0.0
    return v


def dense_case(n, k, seed):
    return (random_dense((n, k), seed, 1, 0.6), random_dense((k, k), seed, 2, 0.5),
            random_dense((n, k), seed, 3, 0.7), random_dense((n, k), seed, 4, 0.9))


def run(fw, k2b, t1, t2, b, dtype=np.float64):
    n, k = k2b.shape
    c = lambda a: tuple(np.asarray(x) for x in dense_to_csr(a.astype(dtype)))  # noqa: E731
    return fw(n, k, c(k2b), c(t1), c(t2), c(b))


def pin_hand_derived(fw):
    g = json.load(open(os.path.join(HERE, "golden", "fw_argmin_hand.json")))
    for c in g["cases"]:
        mats = [tuple(np.array(x) for x in c[name]) for name in ("k2b", "t1", "t2", "b")]
        mats = [(rp, ci, v.astype(np.float64)) for rp, ci, v in mats]
        r = fw(c["n"], c["k"], *mats)
        assert np.array_equal(r["min_val"], c["min_val"]), c["name"]
        assert np.array_equal(r["min_idx"], c["min_idx"]), c["name"]
        assert r["gap"] == c["gap"], c["name"]


def pin_dense_numpy(fw):
    for n, k, seed in ((40, 7, 1), (257, 33, 2)):
        k2b, t1, t2, b = dense_case(n, k, seed)
        r = run(fw, k2b, t1, t2, b)
        G = k2b @ t1 - t2
        assert np.allclose(r["min_val"], G.min(axis=0), rtol=0, atol=1e-12)
        # numpy's argmin takes the first (lowest) row; only exact ties could differ
        assert np.array_equal(r["min_idx"], np.argmin(G, axis=0))
        assert abs(r["gap"] - float((b * G).sum())) <= 1e-12 * max(1.0, r["gap_bound"])
        gb = np.abs(k2b) @ np.abs(t1) + np.abs(t2)
        assert np.allclose(r["col_scale"], gb.max(axis=0), rtol=1e-13)
        assert np.isclose(r["gap_bound"], float((np.abs(b) * gb).sum()), rtol=1e-13)


def pin_tie_goes_to_lowest_row(fw):
    """The page's tie test: t1 = I, K2At = 0, every row of K2B equal, so every
    row ties in every column and the scan must report row 0."""
    n, k = 2048, 4
    k2b = np.tile(-1.0 - np.arange(k, dtype=np.float64), (n, 1))
    r = run(fw, k2b, np.eye(k), np.zeros((n, k)), np.zeros((n, k)))
    assert np.array_equal(r["min_idx"], np.zeros(k))
    assert np.array_equal(r["min_val"], -1.0 - np.arange(k))


def pin_empty_rows_take_part(fw):
    n, k = 64, 9
    k2b, t1, t2, b = dense_case(n, k, 3)
    k2b[::3] = 0.0
    r = run(fw, k2b, t1, t2, b)
    G = k2b @ t1 - t2
    assert np.array_equal(r["min_idx"], np.argmin(G, axis=0))


def pin_gradient_rows(fw):
    n, k = 30, 6
    k2b, t1, t2, _ = dense_case(n, k, 5)
    c = lambda a: dense_to_csr(a)  # noqa: E731
    g, gb = oracle.fw_gradient(n, k, c(k2b), c(t1), c(t2), rows=np.array([29, 0, 7]))
    want = (k2b @ t1 - t2)[[29, 0, 7]]
    assert np.allclose(g, want, rtol=0, atol=1e-13)


def pin_start_value_and_empty(fw):
    """n = 0: the scan never moves from the largest finite value and row 0;
    the same holds for a column whose G never falls below it."""
    k = 3
    e = (np.zeros(1, np.int64), np.zeros(0, np.int64), np.zeros(0, np.float32))
    t1 = (np.zeros(k + 1, np.int64), np.zeros(0, np.int64), np.zeros(0, np.float32))
    r = fw(0, k, e, t1, e, e)
    assert np.array_equal(r["min_val"], np.full(k, F32_MAX)) and r["gap"] == 0.0
    assert np.array_equal(r["min_idx"], np.zeros(k))
    # binary32 rows whose G is +inf in column 0 (K2At = -inf there)
    n = 2
    t2 = np.array([[-np.inf, 1.0], [-np.inf, 2.0]], np.float32)
    r = run(fw, np.zeros((n, 2)), np.eye(2), t2, np.zeros((n, 2)), dtype=np.float32)
    assert r["min_val"][0] == F32_MAX and r["min_idx"][0] == 0
    assert r["min_val"][1] == -2.0 and r["min_idx"][1] == 1


def pin_duplicates_add(fw):
    """Stored duplicates each contribute, in K2B, t1, K2At and B."""
    n, k = 1, 2
    k2b = (np.array([0, 2]), np.array([0, 0]), np.array([1.0, 2.0]))       # 3 at (0,0)
    t1 = (np.array([0, 2, 2]), np.array([1, 1]), np.array([1.0, 1.0]))      # 2 at (0,1)
    t2 = (np.array([0, 2]), np.array([1, 1]), np.array([0.5, 0.5]))        # 1 at (0,1)
    b = (np.array([0, 2]), np.array([1, 1]), np.array([1.0, 1.0]))         # 2 at (0,1)
    r = fw(n, k, k2b, t1, t2, b)
    # G = [0, 3*2 - 1] = [0, 5]; gap = 2 * 5
    assert np.array_equal(r["min_val"], [0.0, 5.0]) and r["gap"] == 10.0


PINS = [pin_hand_derived, pin_dense_numpy, pin_tie_goes_to_lowest_row, pin_empty_rows_take_part,
        pin_gradient_rows, pin_start_value_and_empty, pin_duplicates_add]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_fw_oracle_pin(pin):
    pin(oracle.fw_argmin)


def test_fw_oracle_rejects_bad_csr():
    bad = (np.array([0, 1]), np.array([5]), np.array([1.0]))
    ok1 = (np.array([0, 0, 0]), np.zeros(0, np.int64), np.zeros(0))
    okn = (np.array([0, 0]), np.zeros(0, np.int64), np.zeros(0))
    with pytest.raises(ValueError):
        oracle.fw_argmin(1, 2, bad, ok1, okn, okn)


MUTANTS = {
    "t2_added": ("        g[c] -= t;\n", "        g[c] += t;\n"),
    "t1_transposed": ("for (int64_t q = t1_rp[m]; q < (int64_t)t1_rp[m + 1]; ++q) {\n"
                      "            int64_t c = t1_ci[q];",
                      "for (int64_t q = t1_rp[m]; q < (int64_t)t1_rp[m + 1]; ++q) {\n"
                      "            int64_t c = m; m = t1_ci[q];"),
    "tie_to_last_row": ("if (g[c] < min_val[c]) {", "if (g[c] <= min_val[c]) {"),
    "argmax": ("if (g[c] < min_val[c]) {", "if (g[c] > min_val[c]) {"),
    "gap_without_b": ("*gap += b * g[c];", "*gap += g[c];"),
    "gap_of_k2b_not_g": ("*gap += b * g[c];", "*gap += b;"),
    "start_zero": ("min_val[c] = start;", "min_val[c] = 0.0;"),
    "row_not_reset": ("    for (int64_t c = 0; c < k; ++c) {\n        g[c] = 0.0;\n        gb[c] = 0.0;\n    }",
                      "    for (int64_t c = 0; c < k; ++c) {\n        gb[c] = 0.0;\n    }"),
    "k2b_value_ignored": ("double v = load(k2b_v, p, esize);", "double v = 1.0;"),
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
            "import oracle, test_oracle_fw as t\n"
            "lib = oracle.load_library(%r)\n"
            "bad = t.failing_pins(lambda *a, **k: oracle.fw_argmin(*a, _lib=lib, **k), lib)\n"
            "print('FAILED:' + ','.join(bad))\n") % (os.path.dirname(HERE), HERE, str(so))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode == 0:
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED:")][-1]
        assert line != "FAILED:", f"mutant {name} passed every pin"
    else:
        assert r.returncode < 0 or "Error" in r.stderr, r.stderr


def failing_pins(fw, lib=None):
    failed = []
    saved = oracle.fw_gradient
    if lib is not None:     # pin_gradient_rows calls fw_gradient directly
        oracle.fw_gradient = lambda *a, **k: saved(*a, _lib=lib, **k)
    try:
        for pin in PINS:
            try:
                pin(fw)
            except (AssertionError, ValueError):
                failed.append(pin.__name__)
    finally:
        oracle.fw_gradient = saved
    return failed

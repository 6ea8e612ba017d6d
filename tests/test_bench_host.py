"""Host-side arithmetic of bench.py (no GPU): the clock-sample parser and the
algorithmic byte counts behind the roofline and GB/s figures."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import knn_kernel_graph, power_law, uniform_rows  # noqa: E402


def test_clock_samples_median_max_and_reasons():
    text = "\n".join([
        "0, 2070, 2070, 812.3, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2010, 2070, 1200.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "",
    ])
    c = bench.parse_clock_samples(text)
    assert c["samples"] == 3 and c["sm_mhz"] == 2010.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    hot = "0, 1500, 2070, 900, 0x8, Active, Not Active, Active, Not Active"
    assert bench.parse_clock_samples(hot)["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.parse_clock_samples("")["samples"] == 0


def _all_short_profile(p):
    return {"rows_short": p.m, "rows_medium": 0, "long_nnz": 0}


def test_rows_kernel_bytes_equal_the_whole_product_when_every_row_is_short():
    for p in (knn_kernel_graph(500, 8, 12, 5, seed=1),                       # beta = 0
              uniform_rows(300, 200, 9, 4, seed=2, beta=0.5)):               # beta != 0
        assert bench.rows_kernel_bytes(p, _all_short_profile(p)) == p.algorithmic_bytes()


def test_rows_kernel_bytes_leave_the_long_rows_out():
    p = power_law(5000, 5000, 16, 100_000, 3000, seed=3)
    lens = np.diff(p.row_ptr)
    long_rows = lens >= 1024
    prof = {"rows_short": int((~long_rows).sum()), "rows_medium": 0,
            "long_nnz": int(lens[long_rows].sum())}
    got = bench.rows_kernel_bytes(p, prof)
    es = p.values.itemsize
    entries = p.nnz - prof["long_nnz"]
    want = (4 * (prof["rows_short"] + 1) + (4 + es) * entries
            + entries / p.nnz * es * p.k * p.n + 2 * es * p.n * prof["rows_short"])
    assert got == want and got < p.algorithmic_bytes()


def test_chain_bytes_and_flops():
    p = knn_kernel_graph(400, 6, 10, 4, seed=4)
    p.meta["chain"] = "squared"
    csr, mn = 4 * (p.m + 1) + 8 * p.nnz, 4 * p.m * p.n     # binary32, beta = 0
    # A twice, B once, the intermediate written and read once, C written
    assert bench.problem_bytes(p) == 2 * csr + mn + 2 * mn + mn
    assert bench.problem_flops(p) == 2 * (2 * p.nnz * p.n)


def test_reference_arm_line_on_cpu():
    """`bench.py --impl reference` runs the CPU oracle only (no GPU) and prints
    one JSON line with the contract's keys."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--workload", "tiny_uniform"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GFLOP/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["config"]["workload"] == "tiny_uniform"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


def test_roofline_names_the_binding_unit():
    """binary32 products are set against HBM; a binary64 product whose FP64
    instruction rate is the larger fraction of its peak reports the ALU
    bound, with both fractions on the line."""
    from synth import laplacian_2d
    p32 = uniform_rows(300, 200, 9, 4, seed=2, beta=0.5)
    r = bench.roofline_of(p32, 1e9, 1.0, 6800.0, 6e11)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and "fp64_frac" not in r
    assert abs(r["frac"] - 1e9 / 1e-3 / 1e9 / 6800.0) < 1e-4
    p64 = laplacian_2d(20, 32, seed=3)                      # alpha = 2, beta = -1
    # beta = -1: one FP64 instruction per entry and column, one per output
    assert bench.fp64_pipe_ops(p64) == p64.nnz * 32 + p64.m * 32
    ms = 2.0 * bench.fp64_pipe_ops(p64) / 1e12 * 1e3        # as if at 1 TFLOP/s
    r = bench.roofline_of(p64, 1e3, ms, 6800.0, 0.6e12)     # peak 1.2 TFLOP/s
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - 1.0 / 1.2) < 1e-3 and r["hbm_frac"] < r["frac"]
    p64.beta = 0.5                                           # general beta: a multiply more
    assert bench.fp64_pipe_ops(p64) == p64.nnz * 32 + 2 * p64.m * 32


def test_config_runs_cover_every_product_configuration_and_the_l2_window():
    """The line's `configs` object times the five product configurations once
    each, without the window, and SEACells once more with the persisting-L2
    window on B (its 80 MB B fits the set-aside)."""
    keys = [k for k, _, _ in bench.CONFIG_RUNS]
    assert len(keys) == len(set(keys))
    plain = [(k, w) for k, w, win in bench.CONFIG_RUNS if not win]
    assert [w for _, w in plain] == list(bench.PRODUCT_CONFIGS)
    assert all(k == w for k, w in plain)
    windowed = [(k, w) for k, w, win in bench.CONFIG_RUNS if win]
    assert windowed == [("seacells_knn_l2_window", "seacells_knn")]

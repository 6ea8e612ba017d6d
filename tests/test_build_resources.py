"""Register and spill budget of the kernels that matter, read from ptxas's
resource report (``-Xptxas -v``) while cross-compiling for sm_103a; no GPU
needed.  Guards against a change that makes the headline kernel spill or
drop below its occupancy target."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "csr_spmm_gb300", "csrc")


def _resources(unit):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    from csr_spmm_gb300 import build
    cmd = [nvcc] + build.NVCC_FLAGS + ["-Xptxas", "-v", "-c", os.path.join(CSRC, unit), "-o",
                                       os.devnull]
    err = subprocess.run(cmd, capture_output=True, text=True, check=True).stderr
    out, cur, spill = {}, None, None
    for line in err.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and cur:
            spill = (int(m.group(1)), int(m.group(2)))
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and cur:
            out[cur] = (int(m.group(1)), spill)
            cur = None
    return out


def _find(res, *parts):
    hits = [(k, v) for k, v in res.items() if all(p in k for p in parts)]
    assert hits, f"no kernel matching {parts}"
    return hits


def test_headline_rows_kernel_fits_full_occupancy():
    # rows_kernel<float, 4, 32, 1, false, true>: the SEACells-shaped product
    res = _resources("spmm_rows_f32.cu")
    (name, (regs, spill)), = _find(res, "rows_kernel", "IfLi4ELi32ELi1ELb0ELb1E")
    assert regs <= 64, (name, regs)                 # one 1024-thread block per SM
    assert spill[0] <= 64 and spill[1] <= 64, (name, spill)


def test_scan_and_ilu0_kernels_do_not_spill():
    for unit, kern in (("spmm_fw.cu", "fw_reduce"), ("spmm_ilu0.cu", "ilu0_factor"),
                       ("spmm_ilu0.cu", "ilu0_count")):
        for name, (regs, spill) in _find(_resources(unit), kern):
            assert spill == (0, 0), (name, spill)

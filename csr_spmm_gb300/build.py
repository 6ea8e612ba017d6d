"""Build the CUDA library ``csr_spmm_gb300/lib/libcsrspmm.so`` for sm_103a.

Each translation unit under ``csrc/`` is compiled by its own nvcc process
(in parallel), then the objects are linked into one shared library with the
CUDA runtime linked statically.  A rebuild happens only when a source,
header or flag changed (a content hash is kept beside the library).

Run ``python -m csr_spmm_gb300.build`` or call :func:`build`.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "libcsrspmm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++20", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build csr_spmm_gb300")


def _sources():
    units = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    deps = sorted(f for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    return units, deps


def _digest(units, deps, extra) -> str:
    h = hashlib.sha256()
    for name in units + deps:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    with open(os.path.join(INCLUDE, "csr_spmm.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + list(extra)).encode())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False, extra_flags=(), out: str = LIB,
          flag_units=None) -> str:
    """Compile and link the library if anything changed; return its path.

    ``extra_flags`` (e.g. -D tuning macros) and ``out`` build a variant
    library elsewhere, with its own object directory.  With ``flag_units``
    (names of .cu files) only those units are compiled with ``extra_flags``;
    the others are linked from the library's own objects, which are brought
    up to date first."""
    units, deps = _sources()
    if flag_units is not None:
        flag_units = sorted(flag_units)
        missing = [u for u in flag_units if u not in units]
        if missing:
            raise ValueError(f"no such units: {missing}")
        if out == LIB:
            raise ValueError("a build restricted to some units needs its own output path")
        build(verbose=verbose)
    digest = _digest(units, deps, list(extra_flags) + ["units:"] + list(flag_units or []))
    stamp = out + ".sha256"
    obj_dir = OBJ_DIR if out == LIB else out + ".objs"
    if not force and os.path.exists(out) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return out
    nvcc = _nvcc()
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(os.path.dirname(out), exist_ok=True)

    def compile_one(unit):
        if flag_units is not None and unit not in flag_units:
            return os.path.join(OBJ_DIR, unit[:-3] + ".o")      # the library's own object
        obj = os.path.join(obj_dir, unit[:-3] + ".o")
        cmd = [nvcc] + NVCC_FLAGS + list(extra_flags) + ["-c", os.path.join(CSRC, unit), "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {unit}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(len(units), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, units))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "--cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))

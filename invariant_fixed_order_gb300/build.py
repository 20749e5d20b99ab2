"""Builds libbi.so (the CUDA library behind include/bi.h) in-tree with nvcc.

Each translation unit is compiled for sm_103a only, in parallel, and linked
into ``invariant_fixed_order_gb300/_build/libbi.so``.  The GEMM floor
microbenchmarks (``csrc/probe_floor.cu``, run by ``bench.py --floor``) are
linked into a separate ``libbi_probe.so`` that nothing in the package loads.
A stamp of the sources' contents lets an unchanged tree skip the rebuild.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libbi.so")
PROBE_LIB = os.path.join(BUILD, "libbi_probe.so")
UNITS = ["api.cu", "k_rows.cu", "k_attention.cu", "k_gemm.cu", "k_logits.cu"]
PROBE_UNITS = ["probe_floor.cu"]
HEADERS = ["common.cuh", "internal.h", "tc_ptx.cuh", "prefill_tc.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _stamp() -> str:
    h = hashlib.sha256()
    files = [os.path.join(CSRC, f) for f in UNITS + PROBE_UNITS + HEADERS] + [os.path.join(ROOT, "include", "bi.h")]
    for f in files:
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + FLAGS).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    stamp = _stamp()
    stamp_file = os.path.join(BUILD, "libbi.stamp")
    if not force and os.path.exists(LIB) and os.path.exists(PROBE_LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as fh:
            if fh.read().strip() == stamp:
                return LIB
    cc = nvcc()
    objs = []

    def compile_unit(unit: str) -> str:
        src = os.path.join(CSRC, unit)
        obj = os.path.join(BUILD, unit.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {unit}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(UNITS + PROBE_UNITS)) as ex:
        objs = list(ex.map(compile_unit, UNITS + PROBE_UNITS))
    for lib, lib_objs in ((LIB, objs[:len(UNITS)]), (PROBE_LIB, objs[len(UNITS):])):
        tmp = lib + ".tmp"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *lib_objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    with open(stamp_file, "w") as fh:
        fh.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""Build libgdn_scan.so in-tree for sm_103a (nvcc; translation units in parallel)."""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build", "gdn_scan")
LIB = os.path.join(PKG, "libgdn_scan.so")
SOURCES = ["gdn_api.cu", "gdn_noalloc.cu", "gdn_placement.cpp", "gdn_group.cu", "gdn_tprep.cu", "inst_chunk_tc.cu",
           "inst_chunk_tc_pre.cu", "inst_dk32.cu", "inst_dk64.cu", "inst_dk128.cu"]
HEADERS = [os.path.join(CSRC, f) for f in ("gdn_kernel.cuh", "gdn_chunk.cuh", "gdn_chunk_tc.cuh", "gdn_group.cuh")] + [
    os.path.join(ROOT, "include", "gdn_scan.h")]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + HEADERS):
            jobs.append(["nvcc", *NVCC_FLAGS, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 1)) as ex:
            list(ex.map(run, jobs))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=False))

"""Builds libpgg.so (the C-ABI library) in-tree with nvcc for sm_103a.

Ten translation units compiled in parallel, then linked as a shared
library with the CUDA runtime linked statically; the driver API is reached at
run time through cudaGetDriverEntryPointByVersion, so loading the library
needs no libcuda.

build(checks=True) makes the checked build, libpgg_checks.so in its own
folder: the same sources compiled with -DPGG_CHECKS, which turns on the
kernels' device bounds checks (a failed check writes PGG_ERR_CHECK to the
status word and keeps the access in bounds; nothing traps).
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libpgg.so")
CHECKS_DIR = os.path.join(OUT_DIR, "checks")
LIB_CHECKS = os.path.join(CHECKS_DIR, "libpgg_checks.so")
SOURCES = ["pgg_api.cu", "route_prep.cu", "gmm_dx.cu", "gmm_dx_simt.cu", "gmm_dw.cu",
           "gmm_dw_simt.cu", "gmm_fwd.cu", "gmm_fwd_simt.cu", "unpermute_grad.cu",
           "gmm_dx_owner.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return [*ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
            "-I", INCLUDE, "-I", CSRC, *extra]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), checks: bool = False) -> str:
    out_dir = CHECKS_DIR if checks else OUT_DIR
    lib = LIB_CHECKS if checks else LIB
    if checks:
        extra_flags = (*extra_flags, "-DPGG_CHECKS")
    os.makedirs(out_dir, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "pgg.h"))
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, *headers, __file__]):
            jobs.append([nvcc(), *_flags(extra_flags), "-c", s, "-o", o])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.check_call(cmd)

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        run([nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, checks="--checks" in sys.argv))

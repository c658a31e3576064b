"""Build libgbattn.so in-tree with nvcc for sm_103a.

The kernel instantiations compile as one translation unit per head dimension
(inst.cu with -DGBATTN_HEAD_DIM=<D>), in parallel, plus the C-ABI unit and
the linear cross-entropy unit (lce.cu); the objects link into
bwd_flashattention_fwd_gb300/libgbattn.so (no library besides the CUDA
runtime).  checks.cu becomes libgbattn_checks.so, a test aid.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libgbattn.so")
CHECKS_LIB = os.path.join(PKG, "libgbattn_checks.so")  # device checks of the kernels' math helpers (tests only)
DEBUG_LIB = os.path.join(PKG, "libgbattn_debug.so")  # index checks compiled in (GBATTN_DEBUG_CHECKS)
HEAD_DIMS = (64, 96, 128, 256)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources_mtime() -> float:
    t = 0.0
    for d in (CSRC, os.path.join(ROOT, "include")):
        for f in os.listdir(d):
            t = max(t, os.path.getmtime(os.path.join(d, f)))
    return t


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile (if stale) and return the path of libgbattn.so (with debug:
    libgbattn_debug.so, the kernels' index checks compiled in)."""
    lib = DEBUG_LIB if debug else LIB
    outs_needed = (lib,) if debug else (LIB, CHECKS_LIB)
    if not force and all(os.path.exists(p) and os.path.getmtime(p) >= _sources_mtime() for p in outs_needed):
        return lib
    nvcc = _nvcc()
    bdir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(bdir, exist_ok=True)
    flags = [*FLAGS, *extra_flags] + (["-DGBATTN_DEBUG_CHECKS"] if debug else [])
    jobs = []
    for d in HEAD_DIMS:
        obj = os.path.join(bdir, f"inst_d{d}.o")
        jobs.append([nvcc, *ARCH, *flags, f"-DGBATTN_HEAD_DIM={d}", "-c", os.path.join(CSRC, "inst.cu"), "-o", obj])
    for unit in ("api", "lce"):
        jobs.append([nvcc, *ARCH, *flags, "-c", os.path.join(CSRC, unit + ".cu"), "-o", os.path.join(bdir, unit + ".o")])
    checks_obj = os.path.join(bdir, "checks.o")
    if not debug:
        jobs.append([nvcc, *ARCH, *flags, "-c", os.path.join(CSRC, "checks.cu"), "-o", checks_obj])
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(_run, jobs))
    if verbose:
        for o in outs:
            sys.stdout.write(o)
    objs = [j[-1] for j in jobs if j[-1] != checks_obj]
    tmp = lib + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib)
    if not debug:
        tmp = CHECKS_LIB + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-o", tmp, checks_obj])
        os.replace(tmp, CHECKS_LIB)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else (), debug="--debug" in sys.argv))

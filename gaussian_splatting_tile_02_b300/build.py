"""Builds libgs_b300.so (the C-ABI renderer library) in-tree with nvcc for sm_103a,
and libgs_b300_debug.so, the same sources with the kernels' index checks on
(GS_DEBUG_CHECKS: failures are counted into a device counter, never trapped)."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libgs_b300.so")
DEBUG_LIB = os.path.join(HERE, "libgs_b300_debug.so")
SOURCES = ["api.cu", "preprocess.cu", "binning.cu", "sort.cu", "rasterize.cu", "backward.cu", "splat2d.cu", "densify.cu",
           "bin_static.cu", "measure.cu", "tiledepth.cu", "tilelen.cu"]
HEADERS = ["gs_internal.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "gs.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra: list | None = None, debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    if not force and up_to_date(lib):
        return lib
    tmp = lib + f".{os.getpid()}.tmp"
    defs = ["-DGS_DEBUG_CHECKS"] if debug else []
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *defs, *(extra or []), "-I", os.path.join(ROOT, "include"),
           *[os.path.join(CSRC, f) for f in SOURCES], "-o", tmp]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.check_call(cmd)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    force = "--force" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None
    print(build(force=force or bool(extra), verbose=True, extra=extra, debug="--debug" in sys.argv))

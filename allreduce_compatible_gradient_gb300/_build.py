"""Compile the CUDA library (csrc/*.cu over csrc/gq_kernels.cuh) into libgq.so, in-tree.

Five translation units (the C ABI and the other kernels in gq.cu; the quantise launchers, one per
gradient type and scheme) compiled in parallel with one -gencode (sm_103a), then linked with the
static CUDA runtime: the library depends on nothing but the driver at load time.  -fmad=false
keeps every fp32 operation a separately rounded IEEE operation (the rounding decisions must be
bit-identical to their definition).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
UNITS = ["gq.cu", "gq_quant_f32_l.cu", "gq_quant_f32_e.cu", "gq_quant_bf16_l.cu",
         "gq_quant_bf16_e.cu"]
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgq.so")
# the same library with the kernels' bounds checks compiled in (-DGQ_DEBUG)
DEBUG_LIB = os.path.join(PKG, "libgq_debug.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + [os.path.join(ROOT, "include", "gq.h")])


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libgq.so")
    return cand


def compile_command(unit: str, obj: str, extra=()) -> list:
    return [nvcc(), ARCH, "-O3", "-lineinfo", "-fmad=false", "-std=c++17", "-Xcompiler", "-fPIC",
            "-I" + os.path.join(ROOT, "include"), *extra, "-c", "-o", obj,
            os.path.join(CSRC, unit)]


def link_command(objs: list, out: str) -> list:
    return [nvcc(), ARCH, "-shared", "-o", out, *objs]


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in sources())


def build_library(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build libgq.so (debug: libgq_debug.so, with -DGQ_DEBUG) if missing or older than its
    sources; return its path."""
    lib = DEBUG_LIB if debug else LIB
    if force or is_stale(lib):
        os.makedirs(OBJ_DIR, exist_ok=True)
        extra = (("-Xptxas", "-v") if verbose else ()) + (("-DGQ_DEBUG",) if debug else ())
        tag = ".%d%s" % (os.getpid(), ".dbg" if debug else "")
        objs = [os.path.join(OBJ_DIR, u[:-3] + tag + ".o") for u in UNITS]
        tmp = lib + ".tmp" + tag
        try:
            procs = [subprocess.Popen(compile_command(u, o, extra)) for u, o in zip(UNITS, objs)]
            codes = [p.wait() for p in procs]
            if any(codes):
                raise subprocess.CalledProcessError(next(c for c in codes if c), "nvcc")
            subprocess.run(link_command(objs, tmp), check=True)
            os.replace(tmp, lib)
        finally:
            for f in objs + [tmp]:
                if os.path.exists(f):
                    os.remove(f)
    return lib

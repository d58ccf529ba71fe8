"""Compile the CUDA library (csrc/gq.cu + csrc/gq_kernels.cuh) into libgq.so, in-tree.

One translation unit, one -gencode (sm_103a), static CUDA runtime: the library depends on
nothing but the driver at load time.  -fmad=false keeps every fp32 operation a separately
rounded IEEE operation (the rounding decisions must be bit-identical to their definition).
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", "gq.cu"), os.path.join(PKG, "csrc", "gq_kernels.cuh"),
           os.path.join(ROOT, "include", "gq.h")]
LIB = os.path.join(PKG, "libgq.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libgq.so")
    return cand


def command(out: str, extra=()) -> list:
    return [nvcc(), ARCH, "-O3", "-lineinfo", "-fmad=false", "-std=c++17", "-Xcompiler", "-fPIC",
            "-shared", "-I" + os.path.join(ROOT, "include"), *extra, "-o", out,
            os.path.join(PKG, "csrc", "gq.cu")]


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in SOURCES)


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Build libgq.so if missing or older than its sources; return its path."""
    if force or is_stale():
        tmp = LIB + ".tmp.%d" % os.getpid()
        extra = ("-Xptxas", "-v") if verbose else ()
        subprocess.run(command(tmp, extra), check=True)
        os.replace(tmp, LIB)
    return LIB

"""Compile the CUDA library ``liblowm_gemm.so`` in-tree for sm_103a.

One translation unit (``csrc/lowm_gemm.cu``, which includes the kernel and the
PTX wrappers), one ``-gencode``, no CMake: a few seconds with nvcc 13.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "liblowm_gemm.so")
SOURCES = [os.path.join(HERE, "csrc", "lowm_gemm.cu")]
DEPS = SOURCES + glob.glob(os.path.join(HERE, "csrc", "*.cuh")) + [os.path.join(ROOT, "include", "lowm_gemm.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build liblowm_gemm.so")


def command(out: str, extra=()) -> list:
    return [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
            "-I", os.path.join(ROOT, "include"), *extra, "-o", out, *SOURCES]


def build(force: bool = False, verbose: bool = False) -> str:
    """Build (if stale) and return the path of the shared library."""
    stale = force or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(p) for p in DEPS)
    if stale:
        tmp = LIB + ".%d.tmp" % os.getpid()
        cmd = command(tmp, ("-Xptxas", "-v") if verbose else ())
        subprocess.check_call(cmd)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

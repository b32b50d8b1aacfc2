"""Compile the CUDA library ``liblowm_gemm.so`` in-tree for sm_103a.

Six translation units compiled in parallel with nvcc (one ``-gencode``,
no CMake): the host launcher and C ABI (``csrc/lowm_gemm.cu``) and the kernel
instances for 64- and 128-column tiles (``csrc/kernels_tile64.cu``,
``csrc/kernels_tile128.cu``) and for m_pad 128, 96 and 48
(``csrc/kernels_mpad128.cu``, ``csrc/kernels_mpad96.cu``,
``csrc/kernels_mpad48.cu``), then linked into one shared library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "liblowm_gemm.so")
CSRC = os.path.join(HERE, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in ("lowm_gemm.cu", "kernels_tile64.cu", "kernels_tile128.cu",
                                           "kernels_mpad128.cu", "kernels_mpad96.cu", "kernels_mpad48.cu")]
DEPS = SOURCES + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + [
    os.path.join(ROOT, "include", "lowm_gemm.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build liblowm_gemm.so")


def compile_command(src: str, obj: str, extra=()) -> list:
    return [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I",
            os.path.join(ROOT, "include"), *extra, "-c", "-o", obj, src]


def build(force: bool = False, verbose: bool = False) -> str:
    """Build (if stale) and return the path of the shared library."""
    stale = force or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(p) for p in DEPS)
    if not stale:
        return LIB
    tag = "%d" % os.getpid()
    objs = [os.path.join(CSRC, os.path.basename(src) + "." + tag + ".o") for src in SOURCES]
    extra = ("-Xptxas", "-v") if verbose else ()
    procs = [subprocess.Popen(compile_command(src, obj, extra)) for src, obj in zip(SOURCES, objs)]
    codes = [p.wait() for p in procs]
    try:
        if any(codes):
            raise subprocess.CalledProcessError(max(codes), "nvcc (compile)")
        tmp = LIB + "." + tag + ".tmp"
        subprocess.check_call([nvcc(), ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

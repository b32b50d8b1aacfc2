"""CPU oracle for C[M,N] = A[M,K] . W[N,K]^T (bf16 in, bf16 out).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline call it; the CUDA library never does, and this module imports
nothing from it.  The arithmetic lives in ``oracle.c`` (plain C, host threads);
this module compiles it with the host C compiler and marshals numpy arrays.

Functions (all bf16 values travel as uint16 bit patterns):

* ``gemm_bf16_f64(A, W, nthreads)`` -> ``(C_bits, S)``: fp64 dot products in
  k order, rounded once to bf16 (round-to-nearest-even).  This is the plain
  definition of the product the TensorRT-LLM PR "Fix two synchronization gaps
  in the MiniMax M3 low-M split-K GEMM" (Hardware verification) compares the
  kernel's bf16 output against.
* ``exact_gemm_bf16(A, W)`` -> ``C_bits``: the same product with no rounding
  until the final bf16 rounding (fixed-point accumulation); used to pin the
  fp64 path, in the spirit of the exact-integer construction of the Triton
  issue "warpgroup_mma_wait does not properly synchronize across warpgroups".
* ``f64_to_bf16(x)`` / ``bf16_to_f64(bits)``: the single rounding and the
  exact decode.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (gcc, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-Wall", "-Wextra", "-shared", "-fPIC", "-o", tmp, _SRC, "-lpthread",
        ])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_gemm_bf16_f64.argtypes = [u16p, u16p, u16p, f64p] + [ctypes.c_int] * 4
        lib.oracle_gemm_bf16_f64.restype = ctypes.c_int
        lib.oracle_exact_gemm_bf16.argtypes = [u16p, u16p, u16p] + [ctypes.c_int] * 3
        lib.oracle_exact_gemm_bf16.restype = ctypes.c_int
        _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands are passed as uint16 bit patterns, got %s" % a.dtype)
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def gemm_bf16_f64(A, W, nthreads: int | None = None, want_sum: bool = True):
    """Return ``(C_bits [M,N] uint16, S [M,N] float64 or None)``."""
    A, W = _u16(A), _u16(W)
    if A.ndim != 2 or W.ndim != 2 or A.shape[1] != W.shape[1]:
        raise ValueError("A must be [M,K] and W [N,K]; got %s and %s" % (A.shape, W.shape))
    M, K = A.shape
    N = W.shape[0]
    C = np.empty((M, N), dtype=np.uint16)
    S = np.empty((M, N), dtype=np.float64) if want_sum else None
    rc = _load().oracle_gemm_bf16_f64(
        _ptr(A, ctypes.c_uint16), _ptr(W, ctypes.c_uint16), _ptr(C, ctypes.c_uint16),
        _ptr(S, ctypes.c_double) if S is not None else None,
        M, N, K, int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_gemm_bf16_f64 failed (%d)" % rc)
    return C, S


def exact_gemm_bf16(A, W):
    """Return ``C_bits [M,N]``: exact dot products rounded once to bf16."""
    A, W = _u16(A), _u16(W)
    if A.ndim != 2 or W.ndim != 2 or A.shape[1] != W.shape[1]:
        raise ValueError("A must be [M,K] and W [N,K]; got %s and %s" % (A.shape, W.shape))
    M, K = A.shape
    N = W.shape[0]
    C = np.empty((M, N), dtype=np.uint16)
    rc = _load().oracle_exact_gemm_bf16(
        _ptr(A, ctypes.c_uint16), _ptr(W, ctypes.c_uint16), _ptr(C, ctypes.c_uint16), M, N, K)
    if rc != 0:
        raise RuntimeError("oracle_exact_gemm_bf16 failed (%d)" % rc)
    return C


def f64_to_bf16(x) -> np.ndarray:
    """Elementwise fp64 -> bf16 bits, round-to-nearest-even, one rounding."""
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    out = np.fromiter((lib.oracle_f64_to_bf16_rne(float(v)) for v in x.ravel()),
                      dtype=np.uint16, count=x.size)
    return out.reshape(x.shape)


def bf16_to_f64(bits) -> np.ndarray:
    """Elementwise exact decode of bf16 bit patterns."""
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    out = np.fromiter((lib.oracle_bf16_to_f64(int(v)) for v in b.ravel()),
                      dtype=np.float64, count=b.size)
    return out.reshape(b.shape)

"""Comparison helpers shared by the GPU tests (no GEMM arithmetic here)."""
from __future__ import annotations

import math

import numpy as np


def ordered(bits: np.ndarray) -> np.ndarray:
    """Map bf16 patterns to integers that increase with the value (-0 and +0 adjacent)."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)


def ulp_distance(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two arrays of bf16 patterns."""
    return np.abs(ordered(got) - ordered(want))


def f32_bound(K: int, A_f64: np.ndarray, W_f64: np.ndarray) -> float:
    """Tolerance on the fp32 sums before rounding: 1e-5 * sqrt(K) * max|a| * max|w|."""
    return 1e-5 * math.sqrt(K) * float(np.abs(A_f64).max()) * float(np.abs(W_f64).max())


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 at |x| (2^(e-7) for normals, 2^-133 below 2^-126)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126.0)
    return np.exp2(e - 7.0)


def rne_f32_to_bf16(f: np.ndarray) -> np.ndarray:
    """torch's fp32 -> bf16 conversion (round to nearest even), as bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(f, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def assert_parity(C_bits, F, C_ref, S, tol):
    """The parity bar for random inputs.

    C_bits: kernel bf16 output; F: the kernel's fp32 sums before rounding;
    C_ref / S: the oracle's single-rounded bf16 values and fp64 sums;
    tol: the absolute bound on the fp32 sums.
      (1) |F - S| <= tol everywhere;
      (2) C_bits is exactly the round-to-nearest-even bf16 of F;
      (3) wherever tol <= ulp_bf16(S) / 4, C_bits is within 1 bf16 ulp of C_ref
          (there F and S are too close to round more than one step apart).
    Returns the number of outputs beyond 1 ulp (all of them where (3) does not apply).
    """
    err = np.abs(F - S)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, "fp32 error %.3g at %s > bound %.3g" % (err.max(), worst, tol)
    conv = rne_f32_to_bf16(F)
    bad = np.argwhere(conv != C_bits)
    assert bad.size == 0, "bf16 output is not RNE of the fp32 sums at %s" % bad[:6].tolist()
    d = ulp_distance(C_bits, C_ref)
    strict = tol <= bf16_ulp(S) / 4
    bad = np.argwhere((d > 1) & strict)
    assert bad.size == 0, "%d outputs beyond 1 ulp where the fp32 bound is below a quarter ulp; first %s" % (
        len(bad), bad[:6].tolist())
    return int(np.sum(d > 1))

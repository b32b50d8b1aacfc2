"""Comparison helpers shared by the GPU tests (no GEMM arithmetic here)."""
from __future__ import annotations

import json
import math
import os

import numpy as np

# One record per assert_parity call (shape, outputs beyond 1 ulp, exemptions);
# written to the file named by LOWM_PARITY_LOG at the end of the session.
PARITY_LOG: list = []

# The largest share of a problem's outputs that may take the cancellation
# exemption of assert_parity (rule (3)).
MAX_EXEMPT_FRACTION = 1e-2


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


def f32_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of fp32 at |x| (2^(e-23) for normals, 2^-149 below 2^-126)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126.0)
    return np.exp2(e - 23.0)


def rne_f32_to_bf16(f: np.ndarray) -> np.ndarray:
    """torch's fp32 -> bf16 conversion (round to nearest even), as bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(f, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _f64(x) -> np.ndarray:
    if hasattr(x, "to") and hasattr(x, "numpy"):
        import torch
        return x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def assert_parity(C_bits, F, C_ref, S, A, W, label: str = ""):
    """The parity bar for random inputs, on every output element.

    C_bits: the kernel's bf16 output; F: its fp32 sums before rounding (fp64
    array); C_ref / S: the oracle's single-rounded bf16 values and fp64 sums;
    A [M,K] / W [N,K]: the operands (torch bf16 or arrays).
      (1) |F - S| <= 1e-5 * sqrt(K) * max|a| * max|w| everywhere;
      (2) C_bits is exactly the round-to-nearest-even bf16 of F;
      (3) C_bits is within 1 bf16 ulp of C_ref on every output, except where
          the dot product cancels below fp32's own resolution: the bf16
          spacing at S is smaller than the fp32 spacing at
          R = sum_k |a_k * w_k| (the size of the terms and of the partial
          sums an fp32 accumulator carries), so that a single fp32 rounding
          of a partial sum can move the result by more than one bf16 ulp,
          whatever the summation order.  Exempt outputs still meet (1) and
          (2); at most MAX_EXEMPT_FRACTION of the outputs may be exempt.
    Returns the number of exempt outputs that are beyond 1 ulp.
    """
    A64, W64 = _f64(A), _f64(W)
    K = A64.shape[1]
    tol = f32_bound(K, A64, W64)
    F = np.asarray(F, dtype=np.float64)
    err = np.abs(F - S)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, "fp32 error %.3g at %s > bound %.3g" % (err.max(), worst, tol)
    conv = rne_f32_to_bf16(F)
    bad = np.argwhere(conv != C_bits)
    assert bad.size == 0, "bf16 output is not RNE of the fp32 sums at %s" % bad[:6].tolist()
    d = ulp_distance(C_bits, C_ref)
    R = np.abs(A64) @ np.abs(W64).T
    exempt = bf16_ulp(S) < f32_ulp(R)
    beyond = d > 1
    rec = {"label": label, "shape": [int(A64.shape[0]), int(W64.shape[0]), int(K)], "outputs": int(d.size),
           "beyond_1ulp": int(beyond.sum()), "max_ulp": int(d.max()) if d.size else 0,
           "exempt": int(exempt.sum()), "beyond_1ulp_exempt": int((beyond & exempt).sum())}
    if beyond.any():
        idx = np.argwhere(beyond)[:8]
        rec["worst"] = [{"at": [int(i) for i in ij], "ulp": int(d[tuple(ij)]), "S": float(S[tuple(ij)]),
                         "F_minus_S": float(F[tuple(ij)] - S[tuple(ij)]), "R": float(R[tuple(ij)])} for ij in idx]
    PARITY_LOG.append(rec)
    bad = np.argwhere(beyond & ~exempt)
    assert bad.size == 0, "%d outputs beyond 1 bf16 ulp of the oracle (%d exempt by cancellation); first %s" % (
        len(bad), int((beyond & exempt).sum()), bad[:6].tolist())
    assert exempt.sum() <= max(1, MAX_EXEMPT_FRACTION * d.size), \
        "%d of %d outputs cancel below fp32 resolution: too many to exempt" % (int(exempt.sum()), d.size)
    return int((beyond & exempt).sum())


def write_parity_log():
    path = os.environ.get("LOWM_PARITY_LOG")
    if path and PARITY_LOG:
        with open(path, "w") as f:
            json.dump(PARITY_LOG, f, indent=0)

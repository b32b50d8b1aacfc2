"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no GEMM arithmetic: it only draws operands.  Both the CUDA
path and the CPU oracle receive exactly the tensors made here.

Recipes (the shapes are the pages' workloads; no dataset is involved):

* ``"randn"``: A[M,K] and W[N,K] drawn i.i.d. from N(0,1) in fp32 with a CPU
  ``torch.Generator`` (A from ``seed``, W from ``seed + 1``), scaled by
  1/sqrt(K) and rounded to bf16 (round-to-nearest-even, torch's conversion).
* ``"int"``: the exact-integer construction of the Triton issue
  "warpgroup_mma_wait does not properly synchronize across warpgroups"
  (reproducer): A is all ones and W holds integers uniform in {-3..3}
  (from ``seed + 2``), so every partial sum of a dot product is an exact
  integer of magnitude at most 3*K.
"""
from __future__ import annotations

import math

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(rows: int, cols: int, seed: int, scale: float) -> torch.Tensor:
    """[rows, cols] bf16 on the CPU: N(0,1) * scale, rounded to bf16."""
    x = torch.randn((rows, cols), generator=_gen(seed), dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def make_problem(M: int, N: int, K: int, seed: int = 1234, kind: str = "randn"):
    """Return CPU bf16 tensors ``(A [M,K], W [N,K])`` for one GEMM."""
    if kind == "randn":
        s = 1.0 / math.sqrt(K) if K > 0 else 1.0
        return randn_bf16(M, K, seed, s), randn_bf16(N, K, seed + 1, s)
    if kind == "int":
        A = torch.ones((M, K), dtype=torch.bfloat16)
        W = torch.randint(-3, 4, (N, K), generator=_gen(seed + 2), dtype=torch.int32)
        return A, W.to(torch.bfloat16)
    raise ValueError("unknown input kind %r" % (kind,))


def bits(t: torch.Tensor):
    """uint16 numpy view of a CPU bf16 tensor's bit patterns."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor, got %s" % t.dtype)
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def from_bits(b) -> torch.Tensor:
    """CPU bf16 tensor from a uint16 numpy array of bit patterns."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)

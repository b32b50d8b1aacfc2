"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes a part of the oracle with something independent: values
worked out by hand from the bf16 format (golden files), the closed form of
the exact-integer construction in the Triton issue "warpgroup_mma_wait does
not properly synchronize across warpgroups", exact rational arithmetic on
tiny inputs, torch's own bf16 conversion, and algebraic invariants.  A dropped
term, a wrong sign or index, a transposed operand, a double rounding or a
truncation in the oracle fails at least one of them.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from split_bf16_gemm_swap_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- independent helpers
def frac_of_bf16(b: int) -> Fraction:
    """Exact value of a finite bf16 pattern, straight from the format."""
    s = -1 if b & 0x8000 else 1
    e = (b >> 7) & 0xFF
    m = b & 0x7F
    assert e != 0xFF
    if e == 0:
        return s * Fraction(m, 2 ** 133)
    return s * Fraction(128 + m, 128) * Fraction(2) ** (e - 127)


_POS = None


def _pos_values():
    global _POS
    if _POS is None:
        _POS = [frac_of_bf16(p) for p in range(0x7F80)]  # 0 .. largest finite, increasing
    return _POS


def rne_fraction(x: Fraction) -> int:
    """bf16 pattern nearest to the exact value x, ties to the even pattern."""
    vals = _pos_values()
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    top = vals[0x7F7F]
    if a >= top + (top - vals[0x7F7E]) / 2:
        return sign | 0x7F80
    lo, hi = 0, 0x7F7F                      # vals[lo] <= a < vals[hi] (or a == top)
    if a >= top:
        return sign | 0x7F7F
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if vals[mid] <= a:
            lo = mid
        else:
            hi = mid
    dlo, dhi = a - vals[lo], vals[hi] - a
    p = lo if (dlo < dhi or (dlo == dhi and lo % 2 == 0)) else hi
    return sign | p


def exact_dot(arow, wrow) -> Fraction:
    return sum((frac_of_bf16(int(a)) * frac_of_bf16(int(w)) for a, w in zip(arow, wrow)), Fraction(0))


def random_bf16_bits(rng, shape, emin, emax):
    """Finite bf16 patterns with exponent fields drawn in [emin, emax] and random signs."""
    e = rng.integers(emin, emax + 1, size=shape)
    m = rng.integers(0, 128, size=shape)
    s = rng.integers(0, 2, size=shape)
    return ((s << 15) | (e << 7) | m).astype(np.uint16)


# ---------------------------------------------------------------- rounding and decode
def test_decode_every_pattern_matches_torch():
    pats = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    finite = ((pats >> 7) & 0xFF) != 0xFF
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_to_f64(pats)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(ref[finite]))
    assert np.all(np.isnan(got[~finite]) == np.isnan(ref[~finite]))


def test_rounding_golden_cases():
    path = os.path.join(GOLDEN, "bf16_rounding.txt")
    n = 0
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        fields = line.split()
        x = float.fromhex(fields[0])
        want = int(fields[1], 16)
        got = int(oracle.f64_to_bf16(np.array([x]))[0])
        assert got == want, "%s: got %#06x want %#06x" % (fields[0], got, want)
        if x != 0 and abs(x) != float("inf") and want & 0x7FFF != 0x7F80:  # Fraction has no -0
            assert rne_fraction(Fraction(x)) == want, fields[0]
        n += 1
    assert n >= 20


def test_rounding_agrees_with_torch_on_fp32_values():
    # Values that fp32 holds exactly reach bf16 through torch's RNE conversion
    # with a single rounding, so both must agree bit for bit.
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-38).astype(np.float32),   # subnormal range of bf16
        (rng.standard_normal(5000) * 1e38).clip(-3.3e38, 3.3e38).astype(np.float32),
    ])
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_rounding_agrees_with_exact_rationals_off_fp32_grid():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(3000) * np.exp2(rng.integers(-140, 120, size=3000))
    got = oracle.f64_to_bf16(x)
    for xi, g in zip(x, got):
        assert int(g) == rne_fraction(Fraction(float(xi))), float(xi).hex()


# ---------------------------------------------------------------- exact brute force
@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 0), (2, 3, 5, 1), (3, 4, 16, 2), (4, 5, 33, 3)])
def test_tiny_shapes_against_exact_rationals(M, N, K, seed):
    rng = np.random.default_rng(seed)
    # moderate exponents: every fp64 partial sum is exact, so the fp64 path must
    # return the exact sum itself, not just the same rounding
    A = random_bf16_bits(rng, (M, K), 120, 134)
    W = random_bf16_bits(rng, (N, K), 120, 134)
    C, S = oracle.gemm_bf16_f64(A, W, nthreads=2)
    CX = oracle.exact_gemm_bf16(A, W)
    for r in range(M):
        for c in range(N):
            ex = exact_dot(A[r], W[c])
            assert Fraction(float(S[r, c])) == ex
            assert int(C[r, c]) == rne_fraction(ex)
            assert int(CX[r, c]) == rne_fraction(ex)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_exact_path_over_the_whole_exponent_range(seed):
    # subnormals to near-overflow: fp64 sums are no longer exact, the exact path must be
    rng = np.random.default_rng(100 + seed)
    M, N, K = 2, 3, 12
    A = random_bf16_bits(rng, (M, K), 0, 180)
    W = random_bf16_bits(rng, (N, K), 0, 180)
    CX = oracle.exact_gemm_bf16(A, W)
    for r in range(M):
        for c in range(N):
            assert int(CX[r, c]) == rne_fraction(exact_dot(A[r], W[c]))


def test_cancellation_needs_the_exact_path():
    # 2^60 + 1 + 2^-8 + 2^-30 - 2^60 (all bf16-representable terms): the fp64 sum in
    # k order absorbs the small terms into 2^60 and returns 0; the exact path keeps
    # them and rounds 1 + 2^-8 + 2^-30 once, up to 1 + 2^-7.  The fp64 path is the
    # oracle only where its sums are (near) exact, which the tests below confirm
    # for the benchmark's input distribution.
    vals = [float.fromhex("0x1p+60"), 1.0, float.fromhex("0x1p-8"), float.fromhex("0x1p-30"),
            float.fromhex("-0x1p+60")]
    W = torch.tensor([vals], dtype=torch.float64).to(torch.bfloat16)
    A = torch.ones((1, len(vals)), dtype=torch.bfloat16)
    assert W.to(torch.float64).tolist()[0] == vals
    CX = oracle.exact_gemm_bf16(inputs.bits(A), inputs.bits(W))
    assert int(CX[0, 0]) == rne_fraction(exact_dot(inputs.bits(A)[0], inputs.bits(W)[0])) == 0x3F81
    C, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    assert S[0, 0] == 0.0 and int(C[0, 0]) == 0


def test_gemm_rounds_the_sum_once():
    # Sums that sit 2^-30 off a bf16 tie: rounding the fp64 sum through fp32 first
    # would land exactly on the tie and pick the other neighbour.
    cases = [([1.0, 2.0 ** -8, 2.0 ** -30], 0x3F81),                   # just above 1 + 2^-8
             ([1.0, 2.0 ** -7, 2.0 ** -8, -(2.0 ** -30)], 0x3F81),     # just below 1 + 3*2^-8
             ([-1.0, -(2.0 ** -8), -(2.0 ** -30)], 0xBF81)]
    for vals, want in cases:
        W = torch.tensor([vals], dtype=torch.float64).to(torch.bfloat16)
        assert W.to(torch.float64).tolist()[0] == vals
        A = torch.ones((2, len(vals)), dtype=torch.bfloat16)
        C, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
        assert np.all(C == want), (vals, C)
        assert np.all(oracle.exact_gemm_bf16(inputs.bits(A), inputs.bits(W)) == want)


# ---------------------------------------------------------------- closed forms
def _runs(spec):
    out = []
    for run in spec.split(","):
        v, n = run.split("*")
        out += [int(v)] * int(n)
    return out


def test_closed_form_golden_rows():
    path = os.path.join(GOLDEN, "closed_form_small.txt")
    rows = 0
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        spec, total, pat = line.split()
        w = _runs(spec)
        assert sum(w) == int(total)
        W = torch.tensor([w], dtype=torch.float32).to(torch.bfloat16)
        A = torch.ones((3, len(w)), dtype=torch.bfloat16)
        C, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
        assert np.all(S == float(total))
        assert np.all(C == int(pat, 16)), (spec, C, pat)
        assert np.all(oracle.exact_gemm_bf16(inputs.bits(A), inputs.bits(W)) == int(pat, 16))
        rows += 1
    assert rows == 8


@pytest.mark.parametrize("M,N,K", [(16, 64, 32768), (4, 96, 4096), (1, 7, 100)])
def test_closed_form_integer_construction(M, N, K):
    A, W = inputs.make_problem(M, N, K, seed=5, kind="int")
    col = W.to(torch.int64).sum(dim=1)                       # exact integer column sums
    assert int(col.abs().max()) < 2 ** 24
    C, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W), nthreads=4)
    assert np.array_equal(S, np.broadcast_to(col.numpy().astype(np.float64), (M, N)))
    want = np.array([rne_fraction(Fraction(int(v))) for v in col], dtype=np.uint16)
    assert np.array_equal(C, np.broadcast_to(want, (M, N)))


def test_identity_weight_selects_columns():
    # W[c,k] = 1 if k == c else 0: C[r,c] = A[r,c] exactly.  A transposed operand
    # or a wrong index in the oracle reads the wrong element.
    M, N, K = 5, 40, 64
    A, _ = inputs.make_problem(M, N, K, seed=9)
    W = torch.zeros((N, K), dtype=torch.bfloat16)
    W[torch.arange(N), torch.arange(N)] = 1.0
    C, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    assert np.array_equal(C, inputs.bits(A)[:, :N])
    # a permutation: W[c, perm[c]] = 1 gives C[r,c] = A[r, perm[c]]
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(3))[:N]
    W = torch.zeros((N, K), dtype=torch.bfloat16)
    W[torch.arange(N), perm] = 1.0
    C, _ = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    assert np.array_equal(C, inputs.bits(A)[:, perm.numpy()])


# ---------------------------------------------------------------- invariants
def test_gemv_matches_numpy_within_fp64_bound():
    M, N, K = 1, 256, 4096
    A, W = inputs.make_problem(M, N, K, seed=21)
    a = A.to(torch.float64).numpy()
    w = W.to(torch.float64).numpy()
    _, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    ref = a @ w.T
    bound = K * 2.0 ** -52 * (np.abs(a) @ np.abs(w).T)
    assert np.all(np.abs(S - ref) <= bound)


def test_fp64_and_exact_paths_agree_on_the_bench_distribution():
    M, N, K = 4, 128, 4096
    A, W = inputs.make_problem(M, N, K, seed=1234)
    C, _ = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    assert np.array_equal(C, oracle.exact_gemm_bf16(inputs.bits(A), inputs.bits(W)))


def test_operand_swap_transposes_and_sign_is_odd():
    M, N, K = 3, 50, 257
    A, W = inputs.make_problem(M, N, K, seed=31)
    C, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    Ct, St = oracle.gemm_bf16_f64(inputs.bits(W), inputs.bits(A))
    assert np.array_equal(C, Ct.T) and np.array_equal(S, St.T)
    Cn, Sn = oracle.gemm_bf16_f64(inputs.bits(-A), inputs.bits(W))
    assert np.array_equal(Sn, -S)
    assert np.array_equal(Cn, C ^ np.uint16(0x8000))


def test_zero_and_empty_shapes():
    A = np.zeros((2, 8), dtype=np.uint16)
    W = np.zeros((3, 8), dtype=np.uint16)
    C, S = oracle.gemm_bf16_f64(A, W)
    assert np.all(C == 0) and np.all(S == 0)
    C, S = oracle.gemm_bf16_f64(np.zeros((2, 0), np.uint16), np.zeros((3, 0), np.uint16))
    assert C.shape == (2, 3) and np.all(C == 0)
    C, S = oracle.gemm_bf16_f64(np.zeros((0, 4), np.uint16), np.zeros((3, 4), np.uint16))
    assert C.shape == (0, 3)


def test_thread_count_does_not_change_bits():
    A, W = inputs.make_problem(4, 301, 512, seed=41)
    C1, S1 = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W), nthreads=1)
    C8, S8 = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W), nthreads=8)
    assert np.array_equal(C1, C8) and np.array_equal(S1, S8)


def test_oracle_rejects_non_bf16_operands():
    with pytest.raises(TypeError):
        oracle.gemm_bf16_f64(np.zeros((2, 2), np.float32), np.zeros((2, 2), np.uint16))
    with pytest.raises(ValueError):
        oracle.gemm_bf16_f64(np.zeros((2, 3), np.uint16), np.zeros((2, 2), np.uint16))

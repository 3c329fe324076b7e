"""Pins for the enclosure oracle (lo <= exact A @ B <= hi), independent of it.

The definitions come from the "enclosure-gemm" page (Method: the exact integer
S with exponent Q is rounded outward once; a zero remainder means lo == hi;
overflow saturates to the largest finite value inward and to infinity
outward; the subnormal range needs no special case.  Correctness: the exact
rational product is the reference, integer operands give lo == hi == the
ordinary product).  The checks use what the oracle does not compute itself:
hand-derived IEEE binary64 answers, numpy's BLAS product on exactly
representable cases, fractions.Fraction, and math.fsum (correctly rounded).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import normal_matrices, sample_rows, WORKLOADS

TINY = math.ldexp(1.0, -1074)
MAXF = float.fromhex("0x1.fffffffffffffp+1023")


def _enc(A, B):
    lo, hi = oracle.enclose_f64(np.array(A, dtype=np.float64), np.array(B, dtype=np.float64))
    return lo, hi


def _bits(x):
    return np.array([x], dtype=np.float64).view(np.uint64)[0]


# Hand-derived answers.  Each row: A (1 x K), B (K x 1), expected lo, hi.
HAND_CASES = [
    # 1 + 2^-60 lies strictly between 1 and the next double 1 + 2^-52.
    ([[1.0, 2.0**-60]], [[1.0], [1.0]], 1.0, 1.0 + 2.0**-52),
    # the negative mirror: truncation toward zero is the upper endpoint.
    ([[-1.0, -(2.0**-60)]], [[1.0], [1.0]], -(1.0 + 2.0**-52), -1.0),
    # 2^-1200 is below the smallest subnormal: [+0, 2^-1074].
    ([[2.0**-600]], [[2.0**-600]], 0.0, TINY),
    # -2^-1200: [-2^-1074, -0.0].
    ([[-(2.0**-600)]], [[2.0**-600]], -TINY, -0.0),
    # 3 * 2^-1074 is a subnormal, exactly representable.
    ([[3.0]], [[TINY]], 3 * TINY, 3 * TINY),
    # 2^1200 overflows: [max finite, +inf]; negative: [-inf, -max finite].
    ([[2.0**600]], [[2.0**600]], MAXF, math.inf),
    ([[-(2.0**600)]], [[2.0**600]], -math.inf, -MAXF),
    # 2^1023 + 2^1023 = 2^1024 overflows too.
    ([[2.0**1023, 2.0**1023]], [[1.0], [1.0]], MAXF, math.inf),
    # max finite is representable.
    ([[MAXF]], [[1.0]], MAXF, MAXF),
    # catastrophic cancellation: exactly 1.
    ([[1e300, 1.0, -1e300]], [[1.0], [1.0], [1.0]], 1.0, 1.0),
    # exact zero from cancellation: both endpoints +0.0.
    ([[1.5, -1.5]], [[2.0], [2.0]], 0.0, 0.0),
    # 1/3 is not a double: (0.1 * 3)... use 1 + 3*2^-54: between 1 and 1+2^-52.
    ([[1.0, 3 * 2.0**-54]], [[1.0], [1.0]], 1.0, 1.0 + 2.0**-52),
    # subnormal boundary: 2^-1022 - 2^-1074 (largest subnormal) + 2^-1075 lies
    # between the largest subnormal and the smallest normal.
    ([[2.0**-1022 - TINY, 2.0**-538]], [[1.0], [2.0**-537]], 2.0**-1022 - TINY, 2.0**-1022),
]


@pytest.mark.parametrize("A,B,lo,hi", HAND_CASES)
def test_hand_cases(A, B, lo, hi):
    glo, ghi = _enc(A, B)
    assert _bits(glo[0, 0]) == _bits(lo), (glo[0, 0].hex(), float(lo).hex())
    assert _bits(ghi[0, 0]) == _bits(hi), (ghi[0, 0].hex(), float(hi).hex())
    plo, phi = oracle.enclose_py(A, B)
    assert _bits(plo[0][0]) == _bits(lo) and _bits(phi[0][0]) == _bits(hi)


def test_integer_operands_equal_blas_product():
    # Integer entries below 2^20 with K = 64: every partial sum is an integer
    # below 2^53, so the BLAS product is exact and lo == hi == it.
    rng = np.random.default_rng(0)
    A = rng.integers(-(2**20), 2**20, size=(17, 64)).astype(np.float64)
    B = rng.integers(-(2**20), 2**20, size=(64, 9)).astype(np.float64)
    lo, hi = oracle.enclose_f64(A, B)
    ref = A @ B
    assert np.array_equal(lo, ref) and np.array_equal(hi, ref)


def _check_bracket(A, B, lo, hi):
    for i in range(A.shape[0]):
        for j in range(B.shape[1]):
            ex = oracle.exact_dot_fraction(A[i], B[:, j])
            l, h = float(lo[i, j]), float(hi[i, j])
            assert l <= ex <= h
            if l == h:
                assert Fraction(l) == ex
            else:
                # width of one representable step, and the exact value is not a double
                assert math.nextafter(l, math.inf) == h
                assert Fraction(l) != ex and (math.isinf(h) or Fraction(h) != ex)


@pytest.mark.parametrize("M,N,K,seed", [(3, 4, 8, 0), (5, 2, 33, 1), (2, 3, 128, 2)])
def test_random_normal_bracket_is_tight(M, N, K, seed):
    A, B = normal_matrices(M, N, K, seed)
    lo, hi = oracle.enclose_f64(A, B)
    _check_bracket(A, B, lo, hi)


def test_mixed_scales_and_subnormals():
    rng = np.random.default_rng(3)
    M, N, K = 4, 3, 12
    A = rng.standard_normal((M, K)) * np.exp2(rng.integers(-1070, 1000, size=(M, K)).astype(np.float64) / 1.0)
    B = rng.standard_normal((K, N)) * np.exp2(rng.integers(-200, 10, size=(K, N)).astype(np.float64))
    A[0, :3] = [TINY, -TINY, 5 * TINY]
    lo, hi = oracle.enclose_f64(A, B)
    _check_bracket(A, B, lo, hi)
    plo, phi = oracle.enclose_py(A, B)
    assert np.array_equal(np.array(plo).view(np.uint64), lo.view(np.uint64))
    assert np.array_equal(np.array(phi).view(np.uint64), hi.view(np.uint64))


def test_round_to_nearest_is_an_endpoint():
    # Operands with 26-bit significands make every product exact in binary64;
    # math.fsum then returns the correctly rounded sum, which must be lo or hi
    # and the nearer of the two.
    rng = np.random.default_rng(4)
    M, N, K = 6, 5, 40
    A = np.ldexp(rng.integers(-(2**26), 2**26, size=(M, K)).astype(np.float64), -20)
    B = np.ldexp(rng.integers(-(2**26), 2**26, size=(K, N)).astype(np.float64), -31)
    lo, hi = oracle.enclose_f64(A, B)
    for i in range(M):
        for j in range(N):
            rn = math.fsum(A[i, k] * B[k, j] for k in range(K))
            assert rn == lo[i, j] or rn == hi[i, j]
            ex = oracle.exact_dot_fraction(A[i], B[:, j])
            d_lo, d_hi = ex - Fraction(lo[i, j]), Fraction(hi[i, j]) - ex
            assert (rn == lo[i, j]) == (d_lo < d_hi or (d_lo == d_hi and rn == lo[i, j]))


def test_nonfinite_rejected():
    with pytest.raises(ValueError):
        oracle.enclose_f64(np.array([[1.0, np.nan]]), np.ones((2, 1)))
    with pytest.raises(ValueError):
        oracle.enclose_f64(np.ones((1, 2)), np.array([[np.inf], [1.0]]))


@pytest.mark.slow
def test_normal_workload_width_at_most_one_step():
    # The enclosure page reports width_ulps(lo, hi).max() == 1 for random
    # normal operands of exactly this shape (1024x4096 @ 4096x1024).  Check a
    # few seeded rows of the oracle against that, and the bracket exactly on
    # a handful of entries.
    w = WORKLOADS["enclose_normal"]
    A, B = w.generate()
    rows = sample_rows(w.M, w.seed, n=4)
    lo, hi = oracle.enclose_f64(A, B, rows=rows)
    step = np.array([[math.nextafter(x, math.inf) for x in r] for r in lo])
    assert np.all((hi == lo) | (hi == step))
    assert np.any(hi != lo)
    for r, i in enumerate(rows[:1]):
        for j in range(3):
            ex = oracle.exact_dot_fraction(A[i], B[:, j])
            assert lo[r, j] <= ex <= hi[r, j]

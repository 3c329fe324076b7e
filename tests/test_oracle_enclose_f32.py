"""Pins of the binary32 enclosure oracle (oracle.enclose_f32).

"enclosure-gemm", Usage: operands are float32 or float64; Correctness: the
pair brackets the exact product and, when the scaling is lossless, equals its
floor and ceiling in the format.  The pins below do not go through the
oracle's binary32 search:

* Closed forms written out by hand (subnormal steps, overflow, signed zero,
  cancellation, exactly representable sums).
* The binary64 oracle plus numpy rounding: binary32 values are binary64
  values, so no float lies strictly between the tightest double pair and the
  exact value, and the tightest float pair is that double pair rounded down
  and up to binary32.
* The Fraction brute force on tiny inputs.
"""
import numpy as np
import pytest

import oracle
from workloads import normal_matrices

F32 = np.float32
TINY = float(np.float32(2.0**-149))  # least positive subnormal
FMAX = float(np.finfo(np.float32).max)


def rd32(x):
    """Largest float32 <= x (x float64; may be +-inf)."""
    with np.errstate(over="ignore"):
        c = np.float32(x)
    return np.where(c.astype(np.float64) > x, np.nextafter(c, F32(-np.inf)), c).astype(F32)


def ru32(x):
    with np.errstate(over="ignore"):
        c = np.float32(x)
    return np.where(c.astype(np.float64) < x, np.nextafter(c, F32(np.inf)), c).astype(F32)


def bits(x):
    return np.ascontiguousarray(x, dtype=F32).view(np.uint32)


NEXT_ONE = float(np.nextafter(F32(1.0), F32(2.0)))  # 1 + 2^-23

# (A, B, lo, hi) written out from the definitions
CASES_F32 = [
    ([[1.0, TINY]], [[1.0], [1.0]], 1.0, NEXT_ONE),  # 1 + 2^-149
    ([[1.0, -TINY]], [[1.0], [1.0]], float(np.nextafter(F32(1.0), F32(0.0))), 1.0),
    ([[FMAX, FMAX]], [[1.0], [1.0]], FMAX, np.inf),  # 2 * max finite overflows upward only
    ([[-FMAX, -FMAX]], [[1.0], [1.0]], -np.inf, -FMAX),
    ([[TINY]], [[0.5]], 0.0, TINY),  # 2^-150 lies between 0 and the least subnormal
    ([[-TINY]], [[0.5]], -TINY, -0.0),
    ([[2.0**100, 1.0, -(2.0**100)]], [[1.0], [1.0], [1.0]], 1.0, 1.0),  # cancellation
    ([[3.0, 5.0]], [[7.0], [11.0]], 76.0, 76.0),
    ([[2.0**24, 1.0]], [[1.0], [1.0]], 2.0**24, 2.0**24 + 2.0),  # 2^24 + 1 is not a float
    ([[0.0, -0.0]], [[5.0], [7.0]], 0.0, 0.0),
    ([[TINY, TINY]], [[TINY], [TINY]], 0.0, TINY),  # 2^-297, far below the subnormals
]


@pytest.mark.parametrize("A,B,lo,hi", CASES_F32)
def test_hand_cases(A, B, lo, hi):
    glo, ghi = oracle.enclose_f32(np.array(A, dtype=F32), np.array(B, dtype=F32))
    assert bits(glo)[0, 0] == bits(np.array([lo], dtype=F32))[0]
    assert bits(ghi)[0, 0] == bits(np.array([hi], dtype=F32))[0]


def random_f32(M, N, K, seed, spread=0):
    rng = np.random.default_rng(seed)
    A, B = normal_matrices(M, N, K, seed)
    if spread:
        A = A * np.exp2(rng.integers(-spread, spread + 1, size=A.shape))
        B = B * np.exp2(rng.integers(-spread, spread + 1, size=B.shape))
    with np.errstate(over="ignore", under="ignore"):
        return A.astype(F32), B.astype(F32)


@pytest.mark.parametrize("M,N,K,seed,spread", [(7, 9, 33, 0, 0), (20, 30, 200, 1, 20), (10, 12, 64, 2, 60),
                                               (5, 6, 300, 3, 120)])
def test_equals_binary64_pair_rounded_outward(M, N, K, seed, spread):
    A, B = random_f32(M, N, K, seed, spread)
    lo64, hi64 = oracle.enclose_f64(A.astype(np.float64), B.astype(np.float64))
    lo, hi = oracle.enclose_f32(A, B)
    assert np.array_equal(bits(lo), bits(rd32(lo64)))
    assert np.array_equal(bits(hi), bits(ru32(hi64)))


def test_subnormal_range():
    """Products landing among the binary32 subnormals, both signs."""
    rng = np.random.default_rng(4)
    A = (rng.standard_normal((6, 16)) * 2.0**-70).astype(F32)
    B = (rng.standard_normal((16, 5)) * 2.0**-72).astype(F32)
    lo64, hi64 = oracle.enclose_f64(A.astype(np.float64), B.astype(np.float64))
    lo, hi = oracle.enclose_f32(A, B)
    assert np.array_equal(bits(lo), bits(rd32(lo64))) and np.array_equal(bits(hi), bits(ru32(hi64)))
    assert np.any(np.abs(lo) < np.finfo(F32).tiny)  # the case does reach the subnormals


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fraction_brute_force(seed):
    A, B = random_f32(3, 4, 6, seed, spread=30)
    lo, hi = oracle.enclose_f32(A, B)
    plo, phi = oracle.enclose_py(A, B, dtype=F32)
    assert np.array_equal(bits(lo), bits(np.array(plo, dtype=F32)))
    assert np.array_equal(bits(hi), bits(np.array(phi, dtype=F32)))


def test_rows_subset_and_nonfinite():
    A, B = random_f32(30, 8, 40, 5)
    lo, hi = oracle.enclose_f32(A, B)
    rows = np.array([0, 7, 29])
    slo, shi = oracle.enclose_f32(A, B, rows=rows)
    assert np.array_equal(bits(slo), bits(lo[rows])) and np.array_equal(bits(shi), bits(hi[rows]))
    A[3, 4] = np.inf
    with pytest.raises(ValueError):
        oracle.enclose_f32(A, B)

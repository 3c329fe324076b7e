"""Pins of the interval oracle (oracle.interval): Rump's midpoint-radius
product ("enclosure-gemm", Method: Rump's bound, its products and radius
formed exactly; Correctness: the returned pair must contain the exact product
of every choice of point operands in the intervals).

* Zero radii reduce it to the pinned point enclosure (oracle.enclose_f64/_f32).
* Integer operands keep every sum below 2^53, so numpy's int64 products give
  the exact bounds; and for intervals with mid >= rad >= 0 the upper bound is
  the product of the upper corners (a closed form of the bound).
* Containment of sampled corner products, formed exactly with Fraction.
* The Fraction brute force on tiny inputs, both formats.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import normal_matrices


def bits(x):
    x = np.ascontiguousarray(x)
    return x.view(np.uint32 if x.dtype == np.float32 else np.uint64)


def random_intervals(M, N, K, seed, dtype=np.float64, rad_scale=2.0**-20):
    rng = np.random.default_rng(seed)
    Am, Bm = normal_matrices(M, N, K, seed)
    Ar = np.abs(rng.standard_normal((M, K))) * rad_scale
    Br = np.abs(rng.standard_normal((K, N))) * rad_scale
    return tuple(x.astype(dtype) for x in (Am, Ar, Bm, Br))


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_zero_radius_is_the_point_enclosure(dtype):
    Am, _, Bm, _ = random_intervals(9, 11, 70, 0, dtype)
    lo, hi = oracle.interval(Am, np.zeros_like(Am), Bm, np.zeros_like(Bm))
    enc = oracle.enclose_f32 if dtype == np.float32 else oracle.enclose_f64
    rlo, rhi = enc(Am, Bm)
    assert np.array_equal(bits(lo), bits(rlo)) and np.array_equal(bits(hi), bits(rhi))


def test_integer_operands_exact_bounds():
    rng = np.random.default_rng(1)
    M, N, K = 13, 17, 40
    Am = rng.integers(-2000, 2000, size=(M, K))
    Ar = rng.integers(0, 300, size=(M, K))
    Bm = rng.integers(-2000, 2000, size=(K, N))
    Br = rng.integers(0, 300, size=(K, N))
    mid = Am @ Bm
    rad = np.abs(Am) @ Br + Ar @ np.abs(Bm) + Ar @ Br
    lo, hi = oracle.interval(*(x.astype(np.float64) for x in (Am, Ar, Bm, Br)))
    assert np.array_equal(lo, (mid - rad).astype(np.float64))
    assert np.array_equal(hi, (mid + rad).astype(np.float64))


def test_upper_bound_is_the_upper_corner_product_for_positive_intervals():
    """mid >= rad >= 0 everywhere: the largest point product is (Am+Ar)(Bm+Br), and Rump's bound reaches it."""
    rng = np.random.default_rng(2)
    M, N, K = 8, 9, 30
    Ar = rng.integers(0, 100, size=(M, K))
    Am = Ar + rng.integers(0, 1000, size=(M, K))
    Br = rng.integers(0, 100, size=(K, N))
    Bm = Br + rng.integers(0, 1000, size=(K, N))
    _, hi = oracle.interval(*(x.astype(np.float64) for x in (Am, Ar, Bm, Br)))
    assert np.array_equal(hi, ((Am + Ar) @ (Bm + Br)).astype(np.float64))


@pytest.mark.parametrize("seed", [3, 4])
def test_sampled_corner_products_are_contained(seed):
    """Every point product with A in <Am, Ar> and B in <Bm, Br> lies in [lo, hi] (exact, via Fraction)."""
    rng = np.random.default_rng(seed)
    M, N, K = 3, 4, 12
    Am, Ar, Bm, Br = random_intervals(M, N, K, seed, rad_scale=0.25)
    lo, hi = oracle.interval(Am, Ar, Bm, Br)
    F = np.vectorize(Fraction, otypes=[object])
    for _ in range(40):
        ta = rng.choice([-1, 0, 1], size=Am.shape)
        tb = rng.choice([-1, 0, 1], size=Bm.shape)
        A = F(Am) + F(Ar) * ta  # exact corner (or midpoint) entries
        B = F(Bm) + F(Br) * tb
        P = A.dot(B)
        assert all(Fraction(float(lo[i, j])) <= P[i, j] <= Fraction(float(hi[i, j]))
                   for i in range(M) for j in range(N))


@pytest.mark.parametrize("dtype,seed", [(np.float64, 5), (np.float32, 6), (np.float64, 7)])
def test_fraction_brute_force(dtype, seed):
    Am, Ar, Bm, Br = random_intervals(3, 4, 7, seed, dtype, rad_scale=2.0 ** -(seed * 3))
    Am[0, 0] = -Am[0, 0]
    Ar[1, 2] = 0.0
    lo, hi = oracle.interval(Am, Ar, Bm, Br)
    plo, phi = oracle.interval_py(Am, Ar, Bm, Br, dtype=dtype)
    assert np.array_equal(bits(lo), bits(np.array(plo, dtype=dtype)))
    assert np.array_equal(bits(hi), bits(np.array(phi, dtype=dtype)))


def test_bad_operands_rejected():
    Am, Ar, Bm, Br = random_intervals(4, 4, 4, 8)
    Ar[1, 1] = -1.0
    with pytest.raises(ValueError, match="negative radius"):
        oracle.interval(Am, Ar, Bm, Br)
    Ar[1, 1] = -0.0  # a signed zero is a zero radius
    oracle.interval(Am, Ar, Bm, Br)
    Bm[0, 0] = np.nan
    with pytest.raises(ValueError, match="non-finite"):
        oracle.interval(Am, Ar, Bm, Br)

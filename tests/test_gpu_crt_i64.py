"""The int64 path's two reconstructions.  By default it reconstructs by
balanced Garner; in mode 1 of rg_set_crt_mode, by round-to-nearest CRT
whenever its planned primes already exceed 4 |C| (the prime count for a bound
one bit larger is no larger), and by Garner otherwise.  Operands at
their extremes put |C| at its bound, where the rounded quotient has the least
margin ("Accelerating Multiple-Precision LU Decomposition with Ozaki Scheme
II", CRT by round-to-nearest; "exact-solve", balanced Garner)."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import dev, host, rg  # noqa: F401
from workloads import WORKLOADS

pytestmark = pytest.mark.gpu


def primes_for_bound(primes, T):
    """Fewest leading primes whose product's floor(log2) reaches T + 1 (product > 2^(T+1))."""
    prod = 1
    for n, q in enumerate(primes, 1):
        prod *= q
        if prod.bit_length() - 1 >= T + 1:
            return n
    return 0


@pytest.fixture
def mode(rg):
    lib = rg.library()
    old = lib.rg_set_crt_mode(1)

    def set_mode(m):
        lib.rg_set_crt_mode(m)

    yield set_mode
    lib.rg_set_crt_mode(old)


CASES = [(b, K) for b in (1, 5, 12, 23, 24, 31, 40, 52, 61) for K in (1, 3, 64, 1024)
         if K * (2**b - 1) ** 2 <= 2**63 - 1]


def test_cases_cover_both_reconstructions(rg):
    ps = rg.primes()
    kinds = set()
    for b, K in CASES:
        T = 2 * b + int(np.ceil(np.log2(K)))
        P = primes_for_bound(ps, T)
        kinds.add(primes_for_bound(ps, T + 1) <= P)
    assert kinds == {True, False}


@pytest.mark.parametrize("sign", [1, -1])
@pytest.mark.parametrize("b,K", CASES)
def test_result_at_its_bound(rg, mode, sign, b, K):
    top = 2**b - 1
    M, N = 5, 7
    A = np.full((M, K), top, dtype=np.int64)
    A[1, 0] = -top  # one row a little below the bound
    B = np.full((K, N), sign * top, dtype=np.int64)
    want = oracle.matmul_i64(A, B, lc=1)[:, :, 0]
    T = 2 * b + int(np.ceil(np.log2(K)))
    ps = rg.primes()
    P = primes_for_bound(ps, T)
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    plan = rg.get_plan()
    assert plan["status"] == 0 and plan["bound_bits"] == T and plan["nprimes"] == P
    assert plan["crt_rn"] == (1 if primes_for_bound(ps, T + 1) <= P else 0)
    assert np.array_equal(C, want)
    mode(0)
    C2 = host(rg.res_gemm_i64(dev(A), dev(B)))
    assert rg.get_plan()["crt_rn"] == 0
    assert np.array_equal(C2, want)


def test_headline_workload_both_modes(rg, mode):
    """1024^3, 24-bit entries: 8 primes give the extra bit for free; both reconstructions agree."""
    w = WORKLOADS["exact24_1024"]
    A, B = w.generate()
    dA, dB = dev(A), dev(B)
    C0 = rg.res_gemm_i64(dA, dB)
    plan = rg.get_plan()
    assert plan["nprimes"] == 8 and plan["crt_rn"] == 1
    mode(0)
    C2 = rg.res_gemm_i64(dA, dB)
    assert rg.get_plan()["crt_rn"] == 0
    assert bool((C0 == C2).all())


def test_caller_fixed_prime_count(rg, mode):
    """53 fixed primes hold far more than 4 |C| for 27-bit entries (|C| < 70 * 2^54): round-to-nearest CRT, exact."""
    rng = np.random.default_rng(11)
    A = rng.integers(-(2**27), 2**27, size=(33, 70), dtype=np.int64)
    B = rng.integers(-(2**27), 2**27, size=(70, 45), dtype=np.int64)
    C = host(rg.res_gemm_i64(dev(A), dev(B), nprimes=53))
    plan = rg.get_plan()
    assert plan["nprimes"] == 53 and plan["crt_rn"] == 1
    assert np.array_equal(C, oracle.matmul_i64(A, B, lc=1)[:, :, 0])

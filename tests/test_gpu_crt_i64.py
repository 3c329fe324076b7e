"""The int64 path's three reconstructions.  By default (mode 0 of
rg_set_crt_mode) one-limb results of up to 12 primes are reconstructed by
idempotent sums with a rounded quotient, with the neighbouring quotients tried
when the result falls outside the symmetric range; mode 1 takes
round-to-nearest CRT on balanced digits whenever the planned primes already
exceed 4 |C| (the prime count for a bound one bit larger is no larger), and
Garner otherwise; mode 2 takes balanced Garner.  Operands at their extremes
put |C| at its bound, where the rounded quotient has the least margin
("Accelerating Multiple-Precision LU Decomposition with Ozaki Scheme II", CRT
by round-to-nearest; "exact-solve", balanced Garner)."""
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
    headroom = primes_for_bound(ps, T + 1) <= P
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    plan = rg.get_plan()
    assert plan["status"] == 0 and plan["bound_bits"] == T and plan["nprimes"] == P
    assert plan["crt_rn"] == (1 if headroom else 0)
    assert np.array_equal(C, want)
    mode(0)
    C0 = host(rg.res_gemm_i64(dev(A), dev(B)))
    assert rg.get_plan()["crt_rn"] == 2
    assert np.array_equal(C0, want)
    mode(2)
    C2 = host(rg.res_gemm_i64(dev(A), dev(B)))
    assert rg.get_plan()["crt_rn"] == 0
    assert np.array_equal(C2, want)


def test_headline_workload_all_modes(rg, mode):
    """1024^3, 24-bit entries: 8 primes give the extra bit for free; the three reconstructions agree."""
    w = WORKLOADS["exact24_1024"]
    A, B = w.generate()
    dA, dB = dev(A), dev(B)
    C1 = rg.res_gemm_i64(dA, dB)
    plan = rg.get_plan()
    assert plan["nprimes"] == 8 and plan["crt_rn"] == 1
    mode(0)
    C0 = rg.res_gemm_i64(dA, dB)
    assert rg.get_plan()["crt_rn"] == 2
    mode(2)
    C2 = rg.res_gemm_i64(dA, dB)
    assert rg.get_plan()["crt_rn"] == 0
    assert bool((C0 == C2).all()) and bool((C1 == C2).all())


@pytest.mark.parametrize("P", list(range(1, 13)))
def test_idempotent_sums_every_prime_count(rg, mode, P):
    """Caller-fixed prime counts 1..12, with the a-priori bound T as large as the headroom rule
    allows (P >= 2^(T+2)) and results close to 2^T in both signs: the rounded quotient's margin
    is at its thinnest, and mode 0 takes idempotent sums there."""
    ps = rg.primes()
    prod = 1
    for q in ps[:P]:
        prod *= q
    T = min(prod.bit_length() - 3, 62)
    ta, tb = (T + 1) // 2, T // 2
    a, b = 2**ta - 1, 2**tb - 1  # bits_a + bits_b = T, |a b| close to 2^T
    A = np.array([[a], [-a], [a // 3], [1], [0]], dtype=np.int64)
    B = np.array([[b, -b, 1, 0]], dtype=np.int64)
    mode(0)
    C = host(rg.res_gemm_i64(dev(A), dev(B), nprimes=P))
    plan = rg.get_plan()
    assert plan["bound_bits"] == T and plan["crt_rn"] == 2
    assert np.array_equal(C, oracle.matmul_i64(A, B, lc=1)[:, :, 0])


@pytest.mark.parametrize("P", [1, 2, 3, 5, 8])
def test_idempotent_sums_with_the_callers_guarantee_only(rg, mode, P):
    """A caller-fixed prime count below the a-priori bound: entries near 2^40 whose products cancel
    to results anywhere in the symmetric range, up to +-(P - 1) / 2, where the rounded quotient
    is as likely to be off by one as not and the range test picks the result."""
    ps = rg.primes()
    prod = 1
    for q in ps[:P]:
        prod *= q
    h = (prod - 1) // 2
    big = 2**40
    vals = [h, -h, h - 1, -(h - 1), 0, 1, -1, h // 2, -(h // 3)]
    A = np.array([[v + big, -big] for v in vals], dtype=np.int64)
    B = np.array([[1], [1]], dtype=np.int64)  # C = v
    mode(0)
    C = host(rg.res_gemm_i64(dev(A), dev(B), nprimes=P))
    assert rg.get_plan()["crt_rn"] == 2
    assert np.array_equal(C, oracle.matmul_i64(A, B, lc=1)[:, :, 0])
    assert np.array_equal(C[:, 0], np.array(vals, dtype=np.int64))

"""The two reconstructions of the wide outputs: round-to-nearest CRT (on
request, when the plan can keep P > 4 |x|) and balanced Garner (the default;
always for a caller-fixed prime count and for products at the 332-bit
capacity).  The int64 path's two reconstructions are tested in test_gpu_crt_i64.py.  Extreme
same-sign operands put the result at its bound, where the rounded quotient
has the least margin."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import dev, host, rg, variant  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def crt_mode(rg):
    """Round-to-nearest CRT where the plan allows (Garner is the library's default)."""
    lib = rg.library()
    old = lib.rg_set_crt_mode(1)
    yield
    lib.rg_set_crt_mode(old)


def limbs_of(v, L):
    return oracle.int_to_limbs(v, L)


@pytest.mark.parametrize("sign", [1, -1])
@pytest.mark.parametrize("L,K,bits", [(1, 7, 63), (2, 33, 127), (2, 1000, 127), (3, 2, 165)])
def test_result_at_its_bound(rg, sign, L, K, bits):
    top = 2**bits - 1
    M, N = 5, 6
    A = np.array([[limbs_of(top, L) for _ in range(K)] for _ in range(M)], dtype=np.int64)
    B = np.array([[limbs_of(sign * top, L) for _ in range(N)] for _ in range(K)], dtype=np.int64)
    A[1, 0] = limbs_of(-top, L)  # one row a little below the bound
    lc = min(6, (2 * bits + int(np.ceil(np.log2(K))) + 1) // 64 + 1)
    C = host(rg.res_gemm_limbs(dev(A), dev(B), lc))
    plan = rg.get_plan()
    want = oracle.matmul_py(oracle.to_pyint_matrix(A), oracle.to_pyint_matrix(B))
    assert [[oracle.limbs_to_int(C[i, j]) for j in range(N)] for i in range(M)] == want
    assert plan["crt_rn"] == (1 if plan["bound_bits"] < 332 else 0)


def test_capacity_uses_garner(rg):
    """bits_a + bits_b + ceil(log2 K) = 332 exactly: 53 primes hold the product but not one more bit."""
    K = 4  # 165 + 165 + 2 = 332
    a = 2**165 - 1
    A = np.array([[limbs_of(a, 3)] * K] * 3, dtype=np.int64)
    B = np.array([[limbs_of(-a, 3)] * 2] * K, dtype=np.int64)
    C = host(rg.res_gemm_limbs(dev(A), dev(B), 6))
    plan = rg.get_plan()
    assert plan["bound_bits"] == 332 and plan["crt_rn"] == 0 and plan["nprimes"] == 53
    assert oracle.limbs_to_int(C[0, 0]) == -K * a * a


def test_enclosure_both_paths_agree(rg):
    """A lossless enclosure by RN-CRT equals the oracle; the same product with 53 fixed primes is not
    offered for fp64, so compare the limb form of the scaled integers instead."""
    rng = np.random.default_rng(3)
    A = rng.standard_normal((70, 300))
    B = rng.standard_normal((300, 50))
    lo, hi = rg.mm_enclose(dev(A), dev(B))
    assert rg.get_plan()["crt_rn"] == 1
    rlo, rhi = oracle.enclose_f64(A, B)
    assert np.array_equal(host(lo).view(np.uint64), rlo.view(np.uint64))
    assert np.array_equal(host(hi).view(np.uint64), rhi.view(np.uint64))


def test_fixed_prime_count_uses_garner(rg):
    rng = np.random.default_rng(4)
    full = dict(low=-(2**63), high=2**63 - 1, endpoint=True, dtype=np.int64)
    A = rng.integers(size=(9, 40, 2), **full)
    B = rng.integers(size=(40, 11, 2), **full)
    C_rn = host(rg.res_gemm_limbs(dev(A), dev(B), 6))
    assert rg.get_plan()["crt_rn"] == 1
    C_g = host(rg.res_gemm_limbs(dev(A), dev(B), 6, nprimes=53))
    assert rg.get_plan()["crt_rn"] == 0
    assert np.array_equal(C_rn, C_g) and np.array_equal(C_rn, oracle.matmul_limbs(A, B, 6))


def test_default_is_garner_for_wide_results(rg):
    rg.library().rg_set_crt_mode(0)
    rng = np.random.default_rng(5)
    full = dict(low=-(2**63), high=2**63 - 1, endpoint=True, dtype=np.int64)
    A = rng.integers(size=(9, 40, 2), **full)
    B = rng.integers(size=(40, 11, 2), **full)
    C = host(rg.res_gemm_limbs(dev(A), dev(B), 6))
    assert rg.get_plan()["crt_rn"] == 0
    assert np.array_equal(C, oracle.matmul_limbs(A, B, 6))


"""GPU parity of the multi-limb path (res_gemm_limbs) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import dev, host, rg  # noqa: F401
from workloads import WORKLOADS, limb_matrices

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,la,lb,lc", [
    (33, 65, 70, 2, 2, 6),
    (1, 1, 1, 2, 2, 5),
    (130, 260, 1030, 2, 2, 6),  # two K chunks, ragged tiles
    (20, 30, 40, 1, 3, 5),
    (17, 9, 11, 3, 1, 5),
    (5, 300, 9, 1, 1, 3),
])
def test_random_full_width(rg, M, N, K, la, lb, lc):
    rng = np.random.default_rng(M + 10 * N + 100 * K + la)
    full = dict(low=-(2**63), high=2**63 - 1, endpoint=True, dtype=np.int64)
    A = rng.integers(size=(M, K, la), **full)
    B = rng.integers(size=(K, N, lb), **full)
    C = host(rg.res_gemm_limbs(dev(A), dev(B), lc))
    ref = oracle.matmul_limbs(A, B, lc)
    assert np.array_equal(C, ref)


def test_extremes_and_signs(rg):
    vals = [-(2**127), 2**127 - 1, -1, 0, 1, 2**64, -(2**64), 2**100 + 3, -(2**99)]
    rng = np.random.default_rng(3)
    M, N, K = 7, 6, 9
    A = np.array([[oracle.int_to_limbs(int(rng.choice(vals)), 2) for _ in range(K)] for _ in range(M)], dtype=np.int64)
    B = np.array([[oracle.int_to_limbs(int(rng.choice(vals)), 2) for _ in range(N)] for _ in range(K)], dtype=np.int64)
    C = host(rg.res_gemm_limbs(dev(A), dev(B), 6))
    want = oracle.matmul_py(oracle.to_pyint_matrix(A), oracle.to_pyint_matrix(B))
    got = [[oracle.limbs_to_int(C[i, j]) for j in range(N)] for i in range(M)]
    assert got == want


def test_small_values_in_wide_limbs(rg):
    # 256-bit containers holding small values: the planner reads the real widths.
    A0 = np.random.default_rng(1).integers(-1000, 1000, size=(40, 50))
    B0 = np.random.default_rng(2).integers(-1000, 1000, size=(50, 30))
    A = np.stack([A0] + [np.where(A0 < 0, -1, 0)] * 3, axis=-1).astype(np.int64)
    B = np.stack([B0] + [np.where(B0 < 0, -1, 0)] * 3, axis=-1).astype(np.int64)
    C = host(rg.res_gemm_limbs(dev(A), dev(B), 1))
    assert np.array_equal(C[:, :, 0], A0 @ B0)
    assert rg.get_plan()["nprimes"] <= 5


@pytest.fixture(scope="module")
def wide128_2048():
    """The 2048^3 signed 128-bit workload and its 6-limb oracle product (computed once)."""
    w = WORKLOADS["wide128_2048"]
    A, B = w.generate()
    return w, A, B, oracle.matmul_limbs(A, B, w.out_limbs)


@pytest.mark.parametrize("nprimes,expect", [(0, 38), (53, 53)], ids=["planned", "all_53_primes"])
def test_wide128_2048_full(rg, wide128_2048, nprimes, expect):
    # every entry, with the planned prime count and with the full prime set
    # the workload prescribes (the same integers by CRT uniqueness)
    w, A, B, ref = wide128_2048
    C = host(rg.res_gemm_limbs(dev(A), dev(B), w.out_limbs, nprimes=nprimes))
    assert np.array_equal(C, ref)
    plan = rg.get_plan()
    assert plan["nprimes"] == expect
    if not nprimes:
        # max |x| of values uniform in [-2^127, 2^127) has bit length 127
        assert plan["bits_a"] == 127 and plan["bits_b"] == 127 and plan["bound_bits"] == 127 + 127 + 11


@pytest.mark.parametrize("nprimes", [42, 43, 52, 53])
def test_wide128_fixed_prime_counts(rg, nprimes):
    # both parities of the prime count on the multi-word reconstruction
    A, B = limb_matrices(64, 64, 256, 2, 9)
    C = host(rg.res_gemm_limbs(dev(A), dev(B), 6, nprimes=nprimes))
    assert np.array_equal(C, oracle.matmul_limbs(A, B, 6))


def test_range_errors(rg):
    A, B = limb_matrices(4, 4, 4, 4, 5)
    with pytest.raises(rg.ResGemmError) as e:  # 256 + 256 + 2 > 332
        rg.res_gemm_limbs(dev(A), dev(B), 6)
    assert e.value.code == rg.RG_ERR_RANGE
    A, B = limb_matrices(4, 4, 4, 2, 6)
    with pytest.raises(rg.ResGemmError) as e:  # needs 259 bits, 2 limbs hold 127
        rg.res_gemm_limbs(dev(A), dev(B), 2)
    assert e.value.code == rg.RG_ERR_RANGE


@pytest.mark.parametrize("la,lb", [(2, 2), (4, 4), (2, 4)])
def test_operands_off_16_byte_alignment(rg, la, lb):
    """Operands starting 8 bytes past a 16-byte boundary take the scalar-load paths of the planner and the split."""
    rng = np.random.default_rng(la + 10 * lb)
    M, N, K = 37, 41, 53
    full = dict(low=-(2**63), high=2**63 - 1, endpoint=True, dtype=np.int64)

    def operand(shape, limbs):
        # 128-bit values in `limbs` limbs (upper limbs sign-extend), so the product stays within the 332-bit gate
        x = rng.integers(size=shape + (2,), **full)
        ext = np.repeat((x[..., 1:2] < 0).astype(np.int64) * -1, limbs - 2, axis=-1)
        return np.concatenate([x, ext], axis=-1) if limbs > 2 else x

    A = operand((M, K), la)
    B = operand((K, N), lb)
    bufA = torch.empty(A.size + 1, dtype=torch.int64, device="cuda")
    bufB = torch.empty(B.size + 1, dtype=torch.int64, device="cuda")
    dA = bufA[1:].view(M, K, la)
    dB = bufB[1:].view(K, N, lb)
    dA.copy_(torch.from_numpy(A))
    dB.copy_(torch.from_numpy(B))
    assert dA.data_ptr() % 16 == 8 and dB.data_ptr() % 16 == 8
    C = host(rg.res_gemm_limbs(dA, dB, 6))
    assert np.array_equal(C, oracle.matmul_limbs(A, B, 6))

"""Pins for the integer oracle (exact C = A @ B), independent of the oracle itself.

Each test checks the oracle against something it does not compute itself:
numpy's wrapping integer matmul (a library routine), closed forms, the CRT /
modular identity, a floating-point approximation for the high limbs, and
Python-integer brute force on tiny inputs.  Together they catch a dropped
term, a wrong sign, a wrong index and a transposed operand.
"""
import numpy as np
import pytest

import oracle
from workloads import int_matrices, limb_matrices

U64 = 1 << 64


def _as_int(limbs_row):
    return [oracle.limbs_to_int(e) for e in limbs_row]


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 0), (7, 5, 13, 1), (33, 17, 65, 2), (64, 64, 64, 0)])
def test_i64_equals_numpy_matmul_when_in_range(M, N, K, seed):
    # 24-bit entries: |C| < 2^23 * 2^23 * K < 2^63, so numpy's int64 matmul is exact.
    A, B = int_matrices(M, N, K, -(2**23), 2**23, seed)
    C = oracle.matmul_i64(A, B, lc=1)[:, :, 0]
    assert np.array_equal(C, A @ B)


@pytest.mark.parametrize("M,N,K", [(3, 4, 5), (9, 2, 31)])
def test_i64_low_limb_is_wrapping_product(M, N, K):
    # For any int64 operands the low 64 bits of the exact product equal the
    # product computed with wrap-around uint64 arithmetic (numpy).
    rng = np.random.default_rng(11)
    A = rng.integers(-(2**63), 2**63 - 1, endpoint=True, size=(M, K), dtype=np.int64)
    B = rng.integers(-(2**63), 2**63 - 1, endpoint=True, size=(K, N), dtype=np.int64)
    C = oracle.matmul_i64(A, B, lc=3)
    wrap = A.view(np.uint64) @ B.view(np.uint64)
    assert np.array_equal(C[:, :, 0].view(np.uint64), wrap)


@pytest.mark.parametrize("q", [251, 241, 199, 3, 5, 7])
def test_i64_modular_identity(q):
    # (A B) mod q == ((A mod q)(B mod q)) mod q, evaluated by numpy in int64.
    rng = np.random.default_rng(q)
    A = rng.integers(-(2**63), 2**63 - 1, endpoint=True, size=(6, 40), dtype=np.int64)
    B = rng.integers(-(2**63), 2**63 - 1, endpoint=True, size=(40, 5), dtype=np.int64)
    C = oracle.matmul_i64(A, B, lc=3)
    got = np.array([[oracle.limbs_to_int(C[i, j]) % q for j in range(5)] for i in range(6)])
    want = ((A % q) @ (B % q)) % q
    assert np.array_equal(got, want)


def test_i64_extremes_bruteforce():
    vals = [-(2**63), 2**63 - 1, -1, 0, 1, 2**62, -(2**62) + 7]
    rng = np.random.default_rng(5)
    for trial in range(20):
        M, N, K = rng.integers(1, 4, size=3)
        A = rng.choice(vals, size=(M, K)).astype(np.int64)
        B = rng.choice(vals, size=(K, N)).astype(np.int64)
        C = oracle.matmul_i64(A, B, lc=3)
        want = oracle.matmul_py(oracle.to_pyint_matrix(A), oracle.to_pyint_matrix(B))
        assert [_as_int(row) for row in C] == want


def test_i64_closed_form_long_k_all_minus_128():
    # K = 2^17 entries of (-128)(-128) = 2^14 sum to 2^31 exactly: the int32
    # accumulator bound of the pages' INT8 engine is met with equality here.
    K = 2**17
    A = np.full((2, K), -128, dtype=np.int64)
    B = np.full((K, 3), -128, dtype=np.int64)
    C = oracle.matmul_i64(A, B, lc=1)
    assert (C == 2**31).all()


def test_i64_rank_one_closed_form():
    a = np.array([-(2**63), 2**63 - 1, -3], dtype=np.int64)
    b = np.array([-(2**63), 5, 2**63 - 1, 0], dtype=np.int64)
    K = 3
    A = np.repeat(a[:, None], K, axis=1)
    B = np.repeat(b[None, :], K, axis=0)
    C = oracle.matmul_i64(A, B, lc=3)
    for i in range(3):
        for j in range(4):
            assert oracle.limbs_to_int(C[i, j]) == K * int(a[i]) * int(b[j])


def test_i64_transpose_identity():
    # (A B)^T == B^T A^T on a non-square case: catches swapped operands/indices.
    A, B = int_matrices(5, 11, 7, -(2**40), 2**40, 3)
    C1 = oracle.matmul_i64(A, B, lc=2)
    C2 = oracle.matmul_i64(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T), lc=2)
    assert np.array_equal(C1, C2.transpose(1, 0, 2))


def test_i64_high_limbs_match_float_estimate():
    rng = np.random.default_rng(8)
    A = rng.integers(-(2**62), 2**62, size=(4, 50), dtype=np.int64)
    B = rng.integers(-(2**62), 2**62, size=(50, 6), dtype=np.int64)
    C = oracle.matmul_i64(A, B, lc=3)
    est = A.astype(np.float64) @ B.astype(np.float64)
    got = np.array([[float(oracle.limbs_to_int(C[i, j])) for j in range(6)] for i in range(4)])
    scale = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    assert (np.abs(got - est) <= 1e-12 * scale).all()


def test_i64_overflow_is_reported():
    A = np.full((1, 2), 2**62, dtype=np.int64)
    B = np.full((2, 1), 2, dtype=np.int64)
    with pytest.raises(OverflowError):
        oracle.matmul_i64(A, B, lc=1)  # 2^64 does not fit one limb
    C = oracle.matmul_i64(A, B, lc=2)
    assert oracle.limbs_to_int(C[0, 0]) == 2**64


def test_i64_row_subset():
    A, B = int_matrices(20, 9, 12, -(2**30), 2**30, 4)
    full = oracle.matmul_i64(A, B, lc=1)
    rows = np.array([19, 0, 7])
    part = oracle.matmul_i64(A, B, lc=1, rows=rows)
    assert np.array_equal(part, full[rows])


# --------------------------------------------------------------------------- limbs


def test_limb_codec_roundtrip():
    for v in [0, 1, -1, 2**127 - 1, -(2**127), 2**64, -(2**64), 12345678901234567890123]:
        assert oracle.limbs_to_int(oracle.int_to_limbs(v, 2)) == v
    assert oracle.limbs_to_int([0, 1]) == 2**64
    assert oracle.limbs_to_int([-1, -1]) == -1
    assert oracle.limbs_to_int([0, -(2**63)]) == -(2**127)


@pytest.mark.parametrize("la,lb", [(2, 2), (1, 2), (3, 1), (4, 4)])
def test_limbs_bruteforce(la, lb):
    rng = np.random.default_rng(la * 10 + lb)
    M, N, K = 3, 4, 5
    full = dict(low=-(2**63), high=2**63 - 1, endpoint=True, dtype=np.int64)
    A = rng.integers(size=(M, K, la), **full)
    B = rng.integers(size=(K, N, lb), **full)
    A[0, 0] = oracle.int_to_limbs(-(2 ** (64 * la - 1)), la)  # most negative value
    B[0, 0] = oracle.int_to_limbs(-(2 ** (64 * lb - 1)), lb)
    lc = la + lb + 1
    C = oracle.matmul_limbs(A, B, lc)
    want = oracle.matmul_py(oracle.to_pyint_matrix(A), oracle.to_pyint_matrix(B))
    assert [_as_int(row) for row in C] == want


def test_limbs_low_limb_is_wrapping_product():
    A, B = limb_matrices(6, 7, 9, 2, 21)
    C = oracle.matmul_limbs(A, B, 6)
    wrap = np.ascontiguousarray(A[:, :, 0]).view(np.uint64) @ np.ascontiguousarray(B[:, :, 0]).view(np.uint64)
    assert np.array_equal(C[:, :, 0].view(np.uint64), wrap)


@pytest.mark.parametrize("q", [251, 13, 3])
def test_limbs_modular_identity(q):
    A, B = limb_matrices(4, 3, 10, 2, 22)
    C = oracle.matmul_limbs(A, B, 6)
    Ai = np.array([[oracle.limbs_to_int(e) % q for e in row] for row in A], dtype=np.int64)
    Bi = np.array([[oracle.limbs_to_int(e) % q for e in row] for row in B], dtype=np.int64)
    got = np.array([[oracle.limbs_to_int(C[i, j]) % q for j in range(3)] for i in range(4)])
    assert np.array_equal(got, (Ai @ Bi) % q)


def test_limbs_closed_form_power_of_two_diagonal():
    # A = 2^100 I (as 2 limbs) gives C = 2^100 B exactly.
    n = 4
    A = np.zeros((n, n, 2), dtype=np.int64)
    for i in range(n):
        A[i, i] = oracle.int_to_limbs(2**100, 2)
    _, B = limb_matrices(1, 3, n, 2, 23)
    C = oracle.matmul_limbs(A, B, 6)
    for i in range(n):
        for j in range(3):
            assert oracle.limbs_to_int(C[i, j]) == 2**100 * oracle.limbs_to_int(B[i, j])


def test_limbs_agree_with_i64_path():
    A, B = int_matrices(5, 6, 7, -(2**63), 2**63 - 1, 24)
    C1 = oracle.matmul_i64(A, B, lc=3)
    C2 = oracle.matmul_limbs(A[:, :, None], B[:, :, None], 3)
    assert np.array_equal(C1, C2)

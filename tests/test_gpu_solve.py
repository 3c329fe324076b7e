"""GPU exact solve (rg_solve_i64 / solve; "exact-solve", Method: batched
modular inverse, Dixon lift on the residue engine, rational reconstruction)
against the Fraction Gaussian-elimination oracle on small systems and the
integer identity A N == d b on larger ones ("exact-solve", Correctness)."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import dev, rg  # noqa: F401

pytestmark = pytest.mark.gpu


def nonsingular(n, lo, hi, seed):
    rng = np.random.default_rng(seed)
    while True:
        A = rng.integers(lo, hi, size=(n, n), dtype=np.int64)
        if oracle.solve_fraction(A[: min(n, 12), : min(n, 12)], np.ones((min(n, 12), 1), dtype=np.int64)) is not None:
            return A


def integer_identity(A, X, b):
    """A N == d b with N, d the integer form of X, in Python integers."""
    N, d = oracle.solution_as_integers(X)
    n, c = len(N), len(N[0])
    Ai = [[int(v) for v in row] for row in A]
    for i in range(n):
        for j in range(c):
            if sum(Ai[i][k] * N[k][j] for k in range(n)) != d * int(b[i][j]):
                return False
    return True


@pytest.mark.parametrize("n,c,seed", [(1, 1, 0), (3, 2, 1), (7, 1, 2), (16, 3, 3), (20, 1, 4), (24, 16, 5), (24, 17, 6)])
def test_against_fraction_oracle(rg, n, c, seed):
    rng = np.random.default_rng(seed + 100)
    A = nonsingular(n, -(2**20), 2**20, seed)
    b = rng.integers(-(2**30), 2**30, size=(n, c), dtype=np.int64)
    X = rg.solve(dev(A), dev(b))
    assert X == oracle.solve_fraction(A, b)


@pytest.mark.parametrize("n,seed", [(33, 5), (100, 6), (257, 7)])
def test_planted_integer_solution(rg, n, seed):
    rng = np.random.default_rng(seed)
    A = rng.integers(-(2**24), 2**24, size=(n, n), dtype=np.int64)
    x = rng.integers(-(2**20), 2**20, size=(n, 2), dtype=np.int64)
    b = np.array([[sum(int(A[i, k]) * int(x[k, j]) for k in range(n)) for j in range(2)] for i in range(n)],
                 dtype=object)
    assert all(abs(int(v)) < 2**63 for v in b.ravel())
    info = {}
    X = rg.solve(dev(A), dev(b.astype(np.int64)), info=info)
    assert X == [[Fraction(int(v)) for v in row] for row in x]
    assert info["denominator"] == 1 and info["steps"] >= 1


@pytest.mark.parametrize("n", [128, 600])
def test_rational_solution_integer_identity(rg, n):
    # 600: about 100 lift steps, so the digits' conversion recurses several levels and the numerators'
    # products run through Karatsuba's method and Barrett's reduction
    rng = np.random.default_rng(8 + n)
    A = rng.integers(-(2**23), 2**23, size=(n, n), dtype=np.int64)
    b = rng.integers(-(2**23), 2**23, size=(n, 1), dtype=np.int64)
    info = {}
    X = rg.solve(dev(A), dev(b), info=info)
    assert integer_identity(A, X, b)
    d = info["denominator"]
    assert math.lcm(*[v.denominator for row in X for v in row]) == d  # the least common denominator


def test_pascal_order_30(rg):
    """The pages' example: the order-30 Pascal system (condition ~1e32) has an exact integer solution."""
    n = 30
    P = np.array([[math.comb(i + j, i) for j in range(n)] for i in range(n)], dtype=object)
    assert max(int(v) for v in P.ravel()) * n < 2**63
    b = np.ones((n, 1), dtype=np.int64)
    X = rg.solve(dev(P.astype(np.int64)), dev(b))
    assert all(v.denominator == 1 for row in X for v in row)
    assert integer_identity(P, X, b)
    assert X == oracle.solve_fraction(P, b)


def test_scaled_hilbert_dense_denominators(rg):
    n = 9
    L = math.lcm(*range(1, 2 * n))
    H = np.array([[L // (i + j + 1) for j in range(n)] for i in range(n)], dtype=np.int64)
    b = np.eye(n, 2, dtype=np.int64)
    X = rg.solve(dev(H), dev(b))
    assert X == oracle.solve_fraction(H, b)
    assert max(v.denominator for row in X for v in row) > 1


def test_primes_dividing_det_are_dropped(rg):
    """Every entry a multiple of 3 * 5 * 7: det(A) is divisible by 105^n, so the lift runs without those primes."""
    n = 24
    rng = np.random.default_rng(9)
    A = 105 * rng.integers(-1000, 1000, size=(n, n), dtype=np.int64)
    b = rng.integers(-1000, 1000, size=(n, 1), dtype=np.int64)
    info = {}
    X = rg.solve(dev(A), dev(b), info=info)
    assert info["primes"] <= 50
    assert integer_identity(A, X, b)


def test_host_tensors_and_vector_b(rg):
    n = 12
    A = nonsingular(n, -99, 100, 10)
    b = np.arange(n, dtype=np.int64) - 5
    X = rg.solve(torch.from_numpy(A), torch.from_numpy(b))
    assert X == oracle.solve_fraction(A, b[:, None])


def test_singular_returns_none(rg):
    A = np.array([[1, 2, 3], [2, 4, 6], [7, 1, 1]], dtype=np.int64)
    assert rg.solve(dev(A), dev(np.ones((3, 1), dtype=np.int64))) is None
    Z = np.zeros((4, 4), dtype=np.int64)
    assert rg.solve(dev(Z), dev(np.ones((4, 1), dtype=np.int64))) is None


def test_range_error(rg):
    n = 4
    A = np.full((n, n), 2**62, dtype=np.int64)  # n * max|A| = 2^64
    with pytest.raises(rg.ResGemmError) as e:
        rg.solve(dev(A), dev(np.ones((n, 1), dtype=np.int64)))
    assert e.value.code == rg.RG_ERR_RANGE


def det_is_zero_mod(A, q):
    """Whether q divides det(A), by Gaussian elimination over GF(q) (numpy, exact in int64)."""
    M = np.mod(A, q).astype(np.int64)
    n = len(M)
    for k in range(n):
        nz = np.nonzero(M[k:, k])[0]
        if len(nz) == 0:
            return True
        r = k + nz[0]
        M[[k, r]] = M[[r, k]]
        inv = pow(int(M[k, k]), q - 2, q)
        M[k] = M[k] * inv % q
        f = M[k + 1:, k].copy()
        M[k + 1:] = (M[k + 1:] - np.outer(f, M[k])) % q
    return False


def test_primes_dividing_det_found_in_later_pivot_blocks(rg):
    """Rows made dependent modulo 3, 5 and 7 only (each is another row combination plus a multiple of q times a
    random row), at positions that the elimination reaches in its second, third and fourth block of pivots: exactly
    the primes dividing det(A) are dropped, and the solution is exact."""
    n = 230
    rng = np.random.default_rng(11)
    A = rng.integers(-(2**20), 2**20, size=(n, n), dtype=np.int64)
    for row, q, (a, b) in ((100, 3, (0, 1)), (170, 5, (2, 3)), (229, 7, (4, 5))):
        A[row] = A[a] + A[b] + q * rng.integers(-1000, 1000, size=n)
    b = rng.integers(-(2**20), 2**20, size=(n, 1), dtype=np.int64)
    info = {}
    X = rg.solve(dev(A), dev(b), info=info)
    primes = [q for q in range(3, 256, 2) if all(q % d for d in range(3, int(q ** 0.5) + 1, 2))]
    assert len(primes) == 53
    kept = [q for q in primes if not det_is_zero_mod(A, q)]
    assert 3 not in kept and 5 not in kept and 7 not in kept
    assert info["primes"] == len(kept)
    assert integer_identity(A, X, b)


@pytest.mark.parametrize("n", [1100, 2100, 4200])
def test_planted_solution_at_every_panel_shape(rg, n):
    """Orders past 1024, 2048 and 4096 rows, where the elimination's panel kernel holds 2, 4 and 8 rows per thread
    with blocks of 64, 32 and 16 pivots: a planted integer solution comes back exactly."""
    rng = np.random.default_rng(20 + n)
    A = rng.integers(-(2**10), 2**10, size=(n, n), dtype=np.int64)
    x = rng.integers(-(2**10), 2**10, size=(n, 1), dtype=np.int64)
    b = A @ x  # |entries| < n 2^20: exact in int64
    info = {}
    N, d = rg.solve_integers(dev(A), dev(b), info=info)
    assert d == 1
    assert [row[0] for row in N] == [int(v) for v in x[:, 0]]


def test_denominators_beyond_the_sampled_components(rg):
    """x_i = 1/p_i for distinct primes p_i above 255: every component has its own denominator, so the common
    denominator the first few components give misses the rest, and each missing factor extends it."""
    ps = [257, 263, 269, 271, 277, 281, 283, 293, 307, 311, 313, 317]
    n = len(ps)
    A = np.diag(np.array(ps, dtype=np.int64))  # det(A) = prod p_i: no lift prime divides it
    b = np.ones((n, 1), dtype=np.int64)
    info = {}
    X = rg.solve(dev(A), dev(b), info=info)
    assert X == [[Fraction(1, p)] for p in ps]
    assert info["denominator"] == math.prod(ps)
    assert info["primes"] == 53

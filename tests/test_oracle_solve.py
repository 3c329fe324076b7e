"""Pins of the exact-solve oracle (oracle.solve_fraction; "exact-solve" page,
Correctness: a Fraction Gaussian-elimination oracle, planted integer
solutions, the integer identity A N == d b).

* Planted integer solutions: b = A x for a random integer x must give x back.
* The order-n Pascal matrix is unimodular, so its solutions are integers; the
  solution of P x = e_1 is the first column of P^-1, which has the closed form
  (-1)^(i+j) C(i, j) for the lower-triangular Pascal factor.
* Diagonal and triangular systems with closed-form rational solutions.
* Substitution: A X == b exactly, in Fraction arithmetic, and the integer form
  A N == d b.
* Singular systems return None.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


def matvec(A, X):
    return [[sum(Fraction(int(A[i][k])) * X[k][j] for k in range(len(X))) for j in range(len(X[0]))]
            for i in range(len(A))]


@pytest.mark.parametrize("n,seed", [(1, 0), (5, 1), (12, 2)])
def test_planted_integer_solution(n, seed):
    rng = np.random.default_rng(seed)
    A = rng.integers(-1000, 1000, size=(n, n))
    while round(abs(np.linalg.det(A))) == 0:
        A = rng.integers(-1000, 1000, size=(n, n))
    x = rng.integers(-10**6, 10**6, size=(n, 2))
    b = [[sum(int(A[i, k]) * int(x[k, j]) for k in range(n)) for j in range(2)] for i in range(n)]
    X = oracle.solve_fraction(A, np.array(b, dtype=object))
    assert X == [[Fraction(int(v)) for v in row] for row in x]


def test_pascal_unimodular():
    """Symmetric Pascal S = L L^T with L[i][j] = C(i, j): the solution of S x = e_0 is
    S^-1 e_0 = L^-T L^-1 e_0, with L^-1[i][j] = (-1)^(i+j) C(i, j)."""
    n = 10
    S = np.array([[math.comb(i + j, i) for j in range(n)] for i in range(n)], dtype=object)
    e0 = np.zeros((n, 1), dtype=object)
    e0[0, 0] = 1
    X = oracle.solve_fraction(S, e0)
    Linv = [[(-1) ** (i + j) * math.comb(i, j) if j <= i else 0 for j in range(n)] for i in range(n)]
    y = [Linv[i][0] for i in range(n)]  # L^-1 e_0
    want = [sum(Linv[k][i] * y[k] for k in range(n)) for i in range(n)]  # L^-T y
    assert [row[0] for row in X] == [Fraction(v) for v in want]
    assert all(v.denominator == 1 for row in X for v in row)


def test_diagonal_and_triangular_closed_forms():
    A = np.diag([2, -3, 7])
    X = oracle.solve_fraction(A, np.array([[1], [1], [1]]))
    assert [r[0] for r in X] == [Fraction(1, 2), Fraction(-1, 3), Fraction(1, 7)]
    U = np.array([[2, 1], [0, 4]])  # x1 = 3/4, x0 = (1 - 3/4) / 2 = 1/8
    X = oracle.solve_fraction(U, np.array([[1], [3]]))
    assert [r[0] for r in X] == [Fraction(1, 8), Fraction(3, 4)]


@pytest.mark.parametrize("n,seed", [(8, 3), (15, 4)])
def test_substitution_and_integer_identity(n, seed):
    rng = np.random.default_rng(seed)
    A = rng.integers(-(2**23), 2**23, size=(n, n))
    b = rng.integers(-(2**23), 2**23, size=(n, 3))
    X = oracle.solve_fraction(A, b)
    assert matvec(A, X) == [[Fraction(int(v)) for v in row] for row in b]
    N, d = oracle.solution_as_integers(X)
    assert [[sum(int(A[i, k]) * N[k][j] for k in range(n)) for j in range(3)] for i in range(n)] == \
        [[d * int(v) for v in row] for row in b]


def test_singular_returns_none():
    A = np.array([[1, 2, 3], [2, 4, 6], [0, 1, 1]])
    assert oracle.solve_fraction(A, np.array([[1], [2], [3]])) is None
    assert oracle.solve_fraction(np.zeros((2, 2), dtype=np.int64), np.ones((2, 1), dtype=np.int64)) is None

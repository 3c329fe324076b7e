"""CPU oracle for the exact residue GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's compute path never calls
it, and the two share no code: the oracle computes each result from its plain
definition, not by the residue method.

Two implementations of the same definitions live here:

* ``exact_oracle.c`` (built into ``_build/libexact_oracle.so``): schoolbook
  exact integer products in a wide two's-complement accumulator, and the exact
  fp64 inner product rounded outward by exact comparison and ``nextafter``.
  OpenMP over output rows.  Used at the workload sizes.
* Pure Python (``matmul_py``, ``enclose_py``): Python integers and
  ``fractions.Fraction``, for tiny cases only.

Sources: the "enclosure-gemm" page (Method; Correctness: the reference is
exact rational arithmetic, lo <= exact <= hi, and equality with the floor and
ceiling in the format when scaling is lossless) and the "exact-solve" page
(Method: the residue engine recovers an exact integer product).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from fractions import Fraction

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "exact_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libexact_oracle.so")
_lib = None

# ---------------------------------------------------------------------------
# C oracle
# ---------------------------------------------------------------------------


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP) if needed; return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


def _configure(lib):
    """Declare the C oracle's entry points on a loaded library (this build, or a test's copy)."""
    i64p = ctypes.POINTER(ctypes.c_int64)
    dp = ctypes.POINTER(ctypes.c_double)
    ci = ctypes.c_int
    lib.oracle_matmul_i64.argtypes = [i64p, i64p, i64p, ci, ci, ci, ci, i64p, ci, ci]
    lib.oracle_matmul_i64.restype = ctypes.c_long
    lib.oracle_matmul_limbs.argtypes = [i64p, ci, i64p, ci, i64p, ci, ci, ci, ci, i64p, ci, ci]
    lib.oracle_matmul_limbs.restype = ctypes.c_long
    lib.oracle_enclose_f64.argtypes = [dp, dp, dp, dp, ci, ci, ci, i64p, ci, ci]
    lib.oracle_enclose_f64.restype = ci
    fp = ctypes.POINTER(ctypes.c_float)
    lib.oracle_enclose_f32.argtypes = [fp, fp, fp, fp, ci, ci, ci, i64p, ci, ci]
    lib.oracle_enclose_f32.restype = ci
    lib.oracle_interval_f64.argtypes = [dp, dp, dp, dp, dp, dp, ci, ci, ci, i64p, ci, ci]
    lib.oracle_interval_f64.restype = ci
    lib.oracle_interval_f32.argtypes = [fp, fp, fp, fp, fp, fp, ci, ci, ci, i64p, ci, ci]
    lib.oracle_interval_f32.restype = ci
    lib.oracle_threads.argtypes = [ci]
    lib.oracle_threads.restype = ci
    return lib


def default_threads() -> int:
    env = os.environ.get("ORACLE_THREADS")
    return int(env) if env else (os.cpu_count() or 1)


def threads_used(threads: int | None = None) -> int:
    """How many OpenMP threads the C oracle runs with."""
    return _load().oracle_threads(threads or default_threads())


def _ptr(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if r.size and (r.min() < 0 or r.max() >= M):
        raise IndexError("row index out of range")
    return r, int(r.size)


def matmul_i64(A, B, lc: int = 1, rows=None, threads: int | None = None):
    """Exact C = A @ B for int64 A [M,K], B [K,N]; returns int64 limbs [R,N,lc].

    Raises OverflowError if an entry does not fit in ``lc`` limbs.
    """
    A = np.ascontiguousarray(A, dtype=np.int64)
    B = np.ascontiguousarray(B, dtype=np.int64)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    r, nr = _rows_arg(rows, M)
    C = np.zeros((nr, N, lc), dtype=np.int64)
    rp = _ptr(r, ctypes.c_int64) if r is not None else None
    bad = _load().oracle_matmul_i64(_ptr(A, ctypes.c_int64), _ptr(B, ctypes.c_int64), _ptr(C, ctypes.c_int64),
                                    M, N, K, lc, rp, nr, threads or default_threads())
    if bad:
        raise OverflowError(f"{bad} entries do not fit in {lc} limbs")
    return C


def matmul_limbs(A, B, lc: int, rows=None, threads: int | None = None):
    """Exact C = A @ B for limb operands A [M,K,la], B [K,N,lb]; returns [R,N,lc]."""
    A = np.ascontiguousarray(A, dtype=np.int64)
    B = np.ascontiguousarray(B, dtype=np.int64)
    M, K, la = A.shape
    K2, N, lb = B.shape
    assert K == K2
    r, nr = _rows_arg(rows, M)
    C = np.zeros((nr, N, lc), dtype=np.int64)
    rp = _ptr(r, ctypes.c_int64) if r is not None else None
    bad = _load().oracle_matmul_limbs(_ptr(A, ctypes.c_int64), la, _ptr(B, ctypes.c_int64), lb,
                                      _ptr(C, ctypes.c_int64), lc, M, N, K, rp, nr, threads or default_threads())
    if bad < 0:
        raise ValueError("bad limb counts")
    if bad:
        raise OverflowError(f"{bad} entries do not fit in {lc} limbs")
    return C


def enclose_f64(A, B, rows=None, threads: int | None = None):
    """(lo, hi) float64 [R,N]: the tightest doubles bracketing the exact A @ B."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    r, nr = _rows_arg(rows, M)
    lo = np.zeros((nr, N), dtype=np.float64)
    hi = np.zeros((nr, N), dtype=np.float64)
    rp = _ptr(r, ctypes.c_int64) if r is not None else None
    rc = _load().oracle_enclose_f64(_ptr(A, ctypes.c_double), _ptr(B, ctypes.c_double), _ptr(lo, ctypes.c_double),
                                    _ptr(hi, ctypes.c_double), M, N, K, rp, nr, threads or default_threads())
    if rc == -1:
        raise ValueError("non-finite operand")
    if rc != 0:
        raise RuntimeError("oracle outward search did not converge")
    return lo, hi


def enclose_f32(A, B, rows=None, threads: int | None = None):
    """(lo, hi) float32 [R,N]: the tightest floats bracketing the exact A @ B of float32 matrices."""
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    r, nr = _rows_arg(rows, M)
    lo = np.zeros((nr, N), dtype=np.float32)
    hi = np.zeros((nr, N), dtype=np.float32)
    rp = _ptr(r, ctypes.c_int64) if r is not None else None
    rc = _load().oracle_enclose_f32(_ptr(A, ctypes.c_float), _ptr(B, ctypes.c_float), _ptr(lo, ctypes.c_float),
                                    _ptr(hi, ctypes.c_float), M, N, K, rp, nr, threads or default_threads())
    if rc == -1:
        raise ValueError("non-finite operand")
    if rc == -3:
        raise MemoryError("oracle_enclose_f32")
    if rc != 0:
        raise RuntimeError("oracle outward search did not converge")
    return lo, hi


def interval(Am, Ar, Bm, Br, rows=None, threads: int | None = None):
    """(lo, hi) [R,N] bracketing Rump's midpoint-radius product <Am, Ar> * <Bm, Br>:
    the tightest values of the operands' format (float64 or float32) below
    Am @ Bm - (|Am| @ Br + Ar @ |Bm| + Ar @ Br) and above Am @ Bm + (...), all exact."""
    dt = np.float32 if np.asarray(Am).dtype == np.float32 else np.float64
    Am, Ar, Bm, Br = (np.ascontiguousarray(x, dtype=dt) for x in (Am, Ar, Bm, Br))
    M, K = Am.shape
    K2, N = Bm.shape
    assert K == K2 and Ar.shape == Am.shape and Br.shape == Bm.shape
    r, nr = _rows_arg(rows, M)
    lo = np.zeros((nr, N), dtype=dt)
    hi = np.zeros((nr, N), dtype=dt)
    ct = ctypes.c_float if dt == np.float32 else ctypes.c_double
    fn = _load().oracle_interval_f32 if dt == np.float32 else _load().oracle_interval_f64
    rp = _ptr(r, ctypes.c_int64) if r is not None else None
    rc = fn(*(_ptr(x, ct) for x in (Am, Ar, Bm, Br, lo, hi)), M, N, K, rp, nr, threads or default_threads())
    if rc == -1:
        raise ValueError("non-finite operand")
    if rc == -4:
        raise ValueError("negative radius")
    if rc == -3:
        raise MemoryError("oracle_interval")
    if rc != 0:
        raise RuntimeError("oracle outward search did not converge")
    return lo, hi


# ---------------------------------------------------------------------------
# Pure-Python oracle (tiny cases only)
# ---------------------------------------------------------------------------


def limbs_to_int(limbs) -> int:
    """Little-endian two's-complement int64 limbs -> Python int (top limb signed)."""
    limbs = [int(x) for x in limbs]
    v = 0
    for i, x in enumerate(limbs[:-1]):
        v |= (x & 0xFFFFFFFFFFFFFFFF) << (64 * i)
    return v + (limbs[-1] << (64 * (len(limbs) - 1)))


def int_to_limbs(v: int, L: int):
    """Python int -> L little-endian two's-complement int64 limbs."""
    if not -(1 << (64 * L - 1)) <= v < (1 << (64 * L - 1)):
        raise OverflowError("value does not fit")
    u = v & ((1 << (64 * L)) - 1)
    out = []
    for i in range(L):
        w = (u >> (64 * i)) & 0xFFFFFFFFFFFFFFFF
        out.append(w - (1 << 64) if w >= (1 << 63) else w)
    return out


def to_pyint_matrix(X):
    """numpy int64 [R,C] or limbs [R,C,L] -> nested lists of Python ints."""
    X = np.asarray(X)
    if X.ndim == 2:
        return [[int(v) for v in row] for row in X]
    return [[limbs_to_int(e) for e in row] for row in X]


def matmul_py(A, B):
    """Schoolbook product of nested lists of Python ints (exact, any size)."""
    K = len(B)
    N = len(B[0]) if K else 0
    return [[sum(a[k] * B[k][j] for k in range(K)) for j in range(N)] for a in A]


def enclose_exact_py(exact: Fraction):
    """(lo, hi): largest double <= exact and smallest double >= exact.

    exact == 0 gives (+0.0, +0.0).  Beyond the largest finite double the bound
    away from zero is infinite.
    """
    if exact == 0:
        return 0.0, 0.0
    try:
        c = float(exact)
    except OverflowError:
        c = math.inf if exact > 0 else -math.inf
    while c > exact:
        c = math.nextafter(c, -math.inf)
    while c != math.inf:
        n = math.nextafter(c, math.inf)
        if n <= exact:
            c = n
        else:
            break
    lo = c
    hi = lo if lo == exact else math.nextafter(lo, math.inf)
    return lo, hi


def enclose_exact_py32(exact: Fraction):
    """(lo, hi): largest float32 <= exact and smallest float32 >= exact, as
    numpy float32 (+0 for an exact zero; infinite beyond the largest finite)."""
    f32 = np.float32
    if exact == 0:
        return f32(0.0), f32(0.0)
    top = Fraction(float(np.finfo(np.float32).max))
    if exact > top:
        c = f32(np.inf)
    elif exact < -top:
        c = f32(-np.inf)
    else:
        c = f32(float(exact))  # float() rounds once more; the walk below corrects it
    while c == np.inf or (c != -np.inf and Fraction(float(c)) > exact):
        c = np.nextafter(c, f32(-np.inf))
    while c != np.inf:
        n = np.nextafter(c, f32(np.inf))
        if n == np.inf or Fraction(float(n)) > exact:
            break
        c = n
    lo = c
    hi = lo if (lo != -np.inf and Fraction(float(lo)) == exact) else np.nextafter(lo, f32(np.inf))
    return lo, hi


def enclose_py(A, B, dtype=np.float64):
    """(lo, hi) as nested lists for small float matrices, via Fraction; with
    dtype float32 the operands are binary32 and the bounds are binary32."""
    A = np.asarray(A, dtype=dtype)
    B = np.asarray(B, dtype=dtype)
    rnd = enclose_exact_py32 if dtype == np.float32 else enclose_exact_py
    M, K = A.shape
    N = B.shape[1]
    lo = [[0.0] * N for _ in range(M)]
    hi = [[0.0] * N for _ in range(M)]
    Af = [[Fraction(float(x)) for x in row] for row in A]
    Bf = [[Fraction(float(x)) for x in row] for row in B]
    for i in range(M):
        for j in range(N):
            s = sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0))
            lo[i][j], hi[i][j] = rnd(s)
    return lo, hi


def exact_dot_fraction(a_row, b_col) -> Fraction:
    """The exact real inner product of two float64 vectors."""
    return sum((Fraction(float(x)) * Fraction(float(y)) for x, y in zip(a_row, b_col)), Fraction(0))


def interval_py(Am, Ar, Bm, Br, dtype=np.float64):
    """interval() for tiny matrices via Fraction: midpoint S and radius R as
    exact rationals, then the outward floor of S - R and ceiling of S + R."""
    Am, Ar, Bm, Br = (np.asarray(x, dtype=dtype) for x in (Am, Ar, Bm, Br))
    rnd = enclose_exact_py32 if dtype == np.float32 else enclose_exact_py
    M, K = Am.shape
    N = Bm.shape[1]
    F = [[[Fraction(float(v)) for v in row] for row in X] for X in (Am, Ar, Bm, Br)]
    fam, far, fbm, fbr = F
    lo = [[0.0] * N for _ in range(M)]
    hi = [[0.0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            S = sum((fam[i][k] * fbm[k][j] for k in range(K)), Fraction(0))
            R = sum((abs(fam[i][k]) * fbr[k][j] + far[i][k] * abs(fbm[k][j]) + far[i][k] * fbr[k][j]
                     for k in range(K)), Fraction(0))
            lo[i][j] = rnd(S - R)[0]
            hi[i][j] = rnd(S + R)[1]
    return lo, hi


# ---------------------------------------------------------------------------
# Exact rational solve ("exact-solve" page, Correctness: an exact
# Fraction Gaussian-elimination oracle on small systems)
# ---------------------------------------------------------------------------


def solve_fraction(A, b):
    """The exact solution X of A X = b over the rationals, as a nested list
    [n][c] of Fraction, or None when A is singular.  Gauss-Jordan elimination
    in Fraction arithmetic, pivoting on the first nonzero entry of each column."""
    A = [[Fraction(int(v)) for v in row] for row in np.asarray(A)]
    B = np.asarray(b)
    if B.ndim == 1:
        B = B[:, None]
    Bf = [[Fraction(int(v)) for v in row] for row in B]
    n = len(A)
    c = len(Bf[0]) if n else 0
    M = [A[i] + Bf[i] for i in range(n)]
    for k in range(n):
        piv = next((r for r in range(k, n) if M[r][k] != 0), None)
        if piv is None:
            return None
        M[k], M[piv] = M[piv], M[k]
        inv = 1 / M[k][k]
        M[k] = [v * inv for v in M[k]]
        for r in range(n):
            if r != k and M[r][k] != 0:
                f = M[r][k]
                M[r] = [vr - f * vk for vr, vk in zip(M[r], M[k])]
    return [[M[i][n + j] for j in range(c)] for i in range(n)]


def solution_as_integers(X):
    """(N, d): integer numerators [n][c] and the least common denominator d of
    a rational solution, the form in which the integer identity A N == d b is
    checked."""
    d = 1
    for row in X:
        for v in row:
            d = d * v.denominator // math.gcd(d, v.denominator)
    N = [[int(v * d) for v in row] for row in X]
    return N, d


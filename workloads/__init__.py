"""Seeded synthetic inputs for the exact residue GEMM workloads.

This module only draws random numbers. It holds none of the residue method's
arithmetic, so both the CUDA path's tests and the CPU oracle can take their
inputs from here without sharing any computation.

Generator: numpy ``default_rng(seed)`` (PCG64). A is drawn first, then B, both
row-major. Integer entries use ``rng.integers`` over a half-open range;
multi-limb entries draw every 64-bit limb over the full int64 range, which
makes the value uniform over the signed width of the limbs.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    """One named synthetic workload: shapes, entry distribution and seed."""

    name: str
    kind: str  # "int", "limbs", "normal" (float64), "normal32" (float32) or "interval"
    M: int
    N: int
    K: int
    seed: int
    lo: int = 0  # integer range [lo, hi) for kind == "int"
    hi: int = 0
    limbs: int = 1  # limbs per entry for kind == "limbs"
    out_limbs: int = 1  # limbs of the exact result
    nprimes: int = 0  # primes the call is asked to use (0: as many as the bound needs)

    def generate(self):
        """Return (A, B) as numpy arrays."""
        if self.kind == "int":
            return int_matrices(self.M, self.N, self.K, self.lo, self.hi, self.seed)
        if self.kind == "limbs":
            return limb_matrices(self.M, self.N, self.K, self.limbs, self.seed)
        if self.kind == "normal":
            return normal_matrices(self.M, self.N, self.K, self.seed)
        if self.kind == "normal32":
            A, B = normal_matrices(self.M, self.N, self.K, self.seed)
            return A.astype(np.float32), B.astype(np.float32)
        if self.kind == "interval":
            return interval_matrices(self.M, self.N, self.K, self.seed)
        raise ValueError(self.kind)

    @property
    def macs(self) -> int:
        return self.M * self.N * self.K


# The five workloads of the residue engine, plus the square GEMM-stage case.
#  exact24_64     : 64^3, entries uniform in [-2^23, 2^23), seed 0
#  exact24_1024   : 1024^3, same distribution, seed 1 (|C| < 2^57)
#  wide128_2048   : 2048^3, signed 128-bit entries (2 limbs), seed 2, 6-limb result
#  wide128_2048_p53: the same problem on the full set of 53 primes
#  enclose_normal : fp64 standard normal, M=1024, K=4096, N=1024, seed 3
#  longk_int8     : M=N=512, K=131072, entries in [-128, 128), seed 4
#  exact24_4096   : 4096^3, entries in [-2^23, 2^23), seed 5 (GEMM-stage scale)
#  enclose_f32    : enclose_normal's shape and draw, rounded to float32
#  interval_normal: enclose_normal's shape; midpoints standard normal, radii
#                   uniform in [0, 2^-20) times |midpoint|, seed 7
WORKLOADS = {
    "exact24_64": Workload("exact24_64", "int", 64, 64, 64, 0, -(2**23), 2**23),
    "exact24_1024": Workload("exact24_1024", "int", 1024, 1024, 1024, 1, -(2**23), 2**23),
    "wide128_2048": Workload("wide128_2048", "limbs", 2048, 2048, 2048, 2, limbs=2, out_limbs=6),
    "wide128_2048_p53": Workload("wide128_2048_p53", "limbs", 2048, 2048, 2048, 2, limbs=2, out_limbs=6, nprimes=53),
    "enclose_normal": Workload("enclose_normal", "normal", 1024, 1024, 4096, 3),
    "longk_int8": Workload("longk_int8", "int", 512, 512, 131072, 4, -128, 128),
    "exact24_4096": Workload("exact24_4096", "int", 4096, 4096, 4096, 5, -(2**23), 2**23),
    "enclose_f32": Workload("enclose_f32", "normal32", 1024, 1024, 4096, 3),
    "interval_normal": Workload("interval_normal", "interval", 1024, 1024, 4096, 7),
}


def int_matrices(M, N, K, lo, hi, seed):
    """A [M,K] and B [K,N] int64, entries uniform in [lo, hi)."""
    rng = np.random.default_rng(seed)
    A = rng.integers(lo, hi, size=(M, K), dtype=np.int64)
    B = rng.integers(lo, hi, size=(K, N), dtype=np.int64)
    return A, B


def limb_matrices(M, N, K, limbs, seed):
    """A [M,K,L] and B [K,N,L] int64 limbs, little-endian two's complement.

    Every limb is drawn over the whole int64 range; limb 0..L-2 are read as
    unsigned and the top limb as signed, so each value is uniform over
    [-2^(64L-1), 2^(64L-1)).
    """
    rng = np.random.default_rng(seed)
    full = dict(low=-(2**63), high=2**63 - 1, endpoint=True, dtype=np.int64)
    A = rng.integers(size=(M, K, limbs), **full)
    B = rng.integers(size=(K, N, limbs), **full)
    return A, B


def normal_matrices(M, N, K, seed):
    """A [M,K] and B [K,N] float64, i.i.d. standard normal."""
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((K, N))
    return A, B


def interval_matrices(M, N, K, seed):
    """Interval operands as stacked (midpoint, radius) float64 arrays, A [2,M,K] and B [2,K,N]:
    midpoints i.i.d. standard normal, radii uniform in [0, 2^-20) times the midpoint's magnitude."""
    rng = np.random.default_rng(seed)
    Am = rng.standard_normal((M, K))
    Bm = rng.standard_normal((K, N))
    Ar = rng.random((M, K)) * 2.0**-20 * np.abs(Am)
    Br = rng.random((K, N)) * 2.0**-20 * np.abs(Bm)
    return np.stack([Am, Ar]), np.stack([Bm, Br])


def sample_rows(M, seed, n=64):
    """Seeded distinct row indices used to check large outputs row by row."""
    rng = np.random.default_rng(seed + 1000)
    return np.sort(rng.choice(M, size=min(n, M), replace=False)).astype(np.int64)


def solve_system(n, c=1, bits=24, seed=6):
    """A [n, n] and b [n, c] int64 with entries uniform in [-2^(bits-1), 2^(bits-1)): the
    "exact-solve" page's measured systems (24-bit integer entries), seeded."""
    rng = np.random.default_rng(seed + n)
    A = rng.integers(-(2 ** (bits - 1)), 2 ** (bits - 1), size=(n, n), dtype=np.int64)
    b = rng.integers(-(2 ** (bits - 1)), 2 ** (bits - 1), size=(n, c), dtype=np.int64)
    return A, b


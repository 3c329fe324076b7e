"""Split-K in the per-prime GEMM: products with too few output tiles for the
persistent CTAs cut K into slices of whole 1024-K chunks, and the slices'
residues are summed mod q.  Parity against the CPU oracle on every entry
point, both tensor-core kernels, ragged K, batches and transposed B."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import dev, host, rg, variant  # noqa: F401
from tests.test_oracle_interval import random_intervals
from workloads import int_matrices, normal_matrices

pytestmark = pytest.mark.gpu


def bits(x):
    x = np.ascontiguousarray(x)
    return x.view(np.uint32 if x.dtype == np.float32 else np.uint64)


@pytest.mark.parametrize("M,N,K", [(64, 64, 65536), (100, 70, 30000), (1, 300, 20481), (256, 256, 8192),
                                   (130, 260, 131072)])
def test_i64(rg, variant, M, N, K):
    A, B = int_matrices(M, N, K, -(2**15), 2**15, seed=M + K)
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    assert rg.get_plan()["splits"] > 1
    assert np.array_equal(C, oracle.matmul_i64(A, B, lc=1)[:, :, 0])


def test_i64_extreme_residues(rg, variant):
    """Entries of +-(2^23 - 1): every slice's partial residues are large."""
    M, N, K = 40, 50, 40960
    A = np.full((M, K), 2**23 - 1, dtype=np.int64)
    A[::2, ::3] = -(2**23 - 1)
    B = np.full((K, N), -(2**23 - 1), dtype=np.int64)
    B[1::5, :] = 2**23 - 1
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    assert rg.get_plan()["splits"] > 1
    assert np.array_equal(C, oracle.matmul_i64(A, B, lc=1)[:, :, 0])


def test_limbs(rg, variant):
    rng = np.random.default_rng(3)
    full = dict(low=-(2**63), high=2**63 - 1, endpoint=True, dtype=np.int64)
    A = rng.integers(size=(20, 9000, 2), **full)
    B = rng.integers(size=(9000, 30, 2), **full)
    C = host(rg.res_gemm_limbs(dev(A), dev(B), 6))
    assert rg.get_plan()["splits"] > 1
    assert np.array_equal(C, oracle.matmul_limbs(A, B, 6))


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_enclose(rg, variant, dtype):
    A, B = normal_matrices(30, 40, 16384, seed=4)
    A, B = A.astype(dtype), B.astype(dtype)
    lo, hi = rg.mm_enclose(dev(A), dev(B))
    assert rg.get_plan()["splits"] > 1
    enc = oracle.enclose_f32 if dtype == np.float32 else oracle.enclose_f64
    rlo, rhi = enc(A, B)
    assert np.array_equal(bits(host(lo)), bits(rlo)) and np.array_equal(bits(host(hi)), bits(rhi))


def test_batched_transposed_and_interval(rg, variant):
    A, B = normal_matrices(2 * 16, 24, 12000, seed=5)
    A3 = A.reshape(2, 16, 12000)
    B3 = np.stack([B, -B / 4])
    lo, hi = rg.enclose_gemm(dev(A3), dev(np.ascontiguousarray(B3.transpose(0, 2, 1))), transb=True)
    assert rg.get_plan()["splits"] > 1
    for i in range(2):
        rlo, rhi = oracle.enclose_f64(A3[i], B3[i])
        assert np.array_equal(bits(host(lo)[i]), bits(rlo)) and np.array_equal(bits(host(hi)[i]), bits(rhi))
    Am, Ar, Bm, Br = random_intervals(20, 30, 9000, 6)
    lo, hi = rg.mm_interval(*(dev(x) for x in (Am, Ar, Bm, Br)))
    assert rg.get_plan()["splits"] > 1
    rlo, rhi = oracle.interval(Am, Ar, Bm, Br)
    assert np.array_equal(bits(host(lo)), bits(rlo)) and np.array_equal(bits(host(hi)), bits(rhi))


def test_many_tiles_do_not_split(rg):
    """448 tiles (7 primes, 2048^2) fill the GPU six times over: no split pays for its summing pass."""
    A, B = int_matrices(2048, 2048, 2048, -(2**20), 2**20, seed=7)
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    assert rg.get_plan()["splits"] == 1
    rows = np.array([0, 777, 2047])
    assert np.array_equal(C[rows], oracle.matmul_i64(A, B, lc=1, rows=rows)[:, :, 0])

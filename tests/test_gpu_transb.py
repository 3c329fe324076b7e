"""GPU parity of the transposed-B form (RG_FLAG_TRANS_B; "enclosure-gemm",
Usage: mm_enclose_nt, A @ Bt.T without a transposed copy) against the CPU
oracle, which receives the untransposed B.  Every entry point, both
tensor-core kernels, ragged shapes spanning several tiles and K chunks."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import dev, host, rg, variant  # noqa: F401
from workloads import WORKLOADS, int_matrices, limb_matrices, normal_matrices

pytestmark = pytest.mark.gpu


def bits(x):
    return np.ascontiguousarray(x).view(np.uint64)


SHAPES = [(1, 1, 1), (3, 5, 7), (65, 77, 129), (130, 300, 2049), (300, 520, 1100)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_i64(rg, variant, M, N, K):
    A, B = int_matrices(M, N, K, -(2**23), 2**23, seed=M + N + K)
    Bt = np.ascontiguousarray(B.T)
    C = host(rg.res_gemm_i64(dev(A), dev(Bt), transb=True))
    assert np.array_equal(C, oracle.matmul_i64(A, B, lc=1)[:, :, 0])


def test_i64_workload_1024(rg, variant):
    w = WORKLOADS["exact24_1024"]
    A, B = w.generate()
    C = host(rg.res_gemm_i64(dev(A), dev(np.ascontiguousarray(B.T)), transb=True))
    assert np.array_equal(C, oracle.matmul_i64(A, B, lc=1)[:, :, 0])


def test_i64_host_buffers(rg):
    A, B = int_matrices(70, 90, 300, -(2**26), 2**26, seed=11)  # |C| < 2^61
    C = rg.res_gemm_i64(torch.from_numpy(A), torch.from_numpy(np.ascontiguousarray(B.T)), transb=True)
    assert C.device.type == "cpu"
    assert np.array_equal(C.numpy(), oracle.matmul_i64(A, B, lc=1)[:, :, 0])


@pytest.mark.parametrize("M,N,K,la,lb,lc", [(33, 65, 70, 2, 2, 6), (130, 260, 1030, 2, 2, 6), (17, 9, 11, 3, 1, 5)])
def test_limbs(rg, variant, M, N, K, la, lb, lc):
    rng = np.random.default_rng(M * N + K)
    full = dict(low=-(2**63), high=2**63 - 1, endpoint=True, dtype=np.int64)
    A = rng.integers(size=(M, K, la), **full)
    B = rng.integers(size=(K, N, lb), **full)
    C = host(rg.res_gemm_limbs(dev(A), dev(np.ascontiguousarray(B.transpose(1, 0, 2))), lc, transb=True))
    assert np.array_equal(C, oracle.matmul_limbs(A, B, lc))


@pytest.mark.parametrize("M,N,K", [(3, 4, 8), (65, 77, 129), (130, 260, 1030)])
def test_enclose(rg, variant, M, N, K):
    A, B = normal_matrices(M, N, K, seed=K)
    lo, hi = rg.mm_enclose_nt(dev(A), dev(np.ascontiguousarray(B.T)))
    rlo, rhi = oracle.enclose_f64(A, B)
    assert np.array_equal(bits(host(lo)), bits(rlo))
    assert np.array_equal(bits(host(hi)), bits(rhi))


def test_enclose_nt_digest_equals_nn(rg):
    """The same bracket, bit for bit, whichever way B is handed over."""
    A, B = normal_matrices(200, 333, 2100, seed=5)
    lo, hi = rg.mm_enclose(dev(A), dev(B))
    lo_t, hi_t = rg.mm_enclose_nt(dev(A), dev(np.ascontiguousarray(B.T)))
    assert rg.digest(lo, hi) == rg.digest(lo_t, hi_t)


def test_enclose_nt_wide_operands_lossy(rg):
    """Operands spanning more binades than the fixed point: a valid bracket in the transposed form too."""
    rng = np.random.default_rng(9)
    A = rng.standard_normal((20, 64)) * np.exp2(rng.integers(-260, 260, size=(20, 64)))
    B = rng.standard_normal((64, 30)) * np.exp2(rng.integers(-150, 150, size=(64, 30)))
    lo, hi = rg.mm_enclose_nt(dev(A), dev(np.ascontiguousarray(B.T)))
    rlo, rhi = oracle.enclose_f64(A, B)
    assert np.all(host(lo) <= rlo) and np.all(host(hi) >= rhi)


def test_shape_mismatch_rejected(rg):
    A = torch.zeros((4, 8), dtype=torch.int64, device="cuda")
    Bt = torch.zeros((5, 9), dtype=torch.int64, device="cuda")
    with pytest.raises(ValueError):
        rg.res_gemm_i64(A, Bt, transb=True)

"""GPU parity of the batched forms ("enclosure-gemm", Usage: bmm_enclose; a
batch shares one plan) and of empty problems, against the CPU oracle applied
product by product: a batch is by definition the stack of its products.

Where one shared scale is lossless, every product's bracket must equal the
oracle's tightest pair bit for bit (the shared binary point only adds exact
trailing zero bits); where the batch is wider than the fixed point the
brackets must contain the tightest ones."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import dev, host, rg, variant  # noqa: F401
from workloads import normal_matrices

pytestmark = pytest.mark.gpu


def bits(x):
    return np.ascontiguousarray(x).view(np.uint64)


def normal_batch(b, M, N, K, seed):
    pairs = [normal_matrices(M, N, K, seed + i) for i in range(b)]
    return np.stack([p[0] for p in pairs]), np.stack([p[1] for p in pairs])


def oracle_bracket(A, B):
    lo, hi = zip(*(oracle.enclose_f64(A[i], B[i]) for i in range(A.shape[0])))
    return np.stack(lo), np.stack(hi)


def test_bmm_enclose_five_small_products(rg):
    """The pages' batch: five 20x256x12 products."""
    A, B = normal_batch(5, 20, 12, 256, seed=40)
    lo, hi = rg.bmm_enclose(dev(A), dev(B))
    assert lo.shape == (5, 20, 12)
    rlo, rhi = oracle_bracket(A, B)
    assert np.array_equal(bits(host(lo)), bits(rlo)) and np.array_equal(bits(host(hi)), bits(rhi))
    assert rg.get_plan()["lossless"] == 1


@pytest.mark.parametrize("b,M,N,K", [(3, 65, 77, 129), (4, 130, 300, 1030), (2, 257, 260, 64), (7, 1, 1, 1)])
def test_bmm_enclose_ragged(rg, variant, b, M, N, K):
    A, B = normal_batch(b, M, N, K, seed=M + N + K)
    lo, hi = rg.bmm_enclose(dev(A), dev(B))
    rlo, rhi = oracle_bracket(A, B)
    assert np.array_equal(bits(host(lo)), bits(rlo)) and np.array_equal(bits(host(hi)), bits(rhi))


def test_bmm_enclose_products_of_different_scales(rg):
    """Each product has its own magnitude; the shared plan still scales losslessly."""
    A, B = normal_batch(4, 33, 40, 300, seed=3)
    for i, (sa, sb) in enumerate([(0, 0), (-30, 10), (20, -40), (-10, -20)]):  # ~120 + 120 + 9 bits
        A[i] *= 2.0**sa
        B[i] *= 2.0**sb
    lo, hi = rg.bmm_enclose(dev(A), dev(B))
    assert rg.get_plan()["lossless"] == 1
    rlo, rhi = oracle_bracket(A, B)
    assert np.array_equal(bits(host(lo)), bits(rlo)) and np.array_equal(bits(host(hi)), bits(rhi))


def test_bmm_enclose_wider_than_the_fixed_point(rg):
    """Products 400 binades apart: the batch is coarsened, every bracket stays valid."""
    A, B = normal_batch(2, 20, 30, 64, seed=8)
    A[1] *= 2.0**400
    lo, hi = rg.bmm_enclose(dev(A), dev(B))
    assert rg.get_plan()["lossless"] == 0
    rlo, rhi = oracle_bracket(A, B)
    lo, hi = host(lo), host(hi)
    assert np.all(lo <= rlo) and np.all(hi >= rhi)


def test_bmm_enclose_transposed(rg, variant):
    A, B = normal_batch(3, 70, 90, 500, seed=12)
    Bt = np.ascontiguousarray(B.transpose(0, 2, 1))
    lo, hi = rg.enclose_gemm_f64(dev(A), dev(Bt), transb=True)
    rlo, rhi = oracle_bracket(A, B)
    assert np.array_equal(bits(host(lo)), bits(rlo)) and np.array_equal(bits(host(hi)), bits(rhi))


@pytest.mark.parametrize("b,M,N,K", [(3, 65, 77, 129), (5, 130, 300, 2049)])
def test_batched_i64(rg, variant, b, M, N, K):
    rng = np.random.default_rng(b * M + K)
    A = rng.integers(-(2**23), 2**23, size=(b, M, K), dtype=np.int64)
    B = rng.integers(-(2**23), 2**23, size=(b, K, N), dtype=np.int64)
    A[1] //= 2**20  # products of different magnitudes share the prime count
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    for i in range(b):
        assert np.array_equal(C[i], oracle.matmul_i64(A[i], B[i], lc=1)[:, :, 0]), i


def test_batched_i64_host_buffers_and_transposed(rg):
    rng = np.random.default_rng(5)
    A = rng.integers(-(2**25), 2**25, size=(3, 40, 300), dtype=np.int64)
    B = rng.integers(-(2**25), 2**25, size=(3, 300, 50), dtype=np.int64)
    C = rg.res_gemm_i64(torch.from_numpy(A), torch.from_numpy(np.ascontiguousarray(B.transpose(0, 2, 1))),
                        transb=True)
    assert C.device.type == "cpu" and C.shape == (3, 40, 50)
    for i in range(3):
        assert np.array_equal(C[i].numpy(), oracle.matmul_i64(A[i], B[i], lc=1)[:, :, 0])


def test_batched_limbs(rg, variant):
    rng = np.random.default_rng(6)
    full = dict(low=-(2**63), high=2**63 - 1, endpoint=True, dtype=np.int64)
    A = rng.integers(size=(3, 33, 70, 2), **full)
    B = rng.integers(size=(3, 70, 65, 2), **full)
    C = host(rg.res_gemm_limbs(dev(A), dev(B), 6))
    for i in range(3):
        assert np.array_equal(C[i], oracle.matmul_limbs(A[i], B[i], 6)), i


@pytest.mark.parametrize("b,M,N,K", [(1, 0, 5, 7), (1, 5, 0, 7), (1, 5, 6, 0), (0, 5, 6, 7), (2, 3, 4, 0)])
def test_empty_problems(rg, b, M, N, K):
    """Empty shapes run no kernel; K = 0 is the empty sum, exactly zero."""
    A = torch.ones((b, M, K), dtype=torch.float64, device="cuda")
    B = torch.ones((b, K, N), dtype=torch.float64, device="cuda")
    lo, hi = rg.enclose_gemm_f64(A, B)
    assert lo.shape == (b, M, N)
    assert not bits(host(lo)).any() and not bits(host(hi)).any()  # +0.0 exactly
    C = rg.res_gemm_i64(A.long(), B.long())
    assert C.shape == (b, M, N) and not host(C).any()
    C = rg.res_gemm_limbs(A.long()[..., None].repeat_interleave(2, -1), B.long()[..., None], 3)
    assert C.shape == (b, M, N, 3) and not host(C).any()
    if not (M and N and K):  # the same empty problem through host buffers
        lo, hi = rg.enclose_gemm_f64(torch.ones((M, K), dtype=torch.float64), torch.ones((K, N), dtype=torch.float64))
        assert lo.shape == (M, N) and not bits(lo.numpy()).any() and not bits(hi.numpy()).any()
    assert rg.status() == rg.RG_OK

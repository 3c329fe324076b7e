"""GPU parity of the binary32 enclosure (enclose_gemm_f32; "enclosure-gemm",
Usage: operands are float32 or float64) against the CPU oracle's tightest
float pair, bit for bit wherever the scaling is lossless, containment
otherwise."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import dev, host, rg, variant  # noqa: F401
from tests.test_oracle_enclose_f32 import CASES_F32, random_f32

pytestmark = pytest.mark.gpu
F32 = np.float32


def bits(x):
    return np.ascontiguousarray(x, dtype=F32).view(np.uint32)


def check_equal(rg, A, B, rows=None):
    lo, hi = rg.mm_enclose(dev(A), dev(B))
    assert lo.dtype == torch.float32
    lo, hi = host(lo), host(hi)
    rlo, rhi = oracle.enclose_f32(A, B, rows=rows)
    if rows is not None:
        lo, hi = lo[rows], hi[rows]
    assert np.array_equal(bits(lo), bits(rlo))
    assert np.array_equal(bits(hi), bits(rhi))


@pytest.mark.parametrize("A,B,lo,hi", CASES_F32)
def test_hand_cases(rg, A, B, lo, hi):
    glo, ghi = rg.mm_enclose(dev(np.array(A, dtype=F32)), dev(np.array(B, dtype=F32)))
    assert rg.get_plan()["lossless"] == 1
    assert bits(host(glo))[0, 0] == bits(np.array([lo], dtype=F32))[0]
    assert bits(host(ghi))[0, 0] == bits(np.array([hi], dtype=F32))[0]


@pytest.mark.parametrize("M,N,K,seed,spread", [(3, 4, 8, 0, 0), (65, 77, 129, 1, 0), (130, 260, 1030, 2, 10),
                                               (40, 300, 4096, 3, 0), (129, 257, 2049, 4, 40)])
def test_random(rg, variant, M, N, K, seed, spread):
    A, B = random_f32(M, N, K, seed, spread)
    check_equal(rg, A, B)


def test_uses_binary32_significands(rg):
    """Normal float32 operands plan from 24-bit significands: fewer primes than
    the same values as float64."""
    A, B = random_f32(64, 64, 1024, 5)
    rg.mm_enclose(dev(A), dev(B))
    p32 = rg.get_plan()
    rg.mm_enclose(dev(A.astype(np.float64)), dev(B.astype(np.float64)))
    p64 = rg.get_plan()
    assert p32["lossless"] == 1 and p32["bits_a"] == p64["bits_a"] - 29 and p32["nprimes"] < p64["nprimes"]


def test_subnormal_and_overflow(rg):
    rng = np.random.default_rng(7)
    A = (rng.standard_normal((30, 50)) * 2.0**-70).astype(F32)
    B = (rng.standard_normal((50, 20)) * 2.0**-72).astype(F32)
    A[0, :3] = [2.0**-149, -(2.0**-149), 0.0]
    check_equal(rg, A, B)
    A = (rng.standard_normal((30, 50)) * 2.0**100).astype(F32)
    B = (rng.standard_normal((50, 20)) * 2.0**26).astype(F32)  # sums overflow binary32 in places
    check_equal(rg, A, B)
    lo, hi = rg.mm_enclose(dev(A), dev(B))
    assert bool(torch.isinf(hi).any() | torch.isinf(lo).any())


def test_wide_operands_are_bracketed(rg):
    """The whole binary32 range in one operand (277 bits > 255): a valid, looser bracket."""
    rng = np.random.default_rng(8)
    A = (rng.standard_normal((20, 64)) * np.exp2(rng.integers(-140, 120, size=(20, 64)))).astype(F32)
    B = (rng.standard_normal((64, 30)) * np.exp2(rng.integers(-40, 40, size=(64, 30)))).astype(F32)
    lo, hi = rg.mm_enclose(dev(A), dev(B))
    assert rg.get_plan()["lossless"] == 0
    rlo, rhi = oracle.enclose_f32(A, B)
    lo, hi = host(lo), host(hi)
    assert np.all(lo <= rlo) and np.all(hi >= rhi)


def test_transposed_batched_and_host(rg):
    A, B = random_f32(3 * 40, 50, 300, 9)
    A3, B3 = A.reshape(3, 40, 300), np.stack([B] * 3)
    B3[1] *= 2.0**-12
    lo, hi = rg.bmm_enclose(dev(A3), dev(B3))
    for i in range(3):
        rlo, rhi = oracle.enclose_f32(A3[i], B3[i])
        assert np.array_equal(bits(host(lo)[i]), bits(rlo)) and np.array_equal(bits(host(hi)[i]), bits(rhi))
    lo, hi = rg.mm_enclose_nt(dev(A3[0]), dev(np.ascontiguousarray(B3[0].T)))
    rlo, rhi = oracle.enclose_f32(A3[0], B3[0])
    assert np.array_equal(bits(host(lo)), bits(rlo)) and np.array_equal(bits(host(hi)), bits(rhi))
    lo, hi = rg.mm_enclose(torch.from_numpy(A3[2]), torch.from_numpy(B3[2]))
    assert lo.device.type == "cpu" and lo.dtype == torch.float32
    rlo, rhi = oracle.enclose_f32(A3[2], B3[2])
    assert np.array_equal(bits(lo.numpy()), bits(rlo)) and np.array_equal(bits(hi.numpy()), bits(rhi))


def test_nonfinite_rejected(rg):
    A = np.ones((4, 4), dtype=F32)
    A[1, 2] = np.nan
    with pytest.raises(rg.ResGemmError) as e:
        rg.mm_enclose(dev(A), dev(np.ones((4, 4), dtype=F32)))
    assert e.value.code == rg.RG_ERR_NONFINITE


def test_mixed_dtypes_rejected(rg):
    with pytest.raises(ValueError):
        rg.mm_enclose(torch.ones((4, 4), dtype=torch.float32, device="cuda"),
                      torch.ones((4, 4), dtype=torch.float64, device="cuda"))


def test_enclose_f32_workload_sampled_rows(rg):
    """The bench's float32 enclosure workload at full size (1024 x 4096 x 1024): sample rows bit for bit."""
    from workloads import WORKLOADS, sample_rows

    w = WORKLOADS["enclose_f32"]
    A, B = w.generate()
    lo, hi = rg.enclose_gemm_f32(dev(A), dev(B))
    assert rg.get_plan()["lossless"] == 1
    rows = sample_rows(w.M, w.seed, n=16)
    rlo, rhi = oracle.enclose_f32(A, B, rows=rows)
    assert np.array_equal(host(lo)[rows].view(np.uint32), rlo.view(np.uint32))
    assert np.array_equal(host(hi)[rows].view(np.uint32), rhi.view(np.uint32))

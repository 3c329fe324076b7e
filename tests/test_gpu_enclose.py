"""GPU parity of the fp64 enclosure (enclose_gemm_f64) against the CPU oracle.

Both IEEE endpoints must match the oracle bit for bit wherever the scaling is
lossless ("enclosure-gemm", Correctness: equal to the exact floor and ceiling
in the format).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import dev, host, rg  # noqa: F401
from tests.test_oracle_enclose import HAND_CASES
from workloads import WORKLOADS, normal_matrices

pytestmark = pytest.mark.gpu


def bits(x):
    return np.ascontiguousarray(x).view(np.uint64)


def check_equal(rg, A, B, rows=None):
    lo, hi = rg.enclose_gemm_f64(dev(A), dev(B))
    lo, hi = host(lo), host(hi)
    rlo, rhi = oracle.enclose_f64(A, B, rows=rows)
    if rows is not None:
        lo, hi = lo[rows], hi[rows]
    assert np.array_equal(bits(lo), bits(rlo))
    assert np.array_equal(bits(hi), bits(rhi))


def check_contains(glo, ghi, rlo, rhi):
    """The returned pair brackets the tightest pair (hence the exact value)."""
    assert np.all(glo <= rlo) and np.all(ghi >= rhi)
    assert not np.any(np.isnan(glo)) and not np.any(np.isnan(ghi))


@pytest.mark.parametrize("A,B,lo,hi", HAND_CASES)
def test_hand_cases(rg, A, B, lo, hi):
    A = np.array(A, dtype=np.float64)
    B = np.array(B, dtype=np.float64)
    glo, ghi = rg.enclose_gemm_f64(dev(A), dev(B))
    if rg.get_plan()["lossless"]:
        assert bits(host(glo))[0, 0] == bits(np.array([lo]))[0]
        assert bits(host(ghi))[0, 0] == bits(np.array([hi]))[0]
    else:  # operands wider than the fixed point: a valid, looser bracket
        check_contains(host(glo), host(ghi), np.array([[lo]]), np.array([[hi]]))


@pytest.mark.parametrize("M,N,K,seed", [(3, 4, 8, 0), (65, 77, 129, 1), (130, 260, 1030, 2), (1, 1, 1, 3),
                                        (40, 300, 4096, 4)])
def test_random_normal(rg, M, N, K, seed):
    A, B = normal_matrices(M, N, K, seed)
    check_equal(rg, A, B)


def test_scaled_and_subnormal_operands(rg):
    rng = np.random.default_rng(7)
    A = rng.standard_normal((30, 50)) * 2.0**-1040  # subnormal and tiny normals
    B = rng.standard_normal((50, 20)) * 2.0**-30
    A[0, :4] = [5e-324, -5e-324, 1.5e-323, 0.0]
    check_equal(rg, A, B)
    A = rng.standard_normal((30, 50)) * 2.0**900
    B = rng.standard_normal((50, 20)) * 2.0**120  # overflows to +-inf in places
    check_equal(rg, A, B)
    lo, hi = rg.enclose_gemm_f64(dev(A), dev(B))
    assert bool(torch.isinf(hi).any() | torch.isinf(lo).any())


def test_integer_operands_equal_plain_product(rg):
    rng = np.random.default_rng(0)
    A = rng.integers(-(2**20), 2**20, size=(70, 64)).astype(np.float64)
    B = rng.integers(-(2**20), 2**20, size=(64, 90)).astype(np.float64)
    lo, hi = rg.enclose_gemm_f64(dev(A), dev(B))
    ref = A @ B
    assert np.array_equal(host(lo), ref) and np.array_equal(host(hi), ref)


def test_cancellation(rg):
    # 1e300 .. 2^-60 spans more than 255 bits: coarsened, still a valid bracket
    A = np.array([[1e300, 1.0, -1e300, 2.0**-60]], dtype=np.float64)
    B = np.ones((4, 1))
    lo, hi = rg.enclose_gemm_f64(dev(A), dev(B))
    assert rg.get_plan()["lossless"] == 0
    rlo, rhi = oracle.enclose_f64(A, B)
    check_contains(host(lo), host(hi), rlo, rhi)
    A = np.array([[2.0**100, 1.0, -(2.0**100), 3 * 2.0**-60]], dtype=np.float64)
    check_equal(rg, A, B)
    assert rg.get_plan()["lossless"] == 1


@pytest.mark.parametrize("M,N,K,span,seed", [(9, 7, 33, 520, 0), (40, 50, 300, 520, 1), (20, 30, 2000, 300, 2),
                                             (16, 16, 64, 1500, 3)])
def test_wide_operands_are_bracketed(rg, M, N, K, span, seed):
    """Operands spanning `span` binades ("enclosure-gemm", Correctness: 520
    binades, containment required, tightness not): the pair must contain the
    exact product; where a result is large against the coarsening error the
    bracket is still one step wide."""
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K)) * np.exp2(rng.integers(-span // 2, span // 2, size=(M, K)).astype(np.float64))
    B = rng.standard_normal((K, N)) * np.exp2(rng.integers(-span // 4, span // 4, size=(K, N)).astype(np.float64))
    lo, hi = rg.enclose_gemm_f64(dev(A), dev(B))
    plan = rg.get_plan()
    assert plan["status"] == 0 and plan["lossless"] == 0
    assert plan["bits_a"] + plan["bits_b"] + int(np.ceil(np.log2(K))) <= 332
    rlo, rhi = oracle.enclose_f64(A, B)
    check_contains(host(lo), host(hi), rlo, rhi)
    width = host(rg.width_ulps(lo, hi))
    assert (width <= 1).mean() > 0.5  # most entries are dominated by large terms


def test_nonfinite_rejected(rg):
    A = np.ones((4, 4))
    A[1, 2] = np.nan
    with pytest.raises(rg.ResGemmError) as e:
        rg.enclose_gemm_f64(dev(A), dev(np.ones((4, 4))))
    assert e.value.code == rg.RG_ERR_NONFINITE
    B = np.ones((4, 4))
    B[3, 3] = -np.inf
    with pytest.raises(rg.ResGemmError) as e:
        rg.enclose_gemm_f64(dev(np.ones((4, 4))), dev(B))
    assert e.value.code == rg.RG_ERR_NONFINITE


def test_enclose_normal_workload(rg):
    w = WORKLOADS["enclose_normal"]
    A, B = w.generate()
    lo, hi = rg.enclose_gemm_f64(dev(A), dev(B))
    plan = rg.get_plan()
    assert plan["lossless"] == 1 and plan["status"] == 0
    # one representable step everywhere ("enclosure-gemm", Usage: width_ulps(...).max() == 1)
    width = rg.width_ulps(lo, hi)
    assert int(width.max()) == 1 and int(width.min()) >= 0
    # both endpoints of every entry, bit for bit
    rlo, rhi = oracle.enclose_f64(A, B)
    assert np.array_equal(bits(host(lo)), bits(rlo))
    assert np.array_equal(bits(host(hi)), bits(rhi))


def test_host_buffers_and_digest(rg):
    A, B = normal_matrices(33, 44, 55, 9)
    lo1, hi1 = rg.enclose_gemm_f64(dev(A), dev(B))
    lo2, hi2 = rg.enclose_gemm_f64(torch.from_numpy(A), torch.from_numpy(B))
    assert lo2.device.type == "cpu"
    assert rg.digest(lo1, hi1) == rg.digest(lo2, hi2)


def test_return_info_reports_the_regime(rg):
    """return_info names the regime ("enclosure-gemm", Method: lossless one-step bracket, or coarsened)."""
    B = np.ones((4, 1))
    wide = np.array([[1e300, 1.0, -1e300, 2.0**-60]], dtype=np.float64)
    lo, hi, info = rg.mm_enclose(dev(wide), dev(B), return_info=True)
    assert info["regime"] == "coarsened" and not info["lossless"]
    rlo, rhi = oracle.enclose_f64(wide, B)
    check_contains(host(lo), host(hi), rlo, rhi)
    narrow = np.array([[2.0**100, 1.0, -(2.0**100), 3 * 2.0**-60]], dtype=np.float64)
    lo, hi, info = rg.mm_enclose_nt(dev(narrow), dev(B.T.copy()), return_info=True)
    assert info["regime"] == "lossless" and info["lossless"] and info["nprimes"] >= 1
    rlo, rhi = oracle.enclose_f64(narrow, B)
    assert np.array_equal(host(lo), rlo) and np.array_equal(host(hi), rhi)
    lo, hi = rg.bmm_enclose(dev(narrow[None]), dev(B[None]))
    assert np.array_equal(host(lo)[0], rlo)
    lo, hi, info = rg.bmm_enclose(dev(narrow[None]), dev(B[None]), return_info=True)
    assert info["lossless"]


def test_entry_point_reports_the_regime_in_info(rg):
    """enclose_gemm_f64's info out-argument: 0 for a lossless scaling, 1 for a coarsened one; the bounds
    equal the binding's (which reads the regime from the plan instead)."""
    import ctypes

    lib = rg.library()
    B = np.ones((4, 1))
    for A, want in ((np.array([[1e300, 1.0, -1e300, 2.0**-60]]), 1),
                    (np.array([[2.0**100, 1.0, -(2.0**100), 3 * 2.0**-60]]), 0)):
        dA, dB = dev(A), dev(B)
        lo = torch.empty((1, 1), dtype=torch.float64, device="cuda")
        hi = torch.empty_like(lo)
        ws = rg.workspace(rg.workspace_bytes(rg.RG_OP_ENCLOSE, 1, 1, 4), torch.device("cuda", 0))
        info = ctypes.c_int(-1)
        rc = lib.enclose_gemm_f64(dA.data_ptr(), dB.data_ptr(), lo.data_ptr(), hi.data_ptr(), 1, 1, 4, 0,
                                  ctypes.byref(info), ws.data_ptr(), ws.numel(),
                                  torch.cuda.current_stream().cuda_stream)
        assert rc == rg.RG_OK and info.value == want
        rlo, rhi = rg.enclose_gemm_f64(dA, dB)
        assert torch.equal(lo, rlo) and torch.equal(hi, rhi)


def test_smaller_workspace_caps_the_primes(rg):
    """A workspace for fewer primes than the lossless plan needs gives a coarsened, valid bracket; one
    sized for the count a first call reports gives the same bits as the full workspace."""
    A, B = normal_matrices(64, 48, 256, 21)
    dA, dB = dev(A), dev(B)
    lo, hi = rg.enclose_gemm_f64(dA, dB)
    full = rg.get_plan()
    assert full["lossless"] == 1
    P = full["nprimes"]
    d0 = torch.device("cuda", 0)
    exact = torch.empty(rg.workspace_bytes(rg.RG_OP_ENCLOSE, 64, 48, 256, nprimes=P), dtype=torch.uint8, device=d0)
    lo2, hi2 = rg.enclose_gemm_f64(dA, dB, ws=exact)
    assert torch.equal(lo2, lo) and torch.equal(hi2, hi)
    assert rg.get_plan(ws=exact)["nprimes"] == P and rg.get_plan(ws=exact)["lossless"] == 1
    small = torch.empty(rg.workspace_bytes(rg.RG_OP_ENCLOSE, 64, 48, 256, nprimes=P - 6), dtype=torch.uint8,
                        device=d0)
    lo3, hi3 = rg.enclose_gemm_f64(dA, dB, ws=small)
    plan = rg.get_plan(ws=small)
    assert plan["lossless"] == 0 and plan["nprimes"] <= P - 6
    rlo, rhi = oracle.enclose_f64(A, B)
    check_contains(host(lo3), host(hi3), rlo, rhi)
    tiny = torch.empty(rg.workspace_bytes(rg.RG_OP_ENCLOSE, 64, 48, 256, nprimes=1), dtype=torch.uint8, device=d0)
    with pytest.raises(rg.ResGemmError) as e:  # 7 bits of residue range cannot hold K = 256
        rg.enclose_gemm_f64(dA, dB, ws=tiny)
    assert e.value.code == rg.RG_ERR_WORKSPACE
    with pytest.raises(rg.ResGemmError) as e:
        rg.enclose_gemm_f64(dA, dB, ws=tiny[:4096])
    assert e.value.code == rg.RG_ERR_WORKSPACE

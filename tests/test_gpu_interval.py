"""GPU parity of the interval product (interval_gemm / mm_interval; "enclosure-
gemm", Usage: mm_interval; Method: Rump's midpoint-radius bound, its three
products and radius formed exactly) against the CPU oracle, bit for bit where
the scaling is lossless and by containment where it is coarsened."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import dev, host, rg, variant  # noqa: F401
from tests.test_oracle_interval import random_intervals

pytestmark = pytest.mark.gpu


def bits(x):
    x = np.ascontiguousarray(x)
    return x.view(np.uint32 if x.dtype == np.float32 else np.uint64)


def check_equal(rg, Am, Ar, Bm, Br, rows=None):
    lo, hi = rg.mm_interval(dev(Am), dev(Ar), dev(Bm), dev(Br))
    assert rg.get_plan()["lossless"] == 1
    lo, hi = host(lo), host(hi)
    rlo, rhi = oracle.interval(Am, Ar, Bm, Br, rows=rows)
    if rows is not None:
        lo, hi = lo[rows], hi[rows]
    assert np.array_equal(bits(lo), bits(rlo))
    assert np.array_equal(bits(hi), bits(rhi))


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 0), (3, 5, 7, 1), (65, 77, 129, 2), (130, 260, 1030, 3),
                                        (129, 300, 2049, 4)])
def test_random(rg, variant, dtype, M, N, K, seed):
    check_equal(rg, *random_intervals(M, N, K, seed, dtype))


def test_integer_intervals_exact(rg):
    rng = np.random.default_rng(1)
    M, N, K = 70, 90, 300
    Am = rng.integers(-2000, 2000, size=(M, K))
    Ar = rng.integers(0, 300, size=(M, K))
    Bm = rng.integers(-2000, 2000, size=(K, N))
    Br = rng.integers(0, 300, size=(K, N))
    mid = Am @ Bm
    rad = np.abs(Am) @ Br + Ar @ np.abs(Bm) + Ar @ Br
    lo, hi = rg.mm_interval(*(dev(x.astype(np.float64)) for x in (Am, Ar, Bm, Br)))
    assert np.array_equal(host(lo), (mid - rad).astype(np.float64))
    assert np.array_equal(host(hi), (mid + rad).astype(np.float64))


def test_zero_radius_equals_point_enclosure(rg):
    Am, _, Bm, _ = random_intervals(100, 120, 700, 5)
    lo, hi = rg.mm_interval(dev(Am), dev(np.zeros_like(Am)), dev(Bm), dev(np.zeros_like(Bm)))
    elo, ehi = rg.mm_enclose(dev(Am), dev(Bm))
    assert rg.digest(lo, hi) == rg.digest(elo, ehi)


def test_radius_scales_and_signs(rg):
    """Radii many binades below and above the midpoints, signed zeros, exact zeros."""
    Am, Ar, Bm, Br = random_intervals(40, 50, 300, 6, rad_scale=2.0**-60)
    Ar[:, ::3] *= 2.0**70
    Br[::5, :] = 0.0
    Br[1::7, :] = -0.0
    Am[::4, ::2] = 0.0
    check_equal(rg, Am, Ar, Bm, Br)


def test_transposed_batched_and_host(rg, variant):
    Am, Ar, Bm, Br = random_intervals(3 * 30, 40, 200, 7)
    A3m, A3r = Am.reshape(3, 30, 200), Ar.reshape(3, 30, 200)
    B3m, B3r = np.stack([Bm, 2 * Bm, Bm / 8]), np.stack([Br, Br, 4 * Br])
    lo, hi = rg.interval_gemm(*(dev(x) for x in (A3m, A3r, B3m, B3r)))
    for i in range(3):
        rlo, rhi = oracle.interval(A3m[i], A3r[i], B3m[i], B3r[i])
        assert np.array_equal(bits(host(lo)[i]), bits(rlo)) and np.array_equal(bits(host(hi)[i]), bits(rhi))
    T = lambda x: np.ascontiguousarray(x.T)  # noqa: E731
    lo, hi = rg.interval_gemm(dev(Am), dev(Ar), dev(T(Bm)), dev(T(Br)), transb=True)
    rlo, rhi = oracle.interval(Am, Ar, Bm, Br)
    assert np.array_equal(bits(host(lo)), bits(rlo)) and np.array_equal(bits(host(hi)), bits(rhi))
    lo, hi = rg.mm_interval(*(torch.from_numpy(x) for x in (Am, Ar, Bm, Br)))
    assert lo.device.type == "cpu"
    assert np.array_equal(bits(lo.numpy()), bits(rlo)) and np.array_equal(bits(hi.numpy()), bits(rhi))


def test_wide_operands_are_bracketed(rg):
    """Midpoints and radii spanning more than the fixed point: coarsened, still containing the tight pair."""
    rng = np.random.default_rng(8)
    Am, Ar, Bm, Br = random_intervals(20, 30, 64, 8, rad_scale=2.0**-200)
    Am *= np.exp2(rng.integers(-100, 100, size=Am.shape))
    Bm *= np.exp2(rng.integers(-60, 60, size=Bm.shape))
    lo, hi = rg.mm_interval(*(dev(x) for x in (Am, Ar, Bm, Br)))
    assert rg.get_plan()["lossless"] == 0
    rlo, rhi = oracle.interval(Am, Ar, Bm, Br)
    assert np.all(host(lo) <= rlo) and np.all(host(hi) >= rhi)


def test_negative_radius_rejected(rg):
    Am, Ar, Bm, Br = random_intervals(8, 8, 8, 9)
    Br[3, 4] = -(2.0**-30)
    with pytest.raises(rg.ResGemmError) as e:
        rg.mm_interval(*(dev(x) for x in (Am, Ar, Bm, Br)))
    assert e.value.code == rg.RG_ERR_RADIUS


def test_interval_normal_workload_sampled_rows(rg):
    """The bench's interval workload at full size (1024 x 4096 x 1024): seeded sample rows bit for bit."""
    from workloads import WORKLOADS, sample_rows

    w = WORKLOADS["interval_normal"]
    A, B = w.generate()
    lo, hi = rg.interval_gemm(dev(A[0]), dev(A[1]), dev(B[0]), dev(B[1]))
    assert rg.get_plan()["lossless"] == 1
    rows = sample_rows(w.M, w.seed, n=16)
    rlo, rhi = oracle.interval(A[0], A[1], B[0], B[1], rows=rows)
    assert np.array_equal(host(lo)[rows], rlo) and np.array_equal(host(hi)[rows], rhi)

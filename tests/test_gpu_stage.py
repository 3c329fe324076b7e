"""The per-prime tensor-core stage alone (res_gemm_stage) on chosen residues.

The expected value is the definition: (RA[p] @ RB[p]) mod q_p, formed exactly
with float64 BLAS (integer entries of at most 125 in magnitude and K <= 2^17
keep every partial sum an integer below 2^31).  The adversarial cases drive
every exact fp32 chunk of the kernel to its bound (1024 products of 125^2)
and the int32 bound of the pages' INT8 engine (125^2 * 2^17 = 2.048e9).
"""
import numpy as np
import pytest
import torch

from tests.gpu_util import host, rg, variant  # noqa: F401

pytestmark = pytest.mark.gpu


def expected(ra, rb, ps):
    out = []
    for p, q in enumerate(ps):
        prod = ra[p].astype(np.float64) @ rb[p].astype(np.float64)
        out.append(np.mod(prod.astype(np.int64), q))
    return np.stack(out)


def run_stage(rg, ra, rb, M, N, K, transb=False):
    """rb is [P, K, N]; with transb it is handed to the kernel as [P, N, K]."""
    P = ra.shape[0]
    lda = (K + 7) // 8 * 8
    RA = torch.zeros((P, M, lda), dtype=torch.float16)
    RA[:, :, :K] = torch.from_numpy(ra.astype(np.float16))
    if transb:
        RB = torch.zeros((P, N, lda), dtype=torch.float16)
        RB[:, :, :K] = torch.from_numpy(np.ascontiguousarray(np.swapaxes(rb, 1, 2)).astype(np.float16))
    else:
        RB = torch.zeros((P, K, (N + 63) // 64 * 64), dtype=torch.float16)
        RB[:, :, :N] = torch.from_numpy(rb.astype(np.float16))
    RC = rg.res_gemm_stage(RA.cuda(), RB.cuda(), P, M, N, K, transb=transb)
    return host(RC)[:, :, :N].astype(np.int64)


def patterns(kind, P, M, N, K, rng):
    if kind == "all_plus":
        return np.full((P, M, K), 125), np.full((P, K, N), 125)
    if kind == "all_minus_plus":
        return np.full((P, M, K), -125), np.full((P, K, N), 125)
    if kind == "signs":  # long runs of equal signs with odd partial sums
        s = np.where((np.arange(K) // 700) % 2 == 0, 125, -125)
        ra = np.broadcast_to(s, (P, M, K))
        rb = np.full((P, K, N), 125)
        rb[:, :, 1::2] = 123
        return ra, rb
    if kind == "random_extreme":
        return rng.choice([-125, 125], size=(P, M, K)), rng.choice([-125, 125], size=(P, K, N))
    return rng.integers(-125, 126, size=(P, M, K)), rng.integers(-125, 126, size=(P, K, N))


@pytest.mark.parametrize("kind", ["all_plus", "all_minus_plus", "signs", "random_extreme", "random"])
def test_long_k_adversarial(rg, variant, kind):
    P, M, N, K = 3, 130, 260, 2**17
    rng = np.random.default_rng(1)
    ra, rb = patterns(kind, P, M, N, K, rng)
    got = run_stage(rg, ra, rb, M, N, K)
    assert np.array_equal(got, expected(ra, rb, rg.primes()[:P]))


def test_long_k_unreduced_residues_all_primes(rg, variant):
    """Residues of +-125 for every prime, the smallest (q = 3) included: each
    chunk of 1024 products reaches +-1.6e7, the largest sums the accumulator
    sees, and their quotients by 3 are the largest the reductions see."""
    P, M, N, K = 53, 40, 70, 2**17
    ra = np.full((P, M, K), -125, dtype=np.int8)
    ra[:, 1::2, :] = 125
    rb = np.full((P, K, N), 125, dtype=np.int8)
    rb[:, :, 2::3] = -125
    rb[:, K // 2:, 1::2] = 123
    got = run_stage(rg, ra, rb, M, N, K)
    assert np.array_equal(got, expected(ra, rb, rg.primes()))


@pytest.mark.parametrize("K", [1, 16, 63, 64, 1000, 1024, 1025, 2048, 3000, 5000])
def test_k_tails_all_primes(rg, variant, K):
    P, M, N = 53, 129, 257
    rng = np.random.default_rng(K)
    ra, rb = patterns("random_extreme", P, M, N, K, rng)
    got = run_stage(rg, ra, rb, M, N, K)
    assert np.array_equal(got, expected(ra, rb, rg.primes()))


@pytest.mark.parametrize("kind", ["signs", "random_extreme"])
@pytest.mark.parametrize("M,N,K", [(129, 257, 1025), (40, 70, 2**15 + 8), (256, 512, 64)])
def test_k_major_b(rg, variant, kind, M, N, K):
    """B handed over K-major ([P, N, K]): the same residues as the N-major layout."""
    P = 5
    rng = np.random.default_rng(M + N + K)
    ra, rb = patterns(kind, P, M, N, K, rng)
    got = run_stage(rg, ra, rb, M, N, K, transb=True)
    assert np.array_equal(got, expected(ra, rb, rg.primes()[:P]))


def test_wait_expiry_returns_timeout(rg, variant):
    """A wait that can never complete expires, reports RG_ERR_TIMEOUT, and the context stays usable."""
    lib = rg.library()
    P, M, N, K = 2, 256, 256, 4096
    rng = np.random.default_rng(2)
    ra, rb = patterns("random", P, M, N, K, rng)
    old = lib.rg_set_wait_limit_ns(50_000_000)  # 50 ms
    try:
        lib.rg_inject_fault(1)  # the first accumulator is never signalled
        with pytest.raises(rg.ResGemmError) as e:
            run_stage(rg, ra, rb, M, N, K)
        assert e.value.code == rg.RG_ERR_TIMEOUT
    finally:
        lib.rg_set_wait_limit_ns(old)
    got = run_stage(rg, ra, rb, M, N, K)
    assert np.array_equal(got, expected(ra, rb, rg.primes()[:P]))

"""GPU parity of the exact int64 path (res_gemm_i64) against the CPU oracle.

Bit-exact comparison, element by element: in full on the small and 1024^3
workloads, the long-K workload and the 4096^3 workload (planned and all 53
primes), and on ragged shapes that span several tiles and a tail, plus closed
forms.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import balanced_mod, dev, host, rg, stage_buffers  # noqa: F401
from workloads import WORKLOADS, int_matrices

pytestmark = pytest.mark.gpu


def test_exact24_64_full(rg):
    w = WORKLOADS["exact24_64"]
    A, B = w.generate()
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    ref = oracle.matmul_i64(A, B, lc=1)[:, :, 0]
    assert np.array_equal(C, ref)
    plan = rg.get_plan()
    assert plan["status"] == 0 and plan["nprimes"] == 7  # |C| < 2^(24+24+6): 7 primes


def test_exact24_64_stages(rg):
    """Each stage against its definition: x mod q for the split, (A B) mod q for the GEMM stage."""
    w = WORKLOADS["exact24_64"]
    A, B = w.generate()
    rg.res_gemm_i64(dev(A), dev(B))
    ra, rb, rc, L = stage_buffers(rg, rg.RG_OP_I64, w.M, w.N, w.K)
    P = rg.get_plan()["nprimes"]
    ps = rg.primes()
    C = oracle.matmul_i64(A, B, lc=1)[:, :, 0]
    ra, rb, rc = host(ra.float()).astype(np.int64), host(rb.float()).astype(np.int64), host(rc).astype(np.int64)
    for p in range(P):
        q = ps[p]
        assert np.array_equal(ra[p, :, :w.K], balanced_mod(A, q)), p
        assert np.array_equal(rb[p, :, :w.N], balanced_mod(B, q)), p
        assert np.array_equal(rc[p, :, :w.N], np.mod(C, q)), p
        assert not ra[p, :, w.K:].any() and not rb[p, :, w.N:].any()


def test_exact24_1024_full(rg):
    w = WORKLOADS["exact24_1024"]
    A, B = w.generate()
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    ref = oracle.matmul_i64(A, B, lc=1)[:, :, 0]
    assert np.array_equal(C, ref)
    assert rg.get_plan()["nprimes"] == 8


RAGGED = [
    (1, 1, 1, -(2**23), 2**23),
    (3, 5, 7, -(2**29), 2**29),
    (65, 77, 129, -(2**23), 2**23),
    (127, 129, 1025, -(2**23), 2**23),  # two K chunks
    (130, 300, 2049, -(2**20), 2**20),  # three chunks, ragged M and N tiles
    (257, 513, 4100, -(2**12), 2**12),  # five chunks
    (200, 64, 30, -(2**29), 2**29),  # K * 2^58 < 2^63
    (40, 700, 33, -(2**28), 2**28),
]


@pytest.mark.parametrize("M,N,K,lo,hi", RAGGED)
def test_ragged_shapes(rg, M, N, K, lo, hi):
    A, B = int_matrices(M, N, K, lo, hi, seed=M * 7 + N * 3 + K)
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    assert np.array_equal(C, oracle.matmul_i64(A, B, lc=1)[:, :, 0])


def test_extreme_values(rg):
    # K * max|A| * max|B| <= 2^63 - 1 is the only limit: int64 extremes with K = 1.
    A = np.array([[2**62], [-(2**62)], [-(2**63) + 1], [2**63 - 1]], dtype=np.int64)
    B = np.array([[1, -1, 0]], dtype=np.int64)
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    assert np.array_equal(C, oracle.matmul_i64(A, B, lc=1)[:, :, 0])
    # INT64_MIN against zero
    A = np.full((3, 2), -(2**63), dtype=np.int64)
    B = np.zeros((2, 4), dtype=np.int64)
    assert not host(rg.res_gemm_i64(dev(A), dev(B))).any()


def test_range_error(rg):
    A = np.full((2, 4), 2**40, dtype=np.int64)
    B = np.full((4, 2), 2**40, dtype=np.int64)
    with pytest.raises(rg.ResGemmError) as e:
        rg.res_gemm_i64(dev(A), dev(B))
    assert e.value.code == rg.RG_ERR_RANGE
    # the context stays usable
    A, B = int_matrices(8, 8, 8, -100, 100, 1)
    assert np.array_equal(host(rg.res_gemm_i64(dev(A), dev(B))), A @ B)


@pytest.mark.parametrize("nprimes", [8, 9, 20, 53])
def test_fixed_prime_count(rg, nprimes):
    # CRT uniqueness: any prime count covering the bound gives the same integers.
    A, B = int_matrices(100, 90, 300, -(2**23), 2**23, 17)
    C = host(rg.res_gemm_i64(dev(A), dev(B), nprimes=nprimes))
    assert np.array_equal(C, A @ B)


def test_longk_int8_full(rg):
    # K = 2^17, the longest exact sum ("enclosure-gemm", Requirements and limits)
    w = WORKLOADS["longk_int8"]
    A, B = w.generate()
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    ref = oracle.matmul_i64(A, B, lc=1)[:, :, 0]
    assert np.array_equal(C, ref)
    assert rg.get_plan()["nprimes"] == 5


@pytest.fixture(scope="module")
def exact24_4096():
    """The 4096^3 workload and its oracle product (computed once for the module)."""
    w = WORKLOADS["exact24_4096"]
    A, B = w.generate()
    return A, B, oracle.matmul_i64(A, B, lc=1)[:, :, 0]


@pytest.mark.parametrize("nprimes,expect", [(0, 8), (53, 53)], ids=["planned", "all_53_primes"])
def test_exact24_4096_full(rg, exact24_4096, nprimes, expect):
    # the square workload the GEMM-stage throughput is quoted on, every entry,
    # with the planned prime count and with the whole prime set (CRT uniqueness:
    # the same integers)
    A, B, ref = exact24_4096
    C = rg.res_gemm_i64(dev(A), dev(B), nprimes=nprimes)
    assert rg.get_plan()["nprimes"] == expect
    assert np.array_equal(host(C), ref)


def test_longk_closed_form(rg):
    # all entries -128 at K = 2^17: every entry is exactly 2^31.
    K = 2**17
    A = torch.full((130, K), -128, dtype=torch.int64, device="cuda")
    B = torch.full((K, 70), -128, dtype=torch.int64, device="cuda")
    C = rg.res_gemm_i64(A, B)
    assert bool((C == 2**31).all())


def test_host_buffers(rg):
    A, B = int_matrices(70, 50, 90, -(2**23), 2**23, 5)
    C = rg.res_gemm_i64(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory())
    assert C.device.type == "cpu"
    assert np.array_equal(C.numpy(), A @ B)


def test_async_call_then_status(rg):
    A, B = int_matrices(64, 64, 64, -(2**23), 2**23, 6)
    C = rg.res_gemm_i64(dev(A), dev(B), sync=False)
    assert rg.status() == rg.RG_OK
    assert np.array_equal(host(C), A @ B)


def test_repeatable(rg):
    A, B = int_matrices(300, 200, 1500, -(2**23), 2**23, 8)
    C1 = host(rg.res_gemm_i64(dev(A), dev(B)))
    C2 = host(rg.res_gemm_i64(dev(A), dev(B)))
    assert np.array_equal(C1, C2)


@pytest.mark.parametrize("bits", [1, 4, 8, 12, 16, 20, 24, 28, 31])
def test_every_small_prime_count(rg, bits):
    # value ranges that make the planner pick 1, 2, ..., 9 primes
    # K = 1 keeps K * max|A| * max|B| < 2^62 for 31-bit entries
    A, B = int_matrices(300, 700, 1, -(2**bits) + 1, 2**bits, bits)
    C = host(rg.res_gemm_i64(dev(A), dev(B)))
    assert np.array_equal(C, A @ B)
    T = 2 * bits
    P = rg.get_plan()["nprimes"]
    assert 1 <= P <= 9 and P == next(n for n in range(1, 54) if _log2_prod(rg, n) >= T + 1)


def _log2_prod(rg, n):
    prod = 1
    for q in rg.primes()[:n]:
        prod *= q
    return prod.bit_length() - 1


def test_stage_events_time_a_real_call(rg):
    """The stage-event hook records four ordered events inside a call and leaves its result unchanged."""
    w = WORKLOADS["exact24_64"]
    A, B = w.generate()
    ref = oracle.matmul_i64(A, B, lc=1)[:, :, 0]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    rg.set_stage_events(evs)
    try:
        C = host(rg.res_gemm_i64(dev(A), dev(B)))
    finally:
        rg.set_stage_events(None)
    torch.cuda.synchronize()
    assert np.array_equal(C, ref)
    spans = [evs[i].elapsed_time(evs[i + 1]) for i in range(3)]
    assert all(t > 0 for t in spans), spans
    # with the hook removed the events are not recorded again
    rg.res_gemm_i64(dev(A), dev(B))
    torch.cuda.synchronize()
    assert [evs[i].elapsed_time(evs[i + 1]) for i in range(3)] == spans


def test_out_tensor_is_checked_and_written(rg):
    A, B = int_matrices(33, 20, 17, -1000, 1000, 5)
    dA, dB = dev(A), dev(B)
    out = torch.full((33, 20), 7, dtype=torch.int64, device="cuda")
    C = rg.res_gemm_i64(dA, dB, out=out)
    assert C.data_ptr() == out.data_ptr() and np.array_equal(host(out), A @ B)
    for bad in (torch.empty((33, 21), dtype=torch.int64, device="cuda"),
                torch.empty((33, 20), dtype=torch.int32, device="cuda"),
                torch.empty((20, 33), dtype=torch.int64, device="cuda").t(),
                torch.empty((33, 20), dtype=torch.int64)):
        with pytest.raises(ValueError):
            rg.res_gemm_i64(dA, dB, out=bad)
    lo = torch.empty((33, 20), dtype=torch.float64, device="cuda")
    hi = torch.empty_like(lo)
    Af, Bf = A.astype(np.float64), B.astype(np.float64)
    rlo, rhi = rg.enclose_gemm_f64(dev(Af), dev(Bf), out=(lo, hi))
    assert rlo.data_ptr() == lo.data_ptr() and np.array_equal(host(lo), Af @ Bf) and np.array_equal(host(hi), Af @ Bf)
    with pytest.raises(ValueError):
        rg.enclose_gemm_f64(dev(Af), dev(Bf), out=(lo,))


@pytest.mark.parametrize("pin_in,pin_out", [(True, True), (False, True), (True, False), (False, False)])
def test_host_buffers_pinned_or_pageable(rg, pin_in, pin_out):
    """Pinned host buffers are used in place (int64 operands, every output), pageable ones are
    staged; all four mixes give the exact product, as does the enclosure (operands always staged)."""
    A, B = int_matrices(130, 70, 300, -(2**23), 2**23, 23)
    hA, hB = torch.from_numpy(A), torch.from_numpy(B)
    if pin_in:
        hA, hB = hA.pin_memory(), hB.pin_memory()
    out = torch.empty((130, 70), dtype=torch.int64)
    if pin_out:
        out = out.pin_memory()
    C = rg.res_gemm_i64(hA, hB, out=out)
    assert C.data_ptr() == out.data_ptr() and np.array_equal(C.numpy(), A @ B)
    Af, Bf = (A >> 8).astype(np.float64), (B >> 8).astype(np.float64)
    fA, fB = torch.from_numpy(Af), torch.from_numpy(Bf)
    if pin_in:
        fA, fB = fA.pin_memory(), fB.pin_memory()
    lo, hi = torch.empty((130, 70), dtype=torch.float64), torch.empty((130, 70), dtype=torch.float64)
    if pin_out:
        lo, hi = lo.pin_memory(), hi.pin_memory()
    rlo, rhi = rg.enclose_gemm_f64(fA, fB, out=(lo, hi))
    ref = Af @ Bf  # products of 15-bit integers summed over 300 terms: exact in float64
    assert np.array_equal(rlo.numpy(), ref) and np.array_equal(rhi.numpy(), ref)


_CONCURRENT = r"""
import sys, threading
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import exact_modular_int8_gb300 as rg
import oracle
from workloads import int_matrices
cases = [int_matrices(150 + 40 * i, 130 + 30 * i, 300, -(2**22), 2**22, 40 + i) for i in range(4)]
out, err = [None] * 4, []
start = threading.Barrier(4)
def run(i):
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            A, B = (torch.from_numpy(x).cuda() for x in cases[i])
            start.wait()
            out[i] = rg.res_gemm_i64(A, B).cpu().numpy()
    except Exception as e:  # reported below
        err.append(repr(e))
ts = [threading.Thread(target=run, args=(i,)) for i in range(4)]
for t in ts: t.start()
for t in ts: t.join()
assert not err, err
for i, (A, B) in enumerate(cases):
    assert np.array_equal(out[i], oracle.matmul_i64(A, B, lc=1)[:, :, 0]), i
print("concurrent ok")
"""


def test_concurrent_first_calls_from_host_threads(rg):
    """Four host threads make their first calls at once, each on its own stream (so its own
    workspace), in a fresh process: the per-device setup is taken once, and every product is exact."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CONCURRENT, root], capture_output=True, text=True, timeout=600,
                       cwd=root)
    assert r.returncode == 0 and "concurrent ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


def test_plane_count_hint_and_fixup(rg):
    """Large planner-free int64 calls write as many residue planes as the previous call on the same
    workspace used (a tagged word in the plan block), and a fix-up pass adds the planes a call needs
    beyond them; so every sequence of calls stays exact, whatever the word holds."""
    M = N = K = 2048  # (M + N) K fp16 residues: 16 MiB per plane, the size from which the count is reused
    A24, B24 = int_matrices(M, N, K, -(2**23), 2**23, 31)
    A8, B8 = int_matrices(M, N, K, -128, 128, 32)
    ref24 = oracle.matmul_i64(A24, B24, lc=1)[:, :, 0]
    ref8 = oracle.matmul_i64(A8, B8, lc=1)[:, :, 0]
    ws = torch.empty(rg.workspace_bytes(rg.RG_OP_I64, M, N, K), dtype=torch.uint8, device="cuda")
    word = ws[256:260].view(torch.int32)
    tag = 0x52470000
    # a word claiming one plane: the split writes one, the fix-up the other seven
    word.fill_(tag | 1)
    C = host(rg.res_gemm_i64(dev(A24), dev(B24), ws=ws))
    assert np.array_equal(C, ref24)
    assert rg.get_plan(ws=ws)["nprimes"] == 8 and int(word.item()) == tag | 8
    # fewer primes next: the split writes 8 planes, of which the call uses 4
    C = host(rg.res_gemm_i64(dev(A8), dev(B8), ws=ws))
    assert np.array_equal(C, ref8)
    P8 = rg.get_plan(ws=ws)["nprimes"]
    assert P8 < 8 and int(word.item()) == tag | P8
    # more primes again: the fix-up adds planes P8..7
    C = host(rg.res_gemm_i64(dev(A24), dev(B24), ws=ws))
    assert np.array_equal(C, ref24) and int(word.item()) == tag | 8
    # a garbage word is ignored (all nine planes), and so is a count outside 1..8
    for w in (0x12345678, tag | 0, tag | 9, tag | 40):
        word.fill_(w)
        C = host(rg.res_gemm_i64(dev(A24), dev(B24), ws=ws))
        assert np.array_equal(C, ref24)
    # a caller-fixed prime count neither reads nor writes the word
    word.fill_(tag | 2)
    C = host(rg.res_gemm_i64(dev(A8), dev(B8), nprimes=6, ws=ws))
    assert np.array_equal(C, ref8) and int(word.item()) == tag | 2

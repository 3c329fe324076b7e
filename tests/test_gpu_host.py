"""Host-buffer calls of several MB: ragged row counts, pinned and pageable
buffers, a batch, limbs, the enclosure and the interval product.  Every result
equals the same call on device buffers, and rows sampled across each quarter
of the output equal the oracle."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import dev, host, rg  # noqa: F401
from workloads import int_matrices, interval_matrices, limb_matrices, normal_matrices

pytestmark = pytest.mark.gpu


def spread_rows(rows):
    """Rows at both ends of each quarter of the output, plus a few inside."""
    c = (rows + 3) // 4
    picks = {0, 1, rows - 1}
    for i in range(1, 4):
        picks |= {i * c - 1, i * c, min(rows - 1, i * c + 1)}
    return np.array(sorted(r for r in picks if 0 <= r < rows), dtype=np.int64)


def pinned(x, pin):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.pin_memory() if pin else t


@pytest.mark.parametrize("pin_in,pin_out", [(True, True), (False, False), (True, False)])
def test_int64_ragged_rows(rg, pin_in, pin_out):
    M, N, K = 1027, 1024, 300  # 8.4 MB of int64 results
    A, B = int_matrices(M, N, K, -(2**23), 2**23, 61)
    out = torch.empty((M, N), dtype=torch.int64)
    if pin_out:
        out = out.pin_memory()
    C = rg.res_gemm_i64(pinned(A, pin_in), pinned(B, pin_in), out=out)
    assert C.data_ptr() == out.data_ptr()
    assert np.array_equal(C.numpy(), host(rg.res_gemm_i64(dev(A), dev(B))))
    rows = spread_rows(M)
    assert np.array_equal(C.numpy()[rows], oracle.matmul_i64(A, B, lc=1, rows=rows)[:, :, 0])


def test_int64_batched(rg):
    b, M, N, K = 3, 401, 1024, 128  # 1203 rows of 3 products
    A = np.stack([int_matrices(M, N, K, -(2**20), 2**20, 70 + i)[0] for i in range(b)])
    B = np.stack([int_matrices(M, N, K, -(2**20), 2**20, 70 + i)[1] for i in range(b)])
    C = rg.res_gemm_i64(pinned(A, True), pinned(B, True))
    assert np.array_equal(C.numpy(), host(rg.res_gemm_i64(dev(A), dev(B))))
    for i in range(b):
        rows = spread_rows(M)
        assert np.array_equal(C.numpy()[i][rows], oracle.matmul_i64(A[i], B[i], lc=1, rows=rows)[:, :, 0])


def test_limbs(rg):
    M, N, K = 1100, 512, 64  # 6-limb results: 27 MB
    A, B = limb_matrices(M, N, K, 2, 62)
    C = rg.res_gemm_limbs(pinned(A, True), pinned(B, True), 6)
    assert np.array_equal(C.numpy(), host(rg.res_gemm_limbs(dev(A), dev(B), 6)))
    rows = spread_rows(M)
    assert np.array_equal(C.numpy()[rows], oracle.matmul_limbs(A, B, 6, rows=rows))


@pytest.mark.parametrize("pin", [True, False])
def test_enclosure(rg, pin):
    M, N, K = 1030, 1024, 200
    A, B = normal_matrices(M, N, K, 63)
    lo, hi = rg.enclose_gemm(pinned(A, pin), pinned(B, pin))
    dlo, dhi = rg.enclose_gemm(dev(A), dev(B))
    assert np.array_equal(lo.numpy().view(np.uint64), host(dlo).view(np.uint64))
    assert np.array_equal(hi.numpy().view(np.uint64), host(dhi).view(np.uint64))
    rows = spread_rows(M)
    rlo, rhi = oracle.enclose_f64(A, B, rows=rows)
    assert np.array_equal(lo.numpy()[rows].view(np.uint64), rlo.view(np.uint64))
    assert np.array_equal(hi.numpy()[rows].view(np.uint64), rhi.view(np.uint64))


def test_interval(rg):
    M, N, K = 1025, 1024, 96
    A, B = interval_matrices(M, N, K, 64)
    lo, hi = rg.interval_gemm(*(pinned(x, True) for x in (A[0], A[1], B[0], B[1])))
    dlo, dhi = rg.interval_gemm(dev(A[0]), dev(A[1]), dev(B[0]), dev(B[1]))
    assert np.array_equal(lo.numpy().view(np.uint64), host(dlo).view(np.uint64))
    assert np.array_equal(hi.numpy().view(np.uint64), host(dhi).view(np.uint64))
    rows = spread_rows(M)
    rlo, rhi = oracle.interval(A[0], A[1], B[0], B[1], rows=rows)
    assert np.array_equal(lo.numpy()[rows].view(np.uint64), rlo.view(np.uint64))
    assert np.array_equal(hi.numpy()[rows].view(np.uint64), rhi.view(np.uint64))


@pytest.fixture(scope="module")
def pipelined_case():
    """2500 x 1000 x 3000 int64 (104 MB of operands and result): A goes over the link in two row
    blocks of 1280 and 1220 rows.  The first block's entries are small and the second's full
    24-bit, so the two blocks plan different prime counts (7 and 8)."""
    M, N, K = 2500, 1000, 3000
    A, B = int_matrices(M, N, K, -(2**23), 2**23, 63)
    A[:1280] //= 2**13
    return A, B, oracle.matmul_i64(A, B, lc=1)[:, :, 0]


@pytest.mark.parametrize("pin,transb", [(True, False), (False, False), (True, True)])
def test_int64_pipelined_row_blocks(rg, pipelined_case, pin, transb):
    A, B, ref = pipelined_case
    Bx = np.ascontiguousarray(B.T) if transb else B
    out = torch.empty(ref.shape, dtype=torch.int64)
    if pin:
        out = out.pin_memory()
    for _ in range(2):  # twice: the copy streams and events are reused
        out.fill_(-1)
        C = rg.res_gemm_i64(pinned(A, pin), pinned(Bx, pin), out=out, transb=transb)
        assert np.array_equal(C.numpy(), ref)
    assert rg.get_plan()["nprimes"] == 8


def test_int64_pipelined_four_blocks_ragged(rg):
    # 4100 rows: blocks of 1280, 1280, 1280 and 260 rows (36 MB)
    M, N, K = 4100, 512, 512
    A, B = int_matrices(M, N, K, -(2**23), 2**23, 64)
    C = rg.res_gemm_i64(pinned(A, True), pinned(B, True))
    assert np.array_equal(C.numpy(), host(rg.res_gemm_i64(dev(A), dev(B))))
    rows = spread_rows(M)
    assert np.array_equal(C.numpy()[rows], oracle.matmul_i64(A, B, lc=1, rows=rows)[:, :, 0])

"""The allocation-free entry point res_gemm_i64_noalloc, called through the C ABI.

It serves callers that cannot allocate device memory when they call (a host
framework that owns all device memory, a latency-critical path where
cudaMalloc's implicit synchronisation is not allowed).  Its scratch is a fixed
static device array inside the library, so two calls in a row must each give
exactly what res_gemm_i64 gives (integer results: bit-exact), whatever the
previous call left in that array.  This file is collected last on purpose.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from workloads import int_matrices

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _noalloc(lib):
    f = lib.res_gemm_i64_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int, ctypes.c_uint, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


@pytest.fixture(scope="module")
def rg():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from exact_modular_int8_gb300 import build as b

    b.build()
    import exact_modular_int8_gb300 as rg

    return rg


def test_noalloc_matches_res_gemm_i64_on_two_calls(rg):
    lib = rg.library()
    f = _noalloc(lib)
    lib.rg_noalloc_scratch_bytes.restype = ctypes.c_size_t
    cap = lib.rg_noalloc_scratch_bytes()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(1000, 1000, 1000, -(2**23), 2**23, 11), (700, 900, 1500, -(2**20), 2**20, 12)]
    for M, N, K, lo, hi, seed in cases:  # two calls in a row on the shared scratch
        assert rg.workspace_bytes(rg.RG_OP_I64, M, N, K) <= cap
        A, B = int_matrices(M, N, K, lo, hi, seed)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        want = rg.res_gemm_i64(dA, dB)
        C = torch.full((M, N), -1, dtype=torch.int64, device="cuda")
        rc = f(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, 0, rg.RG_FLAG_SYNC, stream)
        assert rc == rg.RG_OK, rg.strerror(rc)
        assert torch.equal(C, want)
        assert np.array_equal(C.cpu().numpy(), A @ B)
    # beyond the fixed scratch: a clear error before any device work
    M = N = K = 2048
    assert rg.workspace_bytes(rg.RG_OP_I64, M, N, K) > cap
    dummy = torch.zeros(1, dtype=torch.int64, device="cuda")
    rc = f(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), M, N, K, 0, rg.RG_FLAG_SYNC, stream)
    assert rc == rg.RG_ERR_WORKSPACE
    # K beyond the exact int32-class accumulator bound: the status res_gemm_i64 gives
    rc = f(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), 1, 1, 2**17 + 1, 0, rg.RG_FLAG_SYNC, stream)
    assert rc == rg.RG_ERR_RANGE


_FIRST_CALL = r"""
import ctypes, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from workloads import int_matrices
A, B = int_matrices(300, 200, 500, -(2**23), 2**23, 21)
dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
C = torch.full((300, 200), -1, dtype=torch.int64, device="cuda")
torch.cuda.synchronize()
lib = ctypes.CDLL(sys.argv[2])
f = lib.res_gemm_i64_noalloc
f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
              ctypes.c_int, ctypes.c_uint, ctypes.c_void_p]
f.restype = ctypes.c_int
s = torch.cuda.current_stream().cuda_stream
for _ in range(2):  # the library's first call in this process, then a second one
    rc = f(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), 300, 200, 500, 0, 1, s)
    if rc != 0:
        sys.exit(10 + rc)
    np.save(sys.argv[3], C.cpu().numpy())
"""


def test_noalloc_as_the_first_library_call_of_a_process(rg, tmp_path):
    # a fresh process whose first call into the library is a synchronising
    # res_gemm_i64_noalloc: its status read must not need any per-thread
    # state that another entry point would have set up
    out = tmp_path / "C.npy"
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL, ROOT, rg.LIB_PATH, str(out)], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    A, B = int_matrices(300, 200, 500, -(2**23), 2**23, 21)
    ref = oracle.matmul_i64(A, B, lc=1)[:, :, 0]
    assert np.array_equal(np.load(out), ref)


def test_noalloc_binding_copies_strided_operands_and_checks_out(rg):
    A, B = int_matrices(257, 257, 257, -(2**23), 2**23, 22)
    dA = torch.from_numpy(np.ascontiguousarray(A.T)).cuda().T  # strided views of A and B
    dB = torch.from_numpy(np.ascontiguousarray(B.T)).cuda().T
    assert not dA.is_contiguous() and not dB.is_contiguous()
    ref = oracle.matmul_i64(A, B, lc=1)[:, :, 0]
    for _ in range(2):
        C = rg.res_gemm_i64_noalloc(dA, dB)
        assert np.array_equal(C.cpu().numpy(), ref)
    out = torch.empty((257, 257), dtype=torch.int64, device="cuda")
    assert rg.res_gemm_i64_noalloc(dA, dB, out=out) is out
    assert np.array_equal(out.cpu().numpy(), ref)
    for bad in (torch.empty((257, 256), dtype=torch.int64, device="cuda"),
                torch.empty((257, 257), dtype=torch.int32, device="cuda"),
                torch.empty((257, 514), dtype=torch.int64, device="cuda")[:, ::2]):
        with pytest.raises(ValueError):
            rg.res_gemm_i64_noalloc(dA, dB, out=bad)

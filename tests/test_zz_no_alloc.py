"""The allocation-free entry point res_gemm_i64_noalloc, called through the C ABI.

It serves callers that cannot allocate device memory when they call (a host
framework that owns all device memory, a latency-critical path where
cudaMalloc's implicit synchronisation is not allowed).  Its scratch is a fixed
static device array inside the library, so two calls in a row must each give
exactly what res_gemm_i64 gives (integer results: bit-exact), whatever the
previous call left in that array.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import int_matrices

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.res_gemm_i64_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int, ctypes.c_uint, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def test_noalloc_matches_res_gemm_i64_on_two_calls():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from exact_modular_int8_gb300 import build as b

    b.build()
    import exact_modular_int8_gb300 as rg

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

"""Shared helpers for the GPU parity tests (no method arithmetic here)."""
import numpy as np
import pytest
import torch


def library():
    """Build (if needed) and import the binding; a GPU test without a GPU fails."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from exact_modular_int8_gb300 import build as b

    b.build()
    import exact_modular_int8_gb300 as rg

    return rg


@pytest.fixture(scope="module")
def rg():
    return library()


@pytest.fixture(params=[1, 2], ids=["single_cta", "cta_pair"])
def variant(rg, request):
    """Runs the test on the single-CTA and on the CTA-pair tensor-core kernel."""
    lib = rg.library()
    old = lib.rg_set_gemm_variant(request.param)
    yield request.param
    lib.rg_set_gemm_variant(old)


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def balanced_mod(x, q):
    """Balanced residue in [-(q-1)/2, (q-1)/2] of an int64 numpy array (numpy %)."""
    r = np.mod(x, q)
    return np.where(r > (q - 1) // 2, r - q, r)


def stage_buffers(rg, op, M, N, K, la=1, lb=1, lc=1, nprimes=0):
    """Views of the residue planes the last call left in the cached workspace."""
    L = rg.workspace_layout(op, M, N, K, la, lb, lc, nprimes)
    ws = rg.workspace(rg.workspace_bytes(op, M, N, K, la, lb, lc, nprimes), torch.device("cuda", 0))
    P = L.pmax
    ra = ws[L.ra:L.ra + P * M * L.lda * 2].view(torch.float16).view(P, M, L.lda)
    rb = ws[L.rb:L.rb + P * K * L.ldb * 2].view(torch.float16).view(P, K, L.ldb)
    rc = ws[L.rc:L.rc + P * M * L.ldc].view(P, M, L.ldc)
    return ra, rb, rc, L

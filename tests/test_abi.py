"""The C-ABI library loads and exports what include/resgemm.h declares (no GPU).

Only entry points that return before touching the device are called here:
argument validation, workspace sizing and the prime table.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "resgemm.h")


@pytest.fixture(scope="module")
def rg():
    from exact_modular_int8_gb300 import build as b
    b.build()
    import exact_modular_int8_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in {"if", "while", "for", "return", "sizeof"}))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for f in ("res_gemm_i64", "res_gemm_limbs", "enclose_gemm_f64"):
        assert f in names


def test_every_declared_symbol_is_exported(rg):
    lib = ctypes.CDLL(rg.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(rg.EXPORTED) == set(declared_functions())


def _is_prime(n):
    return n > 1 and all(n % d for d in range(2, int(n**0.5) + 1))


def test_prime_base(rg):
    ps = rg.primes()
    assert ps == sorted([p for p in range(3, 256) if _is_prime(p)], reverse=True)
    assert len(ps) == 53 and ps[0] == 251 and ps[-1] == 3
    assert rg.library().rg_prime(53) == 0 and rg.library().rg_prime(-1) == 0
    # The pages' gate bits_a + bits_b + ceil(log2 K) <= 332 is floor(log2((P-1)/2))
    # for the product P of these primes.
    P = 1
    for p in ps:
        P *= p
    assert ((P - 1) // 2).bit_length() - 1 == 332


def test_strerror(rg):
    assert rg.strerror(0) == "ok"
    for code in range(1, 8):
        assert rg.strerror(code) != "unknown status"
    assert rg.strerror(99) == "unknown status"


def test_workspace_sizes(rg):
    # i64 plans for at most 9 primes; planes of fp16 A and B residues and uint8 C residues.
    L = rg.workspace_layout(rg.RG_OP_I64, 64, 64, 64)
    assert L.pmax == 9 and L.lda == 64 and L.ldb == 64 and L.ldc == 64
    n = rg.workspace_bytes(rg.RG_OP_I64, 64, 64, 64)
    assert n >= 4096 + 9 * (64 * 64 * 2 * 2 + 64 * 64)
    assert rg.workspace_bytes(rg.RG_OP_I64, 64, 64, 64, nprimes=7) < n
    L = rg.workspace_layout(rg.RG_OP_I64, 65, 77, 129)
    assert (L.lda, L.ldb, L.ldc) == (136, 128, 80)
    assert L.ra % 4096 == 0 and L.rb % 4096 == 0 and L.rc % 4096 == 0
    assert rg.workspace_layout(rg.RG_OP_ENCLOSE, 8, 8, 8).pmax == 53
    assert rg.workspace_bytes(rg.RG_OP_I64, 64, 64, 64, host=True) > n
    assert rg.workspace_bytes(rg.RG_OP_I64, -1, 64, 64) == 0
    assert rg.workspace_bytes(rg.RG_OP_I64, 0, 64, 64) == 4096  # an empty problem: the plan block only
    assert rg.workspace_bytes(rg.RG_OP_ENCLOSE, 8, 8, 0) == 4096
    assert rg.workspace_bytes(rg.RG_OP_I64, 8, 8, 8, batch=0) == 4096
    assert rg.workspace_bytes(rg.RG_OP_I64, 8, 8, 8, batch=-1) == 0
    # a batch scales every plane: [pmax][batch][rows][ld]
    one, five = (rg.workspace_layout(rg.RG_OP_I64, 65, 77, 129, batch=b) for b in (1, 5))
    assert (five.lda, five.ldb, five.ldc, five.pmax) == (one.lda, one.ldb, one.ldc, one.pmax)
    assert five.rb - five.ra >= 5 * 9 * 65 * 136 * 2 and five.rc - five.rb >= 5 * 9 * 129 * 128 * 2
    assert rg.workspace_bytes(rg.RG_OP_I64, 65, 77, 129, batch=5) > 4 * rg.workspace_bytes(rg.RG_OP_I64, 65, 77, 129)
    Lt = rg.workspace_layout(rg.RG_OP_I64, 65, 77, 129, transb=True)
    assert Lt.ldb == 136 and Lt.rc - Lt.rb >= 9 * 77 * 136 * 2
    assert rg.workspace_bytes(rg.RG_OP_LIMBS, 4, 4, 4, la=5, lb=1, lc=2) == 0
    assert rg.workspace_bytes(rg.RG_OP_LIMBS, 4, 4, 4, la=2, lb=2, lc=7) == 0


def test_layout_reports_k_slices(rg):
    """rc holds as many K slices as the GEMM may use: one for a single 1024-K chunk, one per chunk
    while the tiles alone cannot fill the GPU, at most 16."""
    assert rg.workspace_layout(rg.RG_OP_I64, 1024, 1024, 1024).splits == 1
    assert rg.workspace_layout(rg.RG_OP_ENCLOSE, 1024, 1024, 4096).splits == 4  # 16 pair tiles, 4 chunks
    assert rg.workspace_layout(rg.RG_OP_I64, 512, 512, 131072).splits == 16  # 4 pair tiles, 128 chunks
    assert rg.workspace_layout(rg.RG_OP_I64, 4096, 4096, 4096).splits == 1  # 256 pair tiles fill the GPU
    assert rg.workspace_layout(rg.RG_OP_I64, 0, 8, 8).splits == 1  # an empty problem


def test_workspace_query_refuses_shapes_the_kernels_cannot_index(rg):
    """Shapes past 32-bit rows, columns or batch, K past 2^17, or more than 2^31 - 1 GEMM tiles get 0
    (an invalid problem), never a size wrapped modulo 2^64."""
    big = 2**31 - 1
    assert rg.workspace_bytes(rg.RG_OP_I64, 2**31, 8, 8) == 0
    assert rg.workspace_bytes(rg.RG_OP_I64, 8, 2**40, 8) == 0
    assert rg.workspace_bytes(rg.RG_OP_I64, 8, 8, 2**17 + 1) == 0
    assert rg.workspace_bytes(rg.RG_OP_I64, 8, 8, 8, batch=2**31) == 0
    assert rg.workspace_bytes(rg.RG_OP_INTERVAL, big, big, 64, batch=big) == 0  # about 2^85 tiles
    assert rg.workspace_bytes(rg.RG_OP_I64, 2**22, 2**22, 8) == 0  # 9 primes x 2^15 x 2^14 tiles > 2^31
    n = rg.workspace_bytes(rg.RG_OP_I64, 2**18, 2**18, 8)  # 9 x 2048 x 1024 tiles: valid; C's 9 planes take 620 GB
    assert n > 9 * 2**36 and n < 2**40


def test_argument_errors_need_no_device(rg):
    lib = rg.library()
    buf = (ctypes.c_int64 * 16)()
    p = ctypes.addressof(buf)
    ws = (ctypes.c_uint8 * 8192)()
    wsp = (ctypes.addressof(ws) + 255) // 256 * 256
    # null operand
    assert lib.res_gemm_i64(None, p, p, 2, 2, 2, 0, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    # bad sizes
    assert lib.res_gemm_i64(p, p, p, -1, 2, 2, 0, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.res_gemm_i64(p, p, p, 2, 2, -2, 0, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.res_gemm_i64_batched(p, p, p, -1, 2, 2, 2, 0, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.enclose_gemm_f64_batched(p, p, p, None, 3, 2, 2, 2, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.res_gemm_i64(p, p, p, 2, 2, 2, 54, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    # K > 2^17
    assert lib.res_gemm_i64(p, p, p, 2, 2, 2**17 + 1, 0, 0, wsp, 4096, None) == rg.RG_ERR_RANGE
    # workspace too small
    assert lib.res_gemm_i64(p, p, p, 2, 2, 2, 0, 0, wsp, 16, None) == rg.RG_ERR_WORKSPACE
    # misaligned workspace
    assert lib.res_gemm_i64(p, p, p, 2, 2, 2, 0, 0, wsp + 8, 1 << 20, None) == rg.RG_ERR_ARG
    # limb counts
    assert lib.res_gemm_limbs(p, 5, p, 1, p, 2, 2, 2, 2, 0, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.res_gemm_limbs(p, 1, p, 1, p, 7, 2, 2, 2, 0, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    # enclosure needs both outputs
    assert lib.enclose_gemm_f64(p, p, p, None, 2, 2, 2, 0, None, wsp, 4096, None) == rg.RG_ERR_ARG
    # stage: leading dimensions and prime count
    assert lib.res_gemm_stage(p, 7, p, 64, p, 16, 1, 2, 2, 2, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.res_gemm_stage(p, 8, p, 64, p, 16, 0, 2, 2, 2, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.res_gemm_stage(p, 8, p, 32, p, 16, 1, 2, 2, 2, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.res_gemm_stage(p, 2**17 + 8, p, 64, p, 16, 1, 2, 2, 2**17 + 1, 0, wsp, 4096, None) == rg.RG_ERR_RANGE
    # shapes past the kernels' 32-bit tile numbering
    assert lib.res_gemm_stage(p, 8, p, 2**31 + 64, p, 2**31 + 16, 1, 2, 2**31, 2, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.res_gemm_stage(p, 8, p, 2**21, p, 2**21, 53, 2**21, 2**21, 2, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.res_gemm_i64(p, p, p, 2**31, 2, 2, 0, 0, wsp, 4096, None) == rg.RG_ERR_ARG
    assert lib.res_gemm_i64(p, p, p, 2**22, 2**22, 8, 0, 0, wsp, 1 << 62, None) == rg.RG_ERR_ARG
    assert lib.interval_gemm_f64_batched(p, p, p, p, p, p, 2**31 - 1, 2**31 - 1, 2**31 - 1, 64, 0, wsp, 1 << 62,
                                         None) == rg.RG_ERR_ARG


def test_stage_events_hook_arguments(rg):
    lib = rg.library()
    nulls = (ctypes.c_void_p * 4)()
    assert lib.rg_set_stage_events(None, 3) == rg.RG_ERR_ARG
    assert lib.rg_set_stage_events(None, 4) == rg.RG_ERR_ARG
    assert lib.rg_set_stage_events(nulls, 4) == rg.RG_ERR_ARG
    assert lib.rg_set_stage_events(None, 0) == rg.RG_OK


def test_wait_limit_roundtrip(rg):
    lib = rg.library()
    old = lib.rg_set_wait_limit_ns(12345)
    assert lib.rg_set_wait_limit_ns(old) == 12345


def test_crt_mode_range(rg):
    """Modes 0 (default), 1 and 2 are accepted and return the previous mode; others are refused."""
    lib = rg.library()
    old = lib.rg_set_crt_mode(1)
    assert old in (0, 1)
    assert lib.rg_set_crt_mode(0) == 1
    assert lib.rg_set_crt_mode(2) == 0 and lib.rg_set_crt_mode(0) == 2
    assert lib.rg_set_crt_mode(3) == -1 and lib.rg_set_crt_mode(-1) == -1
    assert lib.rg_set_crt_mode(old) == 0


def test_binding_reports_refused_shapes_like_the_entry_points(rg):
    """The binding sizes the workspace first; a refused shape raises the code the C entry point returns."""
    with pytest.raises(rg.ResGemmError) as e:
        rg._need(rg.RG_OP_I64, 8, 8, rg.MAX_K + 1, "res_gemm_i64")
    assert e.value.code == rg.RG_ERR_RANGE
    with pytest.raises(rg.ResGemmError) as e:
        rg._need(rg.RG_OP_ENCLOSE, 2**31, 8, 8, "enclose_gemm")
    assert e.value.code == rg.RG_ERR_ARG
    assert rg._need(rg.RG_OP_I64, 8, 8, rg.MAX_K, "res_gemm_i64") == rg.workspace_bytes(rg.RG_OP_I64, 8, 8, rg.MAX_K)


def test_probe_rejects_bad_arguments_before_the_device(rg):
    lib = rg.library()
    ops = ctypes.c_double(0.0)
    # no workspace, or an unknown probe kind with no workspace: refused before any CUDA call
    assert lib.rg_probe_mma_rate(rg.RG_PROBE_MMA_S8, 0, 10, None, 4096, None, ctypes.byref(ops)) == rg.RG_ERR_ARG
    assert lib.rg_probe_mma_rate(8, 0, 10, None, 4096, None, ctypes.byref(ops)) == rg.RG_ERR_ARG
    assert lib.rg_probe_mma_rate(rg.RG_PROBE_MMA_S8, 0, 10, 256, 4096, None, None) == rg.RG_ERR_ARG
    assert lib.rg_probe_mma_rate(rg.RG_PROBE_MMA_S8, 0, 10, 256, 128, None, ctypes.byref(ops)) == rg.RG_ERR_ARG

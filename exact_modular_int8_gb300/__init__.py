"""Exact matrix products through residues modulo the odd primes below 256, on GB300.

Thin Python binding of the C-ABI library ``_build/libresgemm.so`` (declared in
``include/resgemm.h``).  The functions here only marshal arguments: they take
torch tensors, allocate outputs and a cached workspace with torch, and pass raw
pointers and the current CUDA stream to the library.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU fallback, and
importing the functions fails loudly if the library has not been built
(``python -m exact_modular_int8_gb300.build`` or ``__graft_entry__.build()``).

Entry points (same names as the C ABI):
  res_gemm_i64(A, B)             exact int64 product
  res_gemm_limbs(A, B, lc)       exact multi-limb product
  enclose_gemm_f64(A, B)         (lo, hi) with lo <= A @ B <= hi exactly
  res_gemm_stage(RA, RB, ...)    the per-prime tensor-core stage alone
Helpers: width_ulps, digest, get_plan, workspace_bytes.
"""
from __future__ import annotations

import contextlib
import ctypes
import functools
import hashlib
from fractions import Fraction
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libresgemm.so")

RG_OK = 0
RG_ERR_ARG = 1
RG_ERR_RANGE = 2
RG_ERR_NONFINITE = 3
RG_ERR_LOSSY = 4
RG_ERR_WORKSPACE = 5
RG_ERR_CUDA = 6
RG_ERR_TIMEOUT = 7
RG_ERR_RADIUS = 8
RG_ERR_SINGULAR = 9
RG_FLAG_SYNC = 1
RG_FLAG_HOST = 2
RG_FLAG_TRANS_B = 4
RG_OP_I64, RG_OP_LIMBS, RG_OP_ENCLOSE, RG_OP_STAGE, RG_OP_ENCLOSE_F32 = 0, 1, 2, 3, 4
RG_OP_INTERVAL, RG_OP_INTERVAL_F32 = 5, 6
RG_PROBE_MMA_S8, RG_PROBE_TCGEN05_F16, RG_PROBE_TCGEN05_E4M3 = 0, 1, 2
RG_PROBE_TCGEN05_F16_BMN, RG_PROBE_TCGEN05_F16_PAIR, RG_PROBE_TCGEN05_F16_PAIR_BMN = 3, 4, 5
RG_PROBE_TCGEN05_F16_PAIR_BMN_SYNC, RG_PROBE_MMA_F16 = 6, 7
MAX_K = 131072
NUM_PRIMES = 53

EXPORTED = (
    "res_gemm_i64", "res_gemm_limbs", "enclose_gemm_f64", "res_gemm_stage", "rg_workspace_bytes",
    "rg_workspace_layout", "rg_get_plan", "rg_status", "rg_prime", "rg_strerror", "rg_set_wait_limit_ns",
    "rg_inject_fault", "res_gemm_i64_noalloc", "rg_noalloc_scratch_bytes", "rg_set_gemm_variant",
    "res_gemm_i64_batched", "res_gemm_limbs_batched", "enclose_gemm_f64_batched", "rg_workspace_bytes_batched",
    "rg_workspace_layout_batched", "enclose_gemm_f32", "enclose_gemm_f32_batched", "interval_gemm_f64",
    "interval_gemm_f32", "interval_gemm_f64_batched", "interval_gemm_f32_batched", "rg_solve_i64",
    "rg_solution_free", "rg_rational_reconstruct", "rg_big_gcd", "rg_set_crt_mode", "rg_set_stage_events",
    "rg_probe_mma_rate", "rg_big_mulmod",
)


class ResGemmError(RuntimeError):
    """A library call returned a non-zero status."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (status {code})")


class Layout(ctypes.Structure):
    _fields_ = [("ra", ctypes.c_size_t), ("rb", ctypes.c_size_t), ("rc", ctypes.c_size_t),
                ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64), ("pmax", ctypes.c_int),
                ("splits", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("status", ctypes.c_int), ("nprimes", ctypes.c_int), ("bits_a", ctypes.c_int),
                ("bits_b", ctypes.c_int), ("bound_bits", ctypes.c_int), ("f_a", ctypes.c_int),
                ("f_b", ctypes.c_int), ("lossless", ctypes.c_int), ("splits", ctypes.c_int), ("crt_rn", ctypes.c_int)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class Solution(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("c", ctypes.c_int64), ("limbs", ctypes.c_int64),
                ("values", ctypes.POINTER(ctypes.c_int64)), ("steps", ctypes.c_int64), ("primes", ctypes.c_int),
                ("ms_inverse", ctypes.c_double), ("ms_lift", ctypes.c_double), ("ms_reconstruct", ctypes.c_double)]


_lib = None
_lib_lock = threading.Lock()


def library():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with `python -m exact_modular_int8_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            vp, i64, ci, cu, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
            lib.res_gemm_i64.argtypes = [vp, vp, vp, i64, i64, i64, ci, cu, vp, sz, vp]
            lib.res_gemm_limbs.argtypes = [vp, ci, vp, ci, vp, ci, i64, i64, i64, ci, cu, vp, sz, vp]
            lib.enclose_gemm_f64.argtypes = [vp, vp, vp, vp, i64, i64, i64, cu, ctypes.POINTER(ci), vp, sz, vp]
            lib.res_gemm_stage.argtypes = [vp, i64, vp, i64, vp, i64, ci, i64, i64, i64, cu, vp, sz, vp]
            lib.res_gemm_i64_batched.argtypes = [vp, vp, vp, i64, i64, i64, i64, ci, cu, vp, sz, vp]
            lib.res_gemm_limbs_batched.argtypes = [vp, ci, vp, ci, vp, ci, i64, i64, i64, i64, ci, cu, vp, sz, vp]
            lib.enclose_gemm_f64_batched.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, cu, vp, sz, vp]
            lib.enclose_gemm_f32.argtypes = [vp, vp, vp, vp, i64, i64, i64, cu, vp, sz, vp]
            lib.enclose_gemm_f32_batched.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, cu, vp, sz, vp]
            for f in ("interval_gemm_f64", "interval_gemm_f32"):
                getattr(lib, f).argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, cu, vp, sz, vp]
            for f in ("interval_gemm_f64_batched", "interval_gemm_f32_batched"):
                getattr(lib, f).argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, cu, vp, sz, vp]
            for f in ("res_gemm_i64", "res_gemm_limbs", "enclose_gemm_f64", "res_gemm_stage", "res_gemm_i64_batched",
                      "res_gemm_limbs_batched", "enclose_gemm_f64_batched", "enclose_gemm_f32",
                      "enclose_gemm_f32_batched", "interval_gemm_f64", "interval_gemm_f32",
                      "interval_gemm_f64_batched", "interval_gemm_f32_batched"):
                getattr(lib, f).restype = ci
            lib.rg_workspace_bytes.argtypes = [ci, i64, i64, i64, ci, ci, ci, ci, cu]
            lib.rg_workspace_bytes.restype = sz
            lib.rg_workspace_bytes_batched.argtypes = [ci, i64, i64, i64, i64, ci, ci, ci, ci, cu]
            lib.rg_workspace_bytes_batched.restype = sz
            lib.rg_workspace_layout.argtypes = [ci, i64, i64, i64, ci, ci, ci, ci, cu, ctypes.POINTER(Layout)]
            lib.rg_workspace_layout.restype = ci
            lib.rg_workspace_layout_batched.argtypes = [ci, i64, i64, i64, i64, ci, ci, ci, ci, cu,
                                                        ctypes.POINTER(Layout)]
            lib.rg_workspace_layout_batched.restype = ci
            lib.rg_get_plan.argtypes = [vp, vp, ctypes.POINTER(PlanInfo)]
            lib.rg_get_plan.restype = ci
            lib.rg_status.argtypes = [vp, vp]
            lib.rg_status.restype = ci
            lib.rg_prime.argtypes = [ci]
            lib.rg_prime.restype = ci
            lib.rg_strerror.argtypes = [ci]
            lib.rg_strerror.restype = ctypes.c_char_p
            lib.rg_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            lib.rg_set_wait_limit_ns.restype = ctypes.c_uint64
            lib.rg_inject_fault.argtypes = [ci]
            lib.rg_inject_fault.restype = None
            lib.rg_set_gemm_variant.argtypes = [ci]
            lib.rg_set_gemm_variant.restype = ci
            lib.rg_set_crt_mode.argtypes = [ci]
            lib.rg_set_crt_mode.restype = ci
            lib.rg_solve_i64.argtypes = [vp, vp, i64, i64, cu, vp, ctypes.POINTER(Solution)]
            lib.rg_solve_i64.restype = ci
            lib.rg_solution_free.argtypes = [ctypes.POINTER(Solution)]
            lib.rg_solution_free.restype = None
            lib.rg_rational_reconstruct.argtypes = [vp, ci, vp, ci, ci, ci, vp, vp, ci]
            lib.rg_rational_reconstruct.restype = ci
            lib.rg_big_gcd.argtypes = [vp, ci, vp, ci, vp, ci]
            lib.rg_big_gcd.restype = ci
            lib.rg_big_mulmod.argtypes = [vp, ci, vp, ci, vp, ci, vp, ci]
            lib.rg_big_mulmod.restype = ci
            lib.rg_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ci]
            lib.rg_set_stage_events.restype = ci
            lib.rg_probe_mma_rate.argtypes = [ci, ci, ci, vp, sz, vp, ctypes.POINTER(ctypes.c_double)]
            lib.rg_probe_mma_rate.restype = ci
            lib.res_gemm_i64_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, ci, cu, vp]
            lib.res_gemm_i64_noalloc.restype = ci
            lib.rg_noalloc_scratch_bytes.argtypes = []
            lib.rg_noalloc_scratch_bytes.restype = sz
            _lib = lib
    return _lib


def strerror(code: int) -> str:
    return library().rg_strerror(int(code)).decode()


def primes() -> list[int]:
    """The residue base, largest first: 251, 241, ..., 3."""
    return [library().rg_prime(i) for i in range(NUM_PRIMES)]


def _layout_flags(host, transb):
    return (RG_FLAG_HOST if host else 0) | (RG_FLAG_TRANS_B if transb else 0)


@functools.lru_cache(maxsize=512)
def _ws_bytes(op, batch, M, N, K, la, lb, lc, nprimes, flags) -> int:
    return int(library().rg_workspace_bytes_batched(op, batch, M, N, K, la, lb, lc, nprimes, flags))


def workspace_bytes(op, M, N, K, la=1, lb=1, lc=1, nprimes=0, host=False, transb=False, batch=1) -> int:
    return _ws_bytes(op, batch, M, N, K, la, lb, lc, nprimes, _layout_flags(host, transb))


def _need(op, M, N, K, where, **kw) -> int:
    """The call's workspace size; a shape the library refuses raises as the C entry point would
    (RG_ERR_RANGE for K above 2^17, RG_ERR_ARG otherwise)."""
    need = workspace_bytes(op, M, N, K, **kw)
    if need == 0:
        raise ResGemmError(RG_ERR_RANGE if K > MAX_K else RG_ERR_ARG, where)
    return need


def workspace_layout(op, M, N, K, la=1, lb=1, lc=1, nprimes=0, host=False, transb=False, batch=1) -> Layout:
    out = Layout()
    rc = library().rg_workspace_layout_batched(op, batch, M, N, K, la, lb, lc, nprimes, _layout_flags(host, transb),
                                               ctypes.byref(out))
    if rc:
        raise ResGemmError(rc, "rg_workspace_layout")
    return out


# ---------------------------------------------------------------------------
# workspace cache: one growing device buffer per (device, stream)
# ---------------------------------------------------------------------------
_ws_cache: dict = {}


def workspace(nbytes: int, device: torch.device, stream=None) -> torch.Tensor:
    """A device buffer of at least nbytes, reused across calls on one stream."""
    stream = stream or torch.cuda.current_stream(device)
    key = (device.index, stream.cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        _ws_cache.pop(key, None)
        buf = torch.empty(max(nbytes, 4096), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def release_workspaces():
    _ws_cache.clear()


def _device_of(*ts):
    devs = {t.device for t in ts}
    if len(devs) != 1:
        raise ValueError("operands must be on one device")
    return devs.pop()


def _call_ctx(A, B):
    """(device for the work, flags) for operands on a CUDA device or on the host."""
    dev = _device_of(A, B)
    if dev.type == "cuda":
        return dev, 0
    if dev.type == "cpu":
        return torch.device("cuda", torch.cuda.current_device()), RG_FLAG_HOST
    raise ValueError(f"unsupported device {dev}")


def _on(dev):
    """The device context of a call: none when `dev` is already the current device."""
    return contextlib.nullcontext() if dev.index == torch.cuda.current_device() else torch.cuda.device(dev)


def _check(rc, where):
    if rc != RG_OK:
        raise ResGemmError(rc, where)


def _shapes(A, B, transb, core):
    """(batch, M, N, K, la, lb) of operands with `core` trailing dims per entry
    (0 for int64/float64 matrices, 1 for limb vectors), batched when they have one
    more leading dimension."""
    if A.dim() != B.dim() or A.dim() not in (2 + core, 3 + core):
        return None
    batched = A.dim() == 3 + core
    if batched and A.shape[0] != B.shape[0]:
        return None
    a, b = A.shape[int(batched):], B.shape[int(batched):]
    M, K = a[0], a[1]
    N, Kb = (b[0], b[1]) if transb else (b[1], b[0])
    if K != Kb:
        return None
    batch = A.shape[0] if batched else 1
    return batched, batch, M, N, K, (a[2] if core else 1), (b[2] if core else 1)


def _prepare(A, B, sync, transb):
    A, B = A.contiguous(), B.contiguous()
    dev, flags = _call_ctx(A, B)
    flags |= (RG_FLAG_SYNC if sync else 0) | (RG_FLAG_TRANS_B if transb else 0)
    return A, B, dev, flags


def _output(out, shape, dtype, like: torch.Tensor, host: bool, what: str) -> torch.Tensor:
    """A new result tensor, or the caller's `out` after checking that the kernels may write it whole."""
    if out is None:
        return torch.empty(shape, dtype=dtype, device=like.device, pin_memory=host)
    if (not isinstance(out, torch.Tensor) or tuple(out.shape) != tuple(shape) or out.dtype != dtype
            or out.device != like.device or not out.is_contiguous()):
        raise ValueError(f"{what}: out must be a contiguous {dtype} tensor of shape {tuple(shape)} on {like.device}")
    return out


def res_gemm_i64(A: torch.Tensor, B: torch.Tensor, nprimes: int = 0, sync: bool = True, out=None,
                 ws: torch.Tensor | None = None, transb: bool = False) -> torch.Tensor:
    """Exact C = A @ B for int64 matrices (CUDA tensors, or CPU tensors staged through the device).
    With transb, B is given as [N, K] and C = A @ B.T, without a transposed copy.  A [b, M, K] and
    B [b, K, N] run as one batched call with one plan."""
    sh = _shapes(A, B, transb, 0) if A.dtype == torch.int64 and B.dtype == torch.int64 else None
    if sh is None:
        raise ValueError("A [M,K] and B [K,N] (transb: [N,K]) int64 expected, optionally with a batch dimension")
    batched, batch, M, N, K, _, _ = sh
    A, B, dev, flags = _prepare(A, B, sync, transb)
    host = bool(flags & RG_FLAG_HOST)
    shape = (batch, M, N) if batched else (M, N)
    C = _output(out, shape, torch.int64, A, host, "res_gemm_i64")
    with _on(dev):
        need = _need(RG_OP_I64, M, N, K, "res_gemm_i64", nprimes=nprimes, host=host, transb=transb, batch=batch)
        w = ws if ws is not None else workspace(need, dev)
        rc = library().res_gemm_i64_batched(A.data_ptr(), B.data_ptr(), C.data_ptr(), batch, M, N, K, nprimes, flags,
                                            w.data_ptr(), w.numel(), torch.cuda.current_stream(dev).cuda_stream)
    _check(rc, "res_gemm_i64")
    return C


def res_gemm_limbs(A: torch.Tensor, B: torch.Tensor, lc: int, nprimes: int = 0, sync: bool = True, out=None,
                   ws: torch.Tensor | None = None, transb: bool = False) -> torch.Tensor:
    """Exact C = A @ B for multi-limb int64 operands A [M,K,la], B [K,N,lb]; returns [M,N,lc].
    With transb, B is given as [N,K,lb] and C = A @ B.T.  A leading batch dimension runs one
    batched call with one plan."""
    sh = _shapes(A, B, transb, 1) if A.dtype == torch.int64 and B.dtype == torch.int64 else None
    if sh is None:
        raise ValueError("A [M,K,la] and B [K,N,lb] (transb: [N,K,lb]) int64 expected, optionally batched")
    batched, batch, M, N, K, la, lb = sh
    A, B, dev, flags = _prepare(A, B, sync, transb)
    host = bool(flags & RG_FLAG_HOST)
    shape = (batch, M, N, lc) if batched else (M, N, lc)
    C = _output(out, shape, torch.int64, A, host, "res_gemm_limbs")
    with _on(dev):
        need = _need(RG_OP_LIMBS, M, N, K, "res_gemm_limbs", la=la, lb=lb, lc=lc, nprimes=nprimes, host=host,
                     transb=transb, batch=batch)
        w = ws if ws is not None else workspace(need, dev)
        rc = library().res_gemm_limbs_batched(A.data_ptr(), la, B.data_ptr(), lb, C.data_ptr(), lc, batch, M, N, K,
                                              nprimes, flags, w.data_ptr(), w.numel(),
                                              torch.cuda.current_stream(dev).cuda_stream)
    _check(rc, "res_gemm_limbs")
    return C


def enclose_gemm(A: torch.Tensor, B: torch.Tensor, sync: bool = True, ws: torch.Tensor | None = None,
                 transb: bool = False, out=None):
    """(lo, hi) with lo <= A @ B <= hi entrywise in exact arithmetic, in the operands' format
    (float64 or float32).  With transb, B is given as [N, K] and the bracket is of A @ B.T.
    A [b, M, K] and B [b, K, N] run as one batched call sharing one plan.  `out` may give the
    (lo, hi) pair to write."""
    if A.dtype != B.dtype or A.dtype not in (torch.float64, torch.float32):
        raise ValueError("float64 or float32 operands of one dtype expected")
    sh = _shapes(A, B, transb, 0)
    if sh is None:
        raise ValueError("A [M,K] and B [K,N] (transb: [N,K]) expected, optionally with a batch dimension")
    batched, batch, M, N, K, _, _ = sh
    f32 = A.dtype == torch.float32
    op = RG_OP_ENCLOSE_F32 if f32 else RG_OP_ENCLOSE
    A, B, dev, flags = _prepare(A, B, sync, transb)
    pin = bool(flags & RG_FLAG_HOST)
    shape = (batch, M, N) if batched else (M, N)
    name = "enclose_gemm_f32" if f32 else "enclose_gemm_f64"
    if out is not None and (not isinstance(out, (tuple, list)) or len(out) != 2):
        raise ValueError(f"{name}: out must be a (lo, hi) pair")
    lo = _output(None if out is None else out[0], shape, A.dtype, A, pin, name)
    hi = _output(None if out is None else out[1], shape, A.dtype, A, pin, name)
    with _on(dev):
        need = _need(op, M, N, K, name, host=pin, transb=transb, batch=batch)
        w = ws if ws is not None else workspace(need, dev)
        rc = getattr(library(), name + "_batched")(A.data_ptr(), B.data_ptr(), lo.data_ptr(), hi.data_ptr(), batch,
                                                   M, N, K, flags, w.data_ptr(), w.numel(),
                                                   torch.cuda.current_stream(dev).cuda_stream)
    _check(rc, name)
    return lo, hi


def enclose_gemm_f64(A: torch.Tensor, B: torch.Tensor, sync: bool = True, ws: torch.Tensor | None = None,
                     transb: bool = False, out=None):
    """enclose_gemm for float64 operands (float64 bounds)."""
    if A.dtype != torch.float64 or B.dtype != torch.float64:
        raise ValueError("float64 operands expected")
    return enclose_gemm(A, B, sync, ws, transb, out)


def enclose_gemm_f32(A: torch.Tensor, B: torch.Tensor, sync: bool = True, ws: torch.Tensor | None = None,
                     transb: bool = False):
    """enclose_gemm for float32 operands (float32 bounds)."""
    if A.dtype != torch.float32 or B.dtype != torch.float32:
        raise ValueError("float32 operands expected")
    return enclose_gemm(A, B, sync, ws, transb)


def _enclose_info(A: torch.Tensor) -> dict:
    """The regime of the last enclosure on A's device ("enclosure-gemm", Method: the lossless
    one-step bracket, or a coarsened fixed point whose flooring bound is added outward)."""
    dev = A.device if A.device.type == "cuda" else None
    plan = get_plan(device=dev)
    lossless = bool(plan["lossless"])
    return {"regime": "lossless" if lossless else "coarsened", "lossless": lossless, "nprimes": plan["nprimes"],
            "scale_exponents": (plan["f_a"], plan["f_b"]), "bound_bits": plan["bound_bits"]}


def mm_enclose(A: torch.Tensor, B: torch.Tensor, return_info: bool = False):
    """lo <= A @ B <= hi entrywise, exactly, for float64 or float32 operands
    ("enclosure-gemm", Usage: mm_enclose).  With return_info, also a dict naming the regime
    (lossless, or coarsened with the flooring bound added outward) and the plan's prime count and
    scale exponents."""
    lo, hi = enclose_gemm(A, B)
    return (lo, hi, _enclose_info(A)) if return_info else (lo, hi)


def mm_enclose_nt(A: torch.Tensor, Bt: torch.Tensor, return_info: bool = False):
    """The bracket of A @ Bt.T without a transposed copy ("enclosure-gemm", Usage: mm_enclose_nt)."""
    lo, hi = enclose_gemm(A, Bt, transb=True)
    return (lo, hi, _enclose_info(A)) if return_info else (lo, hi)


def interval_gemm(Am: torch.Tensor, Ar: torch.Tensor, Bm: torch.Tensor, Br: torch.Tensor, sync: bool = True,
                  ws: torch.Tensor | None = None, transb: bool = False, out=None):
    """(lo, hi) enclosing every product A @ B with A in <Am, Ar>, B in <Bm, Br> (midpoint, radius >= 0),
    by Rump's bound formed exactly and rounded outward once, in the operands' format (float64 or
    float32).  transb gives Bm and Br as [N, K]; a leading batch dimension shares one plan."""
    ts = (Am, Ar, Bm, Br)
    if any(t.dtype != Am.dtype for t in ts) or Am.dtype not in (torch.float64, torch.float32):
        raise ValueError("float64 or float32 operands of one dtype expected")
    if Ar.shape != Am.shape or Br.shape != Bm.shape:
        raise ValueError("each radius must have its midpoint's shape")
    sh = _shapes(Am, Bm, transb, 0)
    if sh is None:
        raise ValueError("Am [M,K] and Bm [K,N] (transb: [N,K]) expected, optionally with a batch dimension")
    batched, batch, M, N, K, _, _ = sh
    f32 = Am.dtype == torch.float32
    op = RG_OP_INTERVAL_F32 if f32 else RG_OP_INTERVAL
    Am, Ar, Bm, Br = (t.contiguous() for t in ts)
    dev, flags = _call_ctx(torch.empty(0, device=Am.device), torch.empty(0, device=Bm.device))
    if {t.device for t in (Am, Ar, Bm, Br)} != {Am.device}:
        raise ValueError("operands must be on one device")
    flags |= (RG_FLAG_SYNC if sync else 0) | (RG_FLAG_TRANS_B if transb else 0)
    pin = bool(flags & RG_FLAG_HOST)
    shape = (batch, M, N) if batched else (M, N)
    name = "interval_gemm_f32" if f32 else "interval_gemm_f64"
    if out is not None and (not isinstance(out, (tuple, list)) or len(out) != 2):
        raise ValueError(f"{name}: out must be a (lo, hi) pair")
    lo = _output(None if out is None else out[0], shape, Am.dtype, Am, pin, name)
    hi = _output(None if out is None else out[1], shape, Am.dtype, Am, pin, name)
    with _on(dev):
        need = _need(op, M, N, K, name, host=pin, transb=transb, batch=batch)
        w = ws if ws is not None else workspace(need, dev)
        rc = getattr(library(), name + "_batched")(Am.data_ptr(), Ar.data_ptr(), Bm.data_ptr(), Br.data_ptr(),
                                                   lo.data_ptr(), hi.data_ptr(), batch, M, N, K, flags,
                                                   w.data_ptr(), w.numel(), torch.cuda.current_stream(dev).cuda_stream)
    _check(rc, name)
    return lo, hi


def mm_interval(A_mid: torch.Tensor, A_rad: torch.Tensor, B_mid: torch.Tensor, B_rad: torch.Tensor):
    """Rump's midpoint-radius product of interval matrices as an outward (lo, hi)
    ("enclosure-gemm", Usage: mm_interval)."""
    return interval_gemm(A_mid, A_rad, B_mid, B_rad)


def bmm_enclose(A: torch.Tensor, B: torch.Tensor, return_info: bool = False):
    """Brackets of the batch A [b, M, K] @ B [b, K, N] with one shared plan
    ("enclosure-gemm", Usage: bmm_enclose)."""
    if A.dim() != 3 or B.dim() != 3:
        raise ValueError("A [b,M,K] and B [b,K,N] expected")
    lo, hi = enclose_gemm(A, B)
    return (lo, hi, _enclose_info(A)) if return_info else (lo, hi)


def res_gemm_stage(RA: torch.Tensor, RB: torch.Tensor, nprimes: int, M: int, N: int, K: int, RC=None,
                   sync: bool = True, transb: bool = False) -> torch.Tensor:
    """RC[p] = (RA[p] @ RB[p]) mod q_p for fp16 residues RA [P,M,lda], RB [P,K,ldb]
    (transb: RB [P,N,ldb], the product RA[p] @ RB[p].T); RC uint8 [P,M,ldc]."""
    if RA.dtype != torch.float16 or RB.dtype != torch.float16:
        raise ValueError("fp16 residues expected")
    if not (RA.is_contiguous() and RB.is_contiguous()):
        raise ValueError("contiguous residue planes expected")
    lda, ldb = RA.shape[-1], RB.shape[-1]
    ldc = (N + 15) // 16 * 16
    if RC is None:
        RC = torch.empty((nprimes, M, ldc), dtype=torch.uint8, device=RA.device)
    dev = RA.device
    flags = (RG_FLAG_SYNC if sync else 0) | (RG_FLAG_TRANS_B if transb else 0)
    with _on(dev):
        w = workspace(4096, dev)
        rc = library().res_gemm_stage(RA.data_ptr(), lda, RB.data_ptr(), ldb, RC.data_ptr(), RC.shape[-1], nprimes,
                                      M, N, K, flags, w.data_ptr(), w.numel(),
                                      torch.cuda.current_stream(dev).cuda_stream)
    _check(rc, "res_gemm_stage")
    return RC


def get_plan(ws: torch.Tensor | None = None, device=None) -> dict:
    """The plan of the last call on the cached workspace of `device` (or on `ws`)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    w = ws if ws is not None else workspace(4096, dev)
    info = PlanInfo()
    with _on(dev):
        _check(library().rg_get_plan(w.data_ptr(), torch.cuda.current_stream(dev).cuda_stream, ctypes.byref(info)),
               "rg_get_plan")
    return info.as_dict()


def set_stage_events(events) -> None:
    """Record four CUDA events around the stages of every later call (before
    the first kernel, before and after the GEMM, after the reconstruction);
    None removes the hook.  `events` are torch.cuda.Event objects (timing
    enabled) that stay alive while the hook is set."""
    lib = library()
    if events is None:
        _check(lib.rg_set_stage_events(None, 0), "rg_set_stage_events")
        return
    evs = list(events)
    if len(evs) != 4:
        raise ValueError("four events expected")
    for e in evs:
        e.record()  # creates the CUDA event behind a lazily created torch event
    arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in evs])
    _check(lib.rg_set_stage_events(arr, 4), "rg_set_stage_events")


def probe_mma_rate(kind: int, iters: int, blocks: int = 0, ws: torch.Tensor | None = None) -> float:
    """Enqueue one launch of a tensor-core rate probe (RG_PROBE_*) on the current stream of
    the current device; returns the operations (2 x multiply-adds) it performs.  Time it with
    events around the call; read its status afterwards with status(ws)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    w = ws if ws is not None else workspace(4096, dev)
    ops = ctypes.c_double(0.0)
    _check(library().rg_probe_mma_rate(int(kind), int(blocks), int(iters), w.data_ptr(), w.numel(),
                                       torch.cuda.current_stream(dev).cuda_stream, ctypes.byref(ops)),
           "rg_probe_mma_rate")
    return ops.value


def status(ws: torch.Tensor | None = None, device=None) -> int:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    w = ws if ws is not None else workspace(4096, dev)
    with _on(dev):
        return int(library().rg_status(w.data_ptr(), torch.cuda.current_stream(dev).cuda_stream))


# ---------------------------------------------------------------------------
# helpers ("enclosure-gemm", Usage: width_ulps and digest)
# ---------------------------------------------------------------------------


def _ordered(x: torch.Tensor) -> torch.Tensor:
    """float64 -> int64 key increasing with the value (+0 and -0 share 0)."""
    b = x.contiguous().view(torch.int64)
    mag = b & 0x7FFFFFFFFFFFFFFF
    return torch.where(b < 0, -mag, mag)


def width_ulps(lo: torch.Tensor, hi: torch.Tensor) -> torch.Tensor:
    """Number of representable steps from lo to hi (0 when lo == hi)."""
    return _ordered(hi) - _ordered(lo)


def digest(lo: torch.Tensor, hi: torch.Tensor) -> str:
    """SHA-256 over the raw bytes of lo then hi."""
    h = hashlib.sha256()
    h.update(lo.detach().contiguous().cpu().numpy().tobytes())
    h.update(hi.detach().contiguous().cpu().numpy().tobytes())
    return h.hexdigest()


def res_gemm_i64_noalloc(A: torch.Tensor, B: torch.Tensor, nprimes: int = 0, sync: bool = True,
                         out=None) -> torch.Tensor:
    """res_gemm_i64 on the library's fixed static scratch, for callers that cannot
    allocate device memory when they call.  A [M,K] and B [K,N] are int64 CUDA tensors; the
    result is allocated here only when `out` is None, and a given `out` must be a contiguous
    int64 [M,N] tensor on A's device.  Non-contiguous operands are copied first (an
    allocation), and the copies stay referenced until the call has returned; with
    sync=False the caller must keep A and B alive until the stream has run the call."""
    if A.dtype != torch.int64 or B.dtype != torch.int64 or A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("A [M,K] and B [K,N] int64 expected")
    if A.device.type != "cuda" or B.device != A.device:
        raise ValueError("device tensors on one GPU expected")
    M, K = A.shape
    N = B.shape[1]
    A, B, dev, flags = _prepare(A, B, sync, False)
    C = _output(out, (M, N), torch.int64, A, False, "res_gemm_i64_noalloc")
    with _on(dev):
        rc = library().res_gemm_i64_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, nprimes, flags,
                                            torch.cuda.current_stream(dev).cuda_stream)
    _check(rc, "res_gemm_i64_noalloc")
    return C


# ---------------------------------------------------------------------------
# exact solve ("exact-solve", Usage: solve)
# ---------------------------------------------------------------------------


def _limbs_to_int(vals) -> int:
    """Little-endian two's-complement int64 limbs -> Python int."""
    v = 0
    for i, x in enumerate(vals):
        v |= (int(x) & 0xFFFFFFFFFFFFFFFF) << (64 * i)
    if vals and int(vals[-1]) < 0:
        v -= 1 << (64 * len(vals))
    return v


def _int_to_limbs(v: int, limbs: int):
    u = v & ((1 << (64 * limbs)) - 1)
    return [((u >> (64 * i)) & 0xFFFFFFFFFFFFFFFF) - ((1 << 64) if (u >> (64 * i + 63)) & 1 else 0)
            for i in range(limbs)]


def solve_integers(A: torch.Tensor, b: torch.Tensor, info: dict | None = None):
    """The exact solution of A X = b in integer form (N, d): numerators N [n][c] (Python
    ints) and the least common denominator d > 0, X = N / d; None if A is singular.  A [n, n]
    and b [n] or [n, c] are int64 (CUDA tensors, or CPU tensors staged through the device).
    `info`, if given, receives the lift's step and prime counts and the phase times."""
    if A.dtype != torch.int64 or b.dtype != torch.int64 or A.dim() != 2 or A.shape[0] != A.shape[1]:
        raise ValueError("A [n, n] and b [n] or [n, c] int64 expected")
    b2 = b.reshape(-1, 1) if b.dim() == 1 else b
    if b2.dim() != 2 or b2.shape[0] != A.shape[0]:
        raise ValueError("b must have n rows")
    A, b2 = A.contiguous(), b2.contiguous()
    dev, flags = _call_ctx(A, b2)
    n, c = A.shape[0], b2.shape[1]
    sol = Solution()
    with _on(dev):
        rc = library().rg_solve_i64(A.data_ptr(), b2.data_ptr(), n, c, flags,
                                    torch.cuda.current_stream(dev).cuda_stream, ctypes.byref(sol))
    if rc == RG_ERR_SINGULAR:
        return None
    _check(rc, "rg_solve_i64")
    try:
        nb = 8 * sol.limbs
        raw = ctypes.string_at(sol.values, (n * c + 1) * nb)
    finally:
        library().rg_solution_free(ctypes.byref(sol))
    vals = [int.from_bytes(raw[k * nb:(k + 1) * nb], "little", signed=True) for k in range(n * c + 1)]
    d = vals[-1]
    if info is not None:
        info.update(steps=int(sol.steps), primes=int(sol.primes), denominator=d, ms_inverse=sol.ms_inverse,
                    ms_lift=sol.ms_lift, ms_reconstruct=sol.ms_reconstruct)
    return [vals[i * c:(i + 1) * c] for i in range(n)], d


def solve(A: torch.Tensor, b: torch.Tensor, info: dict | None = None):
    """The exact solution X of A X = b over the rationals, as a nested list [n][c] of
    fractions.Fraction (c = 1 for a 1-D b), or None if A is singular ("exact-solve", Usage:
    solve).  See solve_integers for the arguments."""
    r = solve_integers(A, b, info)
    if r is None:
        return None
    N, d = r
    return [[Fraction(v, d) for v in row] for row in N]


def big_gcd(a: int, b: int) -> int:
    """gcd of two naturals by the library's host big-integer code (the solve's reconstruction uses it)."""
    al, bl = max(1, (a.bit_length() + 63) // 64), max(1, (b.bit_length() + 63) // 64)
    gl = min(al, bl)
    mask = (1 << 64) - 1
    A = (ctypes.c_uint64 * al)(*[(a >> (64 * i)) & mask for i in range(al)])
    B = (ctypes.c_uint64 * bl)(*[(b >> (64 * i)) & mask for i in range(bl)])
    G = (ctypes.c_uint64 * gl)()
    _check(library().rg_big_gcd(A, al, B, bl, G, gl), "rg_big_gcd")
    return sum(int(G[i]) << (64 * i) for i in range(gl))


def big_mulmod(a: int, b: int, m: int) -> int:
    """(a b) mod m for naturals a, b < m by the library's host big-integer code (the solve's numerators use it)."""
    n = max(1, (m.bit_length() + 63) // 64)
    mask = (1 << 64) - 1
    limbs = lambda x: (ctypes.c_uint64 * n)(*[(x >> (64 * i)) & mask for i in range(n)])  # noqa: E731
    R = (ctypes.c_uint64 * n)()
    _check(library().rg_big_mulmod(limbs(a), n, limbs(b), n, limbs(m), n, R, n), "rg_big_mulmod")
    return sum(int(R[i]) << (64 * i) for i in range(n))


def rational_reconstruct(x: int, m: int, nbits: int, dbits: int):
    """(N, D) with D x == N (mod m), |N| <= 2^nbits, 0 < D <= 2^dbits, in lowest terms,
    by the library's host reconstruction; None if there is none."""
    xl = max(1, (x.bit_length() + 63) // 64)
    ml = max(1, (m.bit_length() + 63) // 64)
    limbs = max(nbits, dbits) // 64 + 2
    X = (ctypes.c_int64 * xl)(*_int_to_limbs(x, xl))
    Mv = (ctypes.c_int64 * ml)(*_int_to_limbs(m, ml))
    num = (ctypes.c_int64 * limbs)()
    den = (ctypes.c_int64 * limbs)()
    rc = library().rg_rational_reconstruct(X, xl, Mv, ml, nbits, dbits, num, den, limbs)
    if rc == RG_ERR_RANGE:
        return None
    _check(rc, "rg_rational_reconstruct")
    return _limbs_to_int(list(num)), _limbs_to_int(list(den))


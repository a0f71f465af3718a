"""Python binding of libbfp8 (blockwise-scaled FP8 quantisation and GEMMs, sm_103a).

Argument marshalling only: every step runs in the library's CUDA kernels,
called through the C ABI declared in ``include/bfp8.h``.  PyTorch provides
device memory and the current stream.  There is no CPU fallback: if the
library is missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbfp8.so")
BLOCK = 128

BFP8_OK, BFP8_ERR_INVALID_ARG, BFP8_ERR_UNSUPPORTED, BFP8_ERR_CUDA, BFP8_ERR_TIMEOUT = range(5)

EXPORTS = [
    "bfp8_last_error", "bfp8_quant_lhs", "bfp8_quant_rhs", "bfp8_quant_weight",
    "bfp8_gemm_1x128_128x128", "bfp8_gemm_1x128_128x1", "bfp8_linear_workspace_size",
    "bfp8_linear_fwd", "bfp8_linear_bwd", "bfp8_cast_e4m3", "bfp8_check_device_errors",
    "bfp8_debug_write_counts", "bfp8_debug_gemm_stall", "bfp8_debug_gemm_pick_bn", "bfp8_debug_launch_pdl", "bfp8_quant_dual",
    "bfp8_linear_train_workspace_size", "bfp8_linear_fwd_train", "bfp8_linear_bwd_saved",
    "bfp8_linear_fwd_static", "bfp8_gemm_grouped_1x128_128x128", "bfp8_gemm_grouped_1x128_128x1",
    "bfp8_quant_dual_weight", "bfp8_mx_cast", "bfp8_linear_step_host_workspace_size",
    "bfp8_linear_step_host", "bfp8_moe_step_host_workspace_size", "bfp8_moe_step_host",
    "bfp8_gemm_1x128_128x128_xq", "bfp8_gemm_1x128_128x1_xq",
]

_lib = None


class Bfp8Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"bfp8 status {status}: {msg}")
        self.status = status


def build(force: bool = False) -> str:
    from . import buildlib as _b
    return _b.build(force=force)


def lib() -> ctypes.CDLL:
    """Loads libbfp8.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with blockwise_scaled_fp8_gb300.build()")
    L = ctypes.CDLL(LIB_PATH)
    i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    L.bfp8_last_error.restype = ctypes.c_char_p
    L.bfp8_last_error.argtypes = []
    L.bfp8_quant_lhs.argtypes = [vp, i64, i64, i64, i32, vp, i64, vp, i64, vp]
    L.bfp8_quant_rhs.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp]
    L.bfp8_quant_weight.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp]
    L.bfp8_gemm_1x128_128x128.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i32, vp, i64, i64, i64, i64, vp]
    L.bfp8_gemm_1x128_128x1.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, i64, vp]
    L.bfp8_linear_workspace_size.argtypes = [i64, i64, i64]
    L.bfp8_linear_workspace_size.restype = sz
    L.bfp8_linear_fwd.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
    L.bfp8_linear_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp, sz, vp]
    L.bfp8_cast_e4m3.argtypes = [vp, i64, vp, vp]
    L.bfp8_check_device_errors.argtypes = [vp]
    L.bfp8_debug_write_counts.argtypes = [i32, i64, i64, i64, i32, vp, vp, ctypes.POINTER(i64)]
    L.bfp8_debug_gemm_pick_bn.argtypes = [i64, i64, i32, i32]
    L.bfp8_debug_launch_pdl.argtypes = [i32, i64, i64, i64]
    L.bfp8_quant_dual.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp]
    L.bfp8_mx_cast.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp]
    L.bfp8_quant_dual_weight.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                         vp, i64, i64, vp, i64, vp, i64, vp, i64, vp]
    L.bfp8_linear_train_workspace_size.argtypes = [i64, i64, i64]
    L.bfp8_linear_train_workspace_size.restype = sz
    L.bfp8_linear_fwd_train.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
    L.bfp8_linear_bwd_saved.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
    L.bfp8_linear_step_host_workspace_size.argtypes = [i64, i64, i64]
    L.bfp8_linear_step_host_workspace_size.restype = sz
    L.bfp8_linear_step_host.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, sz, vp]
    L.bfp8_moe_step_host_workspace_size.argtypes = [i64, i64, i64]
    L.bfp8_moe_step_host_workspace_size.restype = sz
    L.bfp8_moe_step_host.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, i64, i64, i64, i64, vp, sz, vp]
    L.bfp8_linear_fwd_static.argtypes = [vp, vp, vp, i64, i64, i64, vp]
    L.bfp8_gemm_1x128_128x128_xq.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, i64, vp]
    L.bfp8_gemm_1x128_128x1_xq.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, i64, vp]
    L.bfp8_gemm_grouped_1x128_128x128.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i32, vp, i64, vp, i64,
                                                  i64, i64, i64, vp]
    L.bfp8_gemm_grouped_1x128_128x1.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i64,
                                                i64, i64, i64, vp]
    L.bfp8_debug_gemm_stall.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, i64, i64, vp]
    for name in EXPORTS:
        if name not in ("bfp8_last_error", "bfp8_linear_workspace_size", "bfp8_linear_train_workspace_size",
                        "bfp8_linear_step_host_workspace_size", "bfp8_moe_step_host_workspace_size"):
            getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(status: int) -> None:
    if status != BFP8_OK:
        raise Bfp8Error(status, lib().bfp8_last_error().decode(errors="replace"))


def _cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


def _rup(a: int, b: int) -> int:
    return _cdiv(a, b) * b


def _torch():
    import torch
    return torch


def _stream():
    return ctypes.c_void_p(_torch().cuda.current_stream().cuda_stream)


def _p(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(None)


def _need_bf16_2d(t, name):
    torch = _torch()
    if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_cuda or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D CUDA bf16 tensor with unit column stride")


# ---------------------------------------------------------------------------
# Quantisation
# ---------------------------------------------------------------------------

def quant_lhs(x, transposed: bool = False, q=None, s=None):
    """1x128 groups along K of A = x ([M,K]) or A = x^T (x is [K,M]).
    Returns (q [M, ldq] uint8 e4m3 bytes, s [Kb, lds] float32), where s[kb, m]
    is the scale of row m's group kb (the column-major [M, Kb] layout)."""
    torch = _torch()
    _need_bf16_2d(x, "x")
    if transposed:
        K, M = x.shape
    else:
        M, K = x.shape
    Kb = _cdiv(K, BLOCK)
    if q is None:
        q = torch.empty((M, _rup(max(K, 1), 16)), dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty((Kb, max(M, 1)), dtype=torch.float32, device=x.device)
    _check(lib().bfp8_quant_lhs(_p(x), M, K, x.stride(0), int(transposed), _p(q), q.stride(0),
                                _p(s), s.stride(0), _stream()))
    return q, s


def quant_rhs(x, q=None, s=None):
    """128x1 groups along the rows (reduction dim K) of x [K,N]; bytes written
    transposed.  Returns (qT [N, ldq] uint8, s [Kb, lds] float32)."""
    torch = _torch()
    _need_bf16_2d(x, "x")
    K, N = x.shape
    Kb = _cdiv(K, BLOCK)
    if q is None:
        q = torch.empty((N, _rup(max(K, 1), 16)), dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty((Kb, _rup(max(N, 1), 4)), dtype=torch.float32, device=x.device)
    _check(lib().bfp8_quant_rhs(_p(x), K, N, x.stride(0), _p(q), q.stride(0), _p(s), s.stride(0), _stream()))
    return q, s


def quant_weight(w, with_q: bool = True, with_t: bool = False, q=None, qt=None, s=None):
    """128x128 tiles of w [N,K].  Returns (q [N, ldq] or None, qt [K, ldqt] or
    None, s [Nb, lds] float32)."""
    torch = _torch()
    _need_bf16_2d(w, "w")
    N, K = w.shape
    Nb, Kb = _cdiv(N, BLOCK), _cdiv(K, BLOCK)
    if with_q and q is None:
        q = torch.empty((N, _rup(max(K, 1), 16)), dtype=torch.uint8, device=w.device)
    if with_t and qt is None:
        qt = torch.empty((K, _rup(max(N, 1), 16)), dtype=torch.uint8, device=w.device)
    if s is None:
        s = torch.empty((max(Nb, 1), max(Kb, 1)), dtype=torch.float32, device=w.device)
    _check(lib().bfp8_quant_weight(_p(w), N, K, w.stride(0), _p(q), q.stride(0) if q is not None else 0,
                                   _p(qt), qt.stride(0) if qt is not None else 0, _p(s), s.stride(0),
                                   _stream()))
    return q, qt, s


def quant_dual(x, q_row=None, s_row=None, q_col=None, s_col=None):
    """Both quantisations of x [T,C] from one read: (q_row [T, ldq], s_row
    [Cb, lds] as quant_lhs(x)) and (q_col [C, ldq'], s_col [Tb, lds'] as
    quant_rhs(x))."""
    torch = _torch()
    _need_bf16_2d(x, "x")
    T, C = x.shape
    dev = x.device
    if q_row is None:
        q_row = torch.empty((T, _rup(max(C, 1), 16)), dtype=torch.uint8, device=dev)
    if s_row is None:
        s_row = torch.empty((_cdiv(C, BLOCK), _rup(max(T, 1), 4)), dtype=torch.float32, device=dev)
    if q_col is None:
        q_col = torch.empty((C, _rup(max(T, 1), 16)), dtype=torch.uint8, device=dev)
    if s_col is None:
        s_col = torch.empty((_cdiv(T, BLOCK), _rup(max(C, 1), 4)), dtype=torch.float32, device=dev)
    _check(lib().bfp8_quant_dual(_p(x), T, C, x.stride(0), _p(q_row), q_row.stride(0), _p(s_row), s_row.stride(0),
                                 _p(q_col), q_col.stride(0), _p(s_col), s_col.stride(0), _stream()))
    return q_row, s_row, q_col, s_col


def quant_dual_weight(x, w, q_row=None, s_row=None, q_col=None, s_col=None, qw=None, qwt=None, sw=None):
    """quant_dual(x) and quant_weight(w, with_q=True, with_t=True) in one
    launch (x [T,C], w [N,C]).  Returns ((q_row, s_row, q_col, s_col), (qw, qwt, sw))."""
    torch = _torch()
    _need_bf16_2d(x, "x")
    _need_bf16_2d(w, "w")
    T, C = x.shape
    N = w.shape[0]
    if w.shape[1] != C:
        raise ValueError("quant_dual_weight: x and w must share their second dimension")
    dev = x.device
    e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
    q_row = e((T, _rup(max(C, 1), 16)), torch.uint8) if q_row is None else q_row
    s_row = e((_cdiv(C, BLOCK), _rup(max(T, 1), 4)), torch.float32) if s_row is None else s_row
    q_col = e((C, _rup(max(T, 1), 16)), torch.uint8) if q_col is None else q_col
    s_col = e((_cdiv(T, BLOCK), _rup(max(C, 1), 4)), torch.float32) if s_col is None else s_col
    qw = e((N, _rup(max(C, 1), 16)), torch.uint8) if qw is None else qw
    qwt = e((C, _rup(max(N, 1), 16)), torch.uint8) if qwt is None else qwt
    sw = e((max(_cdiv(N, BLOCK), 1), max(_cdiv(C, BLOCK), 1)), torch.float32) if sw is None else sw
    _check(lib().bfp8_quant_dual_weight(_p(x), T, C, x.stride(0), _p(q_row), q_row.stride(0), _p(s_row),
                                        s_row.stride(0), _p(q_col), q_col.stride(0), _p(s_col), s_col.stride(0),
                                        _p(w), N, w.stride(0), _p(qw), qw.stride(0), _p(qwt), qwt.stride(0), _p(sw),
                                        sw.stride(0), _stream()))
    return (q_row, s_row, q_col, s_col), (qw, qwt, sw)


def mx_cast(x, dim0: bool = True, dim1: bool = True, q0=None, e0=None, q1=None, e1=None):
    """MXFP8 casts of x [M,K] (E4M3 codes, E8M0 exponents per 32 elements):
    dim0 -> (q0 [M, ldq0], e0 [M, ceil(K/32)]), dim1 (transposed) -> (q1 [K, ldq1],
    e1 [K, ceil(M/32)]); None for a cast not asked for."""
    torch = _torch()
    _need_bf16_2d(x, "x")
    M, K = x.shape
    dev = x.device
    if dim0:
        q0 = torch.empty((M, _rup(max(K, 1), 16)), dtype=torch.uint8, device=dev) if q0 is None else q0
        e0 = torch.empty((M, max(_cdiv(K, 32), 1)), dtype=torch.uint8, device=dev) if e0 is None else e0
    if dim1:
        q1 = torch.empty((K, _rup(max(M, 1), 16)), dtype=torch.uint8, device=dev) if q1 is None else q1
        e1 = torch.empty((K, max(_cdiv(M, 32), 1)), dtype=torch.uint8, device=dev) if e1 is None else e1
    _check(lib().bfp8_mx_cast(_p(x), M, K, x.stride(0), _p(q0) if dim0 else None, q0.stride(0) if dim0 else 0,
                              _p(e0) if dim0 else None, e0.stride(0) if dim0 else 0,
                              _p(q1) if dim1 else None, q1.stride(0) if dim1 else 0,
                              _p(e1) if dim1 else None, e1.stride(0) if dim1 else 0, _stream()))
    return (q0 if dim0 else None, e0 if dim0 else None), (q1 if dim1 else None, e1 if dim1 else None)


def cast_e4m3(x, q=None):
    """Elementwise RNE fp32 -> e4m3fn with saturation to +-448."""
    torch = _torch()
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA float32 tensor")
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib().bfp8_cast_e4m3(_p(x), x.numel(), _p(q), _stream()))
    return q


# ---------------------------------------------------------------------------
# GEMMs
# ---------------------------------------------------------------------------

def gemm_1x128_128x128(qa, sa, qb, sb, K: int, sb_transposed: bool = False, out=None, M=None, N=None):
    """C = A B with A = qa [M, lda] (1x128 scales sa [Kb, ldsa]), B^T = qb
    [N, ldb] (128x128 tile scales sb, [Nb, ldsb] or transposed [Kb, ldsb]).
    Returns C [M, N] bf16."""
    torch = _torch()
    M = qa.shape[0] if M is None else M
    N = qb.shape[0] if N is None else N
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=qa.device)
    _check(lib().bfp8_gemm_1x128_128x128(_p(qa), qa.stride(0), _p(sa), sa.stride(0), _p(qb), qb.stride(0),
                                         _p(sb), sb.stride(0), int(sb_transposed), _p(out), out.stride(0),
                                         M, N, K, _stream()))
    return out


def gemm_1x128_128x1(qa, sa, qb, sb, K: int, out=None, M=None, N=None):
    """C = A B with A = qa [M, lda] (1x128 scales sa [Kb, ldsa]) and B^T = qb
    [N, ldb] with one scale per column and K-block, sb [Kb, ldsb]."""
    torch = _torch()
    M = qa.shape[0] if M is None else M
    N = qb.shape[0] if N is None else N
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=qa.device)
    _check(lib().bfp8_gemm_1x128_128x1(_p(qa), qa.stride(0), _p(sa), sa.stride(0), _p(qb), qb.stride(0),
                                       _p(sb), sb.stride(0), _p(out), out.stride(0), M, N, K, _stream()))
    return out


def gemm_1x128_128x128_xq(x, qb, sb, out=None, N=None):
    """C = quant_lhs(x) B with x bf16 [M, K] quantised inside the GEMM (one
    launch), B^T = qb [N, ldb] with its 128x128 tile scales sb [Nb, ldsb]
    (bfp8_quant_weight's outputs).  Returns C [M, N] bf16."""
    torch = _torch()
    _need_bf16_2d(x, "x")
    M, K = x.shape
    N = qb.shape[0] if N is None else N
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(lib().bfp8_gemm_1x128_128x128_xq(_p(x), x.stride(0), _p(qb), qb.stride(0), _p(sb), sb.stride(0),
                                            _p(out), out.stride(0), M, N, K, _stream()))
    return out


def gemm_1x128_128x1_xq(qa, sa, x, out=None, M=None):
    """C = A quant_rhs(x) with A = qa [M, lda] (1x128 scales sa [Kb, ldsa])
    and x bf16 [K, N] quantised 128x1 inside the GEMM (one launch; the weight
    gradient dW = dY^T X with qa, sa the transposed 1x128 quantisation of dY).
    Returns C [M, N] bf16."""
    torch = _torch()
    _need_bf16_2d(x, "x")
    K, N = x.shape
    M = qa.shape[0] if M is None else M
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(lib().bfp8_gemm_1x128_128x1_xq(_p(qa), qa.stride(0), _p(sa), sa.stride(0), _p(x), x.stride(0),
                                          _p(out), out.stride(0), M, N, K, _stream()))
    return out


# ---------------------------------------------------------------------------
# Grouped (mixture-of-experts) GEMMs: tokens sorted by expert, expert e owning
# token rows offs[e] .. offs[e+1] (offs: int32 tensor [E+1] on the device)
# ---------------------------------------------------------------------------

def _offs(offs):
    torch = _torch()
    if offs.dtype != torch.int32 or offs.dim() != 1 or not offs.is_contiguous():
        raise ValueError("offs must be a contiguous 1-d int32 tensor of E+1 offsets")
    return offs


def gemm_grouped_1x128_128x128(qa, sa, qb, sb, offs, N: int, K: int, sb_transposed: bool = False, out=None):
    """Per expert e, C[offs[e]:offs[e+1]] = A[offs[e]:offs[e+1]] B_e.  Forward
    (sb_transposed False): qb [E*N, ldb] stacked weight codes, sb [E*Nb, ldsb]
    their tile scales.  Input gradient (True, K = the experts' output
    features): qb [N, ldb] the stacked weight's transposed codes (expert e in
    columns e*K ..), sb [E*Kb, ldsb].  Returns C [M_total, N] bf16 (rows outside
    the experts are left as they were in ``out``)."""
    torch = _torch()
    offs = _offs(offs)
    M_total = qa.shape[0]
    if out is None:
        out = torch.empty((M_total, N), dtype=torch.bfloat16, device=qa.device)
    _check(lib().bfp8_gemm_grouped_1x128_128x128(_p(qa), qa.stride(0), _p(sa), sa.stride(0), _p(qb), qb.stride(0),
                                                 _p(sb), sb.stride(0), int(sb_transposed), _p(offs),
                                                 offs.numel() - 1, _p(out), out.stride(0), M_total, N, K,
                                                 _stream()))
    return out


def gemm_grouped_1x128_128x1(qa, sa, qb, sb, offs, T: int, out=None):
    """Per expert e, dW[e] = A[:, tokens of e] B[tokens of e, :]: qa [M, lda]
    (1x128 along tokens, sa [Tb, ldsa]), qb [N, ldb] (128x1 along tokens,
    transposed; sb [Tb, ldsb]).  Every expert starts on a 128-token boundary.
    Returns dW [E, M, N] bf16."""
    torch = _torch()
    offs = _offs(offs)
    E = offs.numel() - 1
    M, N = qa.shape[0], qb.shape[0]
    if out is None:
        out = torch.empty((E, M, N), dtype=torch.bfloat16, device=qa.device)
    _check(lib().bfp8_gemm_grouped_1x128_128x1(_p(qa), qa.stride(0), _p(sa), sa.stride(0), _p(qb), qb.stride(0),
                                               _p(sb), sb.stride(0), _p(offs), E, _p(out), out.stride(1),
                                               out.stride(0), M, N, T, _stream()))
    return out


def moe_linear_fwd(x, w, offs, y=None):
    """Mixture-of-experts forward y_e = x_e W_e^T: x [M_total, K] bf16 tokens
    sorted by expert, w [E, N, K] bf16 (N % 128 == 0, so the stacked weight's
    128x128 tiles stay inside one expert).  Returns (y, saved) where saved
    holds the quantised operands the backward reuses."""
    E, N, K = w.shape
    if N % 128:
        raise ValueError("moe_linear_fwd: the experts' output features must be a multiple of 128")
    (qx, sx, qxt, sxt), (qw, qwt, sw) = quant_dual_weight(x, w.reshape(E * N, K))
    y = gemm_grouped_1x128_128x128(qx, sx, qw, sw, offs, N, K, out=y)
    return y, (qxt, sxt, qwt, sw)


def moe_linear_bwd(dy, saved, offs, dx=None, dw=None):
    """Mixture-of-experts backward from moe_linear_fwd's saved operands:
    dx_e = dy_e W_e, dW_e = dy_e^T x_e (every expert starting on a 128-token
    boundary).  Returns (dx [M_total, K], dW [E, N, K])."""
    qxt, sxt, qwt, sw = saved
    M_total, N = dy.shape
    K = qxt.shape[0]
    qdy, sdy, qdyt, sdyt = quant_dual(dy)
    dx = gemm_grouped_1x128_128x128(qdy, sdy, qwt, sw, offs, K, N, sb_transposed=True, out=dx)
    dw = gemm_grouped_1x128_128x1(qdyt, sdyt, qxt, sxt, offs, M_total, out=dw)
    return dx, dw


# ---------------------------------------------------------------------------
# Linear layer
# ---------------------------------------------------------------------------

def linear_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib().bfp8_linear_workspace_size(M, N, K))


def _workspace(M, N, K, device, ws):
    torch = _torch()
    need = linear_workspace_size(M, N, K)
    if ws is None:
        ws = torch.empty(max(need, 256) + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    if ws.numel() - off < need:
        raise ValueError(f"workspace too small: {ws.numel() - off} < {need}")
    return ws, ctypes.c_void_p(ws.data_ptr() + off), ws.numel() - off


def linear_fwd(x, w, y=None, ws=None):
    """y = x W^T through blockwise FP8 (x [M,K], w [N,K] bf16 contiguous)."""
    torch = _torch()
    M, K = x.shape
    N = w.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws, wp, wn = _workspace(M, N, K, x.device, ws)
    _check(lib().bfp8_linear_fwd(_p(x), _p(w), _p(y), M, N, K, wp, wn, _stream()))
    return y


def linear_bwd(dy, x, w, dx=None, dw=None, ws=None):
    """dx = dy W, dw = dy^T x through blockwise FP8."""
    torch = _torch()
    M, K = x.shape
    N = w.shape[0]
    if dx is None:
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=x.device)
    if dw is None:
        dw = torch.empty((N, K), dtype=torch.bfloat16, device=x.device)
    ws, wp, wn = _workspace(M, N, K, x.device, ws)
    _check(lib().bfp8_linear_bwd(_p(dy), _p(x), _p(w), _p(dx), _p(dw), M, N, K, wp, wn, _stream()))
    return dx, dw


def debug_gemm_stall(qa, sa, qb, sb, K: int, out, wait_limit_us: int = 50000):
    """Test hook: a GEMM launch whose promotion warps wait on a barrier nothing
    arrives on; returns the launch status (the timeout itself is reported by
    check_device_errors())."""
    M, N = out.shape
    return lib().bfp8_debug_gemm_stall(_p(qa), qa.stride(0), _p(sa), sa.stride(0), _p(qb), qb.stride(0),
                                       _p(sb), sb.stride(0), _p(out), out.stride(0), M, N, K,
                                       wait_limit_us, _stream())


def linear_fwd_static(x, w, y=None):
    """y = x W^T through blockwise FP8 without a caller workspace (the
    library's fixed 32 MiB scratch; see bfp8_linear_fwd_static)."""
    torch = _torch()
    M, K = x.shape
    N = w.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(lib().bfp8_linear_fwd_static(_p(x), _p(w), _p(y), M, N, K, _stream()))
    return y


def linear_train_workspace(M: int, N: int, K: int, device="cuda"):
    """Workspace for linear_fwd_train / linear_bwd_saved (256 bytes of slack
    for alignment)."""
    torch = _torch()
    return torch.empty(int(lib().bfp8_linear_train_workspace_size(M, N, K)) + 256, dtype=torch.uint8, device=device)


def _aligned(ws):
    off = (-ws.data_ptr()) % 256
    return ctypes.c_void_p(ws.data_ptr() + off), ws.numel() - off


def linear_fwd_train(x, w, ws, y=None):
    """Training forward: y = x W^T, keeping in `ws` the quantised operands the
    backward needs (see bfp8_linear_fwd_train)."""
    torch = _torch()
    M, K = x.shape
    N = w.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    wp, wn = _aligned(ws)
    _check(lib().bfp8_linear_fwd_train(_p(x), _p(w), _p(y), M, N, K, wp, wn, _stream()))
    return y


def linear_bwd_saved(dy, ws, M: int, N: int, K: int, dx=None, dw=None):
    """Backward from the workspace a linear_fwd_train call filled."""
    torch = _torch()
    if dx is None:
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device)
    if dw is None:
        dw = torch.empty((N, K), dtype=torch.bfloat16, device=dy.device)
    wp, wn = _aligned(ws)
    _check(lib().bfp8_linear_bwd_saved(_p(dy), _p(dx), _p(dw), M, N, K, wp, wn, _stream()))
    return dx, dw


def linear_step_host_workspace(M: int, N: int, K: int, device="cuda"):
    """Device workspace for linear_step_host (256 bytes of slack for alignment)."""
    torch = _torch()
    return torch.empty(int(lib().bfp8_linear_step_host_workspace_size(M, N, K)) + 256, dtype=torch.uint8,
                       device=device)


def linear_step_host(x, w, dy, ws, y=None, dx=None, dw=None, chunk_n: int = 0):
    """One training step from host tensors (see bfp8_linear_step_host): x [M,K],
    w [N,K], dy [M,N] contiguous bf16 CPU tensors (pinned for overlap); returns
    host (y, dx, dw), allocated pinned when not given.  Enqueued on the current
    CUDA stream: synchronise it before reading the outputs."""
    torch = _torch()
    for name, t in (("x", x), ("w", w), ("dy", dy)):
        if t.device.type != "cpu" or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"linear_step_host: {name} must be a contiguous bf16 CPU tensor")
    M, K = x.shape
    N = w.shape[0]
    if tuple(w.shape) != (N, K) or tuple(dy.shape) != (M, N):
        raise ValueError(f"linear_step_host: shapes x {tuple(x.shape)}, w {tuple(w.shape)}, dy {tuple(dy.shape)}")
    pin = torch.cuda.is_available()
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=pin)
    if dx is None:
        dx = torch.empty((M, K), dtype=torch.bfloat16, pin_memory=pin)
    if dw is None:
        dw = torch.empty((N, K), dtype=torch.bfloat16, pin_memory=pin)
    for name, t, shp in (("y", y, (M, N)), ("dx", dx, (M, K)), ("dw", dw, (N, K))):
        if t.device.type != "cpu" or t.dtype != torch.bfloat16 or not t.is_contiguous() or tuple(t.shape) != shp:
            raise ValueError(f"linear_step_host: {name} must be a contiguous bf16 CPU tensor of shape {shp}")
    wp, wn = _aligned(ws)
    _check(lib().bfp8_linear_step_host(_p(x), _p(w), _p(dy), _p(y), _p(dx), _p(dw), M, N, K, int(chunk_n),
                                       wp, wn, _stream()))
    return y, dx, dw


def moe_step_host_workspace(M_max: int, N: int, K: int, device="cuda"):
    """Device workspace for moe_step_host (M_max: the largest expert's tokens)."""
    torch = _torch()
    return torch.empty(int(lib().bfp8_moe_step_host_workspace_size(M_max, N, K)) + 256, dtype=torch.uint8,
                       device=device)


def moe_step_host(x, w, dy, offs, ws, y=None, dx=None, dw=None, chunk_n: int = 0):
    """Mixture-of-experts training step from host tensors (see
    bfp8_moe_step_host): x [T,K], w [E,N,K], dy [T,N] contiguous bf16 CPU
    tensors (pinned for overlap), offs int32 [E+1] on the CPU.  Returns host
    (y, dx, dw); enqueued on the current CUDA stream."""
    torch = _torch()
    for name, t in (("x", x), ("w", w), ("dy", dy)):
        if t.device.type != "cpu" or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"moe_step_host: {name} must be a contiguous bf16 CPU tensor")
    if offs.device.type != "cpu" or offs.dtype != torch.int32 or not offs.is_contiguous():
        raise ValueError("moe_step_host: offs must be a contiguous int32 CPU tensor")
    T, K = x.shape
    E, N = w.shape[0], w.shape[1]
    if tuple(w.shape) != (E, N, K) or tuple(dy.shape) != (T, N) or offs.numel() != E + 1:
        raise ValueError(f"moe_step_host: shapes x {tuple(x.shape)}, w {tuple(w.shape)}, dy {tuple(dy.shape)}, "
                         f"offs {tuple(offs.shape)}")
    pin = torch.cuda.is_available()
    y = torch.empty((T, N), dtype=torch.bfloat16, pin_memory=pin) if y is None else y
    dx = torch.empty((T, K), dtype=torch.bfloat16, pin_memory=pin) if dx is None else dx
    dw = torch.empty((E, N, K), dtype=torch.bfloat16, pin_memory=pin) if dw is None else dw
    for name, t, shp in (("y", y, (T, N)), ("dx", dx, (T, K)), ("dw", dw, (E, N, K))):
        if t.device.type != "cpu" or t.dtype != torch.bfloat16 or not t.is_contiguous() or tuple(t.shape) != shp:
            raise ValueError(f"moe_step_host: {name} must be a contiguous bf16 CPU tensor of shape {shp}")
    wp, wn = _aligned(ws)
    _check(lib().bfp8_moe_step_host(_p(x), _p(w), _p(dy), _p(offs), E, _p(y), _p(dx), _p(dw), T, N, K,
                                    int(chunk_n), wp, wn, _stream()))
    return y, dx, dw


def check_device_errors() -> None:
    """Synchronises the current stream; raises if a GEMM gave up on a bounded wait."""
    _check(lib().bfp8_check_device_errors(_stream()))


# ---------------------------------------------------------------------------
# Host replay of the kernels' index arithmetic (no GPU)
# ---------------------------------------------------------------------------

def debug_write_counts(kind: int, M: int, N: int, K: int, flag: int = 0):
    """Per-element write counts a launch would produce.  Returns
    (counts [rows, cols], scale_counts or None, out_of_range_writes)."""
    shapes = {0: (M, K), 1: (N, K), 2: (N, K), 3: (M, N), 4: (K, N), 5: (M, K), 6: (K, M)}
    rows, cols = shapes[kind]
    counts = np.zeros((rows, cols), dtype=np.uint32)
    sshape = {0: (_cdiv(K, BLOCK), M), 1: (_cdiv(K, BLOCK), N), 2: (_cdiv(N, BLOCK), _cdiv(K, BLOCK)),
              5: (_cdiv(K, BLOCK), M), 6: (_cdiv(M, BLOCK), K)}.get(kind)
    scounts = np.zeros(sshape, dtype=np.uint32) if sshape else None
    oob = ctypes.c_int64(0)
    _check(lib().bfp8_debug_write_counts(kind, M, N, K, flag, counts.ctypes.data_as(ctypes.c_void_p),
                                         scounts.ctypes.data_as(ctypes.c_void_p) if scounts is not None else None,
                                         ctypes.byref(oob)))
    return counts, scounts, int(oob.value)


def __getattr__(name):
    # the autograd wrapper lives in its own module (it imports torch at load)
    if name in ("Float8BlockwiseLinear", "blockwise_fp8_linear"):
        from . import module
        return getattr(module, name)
    raise AttributeError(name)


"""CPU oracle for blockwise-scaled FP8 quantisation and GEMM.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path
(``blockwise_scaled_fp8_gb300``) never imports this package.

The arithmetic lives in ``bfp8_oracle.c`` (plain C, compiled with gcc without
fast-math or FMA contraction); this module only compiles it, loads it with
ctypes and marshals numpy arrays.  See the header of ``bfp8_oracle.c`` for the
pages each function follows and the readings taken where they are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bfp8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libbfp8_oracle.so")
_lock = threading.Lock()
_lib = None

SB_TILE, SB_TILE_T, SB_COL = 0, 1, 2
BLOCK = 128


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, u64, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
        vp, f32, f64 = ctypes.c_void_p, ctypes.c_float, ctypes.c_double
        lib.ora_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.ora_bf16_to_f32.restype = f32
        lib.ora_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.ora_e4m3_value.restype = f64
        lib.ora_e4m3_rne.argtypes = [f32]
        lib.ora_e4m3_rne.restype = ctypes.c_uint8
        lib.ora_e4m3_nearest.argtypes = [f32]
        lib.ora_e4m3_nearest.restype = ctypes.c_uint8
        lib.ora_sweep_cast.argtypes = [u64, u64, i32, ctypes.POINTER(u64)]
        lib.ora_sweep_cast.restype = u64
        lib.ora_cast_e4m3.argtypes = [vp, i64, vp, i32]
        lib.ora_cast_e4m3.restype = None
        lib.ora_check_cast_range.argtypes = [u64, i64, vp, i32, ctypes.POINTER(u64)]
        lib.ora_check_cast_range.restype = u64
        lib.ora_group_scale.argtypes = [f32]
        lib.ora_group_scale.restype = f32
        lib.ora_quantize_one.argtypes = [f32, f32]
        lib.ora_quantize_one.restype = ctypes.c_uint8
        lib.ora_quant_lhs.argtypes = [vp, i64, i64, i64, i32, vp, i64, vp, i64]
        lib.ora_mx_exponent.argtypes = [f32]
        lib.ora_mx_exponent.restype = i32
        lib.ora_mx_quantize_one.argtypes = [f32, i32]
        lib.ora_mx_quantize_one.restype = ctypes.c_uint8
        lib.ora_mx_cast.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64]
        lib.ora_quant_lhs.restype = None
        lib.ora_quant_rhs.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64]
        lib.ora_quant_rhs.restype = None
        lib.ora_quant_weight.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64]
        lib.ora_quant_weight.restype = None
        lib.ora_gemm.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i32, i64,
                                 vp, i64, vp, i64, vp, i32]
        lib.ora_gemm.restype = None
        lib.ora_sqnr_db.argtypes = [vp, vp, i64]
        lib.ora_sqnr_db.restype = f64
        lib.ora_matmul_bf16_f64.argtypes = [vp, i64, vp, i64, i64, i64, i64, vp]
        lib.ora_matmul_bf16_f64.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


# ---- number formats -------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float32 values."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def e4m3_value(code: int) -> float:
    return _load().ora_e4m3_value(code)


def e4m3_table() -> np.ndarray:
    """Exact value of each of the 256 e4m3fn codes (NaN for 0x7F, 0xFF)."""
    lib = _load()
    return np.array([lib.ora_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_rne(r: float) -> int:
    return _load().ora_e4m3_rne(r)


def e4m3_nearest(r: float) -> int:
    return _load().ora_e4m3_nearest(r)


def sweep_cast(lo: int, hi: int) -> tuple[int, int]:
    """Exhaustive comparison of the rounding rule with a nearest-code search
    over fp32 bit patterns [lo, hi).  Returns (mismatches, first_bad)."""
    first = ctypes.c_uint64(0)
    n = _load().ora_sweep_cast(lo, hi, _threads(), ctypes.byref(first))
    return int(n), int(first.value)


def cast_e4m3(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    _load().ora_cast_e4m3(_ptr(x), x.size, _ptr(q), _threads())
    return q


def check_cast_range(start: int, got: np.ndarray) -> tuple[int, int]:
    """Compare bytes ``got`` (one per fp32 pattern start, start+1, ...) with the
    oracle's rounding.  Returns (mismatches, first_bad_pattern)."""
    got = np.ascontiguousarray(got, dtype=np.uint8)
    first = ctypes.c_uint64(0)
    n = _load().ora_check_cast_range(start, got.size, _ptr(got), _threads(), ctypes.byref(first))
    return int(n), int(first.value)


def group_scale(amax: float) -> float:
    return _load().ora_group_scale(amax)


def quantize_one(x: float, s: float) -> int:
    return _load().ora_quantize_one(x, s)


# ---- quantisation ---------------------------------------------------------

def quant_lhs(x: np.ndarray, transposed: bool = False, ldq: int | None = None,
              lds: int | None = None, q_fill: int = 0, s_fill: float = 0.0):
    """1x128 groups along K of A, where A = x ([M,K]) or x^T (x is [K,M]).
    Returns (q [M, ldq] uint8, s [Kb, lds] float32 -- i.e. column-major [M,Kb])."""
    assert x.dtype == np.uint16 and x.ndim == 2
    x = np.ascontiguousarray(x)
    if transposed:
        K, M = x.shape
    else:
        M, K = x.shape
    Kb = _cdiv(K, BLOCK)
    ldq = ldq or K
    lds = lds or M
    q = np.full((M, ldq), q_fill, dtype=np.uint8)
    s = np.full((Kb, lds), s_fill, dtype=np.float32)
    _load().ora_quant_lhs(_ptr(x), M, K, x.shape[1], int(transposed), _ptr(q), ldq, _ptr(s), lds)
    return q, s


def quant_rhs(x: np.ndarray, ldq: int | None = None, lds: int | None = None,
              q_fill: int = 0, s_fill: float = 0.0):
    """128x1 groups along the rows (reduction dim) of x [K,N].
    Returns (qT [N, ldq] uint8, s [Kb, lds] float32)."""
    assert x.dtype == np.uint16 and x.ndim == 2
    x = np.ascontiguousarray(x)
    K, N = x.shape
    Kb = _cdiv(K, BLOCK)
    ldq = ldq or K
    lds = lds or N
    qT = np.full((N, ldq), q_fill, dtype=np.uint8)
    s = np.full((Kb, lds), s_fill, dtype=np.float32)
    _load().ora_quant_rhs(_ptr(x), K, N, N, _ptr(qT), ldq, _ptr(s), lds)
    return qT, s


def quant_weight(w: np.ndarray, with_t: bool = False, ldq: int | None = None,
                 ldqt: int | None = None, lds: int | None = None, q_fill: int = 0,
                 s_fill: float = 0.0):
    """128x128 tiles of w [N,K].  Returns (q [N,ldq], qt [K,ldqt] or None,
    s [Nb, lds])."""
    assert w.dtype == np.uint16 and w.ndim == 2
    w = np.ascontiguousarray(w)
    N, K = w.shape
    Nb, Kb = _cdiv(N, BLOCK), _cdiv(K, BLOCK)
    ldq = ldq or K
    ldqt = ldqt or N
    lds = lds or Kb
    q = np.full((N, ldq), q_fill, dtype=np.uint8)
    qt = np.full((K, ldqt), q_fill, dtype=np.uint8) if with_t else None
    s = np.full((Nb, lds), s_fill, dtype=np.float32)
    _load().ora_quant_weight(_ptr(w), N, K, K, _ptr(q), ldq, _ptr(qt), ldqt, _ptr(s), lds)
    return q, qt, s


# ---- MXFP8 casts (reading R14: OCP MX v1.0, FLOOR scale) -------------------

MX_BLOCK = 32


def mx_exponent(amax: float) -> int:
    return _load().ora_mx_exponent(amax)


def mx_quantize_one(x: float, e: int) -> int:
    return _load().ora_mx_quantize_one(x, e)


def mx_cast(x: np.ndarray, dim0: bool = True, dim1: bool = True, q_fill: int = 0, e_fill: int = 0):
    """MXFP8 casts of x [M,K] bf16.  Returns (q0 [M,K], e0 [M,ceil(K/32)]) for
    dim0 (blocks of 32 along K) and (q1 [K,M], e1 [K,ceil(M/32)]) for dim1
    (blocks of 32 along M, transposed); None for a cast not asked for.
    Exponents are the biased E8M0 bytes."""
    assert x.dtype == np.uint16 and x.ndim == 2
    x = np.ascontiguousarray(x)
    M, K = x.shape
    q0 = np.full((M, K), q_fill, np.uint8) if dim0 else None
    e0 = np.full((M, max(_cdiv(K, MX_BLOCK), 1)), e_fill, np.uint8) if dim0 else None
    q1 = np.full((K, M), q_fill, np.uint8) if dim1 else None
    e1 = np.full((K, max(_cdiv(M, MX_BLOCK), 1)), e_fill, np.uint8) if dim1 else None
    _load().ora_mx_cast(_ptr(x), M, K, K, _ptr(q0), K, _ptr(e0), e0.shape[1] if dim0 else 0,
                        _ptr(q1), M, _ptr(e1), e1.shape[1] if dim1 else 0)
    return (q0, e0), (q1, e1)


# ---- GEMM -----------------------------------------------------------------

def gemm(qa: np.ndarray, sa: np.ndarray, qb: np.ndarray, sb: np.ndarray, sb_mode: int,
         K: int, rows=None, cols=None) -> np.ndarray:
    """Blockwise-scaled GEMM in fp64.  qa [M, lda] uint8, sa [Kb, ldsa] (column-
    major a_s), qb [N, ldb] uint8 (B^T, K contiguous), sb per ``sb_mode``.
    Returns C[rows][:, cols] as float64."""
    qa = np.ascontiguousarray(qa)
    qb = np.ascontiguousarray(qb)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    M, N = qa.shape[0], qb.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    out = np.empty((rows.size, cols.size), dtype=np.float64)
    if rows.size == 0 or cols.size == 0:
        return out
    _load().ora_gemm(_ptr(qa), qa.shape[1], _ptr(sa), sa.shape[1], _ptr(qb), qb.shape[1],
                     _ptr(sb), sb.shape[1], sb_mode, K, _ptr(rows), rows.size, _ptr(cols),
                     cols.size, _ptr(out), _threads())
    return out


def sqnr_db(ref: np.ndarray, out: np.ndarray) -> float:
    ref = np.ascontiguousarray(ref, dtype=np.float64)
    out = np.ascontiguousarray(out, dtype=np.float64)
    return _load().ora_sqnr_db(_ptr(ref), _ptr(out), ref.size)


def matmul_bf16_f64(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """fp64 C = x w^T of bf16 inputs x [M,K], w [N,K]."""
    x = np.ascontiguousarray(x)
    w = np.ascontiguousarray(w)
    M, K = x.shape
    N = w.shape[0]
    out = np.empty((M, N), dtype=np.float64)
    _load().ora_matmul_bf16_f64(_ptr(x), K, _ptr(w), K, M, N, K, _ptr(out))
    return out


# ---- whole linear (composition of the steps above) -------------------------

def linear_fwd(x: np.ndarray, w: np.ndarray, rows=None, cols=None) -> np.ndarray:
    """y = x W^T through the blockwise FP8 path: x quantised 1x128 along K,
    W quantised in 128x128 tiles, GEMM 1x128 x 128x128."""
    K = x.shape[1]
    qa, sa = quant_lhs(x)
    qb, _, sb = quant_weight(w)
    return gemm(qa, sa, qb, sb, SB_TILE, K, rows, cols)


def linear_dgrad(dy: np.ndarray, w: np.ndarray, rows=None, cols=None) -> np.ndarray:
    """dX = dY W: dY quantised 1x128 along N_out, W's 128x128 tiles read
    transposed (qt, with the tile scales addressed [kb, nb])."""
    N = dy.shape[1]
    qa, sa = quant_lhs(dy)
    _, qt, sw = quant_weight(w, with_t=True)
    return gemm(qa, sa, qt, sw, SB_TILE_T, N, rows, cols)


def linear_wgrad(dy: np.ndarray, x: np.ndarray, rows=None, cols=None) -> np.ndarray:
    """dW = dY^T X: dY^T quantised 1x128 along the token dim, X quantised 128x1
    along the token dim (written transposed), GEMM 1x128 x 128x1."""
    T = dy.shape[0]
    qa, sa = quant_lhs(dy, transposed=True)
    qbT, sb = quant_rhs(x)
    return gemm(qa, sa, qbT, sb, SB_COL, T, rows, cols)


# ---- grouped (mixture-of-experts) GEMMs -------------------------------------
#
# The pages name a mixture-of-experts path beside the dense one ("Enable
# blockwise FP8 dense training kernels on ROCm", description: the same
# FP8_MAX fix made for the MoE path) without spelling it out.  Reading taken
# here: tokens are sorted by expert, expert e owns token rows
# offs[e] .. offs[e+1] (non-decreasing offsets), and each expert's linear is
# exactly the dense method on its slice: forward and input gradient are one
# dense GEMM per expert on its token rows; the weight gradient of expert e
# reduces over its own tokens only.  So that the 128-token quantisation groups
# along the token dim never mix two experts, the weight gradient requires every
# expert to start on a 128-token boundary (offs[e] % 128 == 0 for e < E).
# Expert weights are stacked as [E*N, K] with N % 128 == 0, so their 128x128
# tiles never mix two experts either.

def _group_bounds(offs, e):
    return int(offs[e]), int(offs[e + 1])


def moe_gemm_fwd(qa: np.ndarray, sa: np.ndarray, qw: np.ndarray, sw: np.ndarray,
                 offs, N: int, K: int) -> np.ndarray:
    """y[offs[e]:offs[e+1]] = (tokens of expert e) W_e^T for every expert:
    qa [M_total, lda] 1x128 codes, sa [Kb, ldsa] column-major a_s, qw the
    stacked expert weights' tile codes [E*N, K], sw their tile scales
    [E*Nb, Kb].  Rows past offs[E] are not defined (NaN)."""
    E = len(offs) - 1
    Nb = _cdiv(N, BLOCK)
    out = np.full((qa.shape[0], N), np.nan)
    for e in range(E):
        r0, r1 = _group_bounds(offs, e)
        if r1 > r0:
            out[r0:r1] = gemm(qa[r0:r1], sa[:, r0:r1], qw[e * N:(e + 1) * N], sw[e * Nb:(e + 1) * Nb],
                              SB_TILE, K)
    return out


def moe_gemm_dgrad(qdy: np.ndarray, sdy: np.ndarray, qwt: np.ndarray, sw: np.ndarray,
                   offs, N: int, K: int) -> np.ndarray:
    """dx[offs[e]:offs[e+1]] = dY_e W_e: qdy [M_total, N] codes of dY (1x128
    along N), sdy [Nb, ldsa]; qwt [K, E*N] the stacked weights' transposed
    tile codes (expert e in columns e*N .. (e+1)*N), sw [E*Nb, Kb] read
    transposed."""
    E = len(offs) - 1
    Nb = _cdiv(N, BLOCK)
    out = np.full((qdy.shape[0], K), np.nan)
    for e in range(E):
        r0, r1 = _group_bounds(offs, e)
        if r1 > r0:
            out[r0:r1] = gemm(qdy[r0:r1], sdy[:, r0:r1], qwt[:, e * N:(e + 1) * N],
                              sw[e * Nb:(e + 1) * Nb], SB_TILE_T, N)
    return out


def moe_gemm_wgrad(qdyt: np.ndarray, sdyt: np.ndarray, qxt: np.ndarray, sxt: np.ndarray,
                   offs) -> np.ndarray:
    """dW[e] = dY_e^T X_e, reduced over expert e's tokens only: qdyt [N, ld]
    codes of dY^T (1x128 along tokens), sdyt [Tb, ldsa] column-major; qxt
    [K, ld] codes of X (128x1 along tokens, transposed), sxt [Tb, ldsb].
    Returns dW [E, N, K]; an expert without tokens gets zeros."""
    E = len(offs) - 1
    N, K = qdyt.shape[0], qxt.shape[0]
    out = np.zeros((E, N, K))
    for e in range(E):
        t0, t1 = _group_bounds(offs, e)
        if t1 > t0:
            assert t0 % BLOCK == 0, "an expert's tokens must start on a 128-token boundary"
            b0, b1 = t0 // BLOCK, _cdiv(t1, BLOCK)
            out[e] = gemm(qdyt[:, t0:t1], sdyt[b0:b1], qxt[:, t0:t1], sxt[b0:b1], SB_COL, t1 - t0)
    return out


def moe_linear_fwd(x: np.ndarray, w: np.ndarray, offs) -> np.ndarray:
    """Per expert, the dense method's forward on its tokens: x [M_total, K]
    bf16, w [E, N, K] bf16."""
    out = np.full((x.shape[0], w.shape[1]), np.nan)
    for e in range(len(offs) - 1):
        r0, r1 = _group_bounds(offs, e)
        if r1 > r0:
            out[r0:r1] = linear_fwd(x[r0:r1], w[e])
    return out


def moe_linear_dgrad(dy: np.ndarray, w: np.ndarray, offs) -> np.ndarray:
    out = np.full((dy.shape[0], w.shape[2]), np.nan)
    for e in range(len(offs) - 1):
        r0, r1 = _group_bounds(offs, e)
        if r1 > r0:
            out[r0:r1] = linear_dgrad(dy[r0:r1], w[e])
    return out


def moe_linear_wgrad(dy: np.ndarray, x: np.ndarray, offs) -> np.ndarray:
    E = len(offs) - 1
    out = np.zeros((E, dy.shape[1], x.shape[1]))
    for e in range(E):
        r0, r1 = _group_bounds(offs, e)
        if r1 > r0:
            out[e] = linear_wgrad(dy[r0:r1], x[r0:r1])
    return out

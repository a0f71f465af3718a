"""Host-side tests of the C ABI (no GPU): the library loads and exports every
declared symbol, argument validation rejects bad calls before anything is
launched, and the kernels' own index arithmetic (replayed on the host) writes
every element of the logical outputs exactly once and nothing outside them —
the scale-bounds test idea of "Mask a_s/b_s scale loads in blockwise FP8
training GEMM kernels", generalised from "at least once" to "exactly once"."""
import ctypes
import os
import re

import numpy as np
import pytest

import blockwise_scaled_fp8_gb300 as B
from blockwise_scaled_fp8_gb300 import buildlib as bbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    bbuild.build()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "bfp8.h")).read()
    return sorted(set(re.findall(r"\b(bfp8_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    L = B.lib()
    declared = _declared_symbols()
    assert set(declared) == set(B.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


NULL = ctypes.c_void_p(None)
P16 = ctypes.c_void_p(0x10000)      # fake, 16-byte aligned; never dereferenced
P_ODD = ctypes.c_void_p(0x10001)


def test_quant_argument_validation():
    L = B.lib()
    s = L.bfp8_quant_lhs
    assert s(NULL, 4, 128, 128, 0, P16, 128, P16, 4, NULL) == B.BFP8_ERR_INVALID_ARG
    assert s(P16, 4, 128, 100, 0, P16, 128, P16, 4, NULL) == B.BFP8_ERR_INVALID_ARG      # ldx < K
    assert s(P16, 4, 128, 128, 0, P16, 136, P16, 4, NULL) == B.BFP8_ERR_INVALID_ARG      # ldq % 16
    assert s(P16, 4, 128, 128, 0, P16, 128, P16, 3, NULL) == B.BFP8_ERR_INVALID_ARG      # lds < M
    assert s(P16, 4, 128, 128, 0, P_ODD, 128, P16, 4, NULL) == B.BFP8_ERR_INVALID_ARG    # q misaligned
    assert s(P16, 4, 128, 2, 1, P16, 128, P16, 4, NULL) == B.BFP8_ERR_INVALID_ARG        # transposed: ldx < M
    assert s(P16, -1, 128, 128, 0, P16, 128, P16, 4, NULL) == B.BFP8_ERR_INVALID_ARG
    assert s(P16, 0, 128, 128, 0, P16, 128, P16, 4, NULL) == B.BFP8_OK                   # empty: no-op
    r = L.bfp8_quant_rhs
    assert r(P16, 256, 64, 32, P16, 256, P16, 64, NULL) == B.BFP8_ERR_INVALID_ARG          # ldx < N
    assert r(P16, 256, 64, 64, P16, 256, P16, 63, NULL) == B.BFP8_ERR_INVALID_ARG          # lds < N
    w = L.bfp8_quant_weight
    assert w(P16, 64, 256, 256, NULL, 0, NULL, 0, P16, 2, NULL) == B.BFP8_ERR_INVALID_ARG  # no output
    assert w(P16, 64, 256, 256, P16, 256, NULL, 0, P16, 1, NULL) == B.BFP8_ERR_INVALID_ARG # lds < Kb
    assert w(P16, 64, 256, 256, NULL, 0, P16, 40, P16, 2, NULL) == B.BFP8_ERR_INVALID_ARG  # ldqt < N
    assert L.bfp8_cast_e4m3(NULL, 5, P16, NULL) == B.BFP8_ERR_INVALID_ARG


def test_gemm_argument_validation():
    L = B.lib()
    g = L.bfp8_gemm_1x128_128x128
    ok_args = [P16, 256, P16, 8, P16, 256, P16, 2, 0, P16, 64, 8, 64, 256, NULL]

    def call(**kw):
        a = list(ok_args)
        names = ["qa", "lda", "sa", "ldsa", "qb", "ldb", "sb", "ldsb", "t", "c", "ldc", "M", "N", "K", "st"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return g(*a)

    assert call(lda=200) == B.BFP8_ERR_INVALID_ARG          # lda < K
    assert call(lda=264) == B.BFP8_ERR_INVALID_ARG          # not a multiple of 16
    assert call(ldb=260) == B.BFP8_ERR_INVALID_ARG          # not a multiple of 16
    assert call(ldsa=7) == B.BFP8_ERR_INVALID_ARG           # ldsa < M
    assert call(ldsb=1) == B.BFP8_ERR_INVALID_ARG           # ldsb < Kb
    assert call(t=1, ldsb=0) == B.BFP8_ERR_INVALID_ARG      # transposed: ldsb < Nb
    assert call(ldc=32) == B.BFP8_ERR_INVALID_ARG           # ldc < N
    assert call(qa=P_ODD) == B.BFP8_ERR_INVALID_ARG
    assert call(c=NULL) == B.BFP8_ERR_INVALID_ARG
    assert call(M=0) == B.BFP8_OK
    h = L.bfp8_gemm_1x128_128x1
    assert h(P16, 256, P16, 8, P16, 256, P16, 63, P16, 64, 8, 64, 256, NULL) == B.BFP8_ERR_INVALID_ARG  # ldsb < N


def test_xq_gemm_argument_validation():
    """The GEMM that quantises its bf16 A itself checks x's row stride (TMA:
    a multiple of 8 bf16 values, at least K) and alignment before launching."""
    L = B.lib()
    g = L.bfp8_gemm_1x128_128x128_xq
    ok_args = [P16, 256, P16, 256, P16, 2, P16, 64, 8, 64, 256, NULL]
    names = ["x", "ldx", "qb", "ldb", "sb", "ldsb", "c", "ldc", "M", "N", "K", "st"]

    def call(**kw):
        a = list(ok_args)
        for k, v in kw.items():
            a[names.index(k)] = v
        return g(*a)

    assert call(ldx=200) == B.BFP8_ERR_INVALID_ARG          # ldx < K
    assert call(ldx=260) == B.BFP8_ERR_INVALID_ARG          # not a multiple of 8 (TMA row stride)
    assert call(ldb=264) == B.BFP8_ERR_INVALID_ARG          # not a multiple of 16
    assert call(ldsb=1) == B.BFP8_ERR_INVALID_ARG           # ldsb < Kb
    assert call(ldc=32) == B.BFP8_ERR_INVALID_ARG           # ldc < N
    assert call(x=P_ODD) == B.BFP8_ERR_INVALID_ARG          # x not 16-byte aligned
    assert call(x=NULL) == B.BFP8_ERR_INVALID_ARG
    assert call(M=-1) == B.BFP8_ERR_INVALID_ARG
    assert call(M=0) == B.BFP8_OK


def test_wgrad_xq_gemm_argument_validation():
    """The weight-gradient GEMM that quantises its bf16 rhs itself checks x's
    row stride (TMA: a multiple of 8 bf16 values, at least N), the A operand's
    stride and alignment before launching."""
    L = B.lib()
    g = L.bfp8_gemm_1x128_128x1_xq
    ok_args = [P16, 256, P16, 64, P16, 512, P16, 512, 64, 512, 256, NULL]
    names = ["qa", "lda", "sa", "ldsa", "x", "ldx", "c", "ldc", "M", "N", "K", "st"]

    def call(**kw):
        a = list(ok_args)
        for k, v in kw.items():
            a[names.index(k)] = v
        return g(*a)

    assert call(ldx=500) == B.BFP8_ERR_INVALID_ARG          # ldx < N
    assert call(ldx=516) == B.BFP8_ERR_INVALID_ARG          # not a multiple of 8 (TMA row stride)
    assert call(lda=200) == B.BFP8_ERR_INVALID_ARG          # lda < K
    assert call(lda=264) == B.BFP8_ERR_INVALID_ARG          # not a multiple of 16
    assert call(ldsa=32) == B.BFP8_ERR_INVALID_ARG          # ldsa < M
    assert call(ldc=256) == B.BFP8_ERR_INVALID_ARG          # ldc < N
    assert call(x=P_ODD) == B.BFP8_ERR_INVALID_ARG          # x not 16-byte aligned
    assert call(qa=P_ODD) == B.BFP8_ERR_INVALID_ARG         # qa not 16-byte aligned
    assert call(x=NULL) == B.BFP8_ERR_INVALID_ARG
    assert call(sa=NULL) == B.BFP8_ERR_INVALID_ARG
    assert call(K=-1) == B.BFP8_ERR_INVALID_ARG
    assert call(N=0) == B.BFP8_OK


def test_grouped_and_fused_argument_validation():
    """Host-side checks of the grouped GEMMs and of the one-launch
    quantisation: every rejection happens before anything is launched."""
    L = B.lib()
    g = L.bfp8_gemm_grouped_1x128_128x128
    #       qa   lda  sa   ldsa qb   ldb  sb   ldsb t  offs E  c    ldc Mt   N    K    st
    ok = [P16, 256, P16, 512, P16, 256, P16, 2, 0, P16, 4, P16, 64, 512, 64, 256, NULL]
    names = ["qa", "lda", "sa", "ldsa", "qb", "ldb", "sb", "ldsb", "t", "offs", "E", "c", "ldc", "Mt", "N", "K", "st"]

    def call(**kw):
        a = list(ok)
        for k, v in kw.items():
            a[names.index(k)] = v
        return g(*a)

    assert call(E=0) == B.BFP8_ERR_INVALID_ARG             # no expert
    assert call(E=1025) == B.BFP8_ERR_INVALID_ARG          # more than 1024 experts
    assert call(offs=NULL) == B.BFP8_ERR_INVALID_ARG
    assert call(offs=P_ODD) == B.BFP8_ERR_INVALID_ARG       # offsets not 4-byte aligned
    assert call(lda=200) == B.BFP8_ERR_INVALID_ARG          # lda < K
    assert call(ldsa=511) == B.BFP8_ERR_INVALID_ARG         # ldsa < M_total
    assert call(ldc=32) == B.BFP8_ERR_INVALID_ARG           # ldc < N
    assert call(t=1, K=200, ldb=1024) == B.BFP8_ERR_INVALID_ARG  # input gradient: K % 16 with E > 1
    assert call(t=1, ldb=512) == B.BFP8_ERR_INVALID_ARG     # input gradient: ldb < E*K
    assert call(Mt=0) == B.BFP8_OK                          # no tokens: nothing to do
    r = L.bfp8_gemm_grouped_1x128_128x1
    #          qa   lda  sa   ldsa qb   ldb  sb   ldsb offs E  c    ldc cstride M   N   T    st
    assert r(P16, 512, P16, 64, P16, 512, P16, 64, P16, 4, P16, 64, 64 * 64 - 1, 64, 64, 512, NULL) == \
        B.BFP8_ERR_INVALID_ARG                              # expert stride < M*ldc
    assert r(P16, 500, P16, 64, P16, 512, P16, 64, P16, 4, P16, 64, 64 * 64, 64, 64, 512, NULL) == \
        B.BFP8_ERR_INVALID_ARG                              # lda < T
    f = L.bfp8_quant_dual_weight
    #            x    T    C    ldx  qr   ldqr sr   ldsr qc   ldqc sc   ldsc w    N   ldw  qw   ldqw qwt  ldqwt sw  ldsw st
    args = [P16, 128, 256, 256, P16, 256, P16, 128, P16, 128, P16, 256, P16, 64, 256, P16, 256, P16, 64, P16, 2, NULL]
    assert f(*args[:12], NULL, *args[13:]) == B.BFP8_ERR_INVALID_ARG           # no w
    bad = list(args); bad[18] = 40
    assert f(*bad) == B.BFP8_ERR_INVALID_ARG                                   # ldqwt < N
    bad = list(args); bad[20] = 1
    assert f(*bad) == B.BFP8_ERR_INVALID_ARG                                   # ldsw < Kb
    bad = list(args); bad[14] = 200
    assert f(*bad) == B.BFP8_ERR_INVALID_ARG                                   # ldw < C


def test_mx_cast_argument_validation():
    L = B.lib()
    f = L.bfp8_mx_cast
    #          x    M   K    ldx  q0   ldq0 e0   lde0 q1   ldq1 e1   lde1 st
    ok = [P16, 64, 256, 256, P16, 256, P16, 8, P16, 64, P16, 2, NULL]
    assert f(*ok[:4], NULL, 0, NULL, 0, NULL, 0, NULL, 0, NULL) == B.BFP8_ERR_INVALID_ARG   # no output
    bad = list(ok); bad[6] = NULL
    assert f(*bad) == B.BFP8_ERR_INVALID_ARG                     # codes without exponents
    bad = list(ok); bad[5] = 264
    assert f(*bad) == B.BFP8_ERR_INVALID_ARG                     # ldq0 not a multiple of 16
    bad = list(ok); bad[7] = 7
    assert f(*bad) == B.BFP8_ERR_INVALID_ARG                     # lde0 < ceil(K/32)
    bad = list(ok); bad[11] = 1
    assert f(*bad) == B.BFP8_ERR_INVALID_ARG                     # lde1 < ceil(M/32)
    bad = list(ok); bad[3] = 260
    assert f(*bad) == B.BFP8_ERR_INVALID_ARG                     # ldx not a multiple of 8 (no TMA path)
    bad = list(ok); bad[1] = 0
    assert f(*bad) == B.BFP8_OK                                  # empty: nothing to do


def test_linear_workspace_and_validation():
    L = B.lib()
    assert L.bfp8_linear_workspace_size(0, 10, 10) == 0
    M, N, K = 130, 384, 256
    ws = L.bfp8_linear_workspace_size(M, N, K)
    assert ws > M * K + N * K
    assert L.bfp8_linear_fwd(P16, P16, P16, M, N, K, ctypes.c_void_p(0x10010), ws, NULL) == B.BFP8_ERR_INVALID_ARG
    assert L.bfp8_linear_fwd(P16, P16, P16, M, N, K, ctypes.c_void_p(0x10000), ws - 1, NULL) == B.BFP8_ERR_INVALID_ARG


def test_moe_step_host_validation():
    """The mixture-of-experts host step checks its host offsets and workspace
    before it touches a device."""
    L = B.lib()
    N, K, T = 256, 384, 640
    ws = L.bfp8_moe_step_host_workspace_size(384, N, K)
    assert ws == 2 * L.bfp8_linear_step_host_workspace_size(384, N, K)
    W = ctypes.c_void_p(0x100000)
    f = L.bfp8_moe_step_host

    def call(offs, E=None, T_=T, n=ws, chunk=0):
        o = (ctypes.c_int32 * len(offs))(*offs)
        E = len(offs) - 1 if E is None else E
        return f(P16, P16, P16, o, E, P16, P16, P16, T_, N, K, chunk, W, n, NULL)

    assert call([0, 384, 384, 640], n=ws - 1) == B.BFP8_ERR_INVALID_ARG         # workspace too small
    assert call([0, 400, 300, 640]) == B.BFP8_ERR_INVALID_ARG                   # decreasing offsets
    assert "decrease" in L.bfp8_last_error().decode()
    assert call([0, 384, 700]) == B.BFP8_ERR_INVALID_ARG                        # past T
    assert call([-1, 384, 640]) == B.BFP8_ERR_INVALID_ARG                       # negative
    assert call([0, 384, 640], chunk=100) == B.BFP8_ERR_INVALID_ARG             # chunk not a multiple of 128
    assert call([0, 640], E=0) == B.BFP8_ERR_INVALID_ARG                        # no expert


def test_linear_step_host_workspace_and_validation():
    """The host-buffer training step rejects bad arguments before it touches
    a device or enqueues a copy."""
    L = B.lib()
    assert L.bfp8_linear_step_host_workspace_size(0, 10, 10) == 0
    M, N, K = 256, 1152, 384
    ws = L.bfp8_linear_step_host_workspace_size(M, N, K)
    # device copies of x, W, dY, y, dX, dW plus the training form's quantised operands
    assert ws >= 2 * (2 * M * K + 2 * N * K + 2 * M * N) + L.bfp8_linear_train_workspace_size(M, N, K)
    W = ctypes.c_void_p(0x100000)  # 256-byte aligned, never dereferenced
    f = L.bfp8_linear_step_host

    def call(**kw):
        a = dict(x=P16, w=P16, dy=P16, y=P16, dx=P16, dw=P16, M=M, N=N, K=K, chunk=0, ws=W, n=ws)
        a.update(kw)
        return f(a["x"], a["w"], a["dy"], a["y"], a["dx"], a["dw"], a["M"], a["N"], a["K"], a["chunk"],
                 a["ws"], a["n"], NULL)

    assert call(chunk=100) == B.BFP8_ERR_INVALID_ARG         # not a multiple of 128
    assert "chunk_n" in L.bfp8_last_error().decode()
    assert call(chunk=-128) == B.BFP8_ERR_INVALID_ARG
    assert call(N=128 * 65, chunk=128,
                n=L.bfp8_linear_step_host_workspace_size(M, 128 * 65, K)) == B.BFP8_ERR_INVALID_ARG  # > 64 chunks
    assert call(n=ws - 1) == B.BFP8_ERR_INVALID_ARG           # workspace too small
    assert call(ws=ctypes.c_void_p(0x100010)) == B.BFP8_ERR_INVALID_ARG  # workspace not 256-byte aligned
    assert call(dy=NULL) == B.BFP8_ERR_INVALID_ARG
    assert call(dw=NULL) == B.BFP8_ERR_INVALID_ARG
    assert call(M=0) == B.BFP8_ERR_INVALID_ARG
    assert call(K=-1) == B.BFP8_ERR_INVALID_ARG


SHAPES = [(1, 1, 1), (2, 512, 128), (4, 3584, 640), (130, 384, 256), (129, 130, 131), (257, 65, 300),
          (300, 7, 1000), (1, 1000, 8), (128, 256, 128), (640, 5120, 1280)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("plain", [0, 2])
def test_quant_lhs_index_replay_exactly_once(M, N, K, plain):
    for flag in (0, 1):
        c, s, oob = B.debug_write_counts(0, M, N, K, flag | plain)
        assert oob == 0 and c.shape == (M, K) and np.all(c == 1)
        assert np.all(s == 1)


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("plain", [0, 2])
def test_quant_rhs_and_weight_index_replay_exactly_once(M, N, K, plain):
    c, s, oob = B.debug_write_counts(1, M, N, K, plain)
    assert oob == 0 and np.all(c == 1) and np.all(s == 1)
    c, s, oob = B.debug_write_counts(2, M, N, K, plain)
    assert oob == 0 and np.all(c == 1) and np.all(s == 1)
    c, _, oob = B.debug_write_counts(4, M, N, K, plain)
    assert oob == 0 and c.shape == (K, N) and np.all(c == 1)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_quant_dual_index_replay_exactly_once(M, N, K):
    c, s, oob = B.debug_write_counts(5, M, N, K)
    assert oob == 0 and c.shape == (M, K) and np.all(c == 1) and np.all(s == 1)
    c, s, oob = B.debug_write_counts(6, M, N, K)
    assert oob == 0 and c.shape == (K, M) and np.all(c == 1) and np.all(s == 1)


@pytest.mark.parametrize("M,N,K", SHAPES + [(128, 2048, 2048), (300, 384, 4096), (2, 5120, 1280), (64, 1000, 2048),
                                             (4096, 4096, 128), (2048, 4096, 128), (16384, 1024, 128),
                                             (2048, 4096, 4096), (2000, 4000, 520), (4096, 4096, 8192),
                                             (2048, 4100, 256), (1900, 4090, 128),
                                             (1, 130, 8192), (16, 4096, 4096), (5, 2051, 1100),
                                             (12, 19456, 256), (2, 19584, 256)])
@pytest.mark.parametrize("col_scales", [0, 8])
def test_gemm_epilogue_index_replay_exactly_once(M, N, K, col_scales):
    """The persistent tile schedule stores each output element once (both
    promotion-warp layouts)."""
    c, _, oob = B.debug_write_counts(3, M, N, K, col_scales)
    assert oob == 0 and np.all(c == 1)


def test_launch_policy_programmatic_dependent_launch():
    """Which launches overlap their set-up with the kernel before them (host
    logic): the short kernels of a 2048 x 4096 x 4096 linear step and of small
    problems do, the long ones of the 8192-token and 16384 x 14336 x 4096
    steps do not (measured faster without it)."""
    pdl = lambda kind, a, b=0, c=0: B.lib().bfp8_debug_launch_pdl(kind, a, b, c)
    assert pdl(0, 2048, 4096, 4096) == 1 and pdl(0, 2, 4096, 4096) == 1 and pdl(0, 512, 4096, 4096) == 1
    assert pdl(0, 4096, 4096, 4096) == 0                 # exactly 2^37 FLOPs
    assert pdl(0, 4096, 4096, 8192) == 0 and pdl(0, 16384, 14336, 4096) == 0 and pdl(0, 14336, 4096, 16384) == 0
    mib = 1 << 20
    assert pdl(1, 2 * 2048 * 4096 + 2 * 4096 * 4096) == 1   # x with W, 2048 x 4096 and 4096 x 4096: 48 MiB
    assert pdl(1, 64 * mib - 2) == 1 and pdl(1, 64 * mib) == 0
    assert pdl(1, 2 * 16384 * 14336) == 0                 # dY at MLP-up
    assert pdl(2, 1) == -1 and pdl(0, -1, 1, 1) == -1


def test_gemm_tile_width_choice():
    """Tile widths the launcher picks (host logic, 152 SMs): narrow tiles for
    problems that fill few SMs (1x128 x 128x128 only) -- 32 columns where
    those tiles fit in one wave, else 64 --, 224 columns for the 1x128 x 128x1
    GEMM where they fill the last wave of SMs better than 256, else 256 or
    128."""
    pick = lambda M, N, col=False: B.lib().bfp8_debug_gemm_pick_bn(M, N, int(col), 152)
    assert pick(128, 4096) == 32 and pick(33, 4864) == 32      # 128 / 152 tiles of 32: one wave
    assert pick(256, 2432) == 32 and pick(128, 512) == 32
    assert pick(33, 4865) == 64 and pick(128, 5120) == 64      # 153 / 160 tiles of 32; 38 / 40 of 128
    assert pick(2, 4096, True) == 128                          # the 128x1 GEMM never narrows
    assert pick(2048, 4096) == 256 and pick(2048, 4096, True) == 224   # 256 tiles = 1.68 waves; 304 = 2
    assert pick(4096, 4096, True) == 224                       # 512 tiles = 3.37 waves; 608 = 4
    assert pick(16384, 14336) == 256 and pick(14336, 4096, True) == 256   # many waves: 256 kept
    assert pick(16384, 4096) == 256 and pick(8192, 8192) == 256
    assert pick(512, 4096) == 128                              # 64 tiles of 256 < 152 SMs

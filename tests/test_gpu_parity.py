"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Quantised bytes and scales must match bit for bit; GEMM outputs must satisfy
|gpu - oracle| <= 2^-7 |oracle| + 1e-3 rms(oracle) element by element.
Every output buffer sits inside a guard band pre-filled with a sentinel, with
padding past the logical width, so a write outside the logical tensor shows
up as a changed sentinel (the unmasked-store bugs the pages describe).
"""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from gpu_util import assert_gemm_close, dev_bf16, host_bf16_as_f64, sqnr_db, torch

import blockwise_scaled_fp8_gb300 as B

pytestmark = pytest.mark.gpu

GUARD = 4096
SENT_U8 = 0xA5
SENT_F32_BITS = 0x7FC0DEAD  # a NaN pattern no kernel produces


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    B.build()
    O.build()
    yield
    B.check_device_errors()


def cdiv(a, b):
    return (a + b - 1) // b


def rup(a, b):
    return cdiv(a, b) * b


class Guarded:
    """A 2-D device buffer [rows, ld] inside a sentinel-filled guard band."""

    def __init__(self, rows, ld, dtype):
        self.rows, self.ld, self.dtype = rows, ld, dtype
        n = rows * ld
        if dtype == torch.uint8:
            self.flat = torch.full((n + 2 * GUARD,), SENT_U8, dtype=torch.uint8, device="cuda")
        else:
            self.flat = torch.full((n + 2 * GUARD,), SENT_F32_BITS, dtype=torch.int32, device="cuda").view(torch.float32)
        self.t = self.flat[GUARD:GUARD + n].view(rows, ld)

    def check_outside(self, cols):
        """Sentinels intact in the guard bands and in columns [cols, ld)."""
        f = self.flat.view(torch.uint8) if self.dtype == torch.uint8 else self.flat.view(torch.int32)
        sent = SENT_U8 if self.dtype == torch.uint8 else SENT_F32_BITS
        h = f.cpu().numpy()
        assert np.all(h[:GUARD] == sent) and np.all(h[-GUARD:] == sent), "write outside the buffer"
        body = h[GUARD:GUARD + self.rows * self.ld].reshape(self.rows, self.ld)
        assert np.all(body[:, cols:] == sent), "write into row padding"


def f32_bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


# ------------------------------------------------------------------ the cast

def test_cast_exhaustive_all_fp32_patterns():
    """The device's rounding step equals the oracle's RNE_e4m3 (with the clamp)
    on every non-NaN fp32 bit pattern."""
    n = 1 << 28
    for c in range(16):
        start = c << 28
        lo = start if start < (1 << 31) else start - (1 << 32)   # the same bits as int32
        x = (torch.arange(n, dtype=torch.int32, device="cuda") + lo).view(torch.float32)
        q = B.cast_e4m3(x).cpu().numpy()
        bad, first = O.check_cast_range(start, q)
        assert bad == 0, f"chunk {c}: {bad} mismatches, first pattern 0x{first:08x}"


# ------------------------------------------------------------------ quant_lhs

LHS_SHAPES = [(130, 256), (2, 128), (4, 640), (128, 4096), (512, 1280), (4096, 1024), (300, 1000),
              (3, 136), (5, 72), (1, 1), (7, 77), (2048, 8192)]


def _run_lhs(x, transposed, lds_extra):
    M, K = (x.shape[1], x.shape[0]) if transposed else x.shape
    Kb = cdiv(K, 128)
    ldq, lds = rup(K, 16) + 16, M + lds_extra
    qg, sg = Guarded(M, ldq, torch.uint8), Guarded(Kb, lds, torch.float32)
    B.quant_lhs(dev_bf16(x), transposed=transposed, q=qg.t, s=sg.t)
    torch.cuda.synchronize()
    return qg, sg, M, K


@pytest.mark.parametrize("M,K", LHS_SHAPES)
@pytest.mark.parametrize("lds_extra", [0, 3])
def test_quant_lhs_bit_exact(M, K, lds_extra):
    x = S.normal_bf16((M, K), 1.0, seed=M * 31 + K, outlier_frac=1e-3)
    qg, sg, _, _ = _run_lhs(x, False, lds_extra)
    q_ref, s_ref = O.quant_lhs(x)
    assert np.array_equal(qg.t.cpu().numpy()[:, :K], q_ref)
    assert np.array_equal(f32_bits(sg.t.cpu().numpy()[:, :M]), f32_bits(s_ref))
    qg.check_outside(K)
    sg.check_outside(M)


TLHS_SHAPES = [(256, 130), (300, 70), (129, 64), (128, 1), (1000, 9), (8192, 4096), (16, 4100)]


@pytest.mark.parametrize("T,C", TLHS_SHAPES)
def test_quant_lhs_transposed_bit_exact(T, C):
    """dY^T quantised 1x128 along the token dimension (x is [T, C])."""
    x = S.normal_bf16((T, C), 1e-3, seed=T + 7 * C)
    qg, sg, M, K = _run_lhs(x, True, 1)
    q_ref, s_ref = O.quant_lhs(x, transposed=True)
    assert np.array_equal(qg.t.cpu().numpy()[:, :K], q_ref)
    assert np.array_equal(f32_bits(sg.t.cpu().numpy()[:, :M]), f32_bits(s_ref))
    qg.check_outside(K)
    sg.check_outside(M)


RHS_SHAPES = [(260, 70), (8192, 4096), (128, 8), (1000, 130), (1, 5), (4096, 1024)]


@pytest.mark.parametrize("K,N", RHS_SHAPES)
def test_quant_rhs_bit_exact(K, N):
    x = S.normal_bf16((K, N), 1.0, seed=K + 3 * N)
    Kb = cdiv(K, 128)
    ldq, lds = rup(K, 16) + 32, N + 4
    qg, sg = Guarded(N, ldq, torch.uint8), Guarded(Kb, lds, torch.float32)
    B.quant_rhs(dev_bf16(x), q=qg.t, s=sg.t)
    torch.cuda.synchronize()
    q_ref, s_ref = O.quant_rhs(x)
    assert np.array_equal(qg.t.cpu().numpy()[:, :K], q_ref)
    assert np.array_equal(f32_bits(sg.t.cpu().numpy()[:, :N]), f32_bits(s_ref))
    qg.check_outside(K)
    sg.check_outside(N)


W_SHAPES = [(384, 256), (300, 260), (4096, 4096), (5120, 1280), (3584, 640), (7, 9), (129, 1000)]


@pytest.mark.parametrize("N,K", W_SHAPES)
def test_quant_weight_bit_exact(N, K):
    w = S.normal_bf16((N, K), 0.02, seed=N + K)
    Nb, Kb = cdiv(N, 128), cdiv(K, 128)
    qg = Guarded(N, rup(K, 16) + 16, torch.uint8)
    tg = Guarded(K, rup(N, 16) + 16, torch.uint8)
    sg = Guarded(Nb, Kb + 1, torch.float32)
    B.quant_weight(dev_bf16(w), with_q=True, with_t=True, q=qg.t, qt=tg.t, s=sg.t)
    torch.cuda.synchronize()
    q_ref, qt_ref, s_ref = O.quant_weight(w, with_t=True)
    assert np.array_equal(qg.t.cpu().numpy()[:, :K], q_ref)
    assert np.array_equal(tg.t.cpu().numpy()[:, :N], qt_ref)
    assert np.array_equal(f32_bits(sg.t.cpu().numpy()[:, :Kb]), f32_bits(s_ref))
    qg.check_outside(K)
    tg.check_outside(N)
    sg.check_outside(Kb)


def _adversarial_bf16(rows, cols, seed):
    """Random finite bf16 patterns over the whole exponent range, plus
    all-zero, signed-zero, all-equal and tie-producing groups."""
    rng = np.random.default_rng(seed)
    b = rng.integers(0, 1 << 16, size=(rows, cols), dtype=np.uint32).astype(np.uint16)
    b[(b & 0x7F80) == 0x7F80] &= 0xBF7F  # no Inf/NaN
    b[0, :] = 0
    if rows > 1:
        b[1, ::2] = 0x8000
    if rows > 2:
        b[2, :] = S.f32_to_bf16_bits(np.array([0.3], np.float32))[0]
    if rows > 3:  # amax 448 -> s = 1 exactly: x/s lands on e4m3 ties
        v = (np.arange(cols) % 64).astype(np.float32) / 16.0 + 1.0 / 32.0
        v[0] = 448.0
        b[3, :] = S.f32_to_bf16_bits(v)
    if rows > 4:  # tiny magnitudes: subnormal bf16, subnormal scales
        b[4, :] = rng.integers(1, 0x80, size=cols).astype(np.uint16)
    return b


@pytest.mark.parametrize("M,K", [(8, 128), (64, 1024), (37, 300)])
def test_quant_adversarial_values_bit_exact(M, K):
    x = _adversarial_bf16(M, K, seed=M + K)
    qg, sg, _, _ = _run_lhs(x, False, 0)
    q_ref, s_ref = O.quant_lhs(x)
    assert np.array_equal(qg.t.cpu().numpy()[:, :K], q_ref)
    assert np.array_equal(f32_bits(sg.t.cpu().numpy()[:, :M]), f32_bits(s_ref))
    # same values through the transposed-read and 128x1 kernels
    xt = np.ascontiguousarray(x.T)
    qg2, sg2, _, _ = _run_lhs(xt, True, 0)
    assert np.array_equal(qg2.t.cpu().numpy()[:, :K], q_ref)
    assert np.array_equal(f32_bits(sg2.t.cpu().numpy()[:, :M]), f32_bits(s_ref))
    q3, s3 = B.quant_rhs(dev_bf16(xt))
    assert np.array_equal(q3.cpu().numpy()[:, :K], q_ref)
    assert np.array_equal(f32_bits(s3.cpu().numpy()[:, :M]), f32_bits(s_ref))
    _, _, sw = B.quant_weight(dev_bf16(x))
    _, _, sw_ref = O.quant_weight(x)
    assert np.array_equal(f32_bits(sw.cpu().numpy()), f32_bits(sw_ref))


def _padded_dev(x, pad):
    """Device copy of x [R, C] whose row stride is C + pad (pad not a
    multiple of 8 forces the untiled fallback kernels)."""
    R, C = x.shape
    buf = np.zeros((R, C + pad), dtype=np.uint16)
    buf[:, :C] = x
    return dev_bf16(buf)[:, :C]


@pytest.mark.parametrize("M,K", [(130, 256), (300, 1000), (2048, 4096)])
def test_quant_lhs_fallback_path_bit_exact(M, K):
    """Row stride K+3: the TMA-staged kernel cannot read it; the untiled
    kernels must give the same bytes."""
    x = S.normal_bf16((M, K), 1.0, seed=M + 5 * K, outlier_frac=1e-3)
    q, s = B.quant_lhs(_padded_dev(x, 3))
    q_ref, s_ref = O.quant_lhs(x)
    assert np.array_equal(q.cpu().numpy()[:, :K], q_ref)
    assert np.array_equal(f32_bits(s.cpu().numpy()[:, :M]), f32_bits(s_ref))
    qt, st = B.quant_lhs(_padded_dev(np.ascontiguousarray(x.T), 5), transposed=True)
    assert np.array_equal(qt.cpu().numpy()[:, :K], q_ref)
    assert np.array_equal(f32_bits(st.cpu().numpy()[:, :M]), f32_bits(s_ref))
    w_q, w_qt, w_s = B.quant_weight(_padded_dev(x, 1), with_q=True, with_t=True)
    wq_ref, wqt_ref, ws_ref = O.quant_weight(x, with_t=True)
    assert np.array_equal(w_q.cpu().numpy()[:, :K], wq_ref)
    assert np.array_equal(w_qt.cpu().numpy()[:, :M], wqt_ref)
    assert np.array_equal(f32_bits(w_s.cpu().numpy()), f32_bits(ws_ref))


DUAL_SHAPES = [(130, 256), (257, 300), (2048, 4096), (8, 1000), (1, 136), (4100, 64)]


@pytest.mark.parametrize("T,C", DUAL_SHAPES)
@pytest.mark.parametrize("pad", [0, 3])
def test_quant_dual_bit_exact(T, C, pad):
    """One read of X gives both its 1x128 groups (as quant_lhs) and its 128x1
    groups written transposed (as quant_rhs)."""
    x = S.normal_bf16((T, C), 1.0, seed=T + 11 * C, outlier_frac=1e-3)
    Tb, Cb = cdiv(T, 128), cdiv(C, 128)
    qr, sr = Guarded(T, rup(C, 16) + 16, torch.uint8), Guarded(Cb, T + 2, torch.float32)
    qc, sc = Guarded(C, rup(T, 16) + 16, torch.uint8), Guarded(Tb, C + 2, torch.float32)
    xd = _padded_dev(x, pad) if pad else dev_bf16(x)
    B.quant_dual(xd, q_row=qr.t, s_row=sr.t, q_col=qc.t, s_col=sc.t)
    torch.cuda.synchronize()
    q_ref, s_ref = O.quant_lhs(x)
    qT_ref, sT_ref = O.quant_rhs(x)
    assert np.array_equal(qr.t.cpu().numpy()[:, :C], q_ref)
    assert np.array_equal(f32_bits(sr.t.cpu().numpy()[:, :T]), f32_bits(s_ref))
    assert np.array_equal(qc.t.cpu().numpy()[:, :T], qT_ref)
    assert np.array_equal(f32_bits(sc.t.cpu().numpy()[:, :C]), f32_bits(sT_ref))
    for g, w in ((qr, C), (sr, T), (qc, T), (sc, C)):
        g.check_outside(w)


@pytest.mark.parametrize("T,C,N", [(130, 256, 384), (1, 128, 128), (300, 520, 130), (2048, 4096, 4096),
                                   (257, 1000, 2051)])
def test_quant_dual_weight_one_launch_bit_exact(T, C, N):
    """quant_dual(x) and quant_weight(w) done by one launch over both inputs'
    tiles give exactly the oracle's bytes and scales of each."""
    x = S.normal_bf16((T, C), 1.0, seed=T + 3 * C, outlier_frac=1e-3)
    w = S.normal_bf16((N, C), 0.02, seed=N + 5 * C)
    Tb, Cb, Nb = cdiv(T, 128), cdiv(C, 128), cdiv(N, 128)
    qr, sr = Guarded(T, rup(C, 16) + 16, torch.uint8), Guarded(Cb, T + 2, torch.float32)
    qc, sc = Guarded(C, rup(T, 16) + 16, torch.uint8), Guarded(Tb, C + 2, torch.float32)
    qw, qwt = Guarded(N, rup(C, 16) + 16, torch.uint8), Guarded(C, rup(N, 16) + 16, torch.uint8)
    sw = Guarded(Nb, Cb + 1, torch.float32)
    B.quant_dual_weight(dev_bf16(x), dev_bf16(w), q_row=qr.t, s_row=sr.t, q_col=qc.t, s_col=sc.t,
                        qw=qw.t, qwt=qwt.t, sw=sw.t)
    torch.cuda.synchronize()
    q_ref, s_ref = O.quant_lhs(x)
    qT_ref, sT_ref = O.quant_rhs(x)
    qw_ref, qwt_ref, sw_ref = O.quant_weight(w, with_t=True)
    assert np.array_equal(qr.t.cpu().numpy()[:, :C], q_ref)
    assert np.array_equal(f32_bits(sr.t.cpu().numpy()[:, :T]), f32_bits(s_ref))
    assert np.array_equal(qc.t.cpu().numpy()[:, :T], qT_ref)
    assert np.array_equal(f32_bits(sc.t.cpu().numpy()[:, :C]), f32_bits(sT_ref))
    assert np.array_equal(qw.t.cpu().numpy()[:, :C], qw_ref)
    assert np.array_equal(qwt.t.cpu().numpy()[:, :N], qwt_ref)
    assert np.array_equal(f32_bits(sw.t.cpu().numpy()[:, :Cb]), f32_bits(sw_ref))
    for g, wd in ((qr, C), (sr, T), (qc, T), (sc, C), (qw, C), (qwt, N), (sw, Cb)):
        g.check_outside(wd)


MX_SHAPES = [(130, 256, 0), (1, 32, 0), (64, 1000, 0), (300, 520, 8), (2048, 4096, 0), (257, 72, 0),
             (512, 512, 0), (33, 4104, 0), (4096, 1024, 0), (96, 136, 16)]


@pytest.mark.parametrize("M,K,pad", MX_SHAPES)
@pytest.mark.parametrize("casts", ["both", "dim0", "dim1"])
def test_mx_cast_bit_exact(M, K, pad, casts):
    """MXFP8 casts (dim0 along K; dim1 along M, written transposed) give the
    oracle's codes and E8M0 exponents byte for byte, on tail shapes, padded
    rows, outliers, zero blocks and subnormal inputs; nothing outside the
    outputs is written."""
    x = S.normal_bf16((M, K), 1.0, seed=M + 7 * K, outlier_frac=2e-3)
    x[:, :min(32, K)][: max(1, M // 7)] = 0                      # all-zero blocks
    x[-1, -min(16, K):] = 0x0003                                  # bf16 subnormals
    d0, d1 = casts in ("both", "dim0"), casts in ("both", "dim1")
    q0 = Guarded(M, rup(K, 16) + 16, torch.uint8) if d0 else None
    e0 = Guarded(M, cdiv(K, 32) + 3, torch.uint8) if d0 else None
    q1 = Guarded(K, rup(M, 16) + 16, torch.uint8) if d1 else None
    e1 = Guarded(K, cdiv(M, 32) + 3, torch.uint8) if d1 else None
    xd = _padded_dev(x, pad) if pad else dev_bf16(x)
    B.mx_cast(xd, dim0=d0, dim1=d1, q0=q0.t if d0 else None, e0=e0.t if d0 else None,
              q1=q1.t if d1 else None, e1=e1.t if d1 else None)
    torch.cuda.synchronize()
    (rq0, re0), (rq1, re1) = O.mx_cast(x, dim0=d0, dim1=d1)
    if d0:
        assert np.array_equal(q0.t.cpu().numpy()[:, :K], rq0)
        assert np.array_equal(e0.t.cpu().numpy()[:, :cdiv(K, 32)], re0)
        q0.check_outside(K)
        e0.check_outside(cdiv(K, 32))
    if d1:
        assert np.array_equal(q1.t.cpu().numpy()[:, :M], rq1)
        assert np.array_equal(e1.t.cpu().numpy()[:, :cdiv(M, 32)], re1)
        q1.check_outside(M)
        e1.check_outside(cdiv(M, 32))


# ------------------------------------------------------------------ GEMMs in isolation

def _random_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x00  # no NaN codes
    return c


def _gemm_case(M, N, K, mode, seed, ldc_extra=0, repeats=1):
    """Random e4m3 codes and random scales fed to both sides."""
    rng = np.random.default_rng(seed)
    Kb, Nb = cdiv(K, 128), cdiv(N, 128)
    lda = ldb = rup(K, 16)
    qa = _random_codes(rng, (M, lda))
    qb = _random_codes(rng, (N, ldb))
    sa = rng.uniform(0.01, 2.0, (Kb, M + 1)).astype(np.float32)
    if mode == O.SB_TILE:
        sb = rng.uniform(0.01, 2.0, (Nb, Kb)).astype(np.float32)
    elif mode == O.SB_TILE_T:
        sb = rng.uniform(0.01, 2.0, (Kb, Nb + 1)).astype(np.float32)
    else:
        sb = rng.uniform(0.01, 2.0, (Kb, rup(N, 4))).astype(np.float32)
    ref = O.gemm(qa, sa, qb, sb, mode, K)
    cu = lambda a: torch.from_numpy(a).cuda()
    ldc = N + ldc_extra
    flat16 = torch.full((M * ldc + 2 * GUARD,), 0x7FC1, dtype=torch.int16, device="cuda")
    out = flat16[GUARD:GUARD + M * ldc].view(torch.bfloat16).view(M, ldc)
    for _ in range(repeats):
        out[:, :N].zero_()
        if mode == O.SB_COL:
            B.gemm_1x128_128x1(cu(qa), cu(sa), cu(qb), cu(sb), K, out=out, M=M, N=N)
        else:
            B.gemm_1x128_128x128(cu(qa), cu(sa), cu(qb), cu(sb), K, sb_transposed=(mode == O.SB_TILE_T),
                                 out=out, M=M, N=N)
    torch.cuda.synchronize()
    h = flat16.cpu().numpy()
    assert np.all(h[:GUARD] == 0x7FC1) and np.all(h[-GUARD:] == 0x7FC1), "write outside C"
    body = h[GUARD:GUARD + M * ldc].reshape(M, ldc)
    assert np.all(body[:, N:] == 0x7FC1), "write into C row padding"
    got = out[:, :N].float().cpu().numpy().astype(np.float64)
    return got, ref


GEMM_SHAPES = [(130, 384, 256), (1, 8, 128), (2, 512, 128), (4, 3584, 640), (128, 256, 128),
               (129, 257, 1000), (300, 130, 77), (256, 512, 4096), (64, 1000, 200), (513, 384, 384)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
@pytest.mark.parametrize("mode", [O.SB_TILE, O.SB_TILE_T, O.SB_COL])
def test_gemm_random_codes_matches_oracle(M, N, K, mode):
    got, ref = _gemm_case(M, N, K, mode, seed=M * 7 + N * 3 + K + mode, ldc_extra=8)
    assert_gemm_close(got, ref, f"gemm mode {mode} {M}x{N}x{K}")


# shapes with more tiles than SMs on a 152-SM GB300 and a partly idle last
# wave: persistent CTAs walk several tiles each; launched twice in a row.
# The 1x128 x 128x1 GEMM takes 224-column tiles at all of them (4052: a last
# tile of 20 columns, less than one promotion warp's 56)
MULTIWAVE_SHAPES = [(2048, 4096, 512), (2000, 4000, 520), (1200, 4096, 384), (2048, 4096, 4096), (1600, 4052, 256)]


@pytest.mark.parametrize("M,N,K", MULTIWAVE_SHAPES)
@pytest.mark.parametrize("mode", [O.SB_TILE, O.SB_TILE_T, O.SB_COL])
def test_gemm_multiwave_matches_oracle(M, N, K, mode):
    got, ref = _gemm_case(M, N, K, mode, seed=M + N + K + mode, ldc_extra=8, repeats=2)
    assert_gemm_close(got, ref, f"multi-wave gemm mode {mode} {M}x{N}x{K}")
    B.check_device_errors()


# few output tiles and a deep K: most SMs idle, one CTA walks every K-block of
# its tile; ragged M and N (the tile-scale GEMMs take 64-column tiles here,
# with 16-row A boxes for M <= 16; (3, 12288): 128-column tiles, M <= 16)
DEEP_K_SHAPES = [(128, 2048, 2048), (300, 384, 4096), (2, 5120, 1280), (64, 1000, 2048), (3, 12288, 1024)]


@pytest.mark.parametrize("M,N,K", DEEP_K_SHAPES)
@pytest.mark.parametrize("mode", [O.SB_TILE, O.SB_TILE_T, O.SB_COL])
def test_gemm_few_tiles_deep_k_matches_oracle(M, N, K, mode):
    got, ref = _gemm_case(M, N, K, mode, seed=5 * M + N + K + mode, ldc_extra=8, repeats=2)
    assert_gemm_close(got, ref, f"few-tile deep-K gemm mode {mode} {M}x{N}x{K}")
    B.check_device_errors()


# 128-column tiles (fewer 256-column tiles than SMs, too many 32- or
# 64-column ones for one wave), ragged M, N and K; 512 x 5120 has 160 tiles
# on 152 SMs, so some CTAs walk a second tile; launched twice in a row
MID_M_SHAPES = [(512, 4096, 1024), (500, 4000, 1000), (384, 4004, 640), (512, 5120, 1280)]


@pytest.mark.parametrize("M,N,K", MID_M_SHAPES)
@pytest.mark.parametrize("mode", [O.SB_TILE, O.SB_TILE_T])
def test_gemm_128_column_tiles_match_oracle(M, N, K, mode):
    assert B.lib().bfp8_debug_gemm_pick_bn(M, N, 0, 152) == 128
    got, ref = _gemm_case(M, N, K, mode, seed=13 * M + N + K + mode, ldc_extra=8, repeats=2)
    assert_gemm_close(got, ref, f"128-column-tile gemm mode {mode} {M}x{N}x{K}")
    B.check_device_errors()


# at most 32 rows, tile-scale modes: the operand-swapped kernel whose tiles'
# K-blocks are split over a cluster of CTAs (152 SMs: 16x4096x4096 4 splits;
# 1x130x8192 2; 5x2051x1100 2 over 9 K-blocks; 3x512x384 one; 7x18944 148
# tiles, one split; 12x19456 152 tiles, one split; 2x19584 153 tiles: the
# 64/128-column kernel; 8x1024x8192 8 splits; 17 and 32 rows: its 32-row form),
# and from 33 rows the dense kernel's tiles at the same kind of shapes;
# launched twice in a row
SMALLM_SHAPES = [(16, 4096, 4096), (1, 130, 8192), (5, 2051, 1100), (3, 512, 384), (7, 18944, 384),
                 (12, 19456, 256), (2, 19584, 256), (8, 1024, 8192),
                 (17, 4096, 4096), (32, 512, 2048), (33, 2051, 1100), (64, 4096, 4096), (100, 3000, 2048),
                 (128, 4096, 4096), (128, 18944, 384), (65, 19456, 256), (128, 1024, 16384)]


@pytest.mark.parametrize("M,N,K", SMALLM_SHAPES)
@pytest.mark.parametrize("mode", [O.SB_TILE, O.SB_TILE_T])
def test_gemm_small_m_split_k_matches_oracle(M, N, K, mode):
    got, ref = _gemm_case(M, N, K, mode, seed=11 * M + N + K + mode, ldc_extra=8, repeats=2)
    assert_gemm_close(got, ref, f"small-M gemm mode {mode} {M}x{N}x{K}")
    B.check_device_errors()


def test_gemm_small_m_repeat_is_bit_identical():
    """The split sums are added in a fixed order: two calls give the same bits."""
    rng = np.random.default_rng(3)
    M, N, K = 9, 3000, 6000
    qa, qb = _random_codes(rng, (M, rup(K, 16))), _random_codes(rng, (N, rup(K, 16)))
    sa = rng.uniform(0.01, 2.0, (cdiv(K, 128), M)).astype(np.float32)
    sb = rng.uniform(0.01, 2.0, (cdiv(N, 128), cdiv(K, 128))).astype(np.float32)
    cu = lambda a: torch.from_numpy(a).cuda()
    a = B.gemm_1x128_128x128(cu(qa), cu(sa), cu(qb), cu(sb), K, M=M, N=N)
    b = B.gemm_1x128_128x128(cu(qa), cu(sa), cu(qb), cu(sb), K, M=M, N=N)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(300, 130, 256), (129, 1001, 384), (64, 2051, 128)])
@pytest.mark.parametrize("mode", [O.SB_TILE, O.SB_COL])
def test_gemm_ragged_n_aligned_ldc(M, N, K, mode):
    """N not a multiple of 8 with a 16-byte-aligned row stride: the C row
    padding past N must stay untouched (TMA stores clip the inner dimension
    in 16-byte units, so such shapes take the per-row stores)."""
    ldc_extra = rup(N, 8) + 8 - N
    got, ref = _gemm_case(M, N, K, mode, seed=M + 3 * N + K + mode, ldc_extra=ldc_extra)
    assert_gemm_close(got, ref, f"ragged-N gemm mode {mode} {M}x{N}x{K}")


# ------------------------------------------------------------------ quant + GEMM (linear)

def _dev_linear(M, N, K, seed, x_std=1.0, w_std=0.02, dy_std=1e-3, outliers=0.0):
    x = S.normal_bf16((M, K), x_std, seed=seed * 16, outlier_frac=outliers)
    w = S.normal_bf16((N, K), w_std, seed=seed * 16 + 1)
    dy = S.normal_bf16((M, N), dy_std, seed=seed * 16 + 2)
    return x, w, dy


SMALL_M = [(m, n, k) for m in (2, 4, 128, 512) for (n, k) in ((512, 128), (5120, 1280), (3584, 640), (4096, 4096))]


@pytest.mark.parametrize("M,N,K", [(130, 384, 256)] + SMALL_M)
def test_linear_fwd_matches_oracle(M, N, K):
    x, w, _ = _dev_linear(M, N, K, seed=3)
    y = B.linear_fwd(dev_bf16(x), dev_bf16(w))
    torch.cuda.synchronize()
    assert_gemm_close(host_bf16_as_f64(y), O.linear_fwd(x, w), f"fwd {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(130, 384, 256), (257, 300, 131), (512, 1024, 640), (1024, 256, 512),
                                   (4, 384, 256), (32, 1024, 1280)])
def test_linear_bwd_matches_oracle(M, N, K):
    x, w, dy = _dev_linear(M, N, K, seed=4)
    dx, dw = B.linear_bwd(dev_bf16(dy), dev_bf16(x), dev_bf16(w))
    torch.cuda.synchronize()
    assert_gemm_close(host_bf16_as_f64(dx), O.linear_dgrad(dy, w), f"dgrad {M}x{N}x{K}")
    assert_gemm_close(host_bf16_as_f64(dw), O.linear_wgrad(dy, x), f"wgrad {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(130, 384, 256), (257, 300, 131), (512, 1024, 640), (2048, 4096, 4096),
                                   (2, 4096, 4096), (24, 640, 1280)])
def test_linear_train_form_matches_oracle(M, N, K):
    """fwd_train keeps the quantised x (both forms) and W (both forms) in the
    workspace; bwd_saved quantises dY once and runs both gradient GEMMs."""
    x, w, dy = _dev_linear(M, N, K, seed=6)
    ws = B.linear_train_workspace(M, N, K)
    y = B.linear_fwd_train(dev_bf16(x), dev_bf16(w), ws)
    dx, dw = B.linear_bwd_saved(dev_bf16(dy), ws, M, N, K)
    torch.cuda.synchronize()
    if M * N * K <= 1024 ** 3:
        assert_gemm_close(host_bf16_as_f64(y), O.linear_fwd(x, w), "train fwd")
        assert_gemm_close(host_bf16_as_f64(dx), O.linear_dgrad(dy, w), "train dgrad")
        assert_gemm_close(host_bf16_as_f64(dw), O.linear_wgrad(dy, x), "train wgrad")
    else:
        rows = _sample_idx(M, 16, 1)
        ref, cols = _oracle_fwd_sampled(x, w, rows, _sample_idx(N // 128, 2, 2))
        got = host_bf16_as_f64(y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
        assert_gemm_close(got, ref, "train fwd sampled")
        nrows, kc = _sample_idx(N, 16, 3), _sample_idx(K, 128, 4)
        qa, sa = O.quant_lhs(np.ascontiguousarray(dy[:, nrows]), transposed=True)
        qbT, sb = O.quant_rhs(np.ascontiguousarray(x[:, kc]))
        ref = O.gemm(qa, sa, qbT, sb, O.SB_COL, M)
        got = host_bf16_as_f64(dw[torch.from_numpy(nrows).cuda()][:, torch.from_numpy(kc).cuda()])
        assert_gemm_close(got, ref, "train wgrad sampled")


@pytest.mark.parametrize("M,N,K", [(300, 384, 520), (1024, 2048, 1024)])
def test_training_step_replayed_as_one_graph(M, N, K):
    """The whole training step (one quantisation launch for x and W, forward
    GEMM, dY quantisation, both gradient GEMMs) captured as one CUDA graph and
    replayed back to back: every kernel starts while the one before it
    finishes (programmatic dependent launch) and must still read only
    finished inputs.  New inputs are copied in between replays, so a kernel
    that read its inputs early would produce the previous replay's results."""
    ws = B.linear_train_workspace(M, N, K)
    gx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    gw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    gdy = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    inputs = [_dev_linear(M, N, K, seed=20 + i) for i in range(2)]
    gx.copy_(dev_bf16(inputs[0][0])); gw.copy_(dev_bf16(inputs[0][1])); gdy.copy_(dev_bf16(inputs[0][2]))
    step = lambda: (B.linear_fwd_train(gx, gw, ws, y=y), B.linear_bwd_saved(gdy, ws, M, N, K, dx=dx, dw=dw))
    step()  # one-time attribute set-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for rep in range(4):
        x, w, dy = inputs[rep % 2]
        gx.copy_(dev_bf16(x)); gw.copy_(dev_bf16(w)); gdy.copy_(dev_bf16(dy))
        g.replay()
        g.replay()  # twice in a row: the second replay's kernels overlap the first's tails
        torch.cuda.synchronize()
        B.check_device_errors()
        assert_gemm_close(host_bf16_as_f64(y), O.linear_fwd(x, w), f"graph fwd replay {rep}")
        assert_gemm_close(host_bf16_as_f64(dx), O.linear_dgrad(dy, w), f"graph dgrad replay {rep}")
        assert_gemm_close(host_bf16_as_f64(dw), O.linear_wgrad(dy, x), f"graph wgrad replay {rep}")


def test_float8_blockwise_linear_module_forward_and_backward():
    """The autograd module: y = x W^T forward, dX and dW from y.backward(dY),
    on a 3-d input (the token dims are flattened), against the oracle."""
    M0, M1, N, K = 2, 65, 384, 256
    x, w, dy = _dev_linear(M0 * M1, N, K, seed=60)
    xd = dev_bf16(x).reshape(M0, M1, K).requires_grad_(True)
    layer = B.Float8BlockwiseLinear(K, N, device="cuda")
    with torch.no_grad():
        layer.weight.copy_(dev_bf16(w))
    y = layer(xd)
    assert y.shape == (M0, M1, N) and y.dtype == torch.bfloat16
    y.backward(dev_bf16(dy).reshape(M0, M1, N))
    torch.cuda.synchronize()
    B.check_device_errors()
    assert_gemm_close(host_bf16_as_f64(y.detach().reshape(-1, N)), O.linear_fwd(x, w), "module y")
    assert_gemm_close(host_bf16_as_f64(xd.grad.reshape(-1, K)), O.linear_dgrad(dy, w), "module dX")
    assert_gemm_close(host_bf16_as_f64(layer.weight.grad), O.linear_wgrad(dy, x), "module dW")


@pytest.mark.parametrize("M,N,K,chunk", [(320, 1152, 384, 256),   # five chunks, the last one 128 wide
                                         (1100, 1000, 520, 512),  # chunks of 512 + 488, three dX pieces
                                         (640, 2304, 256, 0),     # automatic: 1024 + 1024 + 256, two pieces
                                         (130, 384, 256, 0),      # one chunk, one piece
                                         (257, 200, 131, 128)])   # ragged everywhere: rows of 131 bf16
                                                                  # (no TMA path for x), chunks 128 + 72
def test_linear_step_host_matches_training_form_and_oracle(M, N, K, chunk):
    """The whole step from pinned host buffers (copies overlapped with the
    kernels, W and dY in column chunks, dX in row pieces) gives the training
    form's results bit for bit, and those meet the oracle's bound."""
    x, w, dy = _dev_linear(M, N, K, seed=62)
    host = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    ws = B.linear_step_host_workspace(M, N, K)
    y, dx, dw = B.linear_step_host(host(x), host(w), host(dy), ws, chunk_n=chunk)
    torch.cuda.current_stream().synchronize()
    B.check_device_errors()
    tws = B.linear_train_workspace(M, N, K)
    ty = B.linear_fwd_train(dev_bf16(x), dev_bf16(w), tws)
    tdx, tdw = B.linear_bwd_saved(dev_bf16(dy), tws, M, N, K)
    torch.cuda.synchronize()
    for name, a, b in (("y", y, ty), ("dX", dx, tdx), ("dW", dw, tdw)):
        assert torch.equal(a.view(torch.int16), b.cpu().view(torch.int16)), f"host step {name} differs"
    assert_gemm_close(y.float().numpy().astype(np.float64), O.linear_fwd(x, w), "host step y")
    assert_gemm_close(dx.float().numpy().astype(np.float64), O.linear_dgrad(dy, w), "host step dX")
    assert_gemm_close(dw.float().numpy().astype(np.float64), O.linear_wgrad(dy, x), "host step dW")


def test_linear_step_host_pageable_memory_and_concurrent_threads():
    """The host step from pageable (not page-locked) buffers gives the same
    bits as from pinned ones; two host threads, each with its own workspace
    and stream, running steps at the same time share the library's copy
    streams and events safely."""
    import threading
    M, N, K = 256, 1280, 384
    x, w, dy = _dev_linear(M, N, K, seed=63)
    pinned = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    pageable = lambda a: torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    ws = B.linear_step_host_workspace(M, N, K)
    ref = B.linear_step_host(pinned(x), pinned(w), pinned(dy), ws, chunk_n=512)
    torch.cuda.synchronize()
    out = B.linear_step_host(pageable(x), pageable(w), pageable(dy), ws, chunk_n=512,
                             y=torch.empty(M, N, dtype=torch.bfloat16), dx=torch.empty(M, K, dtype=torch.bfloat16),
                             dw=torch.empty(N, K, dtype=torch.bfloat16))
    torch.cuda.synchronize()
    for a, b in zip(ref, out):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "pageable host step differs"

    results, errs = [None, None], []

    def work(i):
        try:
            st = torch.cuda.Stream()
            wsi = B.linear_step_host_workspace(M, N, K)
            hx, hw, hdy = pinned(x), pinned(w), pinned(dy)
            with torch.cuda.stream(st):
                for _ in range(5):
                    r = B.linear_step_host(hx, hw, hdy, wsi, chunk_n=256)
                st.synchronize()
            results[i] = r
        except Exception as e:  # reported on the main thread
            errs.append(e)

    ts = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    B.check_device_errors()
    for r in results:
        for a, b in zip(ref, r):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "concurrent host step differs"


def test_library_calls_from_a_thread_that_selected_no_device():
    """Autograd runs backward on a worker thread; a fresh host thread that never
    selected a device must still be able to launch (the library binds the
    thread to its current device)."""
    import threading
    M, N, K = 256, 256, 384
    x, w, dy = _dev_linear(M, N, K, seed=61)
    xd, wd, dyd = dev_bf16(x), dev_bf16(w), dev_bf16(dy)
    out, errs = {}, []

    def work():
        try:
            ws = B.linear_train_workspace(M, N, K, device=xd.device)
            out["y"] = B.linear_fwd_train(xd, wd, ws)
            out["dx"], out["dw"] = B.linear_bwd_saved(dyd, ws, M, N, K)
            torch.cuda.synchronize()
        except Exception as e:  # reported on the main thread
            errs.append(e)

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert not errs, errs
    B.check_device_errors()
    assert_gemm_close(host_bf16_as_f64(out["y"]), O.linear_fwd(x, w), "thread y")
    assert_gemm_close(host_bf16_as_f64(out["dx"]), O.linear_dgrad(dy, w), "thread dX")
    assert_gemm_close(host_bf16_as_f64(out["dw"]), O.linear_wgrad(dy, x), "thread dW")


def _pages_sqnr():
    import os
    rows = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "sqnr_pages.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                m, n, k, db = line.split()
                rows.append((int(m), int(n), int(k), float(db)))
    return rows


@pytest.mark.parametrize("M,N,K,pages_db", _pages_sqnr())
def test_gemm_sqnr_vs_pages(M, N, K, pages_db):
    """SQNR of the device's blockwise FP8 GEMM against an fp64 matmul of the
    bf16 inputs on N(0,1) data: at least 28 dB and within 0.5 dB of the
    pages' printed figure for the same shape."""
    x = S.normal_bf16((M, K), 1.0, seed=11)
    w = S.normal_bf16((N, K), 1.0, seed=12)
    y = host_bf16_as_f64(B.linear_fwd(dev_bf16(x), dev_bf16(w)))
    ref = (torch.from_numpy(S.bf16_bits_to_f32(x)).double().cuda()
           @ torch.from_numpy(S.bf16_bits_to_f32(w)).double().cuda().T).cpu().numpy()
    db = sqnr_db(ref, y)
    assert db >= 28.0 and abs(db - pages_db) <= 0.5, db


# ------------------------------------------------------------------ full-size workloads, sampled

def _sample_idx(n, k, seed):
    rng = np.random.default_rng(seed)
    idx = set(rng.choice(n, size=min(k, n), replace=False).tolist())
    idx.update({0, n - 1})
    return np.array(sorted(idx), dtype=np.int64)


def _blocks_of(idx):
    return np.array(sorted({int(i) // 128 for i in idx}), dtype=np.int64)


def _expand_blocks(blocks, n):
    return np.concatenate([np.arange(b * 128, min(n, b * 128 + 128)) for b in blocks])


def _oracle_fwd_sampled(x, w, rows, col_blocks):
    """Oracle y[rows][:, cols in col_blocks] computed from only the rows of x
    and the 128-row blocks of W it needs (groups and tiles are local to them)."""
    cols = _expand_blocks(col_blocks, w.shape[0])
    qa, sa = O.quant_lhs(np.ascontiguousarray(x[rows]))
    qb, _, sb = O.quant_weight(np.ascontiguousarray(w[cols]))
    return O.gemm(qa, sa, qb, sb, O.SB_TILE, x.shape[1]), cols


@pytest.mark.parametrize("wl", [S.FWD_MID, S.FWD_SQUARE])
def test_fwd_full_size_sampled(wl):
    x, w = wl.x(), wl.w()
    y = B.linear_fwd(dev_bf16(x), dev_bf16(w))
    torch.cuda.synchronize()
    rows = _sample_idx(wl.M, 48, 1)
    cblk = _sample_idx(wl.N // 128, 3, 2)
    ref, cols = _oracle_fwd_sampled(x, w, rows, cblk)
    got = host_bf16_as_f64(y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
    assert_gemm_close(got, ref, wl.name)


def test_wgrad_full_size_sampled():
    wl = S.WGRAD  # dY [8192,4096], X [8192,4096] -> dW [4096,4096]
    dy, x = wl.dy(), wl.x()
    w = wl.w()
    dx, dw = B.linear_bwd(dev_bf16(dy), dev_bf16(x), dev_bf16(w))
    torch.cuda.synchronize()
    rows = _sample_idx(wl.N, 40, 3)     # output-feature rows of dW
    cols = _sample_idx(wl.K, 300, 4)    # input-feature columns of dW
    qa, sa = O.quant_lhs(np.ascontiguousarray(dy[:, rows]), transposed=True)
    qbT, sb = O.quant_rhs(np.ascontiguousarray(x[:, cols]))
    ref = O.gemm(qa, sa, qbT, sb, O.SB_COL, wl.M)
    got = host_bf16_as_f64(dw[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
    assert_gemm_close(got, ref, "wgrad 4096x4096x8192")
    # dgrad of the same step, sampled: dX = dY W
    r2 = _sample_idx(wl.M, 24, 5)
    kblk = _sample_idx(wl.K // 128, 2, 6)
    kcols = _expand_blocks(kblk, wl.K)
    qa2, sa2 = O.quant_lhs(np.ascontiguousarray(dy[r2]))
    _, qt, sw = O.quant_weight(np.ascontiguousarray(w[:, kcols]), with_t=True)
    ref2 = O.gemm(qa2, sa2, qt, sw, O.SB_TILE_T, wl.N)
    got2 = host_bf16_as_f64(dx[torch.from_numpy(r2).cuda()][:, torch.from_numpy(kcols).cuda()])
    assert_gemm_close(got2, ref2, "dgrad 8192x4096x4096")


def test_mlp_up_step_full_size_sampled():
    """The full linear step at 16384 x 14336 x 4096: fwd, dgrad and wgrad,
    each checked on sampled outputs the oracle computes one by one."""
    wl = S.MLP_UP
    x, w, dy = wl.x(), wl.w(), wl.dy()
    xd, wd, dyd = dev_bf16(x), dev_bf16(w), dev_bf16(dy)
    y = B.linear_fwd(xd, wd)
    dx, dw = B.linear_bwd(dyd, xd, wd)
    torch.cuda.synchronize()
    B.check_device_errors()
    rows = _sample_idx(wl.M, 16, 7)
    ref, cols = _oracle_fwd_sampled(x, w, rows, _sample_idx(wl.N // 128, 2, 8))
    got = host_bf16_as_f64(y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
    assert_gemm_close(got, ref, "mlp_up fwd")
    kcols = _expand_blocks(_sample_idx(wl.K // 128, 2, 9), wl.K)
    qa, sa = O.quant_lhs(np.ascontiguousarray(dy[rows]))
    _, qt, sw = O.quant_weight(np.ascontiguousarray(w[:, kcols]), with_t=True)
    ref = O.gemm(qa, sa, qt, sw, O.SB_TILE_T, wl.N)
    got = host_bf16_as_f64(dx[torch.from_numpy(rows).cuda()][:, torch.from_numpy(kcols).cuda()])
    assert_gemm_close(got, ref, "mlp_up dgrad")
    nrows = _sample_idx(wl.N, 12, 10)
    kc = _sample_idx(wl.K, 200, 11)
    qa, sa = O.quant_lhs(np.ascontiguousarray(dy[:, nrows]), transposed=True)
    qbT, sb = O.quant_rhs(np.ascontiguousarray(x[:, kc]))
    ref = O.gemm(qa, sa, qbT, sb, O.SB_COL, wl.M)
    got = host_bf16_as_f64(dw[torch.from_numpy(nrows).cuda()][:, torch.from_numpy(kc).cuda()])
    assert_gemm_close(got, ref, "mlp_up wgrad")


def _bench_step(wl):
    """The benchmark's own step (its buffers, its calls, the whole step as one
    CUDA graph), run once on the workload's inputs."""
    import bench
    x, w, dy = wl.x(), wl.w(), wl.dy()
    step = bench.Step(wl, torch, B, torch.device("cuda", 0))
    step.capture(dev_bf16(x), dev_bf16(w), dev_bf16(dy))
    step.run_step()
    torch.cuda.synchronize()
    B.check_device_errors()
    return step, x, w, dy


def _pick(t, rows, cols):
    return host_bf16_as_f64(t[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])


def _check_linear_sampled(x, w, dy, y, dx, dw, what, seed):
    """y, dX and dW of one dense linear on sampled outputs, each computed by
    the oracle from only the rows / columns it needs."""
    M, K = x.shape
    N = w.shape[0]
    rows = _sample_idx(M, 12, seed)
    ref, cols = _oracle_fwd_sampled(x, w, rows, _sample_idx(N // 128, 2, seed + 1))
    assert_gemm_close(_pick(y, rows, cols), ref, f"{what} y")
    kcols = _expand_blocks(_sample_idx(K // 128, 2, seed + 2), K)
    qa, sa = O.quant_lhs(np.ascontiguousarray(dy[rows]))
    _, qt, sw = O.quant_weight(np.ascontiguousarray(w[:, kcols]), with_t=True)
    assert_gemm_close(_pick(dx, rows, kcols), O.gemm(qa, sa, qt, sw, O.SB_TILE_T, N), f"{what} dx")
    nrows, kc = _sample_idx(N, 12, seed + 3), _sample_idx(K, 160, seed + 4)
    qa, sa = O.quant_lhs(np.ascontiguousarray(dy[:, nrows]), transposed=True)
    qbT, sb = O.quant_rhs(np.ascontiguousarray(x[:, kc]))
    assert_gemm_close(_pick(dw, nrows, kc), O.gemm(qa, sa, qbT, sb, O.SB_COL, M), f"{what} dW")


def test_bench_step_full_size_sampled():
    """The pages' mid shape (2048 x 4096 x 4096) in the launch configuration
    the benchmark times: sampled y, dX and dW against the oracle."""
    step, x, w, dy = _bench_step(S.FWD_MID)
    _check_linear_sampled(x, w, dy, step.y, step.dx, step.dw, "bench step", seed=30)


def _u8_rows(t, rows, ncols):
    return t[torch.from_numpy(np.asarray(rows)).cuda()][:, :ncols].cpu().numpy()


def _f32_cols(t, cols):
    return f32_bits(t[:, torch.from_numpy(np.asarray(cols)).cuda()].cpu().numpy())


def test_bench_mlp_up_step_quant_bytes_bit_exact_and_gemms_sampled():
    """The benchmark's default workload, the MLP-up layer 16384 x 14336 x 4096,
    in the launch configuration it times (one graph of the five calls).  Every
    quantised operand the step makes is compared byte for byte with the
    oracle -- e4m3 codes and fp32 scale bits -- on sampled rows, columns and
    128-row weight blocks that include the last tile of each tensor:
      dY [16384, 14336]: 1x128 groups along N (q_row, s_row) and 1x128 groups
        along M of dY^T (q_col [14336, 16384], s_col);
      x [16384, 4096]: 1x128 groups along K and 128x1 groups along M (x^T);
      W [14336, 4096]: 128x128 tiles as is (q), transposed (qt) and scales.
    Then y, dX and dW on sampled outputs within the GEMM tolerance."""
    wl = S.MLP_UP
    M, N, K = wl.M, wl.N, wl.K
    step, x, w, dy = _bench_step(wl)
    mb, nb, kb = cdiv(M, 128), cdiv(N, 128), cdiv(K, 128)

    # dY, 1x128 along N: whole rows, scales column-major [M, Nb]
    rows = _sample_idx(M, 24, 50)
    q, s = O.quant_lhs(np.ascontiguousarray(dy[rows]))
    assert np.array_equal(_u8_rows(step.qdy, rows, N), q), "q(dY) rows"
    assert np.array_equal(_f32_cols(step.sdy[:nb], rows), f32_bits(s)), "s(dY) rows"
    # dY^T, 1x128 along M: whole columns of dY (rows of q_col), last column included
    ncols = _sample_idx(N, 24, 51)
    q, s = O.quant_lhs(np.ascontiguousarray(dy[:, ncols]), transposed=True)
    assert np.array_equal(_u8_rows(step.qdyt, ncols, M), q), "q(dY^T) rows"
    assert np.array_equal(_f32_cols(step.sdyt[:mb], ncols), f32_bits(s)), "s(dY^T)"
    # x, 1x128 along K
    q, s = O.quant_lhs(np.ascontiguousarray(x[rows]))
    assert np.array_equal(_u8_rows(step.qx, rows, K), q), "q(x) rows"
    assert np.array_equal(_f32_cols(step.sx[:kb], rows), f32_bits(s)), "s(x) rows"
    # x, 128x1 along M, written transposed [K, M]
    kcols = _sample_idx(K, 24, 52)
    q, s = O.quant_rhs(np.ascontiguousarray(x[:, kcols]))
    assert np.array_equal(_u8_rows(step.qxt, kcols, M), q), "q(x^T) rows"
    assert np.array_equal(_f32_cols(step.sxt[:mb], kcols), f32_bits(s)), "s(x^T)"
    # W: 128-row blocks (the last one included), tiles as is and transposed
    for blk in _sample_idx(nb, 3, 53):
        r = np.arange(blk * 128, min(N, blk * 128 + 128))
        q, qt, s = O.quant_weight(np.ascontiguousarray(w[r]), with_t=True)
        assert np.array_equal(_u8_rows(step.qw, r, K), q), f"q(W) block {blk}"
        got_t = step.qwt[:, int(r[0]):int(r[-1]) + 1].cpu().numpy()
        assert np.array_equal(got_t, qt), f"qt(W) block {blk}"
        assert np.array_equal(f32_bits(step.sw[int(blk)].cpu().numpy()), f32_bits(s[0])), f"s(W) block {blk}"
    # the GEMM outputs, sampled
    _check_linear_sampled(x, w, dy, step.y, step.dx, step.dw, "mlp_up bench step", seed=60)


def test_bench_moe_step_full_size_sampled():
    """The mixture-of-experts benchmark step (4096 tokens over 8 experts of
    4096 x 4096, two experts without tokens) in the launch configuration the
    benchmark times: each expert's sampled y, dX and dW against the oracle on
    its token slice; the empty experts' gradients are zero."""
    wl = S.MOE_MID
    step, x, w, dy = _bench_step(wl)
    offs = wl.offsets()
    for e in range(wl.E):
        t0, t1 = int(offs[e]), int(offs[e + 1])
        if t1 == t0:
            assert float(step.dw[e].abs().max()) == 0.0, f"expert {e} without tokens"
            continue
        if e not in (0, 3, 5):
            continue  # three of the experts with tokens, to bound the oracle's time
        we = w[e * wl.N:(e + 1) * wl.N]
        _check_linear_sampled(x[t0:t1], we, dy[t0:t1], step.y[t0:t1], step.dx[t0:t1], step.dw[e],
                              f"moe expert {e}", seed=40 + e)


def test_repeat_runs_are_deterministic():
    x, w, dy = _dev_linear(512, 640, 384, seed=9)
    xd, wd, dyd = dev_bf16(x), dev_bf16(w), dev_bf16(dy)
    a = [B.linear_fwd(xd, wd) for _ in range(2)]
    b = [B.linear_bwd(dyd, xd, wd) for _ in range(2)]
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), a[1].view(torch.int16))
    assert torch.equal(b[0][0].view(torch.int16), b[1][0].view(torch.int16))
    assert torch.equal(b[0][1].view(torch.int16), b[1][1].view(torch.int16))


def test_empty_problems_are_noops():
    e = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s = B.quant_lhs(e)
    assert q.shape[0] == 0
    out = torch.full((4, 8), 1.0, dtype=torch.bfloat16, device="cuda")
    z = torch.zeros((4, 16), dtype=torch.uint8, device="cuda")
    sc = torch.ones((1, 8), dtype=torch.float32, device="cuda")
    B.gemm_1x128_128x128(z, sc, torch.zeros((8, 16), dtype=torch.uint8, device="cuda"), sc, 0, out=out)
    torch.cuda.synchronize()
    assert torch.all(out.float() == 0)

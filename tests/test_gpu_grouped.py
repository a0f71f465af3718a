"""Parity of the grouped (mixture-of-experts) GEMMs with the CPU oracle.

Tokens are sorted by expert; expert e owns token rows offs[e] .. offs[e+1].
The forward / input-gradient GEMMs group the token rows, the weight gradient
groups the reduction.  Outputs must satisfy the dense GEMM's bound
|gpu - oracle| <= 2^-7 |oracle| + 1e-3 rms(oracle) element by element; rows
that belong to no expert, row padding and a guard band around every output
keep their sentinel.
"""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from gpu_util import assert_gemm_close, torch

import blockwise_scaled_fp8_gb300 as B

pytestmark = pytest.mark.gpu

GUARD = 4096
SENT = 0x7FC1  # a bf16 NaN pattern no kernel produces


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


def _codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x00  # no NaN codes
    return c


def _cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _guarded_bf16(n):
    flat = torch.full((n + 2 * GUARD,), SENT, dtype=torch.int16, device="cuda")
    return flat, flat[GUARD:GUARD + n].view(torch.bfloat16)


def _offsets(rng, E, total, align=1, empty=()):
    """E+1 non-decreasing offsets from 0 to total, each expert's start a
    multiple of `align` (the last end may be ragged), experts in `empty`
    without tokens."""
    cuts = np.sort(rng.integers(0, total // align + 1, size=E - 1)) * align
    offs = np.concatenate([[0], cuts, [total]]).astype(np.int64)
    for e in empty:
        offs[e + 1] = offs[e]
    return np.maximum.accumulate(offs).astype(np.int32)


# (E, offsets or None for random, M_total, N, K)
ROW_CASES = [
    (4, [0, 70, 70, 200, 300], 310, 256, 384),     # an empty expert; rows 300.. outside every expert
    (3, [5, 5, 133, 400], 400, 130, 208),          # first expert starts past row 0; ragged N and K
    (1, None, 257, 384, 256),                      # one expert = the dense GEMM
    (8, None, 2048, 512, 1024),
    (16, None, 8192, 1024, 512),                   # more tiles than SMs
    (12, None, 6000, 2056, 256),                   # staged TMA-store epilogue: tiles split at expert ends, 8-column last tile
]


def _row_case(E, offs, M_total, N, K, mode, seed):
    rng = np.random.default_rng(seed)
    if offs is None:
        offs = _offsets(rng, E, M_total, empty=(E // 2,) if E > 2 else ())
    offs = np.asarray(offs, np.int32)
    Kb, Nb = cdiv(K, 128), cdiv(N, 128)
    lda = rup(K, 16)
    qa = _codes(rng, (M_total, lda))
    sa = rng.uniform(0.01, 2.0, (Kb, M_total + 3)).astype(np.float32)
    if mode == O.SB_TILE:       # forward: weights stacked [E*N, K], tile scales [E*Nb, Kb]
        qb = _codes(rng, (E * N, lda))
        sb = rng.uniform(0.01, 2.0, (E * Nb, Kb + 1)).astype(np.float32)
        ref = O.moe_gemm_fwd(qa[:, :K], sa, qb[:, :K], sb[:, :Kb], offs, N, K)
    else:                       # input gradient: B = [N, E*K] (expert e in columns e*K ..), scales [E*Kb, Nb]
        qb = _codes(rng, (N, rup(E * K, 16)))
        sb = rng.uniform(0.01, 2.0, (E * Kb, Nb + 2)).astype(np.float32)
        ref = O.moe_gemm_dgrad(qa[:, :K], sa, qb[:, :E * K], sb[:, :Nb], offs, K, N)
    ldc = N + 8
    flat, body = _guarded_bf16(M_total * ldc)
    out = body.view(M_total, ldc)
    B.gemm_grouped_1x128_128x128(_cu(qa), _cu(sa), _cu(qb), _cu(sb), _cu(offs), N, K,
                                 sb_transposed=(mode == O.SB_TILE_T), out=out)
    torch.cuda.synchronize()
    B.check_device_errors()
    h = flat.cpu().numpy()
    assert np.all(h[:GUARD] == SENT) and np.all(h[-GUARD:] == SENT), "write outside C"
    hb = h[GUARD:GUARD + M_total * ldc].reshape(M_total, ldc)
    assert np.all(hb[:, N:] == SENT), "write into C row padding"
    inside = np.zeros(M_total, bool)
    inside[offs[0]:offs[-1]] = True
    assert np.all(hb[~inside] == SENT), "write into rows of no expert"
    got = out[:, :N].float().cpu().numpy().astype(np.float64)
    return got[inside], ref[inside]


@pytest.mark.parametrize("E,offs,M_total,N,K", ROW_CASES)
@pytest.mark.parametrize("mode", [O.SB_TILE, O.SB_TILE_T])
def test_grouped_rows_matches_oracle(E, offs, M_total, N, K, mode):
    got, ref = _row_case(E, offs, M_total, N, K, mode, seed=E * 13 + M_total + N + K + mode)
    assert_gemm_close(got, ref, f"grouped rows mode {mode} E={E} {M_total}x{N}x{K}")


# (E, offsets or None for random 128-aligned, T tokens, M, N)
RED_CASES = [
    (4, [0, 256, 256, 640, 700], 700, 130, 200),   # an empty expert, ragged last expert, ragged M and N
    (1, [0, 300], 300, 256, 384),                  # one expert = the dense weight gradient
    (8, None, 4096, 512, 384),
    (3, [0, 0, 4096, 4096], 4096, 384, 1024),      # all tokens in one expert
    (16, None, 8192, 1024, 512),                   # more tiles than SMs
    (16, None, 8192, 1000, 512),                   # staged TMA-store epilogue with a last row tile of 104 rows
]


@pytest.mark.parametrize("E,offs,T,M,N", RED_CASES)
def test_grouped_reduction_matches_oracle(E, offs, T, M, N):
    rng = np.random.default_rng(E * 7 + T + M + N)
    if offs is None:
        offs = _offsets(rng, E, T, align=128, empty=(1,))
    offs = np.asarray(offs, np.int32)
    Tb = cdiv(T, 128)
    ld = rup(T, 16)
    qa = _codes(rng, (M, ld))
    qb = _codes(rng, (N, ld))
    sa = rng.uniform(0.01, 2.0, (Tb, M + 1)).astype(np.float32)
    sb = rng.uniform(0.01, 2.0, (Tb, rup(N, 4))).astype(np.float32)
    ref = O.moe_gemm_wgrad(qa[:, :T], sa, qb[:, :T], sb[:, :N], offs)
    ldc = N + 8
    flat, body = _guarded_bf16(E * M * ldc)
    out = body.view(E, M, ldc)
    B.gemm_grouped_1x128_128x1(_cu(qa), _cu(sa), _cu(qb), _cu(sb), _cu(offs), T, out=out)
    torch.cuda.synchronize()
    B.check_device_errors()
    h = flat.cpu().numpy()
    assert np.all(h[:GUARD] == SENT) and np.all(h[-GUARD:] == SENT), "write outside dW"
    assert np.all(h[GUARD:GUARD + E * M * ldc].reshape(E, M, ldc)[:, :, N:] == SENT), "write into row padding"
    got = out[:, :, :N].float().cpu().numpy().astype(np.float64)
    for e in range(E):
        if offs[e + 1] == offs[e]:
            assert np.all(got[e] == 0.0), f"expert {e} without tokens must get zeros"
        else:
            assert_gemm_close(got[e], ref[e], f"grouped reduction E={E} expert {e}")


def test_grouped_input_gradient_needs_aligned_k():
    """Expert e's B starts at K column e*K of the map; the host refuses a K
    that would start a TMA load off a 16-byte boundary."""
    rng = np.random.default_rng(4)
    M_total, N, K = 256, 128, 200
    qa = _cu(_codes(rng, (M_total, rup(K, 16))))
    sa = _cu(np.ones((2, M_total), np.float32))
    qb = _cu(_codes(rng, (N, rup(2 * K, 16))))
    sb = _cu(np.ones((4, 1), np.float32))
    with pytest.raises(B.Bfp8Error, match="K % 16"):
        B.gemm_grouped_1x128_128x128(qa, sa, qb, sb, _cu(np.array([0, 100, 256], np.int32)), N, K,
                                     sb_transposed=True)


def test_grouped_bad_offsets_are_clamped_and_reported():
    """Decreasing offsets (and, for the weight gradient, an expert not starting
    on a 128-token boundary) are clamped on the device and reported by
    check_device_errors; nothing outside the outputs is written."""
    rng = np.random.default_rng(3)
    M_total, N, K = 400, 256, 256
    qa = _cu(_codes(rng, (M_total, K)))
    sa = _cu(rng.uniform(0.5, 1.0, (2, M_total)).astype(np.float32))
    qb = _cu(_codes(rng, (3 * N, K)))
    sb = _cu(rng.uniform(0.5, 1.0, (6, 2)).astype(np.float32))
    offs = _cu(np.array([0, 300, 100, 400], np.int32))
    flat, body = _guarded_bf16(M_total * N)
    B.gemm_grouped_1x128_128x128(qa, sa, qb, sb, offs, N, K, out=body.view(M_total, N))
    with pytest.raises(B.Bfp8Error, match="offsets"):
        B.check_device_errors()
    h = flat.cpu().numpy()
    assert np.all(h[:GUARD] == SENT) and np.all(h[-GUARD:] == SENT)
    # weight gradient with an expert starting at token 100
    T, M = 384, 128
    qdyt = _cu(_codes(rng, (M, T)))
    qxt = _cu(_codes(rng, (N, T)))
    s1 = _cu(rng.uniform(0.5, 1.0, (3, M)).astype(np.float32))
    s2 = _cu(rng.uniform(0.5, 1.0, (3, N)).astype(np.float32))
    flat2, body2 = _guarded_bf16(2 * M * N)
    B.gemm_grouped_1x128_128x1(qdyt, s1, qxt, s2, _cu(np.array([0, 100, 384], np.int32)), T,
                               out=body2.view(2, M, N))
    with pytest.raises(B.Bfp8Error, match="offsets"):
        B.check_device_errors()
    h2 = flat2.cpu().numpy()
    assert np.all(h2[:GUARD] == SENT) and np.all(h2[-GUARD:] == SENT)


@pytest.mark.parametrize("E,T,N,K", [(4, 1024, 256, 384), (8, 4096, 512, 1024)])
def test_moe_linear_matches_oracle(E, T, N, K):
    """The whole mixture-of-experts layer from bf16: forward, input gradient
    and weight gradient, experts on 128-token boundaries (one of them empty)."""
    rng = np.random.default_rng(E + T)
    offs = _offsets(rng, E, T, align=128, empty=(E - 2,))
    x = S.normal_bf16((T, K), 1.0, seed=51)
    w = S.normal_bf16((E * N, K), 0.02, seed=52).reshape(E, N, K)
    dy = S.normal_bf16((T, N), 1e-3, seed=53)
    dev = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    offs_d = _cu(offs)
    y, saved = B.moe_linear_fwd(dev(x), dev(w), offs_d)
    dx, dw = B.moe_linear_bwd(dev(dy), saved, offs_d)
    torch.cuda.synchronize()
    B.check_device_errors()
    assert_gemm_close(y.float().cpu().numpy().astype(np.float64), O.moe_linear_fwd(x, w, offs), "moe y")
    assert_gemm_close(dx.float().cpu().numpy().astype(np.float64), O.moe_linear_dgrad(dy, w, offs), "moe dx")
    ref_dw = O.moe_linear_wgrad(dy, x, offs)
    got_dw = dw.float().cpu().numpy().astype(np.float64)
    for e in range(E):
        if offs[e + 1] == offs[e]:
            assert np.all(got_dw[e] == 0.0)
        else:
            assert_gemm_close(got_dw[e], ref_dw[e], f"moe dW expert {e}")


@pytest.mark.parametrize("E,offs,T,N,K", [(4, [0, 256, 256, 640, 700], 700, 256, 384),  # an empty expert, ragged end
                                          (3, [5, 133, 133, 400], 410, 300, 200)])     # unaligned experts
def test_moe_step_host_matches_oracle(E, offs, T, N, K):
    """The mixture-of-experts step from host buffers, one dense step per
    expert with copies overlapped: against the oracle's per-expert forward,
    input gradient and weight gradient (zeros for an expert without tokens),
    and bit for bit against the grouped device path when the experts start on
    128-token boundaries."""
    offs = np.asarray(offs, np.int32)
    x = S.normal_bf16((T, K), 1.0, seed=71)
    w = S.normal_bf16((E * N, K), 0.02, seed=72).reshape(E, N, K)
    dy = S.normal_bf16((T, N), 1e-3, seed=73)
    host = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    m_max = int(np.max(np.diff(offs)))
    ws = B.moe_step_host_workspace(m_max, N, K)
    y, dx, dw = B.moe_step_host(host(x), host(w), host(dy), torch.from_numpy(offs), ws, chunk_n=128)
    torch.cuda.current_stream().synchronize()
    B.check_device_errors()
    inside = np.zeros(T, bool)
    inside[offs[0]:offs[-1]] = True
    f64 = lambda t: t.float().numpy().astype(np.float64)
    assert_gemm_close(f64(y)[inside], O.moe_linear_fwd(x, w, offs)[inside], "moe host y")
    assert_gemm_close(f64(dx)[inside], O.moe_linear_dgrad(dy, w, offs)[inside], "moe host dx")
    ref_dw = O.moe_linear_wgrad(dy, x, offs)
    got_dw = f64(dw)
    for e in range(E):
        if offs[e + 1] == offs[e]:
            assert np.all(got_dw[e] == 0.0)
        else:
            assert_gemm_close(got_dw[e], ref_dw[e], f"moe host dW expert {e}")
    if np.all(offs[:-1] % 128 == 0):
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
        offs_d = _cu(offs)
        gy, saved = B.moe_linear_fwd(dev(x), dev(w), offs_d)
        gdx, gdw = B.moe_linear_bwd(dev(dy), saved, offs_d)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16)[inside], gy.cpu().view(torch.int16)[inside])
        assert torch.equal(dx.view(torch.int16)[inside], gdx.cpu().view(torch.int16)[inside])
        assert torch.equal(dw.view(torch.int16), gdw.cpu().view(torch.int16))

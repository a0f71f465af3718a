"""Pins of the CPU oracle against facts the pages and the mathematics fix.

None of these compare the oracle with itself: each check uses a value the
pages print, a closed form, an invariant of the method, a library routine on a
special case, or a brute-force search.  A plausible slip in the oracle (a
dropped term, a sign, an index, a transposed operand, a wrong scale layout)
fails at least one of them.
"""
import os

import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def f32(x):
    return float(np.float32(x))


# ---------------------------------------------------------------- e4m3 codes

def test_e4m3_code_values_from_format_definition():
    for code, val in _read_table("e4m3_codes.txt"):
        got = O.e4m3_value(int(code, 16))
        assert got == float(val), (code, got, val)
        if val == "-0":
            assert np.signbit(got)
    assert np.isnan(O.e4m3_value(0x7F)) and np.isnan(O.e4m3_value(0xFF))


def test_e4m3_table_matches_torch_float8_e4m3fn():
    """Library special case: torch's float8_e4m3fn decoding of every code."""
    codes = torch.arange(256, dtype=torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = O.e4m3_table()
    both_nan = np.isnan(lib) & np.isnan(ours)
    assert np.all(both_nan | (lib == ours))
    assert np.sum(np.isnan(ours)) == 2
    finite = ours[~np.isnan(ours)]
    assert finite.max() == 448.0 and finite.min() == -448.0


def test_e4m3_rne_hand_cases():
    # ties to even: 1 + 1/16 lies halfway between 1.0 (0x38) and 1.125 (0x39)
    assert O.e4m3_rne(1.0625) == 0x38
    assert O.e4m3_rne(1.1875) == 0x3A
    # subnormal ties: 2^-10 is halfway between 0 and 2^-9 -> 0 ; 3*2^-10 -> 2*2^-9
    assert O.e4m3_rne(2.0 ** -10) == 0x00
    assert O.e4m3_rne(3 * 2.0 ** -10) == 0x02
    # just above a tie rounds up
    assert O.e4m3_rne(f32(np.nextafter(np.float32(1.0625), np.float32(2)))) == 0x39
    # clamp to +-448 (the method clamps before rounding)
    assert O.e4m3_rne(1e30) == 0x7E and O.e4m3_rne(-1e30) == 0xFE
    assert O.e4m3_rne(464.0) == 0x7E and O.e4m3_rne(447.9) == 0x7E
    # sign of zero kept (reading R4)
    assert O.e4m3_rne(0.0) == 0x00 and O.e4m3_rne(-0.0) == 0x80
    assert O.e4m3_rne(-1e-9) == 0x80
    # subnormal / normal boundary: 2^-6 - 2^-10 rounds up to 2^-6 (0x08)
    assert O.e4m3_rne(2.0 ** -6 - 2.0 ** -10) == 0x08


def test_e4m3_rne_against_torch_cast_in_range():
    """Library special case: torch's RNE cast to float8_e4m3fn agrees on every
    bf16 value inside [-448, 448] (torch does not saturate, so stay in range)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = S.bf16_bits_to_f32(bits)
    ok = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[ok]
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = O.cast_e4m3(v)
    # torch maps tiny negatives to 0x80 too; compare all bytes
    assert np.array_equal(lib, ours)


def test_e4m3_rne_brute_force_small():
    """Direct brute-force nearest search (all 127 magnitudes) on random and
    adversarial values."""
    rng = np.random.default_rng(5)
    vals = list(rng.standard_normal(2000).astype(np.float32) * 50)
    table = [O.e4m3_value(c) for c in range(0x7F)]
    for i in range(len(table) - 1):  # every midpoint and its neighbours
        mid = np.float32((table[i] + table[i + 1]) / 2)
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))]
    for v in vals:
        for s in (1.0, -1.0):
            r = f32(s * v)
            assert O.e4m3_rne(r) == O.e4m3_nearest(r), r


def test_e4m3_rne_exhaustive_sweep():
    """Every fp32 bit pattern with |r| < 512, both signs, against a nearest-code
    search; a stride sample of the rest (all clamp to +-448)."""
    n, first = O.sweep_cast(0x00000000, 0x44000000)          # +0 .. 512
    assert n == 0, hex(first)
    n, first = O.sweep_cast(0x80000000, 0xC4000000)          # -0 .. -512
    assert n == 0, hex(first)
    for lo in range(0x44000000, 0x7F800001, 0x00800000):     # one binade sample each
        n, first = O.sweep_cast(lo, lo + 4096)
        assert n == 0, hex(first)


# --------------------------------------------------------------- quantisation

def _deq(q):
    return O.e4m3_table()[q]


@pytest.mark.parametrize("M,K", [(3, 128), (5, 300), (130, 256), (64, 1000)])
def test_quant_lhs_dequant_error_bound(M, K):
    """|deq(q)*s - x| <= 2^-4 |x| (1 + 2^-20) in e4m3's normal range, and
    <= 2^-10 s (+ the fp32 rounding of x/s) in its subnormal range."""
    x = S.normal_bf16((M, K), 1.0, seed=M * 7 + K, outlier_frac=0.01)
    q, s = O.quant_lhs(x)
    xv = S.bf16_bits_to_f32(x).astype(np.float64)
    kb = np.arange(K) // 128
    sc = s.T[:, kb].astype(np.float64)     # s is column-major [M,Kb] -> s.T is [M,Kb]
    deq = _deq(q[:, :K]) * sc
    r = np.abs(xv / sc)
    err = np.abs(deq - xv)
    normal = r >= 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xv[normal]) * (1 + 2.0 ** -20))
    assert np.all(err[~normal] <= (2.0 ** -10 + 2.0 ** -30) * sc[~normal])


@pytest.mark.parametrize("M,K", [(4, 128), (130, 256), (7, 333)])
def test_quant_lhs_group_max_maps_to_448(M, K):
    """s = amax/448, so each group's largest |x| lands on +-448 (code 0x7E)."""
    x = S.normal_bf16((M, K), 3.0, seed=99)
    q, s = O.quant_lhs(x)
    xv = S.bf16_bits_to_f32(x)
    for m in range(M):
        for kb in range((K + 127) // 128):
            g = slice(kb * 128, min(K, kb * 128 + 128))
            i = np.argmax(np.abs(xv[m, g]))
            assert q[m, g][i] & 0x7F == 0x7E
            amax = np.abs(xv[m, g]).max()
            # scale is within one fp32 rounding of amax/448
            assert abs(float(s[kb, m]) - amax / 448.0) <= 2.0 ** -24 * amax / 448.0 * 1.0000001


def test_quant_lhs_brute_force_tiny():
    """Tiny tensors: every byte equals the brute-force nearest code of the
    fp32 quotient x/s, and s is the fp32 quotient amax/448."""
    for seed in range(6):
        x = S.normal_bf16((2, 16), 1.0 + seed, seed=seed)
        q, s = O.quant_lhs(x)
        xv = S.bf16_bits_to_f32(x)
        for m in range(2):
            amax = np.float32(np.abs(xv[m]).max())
            sc = np.float32(amax) / np.float32(448.0)
            assert s[0, m] == sc
            for k in range(16):
                assert q[m, k] == O.e4m3_nearest(f32(np.float32(xv[m, k]) / sc))


def test_quant_sign_symmetry_and_power_of_two_invariance():
    x = S.normal_bf16((6, 256), 1.0, seed=3)
    q, s = O.quant_lhs(x)
    qn, sn = O.quant_lhs(x ^ np.uint16(0x8000))          # negate every element
    assert np.array_equal(qn, q ^ np.uint8(0x80)) and np.array_equal(sn, s)
    for j in (-7, 5):
        xs = S.f32_to_bf16_bits(S.bf16_bits_to_f32(x) * np.float32(2.0 ** j))
        qs, ss = O.quant_lhs(xs)
        assert np.array_equal(qs, q)
        assert np.array_equal(ss, s * np.float32(2.0 ** j))


def test_quant_all_equal_and_all_zero_groups():
    v = S.f32_to_bf16_bits(np.full((2, 128), 0.3, dtype=np.float32))
    v[1] = S.f32_to_bf16_bits(np.full(128, -0.3, dtype=np.float32))
    q, s = O.quant_lhs(v)
    assert np.all(q[0] == 0x7E) and np.all(q[1] == 0xFE)
    amax = S.bf16_bits_to_f32(v[0, :1])[0]
    assert abs(448.0 * float(s[0, 0]) - amax) <= 2.0 ** -23 * amax
    # amax == 0 (reading R2): scale = fl32(1e-12/448), codes keep the sign
    z = np.zeros((2, 128), dtype=np.uint16)
    z[1, ::2] = 0x8000
    q, s = O.quant_lhs(z)
    assert np.all(s == np.float32(1e-12) / np.float32(448.0))
    assert np.all(q[0] == 0) and np.all(q[1, ::2] == 0x80) and np.all(q[1, 1::2] == 0)


@pytest.mark.parametrize("M,K", [(130, 256), (1, 129), (257, 127)])
def test_quant_lhs_touches_exactly_the_logical_tensor(M, K):
    """Masked tails: only rows m < M of the column-major scale tensor and only
    bytes k < K of each row are written (the pages' unmasked-store bug wrote
    rows >= M into the next K-block's column)."""
    x = S.normal_bf16((M, K), 1.0, seed=1)
    lds, ldq = M + 5, K + 16
    q, s = O.quant_lhs(x, ldq=ldq, lds=lds, q_fill=0xAB, s_fill=np.nan)
    assert np.all(q[:, K:] == 0xAB)
    assert np.all(np.isnan(s[:, M:]))
    assert np.all(np.isfinite(s[:, :M])) and np.all(s[:, :M] > 0)


def test_quant_lhs_transposed_equals_lhs_of_transpose():
    x = S.normal_bf16((300, 140), 1.0, seed=8)          # [K=300, M=140]
    qt, st = O.quant_lhs(x, transposed=True)
    q, s = O.quant_lhs(np.ascontiguousarray(x.T))
    assert np.array_equal(qt, q) and np.array_equal(st, s)


def test_quant_rhs_is_lhs_of_the_transpose():
    """128x1 groups along the rows of X are 1x128 groups along the columns of
    X^T; rhs bytes are written transposed, scales [Kb, N] row-major."""
    x = S.normal_bf16((260, 70), 1.0, seed=9)           # [K=260, N=70]
    qT, s = O.quant_rhs(x)
    q2, s2 = O.quant_lhs(np.ascontiguousarray(x.T))
    assert np.array_equal(qT, q2) and np.array_equal(s, s2)


def test_quant_weight_tile_scale_is_max_of_row_group_scales():
    """amax of a 128x128 tile is the max of its rows' 1x128 amaxes, and
    fl32(a/448) is monotone in a."""
    w = S.normal_bf16((300, 260), 0.02, seed=10)
    q, qt, s = O.quant_weight(w, with_t=True)
    _, sl = O.quant_lhs(w)
    for nb in range(3):
        for kb in range(3):
            assert s[nb, kb] == sl[kb, nb * 128:(nb + 1) * 128].max()
    assert np.array_equal(qt, q.T)
    # bytes: every element quantised with its tile's scale (brute force)
    wv = S.bf16_bits_to_f32(w)
    for (n, k) in [(0, 0), (129, 5), (299, 259), (200, 130), (17, 255)]:
        sc = np.float32(s[n // 128, k // 128])
        assert q[n, k] == O.e4m3_nearest(f32(np.float32(wv[n, k]) / sc))


# ----------------------------------------------------------------------- GEMM

def _int_codes(rng, shape, lo=-8, hi=8):
    """e4m3 codes of small integers (exact in e4m3), plus the integers."""
    ints = rng.integers(lo, hi + 1, size=shape)
    codes = O.cast_e4m3(ints.astype(np.float32))
    return codes, ints


@pytest.mark.parametrize("M,N,K", [(5, 7, 128), (33, 130, 300), (3, 256, 512)])
def test_gemm_integer_inputs_unit_scales_is_integer_matmul(M, N, K):
    rng = np.random.default_rng(M + N + K)
    qa, ia = _int_codes(rng, (M, K))
    qb, ib = _int_codes(rng, (N, K))
    Kb = (K + 127) // 128
    sa = np.ones((Kb, M), np.float32)
    sb = np.ones(((N + 127) // 128, Kb), np.float32)
    c = O.gemm(qa, sa, qb, sb, O.SB_TILE, K)
    assert np.array_equal(c, (ia @ ib.T).astype(np.float64))


@pytest.mark.parametrize("mode", [O.SB_TILE, O.SB_TILE_T, O.SB_COL])
def test_gemm_equals_matmul_of_expanded_dequantised_operands(mode):
    """sum_kb a_s b_s (A_kb . B_kb) == (A * a_s) @ (B * b_s)^T with the scales
    expanded to every element first (a different association of the same
    products); catches scale-layout, index and transposition slips."""
    rng = np.random.default_rng(int(mode) + 1)
    M, N, K = 37, 300, 520
    Kb, Nb = (K + 127) // 128, (N + 127) // 128
    qa = O.cast_e4m3(rng.standard_normal((M, K)).astype(np.float32) * 50)
    qb = O.cast_e4m3(rng.standard_normal((N, K)).astype(np.float32) * 50)
    sa = rng.uniform(0.5, 2, (Kb, M + 3)).astype(np.float32)      # lds > M
    if mode == O.SB_TILE:
        sb = rng.uniform(0.5, 2, (Nb, Kb + 1)).astype(np.float32)
        bscale = sb[np.arange(N)[:, None] // 128, np.arange(K)[None, :] // 128]
    elif mode == O.SB_TILE_T:
        sb = rng.uniform(0.5, 2, (Kb, Nb + 2)).astype(np.float32)
        bscale = sb[np.arange(K)[None, :] // 128, np.arange(N)[:, None] // 128]
    else:
        sb = rng.uniform(0.5, 2, (Kb, N + 1)).astype(np.float32)
        bscale = sb[np.arange(K)[None, :] // 128, np.arange(N)[:, None]]
    T = O.e4m3_table()
    A = T[qa] * sa[np.arange(K)[None, :] // 128, np.arange(M)[:, None]]
    B = T[qb] * bscale
    ref = A @ B.T
    c = O.gemm(qa, sa, qb, sb, mode, K)
    np.testing.assert_allclose(c, ref, rtol=1e-12, atol=1e-9 * np.abs(ref).max())


def test_gemm_one_hot_rows_and_single_block():
    rng = np.random.default_rng(4)
    N, K = 140, 128
    qb = O.cast_e4m3(rng.standard_normal((N, K)).astype(np.float32) * 20)
    qa = np.zeros((3, K), np.uint8)
    qa[0, 5] = 0x38          # 1.0
    qa[1, 127] = 0xC0        # -2.0
    qa[2, 0] = 0x38
    qa[2, 1] = 0x38
    sa = np.array([[0.5, 2.0, 1.0]], np.float32)
    sb = np.array([[3.0], [0.25]], np.float32)          # [Nb=2, Kb=1]
    c = O.gemm(qa, sa, qb, sb, O.SB_TILE, K)
    T = O.e4m3_table()
    bsc = np.where(np.arange(N) < 128, 3.0, 0.25)
    np.testing.assert_array_equal(c[0], 0.5 * bsc * T[qb[:, 5]])
    np.testing.assert_array_equal(c[1], 2.0 * bsc * -2.0 * T[qb[:, 127]])
    np.testing.assert_array_equal(c[2], bsc * (T[qb[:, 0]] + T[qb[:, 1]]))


def test_gemm_k_tail_uses_only_in_range_k():
    """Bytes past K in the operand rows (padding up to ld) never contribute."""
    rng = np.random.default_rng(6)
    M, N, K, ld = 4, 9, 200, 256
    qa = O.cast_e4m3(rng.standard_normal((M, ld)).astype(np.float32))
    qb = O.cast_e4m3(rng.standard_normal((N, ld)).astype(np.float32))
    sa = np.ones((2, M), np.float32)
    sb = np.ones((1, 2), np.float32)
    c1 = O.gemm(qa, sa, qb, sb, O.SB_TILE, K)
    qa2, qb2 = qa.copy(), qb.copy()
    qa2[:, K:] = 0x7E
    qb2[:, K:] = 0x7E
    assert np.array_equal(c1, O.gemm(qa2, sa, qb2, sb, O.SB_TILE, K))
    T = O.e4m3_table()
    np.testing.assert_allclose(c1, T[qa[:, :K]] @ T[qb[:, :K]].T, rtol=1e-13)


def test_gemm_sampled_rows_cols_match_full():
    x = S.normal_bf16((40, 300), 1.0, seed=12)
    w = S.normal_bf16((200, 300), 0.02, seed=13)
    full = O.linear_fwd(x, w)
    rows, cols = np.array([39, 0, 17]), np.array([199, 3, 128, 127])
    np.testing.assert_array_equal(O.linear_fwd(x, w, rows, cols), full[rows][:, cols])


# ------------------------------------------------------------------ SQNR pins

def _sqnr_cases():
    return [tuple(int(v) for v in r[:3]) + (float(r[3]),) for r in _read_table("sqnr_pages.txt")]


@pytest.mark.parametrize("M,N,K,pages_db", [c for c in _sqnr_cases() if c[0] * c[1] * c[2] <= 128 * 4096 * 4096])
def test_sqnr_matches_pages(M, N, K, pages_db):
    """The pages print 28.6-28.8 dB for the FP8 GEMM vs a BF16 matmul on these
    shapes; the oracle pipeline on N(0,1) data lands within 0.5 dB."""
    x = S.normal_bf16((M, K), 1.0, seed=11)
    w = S.normal_bf16((N, K), 1.0, seed=12)
    out = O.linear_fwd(x, w)
    ref = S.bf16_bits_to_f32(x).astype(np.float64) @ S.bf16_bits_to_f32(w).astype(np.float64).T
    db = O.sqnr_db(ref, out)
    assert abs(db - pages_db) <= 0.5, db


def test_sqnr_closed_form_band():
    """Per-operand e4m3 rounding noise (3 mantissa bits, uniform error of half
    a quantum) gives ~31.6 dB per operand and ~28.6 dB for the product of two;
    the oracle lands inside [28.0, 29.5] on an N(0,1) 64x1024x1024 problem, and
    the scale-invariance of block scaling keeps it there for N(0,0.02)."""
    for std in (1.0, 0.02):
        x = S.normal_bf16((64, 1024), 1.0, seed=21)
        w = S.normal_bf16((1024, 1024), std, seed=22)
        out = O.linear_fwd(x, w)
        ref = S.bf16_bits_to_f32(x).astype(np.float64) @ S.bf16_bits_to_f32(w).astype(np.float64).T
        assert 28.0 <= O.sqnr_db(ref, out) <= 29.5


def test_unmasked_scale_store_regression_is_catastrophic():
    """The pages' root-cause comment: rows >= M of the column-major lhs scale
    tensor, written without a mask, alias into the next K-block's column and
    collapse SQNR to 2-10 dB.  Planting that corruption into the oracle's
    scales drops SQNR far below 28 dB, so the SQNR gate catches the bug."""
    M, N, K = 2, 512, 1280
    x = S.normal_bf16((M, K), 1.0, seed=11)
    w = S.normal_bf16((N, K), 1.0, seed=12)
    qa, sa = O.quant_lhs(x)                       # lds == M
    qb, _, sb = O.quant_weight(w)
    ref = S.bf16_bits_to_f32(x).astype(np.float64) @ S.bf16_bits_to_f32(w).astype(np.float64).T
    good = O.gemm(qa, sa, qb, sb, O.SB_TILE, K)
    assert O.sqnr_db(ref, good) > 27.5
    # an autotuned group of 16 rows > M=2: rows 2..15 of column kb are written
    # with the scale of masked (zero) rows, landing on later columns' entries
    bad = sa.copy().reshape(-1)
    tiny = np.float32(1e-12) / np.float32(448)
    for kb in range(sa.shape[0]):
        for r in range(M, 16):
            idx = kb * M + r
            if idx < bad.size:
                bad[idx] = tiny
    c = O.gemm(qa, bad.reshape(sa.shape), qb, sb, O.SB_TILE, K)
    assert O.sqnr_db(ref, c) < 12.0


# ---------------------------------------------------------------- grouped (MoE)

def _finite_codes(rng, shape, scale=30.0):
    return O.cast_e4m3(rng.standard_normal(shape).astype(np.float32) * scale)


def test_moe_fwd_brute_force_tiny():
    """Each token row against its own expert's weight, looked up by scanning
    the offsets, with the scales expanded by hand; an empty expert and rows
    past the last offset included."""
    rng = np.random.default_rng(31)
    E, N, K, M = 3, 128, 200, 11
    offs = [0, 5, 5, 9]
    Kb = 2
    qa = _finite_codes(rng, (M, K))
    qw = _finite_codes(rng, (E * N, K))
    sa = rng.uniform(0.5, 2, (Kb, M)).astype(np.float32)
    sw = rng.uniform(0.5, 2, (E, Kb)).astype(np.float32)       # [E*Nb, Kb], Nb = 1
    got = O.moe_gemm_fwd(qa, sa, qw, sw, offs, N, K)
    T = O.e4m3_table()
    for m in range(M):
        e = next((g for g in range(E) if offs[g] <= m < offs[g + 1]), None)
        if e is None:
            assert np.all(np.isnan(got[m]))
            continue
        for n in range(0, N, 17):
            c = 0.0
            for kb in range(Kb):
                ks = slice(128 * kb, min(128 * kb + 128, K))
                c += float(sa[kb, m]) * float(sw[e, kb]) * float(np.dot(T[qa[m, ks]], T[qw[e * N + n, ks]]))
            assert abs(got[m, n] - c) <= 1e-12 * max(1.0, abs(c)), (m, n)


def test_moe_fwd_is_the_diagonal_blocks_of_one_dense_gemm():
    """Tokens x (all experts stacked) as one dense GEMM: expert e's block of
    that product, on e's token rows, is the grouped result."""
    rng = np.random.default_rng(32)
    E, N, K, M = 4, 256, 384, 300
    offs = [0, 70, 70, 200, 300]
    Kb, Nb = 3, 2
    qa = _finite_codes(rng, (M, K))
    qw = _finite_codes(rng, (E * N, K))
    sa = rng.uniform(0.5, 2, (Kb, M)).astype(np.float32)
    sw = rng.uniform(0.5, 2, (E * Nb, Kb)).astype(np.float32)
    full = O.gemm(qa, sa, qw, sw, O.SB_TILE, K)
    got = O.moe_gemm_fwd(qa, sa, qw, sw, offs, N, K)
    for e in range(E):
        r0, r1 = offs[e], offs[e + 1]
        np.testing.assert_array_equal(got[r0:r1], full[r0:r1, e * N:(e + 1) * N])


def test_moe_dgrad_equals_expanded_dequantised_product():
    """dY_e W_e with W_e's tile scales expanded to every element and the
    transposed codes un-transposed by hand."""
    rng = np.random.default_rng(33)
    E, N, K, M = 3, 256, 200, 50
    offs = [0, 20, 20, 50]
    Nb, Kb = 2, 2
    qdy = _finite_codes(rng, (M, N))
    qwt = _finite_codes(rng, (K, E * N))
    sdy = rng.uniform(0.5, 2, (Nb, M)).astype(np.float32)
    sw = rng.uniform(0.5, 2, (E * Nb, Kb)).astype(np.float32)
    got = O.moe_gemm_dgrad(qdy, sdy, qwt, sw, offs, N, K)
    T = O.e4m3_table()
    A = T[qdy] * sdy[np.arange(N)[None, :] // 128, np.arange(M)[:, None]]
    for e in range(E):
        r0, r1 = offs[e], offs[e + 1]
        We = T[qwt[:, e * N:(e + 1) * N]].T                                  # [N, K]
        We = We * sw[e * Nb + np.arange(N)[:, None] // 128, np.arange(K)[None, :] // 128]
        ref = A[r0:r1] @ We
        if r1 > r0:
            np.testing.assert_allclose(got[r0:r1], ref, rtol=1e-12, atol=1e-9 * np.abs(ref).max())


def test_moe_wgrad_sums_to_the_dense_weight_gradient():
    """With experts starting on 128-token boundaries the K-blocks of the dense
    weight gradient split between the experts, so the experts' gradients add
    up to the dense one; an expert without tokens gets exactly zero."""
    rng = np.random.default_rng(34)
    T_, N, K = 700, 130, 200
    offs = [0, 256, 256, 640, 700]
    Tb = 6
    qdyt = _finite_codes(rng, (N, T_))
    qxt = _finite_codes(rng, (K, T_))
    sdyt = rng.uniform(0.5, 2, (Tb, N)).astype(np.float32)
    sxt = rng.uniform(0.5, 2, (Tb, K)).astype(np.float32)
    got = O.moe_gemm_wgrad(qdyt, sdyt, qxt, sxt, offs)
    dense = O.gemm(qdyt, sdyt, qxt, sxt, O.SB_COL, T_)
    assert np.all(got[1] == 0.0)
    np.testing.assert_allclose(got.sum(axis=0), dense, rtol=1e-11, atol=1e-9 * np.abs(dense).max())
    # one expert alone is the dense GEMM with the other experts' tokens zeroed
    Z = O.e4m3_table()
    keep = np.zeros(T_, bool)
    keep[256:640] = True
    ref = (Z[qdyt] * sdyt[np.arange(T_)[None, :] // 128, np.arange(N)[:, None]] * keep) @ \
          (Z[qxt] * sxt[np.arange(T_)[None, :] // 128, np.arange(K)[:, None]]).T
    np.testing.assert_allclose(got[2], ref, rtol=1e-11, atol=1e-9 * np.abs(ref).max())


def test_moe_linear_with_shared_weights_is_the_dense_linear():
    """When every expert holds the same weight, grouping the tokens changes
    nothing: row-wise quantisation does not see the groups, and (experts on
    128-token boundaries) neither do the token-dim groups of the weight
    gradient, whose expert sums add up to the dense gradient."""
    M, N, K = 384, 256, 256
    offs = [0, 128, 128, 384]
    x = S.normal_bf16((M, K), 1.0, seed=41)
    w = S.normal_bf16((N, K), 0.02, seed=42)
    dy = S.normal_bf16((M, N), 1e-3, seed=43)
    ws = np.stack([w] * 3)
    np.testing.assert_array_equal(O.moe_linear_fwd(x, ws, offs), O.linear_fwd(x, w))
    np.testing.assert_array_equal(O.moe_linear_dgrad(dy, ws, offs), O.linear_dgrad(dy, w))
    dw = O.moe_linear_wgrad(dy, x, offs)
    ref = O.linear_wgrad(dy, x)
    np.testing.assert_allclose(dw.sum(axis=0), ref, rtol=1e-11, atol=1e-12 * np.abs(ref).max())
    assert np.all(dw[1] == 0.0)


# ---------------------------------------------------------------- MXFP8 casts

def _bf16_exponent_field(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.int64) >> 7) & 0xFF


def test_mx_exponent_is_the_largest_power_of_two_at_or_below_amax_over_all_bf16():
    """e + 8 is the exponent field of the bf16 amax minus the bias (normal
    values), clamped at -127 (zero, subnormals and amax < 2^-118): checked for
    every positive finite bf16 value from its bits, not from a logarithm."""
    bits = np.arange(1, 0x7F80, dtype=np.uint16)
    vals = S.bf16_bits_to_f32(bits)
    E = _bf16_exponent_field(bits)
    want = np.maximum(E - 127 - 8, -127)
    got = np.array([O.mx_exponent(float(v)) for v in vals[::7]])
    assert np.array_equal(got, want[::7])
    assert O.mx_exponent(0.0) == -127


def test_mx_quantize_one_is_the_nearest_code_of_the_scaled_value():
    """Brute-force nearest-code search (ties to even) on x * 2^-e, clamped."""
    rng = np.random.default_rng(71)
    xs = S.bf16_bits_to_f32(S.f32_to_bf16_bits(rng.standard_normal(400).astype(np.float32) * 100))
    for x in xs:
        for e in (-9, 0, 3, -127, 60):
            r = float(x) * 2.0 ** -e     # exact in double; the oracle's fp32 product rounds the same way
            r = float(np.float32(max(-1e30, min(1e30, r))))
            r = max(-448.0, min(448.0, r))
            assert O.mx_quantize_one(float(x), e) == O.e4m3_nearest(r), (x, e)


def test_mx_cast_block_maxima_reach_the_top_binade_and_errors_are_half_ulp():
    """With e = floor(log2 amax) - 8 the block maximum scales into [256, 512):
    its code is 256..448 (saturating above 448).  Every other element is
    within half an e4m3 ulp of x * 2^-e (or saturated at 448)."""
    x = S.normal_bf16((37, 200), 1.0, seed=72, outlier_frac=0.01)
    (q0, e0), _ = O.mx_cast(x, dim1=False)
    T = O.e4m3_table()
    xf = S.bf16_bits_to_f32(x).astype(np.float64)
    for m in range(x.shape[0]):
        for b in range(e0.shape[1]):
            blk = slice(32 * b, min(32 * b + 32, x.shape[1]))
            e = int(e0[m, b]) - 127
            r = xf[m, blk] * 2.0 ** -e
            d = T[q0[m, blk]]
            assert 256.0 <= np.abs(d).max() <= 448.0
            sat = np.abs(r) > 448.0
            assert np.all(np.abs(d[sat]) == 448.0)
            ulp = np.where(np.abs(r) >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -6))) - 3),
                           2.0 ** -9)
            assert np.all(np.abs(d[~sat] - r[~sat]) <= ulp[~sat] / 2 + 1e-30)


def test_mx_dim1_cast_is_the_dim0_cast_of_the_transpose_with_tails():
    x = S.normal_bf16((70, 45), 1.0, seed=73)
    (q0, e0), (q1, e1) = O.mx_cast(x)
    (qt0, et0), _ = O.mx_cast(np.ascontiguousarray(x.T), dim1=False)
    assert np.array_equal(q1, qt0) and np.array_equal(e1, et0)
    # tail blocks: the last 32-block of a row holds 45 - 32 = 13 elements, its
    # exponent comes from those alone
    xf = np.abs(S.bf16_bits_to_f32(x))
    for m in range(x.shape[0]):
        assert int(e0[m, 1]) - 127 == O.mx_exponent(float(xf[m, 32:].max()))


def test_mx_cast_power_of_two_invariance_and_zero_blocks():
    x = S.normal_bf16((8, 64), 1.0, seed=74)
    (q0, e0), _ = O.mx_cast(x, dim1=False)
    x4 = S.f32_to_bf16_bits(S.bf16_bits_to_f32(x) * np.float32(16.0))
    (q4, e4), _ = O.mx_cast(x4, dim1=False)
    assert np.array_equal(q0, q4) and np.array_equal(e4.astype(int), e0.astype(int) + 4)
    z = np.zeros((3, 40), np.uint16)
    z[1] = 0x8000  # -0
    (qz, ez), _ = O.mx_cast(z, dim1=False)
    assert np.all(ez == 0) and np.all(qz[0] == 0) and np.all(qz[1] == 0x80)

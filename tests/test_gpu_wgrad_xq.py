"""The weight-gradient GEMM that quantises its bf16 rhs itself
(bfp8_gemm_1x128_128x1_xq, the optional fused quantisation in the GEMM
prologue for the weight gradient's rhs) against the two-launch path it
replaces -- bfp8_quant_rhs of X, then bfp8_gemm_1x128_128x1 with the same
quantised dY^T -- bit for bit, and against the CPU oracle's weight gradient
within the GEMM tolerance ("Enable blockwise FP8 dense training kernels on
ROCm": act_quant_rhs 128x1, the 1x128 x 128x1 GEMM; "Mask a_s/b_s scale loads
in blockwise FP8 training GEMM kernels", Fix: masked scale loads and output
stores).  Shapes: tails in every dimension (rows of dW, features, tokens),
several tile rows and waves of tiles, deep token counts, padded rows of X,
K = 0, and the 8192-token 4096 x 4096 weight gradient on sampled outputs."""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from gpu_util import assert_gemm_close, dev_bf16, host_bf16_as_f64, torch

import blockwise_scaled_fp8_gb300 as B

pytestmark = pytest.mark.gpu

GUARD = 4096
SENT = 0x7FC1  # a bf16 NaN pattern no kernel writes


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    B.build()
    O.build()
    yield
    B.check_device_errors()


# (M rows of dW = output features, N = input features, K = tokens)
TAILS = [(1, 130, 256), (130, 300, 520), (257, 1000, 1024), (128, 128, 128), (200, 64, 4100), (64, 2051, 384)]
WAVES = [(1024, 4096, 1024), (2048, 2304, 512)]
DEEP = [(256, 512, 16384 + 96)]


def _guarded_out(M, N, ldc):
    flat = torch.full((M * ldc + 2 * GUARD,), SENT, dtype=torch.int16, device="cuda")
    return flat, flat[GUARD:GUARD + M * ldc].view(M, ldc).view(torch.bfloat16)


def _dev_x(x: np.ndarray, ldx: int):
    """X [K, N] on the device with row stride ldx >= N (a column slice)."""
    K, N = x.shape
    wide = np.zeros((K, ldx), dtype=x.dtype)
    wide[:, :N] = x
    return dev_bf16(wide)[:, :N]


def _inputs(M, N, K, seed):
    dy = S.normal_bf16((K, M), 1.0, seed=seed, outlier_frac=1e-3)   # dY [tokens, out features]
    x = S.normal_bf16((K, N), 1.0, seed=seed + 1, outlier_frac=1e-3)  # X [tokens, in features]
    return dy, x


@pytest.mark.parametrize("M,N,K", TAILS + WAVES + DEEP)
def test_wgrad_xq_bit_exact_with_two_launch_path_and_oracle(M, N, K):
    dy, x = _inputs(M, N, K, seed=M * 3 + N * 5 + K)
    ldx = (N + 7) // 8 * 8 + (8 if N % 16 else 0)
    xd = _dev_x(x, ldx)
    qa, sa = B.quant_lhs(dev_bf16(dy), transposed=True)
    qb, sb = B.quant_rhs(xd)
    ref = B.gemm_1x128_128x1(qa, sa, qb, sb, K, M=M, N=N)
    ldc = N + 8
    flat, out = _guarded_out(M, N, ldc)
    B.gemm_1x128_128x1_xq(qa, sa, xd, out=out[:, :N], M=M)
    torch.cuda.synchronize()
    B.check_device_errors()
    got = out[:, :N]
    assert torch.equal(got.contiguous().view(torch.int16), ref.view(torch.int16)), f"{M}x{N}x{K}: bits differ"
    h = flat.cpu().numpy()
    assert np.all(h[:GUARD] == SENT) and np.all(h[-GUARD:] == SENT), "write outside the output buffer"
    body = h[GUARD:GUARD + M * ldc].reshape(M, ldc)
    assert np.all(body[:, N:] == SENT), "write into the output's row padding"
    rows = np.unique(np.r_[0:M:max(1, M // 16), M - 1])
    assert_gemm_close(host_bf16_as_f64(got[torch.from_numpy(rows).cuda()]), O.linear_wgrad(dy, x, rows=rows),
                      f"wgrad xq {M}x{N}x{K} vs oracle")


def test_wgrad_xq_full_size_sampled():
    """dW = dY^T X over 8192 tokens, 4096 x 4096: the whole output bit-equal
    to the two-launch path; 16 rows x 256 columns against the oracle."""
    M, N, K = 4096, 4096, 8192
    dy, x = _inputs(M, N, K, seed=77)
    xd, dyd = dev_bf16(x), dev_bf16(dy)
    qa, sa = B.quant_lhs(dyd, transposed=True)
    qb, sb = B.quant_rhs(xd)
    ref = B.gemm_1x128_128x1(qa, sa, qb, sb, K)
    got = B.gemm_1x128_128x1_xq(qa, sa, xd)
    torch.cuda.synchronize()
    B.check_device_errors()
    diff = got.view(torch.int16) != ref.view(torch.int16)
    if bool(diff.any()):
        # say which side is off: both against the oracle at the first differing rows and columns
        idx = diff.nonzero().cpu().numpy()
        rows, cols = np.unique(idx[:, 0])[:4], np.unique(idx[:, 1])[:32]
        qa_o, sa_o = O.quant_lhs(np.ascontiguousarray(dy[:, rows]), transposed=True)
        qb_o, sb_o = O.quant_rhs(np.ascontiguousarray(x[:, cols]))
        want = O.gemm(qa_o, sa_o, qb_o, sb_o, O.SB_COL, K)
        tol = 2.0 ** -7 * np.abs(want) + 1e-3 * np.sqrt(np.mean(want ** 2))
        sel = lambda t: host_bf16_as_f64(t[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
        ok_ref, ok_got = np.mean(np.abs(sel(ref) - want) <= tol), np.mean(np.abs(sel(got) - want) <= tol)
        pytest.fail(f"bits differ from the two-launch path at {len(idx)} elements (rows {rows.tolist()}, "
                    f"columns from {int(cols[0])}); within the oracle bound there: two-launch {ok_ref:.3f}, "
                    f"fused {ok_got:.3f}")
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(M, 16, replace=False))
    cols = np.sort(np.r_[rng.choice(N - 128, 128, replace=False), np.arange(N - 128, N)])
    qa_o, sa_o = O.quant_lhs(np.ascontiguousarray(dy[:, rows]), transposed=True)
    qb_o, sb_o = O.quant_rhs(np.ascontiguousarray(x[:, cols]))
    want = O.gemm(qa_o, sa_o, qb_o, sb_o, O.SB_COL, K)
    have = host_bf16_as_f64(got[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
    assert_gemm_close(have, want, "wgrad xq 4096x4096x8192 sampled vs oracle")


def test_wgrad_xq_repeat_is_deterministic_and_empty_k_zeroes():
    dy, x = _inputs(384, 640, 1280, seed=91)
    xd = dev_bf16(x)
    qa, sa = B.quant_lhs(dev_bf16(dy), transposed=True)
    a = B.gemm_1x128_128x1_xq(qa, sa, xd)
    b = B.gemm_1x128_128x1_xq(qa, sa, xd)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    out = torch.full((4, 8), 1.0, dtype=torch.bfloat16, device="cuda")
    e = torch.zeros((0, 8), dtype=torch.bfloat16, device="cuda")
    B.gemm_1x128_128x1_xq(torch.zeros((4, 16), dtype=torch.uint8, device="cuda"),
                          torch.ones((1, 4), dtype=torch.float32, device="cuda"), e, out=out)
    torch.cuda.synchronize()
    assert torch.all(out.float() == 0)

"""The forward GEMM that quantises its bf16 A operand itself
(bfp8_gemm_1x128_128x128_xq) against the two-launch path it replaces --
bfp8_quant_lhs then bfp8_gemm_1x128_128x128 with the same quantised weight --
bit for bit, and against the CPU oracle's forward within the GEMM tolerance,
on the small-M shapes of "Enable blockwise FP8 dense training kernels on
ROCm" (M in {2, 4, 128, 512} x (N, K) in {(512, 128), (5120, 1280),
(3584, 640), (4096, 4096)}) and on tails (M and N not multiples of 128,
K tails, padded rows of x, several row blocks)."""
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


SMALL_M = [(m, n, k) for m in (2, 4, 128, 512) for (n, k) in ((512, 128), (5120, 1280), (3584, 640), (4096, 4096))]
TAILS = [(1, 130, 256), (3, 384, 136), (130, 300, 520), (257, 1000, 1024), (64, 2051, 128), (300, 640, 4096)]
# M <= 16 with enough columns that 128-column tiles fill more than half the
# SMs; 17..32 rows (the small-M kernel's 32-row form, its quantiser in two
# passes of 16 rows); 153 tiles of 128 columns (beyond one wave: the dense
# forward's tiles on both paths)
WIDE = [(4, 12288, 256), (16, 9856, 520), (24, 4096, 4096), (32, 5120, 1280), (17, 130, 520), (20, 19584, 256)]


def _guarded_out(M, N, ldc):
    flat = torch.full((M * ldc + 2 * GUARD,), SENT, dtype=torch.int16, device="cuda")
    return flat, flat[GUARD:GUARD + M * ldc].view(M, ldc).view(torch.bfloat16)


@pytest.mark.parametrize("M,N,K", SMALL_M + TAILS + WIDE)
def test_xq_forward_bit_exact_with_two_launch_path_and_oracle(M, N, K):
    x = S.normal_bf16((M, K), 1.0, seed=M * 7 + K, outlier_frac=1e-3)
    w = S.normal_bf16((N, K), 0.02, seed=N * 5 + K)
    xd, wd = dev_bf16(x), dev_bf16(w)
    qw, _, sw = B.quant_weight(wd)
    qa, sa = B.quant_lhs(xd)
    ref = B.gemm_1x128_128x128(qa, sa, qw, sw, K, M=M, N=N)
    ldc = N + 8
    flat, out = _guarded_out(M, N, ldc)
    B.gemm_1x128_128x128_xq(xd, qw, sw, out=out[:, :N], N=N)
    torch.cuda.synchronize()
    B.check_device_errors()
    got = out[:, :N]
    assert torch.equal(got.contiguous().view(torch.int16), ref.view(torch.int16)), f"{M}x{N}x{K}: bits differ"
    h = flat.cpu().numpy()
    assert np.all(h[:GUARD] == SENT) and np.all(h[-GUARD:] == SENT), "write outside the output buffer"
    body = h[GUARD:GUARD + M * ldc].reshape(M, ldc)
    assert np.all(body[:, N:] == SENT), "write into the output's row padding"
    rows = np.unique(np.r_[0:M:max(1, M // 16), M - 1])
    assert_gemm_close(host_bf16_as_f64(got[torch.from_numpy(rows).cuda()]), O.linear_fwd(x, w, rows=rows),
                      f"xq {M}x{N}x{K} vs oracle")


def test_xq_forward_padded_activation_rows():
    """x with a row stride above K (a column slice of a wider tensor)."""
    M, N, K, ld = 130, 512, 384, 520
    wide = S.normal_bf16((M, ld), 1.0, seed=91)
    w = S.normal_bf16((N, K), 0.02, seed=92)
    xd = dev_bf16(wide)[:, :K]
    qw, _, sw = B.quant_weight(dev_bf16(w))
    qa, sa = B.quant_lhs(xd)
    ref = B.gemm_1x128_128x128(qa, sa, qw, sw, K, M=M, N=N)
    got = B.gemm_1x128_128x128_xq(xd, qw, sw, N=N)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    x = np.ascontiguousarray(wide[:, :K])
    assert_gemm_close(host_bf16_as_f64(got), O.linear_fwd(x, w), "xq padded rows vs oracle")


def test_xq_forward_repeat_is_deterministic_and_empty_k_zeroes():
    x = dev_bf16(S.normal_bf16((4, 1280), 1.0, seed=93))
    qw, _, sw = B.quant_weight(dev_bf16(S.normal_bf16((5120, 1280), 0.02, seed=94)))
    a = B.gemm_1x128_128x128_xq(x, qw, sw)
    b = B.gemm_1x128_128x128_xq(x, qw, sw)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    out = torch.full((4, 8), 1.0, dtype=torch.bfloat16, device="cuda")
    e = torch.zeros((4, 8), dtype=torch.bfloat16, device="cuda")[:, :0]
    B.gemm_1x128_128x128_xq(e, torch.zeros((8, 16), dtype=torch.uint8, device="cuda"),
                            torch.ones((1, 1), dtype=torch.float32, device="cuda"), out=out, N=8)
    torch.cuda.synchronize()
    assert torch.all(out.float() == 0)

"""bfp8_linear_fwd_static: the linear forward for callers that cannot
allocate device memory (plugins hosted by a framework that owns every
allocation and hands them no allocator, or latency-critical code that must
not enter the driver's allocator).  It keeps its scratch in a fixed 32 MiB
array reserved by the library and runs the same launches as bfp8_linear_fwd
(which takes a caller workspace), so its results must equal those bit for
bit, call after call, since every call reuses the same array -- and meet the
oracle's bound.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import oracle as O
import synthetic as S
from gpu_util import assert_gemm_close, dev_bf16, host_bf16_as_f64, torch

import blockwise_scaled_fp8_gb300 as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    B.build()
    O.build()


def test_static_scratch_forward_matches_workspace_forward_on_two_calls():
    # two calls in a row with different problems: the second reuses the array
    # (and finds the first call's bytes in it)
    for (M, N, K, seed) in ((1024, 2048, 1024, 1), (300, 640, 520, 2), (4, 4096, 2048, 3)):
        x = S.normal_bf16((M, K), 1.0, seed=seed * 16, outlier_frac=1e-3)
        w = S.normal_bf16((N, K), 0.02, seed=seed * 16 + 1)
        xd, wd = dev_bf16(x), dev_bf16(w)
        ref = B.linear_fwd(xd, wd)
        got = B.linear_fwd_static(xd, wd)
        torch.cuda.synchronize()
        B.check_device_errors()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"static scratch {M}x{N}x{K}: bits differ"
        rows = np.unique(np.r_[0:M:max(1, M // 24), M - 1])
        assert_gemm_close(host_bf16_as_f64(got[torch.from_numpy(rows).cuda()]), O.linear_fwd(x, w, rows=rows),
                          f"static scratch {M}x{N}x{K} vs oracle")


def test_static_scratch_rejects_problems_beyond_its_size():
    L = B.lib()
    fake = ctypes.c_void_p(0x10000)
    # 8192 x 8192 x 8192 needs ~128 MiB of quantised operands
    st = L.bfp8_linear_fwd_static(fake, fake, fake, 8192, 8192, 8192, ctypes.c_void_p(None))
    assert st == B.BFP8_ERR_INVALID_ARG
    assert b"scratch" in L.bfp8_last_error()

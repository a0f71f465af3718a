"""Failure detection without a GPU fault: every wait in the GEMM kernels is
bounded in time.  A test hook makes the promotion warps wait on a barrier that
nothing arrives on (with a 50 ms limit); the kernel must give up, record the
timeout, release its resources and return, so that the host reads
BFP8_ERR_TIMEOUT and the context keeps working."""
import numpy as np
import pytest

import oracle as O
from gpu_util import assert_gemm_close, torch

import blockwise_scaled_fp8_gb300 as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    B.build()
    O.build()


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    qa = rng.integers(0, 0x7E, size=(M, K), dtype=np.uint8)
    qb = rng.integers(0, 0x7E, size=(N, K), dtype=np.uint8)
    sa = rng.uniform(0.5, 1.5, ((K + 127) // 128, M)).astype(np.float32)
    sb = rng.uniform(0.5, 1.5, ((N + 127) // 128, (K + 127) // 128)).astype(np.float32)
    return qa, sa, qb, sb


@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (256, 4096, 384), (2048, 4096, 384), (4, 512, 1024)])
def test_stalled_gemm_times_out_and_context_survives(M, N, K):
    """(256, 512, 384): the dense kernel's 32-column tiles (sixteen partial
    buffers); (256, 4096, 384): its 64-column tiles; (2048, 4096, 384): its
    256-column tiles with the staged TMA-store epilogue; (4, 512, 1024): the
    small-M kernel, each of its 4 tiles split over a cluster of 8 CTAs; every
    CTA gives up and the cluster's hand-over of partial sums still completes
    before any CTA leaves."""
    qa, sa, qb, sb = _operands(M, N, K, 1)
    cu = lambda a: torch.from_numpy(a).cuda()
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    B.check_device_errors()  # start clean
    assert B.debug_gemm_stall(cu(qa), cu(sa), cu(qb), cu(sb), K, out, wait_limit_us=50000) == B.BFP8_OK
    with pytest.raises(B.Bfp8Error) as err:
        B.check_device_errors()
    assert err.value.status == B.BFP8_ERR_TIMEOUT
    assert "partial-product" in str(err.value)
    # the flag was cleared and the context is usable: a normal GEMM is right
    B.check_device_errors()
    got = B.gemm_1x128_128x128(cu(qa), cu(sa), cu(qb), cu(sb), K)
    B.check_device_errors()
    ref = O.gemm(qa, sa, qb, sb, O.SB_TILE, K)
    assert_gemm_close(got.float().cpu().numpy().astype(np.float64), ref, "after timeout")

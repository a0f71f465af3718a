"""Helpers shared by the GPU parity tests."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def dev_bf16(bits: np.ndarray):
    """numpy bf16 bit patterns -> CUDA bf16 tensor with the same bytes."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_u8(t) -> np.ndarray:
    return t.cpu().numpy()


def host_f32(t) -> np.ndarray:
    return t.cpu().numpy()


def host_bf16_as_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_gemm_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    """|gpu - oracle| <= 2^-7 |oracle| + 1e-3 rms(oracle), element by element
    (the oracle accumulates in fp64 per K-block; the GPU in fp32 with a bf16
    output rounding, 2^-9 relative)."""
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    tol = 2.0 ** -7 * np.abs(ref) + 1e-3 * rms
    bad = np.abs(got - ref) > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())}/{ref.size} outside tolerance; first at {tuple(i)}: "
                             f"gpu={got[tuple(i)]!r} oracle={ref[tuple(i)]!r} rms={rms:.4g}")


def sqnr_db(ref: np.ndarray, out: np.ndarray) -> float:
    return float(10.0 * np.log10(np.sum(ref * ref) / np.sum((ref - out) ** 2)))

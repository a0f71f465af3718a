"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

Holds none of the method's arithmetic: only random bf16 tensors with the
shapes and value distributions of the blockwise FP8 dense-training workloads
(activations ~N(0,1), optionally with rare x100 outliers; weights ~N(0,0.02);
output gradients ~N(0,1e-3)).  Tensors are returned as bf16 bit patterns in a
numpy ``uint16`` array so that both sides see identical bytes.

Generator: numpy PCG64 seeded per tensor, float32 standard normals, scaled in
float32, rounded to bf16 (nearest, ties to even).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even); returns the uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(shape, std: float = 1.0, seed: int = 0, outlier_frac: float = 0.0,
                outlier_scale: float = 100.0) -> np.ndarray:
    """bf16 bits of N(0, std^2) samples; a Bernoulli(outlier_frac) subset is
    multiplied by outlier_scale."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if outlier_frac > 0.0:
        mask = rng.random(size=shape, dtype=np.float32) < np.float32(outlier_frac)
        a[mask] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(a)


def tensor_seed(config_seed: int, tensor_id: int) -> int:
    """Sub-tensor seeds of one workload: config_seed * 16 + tensor_id."""
    return config_seed * 16 + tensor_id


@dataclass
class Linear:
    """One blockwise-FP8 linear layer problem: x [M,K], W [N,K], dY [M,N]."""
    name: str
    M: int
    N: int
    K: int
    seed: int
    x_std: float = 1.0
    x_outliers: float = 0.0
    w_std: float = 0.02
    dy_std: float = 1e-3
    extra: dict = field(default_factory=dict)

    def x(self) -> np.ndarray:
        return normal_bf16((self.M, self.K), self.x_std, tensor_seed(self.seed, 0), self.x_outliers)

    def w(self) -> np.ndarray:
        return normal_bf16((self.N, self.K), self.w_std, tensor_seed(self.seed, 1))

    def dy(self) -> np.ndarray:
        return normal_bf16((self.M, self.N), self.dy_std, tensor_seed(self.seed, 2))

    @property
    def gemm_flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


# The workloads: shapes and distributions of the pages' tables.
TINY = Linear("tiny_130x384x256", M=130, N=384, K=256, seed=0, w_std=1.0)
FWD_MID = Linear("fwd_2048x4096x4096", M=2048, N=4096, K=4096, seed=1, x_outliers=1e-3)
FWD_SQUARE = Linear("fwd_8192x8192x8192", M=8192, N=8192, K=8192, seed=1, x_outliers=1e-3)
# weight gradient: dY [8192,4096] ~N(0,1e-3), X [8192,4096] ~N(0,1); dW [4096,4096]
WGRAD = Linear("wgrad_tokens8192_4096x4096", M=8192, N=4096, K=4096, seed=2)
SMALL_M = [Linear(f"small_m{m}_{n}x{k}", M=m, N=n, K=k, seed=3)
           for m in (2, 4, 128, 512) for (n, k) in ((512, 128), (5120, 1280), (3584, 640), (4096, 4096))]
MLP_UP = Linear("mlp_up_16384x14336x4096", M=16384, N=14336, K=4096, seed=4)


@dataclass
class MoE(Linear):
    """A mixture-of-experts layer: M tokens sorted by expert, E experts with
    weights W_e [N, K] stacked as [E*N, K]; expert e owns token rows
    offsets()[e] .. offsets()[e+1].  Each expert starts on a 128-token
    boundary; the split is uneven (seeded uniform cut points)."""
    E: int = 8

    def w(self) -> np.ndarray:
        return normal_bf16((self.E * self.N, self.K), self.w_std, tensor_seed(self.seed, 1))

    def offsets(self) -> np.ndarray:
        rng = np.random.Generator(np.random.PCG64(tensor_seed(self.seed, 3)))
        cuts = np.sort(rng.integers(0, self.M // 128 + 1, size=self.E - 1)) * 128
        return np.concatenate([[0], cuts, [self.M]]).astype(np.int32)


# the MLP-up problem routed over 8 experts: same token count and per-expert
# weight shape, so its GEMM rates compare with the dense ones
MOE_UP = MoE("moe_up_8x_16384x14336x4096", M=16384, N=14336, K=4096, seed=5, E=8)
# the mid problem routed over 8 experts (a size a full ncu capture handles)
MOE_MID = MoE("moe_mid_8x_4096x4096x4096", M=4096, N=4096, K=4096, seed=6, E=8)

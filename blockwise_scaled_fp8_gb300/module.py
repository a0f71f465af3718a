"""Autograd wrapper: a bf16 linear layer whose forward and backward run the
blockwise-FP8 training path of this library (the Float8BlockwiseLinear
computation that "Enable blockwise FP8 dense training kernels on ROCm" tests).

Forward: one launch quantises x (1x128 groups along K and 128x1 groups along
the token dim) and W (128x128 tiles, as is and transposed), then the forward
GEMM; the quantised operands stay in a per-call workspace.  Backward: dY is
quantised once (both forms), then the input-gradient and weight-gradient
GEMMs.  Every step runs in the library's kernels through the C ABI; this
module only reshapes, allocates outputs with torch and keeps the workspace
for the backward.  No bias: the method has none.
"""
from __future__ import annotations

import torch

from . import linear_bwd_saved, linear_fwd_train, linear_train_workspace


class _BlockwiseFp8Linear(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight):
        if x.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
            raise TypeError("blockwise_fp8_linear: x and weight must be bfloat16")
        lead = x.shape[:-1]
        K = x.shape[-1]
        N = weight.shape[0]
        if weight.shape[1] != K:
            raise ValueError(f"blockwise_fp8_linear: weight is {tuple(weight.shape)}, x has {K} features")
        x2 = x.reshape(-1, K).contiguous()
        M = x2.shape[0]
        ws = linear_train_workspace(M, N, K, device=x.device)
        y = linear_fwd_train(x2, weight.contiguous(), ws)
        ctx.save_for_backward(ws)
        ctx.dims = (M, N, K)
        ctx.lead = lead
        return y.reshape(*lead, N)

    @staticmethod
    def backward(ctx, dy):
        (ws,) = ctx.saved_tensors
        M, N, K = ctx.dims
        dy2 = dy.reshape(M, N).to(torch.bfloat16).contiguous()
        dx, dw = linear_bwd_saved(dy2, ws, M, N, K)
        return dx.reshape(*ctx.lead, K), dw


def blockwise_fp8_linear(x: torch.Tensor, weight: torch.Tensor) -> torch.Tensor:
    """y = x W^T with blockwise-FP8 forward and backward (x [..., K], weight [N, K], bf16)."""
    return _BlockwiseFp8Linear.apply(x, weight)


class Float8BlockwiseLinear(torch.nn.Module):
    """nn.Linear (no bias) in bf16 whose matmuls run as blockwise-scaled FP8 on the
    5th-generation tensor cores: 1x128 activation / gradient groups, 128x128 weight
    tiles, 128x1 groups for the weight gradient's right operand."""

    def __init__(self, in_features: int, out_features: int, device=None, dtype=torch.bfloat16):
        super().__init__()
        if dtype != torch.bfloat16:
            raise TypeError("Float8BlockwiseLinear keeps its weight in bfloat16")
        self.in_features, self.out_features = in_features, out_features
        self.weight = torch.nn.Parameter(torch.empty(out_features, in_features, device=device, dtype=dtype))
        torch.nn.init.kaiming_uniform_(self.weight, a=5 ** 0.5)

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear) -> "Float8BlockwiseLinear":
        if linear.bias is not None:
            raise ValueError("Float8BlockwiseLinear has no bias")
        m = cls(linear.in_features, linear.out_features, device=linear.weight.device)
        with torch.no_grad():
            m.weight.copy_(linear.weight.to(torch.bfloat16))
        return m

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return blockwise_fp8_linear(x, self.weight)

    def extra_repr(self) -> str:
        return f"in_features={self.in_features}, out_features={self.out_features}, bias=False"

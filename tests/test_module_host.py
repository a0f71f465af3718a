"""Host-side checks of the autograd module (no GPU): argument validation
happens before anything touches a device, and the module mirrors nn.Linear
without a bias."""
import pytest
import torch

import blockwise_scaled_fp8_gb300 as B


def test_module_rejects_other_dtypes_and_bias():
    with pytest.raises(TypeError):
        B.Float8BlockwiseLinear(256, 128, dtype=torch.float32)
    with pytest.raises(ValueError, match="no bias"):
        B.Float8BlockwiseLinear.from_linear(torch.nn.Linear(256, 128, bias=True))
    layer = B.Float8BlockwiseLinear(256, 128)
    assert layer.weight.shape == (128, 256) and layer.weight.dtype == torch.bfloat16
    assert "bias=False" in repr(layer)
    with pytest.raises(TypeError, match="bfloat16"):
        layer(torch.zeros(4, 256))                      # fp32 input
    with pytest.raises(ValueError, match="features"):
        layer(torch.zeros(4, 200, dtype=torch.bfloat16))  # wrong feature count


def test_module_from_linear_copies_the_weight():
    lin = torch.nn.Linear(256, 128, bias=False)
    layer = B.Float8BlockwiseLinear.from_linear(lin)
    assert torch.equal(layer.weight, lin.weight.detach().to(torch.bfloat16))


def test_host_step_binding_validates_before_any_device_call():
    x = torch.zeros(64, 128, dtype=torch.bfloat16)
    w = torch.zeros(256, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="dy"):
        B.linear_step_host(x, w, torch.zeros(64, 256), ws=None)       # fp32 dY
    with pytest.raises(ValueError, match="shapes"):
        B.linear_step_host(x, w, torch.zeros(64, 200, dtype=torch.bfloat16), ws=None)
    with pytest.raises(ValueError, match="offs"):
        B.moe_step_host(x, w.view(2, 128, 128), torch.zeros(64, 128, dtype=torch.bfloat16),
                        torch.zeros(3, dtype=torch.int64), ws=None)

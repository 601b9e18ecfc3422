"""Argument checks of the autograd wrapper, on the host (no GPU needed)."""
import pytest
import torch


def test_module_rejects_sizes_not_multiple_of_64():
    from quantize_block_scaled_amax_gb300.linear import NVFP4Linear
    with pytest.raises(ValueError):
        NVFP4Linear(100, 128, device="cpu")


def test_function_rejects_bad_inputs_before_any_launch():
    from quantize_block_scaled_amax_gb300.linear import nvfp4_linear
    x = torch.zeros(64, 128, dtype=torch.bfloat16)
    w = torch.zeros(64, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):          # CPU tensors
        nvfp4_linear(x, w)
    with pytest.raises(TypeError):           # fp32 input
        nvfp4_linear(x.float(), w)
    with pytest.raises(ValueError):          # K mismatch
        nvfp4_linear(x, torch.zeros(64, 192, dtype=torch.bfloat16))
    with pytest.raises(ValueError):          # M not a multiple of 64
        nvfp4_linear(torch.zeros(48, 128, dtype=torch.bfloat16), w)

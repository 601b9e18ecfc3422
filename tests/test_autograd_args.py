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


def test_precision_flag_and_switch():
    from quantize_block_scaled_amax_gb300.linear import NVFP4Linear, set_precision
    with pytest.raises(ValueError):
        NVFP4Linear(128, 128, device="cpu", precision="fp8")
    model = torch.nn.Sequential(NVFP4Linear(128, 256, device="cpu"), torch.nn.Identity(),
                                torch.nn.Sequential(NVFP4Linear(256, 128, device="cpu", precision="bf16")))
    assert [m.precision for m in model.modules() if isinstance(m, NVFP4Linear)] == ["nvfp4", "bf16"]
    assert set_precision(model, "bf16") == 2
    assert all(m.precision == "bf16" for m in model.modules() if isinstance(m, NVFP4Linear))
    assert "precision=bf16" in repr(model)
    assert set_precision(model[0], "nvfp4") == 1 and model[0].precision == "nvfp4"
    with pytest.raises(ValueError):
        set_precision(model, "fp16")


def test_bf16_function_rejects_bad_inputs_before_any_launch():
    from quantize_block_scaled_amax_gb300.linear import BF16LinearFunction
    w = torch.zeros(64, 128, dtype=torch.bfloat16)
    with pytest.raises(TypeError):           # fp32 input
        BF16LinearFunction.apply(torch.zeros(64, 128), w)
    with pytest.raises(ValueError):          # K mismatch
        BF16LinearFunction.apply(torch.zeros(64, 96, dtype=torch.bfloat16), w)
    with pytest.raises(ValueError):          # M not a multiple of 8
        BF16LinearFunction.apply(torch.zeros(12, 128, dtype=torch.bfloat16), w)

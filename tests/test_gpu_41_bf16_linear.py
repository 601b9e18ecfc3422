"""Layers kept in (or switched back to) BF16: the bf16 transpose kernel is
exact (a transpose is pure data movement, compared with numpy's), and the
BF16 layer's forward and both gradients match float64 products of the same
bf16 operands within the GEMM tolerance for bf16 results."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import assert_gemm_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    return nv


@pytest.mark.parametrize("shape", [(8, 8), (64, 40), (200, 136), (1024, 2056)])
def test_transpose_is_exact(nv, shape):
    x = workloads.normal_with_outliers(*shape, seed=shape[0] + shape[1], dtype=torch.bfloat16)
    y = nv.nvfp4_transpose_bf16(x.cuda())
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    np.testing.assert_array_equal(y.cpu().view(torch.int16).numpy(), x.view(torch.int16).numpy().T)


def test_transpose_of_a_strided_view_into_a_wider_output(nv):
    big = workloads.normal_with_outliers(96, 200, seed=3, dtype=torch.bfloat16).cuda()
    out = torch.full((136, 104), 7.0, dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_transpose_bf16(big[:, 16:152], out=out[:, :96])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out[:, :96].cpu().view(torch.int16).numpy(),
                                  big[:, 16:152].cpu().view(torch.int16).numpy().T)
    assert (out[:, 96:] == 7.0).all()           # columns past ldy's logical rows untouched


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("mnk", [(256, 384, 320), (128, 64, 1024)])
def test_bf16_layer_forward_and_gradients(nv, mnk):
    from quantize_block_scaled_amax_gb300.linear import NVFP4Linear
    m, n, k = mnk
    x, w, dy = workloads.linear_layer(m, n, k)
    x, w, dy = x.cuda(), w.cuda(), dy.cuda()
    layer = NVFP4Linear(k, n, device="cuda", precision="bf16")
    with torch.no_grad():
        layer.weight.copy_(w)
    xin = x.clone().requires_grad_(True)
    y = layer(xin)
    y.backward(dy)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    assert y.dtype == xin.grad.dtype == layer.weight.grad.dtype == torch.bfloat16
    xn, wn, dyn = _f64(x), _f64(w), _f64(dy)
    assert_gemm_close(_f64(y), oracle.bf16_gemm(xn, wn), xn, wn, bf16=True, what="Y = X W^T")
    assert_gemm_close(_f64(xin.grad), oracle.bf16_gemm(dyn, wn.T), dyn, wn.T, bf16=True, what="dX = dY W")
    assert_gemm_close(_f64(layer.weight.grad), oracle.bf16_gemm(dyn.T, xn.T), dyn.T, xn.T, bf16=True,
                      what="dW = dY^T X")


def test_switching_a_model_to_bf16_changes_its_gemms(nv):
    from quantize_block_scaled_amax_gb300.linear import NVFP4Linear, set_precision
    torch.manual_seed(0)
    model = torch.nn.Sequential(NVFP4Linear(256, 512, device="cuda"), NVFP4Linear(512, 256, device="cuda"))
    x = workloads.normal_with_outliers(128, 256, seed=9, dtype=torch.bfloat16).cuda()
    y4 = model(x)
    assert set_precision(model, "bf16") == 2
    y16 = model(x)
    torch.cuda.synchronize()
    # the BF16 model is the plain product chain of its bf16 weights
    w1 = _f64(model[1].weight)
    h = nv.nvfp4_gemm_bf16(x, model[0].weight)
    ref = oracle.bf16_gemm(_f64(h), w1)
    assert_gemm_close(_f64(y16), ref, _f64(h), w1, bf16=True, what="switched model")
    # and it differs from the NVFP4 model's output, which carries FP4 quantization error
    assert not torch.equal(y4, y16)
    rel = (y4.float() - y16.float()).norm() / y16.float().norm()
    assert 0.01 < rel.item() < 0.5

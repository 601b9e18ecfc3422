"""The torch.autograd wrapper (NVFP4Linear) runs exactly the C ABI's linear
calls: its outputs and gradients equal nvfp4_linear_fwd / nvfp4_linear_bwd
called directly with the same inputs and seeds, bit for bit."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    return nv


def _direct(nv, x2, w, gy2, sr_seed, rht_seed):
    m, k = x2.shape
    n = w.shape[0]
    ctx = nv.LinearContext(m, n, k, "cuda")
    y = nv.nvfp4_linear_fwd(x2, w, ctx)
    dx, dw = nv.nvfp4_linear_bwd(gy2, x2, ctx, sr_seed=sr_seed, rht_seed=rht_seed)
    return y, dx, dw


def test_module_matches_direct_calls(nv):
    from quantize_block_scaled_amax_gb300.linear import NVFP4Linear
    m, n, k = 256, 384, 320
    x, w, dy = workloads.linear_layer(m, n, k)
    x, w, dy = x.cuda(), w.cuda(), dy.cuda()
    layer = NVFP4Linear(k, n, device="cuda", seed_base=11, rht_seed=5)
    with torch.no_grad():
        layer.weight.copy_(w)
    xin = x.clone().requires_grad_(True)
    y = layer(xin)
    y.backward(dy)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    y_ref, dx_ref, dw_ref = _direct(nv, x, w, dy, 11, 5)
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)
    assert torch.equal(xin.grad, dx_ref)
    assert torch.equal(layer.weight.grad, dw_ref.to(torch.bfloat16))

    # the next backward draws the next stochastic-rounding seed
    layer.weight.grad = None
    xin.grad = None
    layer(xin).backward(dy)
    _, _, dw_next = _direct(nv, x, w, dy, 12, 5)
    torch.cuda.synchronize()
    assert torch.equal(layer.weight.grad, dw_next.to(torch.bfloat16))
    assert not torch.equal(dw_next, dw_ref)


def test_leading_dims_are_tokens(nv):
    from quantize_block_scaled_amax_gb300.linear import nvfp4_linear
    b, s, n, k = 2, 64, 128, 192
    x, w, dy = workloads.linear_layer(b * s, n, k)
    x, w, dy = x.cuda(), w.cuda(), dy.cuda()
    x3 = x.reshape(b, s, k).clone().requires_grad_(True)
    w_p = w.clone().requires_grad_(True)
    y3 = nvfp4_linear(x3, w_p, sr_seed=3, rht_seed=4)
    assert y3.shape == (b, s, n)
    y3.backward(dy.reshape(b, s, n))
    y_ref, dx_ref, dw_ref = _direct(nv, x, w, dy, 3, 4)
    torch.cuda.synchronize()
    assert torch.equal(y3.reshape(b * s, n), y_ref)
    assert torch.equal(x3.grad.reshape(b * s, k), dx_ref)
    assert torch.equal(w_p.grad, dw_ref.to(torch.bfloat16))

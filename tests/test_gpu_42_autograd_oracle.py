"""The autograd module NVFP4Linear against the oracle composition of the
recipe (paper page "Pretraining Large Language Models with NVFP4", recipe
paragraph: X 1x16 RTN and W 16x16 RTN for Fprop; dY 1x16 SR for Dgrad with
the 16x16 codes of W^T; the 16-point RHT along the tokens with SR on dY and
RTN on X for Wgrad; gradient accumulation in FP32).

Unlike the module-vs-direct-call test, nothing here is compared with the
CUDA path itself: Y, dX and dW are compared element by element with the
oracle's FP64 products of its own quantizations, so a wrong seed, a wrong
reshape of the leading dimensions or a swapped operand in the wrapper fails.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import assert_gemm_close, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    return nv


def _oracle_layer(xn, wn, dyn, sr_seed, rht_seed):
    """Y, dX, dW of the recipe as the oracle computes them (FP64 products of
    the dequantized operands), with the operands' dequantized values."""
    qx, qw = oracle.quantize(xn), oracle.quantize(wn, block="16x16")
    qdy = oracle.quantize(dyn, rounding="sr", seed=sr_seed)
    qwt = oracle.quantize(wn, layout="col", block="16x16")
    qdyt = oracle.quantize(dyn, layout="col", rounding="sr", seed=sr_seed, rht_seed=rht_seed)
    qxt = oracle.quantize(xn, layout="col", rht_seed=rht_seed)
    d = {k: oracle.dequantize(q) for k, q in dict(x=qx, w=qw, dy=qdy, wt=qwt, dyt=qdyt, xt=qxt).items()}
    return d, d["x"] @ d["w"].T, d["dy"] @ d["wt"].T, d["dyt"] @ d["xt"].T


def test_module_against_the_oracle(nv):
    from quantize_block_scaled_amax_gb300.linear import NVFP4Linear
    b, s, n, k = 2, 128, 384, 320          # tokens arrive as [batch, seq, features]
    m = b * s
    x, w, dy = workloads.linear_layer(m, n, k)
    xn, wn, dyn = to_f32_np(x), to_f32_np(w), to_f32_np(dy)
    layer = NVFP4Linear(k, n, device="cuda", seed_base=11, rht_seed=5)
    with torch.no_grad():
        layer.weight.copy_(w.cuda())
    x3 = x.cuda().reshape(b, s, k).clone().requires_grad_(True)
    y3 = layer(x3)
    y3.backward(dy.cuda().reshape(b, s, n))
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    assert y3.shape == (b, s, n) and x3.grad.shape == (b, s, k)
    assert layer.weight.grad.dtype == torch.bfloat16

    d, y_ref, dx_ref, dw_ref = _oracle_layer(xn, wn, dyn, sr_seed=11, rht_seed=5)
    assert_gemm_close(y3.detach().reshape(m, n).float().cpu().numpy(), y_ref, d["x"], d["w"], bf16=True, what="Y")
    assert_gemm_close(x3.grad.reshape(m, k).float().cpu().numpy(), dx_ref, d["dy"], d["wt"], bf16=True, what="dX")
    # dW: FP32 Wgrad, cast once to the bf16 parameter dtype
    assert_gemm_close(layer.weight.grad.float().cpu().numpy(), dw_ref, d["dyt"], d["xt"], bf16=True, what="dW")

    # the second backward draws the next stochastic-rounding seed (12)
    layer.weight.grad = None
    x3.grad = None
    layer(x3).backward(dy.cuda().reshape(b, s, n))
    torch.cuda.synchronize()
    d2, _, dx2_ref, dw2_ref = _oracle_layer(xn, wn, dyn, sr_seed=12, rht_seed=5)
    assert_gemm_close(x3.grad.reshape(m, k).float().cpu().numpy(), dx2_ref, d2["dy"], d2["wt"], bf16=True,
                      what="dX, second backward")
    assert_gemm_close(layer.weight.grad.float().cpu().numpy(), dw2_ref, d2["dyt"], d2["xt"], bf16=True,
                      what="dW, second backward")


def test_fp32_main_grad_accumulates_micro_batches(nv):
    # Two micro-batches through a layer with main_grad=True: weight.main_grad
    # must hold dW(batch 1, seed 21) + dW(batch 2, seed 22) accumulated in
    # FP32, and weight.grad stays unset.
    from quantize_block_scaled_amax_gb300.linear import NVFP4Linear
    m, n, k = 256, 384, 320
    layer = NVFP4Linear(k, n, device="cuda", seed_base=21, rht_seed=7, main_grad=True)
    x1, w, dy1 = workloads.linear_layer(m, n, k)
    x2 = workloads.activations(m, k, seed=workloads.SEED_BASE + 40)
    dy2 = workloads.gradients(m, n, seed=workloads.SEED_BASE + 41)
    with torch.no_grad():
        layer.weight.copy_(w.cuda())
    for xb, dyb in ((x1, dy1), (x2, dy2)):
        layer(xb.cuda().requires_grad_(True)).backward(dyb.cuda())
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    assert layer.weight.grad is None
    g = layer.weight.main_grad
    assert g.dtype == torch.float32 and g.shape == (n, k)

    wn = to_f32_np(w)
    da, _, _, dw_a = _oracle_layer(to_f32_np(x1), wn, to_f32_np(dy1), sr_seed=21, rht_seed=7)
    db, _, _, dw_b = _oracle_layer(to_f32_np(x2), wn, to_f32_np(dy2), sr_seed=22, rht_seed=7)
    # the sum of the two products is one product over the concatenated tokens
    a = np.concatenate([da["dyt"], db["dyt"]], axis=1)
    bm = np.concatenate([da["xt"], db["xt"]], axis=1)
    assert_gemm_close(g.cpu().numpy(), dw_a + dw_b, a, bm, bf16=False, what="main_grad")

    # the accumulation itself is one FP32 add per element: the same two Wgrad
    # GEMMs written out separately and added in FP32 give the same bits
    ctx = nv.LinearContext(m, n, k, "cuda")
    parts = []
    for xb, dyb, seed in ((x1, dy1, 21), (x2, dy2, 22)):
        nv.nvfp4_linear_fwd(xb.cuda(), w.cuda(), ctx)
        _, dwp = nv.nvfp4_linear_bwd(dyb.cuda(), xb.cuda(), ctx, sr_seed=seed, rht_seed=7)
        parts.append(dwp.clone())
    torch.cuda.synchronize()
    expect = (parts[0].cpu().numpy() + parts[1].cpu().numpy()).astype(np.float32)
    assert np.array_equal(g.cpu().numpy().view(np.uint32), expect.view(np.uint32))


def test_gemm_accumulate_into_fp32(nv):
    # nvfp4_gemm with accumulate=True adds into an FP32 C that already holds
    # values: C_after == fl32(C_before + C_product), bit for bit, including a
    # ragged edge (N not a multiple of the tile)
    m, n, k = 200, 136, 320
    a = workloads.normal_with_outliers(m, k, seed=51, dtype=torch.bfloat16).cuda()
    b = workloads.normal_with_outliers(n, k, std=0.05, seed=52, dtype=torch.bfloat16).cuda()
    qa, _ = nv.nvfp4_quantize(a)
    qb, _ = nv.nvfp4_quantize(b)
    prod = nv.nvfp4_gemm(qa, qb, out_dtype=torch.float32)
    base = workloads.normal_with_outliers(m, n, std=3.0, seed=53, device="cuda", dtype=torch.float32)
    c = base.clone()
    nv.nvfp4_gemm(qa, qb, out=c, accumulate=True)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    expect = (base.cpu().numpy() + prod.cpu().numpy()).astype(np.float32)
    assert np.array_equal(c.cpu().numpy().view(np.uint32), expect.view(np.uint32))
    with pytest.raises(ValueError):
        nv.nvfp4_gemm(qa, qb, out=torch.empty(m, n, dtype=torch.bfloat16, device="cuda"), accumulate=True)


def test_two_forwards_before_their_backwards(nv):
    # micro-batches whose forwards both run before either backward (as in a
    # pipelined schedule): each backward must use its own forward's X^T codes
    from quantize_block_scaled_amax_gb300.linear import NVFP4Linear
    m, n, k = 256, 384, 320
    x1, w, dy1 = workloads.linear_layer(m, n, k)
    x2 = workloads.activations(m, k, seed=workloads.SEED_BASE + 50)
    dy2 = workloads.gradients(m, n, seed=workloads.SEED_BASE + 51)
    layer = NVFP4Linear(k, n, device="cuda", seed_base=31, rht_seed=9)
    with torch.no_grad():
        layer.weight.copy_(w.cuda())
    xa, xb = x1.cuda().requires_grad_(True), x2.cuda().requires_grad_(True)
    ya, yb = layer(xa), layer(xb)
    yb.backward(dy2.cuda())                          # seed 31
    g_b = layer.weight.grad.clone()
    layer.weight.grad = None
    ya.backward(dy1.cuda())                          # seed 32
    g_a = layer.weight.grad.clone()
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    wn = to_f32_np(w)
    for xx, dd, seed, g, gx, tag in ((x2, dy2, 31, g_b, xb.grad, "second forward"),
                                     (x1, dy1, 32, g_a, xa.grad, "first forward")):
        d, _, dx_ref, dw_ref = _oracle_layer(to_f32_np(xx), wn, to_f32_np(dd), sr_seed=seed, rht_seed=9)
        assert_gemm_close(gx.float().cpu().numpy(), dx_ref, d["dy"], d["wt"], bf16=True, what=f"dX, {tag}")
        assert_gemm_close(g.float().cpu().numpy(), dw_ref, d["dyt"], d["xt"], bf16=True, what=f"dW, {tag}")

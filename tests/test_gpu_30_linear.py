"""The linear-layer entry points (Fprop, Dgrad, Wgrad with the recipe's
roundings and transforms) against the oracle composed step by step."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import assert_gemm_close, assert_quant_equal, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    return nv


@pytest.mark.parametrize("mnk", [(128, 128, 128), (256, 384, 320), (512, 1024, 768)])
def test_linear_fwd_bwd(nv, mnk):
    m, n, k = mnk
    x, w, dy = workloads.linear_layer(m, n, k)
    ctx = nv.LinearContext(m, n, k, "cuda")
    y = nv.nvfp4_linear_fwd(x.cuda(), w.cuda(), ctx)
    dx, dw = nv.nvfp4_linear_bwd(dy.cuda(), x.cuda(), ctx, sr_seed=workloads.SR_SEED, rht_seed=workloads.RHT_SEED)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    xn, wn, dyn = to_f32_np(x), to_f32_np(w), to_f32_np(dy)
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    o = {
        "xq": oracle.quantize(xn),
        "wq": oracle.quantize(wn, block="16x16"),
        "wtq": oracle.quantize(wn, layout="col", block="16x16"),
        "dyq": oracle.quantize(dyn, rounding="sr", seed=sr),
        "dytq": oracle.quantize(dyn, layout="col", rounding="sr", seed=sr, rht_seed=rh),
        "xtq": oracle.quantize(xn, layout="col", rht_seed=rh),
    }
    for name, ref in o.items():
        assert_quant_equal(getattr(ctx, name), ref, what=name)
    d = {name: oracle.dequantize(q) for name, q in o.items()}
    assert_gemm_close(y.float().cpu().numpy(), d["xq"] @ d["wq"].T, d["xq"], d["wq"], bf16=True, what="Y")
    assert_gemm_close(dx.float().cpu().numpy(), d["dyq"] @ d["wtq"].T, d["dyq"], d["wtq"], bf16=True, what="dX")
    assert_gemm_close(dw.cpu().numpy(), d["dytq"] @ d["xtq"].T, d["dytq"], d["xtq"], bf16=False, what="dW")
    # FP32-output twins of the layer's bf16 Fprop and Dgrad, on the same
    # quantized operands: the strict relative-Frobenius bound
    y32 = nv.nvfp4_gemm(ctx.xq, ctx.wq, out_dtype=torch.float32)
    dx32 = nv.nvfp4_gemm(ctx.dyq, ctx.wtq, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_gemm_close(y32.cpu().numpy(), d["xq"] @ d["wq"].T, d["xq"], d["wq"], bf16=False, what="Y fp32")
    assert_gemm_close(dx32.cpu().numpy(), d["dyq"] @ d["wtq"].T, d["dyq"], d["wtq"], bf16=False, what="dX fp32")
    # fidelity to the unquantized layer (a loose sanity bound, not parity)
    yr = xn.astype(np.float64) @ wn.astype(np.float64).T
    assert np.linalg.norm(y.float().cpu().numpy() - yr) / np.linalg.norm(yr) < 0.2


def test_forward_with_rht_matches_the_two_pass_layer(nv):
    # nvfp4_linear_fwd_rht quantizes X^T for Wgrad in the forward, from the
    # same read of X as xq; the backward then takes X = NULL.  Every
    # quantized operand and Y, dX, dW must equal the plain forward and the
    # backward's own X^T quantization bit for bit.
    m, n, k = 256, 384, 320
    x, w, dy = workloads.linear_layer(m, n, k)
    x, w, dy = x.cuda(), w.cuda(), dy.cuda()
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    a = nv.LinearContext(m, n, k, "cuda")
    ya = nv.nvfp4_linear_fwd(x, w, a)
    dxa, dwa = nv.nvfp4_linear_bwd(dy, x, a, sr_seed=sr, rht_seed=rh)
    b = nv.LinearContext(m, n, k, "cuda")
    yb = nv.nvfp4_linear_fwd(x, w, b, rht_seed=rh)
    xtq_fwd = b.xtq.codes.clone()
    dxb, dwb = nv.nvfp4_linear_bwd(dy, None, b, sr_seed=sr, rht_seed=rh)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    assert torch.equal(xtq_fwd, b.xtq.codes)        # the backward left xtq as the forward wrote it
    for name in ("xq", "wq", "wtq", "dyq", "dytq", "xtq"):
        qa, qb = getattr(a, name), getattr(b, name)
        assert torch.equal(qa.codes, qb.codes) and torch.equal(qa.scales, qb.scales), name
        assert torch.equal(qa.amax[:3], qb.amax[:3]), name      # {A, S_dec, S_enc}
    assert torch.equal(ya, yb) and torch.equal(dxa, dxb) and torch.equal(dwa, dwb)
    assert_quant_equal(b.xtq, oracle.quantize(to_f32_np(x), layout="col", rht_seed=rh), what="xtq from the forward")

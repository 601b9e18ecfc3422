"""The FFN block's two linears over the token sweep (up 5120 -> 20480 and
down 20480 -> 5120, M in {2048, 8192, 32768}; bf16 N(0,1) activations,
N(0, 0.02) weights, Student-t gradients), fwd + bwd through
nvfp4_linear_fwd / nvfp4_linear_bwd.  Sampled rows of every quantized
operand must match the oracle bit for bit (the oracle takes the amax of the
whole tensor), and sampled entries of Y, dX and dW must meet the GEMM
tolerance against the oracle's products of those rows."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import assert_gemm_close, assert_quant_equal, to_f32_np

pytestmark = pytest.mark.gpu

D_MODEL, D_FFN = 5120, 20480


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    return nv


def _row(q, r):
    """dequantized row r of a sampled oracle quantization keyed by its start row"""
    return oracle.dequantize(q)[r - q["row0"]]


@pytest.mark.parametrize("m, which", [(2048, "up"), (2048, "down"), (8192, "up"), (8192, "down"), (32768, "up"),
                                      (32768, "down")])
def test_ffn_linear_sampled(nv, m, which):
    n, k = (D_FFN, D_MODEL) if which == "up" else (D_MODEL, D_FFN)
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    x = workloads.activations(m, k, outliers=False, device="cuda")
    w = workloads.weights(n, k, device="cuda")
    dy = workloads.gradients(m, n, device="cuda")
    ctx = nv.LinearContext(m, n, k, "cuda")
    y = nv.nvfp4_linear_fwd(x, w, ctx)
    dx, dw = nv.nvfp4_linear_bwd(dy, x, ctx, sr_seed=sr, rht_seed=rh)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK

    xn, wn, dyn = to_f32_np(x), to_f32_np(w), to_f32_np(dy)
    lx, lw, lwt = xn, wn, np.ascontiguousarray(wn.T)
    ldy = dyn
    ldyt = oracle.logical_tensor(dyn, "col", rh)
    lxt = oracle.logical_tensor(xn, "col", rh)
    rm = [0, m // 2 + 17, m - 1]          # token rows
    rn = [5, n // 2 + 3, n - 1]           # output-feature rows
    rk = [0, k // 3 + 1, k - 1]           # input-feature rows

    def q16(lt, r, **kw):                 # 16x16 tiles: quantize the tile's 16 rows
        r0 = 16 * (r // 16)
        return oracle.quantize(None, logical=lt, rows=(r0, r0 + 16), block="16x16", **kw)

    def q1(lt, r, **kw):
        return oracle.quantize(None, logical=lt, rows=(r, r + 1), **kw)

    ox = {r: q1(lx, r) for r in rm}
    ow = {r: q16(lw, r) for r in rn}
    owt = {r: q16(lwt, r) for r in rk}
    ody = {r: q1(ldy, r, rounding="sr", seed=sr) for r in rm}
    odyt = {r: q1(ldyt, r, rounding="sr", seed=sr) for r in rn}
    oxt = {r: q1(lxt, r) for r in rk}
    for name, got, refs in (("xq", ctx.xq, ox), ("dyq", ctx.dyq, ody), ("dytq", ctx.dytq, odyt),
                            ("xtq", ctx.xtq, oxt)):
        for r, ref in refs.items():
            assert_quant_equal(got, ref, rows=(r, r + 1), what=f"{which} M={m} {name} row {r}")
    for name, got, refs in (("wq", ctx.wq, ow), ("wtq", ctx.wtq, owt)):
        for r, ref in refs.items():
            r0 = 16 * (r // 16)
            assert_quant_equal(got, ref, rows=(r0, r0 + 16), what=f"{which} M={m} {name} tile rows {r0}")

    a = np.stack([_row(ox[r], r) for r in rm])
    b = np.stack([_row(ow[r], r) for r in rn])
    assert_gemm_close(y[rm][:, rn].float().cpu().numpy(), a @ b.T, a, b, bf16=True, what=f"{which} M={m} Y")
    a = np.stack([_row(ody[r], r) for r in rm])
    b = np.stack([_row(owt[r], r) for r in rk])
    assert_gemm_close(dx[rm][:, rk].float().cpu().numpy(), a @ b.T, a, b, bf16=True, what=f"{which} M={m} dX")
    a = np.stack([_row(odyt[r], r) for r in rn])
    b = np.stack([_row(oxt[r], r) for r in rk])
    assert_gemm_close(dw[rn][:, rk].cpu().numpy(), a @ b.T, a, b, bf16=False, what=f"{which} M={m} dW")

    # FP32-output twins of Fprop and Dgrad on the same quantized operands
    # (the layer returns bf16 Y and dX): the strict relative-Frobenius bound
    # over the sampled entries
    y32 = nv.nvfp4_gemm(ctx.xq, ctx.wq, out_dtype=torch.float32)
    dx32 = nv.nvfp4_gemm(ctx.dyq, ctx.wtq, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    a = np.stack([_row(ox[r], r) for r in rm])
    b = np.stack([_row(ow[r], r) for r in rn])
    assert_gemm_close(y32[rm][:, rn].cpu().numpy(), a @ b.T, a, b, bf16=False, what=f"{which} M={m} Y fp32")
    a = np.stack([_row(ody[r], r) for r in rm])
    b = np.stack([_row(owt[r], r) for r in rk])
    assert_gemm_close(dx32[rm][:, rk].cpu().numpy(), a @ b.T, a, b, bf16=False, what=f"{which} M={m} dX fp32")

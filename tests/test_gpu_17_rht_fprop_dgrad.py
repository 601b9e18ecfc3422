"""The 16-point RHT on the Fprop and Dgrad operands (transform along each
GEMM's K), through nvfp4_rht_quantize_rowwise and nvfp4_rht_quantize:
quantization bit-exact against the oracle, GEMMs within tolerance, and the
shared transform cancelling in the product."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import amax_np, assert_gemm_close, assert_quant_equal, codes_np, scales_np, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    return nv


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_rht_rowwise_nvfp4(nv, dtype, rounding):
    x = workloads.normal_with_outliers(160, 1056, p=0.002, factor=40.0, seed=31, dtype=dtype)
    q = nv.nvfp4_rht_quantize_rowwise(x.cuda(), round=rounding, seed=4, rht_seed=9, scale_layout="linear")
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    assert_quant_equal(q, oracle.quantize(to_f32_np(x), rounding=rounding, seed=4, rht_seed=9), what="rht rows")


def test_rht_rowwise_mxfp4(nv):
    x = workloads.normal_with_outliers(96, 512, seed=32, dtype=torch.bfloat16)
    q = nv.nvfp4_rht_quantize_rowwise(x.cuda(), round="sr", seed=4, rht_seed=9, fmt="mxfp4")
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    ora = oracle.quantize(to_f32_np(x), block="mx1x32", rounding="sr", seed=4, rht_seed=9)
    assert amax_np(q).tolist() == [0.0, 1.0, 1.0]
    assert np.array_equal(scales_np(q), np.repeat(ora["scales"], 2, axis=1))
    assert np.array_equal(codes_np(q), ora["codes"])


def test_fprop_and_dgrad_with_rht(nv):
    m, n, k = 256, 384, 512
    x, w, dy = workloads.linear_layer(m, n, k)
    xc, wc, dyc = x.cuda(), w.cuda(), dy.cuda()
    rh = 12
    # Fprop: X and W transformed along K
    qx = nv.nvfp4_rht_quantize_rowwise(xc, rht_seed=rh)
    qw = nv.nvfp4_rht_quantize_rowwise(wc, rht_seed=rh)
    y = nv.nvfp4_gemm(qx, qw, out_dtype=torch.float32)
    # Dgrad: dY transformed along N (its rows), W^T transformed along N (W's rows)
    qdy = nv.nvfp4_rht_quantize_rowwise(dyc, round="sr", seed=5, rht_seed=rh)
    qwt = nv.nvfp4_rht_quantize(wc, rht_seed=rh)
    dx = nv.nvfp4_gemm(qdy, qwt, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    xn, wn, dyn = to_f32_np(x), to_f32_np(w), to_f32_np(dy)
    ox, ow = oracle.quantize(xn, rht_seed=rh), oracle.quantize(wn, rht_seed=rh)
    ody = oracle.quantize(dyn, rounding="sr", seed=5, rht_seed=rh)
    owt = oracle.quantize(wn, layout="col", rht_seed=rh)
    for got, ref, name in ((qx, ox, "X"), (qw, ow, "W"), (qdy, ody, "dY"), (qwt, owt, "W^T")):
        assert_quant_equal(got, ref, what=name)
    ax, aw, ady, awt = (oracle.dequantize(o) for o in (ox, ow, ody, owt))
    assert_gemm_close(y.cpu().numpy(), ax @ aw.T, ax, aw, bf16=False, what="Y with RHT")
    assert_gemm_close(dx.cpu().numpy(), ady @ awt.T, ady, awt, bf16=False, what="dX with RHT")
    # the shared transform cancels: both products approximate the unquantized ones
    yr = xn.astype(np.float64) @ wn.astype(np.float64).T
    dxr = dyn.astype(np.float64) @ wn.astype(np.float64)
    assert np.linalg.norm(y.cpu().numpy() - yr) / np.linalg.norm(yr) < 0.2
    assert np.linalg.norm(dx.cpu().numpy() - dxr) / np.linalg.norm(dxr) < 0.2

"""GPU parity of the block-scaled FP4 GEMM (tcgen05) against the oracle's
FP64 product of the dequantized operands, through the C ABI.

Tolerance (FP32 output): relative Frobenius 1e-5 and per element
1e-3 * ||A^_row|| * ||B^_col|| / sqrt(K); bf16 output: per element one bf16
ulp of the reference plus the same bound.
"""
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
    assert torch.cuda.is_available()
    return nv


@pytest.mark.parametrize("a_round", ["rtn", "sr"])
def test_tiny_config(nv, a_round):
    # A fp32 128x256 and B fp32 256x256, N(0,1) with 0.5% of entries x40;
    # C = A B with B quantized colwise (blocks along K = 256)
    a, b = workloads.tiny()
    an, bn = a.numpy(), b.numpy()
    qa, _ = nv.nvfp4_quantize(a.cuda(), round=a_round, seed=workloads.SR_SEED)
    _, qb = nv.nvfp4_quantize(b.cuda(), rowwise=False, colwise=True)
    c32 = nv.nvfp4_gemm(qa, qb, out_dtype=torch.float32)
    c16 = nv.nvfp4_gemm(qa, qb, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    oa = oracle.quantize(an, rounding=a_round, seed=workloads.SR_SEED)
    ob = oracle.quantize(bn, layout="col")
    assert_quant_equal(qa, oa, what="A")
    assert_quant_equal(qb, ob, what="B^T")
    ad, bd = oracle.dequantize(oa), oracle.dequantize(ob)
    ref = ad @ bd.T
    assert_gemm_close(c32.cpu().numpy(), ref, ad, bd, bf16=False, what="tiny fp32")
    assert_gemm_close(c16.float().cpu().numpy(), ref, ad, bd, bf16=True, what="tiny bf16")


# N against the 384-column tile (chain 0: columns 0-255, chain 1: 256-383):
# chain 1 out of range (128, 136, 256, 48), partly in range (320, 704: 384 +
# 320), whole tiles (384), a ragged last tile of two (512) and of three (1000)
@pytest.mark.parametrize("mnk", [(128, 128, 64), (128, 128, 256), (200, 136, 320), (384, 512, 1024),
                                 (64, 1000, 512), (1000, 48, 128), (256, 256, 4096), (128, 320, 256),
                                 (256, 384, 512), (130, 704, 192)])
def test_shapes(nv, mnk):
    m, n, k = mnk
    a = workloads.normal_with_outliers(m, k, p=0.005, factor=20.0, seed=m + k, dtype=torch.bfloat16)
    b = workloads.normal_with_outliers(n, k, std=0.05, seed=n + 3 * k, dtype=torch.bfloat16)
    qa, _ = nv.nvfp4_quantize(a.cuda(), round="sr", seed=2)
    qb, _ = nv.nvfp4_quantize(b.cuda())
    c32 = nv.nvfp4_gemm(qa, qb, out_dtype=torch.float32)
    c16 = nv.nvfp4_gemm(qa, qb, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    oa = oracle.quantize(to_f32_np(a), rounding="sr", seed=2)
    ob = oracle.quantize(to_f32_np(b))
    ad, bd = oracle.dequantize(oa), oracle.dequantize(ob)
    ref = ad @ bd.T
    assert_gemm_close(c32.cpu().numpy(), ref, ad, bd, bf16=False, what=f"{mnk} fp32")
    assert_gemm_close(c16.float().cpu().numpy(), ref, ad, bd, bf16=True, what=f"{mnk} bf16")


def test_output_row_stride(nv):
    m, n, k = 256, 128, 256
    a = workloads.normal_with_outliers(m, k, seed=1, dtype=torch.bfloat16)
    b = workloads.normal_with_outliers(n, k, seed=2, dtype=torch.bfloat16)
    qa, _ = nv.nvfp4_quantize(a.cuda())
    qb, _ = nv.nvfp4_quantize(b.cuda())
    big = torch.full((m, 200), 7.0, dtype=torch.float32, device="cuda")
    nv.nvfp4_gemm(qa, qb, out=big[:, :n])
    torch.cuda.synchronize()
    assert torch.all(big[:, n:] == 7.0)
    ad = oracle.dequantize(oracle.quantize(to_f32_np(a)))
    bd = oracle.dequantize(oracle.quantize(to_f32_np(b)))
    assert_gemm_close(big[:, :n].cpu().numpy(), ad @ bd.T, ad, bd, bf16=False, what="strided C")


def _sample_rows(n, size=128):
    return sorted({0, (n // 2 // size) * size, n - size})


def test_full_size_fprop(nv):
    # X 8192x5120 (1x16 RTN) times W^T, W 20480x5120 (16x16 RTN) -> 8192x20480
    x = workloads.activations(device="cuda")
    w = workloads.weights(device="cuda")
    qx, _ = nv.nvfp4_quantize(x)
    qw, _ = nv.nvfp4_quantize(w, block="16x16")
    y16 = nv.nvfp4_gemm(qx, qw, out_dtype=torch.bfloat16)
    y32 = nv.nvfp4_gemm(qx, qw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    wd = oracle.dequantize(oracle.quantize(to_f32_np(w), block="16x16"))
    xn = to_f32_np(x)
    for r0 in _sample_rows(8192):
        xd = oracle.dequantize(oracle.quantize(xn, rows=(r0, r0 + 128)))
        ref = xd @ wd.T
        assert_gemm_close(y32[r0:r0 + 128].cpu().numpy(), ref, xd, wd, bf16=False, what=f"Fprop fp32 rows {r0}")
        assert_gemm_close(y16[r0:r0 + 128].float().cpu().numpy(), ref, xd, wd, bf16=True,
                          what=f"Fprop bf16 rows {r0}")


def test_full_size_dgrad(nv):
    # dX[8192][5120] = dY (1x16 SR) times W (16x16 codes of W^T): a K = 20480
    # reduction.  The bf16 output the layer returns, and its FP32-output twin,
    # which must meet the strict relative-Frobenius bound over the sampled rows.
    dy = workloads.gradients(device="cuda")
    w = workloads.weights(device="cuda")
    qdy, _ = nv.nvfp4_quantize(dy, round="sr", seed=workloads.SR_SEED)
    _, qwt = nv.nvfp4_quantize(w, block="16x16", rowwise=False, colwise=True)
    dx = nv.nvfp4_gemm(qdy, qwt, out_dtype=torch.bfloat16)
    dx32 = nv.nvfp4_gemm(qdy, qwt, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    wtd = oracle.dequantize(oracle.quantize(to_f32_np(w), layout="col", block="16x16"))
    dyn = to_f32_np(dy)
    for r0 in _sample_rows(8192):
        dyd = oracle.dequantize(oracle.quantize(dyn, rounding="sr", seed=workloads.SR_SEED, rows=(r0, r0 + 128)))
        ref = dyd @ wtd.T
        assert_gemm_close(dx32[r0:r0 + 128].cpu().numpy(), ref, dyd, wtd, bf16=False, what=f"Dgrad fp32 rows {r0}")
        assert_gemm_close(dx[r0:r0 + 128].float().cpu().numpy(), ref, dyd, wtd, bf16=True,
                          what=f"Dgrad bf16 rows {r0}")


def test_full_size_wgrad(nv):
    # dW[20480][5120] = (H dY)^T (H X), SR on dY, RTN on X, FP32 out
    dy = workloads.gradients(device="cuda")
    x = workloads.activations(outliers=False, device="cuda")
    qa = nv.nvfp4_rht_quantize(dy, round="sr", seed=workloads.SR_SEED, rht_seed=workloads.RHT_SEED)
    qb = nv.nvfp4_rht_quantize(x, round="rtn", rht_seed=workloads.RHT_SEED)
    dw = nv.nvfp4_gemm(qa, qb, out_dtype=torch.float32)
    torch.cuda.synchronize()
    bd = oracle.dequantize(oracle.quantize(to_f32_np(x), layout="col", rht_seed=workloads.RHT_SEED))
    dyn = to_f32_np(dy)
    ldy = oracle.logical_tensor(dyn, "col", workloads.RHT_SEED)
    for r0 in _sample_rows(20480):
        ad = oracle.dequantize(oracle.quantize(dyn, layout="col", rounding="sr", seed=workloads.SR_SEED,
                                               rht_seed=workloads.RHT_SEED, rows=(r0, r0 + 128), logical=ldy))
        assert_gemm_close(dw[r0:r0 + 128].cpu().numpy(), ad @ bd.T, ad, bd, bf16=False, what=f"Wgrad rows {r0}")
    # the transform cancels: dW approximates dY^T X itself
    ref_rows = dyn[:, :128].T.astype(np.float64) @ to_f32_np(x).astype(np.float64)
    got = dw[:128].cpu().numpy()
    rel = np.linalg.norm(got - ref_rows) / np.linalg.norm(ref_rows)
    assert rel < 0.2


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_full_size_repeatable(nv, out_dtype):
    # The accumulation order of every output element is fixed (K steps in
    # order, one chain per element), so repeated launches on the same operands
    # must agree bit for bit over the whole output, not only on the rows the
    # oracle checks: a launch that read an accumulator or a scale slot at the
    # wrong time shows up here as a difference.
    x = workloads.activations(device="cuda")
    w = workloads.weights(device="cuda")
    qx, _ = nv.nvfp4_quantize(x)
    qw, _ = nv.nvfp4_quantize(w, block="16x16")
    first = nv.nvfp4_gemm(qx, qw, out_dtype=out_dtype)
    for rep in range(6):
        again = nv.nvfp4_gemm(qx, qw, out_dtype=out_dtype)
        torch.cuda.synchronize()
        assert nv.nvfp4_sync_status() == nv.OK
        diff = (again != first).nonzero()
        assert diff.numel() == 0, f"launch {rep + 1} differs from the first at {diff.shape[0]} elements, first {diff[0].tolist()}"

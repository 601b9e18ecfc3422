"""The BF16 fallback GEMM (kind::f16 on the tcgen05 tensor cores, FP32
accumulation) against the oracle's float64 product of the same bf16 inputs,
with the GEMM tolerance of the NVFP4 GEMMs."""
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


@pytest.mark.parametrize("mnk", [(128, 256, 64), (200, 136, 200), (64, 1000, 8), (1000, 48, 128),
                                 (384, 512, 1024), (256, 256, 4096), (128, 320, 64), (96, 712, 40)])
def test_bf16_gemm(nv, mnk):
    m, n, k = mnk
    a = workloads.normal_with_outliers(m, k, p=0.005, factor=20.0, seed=m + 7 * k, dtype=torch.bfloat16)
    b = workloads.normal_with_outliers(n, k, std=0.05, seed=n + 11 * k, dtype=torch.bfloat16)
    c32 = nv.nvfp4_gemm_bf16(a.cuda(), b.cuda(), out_dtype=torch.float32)
    c16 = nv.nvfp4_gemm_bf16(a.cuda(), b.cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    an, bn = a.float().numpy(), b.float().numpy()
    ref = oracle.bf16_gemm(an, bn)
    assert_gemm_close(c32.cpu().numpy(), ref, an.astype(np.float64), bn.astype(np.float64), bf16=False,
                      what=f"bf16 {mnk} fp32")
    assert_gemm_close(c16.float().cpu().numpy(), ref, an.astype(np.float64), bn.astype(np.float64), bf16=True,
                      what=f"bf16 {mnk} bf16")


def test_bf16_gemm_full_size_rows(nv):
    m, n, k = 8192, 20480, 5120
    x = workloads.activations(m, k, device="cuda")
    w = workloads.weights(n, k, device="cuda")
    y = nv.nvfp4_gemm_bf16(x, w, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = [0, 4097, 8191]
    xs = x[rows].float().cpu().numpy()
    wn = w.float().cpu().numpy()
    ref = oracle.bf16_gemm(xs, wn)
    assert_gemm_close(y[rows].cpu().numpy(), ref, xs.astype(np.float64), wn.astype(np.float64), bf16=False,
                      what="bf16 full-size rows")

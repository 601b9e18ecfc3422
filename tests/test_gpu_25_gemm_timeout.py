"""Failure detection in the GEMM without a GPU fault.

Every wait inside the GEMM kernel is bounded.  Here the bound is set far
below the time one tile's MMAs take (K = 8192: 32 pipeline stages per
tile), so the epilogue's wait for the accumulator runs out: the kernel must
record NVFP4_ERR_TIMEOUT, let its MMAs and copies in flight finish, free
its tensor memory and return.  nvfp4_sync_status then reports the timeout,
and the context stays usable: the next GEMM, with the default bound, gives
bit for bit the result of the GEMM run before the abort, which meets the
oracle's tolerance.
"""
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


def test_short_wait_bound_aborts_cleanly(nv):
    m, n, k = 512, 512, 8192
    a = workloads.normal_with_outliers(m, k, p=0.001, factor=30.0, seed=71, dtype=torch.bfloat16).cuda()
    b = workloads.normal_with_outliers(n, k, std=0.05, seed=72, dtype=torch.bfloat16).cuda()
    qa, _ = nv.nvfp4_quantize(a)
    qb, _ = nv.nvfp4_quantize(b)
    before = nv.nvfp4_gemm(qa, qb, out_dtype=torch.float32)
    assert nv.nvfp4_sync_status() == nv.OK

    prev = nv.nvfp4_set_wait_limit_ns(2000)
    try:
        nv.nvfp4_gemm(qa, qb, out_dtype=torch.float32)
        status = nv.nvfp4_sync_status()
    finally:
        nv.nvfp4_set_wait_limit_ns(prev)
    assert status == nv.ERR_TIMEOUT
    assert nv.nvfp4_sync_status() == nv.OK          # the status word was cleared

    after = nv.nvfp4_gemm(qa, qb, out_dtype=torch.float32)
    assert nv.nvfp4_sync_status() == nv.OK
    assert torch.equal(after, before)
    ad = oracle.dequantize(oracle.quantize(to_f32_np(a)))
    bd = oracle.dequantize(oracle.quantize(to_f32_np(b)))
    assert_gemm_close(after.cpu().numpy(), ad @ bd.T, ad, bd, bf16=False, what="GEMM after an aborted launch")

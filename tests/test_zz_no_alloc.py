"""nvfp4_quantize_noalloc: quantization for callers that cannot allocate
device memory (e.g. a plugin whose host framework owns all device memory, or
a loop that must not call cudaMalloc after set-up).  It keeps its amax
scratch in a fixed array inside the library instead of a caller workspace.

Two calls in a row, through the C ABI, must give exactly what nvfp4_quantize
gives for the same inputs (quantization is compared bit for bit, as in the
other quantize tests).  The first call is large and the second small, so a
stale partial left in the shared array by the first call would show up as a
wrong amax in the second.  This file is collected last; it builds the
library itself, so it also passes when run alone in a fresh process.
"""
import pytest
import torch

import workloads
from nvfp4_testing import amax_np, codes_np, scales_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    assert torch.cuda.is_available()
    return nv


def _same(a, b):
    assert amax_np(a).tobytes() == amax_np(b).tobytes()
    assert (codes_np(a) == codes_np(b)).all()
    assert (scales_np(a) == scales_np(b)).all()


def test_noalloc_matches_workspace_path_on_two_calls(nv):
    big = workloads.normal_with_outliers(4096, 4096, p=0.001, factor=50.0, seed=21, device="cuda")
    small = workloads.normal_with_outliers(64, 128, std=1e-3, seed=22, device="cuda", dtype=torch.float32)

    # call 1: large bf16 tensor, SR, both layouts (hundreds of amax CTAs)
    n1r, n1c = nv.nvfp4_quantize_noalloc(big, round="sr", seed=7, rowwise=True, colwise=True)
    # call 2: small fp32 tensor with a far smaller amax, RTN (one amax CTA)
    n2r, n2c = nv.nvfp4_quantize_noalloc(small, rowwise=True, colwise=True, scale_layout="linear")
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK

    r1r, r1c = nv.nvfp4_quantize(big, round="sr", seed=7, rowwise=True, colwise=True)
    r2r, r2c = nv.nvfp4_quantize(small, rowwise=True, colwise=True, scale_layout="linear")
    torch.cuda.synchronize()
    for got, ref in ((n1r, r1r), (n1c, r1c), (n2r, r2r), (n2c, r2c)):
        _same(got, ref)
    assert float(amax_np(n2r)[0]) == float(small.abs().max())


def test_noalloc_rejects_bad_arguments_like_the_workspace_path(nv):
    x = torch.zeros(16, 24, dtype=torch.bfloat16, device="cuda")  # cols not a multiple of 16
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_quantize_noalloc(x)
    assert e.value.status == nv.ERR_INVALID_ARG

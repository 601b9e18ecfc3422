"""The comparison the pages make between the formats: on the same tensors,
NVFP4 (16-element blocks, E4M3 scales, FP32 tensor scale) quantizes with a
smaller error than MXFP4 (32-element blocks, power-of-two scales).  Both
quantizations run on the GPU; the oracle dequantizes their codes and
scales."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import amax_np, codes_np, scales_np, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    return nv


def _rel_err(nv, x, block, rows):
    q, _ = nv.nvfp4_quantize(x, block=block, scale_layout="linear")
    torch.cuda.synchronize()
    codes = codes_np(q)[:rows]
    scales = scales_np(q)[:rows]
    if block == "mx1x32":
        d = dict(codes=codes, scales=np.ascontiguousarray(scales[:, ::2]), fmt="mx", block_h=1, s_dec=1.0)
    else:
        d = dict(codes=codes, scales=scales, block_h=1, s_dec=float(amax_np(q)[1]))
    xd = oracle.dequantize(d)
    xr = to_f32_np(x[:rows]).astype(np.float64)
    return np.linalg.norm(xd - xr) / np.linalg.norm(xr)


@pytest.mark.parametrize("which", ["activations", "gradients"])
def test_nvfp4_error_below_mxfp4(nv, which):
    x = getattr(workloads, which)(1024, 4096, device="cuda")
    e_nv = _rel_err(nv, x, "1x16", 256)
    e_mx = _rel_err(nv, x, "mx1x32", 256)
    assert e_nv < e_mx, (which, e_nv, e_mx)

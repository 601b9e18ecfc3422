"""Quantize calls issued on two streams with no ordering between them.

Each quantize call writes its amax partials into a workspace in its first
kernel and reads them back in its second, so two calls that overlap on the
GPU must not share one workspace.  The binding keeps one workspace per
(device, stream); here the two streams' calls interleave over several rounds
and every result must still equal the oracle bit for bit.
"""
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import assert_quant_equal, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    return nv


def test_two_unordered_streams_keep_their_own_workspace(nv):
    # different amaxes (about 250 and 3e-3), so a partial read from the other
    # stream's call would change the tensor scale
    a = workloads.normal_with_outliers(2048, 4096, p=0.001, factor=50.0, seed=61, device="cuda")
    b = workloads.normal_with_outliers(1024, 2048, std=1e-3, seed=62, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    outs = []
    for rep in range(4):
        with torch.cuda.stream(s1):
            qa, qat = nv.nvfp4_quantize(a, round="sr", seed=3, colwise=True, stream=s1)
        with torch.cuda.stream(s2):
            qb = nv.nvfp4_rht_quantize(b, round="rtn", rht_seed=9, stream=s2)
            qbr, _ = nv.nvfp4_quantize(b, stream=s2)
        outs.append((qa, qat, qb, qbr))
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    an, bn = to_f32_np(a), to_f32_np(b)
    ora = oracle.quantize(an, rounding="sr", seed=3)
    orat = oracle.quantize(an, layout="col", rounding="sr", seed=3)
    orb = oracle.quantize(bn, layout="col", rht_seed=9)
    orbr = oracle.quantize(bn)
    for rep, (qa, qat, qb, qbr) in enumerate(outs):
        assert_quant_equal(qa, ora, what=f"stream 1 rowwise, round {rep}")
        assert_quant_equal(qat, orat, what=f"stream 1 colwise, round {rep}")
        assert_quant_equal(qb, orb, what=f"stream 2 RHT colwise, round {rep}")
        assert_quant_equal(qbr, orbr, what=f"stream 2 rowwise, round {rep}")

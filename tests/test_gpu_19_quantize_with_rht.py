"""GPU parity of nvfp4_quantize_with_rht: the rowwise 1x16 quantization of
an operand and the colwise quantization of its 16-point RHT (along the rows)
from one amax read.  Small cases are compared with the oracle element by
element; the full-size gradient (dY 8192x20480, SR) must equal the two
separate calls (nvfp4_quantize, nvfp4_rht_quantize) bit for bit, codes,
scales and tensor scales alike."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import assert_quant_equal, codes_np, scales_np, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    assert torch.cuda.is_available()
    return nv


@pytest.mark.parametrize("shape", [(16, 16), (64, 48), (208, 336), (400, 272)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
@pytest.mark.parametrize("layout", ["mma", "linear"])
def test_both_outputs_match_the_oracle(nv, shape, dtype, rounding, layout):
    x = workloads.normal_with_outliers(*shape, p=0.01, factor=30.0, seed=101 + shape[1], dtype=dtype)
    xn = to_f32_np(x)
    qr, qc = nv.nvfp4_quantize_with_rht(x.cuda(), round=rounding, seed=55, rht_seed=workloads.RHT_SEED,
                                        scale_layout=layout)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    assert_quant_equal(qr, oracle.quantize(xn, rounding=rounding, seed=55), what="rowwise")
    assert_quant_equal(qc, oracle.quantize(xn, layout="col", rounding=rounding, seed=55, rht_seed=workloads.RHT_SEED),
                       what="rht colwise")


def _same(a, b, what):
    assert torch.equal(a.codes, b.codes), f"{what}: codes differ"
    assert torch.equal(a.scales, b.scales), f"{what}: scales differ"
    # {A, S_dec, S_enc}; the buffer's fourth float is alignment padding
    assert torch.equal(a.amax[:3], b.amax[:3]), f"{what}: tensor scales differ"


def test_full_size_gradient_equals_the_separate_calls(nv):
    dy = workloads.gradients(device="cuda")                # 8192 x 20480, Student-t(3) * 1e-3
    qr, qc = nv.nvfp4_quantize_with_rht(dy, round="sr", seed=workloads.SR_SEED, rht_seed=workloads.RHT_SEED)
    sr_, _ = nv.nvfp4_quantize(dy, round="sr", seed=workloads.SR_SEED)
    sc_ = nv.nvfp4_rht_quantize(dy, round="sr", seed=workloads.SR_SEED, rht_seed=workloads.RHT_SEED)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    _same(qr, sr_, "dY rowwise SR")
    _same(qc, sc_, "dY^T RHT SR")
    # and against the oracle on sampled rows of each output
    dyn = to_f32_np(dy)
    assert_quant_equal(qr, oracle.quantize(dyn, rounding="sr", seed=workloads.SR_SEED, rows=(4096, 4224)),
                       rows=(4096, 4224), what="dY rowwise SR sample")
    ldy = oracle.logical_tensor(dyn, "col", workloads.RHT_SEED)
    assert_quant_equal(qc, oracle.quantize(dyn, layout="col", rounding="sr", seed=workloads.SR_SEED,
                                           rht_seed=workloads.RHT_SEED, rows=(20352, 20480), logical=ldy),
                       rows=(20352, 20480), what="dY^T RHT SR sample")


def test_activation_rtn_equals_the_separate_calls(nv):
    x = workloads.activations(device="cuda")               # 8192 x 5120, 0.1% outliers x50
    qr, qc = nv.nvfp4_quantize_with_rht(x, rht_seed=workloads.RHT_SEED)
    sr_, _ = nv.nvfp4_quantize(x)
    sc_ = nv.nvfp4_rht_quantize(x, rht_seed=workloads.RHT_SEED)
    torch.cuda.synchronize()
    _same(qr, sr_, "X rowwise RTN")
    _same(qc, sc_, "X^T RHT RTN")


@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_nonfinite_input_is_reported(nv, bad):
    x = torch.randn(32, 64, dtype=torch.bfloat16)
    x[21, 5] = bad
    assert nv.nvfp4_sync_status() == nv.OK
    qr, qc = nv.nvfp4_quantize_with_rht(x.cuda(), round="sr", seed=3, rht_seed=4)
    assert nv.nvfp4_sync_status() == nv.ERR_NONFINITE
    assert not codes_np(qr).any() and not scales_np(qr).any()
    assert not codes_np(qc).any() and not scales_np(qc).any()
    assert nv.nvfp4_sync_status() == nv.OK


def test_mxfp4_outputs_are_refused(nv):
    x = torch.randn(32, 64, dtype=torch.bfloat16, device="cuda")
    qr = nv.empty_qtensor(32, 64, x.device, "mma", "mxfp4")
    qc = nv.empty_qtensor(64, 32, x.device, "mma", "mxfp4")
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_quantize_with_rht(x, out_rowwise=qr, out_colwise=qc)

"""GPU parity of the quantize kernels against the oracle, through the C ABI.

Codes, scales and the tensor scales must match bit for bit.  Small cases
compare every element; the full-size workloads (X 8192x5120 with outliers,
W 20480x5120, dY 8192x20480 Student-t) compare sampled rows, which the
oracle quantizes one by one with the amax of the whole tensor.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import assert_quant_equal, codes_np, scales_np, amax_np, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    assert torch.cuda.is_available()
    return nv


E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _probe_values():
    pts = np.array(E2M1, dtype=np.float32)
    mids = ((pts[1:].astype(np.float64) + pts[:-1]) / 2).astype(np.float32)
    base = np.concatenate([pts, mids, np.array([1e-30, 1e-45, 0.1, 0.2, 5.9999], dtype=np.float32)])
    v = np.concatenate([base, np.nextafter(base, np.float32(np.inf)), np.nextafter(base, np.float32(0))])
    v = v[(v >= 0) & (v <= 6)]
    v = np.concatenate([v, -v, np.array([-0.0], dtype=np.float32)])
    return v


def _crafted_rows(values: np.ndarray) -> np.ndarray:
    """Blocks [6, 15 probe values]; a final block holds 2688 so S_enc = 1 and
    every probe block has sb = 1, r = 1 (v = x exactly)."""
    nblk = (len(values) + 14) // 15
    v = np.zeros(nblk * 15, dtype=np.float32)
    v[: len(values)] = values
    blocks = np.concatenate([np.full((nblk, 1), 6.0, np.float32), v.reshape(nblk, 15)], axis=1)
    row = np.concatenate([blocks.reshape(-1), np.zeros(16, np.float32)])
    row[-1] = 2688.0
    pad = (-len(row)) % 64
    return np.concatenate([row, np.zeros(pad, np.float32)]).reshape(1, -1)


@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_element_encoding_on_every_neighbour_pair(nv, rounding):
    x = _crafted_rows(_probe_values())
    xt = torch.from_numpy(x).cuda()
    q, _ = nv.nvfp4_quantize(xt, round=rounding, seed=5, scale_layout="linear")
    torch.cuda.synchronize()
    assert_quant_equal(q, oracle.quantize(x, rounding=rounding, seed=5), what=f"crafted {rounding}")


def test_block_scale_rounding_sweep(nv):
    # block maxima 6*s for s on every E4M3 value, midpoint and the floats next
    # to each midpoint: sweeps the E4M3 rounding of the block scale
    e4 = np.array([oracle.e4m3_decode(c) for c in range(1, 0x7F)], dtype=np.float64)
    mids = (e4[1:] + e4[:-1]) / 2
    s = np.concatenate([e4, mids]).astype(np.float32)
    s = np.concatenate([s, np.nextafter(s, np.float32(0)), np.nextafter(s, np.float32(np.inf)),
                        np.array([2.0 ** -10, 2.0 ** -11, 3e-4, 450.0], np.float32)])
    s = s[s <= 448]
    n = len(s)
    x = np.zeros((n + 1, 16), dtype=np.float32)
    rng = np.random.default_rng(0)
    x[:n, 0] = 6.0 * s
    x[:n, 1:] = (rng.uniform(-1, 1, (n, 15)) * 6.0 * s[:, None]).astype(np.float32)
    x[n, 0] = 2688.0
    x = x.reshape(1, -1)
    x = np.concatenate([x, np.zeros((1, (-x.shape[1]) % 64), np.float32)], axis=1)
    q, _ = nv.nvfp4_quantize(torch.from_numpy(x).cuda(), scale_layout="linear")
    torch.cuda.synchronize()
    assert_quant_equal(q, oracle.quantize(x), what="scale sweep")


SHAPES = [(16, 16), (48, 80), (384, 320), (272, 528), (144, 1040)]


def _input(shape, dtype, seed):
    return workloads.normal_with_outliers(*shape, p=0.01, factor=30.0, seed=seed, dtype=dtype)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
@pytest.mark.parametrize("layout", ["mma", "linear"])
def test_rowwise_and_colwise_1x16(nv, shape, dtype, rounding, layout):
    x = _input(shape, dtype, seed=shape[0] * 7 + shape[1])
    xn = to_f32_np(x)
    qr, qc = nv.nvfp4_quantize(x.cuda(), round=rounding, seed=123, rowwise=True, colwise=True, scale_layout=layout)
    torch.cuda.synchronize()
    assert_quant_equal(qr, oracle.quantize(xn, rounding=rounding, seed=123), what="rowwise")
    assert_quant_equal(qc, oracle.quantize(xn, layout="col", rounding=rounding, seed=123), what="colwise")


@pytest.mark.parametrize("shape", [(16, 16), (64, 128), (208, 336), (400, 272)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("layout", ["mma", "linear"])
def test_2d_16x16_both_layouts(nv, shape, dtype, layout):
    w = workloads.normal_with_outliers(*shape, std=0.02, seed=9 + shape[0], dtype=dtype)
    wn = to_f32_np(w)
    qr, qc = nv.nvfp4_quantize(w.cuda(), block="16x16", rowwise=True, colwise=True, scale_layout=layout)
    torch.cuda.synchronize()
    assert_quant_equal(qr, oracle.quantize(wn, block="16x16"), what="2d rowwise")
    assert_quant_equal(qc, oracle.quantize(wn, layout="col", block="16x16"), what="2d colwise")
    # the two layouts hold the same codes, transposed
    cr, cc = codes_np(qr), codes_np(qc)
    ur = np.stack([cr & 15, cr >> 4], -1).reshape(cr.shape[0], -1)
    uc = np.stack([cc & 15, cc >> 4], -1).reshape(cc.shape[0], -1)
    np.testing.assert_array_equal(ur, uc.T)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("side", ["rowwise", "colwise"])
def test_2d_16x16_one_side_of_a_strided_view(nv, dtype, side):
    # columns 0..335 of a [208][400] tensor: row stride 400 > cols, a last
    # 32-row unit with one 16-row tile, a partial 128-column group
    big = workloads.normal_with_outliers(208, 400, std=0.02, seed=77, dtype=dtype)
    wn = to_f32_np(big[:, :336].contiguous())
    view = big.cuda()[:, :336]
    assert view.stride(0) == 400
    qr, qc = nv.nvfp4_quantize(view, block="16x16", rowwise=side == "rowwise", colwise=side == "colwise")
    torch.cuda.synchronize()
    if side == "rowwise":
        assert qc is None
        assert_quant_equal(qr, oracle.quantize(wn, block="16x16"), what="2d rowwise only")
    else:
        assert qr is None
        assert_quant_equal(qc, oracle.quantize(wn, layout="col", block="16x16"), what="2d colwise only")


@pytest.mark.parametrize("shape", [(16, 16), (64, 48), (256, 320), (400, 272)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_rht_colwise(nv, shape, dtype, rounding):
    x = _input(shape, dtype, seed=31 + shape[1])
    xn = to_f32_np(x)
    q = nv.nvfp4_rht_quantize(x.cuda(), round=rounding, seed=77, rht_seed=workloads.RHT_SEED)
    torch.cuda.synchronize()
    assert_quant_equal(q, oracle.quantize(xn, layout="col", rounding=rounding, seed=77, rht_seed=workloads.RHT_SEED),
                       what="rht colwise")


@pytest.mark.parametrize("rounding", ["rtn", "sr"])
@pytest.mark.parametrize("rht", [False, True])
def test_colwise_several_tiles_per_cta(nv, rounding, rht):
    # 4240 x 4176: 34 x 66 = 2244 tiles of 128 x 64, more than the grid (at
    # most 12 CTAs per SM), so CTAs walk several tiles and the bf16 kernel's
    # double buffer (the next tile copied while one is encoded) turns over;
    # the last tile row and column are partial.  Checked whole against the
    # oracle.
    x = workloads.normal_with_outliers(4240, 4176, p=0.001, factor=20.0, seed=4241, dtype=torch.bfloat16)
    xn = to_f32_np(x)
    if rht:
        q = nv.nvfp4_rht_quantize(x.cuda(), round=rounding, seed=91, rht_seed=workloads.RHT_SEED)
        ref = oracle.quantize(xn, layout="col", rounding=rounding, seed=91, rht_seed=workloads.RHT_SEED)
    else:
        _, q = nv.nvfp4_quantize(x.cuda(), round=rounding, seed=91, rowwise=False, colwise=True)
        ref = oracle.quantize(xn, layout="col", rounding=rounding, seed=91)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    assert_quant_equal(q, ref, what="colwise, several tiles per CTA")


# ---- edge cases ----------------------------------------------------------------

def test_all_zero_tensor(nv):
    x = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
    qr, qc = nv.nvfp4_quantize(x, round="sr", seed=1, rowwise=True, colwise=True)
    torch.cuda.synchronize()
    assert amax_np(qr).tolist() == [0.0, 1.0, 1.0]
    assert not codes_np(qr).any() and not scales_np(qr).any()
    assert not codes_np(qc).any() and not scales_np(qc).any()
    assert nv.nvfp4_sync_status() == nv.OK


def test_negative_zero_and_small_negatives(nv):
    x = torch.zeros(16, 64, dtype=torch.float32)
    x[:, 0] = 6.0
    x[:, 1] = -0.0
    x[:, 2] = -0.1
    x[:, 3] = -1e-30
    q, _ = nv.nvfp4_quantize(x.cuda())
    torch.cuda.synchronize()
    assert_quant_equal(q, oracle.quantize(x.numpy()), what="negative zeros")


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), float("-inf")])
def test_nonfinite_input_is_reported(nv, bad):
    x = torch.randn(32, 64, dtype=torch.bfloat16)
    x[7, 9] = bad
    xd = x.cuda()
    assert nv.nvfp4_sync_status() == nv.OK
    qr, qc = nv.nvfp4_quantize(xd, rowwise=True, colwise=True)
    assert nv.nvfp4_sync_status() == nv.ERR_NONFINITE
    assert not codes_np(qr).any() and not scales_np(qr).any() and not codes_np(qc).any()
    # the status word was cleared by the read
    assert nv.nvfp4_sync_status() == nv.OK
    with pytest.raises(oracle.OracleError):
        oracle.quantize(to_f32_np(x))


def test_tiny_values_saturated_tensor_scale(nv):
    # bf16 subnormals: 2688/A overflows FP32 and S_enc saturates
    x = torch.zeros(16, 64, dtype=torch.float32)
    x[0, :16] = torch.arange(1, 17, dtype=torch.float32) * 1e-40
    x[3, 16:32] = -3e-40
    x[5, 40] = 5e-39
    xb = x.to(torch.bfloat16)
    for t in (x, xb):
        qr, qc = nv.nvfp4_quantize(t.cuda(), round="sr", seed=3, rowwise=True, colwise=True)
        torch.cuda.synchronize()
        tn = to_f32_np(t)
        assert_quant_equal(qr, oracle.quantize(tn, rounding="sr", seed=3), what="tiny rowwise")
        assert_quant_equal(qc, oracle.quantize(tn, layout="col", rounding="sr", seed=3), what="tiny colwise")


def test_huge_values(nv):
    x = torch.randn(32, 64) * 1e37
    x[4, 4] = 3.0e38
    for t in (x, x.to(torch.bfloat16)):
        q, _ = nv.nvfp4_quantize(t.cuda())
        torch.cuda.synchronize()
        assert_quant_equal(q, oracle.quantize(to_f32_np(t)), what="huge")


def test_strided_rows(nv):
    base = _input((96, 256), torch.bfloat16, seed=4)
    view = base.cuda()[:, 64:224]            # ldx = 256, cols = 160
    qr, qc = nv.nvfp4_quantize(view, rowwise=True, colwise=True, round="sr", seed=8)
    q2 = nv.nvfp4_rht_quantize(view, round="rtn", rht_seed=2)
    torch.cuda.synchronize()
    xn = to_f32_np(base[:, 64:224])
    assert_quant_equal(qr, oracle.quantize(xn, rounding="sr", seed=8), what="strided rowwise")
    assert_quant_equal(qc, oracle.quantize(xn, layout="col", rounding="sr", seed=8), what="strided colwise")
    assert_quant_equal(q2, oracle.quantize(xn, layout="col", rht_seed=2), what="strided rht")


def test_repeated_calls_are_deterministic(nv):
    x = _input((256, 512), torch.bfloat16, seed=12).cuda()
    a, _ = nv.nvfp4_quantize(x, round="sr", seed=99)
    b, _ = nv.nvfp4_quantize(x, round="sr", seed=99)
    c, _ = nv.nvfp4_quantize(x, round="sr", seed=100)
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
    assert not torch.equal(a.codes, c.codes)


# ---- full-size workloads, sampled rows --------------------------------------------

def _row_samples(n, k=3, size=128):
    starts = sorted({0, (n // 2 // size) * size, n - size})[:k]
    return [(s, s + size) for s in starts]


def test_full_size_activation_and_weight_quantization(nv):
    x = workloads.activations(device="cuda")               # 8192 x 5120, 0.1% outliers x50
    w = workloads.weights(device="cuda")                   # 20480 x 5120, N(0, 0.02)
    xr, xc = nv.nvfp4_quantize(x, rowwise=True, colwise=True)
    wr, wc = nv.nvfp4_quantize(w, block="16x16", rowwise=True, colwise=True)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    xn, wn = to_f32_np(x), to_f32_np(w)
    lx = oracle.logical_tensor(xn, "col")
    for rows in _row_samples(8192):
        assert_quant_equal(xr, oracle.quantize(xn, rows=rows), rows=rows, what=f"X rowwise {rows}")
    for rows in _row_samples(5120):
        assert_quant_equal(xc, oracle.quantize(xn, layout="col", rows=rows, logical=lx), rows=rows,
                           what=f"X colwise {rows}")
    for rows in _row_samples(20480):
        assert_quant_equal(wr, oracle.quantize(wn, block="16x16", rows=rows), rows=rows, what=f"W 2D {rows}")
    lw = oracle.logical_tensor(wn, "col")
    for rows in _row_samples(5120):
        assert_quant_equal(wc, oracle.quantize(wn, layout="col", block="16x16", rows=rows, logical=lw), rows=rows,
                           what=f"W^T 2D {rows}")


def test_full_size_gradient_sr_and_rht(nv):
    dy = workloads.gradients(device="cuda")                # 8192 x 20480, Student-t(3) * 1e-3
    x = workloads.activations(outliers=False, device="cuda")
    dyr, _ = nv.nvfp4_quantize(dy, round="sr", seed=workloads.SR_SEED)
    dyt = nv.nvfp4_rht_quantize(dy, round="sr", seed=workloads.SR_SEED, rht_seed=workloads.RHT_SEED)
    xt = nv.nvfp4_rht_quantize(x, round="rtn", rht_seed=workloads.RHT_SEED)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    dyn, xn = to_f32_np(dy), to_f32_np(x)
    for rows in _row_samples(8192):
        assert_quant_equal(dyr, oracle.quantize(dyn, rounding="sr", seed=workloads.SR_SEED, rows=rows), rows=rows,
                           what=f"dY rowwise SR {rows}")
    ldy = oracle.logical_tensor(dyn, "col", workloads.RHT_SEED)
    for rows in _row_samples(20480):
        assert_quant_equal(dyt, oracle.quantize(dyn, layout="col", rounding="sr", seed=workloads.SR_SEED,
                                                rht_seed=workloads.RHT_SEED, rows=rows, logical=ldy),
                           rows=rows, what=f"dY^T RHT SR {rows}")
    lx = oracle.logical_tensor(xn, "col", workloads.RHT_SEED)
    for rows in _row_samples(5120):
        assert_quant_equal(xt, oracle.quantize(xn, layout="col", rht_seed=workloads.RHT_SEED, rows=rows, logical=lx),
                           rows=rows, what=f"X^T RHT RTN {rows}")
    # heavy tails: the block holding the tensor max gets the top scale (448)
    # while the typical block scale sits far below it
    s = scales_np(dyr)
    assert s.max() == 0x7E and np.median(s) < 0x60

"""GPU parity of the MXFP4 variant (32-element blocks, UE8M0 power-of-two
scales, no tensor scale) against the oracle, through the C ABI: codes and
scales bit for bit (the GPU keeps each block's scale in both of its
16-element slots), GEMMs within the stated tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import amax_np, assert_gemm_close, codes_np, scales_np, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    return nv


def assert_mx_equal(q, ora, what=""):
    assert q.fmt == "mxfp4"
    assert amax_np(q).tolist() == [0.0, 1.0, 1.0], what
    exp = np.repeat(ora["scales"], 2, axis=1)
    got = scales_np(q)
    bad = np.argwhere(got != exp)
    assert bad.size == 0, f"{what}: {len(bad)} scale mismatches, first {bad[0].tolist()}"
    bad = np.argwhere(codes_np(q) != ora["codes"])
    assert bad.size == 0, f"{what}: {len(bad)} code mismatches, first {bad[0].tolist()}"


def _mixed(rows, cols, seed, dtype):
    """Blocks over many binades, all-zero blocks, subnormal-sized blocks."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * (2.0 ** torch.randint(-40, 40, (rows, cols // 32), generator=g)
                                                 ).float().repeat_interleave(32, dim=1)
    x[0, :32] = 0.0
    if rows > 1:
        x[1, 32:64] = 1e-41
    return x.to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
@pytest.mark.parametrize("layout", ["mma", "linear"])
def test_mx_rowwise_and_colwise(nv, dtype, rounding, layout):
    x = _mixed(96, 1056, seed=4, dtype=dtype)           # 33 blocks per row: ragged warp items
    qr, qc = nv.nvfp4_quantize(x.cuda(), block="mx1x32", round=rounding, seed=9, rowwise=True, colwise=True,
                               scale_layout=layout)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    xf = to_f32_np(x)
    assert_mx_equal(qr, oracle.quantize(xf, block="mx1x32", rounding=rounding, seed=9), "rowwise")
    assert_mx_equal(qc, oracle.quantize(xf, layout="col", block="mx1x32", rounding=rounding, seed=9), "colwise")


@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_mx_rht_colwise(nv, rounding):
    x = _mixed(320, 192, seed=6, dtype=torch.bfloat16)
    q = nv.nvfp4_rht_quantize(x.cuda(), round=rounding, seed=3, rht_seed=8, fmt="mxfp4")
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    assert_mx_equal(q, oracle.quantize(to_f32_np(x), layout="col", block="mx1x32", rounding=rounding, seed=3,
                                       rht_seed=8), "rht colwise")


def test_mx_full_size_gradient_rows(nv):
    dy = workloads.gradients(device="cuda")                 # 8192 x 20480 bf16 Student-t
    q, _ = nv.nvfp4_quantize(dy, block="mx1x32", round="sr", seed=1)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    cols = dy.shape[1]
    c, s = codes_np(q), scales_np(q)
    for r in [0, 4095, 8191]:
        ref = _row_oracle(to_f32_np(dy[r:r + 1])[0], r, cols)
        assert np.array_equal(s[r:r + 1], np.repeat(ref["scales"], 2, axis=1))
        assert np.array_equal(c[r:r + 1], ref["codes"])


def _row_oracle(row, r, cols):
    # quantize one row of a larger tensor: the stochastic-rounding index is
    # r * cols + c, which the oracle takes through its row offset
    big = np.ascontiguousarray(row.reshape(1, cols), dtype=np.float32)
    q = oracle.lib()
    codes = np.zeros((1, cols // 2), dtype=np.uint8)
    scales = np.zeros((1, cols // 32), dtype=np.uint8)
    import ctypes
    st = q.nvfp4_oracle_mx_quantize(big.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), 1, cols, r, 1, 1,
                                    codes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                                    scales.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    assert st == 0
    return dict(codes=codes, scales=scales)


def test_mx_nonfinite_block_is_flagged_and_zeroed(nv):
    x = torch.randn(4, 128, dtype=torch.float32)
    x[2, 40] = float("nan")
    q, _ = nv.nvfp4_quantize(x.cuda(), block="mx1x32", scale_layout="linear")
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.ERR_NONFINITE
    c, s = codes_np(q), scales_np(q)
    assert not c[2, 16:32].any() and not s[2, 2:4].any()
    x[2, 40] = 0.0
    ora = oracle.quantize(x.numpy(), block="mx1x32")
    keep = np.ones_like(c, dtype=bool)
    keep[2, 16:32] = False
    assert np.array_equal(c[keep], ora["codes"][keep])


@pytest.mark.parametrize("mnk", [(128, 128, 64), (200, 136, 320), (384, 512, 1024), (256, 256, 4096)])
def test_mx_gemm(nv, mnk):
    m, n, k = mnk
    a = workloads.normal_with_outliers(m, k, p=0.005, factor=20.0, seed=m + k, dtype=torch.bfloat16)
    b = workloads.normal_with_outliers(n, k, std=0.05, seed=n + 3 * k, dtype=torch.bfloat16)
    qa, _ = nv.nvfp4_quantize(a.cuda(), block="mx1x32", round="sr", seed=2)
    qb, _ = nv.nvfp4_quantize(b.cuda(), block="mx1x32")
    c32 = nv.nvfp4_gemm(qa, qb, out_dtype=torch.float32)
    c16 = nv.nvfp4_gemm(qa, qb, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    oa = oracle.quantize(to_f32_np(a), block="mx1x32", rounding="sr", seed=2)
    ob = oracle.quantize(to_f32_np(b), block="mx1x32")
    assert_mx_equal(qa, oa, "A")
    ad, bd = oracle.dequantize(oa), oracle.dequantize(ob)
    ref = ad @ bd.T
    assert_gemm_close(c32.cpu().numpy(), ref, ad, bd, bf16=False, what=f"mx {mnk} fp32")
    assert_gemm_close(c16.float().cpu().numpy(), ref, ad, bd, bf16=True, what=f"mx {mnk} bf16")


def test_gemm_rejects_mixed_formats(nv):
    a = torch.randn(128, 128, dtype=torch.bfloat16, device="cuda")
    qa, _ = nv.nvfp4_quantize(a)
    qb, _ = nv.nvfp4_quantize(a, block="mx1x32")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_gemm(qa, qb)
    assert e.value.status == nv.ERR_INVALID_ARG

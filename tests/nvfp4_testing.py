"""Shared helpers of the GPU parity tests: fetch the CUDA path's outputs to
the host and compare them with the oracle's, and the GEMM tolerance.

Parity bar (the quantizer is an encoding, so it must match exactly):
  codes, block scales and {A, S_dec, S_enc}: bit-exact.
GEMM bar (FP32 accumulation order is the hardware's):
  FP32 output: ||C - C_ref||_F / ||C_ref||_F <= 1e-5 and, element-wise,
  |C - C_ref| <= 1e-3 * ||A^_row|| * ||B^_col|| / sqrt(K).
  bf16 output: element-wise |C - C_ref| <= ulp_bf16(C_ref) + the same bound
  (bf16 rounding alone is ~2^-9 relative, so the Frobenius bound is checked on
  the FP32-output run of the same GEMM instead).
C_ref is the FP64 product of the oracle's dequantized operands.
"""
import numpy as np
import torch

import quantize_block_scaled_amax_gb300 as nv

REL_FROB = 1e-5
ELEM = 1e-3


def codes_np(q) -> np.ndarray:
    return nv.codes_view(q).cpu().numpy()


def scales_np(q) -> np.ndarray:
    return nv.scales_as_linear(q).cpu().numpy()


def amax_np(q) -> np.ndarray:
    return q.amax[:3].cpu().numpy()


def expand_2d_scales(s: np.ndarray) -> np.ndarray:
    """Oracle 16x16 scales [rows/16][cols/16] -> one row per element row."""
    return np.repeat(s, 16, axis=0)


def assert_quant_equal(q, ora: dict, rows=None, what=""):
    """Bit-exact comparison of a GPU QTensor (optionally a row range of it)
    with an oracle quantization of the same logical rows."""
    r0, r1 = (0, q.rows) if rows is None else rows
    codes = codes_np(q)[r0:r1]
    scales = scales_np(q)[r0:r1]
    exp_scales = ora["scales"] if ora["block_h"] == 1 else expand_2d_scales(ora["scales"])
    a = amax_np(q)
    assert a[0] == np.float32(ora["amax"]), f"{what}: amax {a[0]!r} vs {ora['amax']!r}"
    assert a[1] == np.float32(ora["s_dec"]), f"{what}: S_dec {a[1]!r} vs {ora['s_dec']!r}"
    assert a[2] == np.float32(ora["s_enc"]), f"{what}: S_enc {a[2]!r} vs {ora['s_enc']!r}"
    bad_s = np.argwhere(scales != exp_scales)
    assert bad_s.size == 0, (f"{what}: {len(bad_s)} scale mismatches, first at {bad_s[0].tolist()}: "
                             f"gpu {scales[tuple(bad_s[0])]:#x} oracle {exp_scales[tuple(bad_s[0])]:#x}")
    bad_c = np.argwhere(codes != ora["codes"])
    assert bad_c.size == 0, (f"{what}: {len(bad_c)} code-byte mismatches, first at {bad_c[0].tolist()}: "
                             f"gpu {codes[tuple(bad_c[0])]:#04x} oracle {ora['codes'][tuple(bad_c[0])]:#04x}")


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 7), 2.0 ** -133)


def assert_gemm_close(c_gpu: np.ndarray, c_ref: np.ndarray, a_deq: np.ndarray, b_deq: np.ndarray, bf16: bool,
                      what=""):
    c = c_gpu.astype(np.float64)
    k = a_deq.shape[1]
    bound = ELEM * np.outer(np.linalg.norm(a_deq, axis=1), np.linalg.norm(b_deq, axis=1)) / np.sqrt(k)
    err = np.abs(c - c_ref)
    if bf16:
        bound = bound + ulp_bf16(c_ref)
    else:
        nref = np.linalg.norm(c_ref)
        rel = np.linalg.norm(c - c_ref) / nref if nref > 0 else np.linalg.norm(c)
        assert rel <= REL_FROB, f"{what}: relative Frobenius error {rel:.3e} > {REL_FROB}"
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} elements out of bound, first {bad[0].tolist()}: "
                           f"gpu {c[tuple(bad[0])]!r} ref {c_ref[tuple(bad[0])]!r} bound {bound[tuple(bad[0])]!r}")


def to_f32_np(x: torch.Tensor) -> np.ndarray:
    """Exact float32 copy of a bf16/fp32 tensor for the oracle."""
    return x.detach().to(torch.float32).cpu().numpy()

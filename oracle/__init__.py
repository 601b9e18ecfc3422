"""NVFP4 oracle: plain CPU restatement of the NVFP4 method, for checking only.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
imports, links or calls it, and it never imports the CUDA library.

What it follows ("Pretraining Large Language Models with NVFP4",
arXiv 2509.25149 summary page; NVIDIA blog paraphrase "NVFP4 Trains with
Precision of 16-Bit and Speed and Efficiency of 4-Bit", technique list):

* format paragraph of the paper page: 16 E2M1 elements share one E4M3 block
  scale, plus one FP32 scale per tensor from a full-tensor amax;
* blog technique list: 1x16 blocks, 2D (16x16) blocks for weights,
  stochastic rounding for gradients, Hadamard transforms on GEMM inputs;
* limitations paragraph of the paper page: Hadamard only on the Wgrad GEMM
  inputs, and the extra full-tensor amax scan;
* the GEMM is the FP64 dot product of the dequantized operands.

The element arithmetic lives in ``nvfp4_oracle.c`` (compiled with gcc,
``-O2 -ffp-contract=off``); this module transposes, transforms and calls it,
and does the GEMM with a float64 ``numpy.matmul`` of the dequantized
operands.  All functions are pinned by CPU tests (``tests/test_oracle_*``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libnvfp4_oracle.so")

ORACLE_OK = 0
ORACLE_ERR_INVALID = 1
ORACLE_ERR_NONFINITE = 4

_lib = None
_lock = threading.Lock()


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build`` and return the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u8p = ctypes.POINTER(ctypes.c_uint8)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            u32p = ctypes.POINTER(ctypes.c_uint32)
            i64 = ctypes.c_int64
            L.nvfp4_oracle_e2m1_decode.restype = ctypes.c_double
            L.nvfp4_oracle_e2m1_decode.argtypes = [ctypes.c_uint32]
            L.nvfp4_oracle_e2m1_encode_rtn.restype = ctypes.c_uint32
            L.nvfp4_oracle_e2m1_encode_rtn.argtypes = [ctypes.c_float]
            L.nvfp4_oracle_e2m1_encode_sr.restype = ctypes.c_uint32
            L.nvfp4_oracle_e2m1_encode_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
            L.nvfp4_oracle_e4m3_decode.restype = ctypes.c_double
            L.nvfp4_oracle_e4m3_decode.argtypes = [ctypes.c_uint32]
            L.nvfp4_oracle_e4m3_encode.restype = ctypes.c_uint32
            L.nvfp4_oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.nvfp4_oracle_philox4x32_10.restype = None
            L.nvfp4_oracle_philox4x32_10.argtypes = [u32p, u32p, u32p]
            L.nvfp4_oracle_sr_bits.restype = ctypes.c_uint32
            L.nvfp4_oracle_sr_bits.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            L.nvfp4_oracle_rht16_signs.restype = None
            L.nvfp4_oracle_rht16_signs.argtypes = [ctypes.c_uint64, f32p]
            L.nvfp4_oracle_rht16.restype = None
            L.nvfp4_oracle_rht16.argtypes = [f32p, f32p, f32p]
            L.nvfp4_oracle_rht_rows.restype = ctypes.c_int
            L.nvfp4_oracle_rht_rows.argtypes = [f32p, i64, i64, ctypes.c_uint64]
            L.nvfp4_oracle_tensor_amax.restype = ctypes.c_int
            L.nvfp4_oracle_tensor_amax.argtypes = [f32p, i64, f32p]
            L.nvfp4_oracle_tensor_scales.restype = None
            L.nvfp4_oracle_tensor_scales.argtypes = [ctypes.c_float, f32p, f32p]
            L.nvfp4_oracle_block_scale.restype = ctypes.c_uint32
            L.nvfp4_oracle_block_scale.argtypes = [ctypes.c_float, ctypes.c_float]
            L.nvfp4_oracle_block_multiplier.restype = ctypes.c_float
            L.nvfp4_oracle_block_multiplier.argtypes = [ctypes.c_float, ctypes.c_uint32]
            L.nvfp4_oracle_quantize.restype = ctypes.c_int
            L.nvfp4_oracle_quantize.argtypes = [f32p, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_uint64, f32p, u8p, u8p, f32p]
            L.nvfp4_oracle_dequantize.restype = ctypes.c_int
            L.nvfp4_oracle_dequantize.argtypes = [u8p, u8p, i64, i64, ctypes.c_int, ctypes.c_float, f64p]
            L.nvfp4_oracle_e2m1_encode_rtn_array.restype = None
            L.nvfp4_oracle_e2m1_encode_rtn_array.argtypes = [f32p, i64, u8p]
            L.nvfp4_oracle_e2m1_encode_sr_array.restype = None
            L.nvfp4_oracle_e2m1_encode_sr_array.argtypes = [f32p, u32p, i64, u8p]
            L.nvfp4_oracle_e4m3_encode_array.restype = None
            L.nvfp4_oracle_e4m3_encode_array.argtypes = [f32p, i64, u8p]
            L.nvfp4_oracle_e8m0_decode.restype = ctypes.c_double
            L.nvfp4_oracle_e8m0_decode.argtypes = [ctypes.c_uint32]
            L.nvfp4_oracle_mx_block_scale.restype = ctypes.c_uint32
            L.nvfp4_oracle_mx_block_scale.argtypes = [ctypes.c_float]
            L.nvfp4_oracle_mx_quantize.restype = ctypes.c_int
            L.nvfp4_oracle_mx_quantize.argtypes = [f32p, i64, i64, i64, ctypes.c_int, ctypes.c_uint64, u8p, u8p]
            L.nvfp4_oracle_mx_dequantize.restype = ctypes.c_int
            L.nvfp4_oracle_mx_dequantize.argtypes = [u8p, u8p, i64, i64, f64p]
            _lib = L
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


# ---- scalar element functions -------------------------------------------

def e2m1_decode(code: int) -> float:
    return lib().nvfp4_oracle_e2m1_decode(int(code))


def e2m1_encode_rtn(v: float) -> int:
    return lib().nvfp4_oracle_e2m1_encode_rtn(float(v))


def e2m1_encode_sr(v: float, rbits: int) -> int:
    return lib().nvfp4_oracle_e2m1_encode_sr(float(v), int(rbits) & 0xFFFFFFFF)


def e4m3_decode(b: int) -> float:
    return lib().nvfp4_oracle_e4m3_decode(int(b))


def e4m3_encode(v: float) -> int:
    return lib().nvfp4_oracle_e4m3_encode(float(v))


def e2m1_encode_rtn_array(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.zeros(v.shape, dtype=np.uint8)
    lib().nvfp4_oracle_e2m1_encode_rtn_array(_ptr(v, ctypes.c_float), v.size, _ptr(out, ctypes.c_uint8))
    return out


def e2m1_encode_sr_array(v, rbits) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    rb = np.ascontiguousarray(rbits, dtype=np.uint32)
    assert rb.shape == v.shape
    out = np.zeros(v.shape, dtype=np.uint8)
    lib().nvfp4_oracle_e2m1_encode_sr_array(_ptr(v, ctypes.c_float), _ptr(rb, ctypes.c_uint32), v.size,
                                            _ptr(out, ctypes.c_uint8))
    return out


def e4m3_encode_array(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.zeros(v.shape, dtype=np.uint8)
    lib().nvfp4_oracle_e4m3_encode_array(_ptr(v, ctypes.c_float), v.size, _ptr(out, ctypes.c_uint8))
    return out


def philox4x32_10(ctr, key) -> list[int]:
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().nvfp4_oracle_philox4x32_10(_ptr(c, ctypes.c_uint32), _ptr(k, ctypes.c_uint32),
                                     _ptr(out, ctypes.c_uint32))
    return [int(v) for v in out]


def sr_bits(seed: int, index: int) -> int:
    return lib().nvfp4_oracle_sr_bits(int(seed), int(index))


def rht16_signs(rht_seed: int) -> np.ndarray:
    d = np.zeros(16, dtype=np.float32)
    lib().nvfp4_oracle_rht16_signs(int(rht_seed), _ptr(d, ctypes.c_float))
    return d


def rht16(x, d) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = np.ascontiguousarray(d, dtype=np.float32)
    y = np.zeros(16, dtype=np.float32)
    lib().nvfp4_oracle_rht16(_ptr(x, ctypes.c_float), _ptr(d, ctypes.c_float), _ptr(y, ctypes.c_float))
    return y


def tensor_scales(amax: float) -> tuple[float, float]:
    sd = ctypes.c_float()
    se = ctypes.c_float()
    lib().nvfp4_oracle_tensor_scales(float(amax), ctypes.byref(sd), ctypes.byref(se))
    return sd.value, se.value


def block_scale(bamax: float, s_enc: float) -> int:
    return lib().nvfp4_oracle_block_scale(float(bamax), float(s_enc))


def block_multiplier(s_enc: float, sb: int) -> float:
    return lib().nvfp4_oracle_block_multiplier(float(s_enc), int(sb))


# ---- whole-tensor steps --------------------------------------------------

def rht_rows(x: np.ndarray, rht_seed: int) -> np.ndarray:
    """Return a copy of x [rows][cols] with the 16-point RHT applied to each
    run of 16 consecutive elements of every row."""
    y = np.array(x, dtype=np.float32, order="C", copy=True)
    st = lib().nvfp4_oracle_rht_rows(_ptr(y, ctypes.c_float), y.shape[0], y.shape[1], int(rht_seed))
    if st:
        raise OracleError(f"rht_rows failed with status {st}")
    return y


def tensor_amax(x: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    a = ctypes.c_float()
    st = lib().nvfp4_oracle_tensor_amax(_ptr(x, ctypes.c_float), x.size, ctypes.byref(a))
    if st:
        raise OracleError(f"tensor_amax: status {st} (non-finite input)")
    return a.value


def logical_tensor(x: np.ndarray, layout: str = "row", rht_seed: int | None = None) -> np.ndarray:
    """The tensor the codes describe: x itself (rowwise) or its transpose
    (colwise), then the optional 16-point RHT along its rows."""
    x = np.asarray(x, dtype=np.float32)
    if layout == "row":
        t = np.ascontiguousarray(x)
    elif layout == "col":
        t = np.ascontiguousarray(x.T)
    else:
        raise ValueError(layout)
    if rht_seed is not None:
        t = rht_rows(t, rht_seed)
    return t


def e8m0_decode(b: int) -> float:
    return lib().nvfp4_oracle_e8m0_decode(int(b))


def mx_block_scale(bamax: float) -> int:
    return lib().nvfp4_oracle_mx_block_scale(float(bamax))


def quantize(x: np.ndarray, *, layout: str = "row", block: str = "1x16", rounding: str = "rtn",
             seed: int = 0, rht_seed: int | None = None, rows: tuple[int, int] | None = None,
             logical: np.ndarray | None = None) -> dict:
    """Quantize x [R][C] (float32 values; bf16 inputs passed exactly as float32).

    layout  'row': codes describe x, blocks along C, codes [R][C/2].
            'col': codes describe x^T, blocks along R, codes [C][R/2].
    block   '1x16' or '16x16' (one scale per 16x16 tile of the logical tensor),
            or 'mx1x32' (MXFP4: 32-element blocks, UE8M0 power-of-two
            scales, no tensor scale; then amax, s_dec, s_enc are 0, 1, 1).
    rounding 'rtn' (nearest, ties to even) or 'sr' (stochastic, Philox).
    rht_seed apply the 16-point RHT along the logical rows first.
    rows    (start, stop): quantize only those logical rows; the tensor amax
            still covers the whole logical tensor.
    logical precomputed ``logical_tensor(x, layout, rht_seed)`` to reuse.

    Returns dict(codes, scales, amax, s_dec, s_enc, row0).  scales are
    [rows][C/16] for 1x16 and [rows/16][C/16] for 16x16.
    """
    t = logical if logical is not None else logical_tensor(x, layout, rht_seed)
    if block == "mx1x32":
        return _mx_quantize(t, rounding, seed, rows)
    block_h = {"1x16": 1, "16x16": 16}[block]
    stochastic = {"rtn": 0, "sr": 1}[rounding]
    nrows_all, cols = t.shape
    amax = np.array([tensor_amax(t)], dtype=np.float32)
    r0, r1 = (0, nrows_all) if rows is None else rows
    sub = np.ascontiguousarray(t[r0:r1])
    n = r1 - r0
    codes = np.zeros((n, cols // 2), dtype=np.uint8)
    scales = np.zeros((n // block_h, cols // 16), dtype=np.uint8)
    amax3 = np.zeros(3, dtype=np.float32)
    st = lib().nvfp4_oracle_quantize(_ptr(sub, ctypes.c_float), n, cols, r0, block_h, stochastic,
                                     int(seed), _ptr(amax, ctypes.c_float), _ptr(codes, ctypes.c_uint8),
                                     _ptr(scales, ctypes.c_uint8), _ptr(amax3, ctypes.c_float))
    if st:
        raise OracleError(f"quantize: status {st}")
    return dict(codes=codes, scales=scales, amax=float(amax3[0]), s_dec=float(amax3[1]),
                s_enc=float(amax3[2]), block_h=block_h, row0=r0)


def _mx_quantize(t: np.ndarray, rounding: str, seed: int, rows) -> dict:
    stochastic = {"rtn": 0, "sr": 1}[rounding]
    nrows_all, cols = t.shape
    r0, r1 = (0, nrows_all) if rows is None else rows
    sub = np.ascontiguousarray(t[r0:r1], dtype=np.float32)
    n = r1 - r0
    codes = np.zeros((n, cols // 2), dtype=np.uint8)
    scales = np.zeros((n, cols // 32), dtype=np.uint8)
    st = lib().nvfp4_oracle_mx_quantize(_ptr(sub, ctypes.c_float), n, cols, r0, stochastic, int(seed),
                                        _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8))
    if st:
        raise OracleError(f"mx quantize: status {st}")
    return dict(codes=codes, scales=scales, amax=0.0, s_dec=1.0, s_enc=1.0, block_h=1, row0=r0, fmt="mx")


def dequantize(q: dict) -> np.ndarray:
    """x^ = e2m1(code) * e4m3(block scale) * S_dec in float64 (exact); for
    MXFP4, x^ = e2m1(code) * 2^(scale - 127)."""
    if q.get("fmt") == "mx":
        codes = np.ascontiguousarray(q["codes"], dtype=np.uint8)
        scales = np.ascontiguousarray(q["scales"], dtype=np.uint8)
        rows, cols = codes.shape[0], codes.shape[1] * 2
        out = np.zeros((rows, cols), dtype=np.float64)
        st = lib().nvfp4_oracle_mx_dequantize(_ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8), rows,
                                              cols, _ptr(out, ctypes.c_double))
        if st:
            raise OracleError(f"mx dequantize: status {st}")
        return out
    codes = np.ascontiguousarray(q["codes"], dtype=np.uint8)
    scales = np.ascontiguousarray(q["scales"], dtype=np.uint8)
    rows, cols = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((rows, cols), dtype=np.float64)
    st = lib().nvfp4_oracle_dequantize(_ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8), rows, cols,
                                       q["block_h"], q["s_dec"], _ptr(out, ctypes.c_double))
    if st:
        raise OracleError(f"dequantize: status {st}")
    return out


def bf16_gemm(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """C[m, n] = sum_k a[m, k] * b[n, k] in float64 for bf16-valued inputs
    (given as float32 arrays holding bf16 values exactly): the high-precision
    GEMM the recipe keeps for a few layers, as one float64 matmul."""
    a = np.asarray(a, dtype=np.float32)
    b = np.asarray(b, dtype=np.float32)
    if a.shape[1] != b.shape[1]:
        raise ValueError("K mismatch")
    bits = np.concatenate([a.view(np.uint32).ravel(), b.view(np.uint32).ravel()])
    if np.any(bits & 0xFFFF):
        raise ValueError("inputs must hold bf16 values")
    return a.astype(np.float64) @ b.astype(np.float64).T


def gemm(qa: dict, qb: dict) -> np.ndarray:
    """C[m, n] = sum_k A^[m, k] * B^[n, k] in float64: the FP64 dot of the
    dequantized operands (both quantized along K)."""
    return dequantize(qa) @ dequantize(qb).T

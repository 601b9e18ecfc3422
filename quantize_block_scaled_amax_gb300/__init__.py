"""GB300 (sm_103a) NVFP4 linear-layer engine: Python binding of the C ABI.

The binding only marshals arguments: every step of quantization and of the
GEMMs runs in the CUDA library ``_build/libnvfp4_gb300.so`` (built by
``build.py``).  PyTorch supplies device memory and the current stream.  The
functions carry the names of the C entry points in ``include/nvfp4.h``.

If the library is missing the import of the binding fails loudly; there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "NVFP4Error", "QTensor", "LinearContext", "lib", "nvfp4_quantize", "nvfp4_rht_quantize", "nvfp4_gemm",
    "nvfp4_gemm_pair",
    "nvfp4_quantize_noalloc", "nvfp4_quantize_with_rht", "nvfp4_rht_quantize_rowwise", "nvfp4_gemm_bf16",
    "nvfp4_transpose_bf16",
    "nvfp4_linear_fwd", "nvfp4_linear_bwd", "nvfp4_sync_status", "nvfp4_set_wait_limit_ns", "nvfp4_scales_bytes", "nvfp4_workspace_size",
    "nvfp4_linear_workspace_size",
    "nvfp4_checked_build", "nvfp4_checked_selftest",
    "empty_qtensor", "scales_as_linear",
]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_NONFINITE, ERR_TIMEOUT, ERR_CUDA, ERR_BOUNDS = range(8)
IN_BF16, IN_FP32 = 0, 1
OUT_BF16, OUT_FP32, OUT_FP32_ADD = 0, 1, 2
BLOCK_1x16, BLOCK_16x16, BLOCK_MX1x32 = 0, 1, 2
FORMAT_NVFP4, FORMAT_MXFP4 = 0, 1
RTN, SR = 0, 1
SCALES_LINEAR, SCALES_MMA = 0, 1

_BLOCKS = {"1x16": BLOCK_1x16, "16x16": BLOCK_16x16, "mx1x32": BLOCK_MX1x32}
_FORMATS = {"nvfp4": FORMAT_NVFP4, "mxfp4": FORMAT_MXFP4}
_ROUNDS = {"rtn": RTN, "sr": SR}
_LAYOUTS = {"linear": SCALES_LINEAR, "mma": SCALES_MMA}


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({detail})")


class nvfp4_tensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("amax", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("ld_codes", ctypes.c_int64),
                ("scale_layout", ctypes.c_int32), ("format", ctypes.c_int32)]


class nvfp4_linear_ctx(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("xq", nvfp4_tensor), ("wq", nvfp4_tensor), ("wtq", nvfp4_tensor), ("dyq", nvfp4_tensor),
                ("dytq", nvfp4_tensor), ("xtq", nvfp4_tensor),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("dw_accumulate", ctypes.c_int32)]


_lib = None
_lib_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise ImportError(f"NVFP4 CUDA library not built: {_build.LIB} is missing "
                                  "(run quantize_block_scaled_amax_gb300.build.build())")
            L = ctypes.CDLL(_build.LIB)
            st = ctypes.c_int
            vp = ctypes.c_void_p
            i64 = ctypes.c_int64
            u64 = ctypes.c_uint64
            tp = ctypes.POINTER(nvfp4_tensor)
            L.nvfp4_checked_build.restype = ctypes.c_int32
            L.nvfp4_checked_build.argtypes = []
            L.nvfp4_checked_selftest.restype = st
            L.nvfp4_checked_selftest.argtypes = [vp]
            L.nvfp4_scales_bytes.restype = ctypes.c_size_t
            L.nvfp4_scales_bytes.argtypes = [i64, i64, ctypes.c_int32]
            L.nvfp4_workspace_size.restype = ctypes.c_size_t
            L.nvfp4_workspace_size.argtypes = []
            L.nvfp4_linear_workspace_size.restype = ctypes.c_size_t
            L.nvfp4_linear_workspace_size.argtypes = []
            L.nvfp4_quantize.restype = st
            L.nvfp4_quantize.argtypes = [vp, st, i64, i64, i64, st, st, u64, tp, tp, vp, ctypes.c_size_t, vp]
            L.nvfp4_quantize_noalloc.restype = st
            L.nvfp4_quantize_noalloc.argtypes = [vp, st, i64, i64, i64, st, st, u64, tp, tp, vp]
            L.nvfp4_rht_quantize.restype = st
            L.nvfp4_rht_quantize.argtypes = [vp, st, i64, i64, i64, st, u64, u64, tp, vp, ctypes.c_size_t, vp]
            L.nvfp4_rht_quantize_rowwise.restype = st
            L.nvfp4_transpose_bf16.restype = st
            L.nvfp4_transpose_bf16.argtypes = [vp, i64, i64, i64, vp, i64, vp]
            L.nvfp4_quantize_with_rht.restype = st
            L.nvfp4_quantize_with_rht.argtypes = [vp, st, i64, i64, i64, st, u64, u64, tp, tp, vp, ctypes.c_size_t,
                                                  vp]
            L.nvfp4_rht_quantize_rowwise.argtypes = [vp, st, i64, i64, i64, st, u64, u64, tp, vp, ctypes.c_size_t,
                                                     vp]
            L.nvfp4_gemm.restype = st
            L.nvfp4_gemm.argtypes = [tp, tp, vp, st, i64, vp, ctypes.c_size_t, vp]
            L.nvfp4_gemm_pair.restype = st
            L.nvfp4_gemm_pair.argtypes = [tp, tp, vp, st, i64, tp, tp, vp, st, i64, vp]
            L.nvfp4_gemm_bf16.restype = st
            L.nvfp4_gemm_bf16.argtypes = [vp, i64, vp, i64, vp, st, i64, i64, i64, i64, vp]
            L.nvfp4_linear_fwd.restype = st
            L.nvfp4_linear_fwd.argtypes = [vp, vp, vp, ctypes.POINTER(nvfp4_linear_ctx), vp]
            L.nvfp4_linear_fwd_rht.restype = st
            L.nvfp4_linear_fwd_rht.argtypes = [vp, vp, vp, u64, ctypes.POINTER(nvfp4_linear_ctx), vp]
            L.nvfp4_linear_bwd.restype = st
            L.nvfp4_linear_bwd.argtypes = [vp, vp, vp, vp, u64, u64, ctypes.POINTER(nvfp4_linear_ctx), vp]
            L.nvfp4_set_wait_limit_ns.restype = ctypes.c_uint64
            L.nvfp4_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.nvfp4_sync_status.restype = st
            L.nvfp4_sync_status.argtypes = [vp]
            L.nvfp4_status_string.restype = ctypes.c_char_p
            L.nvfp4_status_string.argtypes = [st]
            L.nvfp4_last_error.restype = ctypes.c_char_p
            L.nvfp4_last_error.argtypes = []
            _lib = L
    return _lib


def _check(status: int, where: str):
    if status != OK:
        L = lib()
        detail = (L.nvfp4_last_error() or b"").decode() or L.nvfp4_status_string(status).decode()
        raise NVFP4Error(status, where, detail)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def nvfp4_scales_bytes(rows: int, cols: int, scale_layout: str = "mma") -> int:
    return int(lib().nvfp4_scales_bytes(rows, cols, _LAYOUTS[scale_layout]))


def nvfp4_workspace_size() -> int:
    return int(lib().nvfp4_workspace_size())


def nvfp4_linear_workspace_size() -> int:
    return int(lib().nvfp4_linear_workspace_size())


_ws: dict = {}
_ws_lock = threading.Lock()


def _workspace(device, stream_handle: int) -> torch.Tensor:
    """The amax-partials workspace of the quantize wrappers, one per
    (device, stream).  A quantize call writes its workspace in its first
    kernel and reads it back in the next, so two calls whose work can overlap
    on the GPU must not share one: calls on one stream run in order, calls on
    different streams get different buffers.  Each buffer lives as long as
    the process (16 KB per stream used)."""
    key = (device.index if device.index is not None else torch.cuda.current_device(), int(stream_handle))
    with _ws_lock:
        w = _ws.get(key)
        if w is None:
            w = torch.empty(nvfp4_workspace_size(), dtype=torch.uint8, device=device)
            _ws[key] = w
        return w


class QTensor:
    """A quantized tensor held in torch device buffers.

    codes  uint8 [rows][ld_codes] (two E2M1 codes per byte, low nibble first)
    scales uint8 flat buffer of block scales in ``scale_layout``: E4M3 per 16
           elements (fmt "nvfp4"), or UE8M0 per 32 elements stored in both of
           the block's 16-element slots (fmt "mxfp4")
    amax   float32 [3] = (A, S_dec, S_enc); (0, 1, 1) for "mxfp4"
    """

    def __init__(self, codes, scales, amax, rows, cols, scale_layout, fmt="nvfp4"):
        self.codes, self.scales, self.amax = codes, scales, amax
        self.rows, self.cols = int(rows), int(cols)
        self.scale_layout = scale_layout
        self.fmt = fmt

    @property
    def ld_codes(self) -> int:
        return int(self.codes.stride(0))

    def c(self) -> nvfp4_tensor:
        return nvfp4_tensor(self.codes.data_ptr(), self.scales.data_ptr(), self.amax.data_ptr(), self.rows,
                            self.cols, self.ld_codes, _LAYOUTS[self.scale_layout], _FORMATS[self.fmt])


def empty_qtensor(rows: int, cols: int, device, scale_layout: str = "mma", fmt: str = "nvfp4") -> QTensor:
    ld = ((cols // 2 + 15) // 16) * 16
    codes = torch.empty(rows, ld, dtype=torch.uint8, device=device)
    scales = torch.empty(max(nvfp4_scales_bytes(rows, cols, scale_layout), 16), dtype=torch.uint8, device=device)
    amax = torch.empty(4, dtype=torch.float32, device=device)
    return QTensor(codes, scales, amax, rows, cols, scale_layout, fmt)


def _in_dtype(x: torch.Tensor) -> int:
    if x.dtype == torch.bfloat16:
        return IN_BF16
    if x.dtype == torch.float32:
        return IN_FP32
    raise TypeError(f"input dtype {x.dtype} not supported (bf16 or fp32)")


def _check_input(x: torch.Tensor):
    if not x.is_cuda:
        raise ValueError("input must be a CUDA tensor")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("input must be a 2D row-major tensor")


def nvfp4_quantize(x: torch.Tensor, block: str = "1x16", round: str = "rtn", seed: int = 0, *,
                   rowwise: bool = True, colwise: bool = False, scale_layout: str = "mma",
                   out_rowwise: QTensor | None = None, out_colwise: QTensor | None = None, stream=None):
    """Quantize x [rows][cols]; returns (rowwise QTensor or None, colwise QTensor or None).
    block "1x16" / "16x16" give NVFP4, "mx1x32" MXFP4."""
    _check_input(x)
    rows, cols = x.shape
    fmt = "mxfp4" if block == "mx1x32" else "nvfp4"
    if rowwise and out_rowwise is None:
        out_rowwise = empty_qtensor(rows, cols, x.device, scale_layout, fmt)
    if colwise and out_colwise is None:
        out_colwise = empty_qtensor(cols, rows, x.device, scale_layout, fmt)
    r = out_rowwise.c() if rowwise else None
    c = out_colwise.c() if colwise else None
    sh = _stream(stream)
    ws = _workspace(x.device, sh)
    st = lib().nvfp4_quantize(x.data_ptr(), _in_dtype(x), rows, cols, x.stride(0), _BLOCKS[block], _ROUNDS[round],
                              seed, ctypes.byref(r) if r is not None else None,
                              ctypes.byref(c) if c is not None else None, ws.data_ptr(), ws.numel(), sh)
    _check(st, "nvfp4_quantize")
    return (out_rowwise if rowwise else None), (out_colwise if colwise else None)


def nvfp4_quantize_noalloc(x: torch.Tensor, block: str = "1x16", round: str = "rtn", seed: int = 0, *,
                           rowwise: bool = True, colwise: bool = False, scale_layout: str = "mma",
                           out_rowwise: QTensor | None = None, out_colwise: QTensor | None = None, stream=None):
    """nvfp4_quantize without a workspace: for callers that cannot allocate
    device memory, the library keeps the amax scratch in a fixed device array
    of its own.  Pass preallocated outputs to allocate nothing here either."""
    _check_input(x)
    rows, cols = x.shape
    fmt = "mxfp4" if block == "mx1x32" else "nvfp4"
    if rowwise and out_rowwise is None:
        out_rowwise = empty_qtensor(rows, cols, x.device, scale_layout, fmt)
    if colwise and out_colwise is None:
        out_colwise = empty_qtensor(cols, rows, x.device, scale_layout, fmt)
    r = out_rowwise.c() if rowwise else None
    c = out_colwise.c() if colwise else None
    st = lib().nvfp4_quantize_noalloc(x.data_ptr(), _in_dtype(x), rows, cols, x.stride(0), _BLOCKS[block],
                                      _ROUNDS[round], seed, ctypes.byref(r) if r is not None else None,
                                      ctypes.byref(c) if c is not None else None, _stream(stream))
    _check(st, "nvfp4_quantize_noalloc")
    return (out_rowwise if rowwise else None), (out_colwise if colwise else None)


def nvfp4_rht_quantize(x: torch.Tensor, round: str = "rtn", seed: int = 0, rht_seed: int = 0, *,
                       scale_layout: str = "mma", fmt: str = "nvfp4", out_colwise: QTensor | None = None,
                       stream=None) -> QTensor:
    """16-point RHT along the rows of x, then colwise quantization of the
    result's transpose: 1x16 NVFP4 (fmt "nvfp4") or 1x32 MXFP4 ("mxfp4");
    a given out_colwise decides by its own fmt."""
    _check_input(x)
    rows, cols = x.shape
    if out_colwise is None:
        out_colwise = empty_qtensor(cols, rows, x.device, scale_layout, fmt)
    c = out_colwise.c()
    sh = _stream(stream)
    ws = _workspace(x.device, sh)
    st = lib().nvfp4_rht_quantize(x.data_ptr(), _in_dtype(x), rows, cols, x.stride(0), _ROUNDS[round], seed,
                                  rht_seed, ctypes.byref(c), ws.data_ptr(), ws.numel(), sh)
    _check(st, "nvfp4_rht_quantize")
    return out_colwise


def nvfp4_quantize_with_rht(x: torch.Tensor, round: str = "rtn", seed: int = 0, rht_seed: int = 0, *,
                            scale_layout: str = "mma", out_rowwise: QTensor | None = None,
                            out_colwise: QTensor | None = None, stream=None) -> tuple[QTensor, QTensor]:
    """Both quantizations of one linear-layer operand from one amax read:
    (1x16 NVFP4 of x, 1x16 NVFP4 of the RHT of x along its rows, transposed).
    Bit for bit nvfp4_quantize(x) and nvfp4_rht_quantize(x) with the same
    round and seed."""
    _check_input(x)
    rows, cols = x.shape
    if out_rowwise is None:
        out_rowwise = empty_qtensor(rows, cols, x.device, scale_layout)
    if out_colwise is None:
        out_colwise = empty_qtensor(cols, rows, x.device, scale_layout)
    r, c = out_rowwise.c(), out_colwise.c()
    sh = _stream(stream)
    ws = _workspace(x.device, sh)
    st = lib().nvfp4_quantize_with_rht(x.data_ptr(), _in_dtype(x), rows, cols, x.stride(0), _ROUNDS[round], seed,
                                       rht_seed, ctypes.byref(r), ctypes.byref(c), ws.data_ptr(), ws.numel(), sh)
    _check(st, "nvfp4_quantize_with_rht")
    return out_rowwise, out_colwise


def nvfp4_rht_quantize_rowwise(x: torch.Tensor, round: str = "rtn", seed: int = 0, rht_seed: int = 0, *,
                               scale_layout: str = "mma", fmt: str = "nvfp4", out_rowwise: QTensor | None = None,
                               stream=None) -> QTensor:
    """16-point RHT along the columns of each row of x (in 16-element chunks),
    then rowwise quantization of the result: 1x16 NVFP4 or 1x32 MXFP4."""
    _check_input(x)
    rows, cols = x.shape
    if out_rowwise is None:
        out_rowwise = empty_qtensor(rows, cols, x.device, scale_layout, fmt)
    r = out_rowwise.c()
    sh = _stream(stream)
    ws = _workspace(x.device, sh)
    st = lib().nvfp4_rht_quantize_rowwise(x.data_ptr(), _in_dtype(x), rows, cols, x.stride(0), _ROUNDS[round], seed,
                                          rht_seed, ctypes.byref(r), ws.data_ptr(), ws.numel(), sh)
    _check(st, "nvfp4_rht_quantize_rowwise")
    return out_rowwise


def _out_mode(out: torch.Tensor, accumulate: bool) -> int:
    if accumulate:
        if out.dtype != torch.float32:
            raise ValueError("accumulate=True needs an FP32 output to add into")
        return OUT_FP32_ADD
    return {torch.bfloat16: OUT_BF16, torch.float32: OUT_FP32}[out.dtype]


def nvfp4_gemm(a: QTensor, b: QTensor, out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
               stream=None, accumulate: bool = False) -> torch.Tensor:
    """C[M][N] = dequant(a) @ dequant(b)^T on the FP4 tensor cores (FP32
    accumulation); accumulate=True adds the result into the FP32 ``out``."""
    if out is None:
        if accumulate:
            raise ValueError("accumulate=True needs an existing FP32 output")
        out = torch.empty(a.rows, b.rows, dtype=out_dtype, device=a.codes.device)
    od = _out_mode(out, accumulate)
    ca, cb = a.c(), b.c()
    st = lib().nvfp4_gemm(ctypes.byref(ca), ctypes.byref(cb), out.data_ptr(), od, out.stride(0), None, 0,
                          _stream(stream))
    _check(st, "nvfp4_gemm")
    return out


def nvfp4_gemm_pair(a0: QTensor, b0: QTensor, out0: torch.Tensor, a1: QTensor, b1: QTensor, out1: torch.Tensor,
                    stream=None, accumulate0: bool = False, accumulate1: bool = False):
    """nvfp4_gemm(a0, b0, out=out0) and nvfp4_gemm(a1, b1, out=out1) in one
    launch (bit for bit the same outputs)."""
    od0, od1 = _out_mode(out0, accumulate0), _out_mode(out1, accumulate1)
    c = [t.c() for t in (a0, b0, a1, b1)]
    st = lib().nvfp4_gemm_pair(ctypes.byref(c[0]), ctypes.byref(c[1]), out0.data_ptr(), od0, out0.stride(0),
                               ctypes.byref(c[2]), ctypes.byref(c[3]), out1.data_ptr(), od1, out1.stride(0),
                               _stream(stream))
    _check(st, "nvfp4_gemm_pair")
    return out0, out1


def nvfp4_gemm_bf16(a: torch.Tensor, b: torch.Tensor, out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
                    stream=None, accumulate: bool = False) -> torch.Tensor:
    """C[M][N] = a @ b^T for bf16 a [M][K], b [N][K] on the tensor cores (FP32
    accumulation); accumulate=True adds the result into the FP32 ``out``."""
    for t in (a, b):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("a and b must be 2D row-major bf16 CUDA tensors")
    if a.shape[1] != b.shape[1]:
        raise ValueError(f"K mismatch: {tuple(a.shape)} vs {tuple(b.shape)}")
    if out is None:
        if accumulate:
            raise ValueError("accumulate=True needs an existing FP32 output")
        out = torch.empty(a.shape[0], b.shape[0], dtype=out_dtype, device=a.device)
    od = _out_mode(out, accumulate)
    st = lib().nvfp4_gemm_bf16(a.data_ptr(), a.stride(0), b.data_ptr(), b.stride(0), out.data_ptr(), od,
                               out.stride(0), a.shape[0], b.shape[0], a.shape[1], _stream(stream))
    _check(st, "nvfp4_gemm_bf16")
    return out


def nvfp4_transpose_bf16(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """x^T of a 2D row-major bf16 CUDA tensor (rows, cols multiples of 8)."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2D row-major bf16 CUDA tensor")
    rows, cols = x.shape
    if out is None:
        out = torch.empty(cols, rows, dtype=torch.bfloat16, device=x.device)
    st = lib().nvfp4_transpose_bf16(x.data_ptr(), rows, cols, x.stride(0), out.data_ptr(), out.stride(0),
                                    _stream(stream))
    _check(st, "nvfp4_transpose_bf16")
    return out


class LinearContext:
    """Caller-owned quantized buffers of one NVFP4 linear layer Y = X W^T
    (X [M][K], W [N][K]); see nvfp4_linear_fwd / nvfp4_linear_bwd."""

    def __init__(self, M: int, N: int, K: int, device, two_streams: bool = True):
        self.M, self.N, self.K = M, N, K
        self.xq = empty_qtensor(M, K, device)
        self.wq = empty_qtensor(N, K, device)
        self.wtq = empty_qtensor(K, N, device)
        self.dyq = empty_qtensor(M, N, device)
        self.dytq = empty_qtensor(N, M, device)
        self.xtq = empty_qtensor(K, M, device)
        # the larger workspace lets the forward quantize W on a second stream
        ws = nvfp4_linear_workspace_size() if two_streams else nvfp4_workspace_size()
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)

    def c(self, dw_accumulate: bool = False) -> nvfp4_linear_ctx:
        return nvfp4_linear_ctx(self.M, self.N, self.K, self.xq.c(), self.wq.c(), self.wtq.c(), self.dyq.c(),
                                self.dytq.c(), self.xtq.c(), self.workspace.data_ptr(), self.workspace.numel(),
                                1 if dw_accumulate else 0)


def nvfp4_linear_fwd(X: torch.Tensor, W: torch.Tensor, ctx: LinearContext, Y: torch.Tensor | None = None,
                     stream=None, rht_seed: int | None = None) -> torch.Tensor:
    """Y = X W^T.  With rht_seed: nvfp4_linear_fwd_rht, which also fills
    ctx.xtq (X^T after the RHT, for Wgrad) from the same read of X; the
    backward then takes X=None."""
    if Y is None:
        Y = torch.empty(ctx.M, ctx.N, dtype=torch.bfloat16, device=X.device)
    for t, shape in ((X, (ctx.M, ctx.K)), (W, (ctx.N, ctx.K)), (Y, (ctx.M, ctx.N))):
        if t.dtype != torch.bfloat16 or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"expected contiguous bf16 {shape}, got {t.dtype} {tuple(t.shape)}")
    c = ctx.c()
    if rht_seed is None:
        _check(lib().nvfp4_linear_fwd(X.data_ptr(), W.data_ptr(), Y.data_ptr(), ctypes.byref(c), _stream(stream)),
               "nvfp4_linear_fwd")
    else:
        _check(lib().nvfp4_linear_fwd_rht(X.data_ptr(), W.data_ptr(), Y.data_ptr(), int(rht_seed), ctypes.byref(c),
                                          _stream(stream)), "nvfp4_linear_fwd_rht")
    return Y


def nvfp4_linear_bwd(dY: torch.Tensor, X: torch.Tensor | None, ctx: LinearContext, sr_seed: int, rht_seed: int,
                     dX: torch.Tensor | None = None, dW: torch.Tensor | None = None, stream=None,
                     accumulate_dw: bool = False):
    """Dgrad and Wgrad of the layer; with accumulate_dw=True the FP32 Wgrad
    result is added into the given dW instead of overwriting it.  X=None:
    ctx.xtq already holds X^T's codes (nvfp4_linear_fwd with rht_seed)."""
    if dX is None:
        dX = torch.empty(ctx.M, ctx.K, dtype=torch.bfloat16, device=dY.device)
    if dW is None:
        if accumulate_dw:
            raise ValueError("accumulate_dw=True needs an existing FP32 dW")
        dW = torch.empty(ctx.N, ctx.K, dtype=torch.float32, device=dY.device)
    for t, shape, dt in ((dY, (ctx.M, ctx.N), torch.bfloat16), (X, (ctx.M, ctx.K), torch.bfloat16),
                         (dX, (ctx.M, ctx.K), torch.bfloat16), (dW, (ctx.N, ctx.K), torch.float32)):
        if t is None:
            continue
        if t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"expected contiguous {dt} {shape}, got {t.dtype} {tuple(t.shape)}")
    c = ctx.c(dw_accumulate=accumulate_dw)
    _check(lib().nvfp4_linear_bwd(dY.data_ptr(), None if X is None else X.data_ptr(), dX.data_ptr(), dW.data_ptr(),
                                  sr_seed, rht_seed, ctypes.byref(c), _stream(stream)), "nvfp4_linear_bwd")
    return dX, dW


def nvfp4_set_wait_limit_ns(limit_ns: int) -> int:
    """Bound of every device-side wait in the GEMM kernels (0: the default,
    4 s); returns the previous setting.  For tests and diagnostics."""
    return int(lib().nvfp4_set_wait_limit_ns(int(limit_ns)))


def nvfp4_sync_status(stream=None) -> int:
    """Synchronize the stream and return (and clear) the device status code."""
    return int(lib().nvfp4_sync_status(_stream(stream)))


def nvfp4_checked_build() -> bool:
    """True when the loaded library is the checked build (NVFP4_CHECKED=1)."""
    return bool(lib().nvfp4_checked_build())


def nvfp4_checked_selftest(stream=None) -> int:
    """Checked build: one guarded store past its buffer must be skipped and
    reported (returns ERR_BOUNDS); ERR_UNSUPPORTED in the normal build."""
    return int(lib().nvfp4_checked_selftest(_stream(stream)))


def scales_as_linear(q: QTensor) -> torch.Tensor:
    """The block scales of q as a [rows][cols/16] uint8 tensor (undoes the
    MMA layout's index permutation; a pure gather, no arithmetic)."""
    nkb = q.cols // 16
    if q.scale_layout == "linear":
        return q.scales[: q.rows * nkb].view(q.rows, nkb)
    n_katoms = 4 * ((q.cols + 255) // 256)
    dev = q.scales.device
    r = torch.arange(q.rows, device=dev, dtype=torch.int64)[:, None]
    kb = torch.arange(nkb, device=dev, dtype=torch.int64)[None, :]
    off = ((r // 128) * n_katoms + kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    return q.scales[off]


def codes_view(q: QTensor) -> torch.Tensor:
    """The packed codes of q without row padding: [rows][cols/2] uint8."""
    return q.codes[:, : q.cols // 2]

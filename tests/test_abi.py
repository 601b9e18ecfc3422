"""The C-ABI library builds, loads and exports every entry point that
include/nvfp4.h declares; host-side argument checks answer without a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nvfp4.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(nvfp4_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as q
    return q.lib()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ["nvfp4_quantize", "nvfp4_rht_quantize", "nvfp4_gemm", "nvfp4_linear_fwd", "nvfp4_linear_bwd",
                     "nvfp4_sync_status", "nvfp4_status_string", "nvfp4_workspace_size", "nvfp4_scales_bytes",
                     "nvfp4_last_error"]:
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_normal_build_has_no_bounds_checks(L):
    # the checked build is a separate library (NVFP4_CHECKED=1); this one
    # answers that it is not, and its self-test refuses before any launch
    import quantize_block_scaled_amax_gb300 as q
    from quantize_block_scaled_amax_gb300 import build
    if build.CHECKED:
        pytest.skip("this process runs the checked build")
    assert L.nvfp4_checked_build() == 0
    assert L.nvfp4_checked_selftest(None) == q.ERR_UNSUPPORTED
    assert q.ERR_BOUNDS == 7 and L.nvfp4_status_string(q.ERR_BOUNDS).startswith(b"device index out of bounds")


def test_struct_layout_matches_header(L, tmp_path):
    # the binding's ctypes structures against the C compiler's view of the
    # header: every field's offset and each struct's size
    import subprocess
    import quantize_block_scaled_amax_gb300 as q
    structs = {"nvfp4_tensor": q.nvfp4_tensor, "nvfp4_linear_ctx": q.nvfp4_linear_ctx}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "nvfp4.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'printf("{name} sizeof %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for name, cls in structs.items():
        assert got[(name, "sizeof")] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert got[(name, field)] == getattr(cls, field).offset, (name, field)


def test_status_strings(L):
    for code in range(7):
        assert L.nvfp4_status_string(code)
    assert L.nvfp4_status_string(4) == b"non-finite input"


def test_scales_bytes(L):
    import quantize_block_scaled_amax_gb300 as q
    # linear: one byte per 1x16 block
    assert q.nvfp4_scales_bytes(8192, 5120, "linear") == 8192 * 320
    # MMA layout: 128-row groups x 4*ceil(K/256) atoms of 512 bytes
    assert q.nvfp4_scales_bytes(8192, 5120, "mma") == 64 * 80 * 512
    assert q.nvfp4_scales_bytes(200, 320, "mma") == 2 * 8 * 512
    assert q.nvfp4_scales_bytes(16, 17, "mma") == 0          # cols not a multiple of 16
    assert q.nvfp4_workspace_size() >= 4096
    # the layer's workspace: nvfp4_quantize_with_rht's 16 KB plus the 8 KB
    # of W's quantization on the second stream
    assert q.nvfp4_linear_workspace_size() == q.nvfp4_workspace_size() * 3 // 2


def test_host_argument_checks_need_no_gpu(L):
    # every call below must fail its host-side checks before any launch: the
    # pointers are placeholders, never dereferenced
    import quantize_block_scaled_amax_gb300 as q
    t = q.nvfp4_tensor(16, 16, 16, 16, 32, 16, 1, 0)
    # null input
    assert L.nvfp4_quantize(None, 0, 16, 32, 32, 0, 0, 0, ctypes.byref(t), None, 16, 8192, None) == q.ERR_INVALID_ARG
    # cols not a multiple of 16
    assert L.nvfp4_quantize(16, 0, 16, 24, 24, 0, 0, 0, ctypes.byref(t), None, 16, 8192, None) == q.ERR_INVALID_ARG
    # empty input
    assert L.nvfp4_quantize(16, 0, 0, 32, 32, 0, 0, 0, ctypes.byref(t), None, 16, 8192, None) == q.ERR_INVALID_ARG
    # no output
    assert L.nvfp4_quantize(16, 0, 16, 32, 32, 0, 0, 0, None, None, 16, 8192, None) == q.ERR_INVALID_ARG
    # misaligned input pointer
    assert L.nvfp4_quantize(24, 0, 16, 32, 32, 0, 0, 0, ctypes.byref(t), None, 16, 8192, None) == q.ERR_INVALID_ARG
    # output shape mismatch
    bad = q.nvfp4_tensor(16, 16, 16, 16, 64, 32, 1, 0)
    assert L.nvfp4_quantize(16, 0, 16, 32, 32, 0, 0, 0, ctypes.byref(bad), None, 16, 8192, None) == q.ERR_INVALID_ARG
    # 16x16 with SR is not offered
    assert L.nvfp4_quantize(16, 0, 16, 32, 32, 1, 1, 0, ctypes.byref(t), None, 16, 8192, None) == q.ERR_UNSUPPORTED
    # workspace too small
    assert L.nvfp4_quantize(16, 0, 16, 32, 32, 0, 0, 0, ctypes.byref(t), None, 16, 64, None) == q.ERR_WORKSPACE
    assert b"workspace" in L.nvfp4_last_error()
    # MXFP4: 32-element blocks, and outputs of the MXFP4 format
    tm = q.nvfp4_tensor(16, 16, 16, 16, 48, 32, 1, 1)
    assert L.nvfp4_quantize(16, 0, 16, 48, 48, 2, 0, 0, ctypes.byref(tm), None, 16, 8192, None) == q.ERR_INVALID_ARG
    tm = q.nvfp4_tensor(16, 16, 16, 16, 64, 32, 1, 0)      # NVFP4-format output for an MX block
    assert L.nvfp4_quantize(16, 0, 16, 64, 64, 2, 0, 0, ctypes.byref(tm), None, 16, 8192, None) == q.ERR_INVALID_ARG
    tm = q.nvfp4_tensor(16, 16, 16, 16, 64, 32, 1, 7)      # unknown format
    assert L.nvfp4_quantize(16, 0, 16, 64, 64, 0, 0, 0, ctypes.byref(tm), None, 16, 8192, None) == q.ERR_INVALID_ARG
    # RHT needs rows % 16 == 0
    tc2 = q.nvfp4_tensor(16, 16, 16, 32, 24, 16, 1, 0)
    assert L.nvfp4_rht_quantize(16, 0, 24, 32, 32, 0, 0, 0, ctypes.byref(tc2), 16, 8192, None) == q.ERR_INVALID_ARG


def test_quantize_with_rht_argument_checks_need_no_gpu(L):
    import quantize_block_scaled_amax_gb300 as q
    r = q.nvfp4_tensor(16, 16, 16, 32, 64, 32, 1, 0)       # x^T... rowwise [32][64]
    c = q.nvfp4_tensor(16, 16, 16, 64, 32, 16, 1, 0)       # colwise [64][32]
    ws = 2 * 8192
    # both outputs required
    assert L.nvfp4_quantize_with_rht(16, 0, 32, 64, 64, 0, 0, 0, ctypes.byref(r), None, 16, ws, None) == \
        q.ERR_INVALID_ARG
    # rows % 16
    r24 = q.nvfp4_tensor(16, 16, 16, 24, 64, 32, 1, 0)
    c24 = q.nvfp4_tensor(16, 16, 16, 64, 24, 16, 1, 0)
    assert L.nvfp4_quantize_with_rht(16, 0, 24, 64, 64, 0, 0, 0, ctypes.byref(r24), ctypes.byref(c24), 16, ws,
                                     None) == q.ERR_INVALID_ARG
    # MXFP4 outputs
    rm = q.nvfp4_tensor(16, 16, 16, 32, 64, 32, 1, 1)
    cm = q.nvfp4_tensor(16, 16, 16, 64, 32, 16, 1, 1)
    assert L.nvfp4_quantize_with_rht(16, 0, 32, 64, 64, 0, 0, 0, ctypes.byref(rm), ctypes.byref(cm), 16, ws,
                                     None) == q.ERR_INVALID_ARG
    # 8 KB is enough for the single calls but not for this one
    assert L.nvfp4_quantize_with_rht(16, 0, 32, 64, 64, 0, 0, 0, ctypes.byref(r), ctypes.byref(c), 16, 8192,
                                     None) == q.ERR_WORKSPACE
    assert b"workspace" in L.nvfp4_last_error()
    assert q.nvfp4_workspace_size() >= ws


def test_transpose_argument_checks_need_no_gpu(L):
    import quantize_block_scaled_amax_gb300 as q
    assert L.nvfp4_transpose_bf16(None, 8, 8, 8, 16, 8, None) == q.ERR_INVALID_ARG      # null x
    assert L.nvfp4_transpose_bf16(16, 12, 8, 8, 16, 16, None) == q.ERR_INVALID_ARG     # rows % 8
    assert L.nvfp4_transpose_bf16(16, 8, 8, 4, 16, 8, None) == q.ERR_INVALID_ARG       # ldx < cols
    assert L.nvfp4_transpose_bf16(16, 8, 8, 8, 16, 4, None) == q.ERR_INVALID_ARG       # ldy < rows
    assert L.nvfp4_transpose_bf16(24, 8, 8, 8, 16, 8, None) == q.ERR_INVALID_ARG       # misaligned x
    assert L.nvfp4_transpose_bf16(16, 8, 8, 8, 0, 8, None) == q.ERR_INVALID_ARG        # null y


def test_bf16_gemm_argument_checks_need_no_gpu(L):
    import quantize_block_scaled_amax_gb300 as q
    # K % 8 != 0
    assert L.nvfp4_gemm_bf16(16, 12, 16, 12, 16, 0, 64, 64, 64, 12, None) == q.ERR_INVALID_ARG
    # misaligned A
    assert L.nvfp4_gemm_bf16(24, 64, 16, 64, 16, 0, 64, 64, 64, 64, None) == q.ERR_INVALID_ARG
    # lda < K
    assert L.nvfp4_gemm_bf16(16, 32, 16, 64, 16, 0, 64, 64, 64, 64, None) == q.ERR_INVALID_ARG


def test_gemm_argument_checks_need_no_gpu(L):
    import quantize_block_scaled_amax_gb300 as q
    a = q.nvfp4_tensor(16, 16, 16, 128, 128, 64, 1, 0)
    b = q.nvfp4_tensor(16, 16, 16, 64, 64, 32, 1, 0)      # K mismatch
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), 16, 0, 64, None, 0, None) == q.ERR_INVALID_ARG
    b = q.nvfp4_tensor(16, 16, 16, 64, 128, 64, 0, 0)     # row-major (LINEAR) scales
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), 16, 0, 64, None, 0, None) == q.ERR_INVALID_ARG
    b = q.nvfp4_tensor(16, 24, 16, 64, 128, 64, 1, 0)     # scale buffer not 16-byte aligned
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), 16, 0, 64, None, 0, None) == q.ERR_INVALID_ARG
    b = q.nvfp4_tensor(16, 16, 16, 64, 128, 64, 1, 1)     # MXFP4 B with an NVFP4 A
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), 16, 0, 64, None, 0, None) == q.ERR_INVALID_ARG
    a = q.nvfp4_tensor(16, 16, 16, 128, 96, 48, 1, 0)     # K % 64 != 0
    b = q.nvfp4_tensor(16, 16, 16, 64, 96, 48, 1, 0)
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), 16, 0, 64, None, 0, None) == q.ERR_INVALID_ARG


def test_gemm_pair_argument_checks_need_no_gpu(L):
    # nvfp4_gemm_pair checks both problems (the same checks as nvfp4_gemm)
    # and refuses two formats, all before any launch
    import quantize_block_scaled_amax_gb300 as q
    a = q.nvfp4_tensor(16, 16, 16, 128, 128, 64, 1, 0)
    b = q.nvfp4_tensor(16, 16, 16, 64, 128, 64, 1, 0)
    bad = q.nvfp4_tensor(16, 16, 16, 64, 64, 32, 1, 0)     # K mismatch with a
    pair = lambda a0, b0, c0, a1, b1, c1: L.nvfp4_gemm_pair(ctypes.byref(a0), ctypes.byref(b0), c0, 0, 64,
                                                             ctypes.byref(a1), ctypes.byref(b1), c1, 0, 64, None)
    assert pair(a, bad, 16, a, b, 16) == q.ERR_INVALID_ARG      # first problem invalid
    assert pair(a, b, 16, a, bad, 16) == q.ERR_INVALID_ARG      # second problem invalid
    assert pair(a, b, None, a, b, 16) == q.ERR_INVALID_ARG      # null C0
    assert pair(a, b, 16, a, b, 24) == q.ERR_INVALID_ARG        # C1 not 16-byte aligned
    am = q.nvfp4_tensor(16, 16, 16, 128, 128, 64, 1, 1)
    bm = q.nvfp4_tensor(16, 16, 16, 64, 128, 64, 1, 1)
    assert pair(a, b, 16, am, bm, 16) == q.ERR_INVALID_ARG      # NVFP4 with MXFP4
    assert b"format" in L.nvfp4_last_error()


def test_rht_quantize_rowwise_argument_checks_need_no_gpu(L):
    import quantize_block_scaled_amax_gb300 as q
    t = q.nvfp4_tensor(16, 16, 16, 16, 64, 32, 1, 0)       # y [16][64], NVFP4
    ws = 8192
    args = lambda x, cols, rnd, out, wsb: L.nvfp4_rht_quantize_rowwise(x, 0, 16, cols, cols, rnd, 0, 0, out, 16,
                                                                        wsb, None)
    assert args(None, 64, 0, ctypes.byref(t), ws) == q.ERR_INVALID_ARG                 # null x
    assert args(16, 40, 0, ctypes.byref(t), ws) == q.ERR_INVALID_ARG                   # cols % 16
    assert args(16, 64, 5, ctypes.byref(t), ws) == q.ERR_INVALID_ARG                   # no such rounding
    assert args(16, 64, 0, None, ws) == q.ERR_INVALID_ARG                              # no output
    wrong = q.nvfp4_tensor(16, 16, 16, 32, 64, 32, 1, 0)    # [32][64] for a [16][64] input
    assert args(16, 64, 0, ctypes.byref(wrong), ws) == q.ERR_INVALID_ARG
    mx = q.nvfp4_tensor(16, 16, 16, 16, 48, 32, 1, 1)       # MXFP4 needs cols % 32
    assert args(16, 48, 0, ctypes.byref(mx), ws) == q.ERR_INVALID_ARG
    assert args(16, 64, 0, ctypes.byref(t), 64) == q.ERR_WORKSPACE                     # workspace too small
    assert b"workspace" in L.nvfp4_last_error()


def test_linear_argument_checks_need_no_gpu(L):
    # the layer entry points check the context before their first call
    import quantize_block_scaled_amax_gb300 as q
    M, N, K = 64, 128, 64

    def t(rows, cols, layout=1):
        return q.nvfp4_tensor(16, 16, 16, rows, cols, max(16, cols // 2), layout, 0)

    def ctx(**over):
        c = q.nvfp4_linear_ctx(M, N, K, t(M, K), t(N, K), t(K, N), t(M, N), t(N, M), t(K, M), 16, 16384)
        for k, v in over.items():
            setattr(c, k, v)
        return c

    fwd = lambda c, x=16: L.nvfp4_linear_fwd(x, 16, 16, ctypes.byref(c) if c is not None else None, None)
    assert fwd(None) == q.ERR_INVALID_ARG                                             # no context
    assert fwd(ctx(), x=None) == q.ERR_INVALID_ARG                                    # null X
    assert fwd(ctx(M=96)) == q.ERR_INVALID_ARG                                        # M % 64
    assert fwd(ctx(xq=t(M, 2 * K))) == q.ERR_INVALID_ARG                              # xq shape
    assert fwd(ctx(wq=t(N, K, layout=0))) == q.ERR_INVALID_ARG                        # wq needs MMA scales
    assert fwd(ctx(wtq=t(N, K))) == q.ERR_INVALID_ARG                                 # wtq is [K][N]
    assert b"wtq" in L.nvfp4_last_error()
    assert fwd(ctx(workspace_bytes=8192)) == q.ERR_WORKSPACE                          # below 16 KB
    # a W that its own quantization refuses (not 16-byte aligned): the error
    # comes back through the forward's fork/join, whichever stream W was on
    lw = q.nvfp4_linear_workspace_size()
    assert L.nvfp4_linear_fwd(16, 24, 16, ctypes.byref(ctx(workspace_bytes=lw)), None) == q.ERR_INVALID_ARG
    assert b"aligned" in L.nvfp4_last_error()

    # the forward that also writes Wgrad's X^T codes checks xtq as well
    fwd_rht = lambda c, x=16: L.nvfp4_linear_fwd_rht(x, 16, 16, 5, ctypes.byref(c) if c is not None else None, None)
    assert fwd_rht(None) == q.ERR_INVALID_ARG                                         # no context
    assert fwd_rht(ctx(), x=None) == q.ERR_INVALID_ARG                                # null X
    assert fwd_rht(ctx(xtq=t(N, M))) == q.ERR_INVALID_ARG                             # xtq is [K][M]
    assert b"xtq" in L.nvfp4_last_error()

    bwd = lambda c, dw=16: L.nvfp4_linear_bwd(16, 16, 16, dw, 1, 2, ctypes.byref(c), None)
    assert bwd(ctx(), dw=None) == q.ERR_INVALID_ARG                                   # null dW
    assert bwd(ctx(K=0)) == q.ERR_INVALID_ARG                                         # empty
    assert bwd(ctx(dyq=t(N, M))) == q.ERR_INVALID_ARG                                 # dyq is [M][N]
    assert bwd(ctx(dytq=t(M, N))) == q.ERR_INVALID_ARG                                # dytq is [N][M]
    assert bwd(ctx(xtq=t(K, M, layout=0))) == q.ERR_INVALID_ARG                       # xtq needs MMA scales
    assert b"xtq" in L.nvfp4_last_error()

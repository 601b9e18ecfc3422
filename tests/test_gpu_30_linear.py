"""The linear-layer entry points (Fprop, Dgrad, Wgrad with the recipe's
roundings and transforms) against the oracle composed step by step."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import assert_gemm_close, assert_quant_equal, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    return nv


@pytest.mark.parametrize("mnk", [(128, 128, 128), (256, 384, 320), (512, 1024, 768)])
def test_linear_fwd_bwd(nv, mnk):
    m, n, k = mnk
    x, w, dy = workloads.linear_layer(m, n, k)
    ctx = nv.LinearContext(m, n, k, "cuda")
    y = nv.nvfp4_linear_fwd(x.cuda(), w.cuda(), ctx)
    dx, dw = nv.nvfp4_linear_bwd(dy.cuda(), x.cuda(), ctx, sr_seed=workloads.SR_SEED, rht_seed=workloads.RHT_SEED)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    xn, wn, dyn = to_f32_np(x), to_f32_np(w), to_f32_np(dy)
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    o = {
        "xq": oracle.quantize(xn),
        "wq": oracle.quantize(wn, block="16x16"),
        "wtq": oracle.quantize(wn, layout="col", block="16x16"),
        "dyq": oracle.quantize(dyn, rounding="sr", seed=sr),
        "dytq": oracle.quantize(dyn, layout="col", rounding="sr", seed=sr, rht_seed=rh),
        "xtq": oracle.quantize(xn, layout="col", rht_seed=rh),
    }
    for name, ref in o.items():
        assert_quant_equal(getattr(ctx, name), ref, what=name)
    d = {name: oracle.dequantize(q) for name, q in o.items()}
    assert_gemm_close(y.float().cpu().numpy(), d["xq"] @ d["wq"].T, d["xq"], d["wq"], bf16=True, what="Y")
    assert_gemm_close(dx.float().cpu().numpy(), d["dyq"] @ d["wtq"].T, d["dyq"], d["wtq"], bf16=True, what="dX")
    assert_gemm_close(dw.cpu().numpy(), d["dytq"] @ d["xtq"].T, d["dytq"], d["xtq"], bf16=False, what="dW")
    # FP32-output twins of the layer's bf16 Fprop and Dgrad, on the same
    # quantized operands: the strict relative-Frobenius bound
    y32 = nv.nvfp4_gemm(ctx.xq, ctx.wq, out_dtype=torch.float32)
    dx32 = nv.nvfp4_gemm(ctx.dyq, ctx.wtq, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_gemm_close(y32.cpu().numpy(), d["xq"] @ d["wq"].T, d["xq"], d["wq"], bf16=False, what="Y fp32")
    assert_gemm_close(dx32.cpu().numpy(), d["dyq"] @ d["wtq"].T, d["dyq"], d["wtq"], bf16=False, what="dX fp32")
    # fidelity to the unquantized layer (a loose sanity bound, not parity)
    yr = xn.astype(np.float64) @ wn.astype(np.float64).T
    assert np.linalg.norm(y.float().cpu().numpy() - yr) / np.linalg.norm(yr) < 0.2


def test_forward_with_rht_matches_the_two_pass_layer(nv):
    # nvfp4_linear_fwd_rht quantizes X^T for Wgrad in the forward, from the
    # same read of X as xq; the backward then takes X = NULL.  Every
    # quantized operand and Y, dX, dW must equal the plain forward and the
    # backward's own X^T quantization bit for bit.
    m, n, k = 256, 384, 320
    x, w, dy = workloads.linear_layer(m, n, k)
    x, w, dy = x.cuda(), w.cuda(), dy.cuda()
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    a = nv.LinearContext(m, n, k, "cuda")
    ya = nv.nvfp4_linear_fwd(x, w, a)
    dxa, dwa = nv.nvfp4_linear_bwd(dy, x, a, sr_seed=sr, rht_seed=rh)
    b = nv.LinearContext(m, n, k, "cuda")
    yb = nv.nvfp4_linear_fwd(x, w, b, rht_seed=rh)
    xtq_fwd = b.xtq.codes.clone()
    dxb, dwb = nv.nvfp4_linear_bwd(dy, None, b, sr_seed=sr, rht_seed=rh)
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    assert torch.equal(xtq_fwd, b.xtq.codes)        # the backward left xtq as the forward wrote it
    for name in ("xq", "wq", "wtq", "dyq", "dytq", "xtq"):
        qa, qb = getattr(a, name), getattr(b, name)
        assert torch.equal(qa.codes, qb.codes) and torch.equal(qa.scales, qb.scales), name
        assert torch.equal(qa.amax[:3], qb.amax[:3]), name      # {A, S_dec, S_enc}
    assert torch.equal(ya, yb) and torch.equal(dxa, dxb) and torch.equal(dwa, dwb)
    assert_quant_equal(b.xtq, oracle.quantize(to_f32_np(x), layout="col", rht_seed=rh), what="xtq from the forward")


def _quantized_equal(a, b, names=("xq", "wq", "wtq", "dyq", "dytq", "xtq")):
    for name in names:
        qa, qb = getattr(a, name), getattr(b, name)
        assert torch.equal(qa.codes, qb.codes) and torch.equal(qa.scales, qb.scales), name
        assert torch.equal(qa.amax[:3], qb.amax[:3]), name


def test_two_stream_forward_equals_one_stream(nv):
    # With the larger workspace the forward quantizes W on the library's
    # second stream while X is quantized on the caller's; the results must
    # equal the one-stream forward bit for bit, repeatedly, and the caller's
    # stream must see them without any synchronization of its own.
    m, n, k = 512, 1024, 768
    x, w, dy = workloads.linear_layer(m, n, k)
    x, w, dy = x.cuda(), w.cuda(), dy.cuda()
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    one = nv.LinearContext(m, n, k, "cuda", two_streams=False)
    two = nv.LinearContext(m, n, k, "cuda")
    assert one.workspace.numel() == nv.nvfp4_workspace_size()
    assert two.workspace.numel() == nv.nvfp4_linear_workspace_size()
    y1 = nv.nvfp4_linear_fwd(x, w, one, rht_seed=rh)
    dx1, dw1 = nv.nvfp4_linear_bwd(dy, None, one, sr_seed=sr, rht_seed=rh)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        s.wait_stream(torch.cuda.default_stream())
        for _ in range(3):
            y2 = nv.nvfp4_linear_fwd(x, w, two, rht_seed=rh)
            dx2, dw2 = nv.nvfp4_linear_bwd(dy, None, two, sr_seed=sr, rht_seed=rh)
            # read on the caller's stream right after the forward's join
            wsum = two.wtq.codes.to(torch.int64).sum()
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    _quantized_equal(one, two)
    assert torch.equal(y1, y2) and torch.equal(dx1, dx2) and torch.equal(dw1, dw2)
    assert int(wsum) == int(one.wtq.codes.to(torch.int64).sum())


def test_layer_step_captured_in_a_cuda_graph(nv):
    # The layer's forward and backward captured into one CUDA graph and
    # replayed: the same results as the eager calls (under capture the
    # forward keeps both quantizations on the capturing stream).
    m, n, k = 256, 384, 320
    x, w, dy = workloads.linear_layer(m, n, k)
    x, w, dy = x.cuda(), w.cuda(), dy.cuda()
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    eager = nv.LinearContext(m, n, k, "cuda")
    ye = nv.nvfp4_linear_fwd(x, w, eager, rht_seed=rh)
    dxe, dwe = nv.nvfp4_linear_bwd(dy, None, eager, sr_seed=sr, rht_seed=rh)
    torch.cuda.synchronize()
    cap = nv.LinearContext(m, n, k, "cuda")
    y = torch.empty_like(ye)
    dx, dw = torch.empty_like(dxe), torch.empty_like(dwe)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nv.nvfp4_linear_fwd(x, w, cap, Y=y, rht_seed=rh)
        nv.nvfp4_linear_bwd(dy, None, cap, sr_seed=sr, rht_seed=rh, dX=dx, dW=dw)
    for _ in range(2):
        y.zero_(); dx.zero_(); dw.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert nv.nvfp4_sync_status() == nv.OK
        _quantized_equal(eager, cap)
        assert torch.equal(ye, y) and torch.equal(dxe, dx) and torch.equal(dwe, dw)


def test_two_stream_forwards_from_two_threads(nv):
    # Two host threads, each with its own context and stream, run forwards
    # at the same time: the library's second stream and its fork/join
    # events are shared by both, so their record-to-wait sequences must not
    # interleave.  Every result must equal the one-stream forward.
    import threading
    m, n, k = 256, 384, 320
    rh = workloads.RHT_SEED
    inputs = [(workloads.activations(m, k, seed=workloads.SEED_BASE + 40 + t),
               workloads.weights(n, k, seed=workloads.SEED_BASE + 42 + t), None) for t in (0, 1)]
    refs = []
    for x, w, _ in inputs:
        c = nv.LinearContext(m, n, k, "cuda", two_streams=False)
        refs.append((nv.nvfp4_linear_fwd(x.cuda(), w.cuda(), c, rht_seed=rh), c))
    torch.cuda.synchronize()
    outs, errors = [None, None], []

    def run(t):
        try:
            x, w, _ = inputs[t]
            x, w = x.cuda(), w.cuda()
            c = nv.LinearContext(m, n, k, "cuda")
            s = torch.cuda.Stream()
            ys = []
            with torch.cuda.stream(s):
                for _ in range(20):
                    ys.append(nv.nvfp4_linear_fwd(x, w, c, rht_seed=rh))
            s.synchronize()
            outs[t] = (ys, c)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(t,)) for t in (0, 1)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert nv.nvfp4_sync_status() == nv.OK
    for t in (0, 1):
        ys, c = outs[t]
        y_ref, c_ref = refs[t]
        for y in ys:
            assert torch.equal(y, y_ref)
        _quantized_equal(c_ref, c, names=("xq", "wq", "wtq", "xtq"))

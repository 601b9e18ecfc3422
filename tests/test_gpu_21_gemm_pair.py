"""nvfp4_gemm_pair: two block-scaled GEMMs in one persistent launch.  Each
output must equal nvfp4_gemm's for the same problem bit for bit (a tile is
computed by one SM pair, its K steps in order, wherever the schedule puts
it), at the layer's Dgrad + Wgrad shapes, on ragged shapes, with either
problem the costlier one, with MXFP4 operands, and with the FP32 add mode.
The single GEMM is itself checked against the oracle in test_gpu_20_gemm.py;
one small pair here is also compared with the oracle directly."""
import pytest
import torch

import oracle
import workloads
from nvfp4_testing import assert_gemm_close, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from quantize_block_scaled_amax_gb300 import build
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    assert torch.cuda.is_available()
    return nv


def _inputs(m, n, k, seed):
    a = workloads.normal_with_outliers(m, k, p=0.01, factor=30.0, seed=seed, dtype=torch.bfloat16)
    b = workloads.normal_with_outliers(n, k, p=0.01, factor=30.0, seed=seed + 1, dtype=torch.bfloat16)
    return a, b


def _operands(nv, m, n, k, seed, fmt="nvfp4"):
    a, b = _inputs(m, n, k, seed)
    block = "mx1x32" if fmt == "mxfp4" else "1x16"
    qa, _ = nv.nvfp4_quantize(a.cuda(), block=block)
    qb, _ = nv.nvfp4_quantize(b.cuda(), block=block)
    return qa, qb


def _pair_equals_singles(nv, shapes, dtypes, fmt="nvfp4", accumulate1=False):
    (m0, n0, k0), (m1, n1, k1) = shapes
    qa0, qb0 = _operands(nv, m0, n0, k0, 301, fmt)
    qa1, qb1 = _operands(nv, m1, n1, k1, 401, fmt)
    init1 = torch.randn(m1, n1, device="cuda", dtype=torch.float32) if accumulate1 else None
    c0 = torch.empty(m0, n0, dtype=dtypes[0], device="cuda")
    c1 = init1.clone() if accumulate1 else torch.empty(m1, n1, dtype=dtypes[1], device="cuda")
    s0 = torch.empty_like(c0)
    s1 = init1.clone() if accumulate1 else torch.empty_like(c1)
    for _ in range(2):   # twice: the pair must not depend on leftover state
        if accumulate1:
            c1.copy_(init1)
            s1.copy_(init1)
        nv.nvfp4_gemm_pair(qa0, qb0, c0, qa1, qb1, c1, accumulate1=accumulate1)
        nv.nvfp4_gemm(qa0, qb0, out=s0)
        nv.nvfp4_gemm(qa1, qb1, out=s1, accumulate=accumulate1)
        torch.cuda.synchronize()
        assert nv.nvfp4_sync_status() == nv.OK
        assert torch.equal(c0, s0), "problem 0 differs from its single GEMM"
        assert torch.equal(c1, s1), "problem 1 differs from its single GEMM"
    return qa0, qb0, c0, qa1, qb1, c1


def test_layer_dgrad_and_wgrad(nv):
    # Dgrad dX = dY W: 8192 x 5120 x 20480, bf16 out; Wgrad dW = dY^T X:
    # 20480 x 5120 x 8192, FP32 out
    _pair_equals_singles(nv, [(8192, 5120, 20480), (20480, 5120, 8192)], (torch.bfloat16, torch.float32))


def test_layer_wgrad_accumulates_into_fp32(nv):
    _pair_equals_singles(nv, [(8192, 5120, 20480), (20480, 5120, 8192)], (torch.bfloat16, torch.float32),
                         accumulate1=True)


@pytest.mark.parametrize("shapes", [
    [(300, 200, 128), (500, 260, 192)],          # fewer tiles than SM pairs in both
    [(1000, 704, 512), (2048, 4096, 256)],       # the second problem costlier per tile: swapped
    [(4096, 4864, 2048), (3072, 1536, 1024)],    # a partial last round in the first
    [(256, 256, 64), (19712, 256, 64)],          # one tile, then many
])
def test_ragged_pairs(nv, shapes):
    _pair_equals_singles(nv, shapes, (torch.bfloat16, torch.float32))


def test_mxfp4_pair(nv):
    _pair_equals_singles(nv, [(2048, 3072, 1024), (1024, 2048, 4096)], (torch.float32, torch.bfloat16), fmt="mxfp4")


def test_small_pair_against_the_oracle(nv):
    shapes = [(200, 136, 192), (136, 264, 320)]
    _, _, c0, _, _, c1 = _pair_equals_singles(nv, shapes, (torch.float32, torch.float32))
    for (m, n, k), seed, c in zip(shapes, (301, 401), (c0, c1)):
        a, b = _inputs(m, n, k, seed)
        ad = oracle.dequantize(oracle.quantize(to_f32_np(a)))
        bd = oracle.dequantize(oracle.quantize(to_f32_np(b)))
        assert_gemm_close(c.cpu().numpy(), ad @ bd.T, ad, bd, bf16=False, what=f"pair output {m}x{n}x{k}")


def test_mixed_formats_are_refused(nv):
    qa0, qb0 = _operands(nv, 256, 256, 128, 501)
    qa1, qb1 = _operands(nv, 256, 256, 128, 601, fmt="mxfp4")
    c0 = torch.empty(256, 256, dtype=torch.bfloat16, device="cuda")
    c1 = torch.empty_like(c0)
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_gemm_pair(qa0, qb0, c0, qa1, qb1, c1)

"""``torch.autograd`` wrapper of the NVFP4 linear layer Y = X W^T.

The forward and backward passes are the C ABI's ``nvfp4_linear_fwd`` and
``nvfp4_linear_bwd`` (through the binding): X 1x16 RTN, W 16x16 RTN in both
layouts, Y in bf16; dY 1x16 SR for Dgrad, and the 16-point RHT along the
tokens with SR on dY and RTN on X for Wgrad (paper page "Pretraining Large
Language Models with NVFP4", recipe paragraph; blog "NVFP4 Trains with
Precision of 16-Bit...", technique list).  Nothing here computes: the module
keeps the caller-side state the C calls need (quantized-operand buffers per
shape and device, and the random seeds).

Seeds: every backward pass draws a fresh stochastic-rounding seed from a
counter (``seed_base + call index``), so repeated steps do not reuse the
rounding decisions, and a run started from the same ``seed_base`` repeats
them exactly.  The RHT sign vector uses ``rht_seed`` (one per layer; both
Wgrad operands of a call share it, as the transform requires).

FP32 gradient accumulation: the recipe keeps gradient accumulation in FP32
(paper page, recipe paragraph).  With ``main_grad=True`` a layer adds each
backward's FP32 Wgrad result into ``weight.main_grad`` (an FP32 tensor of
the weight's shape, zeros when first created; the optimizer reads it and
zeroes it between steps) inside the Wgrad GEMM itself, and leaves
``weight.grad`` unset; otherwise ``weight.grad`` gets the Wgrad result cast
to the weight's dtype.

Saved state: the forward quantizes X twice from one read of it (1x16 RTN
for Fprop, and X^T after the RHT, RTN, for Wgrad: the C ABI's
``nvfp4_linear_fwd_rht``), and keeps only the Wgrad operand for the
backward, a fresh buffer per forward: 0.5625 bytes per element of X instead
of X's 2.  Several forwards may run before their backwards.

Precision: the paper page keeps some linear layers in BF16 (the last blocks
of the network) and switches the whole model to BF16 for the final part of
training to close the remaining loss gap.  A layer's ``precision`` is
"nvfp4" or "bf16"; "bf16" runs the same three GEMMs on bf16 operands with
the library's BF16 tensor-core GEMM (FP32 accumulation, bf16 results) and
its transpose kernel for the K-major operands of Dgrad and Wgrad.
``set_precision(model, "bf16")`` switches every such layer of a model at
once.
"""
from __future__ import annotations

import threading

import torch

from . import LinearContext, empty_qtensor, nvfp4_gemm_bf16, nvfp4_linear_bwd, nvfp4_linear_fwd, nvfp4_transpose_bf16

__all__ = ["NVFP4LinearFunction", "BF16LinearFunction", "NVFP4Linear", "nvfp4_linear", "set_precision"]

PRECISIONS = ("nvfp4", "bf16")


class _SeedCounter:
    def __init__(self, base: int):
        self._next = int(base)
        self._lock = threading.Lock()

    def take(self) -> int:
        with self._lock:
            s = self._next
            self._next += 1
            return s & 0xFFFFFFFFFFFFFFFF


class _Contexts:
    """Quantized-operand buffers, one set per (M, N, K, device)."""

    def __init__(self):
        self._ctx = {}
        self._lock = threading.Lock()

    def get(self, m: int, n: int, k: int, device) -> LinearContext:
        key = (m, n, k, str(device))
        with self._lock:
            c = self._ctx.get(key)
            if c is None:
                c = LinearContext(m, n, k, device)
                self._ctx[key] = c
            return c


def _check_shapes(x2: torch.Tensor, w: torch.Tensor) -> None:
    if x2.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise TypeError(f"NVFP4 linear takes bf16 X and W, got {x2.dtype} and {w.dtype}")
    if w.dim() != 2 or x2.shape[1] != w.shape[1]:
        raise ValueError(f"X [..., K] and W [N, K] disagree: {tuple(x2.shape)} vs {tuple(w.shape)}")
    m, k = x2.shape
    n = w.shape[0]
    if m % 64 or n % 64 or k % 64 or m == 0 or n == 0 or k == 0:
        raise ValueError(f"M, N, K must be positive multiples of 64, got M={m} N={n} K={k}")
    if not x2.is_cuda or not w.is_cuda or x2.device != w.device:
        raise ValueError("X and W must be CUDA tensors on the same device")


class NVFP4LinearFunction(torch.autograd.Function):
    """Y = X W^T with the NVFP4 recipe; X [..., K] bf16, W [N, K] bf16.

    Returns Y [..., N] bf16.  Gradients: dX bf16, dW in W's dtype (the Wgrad
    GEMM accumulates and writes FP32; the cast to bf16 is the one rounding
    this wrapper adds), or, when ``main_grad`` (an FP32 [N, K] tensor) is
    given, no dW: the Wgrad GEMM adds its FP32 result into ``main_grad``."""

    @staticmethod
    def forward(ctx, x, w, contexts: _Contexts, seeds: _SeedCounter, rht_seed: int, main_grad=None):
        lead = x.shape[:-1]
        x2 = x.reshape(-1, x.shape[-1]).contiguous()
        w = w.contiguous()
        _check_shapes(x2, w)
        m, k = x2.shape
        n = w.shape[0]
        lc = contexts.get(m, n, k, x2.device)
        # this forward's X^T codes, kept for its own backward
        lc.xtq = empty_qtensor(k, m, x2.device)
        y = nvfp4_linear_fwd(x2, w, lc, rht_seed=rht_seed)
        ctx.xtq = lc.xtq
        ctx.lc = lc
        ctx.lead = lead
        ctx.seeds = seeds
        ctx.rht_seed = rht_seed
        ctx.w_dtype = w.dtype
        ctx.main_grad = main_grad
        return y.reshape(*lead, n)

    @staticmethod
    def backward(ctx, dy):
        lc = ctx.lc
        dy2 = dy.reshape(-1, dy.shape[-1]).to(torch.bfloat16).contiguous()
        # Dgrad reads lc.wtq, which every forward of this layer writes from
        # the same W; Wgrad reads this forward's own X^T codes
        lc.xtq = ctx.xtq
        if ctx.main_grad is not None:
            dx, _ = nvfp4_linear_bwd(dy2, None, lc, sr_seed=ctx.seeds.take(), rht_seed=ctx.rht_seed,
                                     dW=ctx.main_grad, accumulate_dw=True)
            return dx.reshape(*ctx.lead, lc.K), None, None, None, None, None
        dx, dw = nvfp4_linear_bwd(dy2, None, lc, sr_seed=ctx.seeds.take(), rht_seed=ctx.rht_seed)
        return dx.reshape(*ctx.lead, lc.K), dw.to(ctx.w_dtype), None, None, None, None


class BF16LinearFunction(torch.autograd.Function):
    """Y = X W^T with bf16 operands on the tensor cores (FP32 accumulation):
    the layers the recipe keeps in high precision.  X [..., K] bf16, W [N, K]
    bf16; Y, dX and dW are bf16.  M, N, K must be multiples of 8."""

    @staticmethod
    def forward(ctx, x, w, main_grad=None):
        lead = x.shape[:-1]
        x2 = x.reshape(-1, x.shape[-1]).contiguous()
        w = w.contiguous()
        if x2.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
            raise TypeError(f"BF16 linear takes bf16 X and W, got {x2.dtype} and {w.dtype}")
        if w.dim() != 2 or x2.shape[1] != w.shape[1]:
            raise ValueError(f"X [..., K] and W [N, K] disagree: {tuple(x2.shape)} vs {tuple(w.shape)}")
        if x2.shape[0] % 8 or w.shape[0] % 8 or w.shape[1] % 8:
            raise ValueError(f"M, N, K must be multiples of 8, got {x2.shape[0]}, {w.shape[0]}, {w.shape[1]}")
        y = nvfp4_gemm_bf16(x2, w)                          # [M][N] = X W^T
        ctx.save_for_backward(x2, w)
        ctx.lead = lead
        ctx.main_grad = main_grad
        return y.reshape(*lead, w.shape[0])

    @staticmethod
    def backward(ctx, dy):
        x2, w = ctx.saved_tensors
        dy2 = dy.reshape(-1, w.shape[0]).to(torch.bfloat16).contiguous()
        dx = nvfp4_gemm_bf16(dy2, nvfp4_transpose_bf16(w))  # [M][K] = dY W
        if ctx.main_grad is not None:                      # main_grad += dY^T X, FP32
            nvfp4_gemm_bf16(nvfp4_transpose_bf16(dy2), nvfp4_transpose_bf16(x2), out=ctx.main_grad, accumulate=True)
            return dx.reshape(*ctx.lead, w.shape[1]), None, None
        dw = nvfp4_gemm_bf16(nvfp4_transpose_bf16(dy2), nvfp4_transpose_bf16(x2))  # [N][K] = dY^T X
        return dx.reshape(*ctx.lead, w.shape[1]), dw, None


class NVFP4Linear(torch.nn.Module):
    """A bias-free linear layer whose three GEMMs run in NVFP4 on the tcgen05
    tensor cores.  ``weight`` is a bf16 parameter [out_features, in_features]
    (the high-precision master copy stays with the optimizer, as in the
    recipe); in_features, out_features and the token count must be multiples
    of 64.  ``main_grad=True``: the Wgrad result is accumulated in FP32 into
    ``weight.main_grad`` instead of being returned as ``weight.grad``."""

    def __init__(self, in_features: int, out_features: int, device=None, seed_base: int = 1, rht_seed: int = 2,
                 precision: str = "nvfp4", main_grad: bool = False):
        super().__init__()
        if in_features % 64 or out_features % 64:
            raise ValueError("in_features and out_features must be multiples of 64")
        if precision not in PRECISIONS:
            raise ValueError(f"precision must be one of {PRECISIONS}, got {precision!r}")
        self.precision = precision
        self.weight = torch.nn.Parameter(torch.empty(out_features, in_features, dtype=torch.bfloat16, device=device))
        torch.nn.init.normal_(self.weight, std=0.02)
        self._contexts = _Contexts()
        self._seeds = _SeedCounter(seed_base)
        self.rht_seed = int(rht_seed)
        self.use_main_grad = bool(main_grad)

    def _main_grad(self):
        if not self.use_main_grad:
            return None
        g = getattr(self.weight, "main_grad", None)
        if g is None or g.shape != self.weight.shape or g.device != self.weight.device:
            g = torch.zeros(self.weight.shape, dtype=torch.float32, device=self.weight.device)
            self.weight.main_grad = g
        return g

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if self.precision == "bf16":
            return BF16LinearFunction.apply(x, self.weight, self._main_grad())
        return NVFP4LinearFunction.apply(x, self.weight, self._contexts, self._seeds, self.rht_seed,
                                         self._main_grad())

    def extra_repr(self) -> str:
        return (f"in_features={self.weight.shape[1]}, out_features={self.weight.shape[0]}, precision={self.precision}, "
                f"main_grad={self.use_main_grad}")


def set_precision(module: torch.nn.Module, precision: str) -> int:
    """Set ``precision`` ("nvfp4" or "bf16") on every NVFP4Linear in
    ``module`` (itself included), e.g. for the switch to BF16 near the end of
    training; returns how many layers were set."""
    if precision not in PRECISIONS:
        raise ValueError(f"precision must be one of {PRECISIONS}, got {precision!r}")
    n = 0
    for m in module.modules():
        if isinstance(m, NVFP4Linear):
            m.precision = precision
            n += 1
    return n


def nvfp4_linear(x: torch.Tensor, w: torch.Tensor, sr_seed: int = 1, rht_seed: int = 2) -> torch.Tensor:
    """Functional form with a fixed stochastic-rounding seed (every backward
    of this call uses ``sr_seed``)."""
    return NVFP4LinearFunction.apply(x, w, _Contexts(), _SeedCounter(sr_seed), int(rht_seed))

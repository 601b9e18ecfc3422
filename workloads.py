"""Seeded synthetic inputs shaped like the linear layers of the 12B hybrid
Mamba-Transformer of "Pretraining Large Language Models with NVFP4" (model
paragraph: sequence length 8192), with the value distributions of the
workloads this library is checked and measured on.

This module holds no NVFP4 arithmetic.  It only draws random tensors; both
the CUDA path and the oracle consume the same bits (bf16 values are passed to
the oracle exactly, as float32).

Recipes (all draws from one ``torch.Generator`` per tensor):

* ``normal_with_outliers``: N(0, std), then a Bernoulli(p) mask of entries
  multiplied by ``factor`` (activations with outliers).
* ``student_t``: Student-t(nu) * scale, as Z / sqrt(chi2_nu / nu) with chi2_nu
  a sum of nu squared standard normals (heavy-tailed gradients: many block
  maxima far below the tensor max, so many E4M3 block scales are subnormal).
* every tensor is drawn in float32 and then cast to bf16 (round to nearest
  even) when a bf16 workload is asked for.

Seeds: tensor j of a workload uses seed 0x1000 + j; stochastic-rounding seed 1;
RHT seed 2.
"""
from __future__ import annotations

import torch

SEED_BASE = 0x1000
SR_SEED = 1
RHT_SEED = 2

# layer dims of the 12B model's FFN (hidden 5120, FFN 20480) at seq 8192
M_TOKENS = 8192
D_MODEL = 5120
D_FFN = 20480


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_with_outliers(rows: int, cols: int, *, std: float = 1.0, p: float = 0.0, factor: float = 1.0,
                         seed: int = SEED_BASE, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if p > 0.0:
        mask = torch.rand(rows, cols, generator=g, device=device) < p
        x = torch.where(mask, x * factor, x)
    return x.to(dtype)


def student_t(rows: int, cols: int, *, nu: int = 3, scale: float = 1e-3, seed: int = SEED_BASE,
              device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    g = _gen(seed, device)
    z = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(rows, cols, device=device, dtype=torch.float32)
    for _ in range(nu):
        n = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
        chi2.addcmul_(n, n)
    t = z / torch.sqrt(chi2 / nu)
    return (t * scale).to(dtype)


# ---- the named workloads -------------------------------------------------

def tiny(device="cpu"):
    """A fp32 128x256 and B fp32 256x256, N(0,1) with 0.5% of entries x40."""
    a = normal_with_outliers(128, 256, p=0.005, factor=40.0, seed=SEED_BASE + 0, device=device,
                             dtype=torch.float32)
    b = normal_with_outliers(256, 256, p=0.005, factor=40.0, seed=SEED_BASE + 1, device=device,
                             dtype=torch.float32)
    return a, b


def activations(rows: int = M_TOKENS, cols: int = D_MODEL, *, outliers: bool = True, seed: int = SEED_BASE + 0,
                device="cpu", dtype=torch.bfloat16):
    """X bf16 N(0,1); with outliers, 0.1% of entries x50 (amax ~ 250)."""
    if outliers:
        return normal_with_outliers(rows, cols, p=0.001, factor=50.0, seed=seed, device=device, dtype=dtype)
    return normal_with_outliers(rows, cols, seed=seed, device=device, dtype=dtype)


def weights(rows: int = D_FFN, cols: int = D_MODEL, *, seed: int = SEED_BASE + 1, device="cpu",
            dtype=torch.bfloat16):
    """W bf16 N(0, 0.02)."""
    return normal_with_outliers(rows, cols, std=0.02, seed=seed, device=device, dtype=dtype)


def gradients(rows: int = M_TOKENS, cols: int = D_FFN, *, seed: int = SEED_BASE + 2, device="cpu",
              dtype=torch.bfloat16):
    """dY bf16 Student-t(nu=3) * 1e-3."""
    return student_t(rows, cols, nu=3, scale=1e-3, seed=seed, device=device, dtype=dtype)


def linear_layer(m: int = M_TOKENS, n: int = D_FFN, k: int = D_MODEL, device="cpu"):
    """One linear layer's fwd+bwd inputs: X [m][k] (outliers), W [n][k], dY [m][n]."""
    x = activations(m, k, device=device)
    w = weights(n, k, device=device)
    dy = gradients(m, n, device=device)
    return x, w, dy

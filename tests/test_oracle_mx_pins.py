"""Pins of the oracle's MXFP4 variant (paper summary page, format
paragraph; explainer page, comparison paragraph: 32-element blocks, one
power-of-two UE8M0 scale, no tensor scale, at worst the +-4 and +-6 levels
unused).  Each check compares against something other than the oracle's own
code: IEEE bit layouts, hand-worked cases, the pages' stated worst case, and
brute force over the E2M1 grid."""
from fractions import Fraction

import numpy as np
import pytest

import oracle

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e8m0_decode_matches_ieee_exponent_field():
    # a float32 with exponent field b and zero mantissa is 2^(b-127) (b >= 1);
    # b = 0 is the subnormal 2^-127 = mantissa bit 22
    for b in range(1, 255):
        ieee = np.array([b << 23], dtype=np.uint32).view(np.float32)[0]
        assert oracle.e8m0_decode(b) == float(ieee)
    assert oracle.e8m0_decode(0) == float(np.array([1 << 22], dtype=np.uint32).view(np.float32)[0])
    assert np.isnan(oracle.e8m0_decode(255))


@pytest.mark.parametrize("bamax, e", [
    (6.0, 0),                        # 6 * 2^0 = 6 covers it exactly
    (float(np.nextafter(np.float32(6.0), np.float32(7.0))), 1),
    (1.0, -2),                       # 6 / 4 = 1.5 >= 1 > 0.75
    (0.75, -3),                      # 6 / 8 = 0.75
    (3.0, -1),                       # the block max lands exactly on 6
    (float(np.nextafter(np.float32(3.0), np.float32(4.0))), 0),   # just above 3: 4 and 6 go unused
    (250.0, 6),                      # 6 * 64 = 384 >= 250 > 192
    (1e-40, -127),                   # below the UE8M0 range: clamped
])
def test_mx_block_scale_worked_examples(bamax, e):
    assert oracle.mx_block_scale(bamax) == e + 127


def test_mx_block_scale_is_the_smallest_covering_power_of_two():
    rng = np.random.default_rng(7)
    vals = np.concatenate([np.float32(2.0) ** rng.integers(-120, 120, 2000).astype(np.float32) *
                           rng.uniform(0.5, 1.0, 2000).astype(np.float32),
                           rng.uniform(0, 10, 2000).astype(np.float32)])
    for a in vals.astype(np.float32):
        a = Fraction(float(a))
        if a == 0:
            continue
        e = oracle.mx_block_scale(float(a)) - 127
        assert 6 * Fraction(2) ** e >= a
        assert e == -127 or 6 * Fraction(2) ** (e - 1) < a
        if e > -127:
            # the pages' worst case: the scaled block max stays above 3
            assert Fraction(3) < a / Fraction(2) ** e <= 6


def _nearest_even_grid(v: Fraction) -> Fraction:
    # brute force over the signed grid; ties to the value whose magnitude has
    # an even code (0, 1, 2, 4 are the even-mantissa points)
    cands = sorted({Fraction(s) * Fraction(g) for g in GRID for s in (1, -1)})
    best = min(abs(c - v) for c in cands)
    ties = [c for c in cands if abs(c - v) == best]
    if len(ties) == 1:
        return ties[0]
    even = [c for c in ties if GRID.index(float(abs(c))) % 2 == 0]
    return even[0]


def test_mx_quantize_rtn_is_nearest_grid_point_times_block_scale():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((4, 64)) * np.float32(2.0) ** rng.integers(-3, 4, (4, 1))).astype(np.float32)
    x[1, 5] = 0.0
    x[2, :32] = 0.0                  # an all-zero block
    q = oracle.quantize(x, block="mx1x32")
    assert q["s_dec"] == 1.0 and q["scales"].shape == (4, 2)
    xd = oracle.dequantize(q)
    for r in range(4):
        for b in range(2):
            blk = x[r, 32 * b:32 * b + 32]
            sb = int(q["scales"][r, b])
            if not np.any(blk):
                assert sb == 0 and not np.any(xd[r, 32 * b:32 * b + 32])
                continue
            scale = Fraction(2) ** (sb - 127)
            for c in range(32):
                want = _nearest_even_grid(Fraction(float(blk[c])) / scale) * scale
                assert Fraction(xd[r, 32 * b + c]) == want


def test_mx_representable_values_round_trip():
    # every value code * 2^e with the block max on the top binade comes back exactly
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 16, (3, 96))
    vals = np.array([[(-1.0 if c & 8 else 1.0) * GRID[c & 7] for c in row] for row in codes], dtype=np.float64)
    vals[:, ::32] = 6.0              # pin each block's max at 6 * 2^e
    e = rng.integers(-20, 20, (3, 3))
    x = (vals * np.repeat(2.0 ** e, 32, axis=1)).astype(np.float32)
    xd = oracle.dequantize(oracle.quantize(x, block="mx1x32"))
    assert np.array_equal(xd, x.astype(np.float64))


def test_mx_gemm_against_exact_brute_force():
    rng = np.random.default_rng(11)
    a = rng.standard_normal((3, 64)).astype(np.float32)
    b = (rng.standard_normal((2, 64)) * 30).astype(np.float32)
    qa, qb = oracle.quantize(a, block="mx1x32"), oracle.quantize(b, block="mx1x32")
    c = oracle.gemm(qa, qb)
    ad, bd = oracle.dequantize(qa), oracle.dequantize(qb)
    for i in range(3):
        for j in range(2):
            exact = sum(Fraction(ad[i, k]) * Fraction(bd[j, k]) for k in range(64))
            assert Fraction(c[i, j]) == exact


def test_mx_needs_blocks_of_32():
    with pytest.raises(oracle.OracleError):
        oracle.quantize(np.zeros((2, 48), dtype=np.float32), block="mx1x32")


def test_bf16_gemm_against_exact_brute_force():
    import torch
    g = torch.Generator().manual_seed(2)
    a = (torch.randn(4, 48, generator=g) * 3).bfloat16().float().numpy()
    b = torch.randn(3, 48, generator=g).bfloat16().float().numpy()
    c = oracle.bf16_gemm(a, b)
    for i in range(4):
        for j in range(3):
            assert Fraction(c[i, j]) == sum(Fraction(float(a[i, k])) * Fraction(float(b[j, k])) for k in range(48))
    with pytest.raises(ValueError):
        oracle.bf16_gemm(np.full((1, 16), 1.0 + 2.0 ** -20, np.float32), np.ones((1, 16), np.float32))

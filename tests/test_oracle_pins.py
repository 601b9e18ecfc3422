"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the oracle against the pages' printed facts, a library
routine that implements the same standard format independently (torch's
float8_e4m3fn, scipy's Hadamard matrix), a closed form, an invariant, a
hand-derived example or brute force -- never against a retyping of the
oracle's own formula.  No GPU is needed.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ---- E2M1 -----------------------------------------------------------------

def test_e2m1_decode_matches_page_grid():
    _, rows = read_golden("e2m1_grid.txt")
    assert len(rows) == 16
    for code_hex, value in rows:
        code = int(code_hex, 16)
        got = oracle.e2m1_decode(code)
        assert got == float(value)
        assert np.signbit(got) == (code >= 8)


def _brute_nearest_e2m1(v: np.ndarray) -> np.ndarray:
    """Brute force: nearest of the 8 magnitudes (after saturating at 6); on a
    tie take the point with the even mantissa bit (the even code)."""
    a = np.minimum(np.abs(v.astype(np.float64)), 6.0)
    grid = np.array(E2M1_GRID)
    d = np.abs(a[:, None] - grid[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among tied candidates prefer the even code index
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    return (pick | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def _neighbour_values():
    pts = np.array(E2M1_GRID, dtype=np.float32)
    mids = ((pts[1:].astype(np.float64) + pts[:-1]) / 2).astype(np.float32)
    base = np.concatenate([pts, mids, np.array([6.5, 7.0, 8.0, 1e30, np.inf], dtype=np.float32)])
    vals = [base, np.nextafter(base, np.float32(np.inf)), np.nextafter(base, np.float32(-np.inf))]
    v = np.concatenate(vals)
    v = v[v >= 0]
    return np.concatenate([v, -v])


def test_e2m1_rtn_every_neighbour_pair():
    v = _neighbour_values()
    got = oracle.e2m1_encode_rtn_array(v)
    np.testing.assert_array_equal(got, _brute_nearest_e2m1(v))


def test_e2m1_rtn_ties_go_to_even_mantissa():
    # the midpoints between grid points, by hand
    expect = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, code in expect.items():
        assert oracle.e2m1_encode_rtn(v) == code
        assert oracle.e2m1_encode_rtn(-v) == code | 8


def test_e2m1_rtn_sweep_against_brute_force():
    # every 61st float32 bit pattern in [0, 8] (~18M values) and some negations
    hi = np.float32(8.0).view(np.uint32)
    bits = np.arange(0, int(hi) + 1, 61, dtype=np.uint32)
    v = bits.view(np.float32)
    for chunk in np.array_split(v, 16):
        np.testing.assert_array_equal(oracle.e2m1_encode_rtn_array(chunk), _brute_nearest_e2m1(chunk))
    neg = -v[::7]
    np.testing.assert_array_equal(oracle.e2m1_encode_rtn_array(neg), _brute_nearest_e2m1(neg))


def test_e2m1_rtn_saturates_and_keeps_sign_of_zero():
    assert oracle.e2m1_encode_rtn(1e30) == 7
    assert oracle.e2m1_encode_rtn(float("inf")) == 7
    assert oracle.e2m1_encode_rtn(-7.0) == 0xF
    assert oracle.e2m1_encode_rtn(-0.0) == 8
    assert oracle.e2m1_encode_rtn(-0.1) == 8
    assert oracle.e2m1_encode_rtn(0.1) == 0


# ---- E4M3 -----------------------------------------------------------------

def test_e4m3_decode_all_codes_against_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if np.isnan(ref[c]):
            assert np.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_against_torch_round_to_nearest_even():
    # every 997th float32 bit pattern in [0, 448] plus every E4M3 value, every
    # midpoint and the floats on either side of each midpoint
    hi = np.float32(448.0).view(np.uint32)
    bits = np.arange(0, int(hi) + 1, 997, dtype=np.uint32)
    v = bits.view(np.float32)
    e4 = np.array([oracle.e4m3_decode(c) for c in range(0x7F)], dtype=np.float64)
    mids = ((e4[1:] + e4[:-1]) / 2).astype(np.float32)
    extra = np.concatenate([e4.astype(np.float32), mids, np.nextafter(mids, np.float32(0)),
                            np.nextafter(mids, np.float32(np.inf))])
    v = np.concatenate([v, extra[(extra >= 0) & (extra <= 448)]])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode_array(v)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_saturates():
    for v in [448.0, 449.0, 464.0, 479.0, 480.0, 1e6, 3.4e38]:
        assert oracle.e4m3_encode(v) == 0x7E
    assert oracle.e4m3_encode(0.0) == 0
    assert oracle.e4m3_encode(2.0 ** -10) == 0          # tie between 0 and 2^-9 -> even (0)
    assert oracle.e4m3_encode(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 1


# ---- Philox ---------------------------------------------------------------

def test_philox_known_answer_vectors():
    _, rows = read_golden("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        vals = [int(x, 16) for x in r]
        assert oracle.philox4x32_10(vals[0:4], vals[4:6]) == vals[6:10]


def test_sr_bits_counter_mapping():
    # elements 8j..8j+7 share the block with counter (j low, j high, 0, 0);
    # element i takes 16-bit half i%8 of it (low half of each word first),
    # returned in the top half of the word
    kat0 = [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]    # seed 0, counter 0
    halves = [0xE8D5, 0x6627, 0xC58D, 0xE169, 0xAC4C, 0xBC57, 0xDBD8, 0x9B00]
    assert [oracle.sr_bits(0, i) for i in range(8)] == [h << 16 for h in halves]
    assert [oracle.sr_bits(0, i) >> 16 for i in range(8)] == [
        (kat0[k >> 1] >> (16 * (k & 1))) & 0xFFFF for k in range(8)]
    i = (1 << 35) + 13
    w = oracle.philox4x32_10([(i >> 3) & 0xFFFFFFFF, i >> 35, 0, 0], [7, 0])
    assert oracle.sr_bits(7, i) == (w[2] >> 16) << 16


# ---- tensor and block scales ----------------------------------------------

@pytest.mark.parametrize("amax", [250.0, 1.0, 2688.0, 0.0302734375, 3.0e4, 1e-30, 1e-41])
def test_tensor_scales_closed_form(amax):
    s_dec, s_enc = oracle.tensor_scales(amax)
    # S_dec * 2688 = A and S_enc * A = 2688, each to within one FP32 rounding
    # (an S_dec in the FP32 subnormal range has the subnormal spacing 2^-149;
    # an S_enc beyond the FP32 range saturates to the largest float)
    amax = float(np.float32(amax))
    assert abs(s_dec * 2688.0 - amax) <= max(amax * 2.0 ** -23, 2688.0 * 2.0 ** -149)
    if 2688.0 / amax < float(np.finfo(np.float32).max):
        assert abs(s_enc * amax - 2688.0) <= 2688.0 * 2.0 ** -23
    else:
        assert s_enc == float(np.finfo(np.float32).max)


def test_tensor_scales_degenerate():
    assert oracle.tensor_scales(0.0) == (1.0, 1.0)
    # 2688 / 1e-40 overflows FP32: S_enc saturates to the largest finite float
    _, s_enc = oracle.tensor_scales(1e-40)
    assert s_enc == np.finfo(np.float32).max


def test_block_max_recoverable_near_fp8_precision():
    # format paragraph: the block max is recovered at near-FP8 precision,
    # i.e. within the E4M3 relative rounding error 2^-4 for normal scales.
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 512)) * np.exp(rng.uniform(-6, 6, (64, 1)))).astype(np.float32)
    q = oracle.quantize(x)
    deq = oracle.dequantize(q)
    xb = np.abs(x.astype(np.float64)).reshape(64, 32, 16)
    db = np.abs(deq).reshape(64, 32, 16)
    bamax = xb.max(axis=2)
    recovered = db.max(axis=2)
    # sb >= 0x09 (1.125 * 2^-6) implies the unrounded scale was a normal E4M3
    # value; 0x08 itself can be a subnormal-range scale rounded up.
    normal = q["scales"] >= 0x09
    assert normal.sum() > 1500
    rel = np.abs(recovered - bamax)[normal] / bamax[normal]
    assert rel.max() <= 2.0 ** -4


# ---- quantizer worked examples ----------------------------------------------

def test_worked_example_rtn():
    kv, _ = read_golden("worked_example_rtn.txt")
    x = np.array([float(v) for v in kv["x"]], dtype=np.float32).reshape(1, 32)
    q = oracle.quantize(x)
    assert q["codes"].reshape(-1).tolist() == [int(b, 16) for b in kv["packed_bytes"]]
    assert q["scales"].reshape(-1).tolist() == [int(b, 16) for b in kv["scales"]]
    assert q["amax"] == float(kv["amax"][0])
    assert q["s_dec"] == float(kv["s_dec"][0]) and q["s_enc"] == float(kv["s_enc"][0])
    # element codes unpacked, low nibble first
    codes = q["codes"].reshape(-1)
    unpacked = np.stack([codes & 0xF, codes >> 4], axis=1).reshape(-1)
    assert unpacked.tolist() == [int(c, 16) for c in kv["codes_per_element"]]


def test_worked_example_sr():
    kv, _ = read_golden("worked_example_sr.txt")
    x = np.array([float(v) for v in kv["x"]], dtype=np.float32).reshape(1, 32)
    q = oracle.quantize(x, rounding="sr", seed=int(kv["seed"][0]))
    codes = q["codes"].reshape(-1)
    unpacked = np.stack([codes & 0xF, codes >> 4], axis=1).reshape(-1)
    assert unpacked[:4].tolist() == [int(c, 16) for c in kv["codes_first4"]]


def test_exactly_representable_values_round_trip():
    # x = grid value * block scale * S_dec for a chosen scale per block: both
    # RTN and SR must return x exactly (no rounding happens).
    rng = np.random.default_rng(1)
    rows, cols = 8, 64
    grid = np.array(E2M1_GRID + [-g for g in E2M1_GRID[1:]], dtype=np.float64)
    vals = rng.choice(grid, size=(rows, cols))
    vals.reshape(rows, cols // 16, 16)[:, :, 0] = 6.0          # every block reaches 6
    bscale = 2.0 ** rng.integers(-3, 4, size=(rows, cols // 16, 1))
    x = (vals.reshape(rows, cols // 16, 16) * bscale).reshape(rows, cols)
    # first block holds only the tensor amax 2688, so S_enc = S_dec = 1; a
    # block with bamax = 6 * 2^j then gets sb = 2^j exactly and r = 2^-j, and
    # 2688 * fl32(1/448) rounds to exactly 6.
    x[0, :16] = 0.0
    x[0, 0] = 2688.0
    x = x.astype(np.float32)
    for rounding in ("rtn", "sr"):
        q = oracle.quantize(x, rounding=rounding, seed=3)
        np.testing.assert_array_equal(oracle.dequantize(q), x.astype(np.float64))


def test_zero_tensor_and_nonfinite():
    q = oracle.quantize(np.zeros((4, 32), dtype=np.float32))
    assert q["amax"] == 0.0 and q["s_dec"] == 1.0 and q["s_enc"] == 1.0
    assert not q["codes"].any() and not q["scales"].any()
    bad = np.ones((2, 32), dtype=np.float32)
    bad[1, 5] = np.nan
    with pytest.raises(oracle.OracleError):
        oracle.quantize(bad)
    bad[1, 5] = np.inf
    with pytest.raises(oracle.OracleError):
        oracle.quantize(bad)


def test_negative_values_rounding_to_zero_keep_sign_bit():
    x = np.zeros((1, 16), dtype=np.float32)
    x[0, 0] = 6.0
    x[0, 1] = -0.2          # |v| < 0.25 -> magnitude 0, sign kept
    x[0, 2] = -0.0
    q = oracle.quantize(x)
    c = q["codes"].reshape(-1)
    assert (c[0] & 0xF) == 7 and (c[0] >> 4) == 8 and (c[1] & 0xF) == 8


def test_tiny_tensor_saturated_scales_stay_finite():
    # amax ~ 1e-39: S_enc saturates; codes must still decode near the input
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :16] = np.float32(1e-39) * np.arange(1, 17, dtype=np.float32) / 16
    x[0, 16:] = -np.float32(3e-40)
    q = oracle.quantize(x)
    assert q["s_enc"] == np.finfo(np.float32).max
    assert np.all(q["scales"] > 0)
    c = q["codes"].reshape(-1)
    assert np.all((c[8:] & 0x8) == 0x8) and np.all((c[8:] >> 4) >= 8)  # negatives keep sign


# ---- stochastic rounding -----------------------------------------------------

@pytest.mark.parametrize("v", [0.1, 0.3, 0.75, 1.2, 2.2, 3.7, 5.0, 5.9, -2.7, -0.05])
def test_sr_unbiased_over_a_million_draws(v):
    # blocks of [6, v x 15] with A = 2688: sb = 1, r = 1, so element value = v
    nblk = 70000
    x = np.full((nblk, 16), np.float32(v), dtype=np.float32)
    x[:, 0] = 6.0
    x = x.reshape(1, -1)
    x = np.concatenate([x, np.zeros((1, 16), np.float32)], axis=1)
    x[0, -1] = 2688.0
    q = oracle.quantize(x, rounding="sr", seed=11)
    deq = oracle.dequantize(q).reshape(-1)[:-16].reshape(nblk, 16)[:, 1:]
    vv = float(np.float32(v))
    n = deq.size
    assert n >= 10 ** 6
    a = abs(vv)
    lo = max(g for g in E2M1_GRID if g <= a)
    hi = min(g for g in E2M1_GRID if g > a)
    frac = (a - lo) / (hi - lo)
    sigma = (hi - lo) * np.sqrt(frac * (1 - frac) / n)
    err = deq.mean() - vv
    assert abs(err) <= 4 * sigma + 1e-12
    # empirical probability of rounding up
    p_up = np.mean(np.abs(deq) == hi)
    # (16-bit random values: P(up) = ceil(frac * 2^16) / 2^16)
    assert abs(p_up - frac) <= 4 * np.sqrt(frac * (1 - frac) / n) + 2.0 ** -16


def test_sr_extreme_random_words():
    # u = 0 rounds up whenever frac > 0; u = 2^24 - 1 rounds down unless frac
    # exceeds 1 - 2^-24; grid points never move.
    for v in [0.26, 1.01, 2.5, 4.1, 5.99]:
        up = oracle.e2m1_encode_sr(v, 0)
        down = oracle.e2m1_encode_sr(v, 0xFFFFFFFF)
        a = float(np.float32(v))
        lo = max(g for g in E2M1_GRID if g <= a)
        hi = min(g for g in E2M1_GRID if g > a)
        assert oracle.e2m1_decode(up) == hi and oracle.e2m1_decode(down) == lo
    for g in E2M1_GRID:
        for rb in (0, 0x12345678, 0xFFFFFFFF):
            assert oracle.e2m1_decode(oracle.e2m1_encode_sr(g, rb)) == g


# ---- random Hadamard transform -----------------------------------------------

def test_rht_butterfly_is_sylvester_hadamard():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(16).astype(np.float64)   # Sylvester construction
    ones = np.ones(16, dtype=np.float32)
    cols = []
    for j in range(16):
        e = np.zeros(16, dtype=np.float32)
        e[j] = 4.0
        cols.append(oracle.rht16(e, ones))
    Hb = np.stack(cols, axis=1).astype(np.float64)
    np.testing.assert_array_equal(Hb, H)
    np.testing.assert_array_equal(H @ H.T, 16 * np.eye(16))


def test_rht_matches_dense_product_on_exact_inputs():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(16).astype(np.float64)
    rng = np.random.default_rng(2)
    d = oracle.rht16_signs(2)
    for _ in range(50):
        x = rng.integers(-64, 65, size=16).astype(np.float32)
        y = oracle.rht16(x, d)
        np.testing.assert_array_equal(y.astype(np.float64), 0.25 * H @ (d.astype(np.float64) * x))


def test_rht_is_an_involution_without_signs():
    rng = np.random.default_rng(3)
    ones = np.ones(16, dtype=np.float32)
    for _ in range(50):
        x = rng.integers(-1000, 1001, size=16).astype(np.float32)
        np.testing.assert_array_equal(oracle.rht16(oracle.rht16(x, ones), ones), x)


def test_rht_signs_come_from_philox_stream_one():
    w = oracle.philox4x32_10([0, 0, 1, 0], [2, 0])[0]
    d = oracle.rht16_signs(2)
    assert d.tolist() == [(-1.0 if (w >> j) & 1 else 1.0) for j in range(16)]
    assert set(d.tolist()) <= {-1.0, 1.0}


def test_rht_is_transparent_to_the_gemm():
    # (Q A)^T (Q B) = A^T B when both operands get the same transform along
    # the shared (token) dimension: Q = blockdiag(H16 D / 4) is orthogonal.
    rng = np.random.default_rng(4)
    a = rng.standard_normal((64, 8)).astype(np.float32)     # [tokens][n]
    b = rng.standard_normal((64, 5)).astype(np.float32)     # [tokens][k]
    qa = oracle.rht_rows(np.ascontiguousarray(a.T), 2)      # rows = n, along tokens
    qb = oracle.rht_rows(np.ascontiguousarray(b.T), 2)
    lhs = qa.astype(np.float64) @ qb.astype(np.float64).T
    rhs = a.T.astype(np.float64) @ b.astype(np.float64)
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=64 * 8 * 2.0 ** -23)


# ---- 2D blocks, layouts ------------------------------------------------------

def _unpack(codes):
    return np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(codes.shape[0], -1)


def test_2d_blocks_share_one_scale_and_transpose_consistently():
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((48, 64)) * 0.02).astype(np.float32)
    qw = oracle.quantize(w, block="16x16")
    qwt = oracle.quantize(w, layout="col", block="16x16")
    assert qw["scales"].shape == (3, 4) and qwt["scales"].shape == (4, 3)
    np.testing.assert_array_equal(qw["scales"], qwt["scales"].T)
    np.testing.assert_array_equal(_unpack(qw["codes"]), _unpack(qwt["codes"]).T)
    # every scale equals the 1x16 rule applied to the 16x16 tile's amax
    _, s_enc = oracle.tensor_scales(float(np.abs(w).max()))
    for i in range(3):
        for j in range(4):
            tile = np.abs(w[16 * i:16 * i + 16, 16 * j:16 * j + 16]).max()
            assert qw["scales"][i, j] == oracle.block_scale(float(tile), s_enc)


def test_colwise_is_rowwise_of_the_transpose():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((32, 48)).astype(np.float32)
    qc = oracle.quantize(x, layout="col", rounding="sr", seed=9)
    qr = oracle.quantize(np.ascontiguousarray(x.T), layout="row", rounding="sr", seed=9)
    np.testing.assert_array_equal(qc["codes"], qr["codes"])
    np.testing.assert_array_equal(qc["scales"], qr["scales"])


def test_row_sample_matches_full_quantization():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((64, 64)).astype(np.float32)
    full = oracle.quantize(x, rounding="sr", seed=5, block="16x16")
    part = oracle.quantize(x, rounding="sr", seed=5, block="16x16", rows=(16, 48))
    np.testing.assert_array_equal(part["codes"], full["codes"][16:48])
    np.testing.assert_array_equal(part["scales"], full["scales"][1:3])


# ---- GEMM ----------------------------------------------------------------------

def test_gemm_against_exact_rational_brute_force():
    # C[m,n] = S_dec,A S_dec,B sum_b sbA sbB sum_16 qA qB, computed in exact
    # rationals from the codes and scales, with the page grid for E2M1 and
    # torch's E4M3 decode for the scales.
    rng = np.random.default_rng(9)
    a = rng.standard_normal((3, 48)).astype(np.float32) * 3
    b = rng.standard_normal((5, 48)).astype(np.float32)
    qa, qb = oracle.quantize(a), oracle.quantize(b, rounding="sr", seed=4)
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    _, rows = read_golden("e2m1_grid.txt")
    e2 = {int(c, 16): Fraction(v) for c, v in rows}

    def q_at(q, r, k):
        byte = int(q["codes"][r, k // 2])
        return e2[(byte >> 4) if k % 2 else (byte & 0xF)]

    got = oracle.gemm(qa, qb)
    for m in range(3):
        for n in range(5):
            acc = Fraction(0)
            for blk in range(3):
                inner = sum(q_at(qa, m, k) * q_at(qb, n, k) for k in range(16 * blk, 16 * blk + 16))
                acc += Fraction(e4[qa["scales"][m, blk]]) * Fraction(e4[qb["scales"][n, blk]]) * inner
            exact = acc * Fraction(qa["s_dec"]) * Fraction(qb["s_dec"])
            assert abs(Fraction(got[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)


def test_gemm_closed_form_constant_operands():
    # a = ones(2, 64) with a[0, 0] = 6, worked by hand:
    #   A = 6 -> S_enc = 448, S_dec = fl32(6/2688)
    #   row 0, block 0: bamax 6 -> sb = 448, r = 1: codes 6 and fifteen 1s
    #   every other block: bamax 1 -> sbf = fl32(fl32(1/6) * 448) = 74.67 ->
    #   sb = 72 (nearest E4M3), v = 448/72 = 6.22 -> saturates to 6
    # so x^ = 2688 S_dec, 448 S_dec (x15) in row 0 block 0 and 432 S_dec elsewhere.
    k = 64
    a = np.ones((2, k), np.float32)
    a[0, 0] = 6.0
    qa = oracle.quantize(a)
    assert qa["scales"].tolist() == [[0x7E, 0x69, 0x69, 0x69], [0x69] * 4]   # 72 = 1.125 * 2^6
    assert oracle.e4m3_decode(0x69) == 72.0
    sd = Fraction(qa["s_dec"])
    assert qa["s_dec"] == float(np.float32(6.0 / 2688.0))
    r0 = [2688 * sd] + [448 * sd] * 15 + [432 * sd] * 48
    r1 = [432 * sd] * 64
    expect = [[sum(x * y for x, y in zip(u, v)) for v in (r0, r1)] for u in (r0, r1)]
    c = oracle.gemm(qa, qa)
    for i in range(2):
        for j in range(2):
            assert abs(Fraction(c[i, j]) - expect[i][j]) <= expect[i][j] * Fraction(1, 2 ** 48)

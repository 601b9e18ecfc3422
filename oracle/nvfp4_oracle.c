/*
 * NVFP4 oracle: a plain, slow, obviously-correct CPU restatement of the NVFP4
 * quantization method of "Pretraining Large Language Models with NVFP4"
 * (arXiv 2509.25149 summary page, the paragraph defining the format and the
 * closing limitations paragraph) and of the NVIDIA blog paraphrase "NVFP4
 * Trains with Precision of 16-Bit..." (the technique list: 16-element
 * micro-blocks, E4M3 scales, Hadamard transforms, 2D blocks, stochastic
 * rounding).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header or table with
 * the CUDA library.
 *
 * Arithmetic contract.  Every FP32 operation of the method is emulated as
 * "compute in FP64, round once to FP32" (the C cast).  For +, -, *, / this is
 * bit-identical to one correctly rounded FP32 operation because FP64 carries
 * 53 >= 2*24+2 bits (innocuous double rounding).  Build with
 * -ffp-contract=off so no multiply-add is fused.
 *
 * Parity status: every function below is pinned by a CPU test (see the test
 * files named oracle pins); Philox4x32-10 is pinned by known-answer vectors.
 *
 * Threads: loops over independent rows (or row blocks) carry an OpenMP
 * pragma, so with -fopenmp they run on all host cores.  Each row's
 * arithmetic is the same single-threaded code either way, and no value
 * depends on which thread computed it.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_INVALID 1
#define ORACLE_ERR_NONFINITE 4

/* Product of E2M1 max (6) and E4M3 max (448): maps the tensor amax to the
 * top of both grids (format paragraph: the block max is recoverable at
 * near-FP8 precision). */
#define NVFP4_TENSOR_RANGE 2688.0

static float f32(double v) { return (float)v; }

/* ---- E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit ------------- */

/* Decode a 4-bit E2M1 code straight from its bit fields. */
double nvfp4_oracle_e2m1_decode(uint32_t code) {
    uint32_t s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* Magnitude code of a grid value (0, .5, 1, 1.5, 2, 3, 4, 6) -> 0..7. */
static uint32_t e2m1_code_of_grid_value(double g) {
    if (g == 0.0) return 0;
    if (g == 0.5) return 1;
    if (g == 1.0) return 2;
    if (g == 1.5) return 3;
    if (g == 2.0) return 4;
    if (g == 3.0) return 5;
    if (g == 4.0) return 6;
    return 7; /* 6.0 */
}

/* Round-to-nearest, ties to the even mantissa, saturating at 6.
 * Works binade by binade: inside each binade the E2M1 points are evenly
 * spaced, so the nearest point is lo + gap*nearbyint((a-lo)/gap) and the
 * parity of that integer is the parity of the mantissa bit. */
uint32_t nvfp4_oracle_e2m1_encode_rtn(float v) {
    uint32_t sign = signbit(v) ? 8u : 0u;
    double a = fabs((double)v);
    if (a > 6.0) a = 6.0; /* saturate (inf included) */
    double lo, gap;
    if (a < 1.0)      { lo = 0.0; gap = 0.5; }
    else if (a < 2.0) { lo = 1.0; gap = 0.5; }
    else if (a < 4.0) { lo = 2.0; gap = 1.0; }
    else              { lo = 4.0; gap = 2.0; }
    double n = nearbyint((a - lo) / gap); /* default mode: ties to even */
    double g = lo + gap * n;
    return sign | e2m1_code_of_grid_value(g);
}

/* Stochastic rounding: round |v| (saturated at 6) up to the next grid point
 * with probability equal to its fractional distance from the lower point.
 * rbits is the element's 32-bit random word; its top 24 bits u give the
 * decision "up iff u * 2^-24 < frac", an exact comparison. */
uint32_t nvfp4_oracle_e2m1_encode_sr(float v, uint32_t rbits) {
    static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint32_t sign = signbit(v) ? 8u : 0u;
    double a = fabs((double)v);
    if (a >= 6.0) return sign | 7u;
    int k = 0;
    while (k < 7 && grid[k + 1] <= a) k++;
    double lo = grid[k], hi = grid[k + 1];
    double frac = (a - lo) / (hi - lo); /* exact: gap is a power of two */
    double u = (double)(rbits >> 8) * ldexp(1.0, -24);
    double g = (u < frac) ? hi : lo;
    return sign | e2m1_code_of_grid_value(g);
}

/* ---- E4M3 (unsigned use): 4 exponent bits (bias 7), 3 mantissa bits ---- */

double nvfp4_oracle_e4m3_decode(uint32_t b) {
    uint32_t s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);
    else        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* Nearest non-negative finite E4M3 value, ties to the even code, values
 * above the largest finite value (448) saturate to it.  Brute force over the
 * 127 finite non-negative codes. */
uint32_t nvfp4_oracle_e4m3_encode(float v) {
    double a = (double)v;
    if (!(a > 0.0)) return 0;
    if (a >= 448.0) return 0x7E;
    uint32_t best = 0;
    double best_err = INFINITY;
    for (uint32_t c = 0; c <= 0x7E; c++) {
        double err = fabs(nvfp4_oracle_e4m3_decode(c) - a);
        if (err < best_err || (err == best_err && (c & 1u) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return best;
}

/* ---- Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) ----------------- */

static void mulhilo32(uint32_t a, uint32_t b, uint32_t* hi, uint32_t* lo) {
    uint64_t p = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(p >> 32);
    *lo = (uint32_t)p;
}

void nvfp4_oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; round++) {
        uint32_t hi0, lo0, hi1, lo1;
        mulhilo32(M0, c0, &hi0, &lo0);
        mulhilo32(M1, c2, &hi1, &lo1);
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += W0;
        k1 += W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Random word of element i of a logical tensor for stochastic rounding.
 * One Philox4x32-10 block (key = seed, counter = (i/8 low, i/8 high, 0, 0))
 * gives the 16-bit random values of eight consecutive elements: element i
 * takes half (i mod 8) of the block read as eight 16-bit halves, low half of
 * each word first, i.e. half (i mod 2) of word (i mod 8)/2.  It is returned
 * in the top 16 bits of the word (the low 16 bits zero), so the encode's
 * decision "up iff u * 2^-24 < frac" with u = word >> 8 reads it as
 * h * 2^-16 < frac: P(up) = ceil(frac * 2^16) / 2^16, within 2^-16 of the
 * fractional distance the blog's technique list asks for. */
uint32_t nvfp4_oracle_sr_bits(uint64_t seed, uint64_t i) {
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint64_t q = i >> 3;
    uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), 0u, 0u};
    uint32_t out[4];
    nvfp4_oracle_philox4x32_10(ctr, key, out);
    uint32_t word = out[(i & 7u) >> 1];
    uint32_t half = (i & 1u) ? (word >> 16) : (word & 0xFFFFu);
    return half << 16;
}

/* ---- 16-point random Hadamard transform -------------------------------- */

/* Random signs: bit j of word 0 of Philox(key = rht_seed, counter =
 * (0, 0, 1, 0)) gives d_j = +1 (bit clear) or -1 (bit set). */
void nvfp4_oracle_rht16_signs(uint64_t rht_seed, float d[16]) {
    uint32_t key[2] = {(uint32_t)rht_seed, (uint32_t)(rht_seed >> 32)};
    uint32_t ctr[4] = {0u, 0u, 1u, 0u};
    uint32_t out[4];
    nvfp4_oracle_philox4x32_10(ctr, key, out);
    for (int j = 0; j < 16; j++) d[j] = ((out[0] >> j) & 1u) ? -1.0f : 1.0f;
}

/* y = (1/4) * H16 * (d (.) x) with H16 the Sylvester (natural order)
 * Hadamard matrix, evaluated as four add/subtract stages over index bit s =
 * 0, 1, 2, 3, each sum rounded to FP32, then the exact scaling by 1/4. */
void nvfp4_oracle_rht16(const float x[16], const float d[16], float y[16]) {
    float t[16];
    for (int j = 0; j < 16; j++) t[j] = f32((double)d[j] * (double)x[j]);
    for (int s = 0; s < 4; s++) {
        int h = 1 << s;
        for (int j = 0; j < 16; j++) {
            if (j & h) continue;
            float a = t[j], b = t[j + h];
            t[j] = f32((double)a + (double)b);
            t[j + h] = f32((double)a - (double)b);
        }
    }
    for (int j = 0; j < 16; j++) y[j] = f32((double)t[j] * 0.25);
}

/* Apply the transform in place to every run of 16 consecutive elements of
 * each row of a [rows][cols] tensor (cols % 16 == 0). */
int nvfp4_oracle_rht_rows(float* x, int64_t rows, int64_t cols, uint64_t rht_seed) {
    if (rows < 0 || cols < 0 || cols % 16) return ORACLE_ERR_INVALID;
    float d[16], y[16];
    nvfp4_oracle_rht16_signs(rht_seed, d);
#pragma omp parallel for schedule(static) private(y)
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c += 16) {
            nvfp4_oracle_rht16(x + r * cols + c, d, y);
            memcpy(x + r * cols + c, y, sizeof y);
        }
    return ORACLE_OK;
}

/* ---- tensor amax and the FP32 tensor scales ---------------------------- */

/* A = max |x| over n values; non-finite input is an error. */
int nvfp4_oracle_tensor_amax(const float* x, int64_t n, float* amax) {
    double a = 0.0;
    int nonfinite = 0;
#pragma omp parallel for schedule(static) reduction(max : a) reduction(| : nonfinite)
    for (int64_t i = 0; i < n; i++) {
        if (!isfinite(x[i])) {
            nonfinite = 1;
            continue;
        }
        double v = fabs((double)x[i]);
        if (v > a) a = v;
    }
    if (nonfinite) return ORACLE_ERR_NONFINITE;
    *amax = (float)a; /* exact: a is one of the inputs */
    return ORACLE_OK;
}

/* S_dec = A / 2688 and S_enc = 2688 / A in FP32; A == 0 gives 1 and 1.  An
 * S_enc that overflows FP32 (A below ~7.9e-36) saturates to FLT_MAX. */
void nvfp4_oracle_tensor_scales(float amax, float* s_dec, float* s_enc) {
    if (amax == 0.0f) {
        *s_dec = 1.0f;
        *s_enc = 1.0f;
        return;
    }
    *s_dec = f32((double)amax / NVFP4_TENSOR_RANGE);
    float e = f32(NVFP4_TENSOR_RANGE / (double)amax);
    *s_enc = isinf(e) ? FLT_MAX : e;
}

/* E4M3 block scale from a block amax: sb = E4M3(fl32(fl32(bamax/6) * S_enc)). */
uint32_t nvfp4_oracle_block_scale(float bamax, float s_enc) {
    float t = f32((double)bamax / 6.0);
    float sbf = f32((double)t * (double)s_enc);
    return nvfp4_oracle_e4m3_encode(sbf);
}

/* Per-element encode multiplier r = fl32(S_enc / sb), saturated to FLT_MAX. */
float nvfp4_oracle_block_multiplier(float s_enc, uint32_t sb) {
    float r = f32((double)s_enc / nvfp4_oracle_e4m3_decode(sb));
    return isinf(r) ? FLT_MAX : r;
}

/* ---- the quantizer ------------------------------------------------------
 * x holds rows [row0, row0 + rows) of a logical [*, cols] tensor (the
 * tensor the codes describe: already transposed / transformed).  Blocks run
 * along cols: 1x16 (block_h = 1) or 16x16 (block_h = 16, rows % 16 == 0 and
 * row0 % 16 == 0).  amax_in, if non-NULL, is the amax of the whole logical
 * tensor (so a sample of rows can be quantized); else it is taken over x.
 *
 * Outputs: codes [rows][cols/2], element 2j in the low nibble of byte j;
 * scales [rows/block_h][cols/16]; amax3 = {A, S_dec, S_enc}.
 * Stochastic rounding draws element (row0 + r) * cols + c. */
int nvfp4_oracle_quantize(const float* x, int64_t rows, int64_t cols, int64_t row0, int block_h,
                          int stochastic, uint64_t seed, const float* amax_in, uint8_t* codes,
                          uint8_t* scales, float* amax3) {
    if (rows < 0 || cols < 0 || cols % 16 || (block_h != 1 && block_h != 16)) return ORACLE_ERR_INVALID;
    if (block_h == 16 && (rows % 16 || row0 % 16)) return ORACLE_ERR_INVALID;

    /* 1. tensor amax and the FP32 tensor scales */
    float A;
    if (amax_in) {
        if (!isfinite(*amax_in)) return ORACLE_ERR_NONFINITE;
        A = *amax_in;
    } else {
        int st = nvfp4_oracle_tensor_amax(x, rows * cols, &A);
        if (st) return st;
    }
    float s_dec, s_enc;
    nvfp4_oracle_tensor_scales(A, &s_dec, &s_enc);
    amax3[0] = A;
    amax3[1] = s_dec;
    amax3[2] = s_enc;

    int64_t nkb = cols / 16;
#pragma omp parallel for schedule(static)
    for (int64_t rb = 0; rb < rows; rb += block_h) {
        for (int64_t kb = 0; kb < nkb; kb++) {
            /* 2. block amax over the 1x16 or 16x16 block, then its E4M3 scale */
            float bamax = 0.0f;
            for (int64_t r = rb; r < rb + block_h; r++)
                for (int64_t c = kb * 16; c < kb * 16 + 16; c++) {
                    float v = fabsf(x[r * cols + c]);
                    if (v > bamax) bamax = v;
                }
            uint32_t sb = nvfp4_oracle_block_scale(bamax, s_enc);
            scales[(rb / block_h) * nkb + kb] = (uint8_t)sb;

            /* 3. scale every element and round it to an E2M1 code */
            float rmul = sb ? nvfp4_oracle_block_multiplier(s_enc, sb) : 0.0f;
            for (int64_t r = rb; r < rb + block_h; r++)
                for (int64_t c = kb * 16; c < kb * 16 + 16; c++) {
                    uint32_t code = 0;
                    if (sb) {
                        float v = f32((double)x[r * cols + c] * (double)rmul);
                        if (stochastic) {
                            uint64_t i = (uint64_t)(row0 + r) * (uint64_t)cols + (uint64_t)c;
                            code = nvfp4_oracle_e2m1_encode_sr(v, nvfp4_oracle_sr_bits(seed, i));
                        } else {
                            code = nvfp4_oracle_e2m1_encode_rtn(v);
                        }
                    }
                    uint8_t* byte = &codes[r * (cols / 2) + c / 2];
                    if (c % 2 == 0) *byte = (uint8_t)((*byte & 0xF0u) | code);
                    else            *byte = (uint8_t)((*byte & 0x0Fu) | (code << 4));
                }
        }
    }
    return ORACLE_OK;
}

/* Array forms of the element encoders, for exhaustive checks. */
void nvfp4_oracle_e2m1_encode_rtn_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)nvfp4_oracle_e2m1_encode_rtn(v[i]);
}

void nvfp4_oracle_e2m1_encode_sr_array(const float* v, const uint32_t* rbits, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)nvfp4_oracle_e2m1_encode_sr(v[i], rbits[i]);
}

void nvfp4_oracle_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)nvfp4_oracle_e4m3_encode(v[i]);
}

/* Dequantize: x^ = e2m1(code) * e4m3(sb) * S_dec, exact in FP64. */
int nvfp4_oracle_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                            int block_h, float s_dec, double* out) {
    if (rows < 0 || cols % 16 || (block_h != 1 && block_h != 16)) return ORACLE_ERR_INVALID;
    int64_t nkb = cols / 16;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++) {
            uint32_t byte = codes[r * (cols / 2) + c / 2];
            uint32_t code = (c % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
            double sb = nvfp4_oracle_e4m3_decode(scales[(r / block_h) * nkb + c / 16]);
            out[r * cols + c] = nvfp4_oracle_e2m1_decode(code) * sb * (double)s_dec;
        }
    return ORACLE_OK;
}

/* ---- MXFP4: the format NVFP4 is compared against -------------------------
 * Paper summary page, format paragraph and the explainer's comparison
 * paragraph: MXFP4 (OCP) groups 32 E2M1 elements under one power-of-two
 * scale stored as UE8M0, and has no tensor-level scale; its power-of-two
 * scale can leave the block maximum as low as just above 3, so at worst the
 * +-4 and +-6 levels go unused.  Reading: the block scale is the smallest
 * power of two 2^e with 6 * 2^e >= bamax (no element clips), e clamped to
 * the UE8M0 range [-127, 127]; the code is e + 127.  An all-zero block gets
 * code 0 and zero elements. */

/* UE8M0 decode: 2^(b - 127); 255 is NaN. */
double nvfp4_oracle_e8m0_decode(uint32_t b) {
    if (b == 255u) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* The block scale exponent by search: start below the answer and step up
 * until 6 * 2^e covers bamax (every comparison exact in FP64). */
uint32_t nvfp4_oracle_mx_block_scale(float bamax) {
    double a = (double)bamax;
    if (!(a > 0.0)) return 0;
    int ex;
    (void)frexp(a, &ex); /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 4;      /* 6 * 2^(ex-4) = 0.375 * 2^ex < a */
    while (6.0 * ldexp(1.0, e) < a) e++;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint32_t)(e + 127);
}

/* Quantize a [rows][cols] tensor to MXFP4 with 1x32 blocks along cols
 * (cols % 32 == 0).  Element: v = fl32(x * 2^-e) (a power-of-two scaling),
 * then the same E2M1 rounding as NVFP4 (nearest-even, or stochastic with the
 * element's Philox word: element (row0 + r) * cols + c).  Outputs codes
 * [rows][cols/2] and scales [rows][cols/32] (UE8M0 codes). */
int nvfp4_oracle_mx_quantize(const float* x, int64_t rows, int64_t cols, int64_t row0, int stochastic,
                             uint64_t seed, uint8_t* codes, uint8_t* scales) {
    if (rows < 0 || cols < 0 || cols % 32) return ORACLE_ERR_INVALID;
    for (int64_t i = 0; i < rows * cols; i++)
        if (!isfinite(x[i])) return ORACLE_ERR_NONFINITE;
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < nb; b++) {
            float bamax = 0.0f;
            for (int64_t c = b * 32; c < b * 32 + 32; c++) {
                float v = fabsf(x[r * cols + c]);
                if (v > bamax) bamax = v;
            }
            uint32_t sb = nvfp4_oracle_mx_block_scale(bamax);
            scales[r * nb + b] = (uint8_t)sb;
            double mul = ldexp(1.0, 127 - (int)sb); /* 2^-e */
            for (int64_t c = b * 32; c < b * 32 + 32; c++) {
                uint32_t code = 0;
                if (bamax > 0.0f) {
                    float v = f32((double)x[r * cols + c] * mul);
                    if (stochastic) {
                        uint64_t i = (uint64_t)(row0 + r) * (uint64_t)cols + (uint64_t)c;
                        code = nvfp4_oracle_e2m1_encode_sr(v, nvfp4_oracle_sr_bits(seed, i));
                    } else {
                        code = nvfp4_oracle_e2m1_encode_rtn(v);
                    }
                }
                uint8_t* byte = &codes[r * (cols / 2) + c / 2];
                if (c % 2 == 0) *byte = (uint8_t)((*byte & 0xF0u) | code);
                else            *byte = (uint8_t)((*byte & 0x0Fu) | (code << 4));
            }
        }
    }
    return ORACLE_OK;
}

/* MXFP4 dequantize: x^ = e2m1(code) * 2^(sb - 127), exact in FP64. */
int nvfp4_oracle_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                               double* out) {
    if (rows < 0 || cols % 32) return ORACLE_ERR_INVALID;
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++) {
            uint32_t byte = codes[r * (cols / 2) + c / 2];
            uint32_t code = (c % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
            out[r * cols + c] = nvfp4_oracle_e2m1_decode(code) * nvfp4_oracle_e8m0_decode(scales[r * nb + c / 32]);
        }
    return ORACLE_OK;
}

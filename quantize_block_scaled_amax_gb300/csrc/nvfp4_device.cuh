// Device-side building blocks of the NVFP4 quantizer (sm_103a).
//
// Format ("Pretraining Large Language Models with NVFP4", summary page,
// format paragraph): E2M1 elements, one E4M3 scale per 16 elements, one FP32
// scale per tensor.  Every FP32 step below is a single correctly rounded
// operation (explicit __f*_rn intrinsics, so no contraction into FMA).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

constexpr float kTensorRange = 2688.0f;  // E2M1 max (6) * E4M3 max (448)
constexpr float kFltMax = 3.402823466e+38f;

// Bits of the per-device status word.
constexpr uint32_t kStatusNonfinite = 1u;
constexpr uint32_t kStatusTimeout = 2u;
constexpr uint32_t kStatusBounds = 4u;

// Device bounds checks of the checked build (compiled with -DNVFP4_CHECKED):
// NVFP4_IN_BOUNDS(cond, status) is true when the index condition holds;
// otherwise it records kStatusBounds in the status word (read back as
// NVFP4_ERR_BOUNDS) and the caller skips the access.  In the normal build it
// is the constant true and costs nothing.
#ifdef NVFP4_CHECKED
#define NVFP4_IN_BOUNDS(cond, status) ((cond) || (atomicOr((status), kStatusBounds), false))
#else
#define NVFP4_IN_BOUNDS(cond, status) true
#endif

// ---------------------------------------------------------------------------
// Tensor scales from the tensor amax A (given as the bit pattern of |A|).
struct TensorScales {
    float amax, s_dec, s_enc;
    bool finite;
};

__device__ __forceinline__ TensorScales tensor_scales_from_bits(uint32_t amax_bits) {
    TensorScales t;
    t.finite = amax_bits < 0x7f800000u;
    t.amax = __uint_as_float(amax_bits);
    if (!t.finite || amax_bits == 0u) {
        t.s_dec = 1.0f;
        t.s_enc = 1.0f;
        if (!t.finite) t.amax = __uint_as_float(amax_bits);
        return t;
    }
    t.s_dec = __fdiv_rn(t.amax, kTensorRange);
    float e = __fdiv_rn(kTensorRange, t.amax);
    t.s_enc = isinf(e) ? kFltMax : e;
    return t;
}

// ---------------------------------------------------------------------------
// E4M3 block scale: sb = E4M3_rne_satfinite(fl(fl(bamax / 6) * S_enc)).
__device__ __forceinline__ uint32_t e4m3_from_float(float v) {
    uint16_t out;
    // v goes to the low byte (second source operand)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(v));
    return out & 0xFFu;
}

__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
    // unsigned use only: normal (1 + m/8) 2^(e-7) re-biased into FP32, or
    // subnormal m * 2^-9
    return (b & 0x78u) ? __uint_as_float(((b & 0x7Fu) << 20) + (120u << 23))
                       : __fmul_rn((float)(b & 7u), 0.001953125f);
}

struct BlockScale {
    uint32_t sb;  // E4M3 code (0 = all codes zero)
    float r;      // per-element multiplier S_enc / sb
};

// x / 6 correctly rounded, for x >= 0.  q = x * RN(1/6) is within one ulp of
// the quotient, the remainder x - 6q is exact in one FMA, and one more FMA
// q + rem * RN(1/6) gives the correctly rounded quotient (the correction step
// of Markstein's division, P. Markstein, IBM J. Res. Develop. 34(1), 1990).
// Checked exhaustively against the IEEE division for every finite x >= 0:
// equal for all x >= 2^-125; below that the quotient is subnormal and the
// correction can be off, so those x take the IEEE division.
__device__ __forceinline__ float div6_rn(float x) {
    if (__float_as_uint(x) < 0x01000000u) return __fdiv_rn(x, 6.0f);
    const float inv6 = 0.16666667163372039794921875f;  // RN(1/6)
    const float q = __fmul_rn(x, inv6);
    return __fmaf_rn(__fmaf_rn(-q, 6.0f, x), inv6, q);
}

// The multipliers r = S_enc / e4m3(sb) of a tensor, one per E4M3 code, built
// by a CTA in shared memory before its first block: r saturates to FLT_MAX
// where the quotient overflows, and sb = 0 (and the unused NaN code) get 0.
// Ends with a barrier: every thread of the CTA must call it.
__device__ __forceinline__ void build_r_table(float* tab, float s_enc) {
    for (int i = threadIdx.x; i < 128; i += blockDim.x) {
        float r = 0.0f;
        if (i > 0 && i < 127) {
            r = __fdiv_rn(s_enc, e4m3_to_float((uint32_t)i));
            if (isinf(r)) r = kFltMax;
        }
        tab[i] = r;
    }
    __syncthreads();
}

// sb = E4M3_RN_sat(fl(bamax / 6) * S_enc) and its multiplier from the table
__device__ __forceinline__ BlockScale block_scale(float bamax, float s_enc, const float* r_tab) {
    BlockScale b;
    b.sb = e4m3_from_float(__fmul_rn(div6_rn(bamax), s_enc));
    b.r = r_tab[b.sb];
    return b;
}

// ---------------------------------------------------------------------------
// MXFP4 block scale (the format NVFP4 is compared against: paper summary
// page, format paragraph; 32-element blocks, power-of-two UE8M0 scale, no
// tensor scale): the smallest e with 6 * 2^e >= bamax, clamped to
// [-127, 127], from the bits of bamax = 1.m * 2^(E-127): 6 * 2^e = 1.5 *
// 2^(e+2) covers it at e = E - 129 when 1.m <= 1.5, else at e = E - 128; a
// subnormal bamax (< 2^-126) is covered by the smallest scale.  Returns the
// UE8M0 code e + 127 (0 for an all-zero block).
__device__ __forceinline__ uint32_t mx_block_scale(float bamax) {
    const uint32_t b = __float_as_uint(bamax);
    const int E = (int)(b >> 23);
    if (E == 0) return 0u;  // zero or subnormal: e = -127
    int e = E - 129 + ((b & 0x7FFFFFu) > 0x400000u ? 1 : 0);
    e = max(-127, min(127, e));
    return (uint32_t)(e + 127);
}

// 2^-e for the UE8M0 code sb = e + 127 (exact; 2^-127 is an FP32 subnormal).
__device__ __forceinline__ float mx_multiplier(uint32_t sb) {
    return sb == 254u ? __uint_as_float(0x00400000u) : __uint_as_float((254u - sb) << 23);
}

// ---------------------------------------------------------------------------
// E2M1 codes of values, two at a time: the hardware conversion rounds to
// nearest (ties to even) and saturates to +-6; it keeps the sign of a value
// that rounds to zero (code 0x8 for -0).  It places its first source operand
// in the high nibble, so element 2j (low nibble) is the second operand.  Each
// 8-bit result is widened on its own (cvt.u32.u8) before packing: packing four
// 8-bit registers with one vector mov produced wrong bytes inside the 16x16
// kernel with this toolchain.
__device__ __forceinline__ uint32_t e2m1x2_rtn(float lo, float hi) {
    uint32_t h;
    asm volatile(
        "{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(h)
        : "f"(hi), "f"(lo));
    return h & 0xFFu;
}

// eight values -> one word, v[0] in the lowest nibble (the four converted
// bytes are packed by one vector move instead of shifts and ORs)
__device__ __forceinline__ uint32_t e2m1x8_rtn(const float v[8]) {
    uint32_t out;
    asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
        : "=r"(out)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return out;
}

// ---------------------------------------------------------------------------
// Packed FP32x2 operations on a register pair (lane 0 in the low word): each
// lane is the correctly rounded FP32 operation.
__device__ __forceinline__ uint64_t x2_pack(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float x2_lo(uint64_t a) { return __uint_as_float((uint32_t)a); }
__device__ __forceinline__ float x2_hi(uint64_t a) { return __uint_as_float((uint32_t)(a >> 32)); }
__device__ __forceinline__ uint64_t x2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t x2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t x2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t x2_add_rp(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rp.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t x2_fma_rp(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rp.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).  Round i uses the key
// (k0 + i * 0x9E3779B9, k1 + i * 0xBB67AE85); PhiloxKey holds the ten round
// keys of one seed, built once on the host, so a kernel that takes it as a
// __grid_constant__ parameter reads them from the constant bank instead of
// recomputing the key schedule in every call.
struct PhiloxKey {
    uint32_t k0[10], k1[10];
};

__host__ __device__ inline PhiloxKey philox_key(uint64_t seed) {
    PhiloxKey k;
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
    for (int i = 0; i < 10; ++i) {
        k.k0[i] = a;
        k.k1[i] = b;
        a += 0x9E3779B9u;
        b += 0xBB67AE85u;
    }
    return k;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKey& k) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        const uint64_t p0 = 0xD2511F53ull * c.x;  // one 32x32 -> 64-bit multiply each
        const uint64_t p1 = 0xCD9E8D57ull * c.z;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k.k0[i], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k.k1[i],
                       (uint32_t)p0);
    }
    return c;
}

// Random values of elements i0..i0+7 (i0 % 8 == 0) of a logical tensor for
// stochastic rounding: one Philox block, key = seed, counter = (i0/8 low,
// i0/8 high, 0, 0), read as eight 16-bit halves, low half of each word
// first; element i0 + k takes half k.
__device__ __forceinline__ uint4 sr_words(const PhiloxKey& key, uint64_t i0) {
    uint64_t q = i0 >> 3;
    return philox4x32_10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), 0u, 0u), key);
}

// E2M1 stochastic rounding.  The contract: with a = min(|v|, 6), lo <= a < hi
// the neighbouring grid points, frac = (a - lo) / (hi - lo) and h the
// element's 16-bit random value (see sr_words), a goes up to hi iff
// h * 2^-16 < frac.
//
// Computed with directed rounding instead of a compare.  Let s = hi - lo be
// the grid spacing of a's binade (0.5 below 2, otherwise half the binade's
// power of two) and t = h * 2^-16.  Then lo + s * ceil(frac - t) is hi exactly
// when frac > t, and ceil(frac - t) = ceil(a/s - t) - lo/s, so the rounded
// value is s * ceil((a - s t) / s).  a - s t is formed by one FMA rounded
// upward (s t is exact: a power of two times a 16-bit integer), and rounding
// upward never moves a value past the next multiple of s (those are
// representable), so the ceiling is unchanged; adding M = 1.5 * 2^23 * s,
// whose binade has spacing s, rounded upward again, lands on M + that
// multiple, and subtracting M is exact.  For |v| > 6 the result is >= 6 and
// the saturating conversion gives code 7, which is what clamping to 6 first
// gives; so no clamp is needed (|v| stays finite: |v| <= ~12 by construction
// of the block scale).

// Two elements at once, the FP steps on packed pairs (each lane the same
// correctly rounded operation, directed roundings included): the scaled
// magnitudes a0, a1 (>= 0) with the 16-bit random values h0 (low half of w)
// and h1 (high half); the results take the signs of s0, s1.  p = 2^max(e, 0)
// for a in [2^e, 2^(e+1)), so s = p / 2; uf = h exactly, and
// uf * (p * -2^-17) = -s t; M = 1.5 * 2^22 * p.  The 16-bit halves go
// straight into the conversions and |x| comes out of the scaling multiply
// (encode16_scaled), which saves the logic operations that masked them.
__device__ __forceinline__ void e2m1_sr_pair_mag(float a0, float a1, float s0, float s1, uint32_t w, float& y0,
                                                 float& y1) {
    const uint64_t p = x2_pack(fmaxf(__uint_as_float(__float_as_uint(a0) & 0x7F800000u), 1.0f),
                               fmaxf(__uint_as_float(__float_as_uint(a1) & 0x7F800000u), 1.0f));
    float u0, u1;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f32.u16 %0, lo;\n\tcvt.rn.f32.u16 %1, hi;\n\t}"
        : "=f"(u0), "=f"(u1)
        : "r"(w));
    const float c = -7.62939453125e-06f;  // -2^-17
    const uint64_t z = x2_fma_rp(x2_pack(u0, u1), x2_mul(p, x2_pack(c, c)), x2_pack(a0, a1));
    const uint64_t m = x2_mul(p, x2_pack(6291456.0f, 6291456.0f));
    const uint64_t y = x2_sub(x2_add_rp(z, m), m);
    y0 = __uint_as_float(__float_as_uint(x2_lo(y)) | (__float_as_uint(s0) & 0x80000000u));
    y1 = __uint_as_float(__float_as_uint(x2_hi(y)) | (__float_as_uint(s1) & 0x80000000u));
}

// Encode 16 consecutive elements of one block (already multiplied by r, RTN)
// into 8 bytes.
__device__ __forceinline__ uint2 encode16_rtn(const float v[16]) {
    uint2 out;
    out.x = e2m1x8_rtn(v);
    out.y = e2m1x8_rtn(v + 8);
    return out;
}

// Encode the 16 elements x[k] * r of one block (r > 0, each product rounded
// as __fmul_rn) into 8 bytes.  SR: i0 is the logical index of element 0
// (a multiple of 16); the magnitudes |x| * r come straight out of the
// multiply and the signs from x, the same values as scaling first and taking
// |v| after.
template <bool kSR>
__device__ __forceinline__ uint2 encode16_scaled(const float x[16], float r, const PhiloxKey& key, uint64_t i0) {
    if constexpr (!kSR) {
        float v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = __fmul_rn(x[k], r);
        return encode16_rtn(v);
    } else {
        float y[16];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint4 rw = sr_words(key, i0 + 8 * q);
            const uint32_t w[4] = {rw.x, rw.y, rw.z, rw.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = 8 * q + 2 * k;
                e2m1_sr_pair_mag(__fmul_rn(fabsf(x[e]), r), __fmul_rn(fabsf(x[e + 1]), r), x[e], x[e + 1], w[k], y[e],
                                 y[e + 1]);
            }
        }
        uint2 out;
        out.x = e2m1x8_rtn(y);  // exact: every y is a grid value
        out.y = e2m1x8_rtn(y + 8);
        return out;
    }
}

// 16-point random Hadamard transform of one chunk, in place:
// y = (1/4) H16 (d . x), stages over index bits 0, 1, 2, 3, each sum rounded.
// `dmask` bit j set means d_j = -1.  Stage 0 pairs neighbours (j, j + 1);
// stages 1-3 pair (j, j + h) with h even, so they run on packed pairs
// (x[j], x[j + 1]) against (x[j + h], x[j + h + 1]), as does the x1/4: the same
// correctly rounded operations, half the instructions.
__device__ __forceinline__ void rht16(float x[16], uint32_t dmask) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if ((dmask >> j) & 1u) x[j] = -x[j];
    uint64_t p[8];  // p[k] = (x[2k], x[2k + 1])
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float a = x[2 * k], b = x[2 * k + 1];
        p[k] = x2_pack(__fadd_rn(a, b), __fsub_rn(a, b));  // stage 0
    }
#pragma unroll
    for (int s = 1; s < 4; ++s) {
        const int hp = 1 << (s - 1);  // stride in pairs
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k & hp) continue;
            const uint64_t a = p[k], b = p[k + hp];
            p[k] = x2_add(a, b);
            p[k + hp] = x2_sub(a, b);
        }
    }
    const uint64_t quarter = x2_pack(0.25f, 0.25f);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint64_t y = x2_mul(p[k], quarter);
        x[2 * k] = x2_lo(y);
        x[2 * k + 1] = x2_hi(y);
    }
}

__device__ __forceinline__ uint32_t rht_sign_mask(uint64_t rht_seed) {
    uint4 w = philox4x32_10(make_uint4(0u, 0u, 1u, 0u), philox_key(rht_seed));
    return w.x & 0xFFFFu;
}

// ---------------------------------------------------------------------------
// Scale-buffer addressing (see nvfp4.h, NVFP4_SCALES_MMA).
__device__ __forceinline__ int64_t mma_scale_offset(int64_t r, int64_t kb, int64_t n_katoms) {
    return ((r >> 7) * n_katoms + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

struct ScaleOut {
    uint8_t* p;
    int64_t bytes;     // the layout's size for this tensor (nvfp4_scales_bytes)
    int64_t n_katoms;  // MMA layout
    int64_t nkb;       // linear layout: blocks per row (cols / 16)
    int mma;
    __device__ __forceinline__ int64_t offset(int64_t r, int64_t kb) const {
        return mma ? mma_scale_offset(r, kb, n_katoms) : r * nkb + kb;
    }
    // offset(r + k, kb) = offset(r, kb) + k * row_step() when r % 4 == 0 and k < 4
    __device__ __forceinline__ int64_t row_step() const { return mma ? 16 : nkb; }
};

// ---------------------------------------------------------------------------
// Element loads.  Input rows are 16-byte aligned.
template <typename T>
struct In;

template <>
struct In<__nv_bfloat16> {
    static constexpr int kVec = 8;  // elements per 16-byte load
    __device__ __forceinline__ static void load8(const __nv_bfloat16* p, float f[8]) {
        uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = __uint_as_float(w[j] << 16);
            f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
};

template <>
struct In<float> {
    static constexpr int kVec = 4;
    __device__ __forceinline__ static void load8(const float* p, float f[8]) {
        float4 a = __ldg(reinterpret_cast<const float4*>(p));
        float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
};

__device__ __forceinline__ uint32_t abs_bits(float f) { return __float_as_uint(f) & 0x7FFFFFFFu; }

}  // namespace nvfp4

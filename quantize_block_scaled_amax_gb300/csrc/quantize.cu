// NVFP4 quantization kernels (sm_103a): tensor amax, then block scales and
// E2M1 codes.
//
// Method ("Pretraining Large Language Models with NVFP4", summary page):
// the format paragraph (E2M1 elements, E4M3 scale per 16 elements, FP32
// tensor scale) and the limitations paragraph (the tensor scale costs an
// extra full-tensor amax scan; Hadamard only on the Wgrad inputs); NVIDIA
// blog "NVFP4 Trains with Precision of 16-Bit...", technique list (1x16
// micro-blocks, 2D blocks for weights, stochastic rounding, Hadamard).
//
// Every kernel is HBM-bound.  Pass 1 (amax) reads the input once and writes
// one partial max per CTA into the caller's workspace; pass 2 reduces those
// partials in every CTA (a few KB from L2), derives the tensor scales and
// quantizes, visiting the input in the reverse order of pass 1 so that the
// most recently read part of the input is still in L2.
#include "nvfp4_device.cuh"
#include "nvfp4_launch.h"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// block-wide max of a uint32 (all threads get the result)
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* red) {
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
        w = __reduce_max_sync(0xFFFFFFFFu, w);
        if (lane == 0) red[32] = w;
    }
    __syncthreads();
    uint32_t r = red[32];
    __syncthreads();
    return r;
}

// Tensor scales from the pass-1 partials; CTA 0 publishes {A, S_dec, S_enc}
// and flags a non-finite input.
__device__ __forceinline__ TensorScales reduce_partials(const uint32_t* __restrict__ partials, int npartials,
                                                        float* amax_out, uint32_t* status, uint32_t* red) {
    uint32_t m = 0;
    for (int i = threadIdx.x; i < npartials; i += blockDim.x) m = max(m, __ldcg(partials + i));
    m = block_max_u32(m, red);
    TensorScales ts = tensor_scales_from_bits(m);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        amax_out[0] = ts.amax;
        amax_out[1] = ts.s_dec;
        amax_out[2] = ts.s_enc;
        if (!ts.finite) atomicOr(status, kStatusNonfinite);
    }
    return ts;
}

// max of |x| bit patterns of the 8 elements of one 16-byte vector
template <typename T>
__device__ __forceinline__ uint32_t vec_absmax_bits(uint4 u);

template <>
__device__ __forceinline__ uint32_t vec_absmax_bits<__nv_bfloat16>(uint4 u) {
    // packed 16-bit maxima of the bf16 magnitudes, widened to FP32 bit patterns
    uint32_t m = __vmaxu2(__vmaxu2(u.x & 0x7FFF7FFFu, u.y & 0x7FFF7FFFu),
                          __vmaxu2(u.z & 0x7FFF7FFFu, u.w & 0x7FFF7FFFu));
    return max(m & 0xFFFFu, m >> 16) << 16;
}

template <>
__device__ __forceinline__ uint32_t vec_absmax_bits<float>(uint4 u) {
    return max(max(u.x & 0x7FFFFFFFu, u.y & 0x7FFFFFFFu), max(u.z & 0x7FFFFFFFu, u.w & 0x7FFFFFFFu));
}

// Packed bf16 maxima of magnitudes: max(|a|, |b|) in each half, the sign
// bit of each half the XOR of the inputs' signs (callers mask it); a NaN in
// either input gives the canonical NaN 0x7FFF, so a block holding a NaN still
// has a maximum pattern >= 0x7f800000 once widened.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The larger magnitude of the two halves of a packed bf16x2 magnitude word,
// as the FP32 bit pattern of that bf16 value.
__device__ __forceinline__ uint32_t bf16x2_widen_max(uint32_t m) {
    return bf16x2_absmax(m, __byte_perm(m, 0u, 0x1032)) & 0x7FFF0000u;
}

// vec_absmax_bits by packed maxima (the encode passes; the amax pass keeps
// the integer form, whose NaN patterns it reports as they are)
template <typename T>
__device__ __forceinline__ uint32_t vec_absmax_bits_enc(uint4 u) {
    return vec_absmax_bits<T>(u);
}

template <>
__device__ __forceinline__ uint32_t vec_absmax_bits_enc<__nv_bfloat16>(uint4 u) {
    return bf16x2_widen_max(bf16x2_absmax(bf16x2_absmax(u.x, u.y), bf16x2_absmax(u.z, u.w)));
}

// element c of a 16-byte vector, as FP32
template <typename T>
__device__ __forceinline__ float vec_elem(const uint4& u, int c);

template <>
__device__ __forceinline__ float vec_elem<__nv_bfloat16>(const uint4& u, int c) {
    const uint32_t w = c < 2 ? u.x : c < 4 ? u.y : c < 6 ? u.z : u.w;
    return __uint_as_float((c & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

template <>
__device__ __forceinline__ float vec_elem<float>(const uint4& u, int c) {
    return __uint_as_float(c == 0 ? u.x : c == 1 ? u.y : c == 2 ? u.z : u.w);
}

// ---------------------------------------------------------------------------
// Pass 1: tensor amax (as FP32 magnitude bit patterns; a NaN or an infinity
// gives a pattern >= 0x7f800000).  A dense input is cut into chunks of
// kAmaxThreads * kAmaxUnroll 16-byte vectors; a CTA reads whole chunks (every
// thread issues its kAmaxUnroll loads before using any) and walks the chunks
// with a grid stride, so each CTA streams long contiguous runs.
template <typename T>
__global__ void __launch_bounds__(kAmaxThreads) amax_kernel(const T* __restrict__ x, int64_t rows, int64_t cols,
                                                            int64_t ldx, uint32_t* __restrict__ partials) {
    __shared__ uint32_t red[33];
    constexpr int V = 16 / sizeof(T);
    uint32_t m = 0;
    if (ldx == cols) {
        const uint4* p = reinterpret_cast<const uint4*>(x);
        const int64_t nvec = rows * cols / V;
        constexpr int64_t kChunk = (int64_t)kAmaxThreads * kAmaxUnroll;
        const int64_t nchunks = nvec / kChunk;
        for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
            const uint4* q = p + c * kChunk + threadIdx.x;
            uint4 v[kAmaxUnroll];
#pragma unroll
            for (int k = 0; k < kAmaxUnroll; ++k) v[k] = __ldg(q + k * kAmaxThreads);
#pragma unroll
            for (int k = 0; k < kAmaxUnroll; ++k) m = max(m, vec_absmax_bits<T>(v[k]));
        }
        for (int64_t i = nchunks * kChunk + (int64_t)blockIdx.x * kAmaxThreads + threadIdx.x; i < nvec;
             i += (int64_t)gridDim.x * kAmaxThreads)
            m = max(m, vec_absmax_bits<T>(__ldg(p + i)));
    } else {
        const int64_t vpr = cols / V;
        for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
            const uint4* p = reinterpret_cast<const uint4*>(x + r * ldx);
            for (int64_t c = threadIdx.x; c < vpr; c += blockDim.x) m = max(m, vec_absmax_bits<T>(__ldg(p + c)));
        }
    }
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

// Pass 1 of the RHT path: amax of the transformed tensor.  One unit is 16
// consecutive rows x one 8-byte column vector (4 bf16 or 2 fp32 columns);
// every column of the unit is one 16-point chunk.  The butterfly runs on
// column pairs with packed FP32x2 adds (each lane of add.rn.f32x2 is one
// correctly rounded FP32 add, so the values are those of rht16); the signs
// d_j are applied to the inputs, and the final exact x1/4 is applied to the
// maximum (scaling by 1/4 is monotone, so the max of the scaled values is the
// scaled max).
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}

// 16-point butterfly of two columns at once (x[j] holds row j of both),
// without the signs (applied by the caller) and without the final x1/4.
__device__ __forceinline__ void rht16_pair_unscaled(uint64_t x[16]) {
#pragma unroll
    for (int st = 0; st < 4; ++st) {
        const int h = 1 << st;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j & h) continue;
            const uint64_t a = x[j], b = x[j + h];
            x[j] = f32x2_add(a, b);
            x[j + h] = f32x2_sub(a, b);
        }
    }
}

// one column pair of the unit: FP32 values of rows 0..15 (signs applied)
template <typename T>
__device__ __forceinline__ void unit_pair(const uint2 raw[16], int pr, uint32_t dmask, uint64_t x[16]);

template <>
__device__ __forceinline__ void unit_pair<__nv_bfloat16>(const uint2 raw[16], int pr, uint32_t dmask,
                                                         uint64_t x[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t w = pr ? raw[i].y : raw[i].x;  // two bf16: columns 2pr, 2pr+1
        if ((dmask >> i) & 1u) w ^= 0x80008000u;
        x[i] = f32x2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
}

template <>
__device__ __forceinline__ void unit_pair<float>(const uint2 raw[16], int pr, uint32_t dmask, uint64_t x[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t s = ((dmask >> i) & 1u) << 31;
        x[i] = f32x2_pack(__uint_as_float(raw[i].x ^ s), __uint_as_float(raw[i].y ^ s));
    }
}

// kPlain: the same pass also takes the amax of x itself (partials_plain),
// so an operand quantized both rowwise and transformed-colwise is read once
// for its two tensor scales.
template <typename T>
__device__ __forceinline__ uint32_t raw_absmax_acc(uint32_t acc, uint2 w);

template <>
__device__ __forceinline__ uint32_t raw_absmax_acc<__nv_bfloat16>(uint32_t acc, uint2 w) {
    return bf16x2_absmax(bf16x2_absmax(acc, w.x), w.y);  // packed bf16 magnitudes (sign bits: don't-cares)
}

// max(|a|, |b|, |c|); any NaN input gives the canonical NaN
__device__ __forceinline__ float absmax3_nan(float a, float b, float c) {
    float d;
    asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <>
__device__ __forceinline__ uint32_t raw_absmax_acc<float>(uint32_t acc, uint2 w) {
    return max(acc, max(w.x & 0x7FFFFFFFu, w.y & 0x7FFFFFFFu));
}

template <typename T, bool kPlain>
__global__ void __launch_bounds__(kRhtAmaxThreads, 3) rht_amax_kernel(const T* __restrict__ x, int64_t rows,
                                                                     int64_t cols, int64_t ldx, uint64_t rht_seed,
                                                                     uint32_t* __restrict__ partials,
                                                                     uint32_t* __restrict__ partials_plain) {
    __shared__ uint32_t red[33];
    constexpr int V = 8 / sizeof(T);        // columns per 8-byte vector
    constexpr int kPairs = V / 2;           // column pairs per vector (bf16: 2, fp32: 1)
    const uint32_t dmask = rht_sign_mask(rht_seed);
    const int64_t vpr = cols / V;  // column vectors per row block
    const int64_t nunits = (rows / 16) * vpr;
    float my = 0.0f;  // max |y| (a NaN propagates)
    uint32_t mp = 0;  // kPlain: max |x| (packed 16-bit patterns for bf16)
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < nunits;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rb = u / vpr, cv = u - rb * vpr;
        const T* src = x + rb * 16 * ldx + cv * V;
        uint2 raw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) raw[i] = __ldg(reinterpret_cast<const uint2*>(src + i * ldx));
        if constexpr (kPlain) {
#pragma unroll
            for (int i = 0; i < 16; ++i) mp = raw_absmax_acc<T>(mp, raw[i]);
        }
#pragma unroll
        for (int pr = 0; pr < kPairs; ++pr) {
            uint64_t v[16];
            unit_pair<T>(raw, pr, dmask, v);
            rht16_pair_unscaled(v);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                my = absmax3_nan(my, __uint_as_float((uint32_t)v[i]), __uint_as_float((uint32_t)(v[i] >> 32)));
        }
    }
    // the maximum of fl(|y| / 4) is fl(max |y| / 4) (monotone); a NaN or an
    // infinity stays a pattern >= 0x7f800000
    uint32_t m = __float_as_uint(__fmul_rn(my, 0.25f)) & 0x7FFFFFFFu;
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) partials[blockIdx.x] = m;
    if constexpr (kPlain) {
        if (sizeof(T) == 2) mp = bf16x2_widen_max(mp);  // to an FP32 pattern
        mp = block_max_u32(mp, red);
        if (threadIdx.x == 0) partials_plain[blockIdx.x] = mp;
    }
}

// Pass 1 of the rowwise RHT path (the transform along each row, i.e. along
// the GEMM's K of a rowwise operand): amax of the transformed tensor.  Warp
// items as in the rowwise quantizer: 64 consecutive 16-element chunks of a
// row, lane l taking chunks l and l + 32.
template <typename T>
__global__ void __launch_bounds__(kQuantThreads) rht_rows_amax_kernel(const T* __restrict__ x, int64_t rows,
                                                                      int64_t cols, int64_t ldx, uint64_t rht_seed,
                                                                      uint32_t* __restrict__ partials);

// ---------------------------------------------------------------------------
// Quantize one block of 16 values in place into 8 bytes of codes.
template <bool kSR>
__device__ __forceinline__ uint2 quantize_block(float v[16], const TensorScales& ts, const float* r_tab,
                                                const PhiloxKey& key, uint64_t i0, uint32_t& sb_out) {
    float bamax = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) bamax = fmaxf(bamax, fabsf(v[k]));
    BlockScale bs = block_scale(bamax, ts.s_enc, r_tab);
    if (!ts.finite) bs.sb = 0u;
    sb_out = bs.sb;
    if (bs.sb == 0u) return make_uint2(0u, 0u);
    return encode16_scaled<kSR>(v, bs.r, key, i0);
}

// ---------------------------------------------------------------------------
// One 1x16 block of T in 16-byte vectors: load, block amax, unpack to FP32.
template <typename T>
struct Block16 {
    static constexpr int kVecs = 16 * sizeof(T) / 16;
    uint4 raw[kVecs];
    __device__ __forceinline__ void load(const T* p) {
#pragma unroll
        for (int k = 0; k < kVecs; ++k) raw[k] = __ldg(reinterpret_cast<const uint4*>(p) + k);
    }
    // bit pattern of the largest magnitude (>= 0x7f800000 for a NaN or an infinity)
    __device__ __forceinline__ uint32_t absmax_bits() const {
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < kVecs; ++k) m = max(m, vec_absmax_bits_enc<T>(raw[k]));
        return m;
    }
    __device__ __forceinline__ void unpack(float v[16]) const {
#pragma unroll
        for (int k = 0; k < kVecs; ++k)
#pragma unroll
            for (int c = 0; c < 16 / kVecs; ++c) v[k * (16 / kVecs) + c] = vec_elem<T>(raw[k], c);
    }
};

template <typename T>
__global__ void __launch_bounds__(kQuantThreads) rht_rows_amax_kernel(const T* __restrict__ x, int64_t rows,
                                                                      int64_t cols, int64_t ldx, uint64_t rht_seed,
                                                                      uint32_t* __restrict__ partials) {
    __shared__ uint32_t red[33];
    const uint32_t dmask = rht_sign_mask(rht_seed);
    const int lane = threadIdx.x & 31;
    const int64_t bpr = cols / 16;
    const int64_t ipr = (bpr + kRowItemBlocks - 1) / kRowItemBlocks;
    const int64_t nitems = rows * ipr;
    const int64_t nwarps = (int64_t)gridDim.x * (kQuantThreads / 32);
    uint32_t m = 0;
    for (int64_t it = (int64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5); it < nitems; it += nwarps) {
        const int64_t r = it / ipr;
        const int64_t kb0 = (it - r * ipr) * kRowItemBlocks + lane;
        Block16<T> blk[2];
        bool ok[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            ok[h] = kb0 + 32 * h < bpr;
            if (ok[h]) blk[h].load(x + r * ldx + (kb0 + 32 * h) * 16);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (!ok[h]) continue;
            float v[16];
            blk[h].unpack(v);
            rht16(v, dmask);
#pragma unroll
            for (int k = 0; k < 16; ++k) m = max(m, abs_bits(v[k]));
        }
    }
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

// ---------------------------------------------------------------------------
// MXFP4 element encode of 16 values that share the UE8M0 scale sb of their
// 32-element block (bmax_bits: the block's largest magnitude).  A block
// holding a NaN or an infinity flags the status word and gets zero codes and
// scale; an all-zero block gets zero codes and scale 0.
template <bool kSR>
__device__ __forceinline__ uint2 mx_encode16(float v[16], uint32_t bmax_bits, const PhiloxKey& key, uint64_t i0,
                                             uint32_t* status, uint32_t& sb_out) {
    if (bmax_bits >= 0x7f800000u) {
        atomicOr(status, kStatusNonfinite);
        sb_out = 0u;
        return make_uint2(0u, 0u);
    }
    const uint32_t sb = mx_block_scale(__uint_as_float(bmax_bits));
    sb_out = sb;
    if (bmax_bits == 0u) return make_uint2(0u, 0u);
    return encode16_scaled<kSR>(v, mx_multiplier(sb), key, i0);
}

// ---------------------------------------------------------------------------
// Pass 2, rowwise 1x16.  A warp takes 64 consecutive blocks of one row (lane l
// blocks l and l + 32: two coalesced 1 KB runs of bf16), loads both before
// encoding either, and writes 8 bytes of codes and one scale byte per block.
// Warp items run in the reverse of the amax pass's order, so the part of the
// input read last by that pass (still in L2) is read first here.
// kMX: MXFP4 instead (no amax pass, no tensor scale): a 32-element block is
// the 16-blocks of lanes 2j and 2j+1, which exchange their block maxima; its
// UE8M0 scale is written in both 16-block slots.
// kRHT: each 16-element block is first transformed by the 16-point RHT (the
// block is the transform's chunk), and block maxima are taken afterwards.
// Launch bounds: 4 CTAs of 256 threads per SM (64 registers) except the RHT
// forms with SR or FP32 input, whose transformed blocks need more registers
// (2 CTAs; at 3 or 4 they spilled and the SR one ran 6% slower).
template <typename T, bool kSR, bool kMX, bool kRHT>
__global__ void __launch_bounds__(kQuantThreads, kRHT ? ((kSR || sizeof(T) == 4) ? 2 : 4) : (sizeof(T) == 2 ? 4 : 3))
    quantize_rowwise_kernel(
    const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, const uint32_t* __restrict__ partials,
    int npartials, uint8_t* __restrict__ codes, int64_t ld_codes, ScaleOut so, float* amax_out, uint32_t* status,
    const __grid_constant__ PhiloxKey key, uint64_t rht_seed) {
    __shared__ uint32_t red[33];
    __shared__ float r_tab[128];
    TensorScales ts{};
    if constexpr (!kMX) {
        ts = reduce_partials(partials, npartials, amax_out, status, red);
        build_r_table(r_tab, ts.s_enc);
    } else if (blockIdx.x == 0 && threadIdx.x == 0) {
        amax_out[0] = 0.0f;  // MXFP4 has no tensor scale
        amax_out[1] = 1.0f;
        amax_out[2] = 1.0f;
    }
    const uint32_t dmask = kRHT ? rht_sign_mask(rht_seed) : 0u;
    const int lane = threadIdx.x & 31;
    const int64_t bpr = cols / 16;
    const int64_t ipr = (bpr + kRowItemBlocks - 1) / kRowItemBlocks;
    const int64_t nitems = rows * ipr;
    const int64_t nwarps = (int64_t)gridDim.x * (kQuantThreads / 32);
    for (int64_t it = (int64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5); it < nitems; it += nwarps) {
        const int64_t item = nitems - 1 - it;
        const int64_t r = item / ipr;
        const int64_t kb0 = (item - r * ipr) * kRowItemBlocks + lane;
        Block16<T> blk[2];
        bool ok[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            ok[h] = kb0 + 32 * h < bpr &&
                    NVFP4_IN_BOUNDS(r >= 0 && r < rows && kb0 + 32 * h >= 0 && (kb0 + 32 * h) * 16 + 16 <= cols, status);
            if (ok[h]) blk[h].load(x + r * ldx + (kb0 + 32 * h) * 16);
        }
        uint32_t bm[2];
        float tv[kRHT ? 2 : 1][16];  // transformed blocks (RHT only)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if constexpr (kRHT) {
                bm[h] = 0u;
                if (ok[h]) {
                    blk[h].unpack(tv[h]);
                    rht16(tv[h], dmask);
#pragma unroll
                    for (int k = 0; k < 16; ++k) bm[h] = max(bm[h], abs_bits(tv[h][k]));
                }
            } else {
                bm[h] = ok[h] ? blk[h].absmax_bits() : 0u;
            }
            if constexpr (kMX) bm[h] = max(bm[h], __shfl_xor_sync(0xFFFFFFFFu, bm[h], 1));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (!ok[h]) continue;
            const int64_t kb = kb0 + 32 * h;
            const uint64_t i0 = (uint64_t)r * (uint64_t)cols + (uint64_t)kb * 16;
            uint2 c = make_uint2(0u, 0u);
            uint32_t sb;
            float v[16];
            if constexpr (kRHT) {
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] = tv[h][k];
            } else {
                blk[h].unpack(v);
            }
            if constexpr (kMX) {
                c = mx_encode16<kSR>(v, bm[h], key, i0, status, sb);
            } else {
                BlockScale bs = block_scale(__uint_as_float(bm[h]), ts.s_enc, r_tab);
                if (!ts.finite) bs.sb = 0u;
                sb = bs.sb;
                if (bs.sb != 0u) c = encode16_scaled<kSR>(v, bs.r, key, i0);
            }
            if (NVFP4_IN_BOUNDS(kb * 8 + 8 <= ld_codes, status))
                *reinterpret_cast<uint2*>(codes + r * ld_codes + kb * 8) = c;
            const int64_t soff = so.offset(r, kb);
            if (NVFP4_IN_BOUNDS(soff >= 0 && soff < so.bytes, status)) so.p[soff] = (uint8_t)sb;
        }
    }
}

// ---------------------------------------------------------------------------
// Pass 2, colwise 1x16 (optionally after the 16-point RHT): the output
// describes x^T.  A CTA stages 128-row x 64-column tiles in shared memory
// (bf16: double-buffered, the next tile copied by cp.async while this one
// is encoded); thread t takes column t % 64 and rows 64 * (t / 64) .. +63,
// i.e. 4 blocks of one output row: 32 contiguous bytes of codes and 4 scale
// bytes.
constexpr int kColTileRows = 128;
constexpr int kColTileCols = 64;

template <typename T, bool kSR, bool kRHT, bool kMX>
__global__ void __launch_bounds__(kColThreads) quantize_colwise_kernel(
    const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, const uint32_t* __restrict__ partials,
    int npartials, uint8_t* __restrict__ codes, int64_t ld_codes, ScaleOut so, float* amax_out, uint32_t* status,
    const __grid_constant__ PhiloxKey key, uint64_t rht_seed) {
    // bf16: two tile buffers, the next tile's copies in flight (cp.async)
    // while this one is encoded (the FFN's 8192 x 20480 RTN operand 0.254 ->
    // 0.241 ms); FP32 tiles are twice as large, so one
    constexpr int kBufs = sizeof(T) == 2 ? 2 : 1;
    __shared__ uint32_t red[33];
    __shared__ __align__(16) T tiles[kBufs][kColTileRows][kColTileCols];
    __shared__ float r_tab[128];
    TensorScales ts{};
    if constexpr (!kMX) {
        ts = reduce_partials(partials, npartials, amax_out, status, red);
        build_r_table(r_tab, ts.s_enc);
    } else if (blockIdx.x == 0 && threadIdx.x == 0) {
        amax_out[0] = 0.0f;  // MXFP4 has no tensor scale
        amax_out[1] = 1.0f;
        amax_out[2] = 1.0f;
    }
    const uint32_t dmask = kRHT ? rht_sign_mask(rht_seed) : 0u;

    constexpr int V = 16 / sizeof(T);
    constexpr int kVecPerRow = kColTileCols / V;
    constexpr int kLoads = kColTileRows * kVecPerRow / kColThreads;
    const int64_t tiles_r = (rows + kColTileRows - 1) / kColTileRows;
    const int64_t tiles_c = (cols + kColTileCols - 1) / kColTileCols;
    const int64_t ntiles = tiles_r * tiles_c;
    const int col = threadIdx.x % kColTileCols;
    const int half = threadIdx.x / kColTileCols;

    // first row and column of the t-th tile of this CTA's stream
    auto tile_origin = [&](int64_t t, int64_t& r0, int64_t& c0) {
        const int64_t tile_id = ntiles - 1 - t;
        const int64_t tr = tile_id / tiles_c;
        r0 = tr * kColTileRows;
        c0 = (tile_id - tr * tiles_c) * kColTileCols;
    };
    // stage tile t into buffer b (rows and columns beyond the tensor are not
    // read); with two buffers by cp.async, one commit group per tile
    auto stage = [&](int64_t t, int b) {
        int64_t r0, c0;
        tile_origin(t, r0, c0);
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
            const int L = threadIdx.x + kColThreads * k;
            const int lr = L / kVecPerRow, seg = L % kVecPerRow;
            if (r0 + lr < rows && c0 + seg * V < cols &&
                NVFP4_IN_BOUNDS(r0 + lr >= 0 && c0 + seg * V >= 0 && c0 + seg * V + V <= cols, status)) {
                const T* src = x + (r0 + lr) * ldx + c0 + seg * V;
                if constexpr (kBufs == 2)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                     (uint32_t)__cvta_generic_to_shared(&tiles[b][lr][seg * V])),
                                 "l"(src)
                                 : "memory");
                else
                    *reinterpret_cast<uint4*>(&tiles[b][lr][seg * V]) = __ldg(reinterpret_cast<const uint4*>(src));
            }
        }
        if constexpr (kBufs == 2) asm volatile("cp.async.commit_group;" ::: "memory");
    };
    int buf = 0;
    if (kBufs == 2 && (int64_t)blockIdx.x < ntiles) stage(blockIdx.x, 0);
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        int64_t r0, c0;
        tile_origin(t, r0, c0);
        if constexpr (kBufs == 2) {
            // the next tile's copies go out before this tile is encoded
            if (t + gridDim.x < ntiles) {
                stage(t + gridDim.x, buf ^ 1);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
        } else {
            stage(t, 0);
        }
        __syncthreads();
        const T(&tile)[kColTileRows][kColTileCols] = tiles[buf];
        const int64_t oc = c0 + col;  // output row
        if (oc < cols) {
            const int64_t orow0 = r0 + 64 * half;  // first element of this thread's 64
            uint32_t w[8];
            uint32_t sbs = 0;
            int nb = 0;
            auto load_chunk = [&](int b, float v[16]) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    T e = tile[64 * half + 16 * b + i][col];
                    if constexpr (sizeof(T) == 2)
                        v[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(&e));
                    else
                        v[i] = *reinterpret_cast<const float*>(&e);
                }
                if constexpr (kRHT) rht16(v, dmask);
            };
#pragma unroll
            for (int b = 0; b < 8; ++b) w[b] = 0u;
            if constexpr (kMX) {
                // two 32-element blocks (chunk pairs 0-1 and 2-3); rows % 32 == 0
#pragma unroll
                for (int pb = 0; pb < 2; ++pb) {
                    if (orow0 + 32 * pb < rows) {
                        float v0[16], v1[16];
                        load_chunk(2 * pb, v0);
                        load_chunk(2 * pb + 1, v1);
                        uint32_t bm = 0;
#pragma unroll
                        for (int i = 0; i < 16; ++i) bm = max(bm, max(abs_bits(v0[i]), abs_bits(v1[i])));
                        const uint64_t i0 = (uint64_t)oc * (uint64_t)rows + orow0 + 32 * pb;
                        uint32_t sb;
                        const uint2 c0 = mx_encode16<kSR>(v0, bm, key, i0, status, sb);
                        const uint2 c1 = mx_encode16<kSR>(v1, bm, key, i0 + 16, status, sb);
                        w[4 * pb] = c0.x;
                        w[4 * pb + 1] = c0.y;
                        w[4 * pb + 2] = c1.x;
                        w[4 * pb + 3] = c1.y;
                        sbs |= (sb | (sb << 8)) << (16 * pb);
                        nb = 2 * pb + 2;
                    }
                }
            } else {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if (orow0 + 16 * b < rows) {
                        float v[16];
                        load_chunk(b, v);
                        uint32_t sb;
                        uint2 c = quantize_block<kSR>(v, ts, r_tab, key, (uint64_t)oc * (uint64_t)rows + orow0 + 16 * b, sb);
                        w[2 * b] = c.x;
                        w[2 * b + 1] = c.y;
                        sbs |= sb << (8 * b);
                        nb = b + 1;
                    }
                }
            }
            // output row oc of x^T holds `rows` codes; this thread's nb blocks
            // from element orow0; its scale bytes from block orow0 / 16
            if (nb > 0 && NVFP4_IN_BOUNDS(orow0 / 2 + 8 * nb <= ld_codes && orow0 + 16 * nb <= rows &&
                                              so.offset(oc, orow0 / 16 + nb - 1) < so.bytes && so.offset(oc, orow0 / 16) >= 0,
                                          status)) {
                uint8_t* dst = codes + oc * ld_codes + orow0 / 2;
                if (nb == 4) {
                    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                } else {
                    for (int b = 0; b < nb; ++b) reinterpret_cast<uint2*>(dst)[b] = make_uint2(w[2 * b], w[2 * b + 1]);
                }
                const int64_t kb0 = orow0 / 16;
                const int64_t off = so.offset(oc, kb0);
                if (nb == 4 && (off & 3) == 0) {
                    *reinterpret_cast<uint32_t*>(so.p + off) = sbs;
                } else {
                    for (int b = 0; b < nb; ++b) so.p[so.offset(oc, kb0 + b)] = (uint8_t)(sbs >> (8 * b));
                }
            }
        }
        __syncthreads();  // every thread is done with this buffer before it is refilled
        if constexpr (kBufs == 2) buf ^= 1;
    }
}

// ---------------------------------------------------------------------------
// Pass 2, 16x16 blocks (weights, RTN): one E4M3 scale per 16x16 tile, codes
// for x (rowwise) and for x^T (colwise) from one read.  A warp takes a unit
// of 128 columns by one or two tiles of 16 rows; lane l holds columns
// 4l..4l+3 of every row of the unit, so a tile's 16 columns sit in four
// neighbouring lanes and its maximum is two shuffles.  Under RTN a code
// depends only on the element and its tile's scale, so neighbouring values
// are converted in pairs twice: along the row for the codes of x, and down
// the column (rows 2i, 2i+1) for the codes of x^T, which each lane then
// holds whole for its four columns.  No shared memory is used after the
// tensor-scale reduction and warps never wait on one another.

// four consecutive elements of one row
template <typename T>
struct Quad;

template <>
struct Quad<__nv_bfloat16> {
    uint2 u;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = __ldg(reinterpret_cast<const uint2*>(p)); }
    // running maximum of the magnitudes, packed bf16 (sign bits are
    // don't-cares until widen)
    __device__ __forceinline__ uint32_t absmax_acc(uint32_t acc) const {
        return bf16x2_absmax(bf16x2_absmax(acc, u.x), u.y);
    }
    __device__ __forceinline__ static uint32_t widen(uint32_t acc) { return bf16x2_widen_max(acc); }
    __device__ __forceinline__ void pairs(uint64_t& p01, uint64_t& p23) const {
        p01 = f32x2_pack(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u));
        p23 = f32x2_pack(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    }
};

template <>
struct Quad<float> {
    uint4 u;
    __device__ __forceinline__ void load(const float* p) { u = __ldg(reinterpret_cast<const uint4*>(p)); }
    __device__ __forceinline__ uint32_t absmax_acc(uint32_t acc) const { return max(acc, vec_absmax_bits<float>(u)); }
    __device__ __forceinline__ static uint32_t widen(uint32_t acc) { return acc; }
    __device__ __forceinline__ void pairs(uint64_t& p01, uint64_t& p23) const {
        p01 = (uint64_t)u.x | ((uint64_t)u.y << 32);
        p23 = (uint64_t)u.z | ((uint64_t)u.w << 32);
    }
};

__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float f32x2_lo(uint64_t a) { return __uint_as_float((uint32_t)a); }
__device__ __forceinline__ float f32x2_hi(uint64_t a) { return __uint_as_float((uint32_t)(a >> 32)); }

// E2M1 codes (RTN) of v0..v3 in the low 16 bits, v0 in the lowest nibble
__device__ __forceinline__ uint32_t e2m1x4_rtn(float v0, float v1, float v2, float v3) {
    uint32_t out;
    asm("{\n\t.reg .b8 t0, t1;\n\t.reg .b16 h;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
        "mov.b16 h, {t0, t1};\n\t"
        "cvt.u32.u16 %0, h;\n\t}"
        : "=r"(out)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
    return out;
}

// E2M1 codes (RTN) of four pairs: byte k holds lo[k] in its low nibble and
// hi[k] in its high nibble
__device__ __forceinline__ uint32_t e2m1_pairs4_rtn(const float lo[4], const float hi[4]) {
    uint32_t out;
    asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
        : "=r"(out)
        : "f"(lo[0]), "f"(hi[0]), "f"(lo[1]), "f"(hi[1]), "f"(lo[2]), "f"(hi[2]), "f"(lo[3]), "f"(hi[3]));
    return out;
}

// 4x4 byte transpose: byte k of out[j] = byte j of w[k]
__device__ __forceinline__ void byte_transpose4(const uint32_t w[4], uint32_t out[4]) {
    const uint32_t t0 = __byte_perm(w[0], w[1], 0x5140), t1 = __byte_perm(w[0], w[1], 0x7362);
    const uint32_t t2 = __byte_perm(w[2], w[3], 0x5140), t3 = __byte_perm(w[2], w[3], 0x7362);
    out[0] = __byte_perm(t0, t2, 0x5410);
    out[1] = __byte_perm(t0, t2, 0x7632);
    out[2] = __byte_perm(t1, t3, 0x5410);
    out[3] = __byte_perm(t1, t3, 0x7632);
}

template <typename T>
struct Unit2d {
    static constexpr int kTiles = sizeof(T) == 2 ? 2 : 1;  // 16-row tiles per unit (register budget)
    static constexpr int kRows = 16 * kTiles;
    static constexpr int kCols = 128;
};

template <int N>
struct TileIdx {
    static constexpr int value = N;
};

template <typename T>
__global__ void __launch_bounds__(k2dThreads, 2) quantize_2d_kernel(
    const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, const uint32_t* __restrict__ partials,
    int npartials, uint8_t* __restrict__ codes_r, int64_t ld_r, ScaleOut so_r, float* amax_r,
    uint8_t* __restrict__ codes_c, int64_t ld_c, ScaleOut so_c, float* amax_c, uint32_t* status) {
    using U = Unit2d<T>;
    // bf16: two 16-row register buffers, the loads of the next tile in flight
    // while one tile is encoded; fp32 quads are twice as wide, so one buffer
    constexpr bool kPipe = U::kTiles == 2;
    __shared__ uint32_t red[33];
    __shared__ float r_tab[128];
    float* amax_out = amax_r ? amax_r : amax_c;
    const TensorScales ts = reduce_partials(partials, npartials, amax_out, status, red);
    build_r_table(r_tab, ts.s_enc);
    if (amax_r && amax_c && blockIdx.x == 0 && threadIdx.x == 0) {
        amax_c[0] = ts.amax;
        amax_c[1] = ts.s_dec;
        amax_c[2] = ts.s_enc;
    }
    const int lane = threadIdx.x & 31;
    const int qd = lane & 3;  // position of the lane among the four of its tile
    const int64_t groups = (cols + U::kCols - 1) / U::kCols;
    const int64_t nunits = ((rows + U::kRows - 1) / U::kRows) * groups;
    const int64_t nwarps = (int64_t)gridDim.x * (k2dThreads / 32);
    const int64_t first = (int64_t)blockIdx.x * (k2dThreads / 32) + (threadIdx.x >> 5);
    const int64_t step_r = so_r.row_step(), step_c = so_c.row_step();

    // Tile s of this warp's stream is tile s % kTiles of its unit s / kTiles.
    struct TilePos {
        int64_t r, col;  // first row of the tile, first column of the lane
        bool valid;      // the unit exists (warp-uniform)
        bool has;        // the tile exists: the last unit may have fewer rows (warp-uniform)
        bool ok;         // the lane's columns exist
    };
    auto tile_pos = [&](int64_t s) {
        TilePos p{0, 0, false, false, false};
        const int64_t u = first + (s / U::kTiles) * nwarps;
        if (u >= nunits) return p;
        const int64_t unit = nunits - 1 - u;  // last unit first: the end of x is what the amax pass left in L2
        const int64_t ur = unit / groups;
        p.col = (unit - ur * groups) * U::kCols + 4 * lane;
        p.r = ur * U::kRows + 16 * (s % U::kTiles);
        p.valid = true;
        p.has = p.r < rows;  // rows % 16 == 0
        p.ok = p.has && p.col < cols;  // cols % 16 == 0
        return p;
    };
    auto load16 = [&](Quad<T>(&q)[16], const TilePos& p) {
        if (!NVFP4_IN_BOUNDS(p.r >= 0 && p.r + 16 <= rows && p.col >= 0 && p.col + 4 <= cols, status)) return;
        const T* src = x + p.r * ldx + p.col;
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i].load(src + i * ldx);
    };

    uint32_t cw[4][2 * U::kTiles];  // codes of x^T: 8 bytes per column and tile
    auto process = [&](const Quad<T>(&q)[16], const TilePos& p, auto tile) {
        constexpr int t = decltype(tile)::value;
        if (p.has) {
            uint32_t acc = 0;
            if (p.ok) {
#pragma unroll
                for (int i = 0; i < 16; ++i) acc = q[i].absmax_acc(acc);
            }
            uint32_t m = Quad<T>::widen(acc);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            BlockScale bs = block_scale(__uint_as_float(m), ts.s_enc, r_tab);
            if (!ts.finite) bs.sb = 0u;
            const bool zero = bs.sb == 0u;  // every code of the tile is 0
            const uint64_t r2 = f32x2_pack(bs.r, bs.r);
            uint32_t wk[4];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                uint64_t a01, a23, b01, b23;
                q[i].pairs(a01, a23);
                q[i + 1].pairs(b01, b23);
                a01 = f32x2_mul(a01, r2);
                a23 = f32x2_mul(a23, r2);
                b01 = f32x2_mul(b01, r2);
                b23 = f32x2_mul(b23, r2);
                const float a[4] = {f32x2_lo(a01), f32x2_hi(a01), f32x2_lo(a23), f32x2_hi(a23)};
                const float b[4] = {f32x2_lo(b01), f32x2_hi(b01), f32x2_lo(b23), f32x2_hi(b23)};
                if (codes_r && p.ok && NVFP4_IN_BOUNDS(p.r + i + 1 < rows && p.col / 2 + 2 <= ld_r, status)) {
                    const int64_t r = p.r + i;
                    const uint32_t ca = zero ? 0u : e2m1x4_rtn(a[0], a[1], a[2], a[3]);
                    const uint32_t cb = zero ? 0u : e2m1x4_rtn(b[0], b[1], b[2], b[3]);
                    *reinterpret_cast<uint16_t*>(codes_r + r * ld_r + p.col / 2) = (uint16_t)ca;
                    *reinterpret_cast<uint16_t*>(codes_r + (r + 1) * ld_r + p.col / 2) = (uint16_t)cb;
                }
                // rows i, i+1 of the four columns: byte j of wk = column j
                wk[(i / 2) % 4] = e2m1_pairs4_rtn(a, b);
                if ((i / 2) % 4 == 3) {
                    uint32_t c4[4];
                    byte_transpose4(wk, c4);
#pragma unroll
                    for (int j = 0; j < 4; ++j) cw[j][2 * t + i / 8] = zero ? 0u : c4[j];
                }
            }
            if (p.ok) {
                if (codes_r && NVFP4_IN_BOUNDS(so_r.offset(p.r + 4 * qd, p.col / 16) >= 0 &&
                                                   so_r.offset(p.r + 4 * qd, p.col / 16) + 3 * step_r < so_r.bytes,
                                               status)) {
                    uint8_t* sp = so_r.p + so_r.offset(p.r + 4 * qd, p.col / 16);
#pragma unroll
                    for (int k = 0; k < 4; ++k) sp[k * step_r] = (uint8_t)bs.sb;
                }
                if (codes_c && NVFP4_IN_BOUNDS(so_c.offset(p.col, p.r / 16) >= 0 &&
                                                   so_c.offset(p.col, p.r / 16) + 3 * step_c < so_c.bytes,
                                               status)) {
                    uint8_t* sp = so_c.p + so_c.offset(p.col, p.r / 16);
#pragma unroll
                    for (int j = 0; j < 4; ++j) sp[j * step_c] = (uint8_t)bs.sb;
                }
            }
        }
        if (t == U::kTiles - 1 && codes_c && p.valid && p.col < cols &&
            NVFP4_IN_BOUNDS(p.col + 4 <= cols && (p.r - 16 * t) / 2 + 8 * U::kTiles <= ld_c, status)) {
            // the unit is done: 8 bytes of x^T per column and tile
            const int64_t r0 = p.r - 16 * t;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint8_t* dst = codes_c + (p.col + j) * ld_c + r0 / 2;
                bool stored = false;
                if constexpr (t == 1) {
                    if (p.has) {
                        *reinterpret_cast<uint4*>(dst) = make_uint4(cw[j][0], cw[j][1], cw[j][2], cw[j][3]);
                        stored = true;
                    }
                }
                if (!stored) *reinterpret_cast<uint2*>(dst) = make_uint2(cw[j][0], cw[j][1]);
            }
        }
    };

    Quad<T> qa[16];
    TilePos pa = tile_pos(0);
    if (pa.ok) load16(qa, pa);
    if constexpr (kPipe) {
        Quad<T> qb[16];
        for (int64_t s = 0; pa.valid; s += 2) {
            const TilePos pb = tile_pos(s + 1);  // tile 1 of this unit
            if (pb.ok) load16(qb, pb);
            process(qa, pa, TileIdx<0>{});
            pa = tile_pos(s + 2);  // tile 0 of the next unit
            if (pa.ok) load16(qa, pa);
            process(qb, pb, TileIdx<1>{});
        }
    } else {
        for (int64_t s = 0; pa.valid;) {
            process(qa, pa, TileIdx<0>{});
            pa = tile_pos(++s);
            if (pa.ok) load16(qa, pa);
        }
    }
}

// ---------------------------------------------------------------------------
// bf16 transpose, y[c][r] = x[r][c] (the BF16 fallback GEMM takes K-major
// operands; its Dgrad and Wgrad need W^T, dY^T and X^T).  A thread moves an
// 8 x 8 block: eight 16-byte row loads (a warp's 32 neighbouring blocks read
// 512 contiguous bytes per row), one byte permute per output word (word k of
// output row j holds rows 2k and 2k + 1 of input column j, i.e. halves of
// input words [2k][j/2] and [2k+1][j/2]) and eight 16-byte stores.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint4* __restrict__ x, int64_t rows, int64_t cols,
                                                            int64_t ldx_vec, uint4* __restrict__ y, int64_t ldy_vec) {
    const int64_t cb_n = cols / 8;
    const int64_t nunits = (rows / 8) * cb_n;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < nunits; u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rb = u / cb_n, cb = u - rb * cb_n;
        uint32_t w[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 v = __ldg(x + (8 * rb + i) * ldx_vec + cb);
            w[i][0] = v.x;
            w[i][1] = v.y;
            w[i][2] = v.z;
            w[i][3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;  // high halves : low halves
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) o[k] = __byte_perm(w[2 * k][j / 2], w[2 * k + 1][j / 2], sel);
            y[(8 * cb + j) * ldy_vec + rb] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// ---------------------------------------------------------------------------
// Host-side launchers.

template <typename T>
static void launch_amax_t(const void* x, int64_t rows, int64_t cols, int64_t ldx, uint32_t* partials, int grid,
                          cudaStream_t s) {
    amax_kernel<T><<<grid, kAmaxThreads, 0, s>>>(static_cast<const T*>(x), rows, cols, ldx, partials);
}

void launch_amax(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx, uint32_t* partials, int grid,
                 cudaStream_t s) {
    if (fp32) launch_amax_t<float>(x, rows, cols, ldx, partials, grid, s);
    else launch_amax_t<__nv_bfloat16>(x, rows, cols, ldx, partials, grid, s);
}

void launch_rht_rows_amax(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx, uint64_t rht_seed,
                          uint32_t* partials, int grid, cudaStream_t s) {
    if (fp32)
        rht_rows_amax_kernel<float><<<grid, kQuantThreads, 0, s>>>(static_cast<const float*>(x), rows, cols, ldx,
                                                                   rht_seed, partials);
    else
        rht_rows_amax_kernel<__nv_bfloat16><<<grid, kQuantThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                                                                           rows, cols, ldx, rht_seed, partials);
}

void launch_rht_amax(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx, uint64_t rht_seed,
                     uint32_t* partials, int grid, cudaStream_t s, uint32_t* partials_plain) {
#define NVFP4_RHT_AMAX(T, P)                                                                                 \
    rht_amax_kernel<T, P><<<grid, kRhtAmaxThreads, 0, s>>>(static_cast<const T*>(x), rows, cols, ldx, rht_seed, \
                                                           partials, partials_plain)
    if (fp32) {
        if (partials_plain) NVFP4_RHT_AMAX(float, true); else NVFP4_RHT_AMAX(float, false);
    } else {
        if (partials_plain) NVFP4_RHT_AMAX(__nv_bfloat16, true); else NVFP4_RHT_AMAX(__nv_bfloat16, false);
    }
#undef NVFP4_RHT_AMAX
}

void launch_quantize_rowwise(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx,
                             const uint32_t* partials, int npartials, uint8_t* codes, int64_t ld_codes, ScaleOut so,
                             float* amax_out, uint32_t* status, bool sr, bool mx, uint64_t seed, bool rht,
                             uint64_t rht_seed, int grid, cudaStream_t s) {
    const PhiloxKey key = philox_key(seed);
#define NVFP4_ROW(T, SR, MX, RHT)                                                                               \
    quantize_rowwise_kernel<T, SR, MX, RHT><<<grid, kQuantThreads, 0, s>>>(                                    \
        static_cast<const T*>(x), rows, cols, ldx, partials, npartials, codes, ld_codes, so, amax_out, status, \
        key, rht_seed)
#define NVFP4_ROW_MX(T, SR, RHT) \
    if (mx) NVFP4_ROW(T, SR, true, RHT); else NVFP4_ROW(T, SR, false, RHT)
#define NVFP4_ROW_RHT(T, SR) \
    if (rht) { NVFP4_ROW_MX(T, SR, true); } else { NVFP4_ROW_MX(T, SR, false); }
    if (fp32) {
        if (sr) { NVFP4_ROW_RHT(float, true) } else { NVFP4_ROW_RHT(float, false) }
    } else {
        if (sr) { NVFP4_ROW_RHT(__nv_bfloat16, true) } else { NVFP4_ROW_RHT(__nv_bfloat16, false) }
    }
#undef NVFP4_ROW_RHT
#undef NVFP4_ROW_MX
#undef NVFP4_ROW
}

void launch_quantize_colwise(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx,
                             const uint32_t* partials, int npartials, uint8_t* codes, int64_t ld_codes, ScaleOut so,
                             float* amax_out, uint32_t* status, bool sr, bool mx, uint64_t seed, bool rht,
                             uint64_t rht_seed, int grid, cudaStream_t s) {
    const PhiloxKey key = philox_key(seed);
#define NVFP4_COL(T, SR, RHT, MX)                                                                                    \
    quantize_colwise_kernel<T, SR, RHT, MX><<<grid, kColThreads, 0, s>>>(static_cast<const T*>(x), rows, cols, ldx,  \
                                                                         partials, npartials, codes, ld_codes, so,   \
                                                                         amax_out, status, key, rht_seed)
#define NVFP4_COL_MX(T, SR, RHT) \
    if (mx) NVFP4_COL(T, SR, RHT, true); else NVFP4_COL(T, SR, RHT, false)
#define NVFP4_COL_RHT(T, SR) \
    if (rht) { NVFP4_COL_MX(T, SR, true); } else { NVFP4_COL_MX(T, SR, false); }
    if (fp32) {
        if (sr) { NVFP4_COL_RHT(float, true) } else { NVFP4_COL_RHT(float, false) }
    } else {
        if (sr) { NVFP4_COL_RHT(__nv_bfloat16, true) } else { NVFP4_COL_RHT(__nv_bfloat16, false) }
    }
#undef NVFP4_COL_RHT
#undef NVFP4_COL_MX
#undef NVFP4_COL
}

void launch_quantize_2d(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx, const uint32_t* partials,
                        int npartials, uint8_t* codes_r, int64_t ld_r, ScaleOut so_r, float* amax_r, uint8_t* codes_c,
                        int64_t ld_c, ScaleOut so_c, float* amax_c, uint32_t* status, int grid, cudaStream_t s) {
    if (fp32)
        quantize_2d_kernel<float><<<grid, k2dThreads, 0, s>>>(static_cast<const float*>(x), rows, cols, ldx, partials,
                                                              npartials, codes_r, ld_r, so_r, amax_r, codes_c, ld_c,
                                                              so_c, amax_c, status);
    else
        quantize_2d_kernel<__nv_bfloat16><<<grid, k2dThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(x), rows,
                                                                      cols, ldx, partials, npartials, codes_r, ld_r,
                                                                      so_r, amax_r, codes_c, ld_c, so_c, amax_c,
                                                                      status);
}

int64_t colwise_tiles(int64_t rows, int64_t cols) {
    return ((rows + kColTileRows - 1) / kColTileRows) * ((cols + kColTileCols - 1) / kColTileCols);
}

int quantize_2d_grid(int64_t rows, int64_t cols, bool fp32, int num_sms) {
    // the kernel loops over its units, so the grid is what stays resident at once
    static int occ[2] = {0, 0};
    int& o = occ[fp32 ? 1 : 0];
    if (o == 0) {
        int n = 0;
        cudaError_t e = fp32 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_2d_kernel<float>, k2dThreads, 0)
                             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_2d_kernel<__nv_bfloat16>,
                                                                             k2dThreads, 0);
        o = (e == cudaSuccess && n > 0) ? n : 2;
    }
    const int64_t unit_rows = fp32 ? Unit2d<float>::kRows : Unit2d<__nv_bfloat16>::kRows;
    const int64_t units = ((rows + unit_rows - 1) / unit_rows) * ((cols + 127) / 128);
    const int64_t ctas = (units + k2dThreads / 32 - 1) / (k2dThreads / 32);
    return (int)std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)o * num_sms));
}

void launch_transpose_bf16(const void* x, int64_t rows, int64_t cols, int64_t ldx, void* y, int64_t ldy, int grid,
                           cudaStream_t s) {
    transpose_bf16_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(x), rows, cols, ldx / 8,
                                               static_cast<uint4*>(y), ldy / 8);
}

}  // namespace nvfp4

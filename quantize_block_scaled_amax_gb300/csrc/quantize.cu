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

template <typename T>
__global__ void __launch_bounds__(kRhtAmaxThreads, 3) rht_amax_kernel(const T* __restrict__ x, int64_t rows,
                                                                     int64_t cols, int64_t ldx, uint64_t rht_seed,
                                                                     uint32_t* __restrict__ partials) {
    __shared__ uint32_t red[33];
    constexpr int V = 8 / sizeof(T);        // columns per 8-byte vector
    constexpr int kPairs = V / 2;           // column pairs per vector (bf16: 2, fp32: 1)
    const uint32_t dmask = rht_sign_mask(rht_seed);
    const int64_t vpr = cols / V;  // column vectors per row block
    const int64_t nunits = (rows / 16) * vpr;
    uint32_t m = 0;  // max |y| bit pattern (a NaN or an infinity gives >= 0x7f800000)
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < nunits;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rb = u / vpr, cv = u - rb * vpr;
        const T* src = x + rb * 16 * ldx + cv * V;
        uint2 raw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) raw[i] = __ldg(reinterpret_cast<const uint2*>(src + i * ldx));
#pragma unroll
        for (int pr = 0; pr < kPairs; ++pr) {
            uint64_t v[16];
            unit_pair<T>(raw, pr, dmask, v);
            rht16_pair_unscaled(v);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                m = max(m, max((uint32_t)v[i] & 0x7FFFFFFFu, (uint32_t)(v[i] >> 32) & 0x7FFFFFFFu));
        }
    }
    // the maximum of fl(|y| / 4) is fl(max |y| / 4) (monotone); a NaN or an
    // infinity stays a pattern >= 0x7f800000
    m = __float_as_uint(__fmul_rn(__uint_as_float(m), 0.25f)) & 0x7FFFFFFFu;
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) partials[blockIdx.x] = m;
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
__device__ __forceinline__ uint2 quantize_block(float v[16], const TensorScales& ts, uint64_t seed, uint64_t i0,
                                                uint32_t& sb_out) {
    float bamax = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) bamax = fmaxf(bamax, fabsf(v[k]));
    BlockScale bs = block_scale(bamax, ts.s_enc);
    if (!ts.finite) bs.sb = 0u;
    sb_out = bs.sb;
    if (bs.sb == 0u) return make_uint2(0u, 0u);
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __fmul_rn(v[k], bs.r);
    return encode16<kSR>(v, seed, i0);
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
        for (int k = 0; k < kVecs; ++k) m = max(m, vec_absmax_bits<T>(raw[k]));
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
__device__ __forceinline__ uint2 mx_encode16(float v[16], uint32_t bmax_bits, uint64_t seed, uint64_t i0,
                                             uint32_t* status, uint32_t& sb_out) {
    if (bmax_bits >= 0x7f800000u) {
        atomicOr(status, kStatusNonfinite);
        sb_out = 0u;
        return make_uint2(0u, 0u);
    }
    const uint32_t sb = mx_block_scale(__uint_as_float(bmax_bits));
    sb_out = sb;
    if (bmax_bits == 0u) return make_uint2(0u, 0u);
    const float mul = mx_multiplier(sb);
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __fmul_rn(v[k], mul);
    return encode16<kSR>(v, seed, i0);
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
template <typename T, bool kSR, bool kMX, bool kRHT>
__global__ void __launch_bounds__(kQuantThreads, sizeof(T) == 2 ? 4 : 3) quantize_rowwise_kernel(
    const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, const uint32_t* __restrict__ partials,
    int npartials, uint8_t* __restrict__ codes, int64_t ld_codes, ScaleOut so, float* amax_out, uint32_t* status,
    uint64_t seed, uint64_t rht_seed) {
    __shared__ uint32_t red[33];
    TensorScales ts{};
    if constexpr (!kMX) {
        ts = reduce_partials(partials, npartials, amax_out, status, red);
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
            ok[h] = kb0 + 32 * h < bpr;
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
                c = mx_encode16<kSR>(v, bm[h], seed, i0, status, sb);
            } else {
                BlockScale bs = block_scale(__uint_as_float(bm[h]), ts.s_enc);
                if (!ts.finite) bs.sb = 0u;
                sb = bs.sb;
                if (bs.sb != 0u) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[k] = __fmul_rn(v[k], bs.r);
                    c = encode16<kSR>(v, seed, i0);
                }
            }
            *reinterpret_cast<uint2*>(codes + r * ld_codes + kb * 8) = c;
            so.p[so.offset(r, kb)] = (uint8_t)sb;
        }
    }
}

// ---------------------------------------------------------------------------
// Pass 2, colwise 1x16 (optionally after the 16-point RHT): the output
// describes x^T.  A CTA stages a 128-row x 64-column tile in shared memory;
// thread t takes column t % 64 and rows 64 * (t / 64) .. +63, i.e. 4 blocks
// of one output row: 32 contiguous bytes of codes and 4 scale bytes.
constexpr int kColTileRows = 128;
constexpr int kColTileCols = 64;

template <typename T, bool kSR, bool kRHT, bool kMX>
__global__ void __launch_bounds__(kColThreads) quantize_colwise_kernel(
    const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, const uint32_t* __restrict__ partials,
    int npartials, uint8_t* __restrict__ codes, int64_t ld_codes, ScaleOut so, float* amax_out, uint32_t* status,
    uint64_t seed, uint64_t rht_seed) {
    __shared__ uint32_t red[33];
    __shared__ __align__(16) T tile[kColTileRows][kColTileCols];
    TensorScales ts{};
    if constexpr (!kMX) {
        ts = reduce_partials(partials, npartials, amax_out, status, red);
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

    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t tile_id = ntiles - 1 - t;
        const int64_t tr = tile_id / tiles_c;
        const int64_t r0 = tr * kColTileRows, c0 = (tile_id - tr * tiles_c) * kColTileCols;
        // stage the tile (rows and columns beyond the tensor are not read)
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
            const int L = threadIdx.x + kColThreads * k;
            const int lr = L / kVecPerRow, seg = L % kVecPerRow;
            if (r0 + lr < rows && c0 + seg * V < cols)
                *reinterpret_cast<uint4*>(&tile[lr][seg * V]) =
                    __ldg(reinterpret_cast<const uint4*>(x + (r0 + lr) * ldx + c0 + seg * V));
        }
        __syncthreads();
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
                        const uint2 c0 = mx_encode16<kSR>(v0, bm, seed, i0, status, sb);
                        const uint2 c1 = mx_encode16<kSR>(v1, bm, seed, i0 + 16, status, sb);
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
                        uint2 c = quantize_block<kSR>(v, ts, seed, (uint64_t)oc * (uint64_t)rows + orow0 + 16 * b, sb);
                        w[2 * b] = c.x;
                        w[2 * b + 1] = c.y;
                        sbs |= sb << (8 * b);
                        nb = b + 1;
                    }
                }
            }
            if (nb > 0) {
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
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Pass 2, 16x16 blocks (weights, RTN): one E4M3 scale per 16x16 tile, codes
// for x (rowwise) and for x^T (colwise) from one read.  Under RTN the code of
// an element depends only on the element and its tile's scale, so the codes
// of x^T are the transpose of those of x.  A CTA covers 64 rows x 128
// columns (4 x 8 tiles); thread t takes row t/4 and columns 32*(t%4)..+31.
constexpr int k2dRows = 64;
constexpr int k2dCols = 128;

template <typename T>
__global__ void __launch_bounds__(k2dThreads) quantize_2d_kernel(
    const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, const uint32_t* __restrict__ partials,
    int npartials, uint8_t* __restrict__ codes_r, int64_t ld_r, ScaleOut so_r, float* amax_r,
    uint8_t* __restrict__ codes_c, int64_t ld_c, ScaleOut so_c, float* amax_c, uint32_t* status) {
    __shared__ uint32_t red[33];
    __shared__ float bam[k2dRows][k2dCols / 16];
    __shared__ float tile_r[k2dRows / 16][k2dCols / 16];
    __shared__ uint32_t tile_sb[k2dRows / 16][k2dCols / 16];
    __shared__ __align__(16) uint8_t ctile[k2dRows][k2dCols / 2];

    float* amax_out = amax_r ? amax_r : amax_c;
    const TensorScales ts = reduce_partials(partials, npartials, amax_out, status, red);
    if (amax_r && amax_c && blockIdx.x == 0 && threadIdx.x == 0) {
        amax_c[0] = ts.amax;
        amax_c[1] = ts.s_dec;
        amax_c[2] = ts.s_enc;
    }
    const int64_t tiles_r = (rows + k2dRows - 1) / k2dRows;
    const int64_t tiles_c = (cols + k2dCols - 1) / k2dCols;
    const int64_t ntiles = tiles_r * tiles_c;
    const int lr = threadIdx.x / 4, seg = threadIdx.x % 4;

    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t tile_id = ntiles - 1 - t;
        const int64_t trow = tile_id / tiles_c;
        const int64_t r0 = trow * k2dRows, c0 = (tile_id - trow * tiles_c) * k2dCols;
        const int64_t r = r0 + lr;
        float v[2][16];
        bool ok[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int64_t c = c0 + 32 * seg + 16 * b;
            ok[b] = (r < rows) && (c < cols);
            float m = 0.0f;
            if (ok[b]) {
                In<T>::load8(x + r * ldx + c, v[b]);
                In<T>::load8(x + r * ldx + c + 8, v[b] + 8);
#pragma unroll
                for (int k = 0; k < 16; ++k) m = fmaxf(m, fabsf(v[b][k]));
            }
            bam[lr][2 * seg + b] = m;
        }
        __syncthreads();
        if (threadIdx.x < (k2dRows / 16) * (k2dCols / 16)) {
            const int ti = threadIdx.x / (k2dCols / 16), tj = threadIdx.x % (k2dCols / 16);
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) m = fmaxf(m, bam[16 * ti + i][tj]);
            BlockScale bs = block_scale(m, ts.s_enc);
            if (!ts.finite) bs.sb = 0u;
            tile_sb[ti][tj] = bs.sb;
            tile_r[ti][tj] = bs.r;
        }
        __syncthreads();
        uint2 c[2];
        uint32_t sb[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int tj = 2 * seg + b;
            sb[b] = tile_sb[lr / 16][tj];
            c[b] = make_uint2(0u, 0u);
            if (ok[b] && sb[b] != 0u) {
                const float rm = tile_r[lr / 16][tj];
#pragma unroll
                for (int k = 0; k < 16; ++k) v[b][k] = __fmul_rn(v[b][k], rm);
                c[b] = encode16<false>(v[b], 0, 0);
            }
        }
        *reinterpret_cast<uint4*>(&ctile[lr][16 * seg]) = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
        if (codes_r) {
            uint8_t* dst = codes_r + r * ld_r + (c0 + 32 * seg) / 2;
            if (ok[0] && ok[1]) {
                *reinterpret_cast<uint4*>(dst) = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
            } else if (ok[0]) {
                *reinterpret_cast<uint2*>(dst) = c[0];
            }
#pragma unroll
            for (int b = 0; b < 2; ++b)
                if (ok[b]) so_r.p[so_r.offset(r, (c0 + 32 * seg) / 16 + b)] = (uint8_t)sb[b];
        }
        __syncthreads();
        if (codes_c) {
            // output row oc = c0 + cc of x^T; 32 rows of x per thread -> 16 bytes
            const int cc = threadIdx.x / 2, hh = threadIdx.x % 2;
            const int64_t oc = c0 + cc;
            const int64_t orow0 = r0 + 32 * hh;
            if (oc < cols && orow0 < rows) {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const uint32_t byte = ctile[32 * hh + i][cc / 2];
                    const uint32_t nib = (cc & 1) ? (byte >> 4) : (byte & 0xFu);
                    w[i / 8] |= nib << (4 * (i % 8));
                }
                uint8_t* dst = codes_c + oc * ld_c + orow0 / 2;
                const bool full = orow0 + 32 <= rows;
                if (full) {
                    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
                    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
                }
                const int tj = cc / 16;
                so_c.p[so_c.offset(oc, orow0 / 16)] = (uint8_t)tile_sb[2 * hh][tj];
                if (full) so_c.p[so_c.offset(oc, orow0 / 16 + 1)] = (uint8_t)tile_sb[2 * hh + 1][tj];
            }
        }
        __syncthreads();
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
                     uint32_t* partials, int grid, cudaStream_t s) {
    if (fp32)
        rht_amax_kernel<float><<<grid, kRhtAmaxThreads, 0, s>>>(static_cast<const float*>(x), rows, cols, ldx, rht_seed,
                                                             partials);
    else
        rht_amax_kernel<__nv_bfloat16><<<grid, kRhtAmaxThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(x), rows,
                                                                     cols, ldx, rht_seed, partials);
}

void launch_quantize_rowwise(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx,
                             const uint32_t* partials, int npartials, uint8_t* codes, int64_t ld_codes, ScaleOut so,
                             float* amax_out, uint32_t* status, bool sr, bool mx, uint64_t seed, bool rht,
                             uint64_t rht_seed, int grid, cudaStream_t s) {
#define NVFP4_ROW(T, SR, MX, RHT)                                                                               \
    quantize_rowwise_kernel<T, SR, MX, RHT><<<grid, kQuantThreads, 0, s>>>(                                    \
        static_cast<const T*>(x), rows, cols, ldx, partials, npartials, codes, ld_codes, so, amax_out, status, \
        seed, rht_seed)
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
#define NVFP4_COL(T, SR, RHT, MX)                                                                                    \
    quantize_colwise_kernel<T, SR, RHT, MX><<<grid, kColThreads, 0, s>>>(static_cast<const T*>(x), rows, cols, ldx,  \
                                                                         partials, npartials, codes, ld_codes, so,   \
                                                                         amax_out, status, seed, rht_seed)
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

int64_t tiles_2d(int64_t rows, int64_t cols) {
    return ((rows + k2dRows - 1) / k2dRows) * ((cols + k2dCols - 1) / k2dCols);
}

}  // namespace nvfp4

// Block-scaled NVFP4 GEMM on the sm_103a tensor cores (tcgen05 + TMEM).
//
//   C[m][n] = S_dec(A) S_dec(B) sum_kb sbA[m][kb] sbB[n][kb] sum_16 a[m][k] b[n][k]
//
// The blog "NVFP4 Trains with Precision of 16-Bit..." (Blackwell FP4 tensor
// cores; GEMM speed-up figure) and the paper page ("Pretraining Large
// Language Models with NVFP4", FP4 tensor-core throughput vs FP8 on GB300)
// put the linear layers' Fprop/Dgrad/Wgrad on block-scaled FP4 MMA with FP32
// accumulation; this kernel is that MMA.
//
// Structure (one persistent CTA per SM, 6 warps):
//   warp 0      TMA producer: A/B code tiles (128 rows x 128 bytes, 128-byte
//               swizzle) and the matching 2 KB scale atoms (bulk copies) into
//               a ring of smem stages, one mbarrier per stage.
//   warp 1      TMEM owner and MMA issuer: per stage, tcgen05.cp moves the
//               scale atoms to TMEM, then four
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
//               (M=128, N=128, K=64 each) accumulate into one of two TMEM
//               accumulators; tcgen05.commit releases the stage / signals
//               the epilogue.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (thread = row),
//               x alpha, convert, store; then release the accumulator.
// Every mbarrier wait is bounded: past the limit the waiter records
// NVFP4_ERR_TIMEOUT in the status word, raises a CTA-wide abort flag and all
// roles drain out to the final barrier, where TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "nvfp4_device.cuh"
#include "nvfp4_launch.h"

namespace nvfp4 {
namespace gemm {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 256;            // K elements per stage
constexpr int BKB = BK / 2;        // bytes per row per stage (= 128, the swizzle width)
constexpr int kStages = 6;
constexpr int kMmaK = 64;          // K per tcgen05.mma (FP4)
constexpr int kMmaPerStage = BK / kMmaK;
constexpr int kATileBytes = BM * BKB;      // 16 KB
constexpr int kBTileBytes = BN * BKB;      // 16 KB
constexpr int kSfTileBytes = 128 * BK / 16; // 2 KB: 128 rows x 16 scales
constexpr int kStageBytes = kATileBytes + kBTileBytes + 2 * kSfTileBytes;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = BN;          // fp32 accumulator columns per buffer
constexpr uint32_t kSfColsPerStage = 2 * kMmaPerStage * 4;  // SFA + SFB, 4 columns per MMA each
constexpr uint64_t kTimeoutNs = 4000000000ull;               // 4 s per wait

struct __align__(8) SharedState {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + (size_t)kStages * kStageBytes + sizeof(SharedState);

// ---- PTX wrappers ----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity; false on abort/timeout.
__device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, SharedState* ss, uint32_t* status) {
    uint64_t t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u) {
            if (*reinterpret_cast<volatile int*>(&ss->abort_flag)) return false;
            const uint64_t now = globaltimer();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kTimeoutNs) {
                atomicOr(status, kStatusTimeout);
                *reinterpret_cast<volatile int*>(&ss->abort_flag) = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start address, leading/stride
// byte offsets (>> 4), descriptor version 1 (bits 46-48), swizzle mode in
// bits 61-63 (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= (uint64_t)(swizzle & 7u) << 61;
    return d;
}

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B (format 1),
// K-major both, N >> 3 at bit 17, UE4M3 scales (bit 23 = 0), M >> 7 at
// bit 27, scale-factor data ids 0.
__host__ __device__ constexpr uint32_t instr_desc_nvf4(int m, int n) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 7) << 27);
}

__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
        "}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// ---- the kernel ----------------------------------------------------------------
struct Params {
    const uint8_t* a_scales;
    const uint8_t* b_scales;
    const float* a_amax;
    const float* b_amax;
    void* c;
    int64_t ldc;
    int M, N, K;
    int num_m, num_n, num_k;  // tiles
    int n_katoms;             // scale atoms per 128-row group
    int out_fp32;
    uint32_t* status;
};

__global__ void __launch_bounds__(kThreads, 1)
    nvf4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + kStages * kATileBytes;
    uint8_t* sSFA = sB + kStages * kBTileBytes;
    uint8_t* sSFB = sSFA + kStages * kSfTileBytes;
    SharedState* ss = reinterpret_cast<SharedState*>(sSFB + kStages * kSfTileBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_tiles = p.num_m * p.num_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ss->full[s], 1);
            mbar_init(&ss->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&ss->acc_full[a], 1);
            mbar_init(&ss->acc_empty[a], kEpiWarps);
        }
        ss->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_a) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_b) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&ss->tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ss->tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            uint32_t it = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                const int mb = tile % p.num_m, nb = tile / p.num_m;
                const uint8_t* sfa_src = p.a_scales + (size_t)mb * p.n_katoms * 512;
                const uint8_t* sfb_src = p.b_scales + (size_t)nb * p.n_katoms * 512;
                bool ok = true;
                for (int kt = 0; kt < p.num_k; ++kt, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(&ss->empty[s], ph ^ 1u, ss, p.status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&ss->full[s], kStageBytes);
                    tma_load_2d(sA + s * kATileBytes, &tmap_a, &ss->full[s], kt * BKB, mb * BM);
                    tma_load_2d(sB + s * kBTileBytes, &tmap_b, &ss->full[s], kt * BKB, nb * BN);
                    bulk_load(sSFA + s * kSfTileBytes, sfa_src + (size_t)kt * kSfTileBytes, kSfTileBytes,
                              &ss->full[s]);
                    bulk_load(sSFB + s * kSfTileBytes, sfb_src + (size_t)kt * kSfTileBytes, kSfTileBytes,
                              &ss->full[s]);
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = instr_desc_nvf4(BM, BN);
            const uint32_t sf_base = tmem_base + 2 * kAccCols;
            uint32_t it = 0;
            uint32_t tc = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tc) {
                const uint32_t a = tc & 1u;
                const uint32_t aph = (tc >> 1) & 1u;
                if (!mbar_wait(&ss->acc_empty[a], aph ^ 1u, ss, p.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + a * kAccCols;
                bool ok = true;
                for (int kt = 0; kt < p.num_k; ++kt, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(&ss->full[s], ph, ss, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sfa_t = sf_base + s * kSfColsPerStage;
                    const uint32_t sfb_t = sfa_t + kMmaPerStage * 4;
                    const uint32_t sfa_s = smem_u32(sSFA + s * kSfTileBytes);
                    const uint32_t sfb_s = smem_u32(sSFB + s * kSfTileBytes);
#pragma unroll
                    for (int j = 0; j < kMmaPerStage; ++j) {
                        tmem_cp_32x128b_x4(sfa_t + 4 * j, smem_desc(sfa_s + 512 * j, 0, 128, 0));
                        tmem_cp_32x128b_x4(sfb_t + 4 * j, smem_desc(sfb_s + 512 * j, 0, 128, 0));
                    }
                    const uint32_t a_s = smem_u32(sA + s * kATileBytes);
                    const uint32_t b_s = smem_u32(sB + s * kBTileBytes);
#pragma unroll
                    for (int j = 0; j < kMmaPerStage; ++j) {
                        const uint64_t adesc = smem_desc(a_s + 32 * j, 16, 1024, 2);
                        const uint64_t bdesc = smem_desc(b_s + 32 * j, 16, 1024, 2);
                        mma_nvf4(d_tmem, adesc, bdesc, idesc, sfa_t + 4 * j, sfb_t + 4 * j,
                                 (kt > 0 || j > 0) ? 1u : 0u);
                    }
                    mma_commit(&ss->empty[s]);
                }
                if (!ok) break;
                mma_commit(&ss->acc_full[a]);
            }
        }
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const float alpha = __fmul_rn(__ldg(p.a_amax + 1), __ldg(p.b_amax + 1));
        uint32_t tc = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tc) {
            const int mb = tile % p.num_m, nb = tile / p.num_m;
            const uint32_t a = tc & 1u;
            const uint32_t aph = (tc >> 1) & 1u;
            const bool ok = mbar_wait(&ss->acc_full[a], aph, ss, p.status);
            __syncwarp();
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            const int row = mb * BM + q * 32 + lane;
            const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + a * kAccCols;
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + ch * 32, r);
                const int col0 = nb * BN + ch * 32;
                if (row < p.M) {
                    if (p.out_fp32) {
                        float* dst = static_cast<float*>(p.c) + (int64_t)row * p.ldc + col0;
                        if (col0 + 32 <= p.N) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4)
                                *reinterpret_cast<float4*>(dst + j) =
                                    make_float4(__fmul_rn(__uint_as_float(r[j]), alpha),
                                                __fmul_rn(__uint_as_float(r[j + 1]), alpha),
                                                __fmul_rn(__uint_as_float(r[j + 2]), alpha),
                                                __fmul_rn(__uint_as_float(r[j + 3]), alpha));
                        } else {
                            for (int j = 0; j < 32 && col0 + j < p.N; ++j)
                                dst[j] = __fmul_rn(__uint_as_float(r[j]), alpha);
                        }
                    } else {
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.c) + (int64_t)row * p.ldc + col0;
                        if (col0 + 32 <= p.N) {
#pragma unroll
                            for (int j = 0; j < 32; j += 8) {
                                uint4 v;
                                v.x = pack_bf16x2(__fmul_rn(__uint_as_float(r[j]), alpha),
                                                  __fmul_rn(__uint_as_float(r[j + 1]), alpha));
                                v.y = pack_bf16x2(__fmul_rn(__uint_as_float(r[j + 2]), alpha),
                                                  __fmul_rn(__uint_as_float(r[j + 3]), alpha));
                                v.z = pack_bf16x2(__fmul_rn(__uint_as_float(r[j + 4]), alpha),
                                                  __fmul_rn(__uint_as_float(r[j + 5]), alpha));
                                v.w = pack_bf16x2(__fmul_rn(__uint_as_float(r[j + 6]), alpha),
                                                  __fmul_rn(__uint_as_float(r[j + 7]), alpha));
                                *reinterpret_cast<uint4*>(dst + j) = v;
                            }
                        } else {
                            for (int j = 0; j < 32 && col0 + j < p.N; ++j)
                                dst[j] = __float2bfloat16_rn(__fmul_rn(__uint_as_float(r[j]), alpha));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ss->acc_empty[a]);
        }
    }

    // Drain: every role reaches this barrier, then warp 1 frees TMEM.
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols));
    }
}

// ---- host side ---------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encoder(const char** msg) {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) {
        *msg = "cuTensorMapEncodeTiled is not available from the driver";
        return 1;
    }
    return 0;
}

// 2D tensor map over a [rows][row_bytes] byte matrix with row stride ld,
// box 128 x 128 bytes, 128-byte swizzle, zero fill outside the matrix.
int make_code_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, int64_t ld, const char** msg) {
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {(cuuint32_t)BKB, (cuuint32_t)BM};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *msg = "cuTensorMapEncodeTiled failed";
        return 1;
    }
    return 0;
}

bool g_attr_set[64] = {};
std::mutex g_attr_mu;

}  // namespace gemm

int launch_gemm(const GemmArgs& g, cudaStream_t s, const char** msg) {
    using namespace gemm;
    if (get_encoder(msg)) return 1;
    if (g.M > INT32_MAX || g.N > INT32_MAX || g.K > INT32_MAX) {
        *msg = "dimension exceeds 2^31";
        return -1;
    }
    CUtensorMap ta, tb;
    if (make_code_map(&ta, g.a_codes, g.M, g.K / 2, g.lda, msg)) return 1;
    if (make_code_map(&tb, g.b_codes, g.N, g.K / 2, g.ldb, msg)) return 1;
    {
        int dev = 0;
        cudaGetDevice(&dev);
        std::lock_guard<std::mutex> lk(g_attr_mu);
        if (dev >= 0 && dev < 64 && !g_attr_set[dev]) {
            cudaError_t e =
                cudaFuncSetAttribute(nvf4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
            if (e != cudaSuccess) return (int)e;
            g_attr_set[dev] = true;
        }
    }
    Params p;
    p.a_scales = g.a_scales;
    p.b_scales = g.b_scales;
    p.a_amax = g.a_amax;
    p.b_amax = g.b_amax;
    p.c = g.c;
    p.ldc = g.ldc;
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.num_m = (int)((g.M + BM - 1) / BM);
    p.num_n = (int)((g.N + BN - 1) / BN);
    p.num_k = (int)((g.K + BK - 1) / BK);
    p.n_katoms = (int)(4 * ((g.K + 255) / 256));
    p.out_fp32 = g.out_fp32;
    p.status = g.status;
    const int tiles = p.num_m * p.num_n;
    const int grid = tiles < g.num_sms ? tiles : g.num_sms;
    nvf4_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(ta, tb, p);
    return (int)cudaGetLastError();
}

}  // namespace nvfp4

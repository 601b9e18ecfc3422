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
// Tile 128 x 384 (M x N), K staged 256 at a time; one persistent CTA per SM,
// 16 warps in four warpgroups.  The tile's N is computed by two independent
// accumulation chains: chain 0 takes B rows 0-255 (N = 256 MMAs into TMEM
// columns 0-255), chain 1 rows 256-383 (N = 128 into columns 256-383), each
// issued by its own warp.  Back-to-back MMAs into one accumulator wait on
// each other (about 275 cycles per M=128 N=256 K=64 MMA on this part, against
// about 182 cycles of tensor-pipe time), so two chains keep the pipe busier
// than one; 384 accumulator columns leave TMEM room for two scale slots.
//   warp 0      producer: A (128 rows) and B (three 128-row boxes) code tiles
//               by TMA (128-byte swizzle) into a 3-stage smem ring (64 KB
//               per stage).
//   warp 2      scale producer: the stage's block scales (MMA layout:
//               contiguous 2 KB runs of 512-byte atoms, A's 128 rows and B's
//               three 128-row groups) by bulk copies into a 2-slot ring of its
//               own, whose slots free as soon as the scale writers have read
//               them.
//   warp 1      TMEM owner and chain-0 MMA issuer; warp 3 chain-1 issuer:
//               four tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
//               (M=128, K=64) per stage each.
//   warps 4-7   scale-factor writers, one per TMEM lane quarter: they read
//               the stage's scale atoms from smem and write them into one of
//               two TMEM scale slots with tcgen05.st (layout at scale_role).
//               Scale copies through the tensor pipe (tcgen05.cp) would
//               serialize with the MMAs, and a TMA box of 256 rows x 16 bytes
//               costs about one cycle per row of the SM's copy bandwidth, so
//               the scales come as long contiguous runs.
//   warps 8-15  epilogue: two warps per lane quarter drain chain 1 (64
//               columns each) and release it, store it, then drain chain 0
//               (128 columns each, 64 at a time, released after the second
//               load); stores scale by alpha, convert and go through two 1 KB
//               swizzled smem staging tiles per warp with TMA tensor stores.
// Registers: at most 128 per thread (512 threads fill the register file).
// The epilogue keeps at most 64 accumulator words live and takes each TMEM
// load together with its wait, so nothing is spilled: a spill of registers
// that a tcgen05.ld has not finished writing made repeated launches differ.
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
constexpr int BN = 384;            // tile N: chain 0 (256) + chain 1 (128)
constexpr int kChain0N = 256;
constexpr int kChain1N = BN - kChain0N;
constexpr int kBBoxRows = 128;     // B rows per TMA box (a box has at most 256 rows)
constexpr int kBGroups = BN / 128; // 128-row groups of B per tile
constexpr int BK = 256;            // K elements per stage
constexpr int BKB = BK / 2;        // bytes per row per stage (= 128, the swizzle width)
constexpr int kStages = 3;         // code-tile ring (smem)
constexpr int kSfSlots = 2;        // scale-atom ring (smem)
constexpr int kTmemSlots = 2;      // scale-factor slots in TMEM
constexpr int kChains = 2;
constexpr int kMmaK = 64;          // K per tcgen05.mma (FP4)
constexpr int kMmaPerStage = BK / kMmaK;
constexpr int kATileBytes = BM * BKB;      // 16 KB
constexpr int kBTileBytes = BN * BKB;      // 48 KB (three 128-row boxes)
constexpr int kSfAtomBytes = 512;           // 128 rows x 4 K blocks (MMA scale layout)
constexpr int kSfRunBytes = 4 * kSfAtomBytes;  // one 128-row group, one stage (16 K blocks)
constexpr int kSfStageBytes = (1 + kBGroups) * kSfRunBytes; // A, then B's three 128-row groups
constexpr int kStageBytes = kATileBytes + kBTileBytes;
constexpr int kThreads = 512;
constexpr int kEpiWarps = 8;
constexpr int kSfWarps = 4;
constexpr int kStagingBytes = 32 * 32;     // one staging tile: 32 rows x 32 bytes
constexpr int kStagingBufs = 2;            // per epilogue warp, filled as a pair
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = BN;          // fp32 accumulator columns (chain 0: 0-255, chain 1: 256-383)
constexpr uint32_t kSfaCols = kMmaPerStage * 4;         // 4 columns per MMA
constexpr uint32_t kSfb0Cols = kMmaPerStage * 8;        // chain 0, N = 256: two 128-row groups per MMA
constexpr uint32_t kSfb1Cols = kMmaPerStage * 4;        // chain 1, N = 128: one group per MMA
constexpr uint32_t kSfColsPerSlot = kSfaCols + kSfb0Cols + kSfb1Cols;
constexpr uint64_t kTimeoutNs = 4000000000ull;          // 4 s per wait
static_assert(kAccCols + kTmemSlots * kSfColsPerSlot <= kTmemCols, "TMEM budget");
static_assert(kSfColsPerSlot % 4 == 0 && kSfaCols % 4 == 0 && kSfb0Cols % 4 == 0, "TMEM columns 4-aligned");

struct __align__(8) SharedState {
    uint64_t full[kStages];             // A/B tiles landed (TMA transaction count)
    uint64_t empty[kStages];            // MMAs of the stage done (tcgen05.commit, both chains)
    uint64_t sf_in[kSfSlots];           // scale atoms of the slot landed (bulk-copy transaction count)
    uint64_t sf_free[kSfSlots];         // scale atoms of the slot read out of smem (4 scale warps)
    uint64_t sf_full[kTmemSlots];       // scales written to the TMEM slot (4 scale warps)
    uint64_t tmem_free[kTmemSlots];     // MMAs reading the TMEM slot done (tcgen05.commit, both chains)
    uint64_t acc_full[kChains];         // chain's accumulator complete (tcgen05.commit)
    uint64_t acc_empty[kChains];        // chain's accumulator drained (8 epilogue warps)
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + (size_t)kStages * kStageBytes +
                              (size_t)kSfSlots * kSfStageBytes + (size_t)kEpiWarps * kStagingBufs * kStagingBytes +
                              sizeof(SharedState);
static_assert(kSmemBytes <= 232448, "shared memory budget");

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
// K-major both, N >> 3 at bit 17, scale type at bit 23 (0 = UE4M3 for
// NVFP4, 1 = UE8M0 for MXFP4), M >> 7 at bit 27, scale-factor data ids 0
// (with scale_vec::2X the MMA reads bytes 0 and 1 of each scale word).
__host__ __device__ constexpr uint32_t instr_desc_nvf4(int m, int n, bool ue8m0) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((ue8m0 ? 1u : 0u) << 23) |
           ((uint32_t)(m >> 7) << 27);
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

// BF16 operands (the high-precision fallback GEMM): kind::f16, K = 16 per
// instruction, FP32 accumulation.  Instruction descriptor: D = F32 (bits
// 4-5 = 1), A = B = BF16 (bits 7-9 and 10-12 = 1), both K-major, N >> 3 at
// bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t instr_desc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// MXFP4: two UE8M0 scales per row per K = 64 (32-element blocks).
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
        "}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// A bounded wait taken by every lane of a warp, returning the warp's verdict.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, SharedState* ss, uint32_t* status) {
    const bool ok = mbar_wait(bar, parity, ss, status);
    __syncwarp();
    return __all_sync(0xFFFFFFFFu, ok);
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}

// The same tile added element-wise into global memory (FP32 adds, done by
// the memory system): C += tile, for accumulating into an FP32 gradient.
__device__ __forceinline__ void tma_add_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     map),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// 64 accumulator columns of the warp's 32 lanes, returned only once the
// load has completed: the load and its wait are one statement, so no use of
// the registers (a spill included) can be placed between them.
__device__ __forceinline__ void tmem_ld_x64_sync(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Contiguous global -> shared copy (16-byte aligned, size a multiple of 16)
// completing on an mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---- the kernel ----------------------------------------------------------------
struct Params {
    const uint8_t* a_scales;  // MMA layout (512-byte atoms), rows padded to 128
    const uint8_t* b_scales;
    const float* a_amax;
    const float* b_amax;
    int M, N, K;
    int num_m, num_n, num_k;  // tiles
    int n_katoms;             // atoms per 128-row group: 4 * ceil(K / 256)
    int b_groups;             // 128-row groups of B: ceil(N / 128)
    int out_fp32;
    int accumulate;           // FP32 output added into C instead of stored
    int mx;                   // MXFP4 operands (UE8M0 scales, 32-element blocks)
    int bf16;                 // BF16 operands: no scales, 64 K elements per stage, alpha = 1
    uint32_t* status;
};

// Tile schedule: CTA c takes tiles c, c + gridDim.x, ... with M fastest.
struct Sched {
    int num_tiles;
    __device__ explicit Sched(const Params& p) { num_tiles = p.num_m * p.num_n; }
    __device__ int count() const {
        return (int)blockIdx.x < num_tiles ? (num_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    }
    __device__ void tile(int i, const Params& p, int& mb, int& nb) const {
        const int t = (int)blockIdx.x + i * (int)gridDim.x;
        nb = t / p.num_m;
        mb = t - nb * p.num_m;
    }
};

__device__ __forceinline__ void producer_role(const CUtensorMap* tmap_a, const CUtensorMap* tmap_b, const Params& p,
                                              SharedState* ss, uint8_t* sA, uint8_t* sB) {
    const Sched S(p);
    uint32_t it = 0;
    for (int i = 0; i < S.count(); ++i) {
        int mb, nb;
        S.tile(i, p, mb, nb);
        for (int kt = 0; kt < p.num_k; ++kt, ++it) {
            const int s = it % kStages;
            const uint32_t ph = (it / kStages) & 1u;
            if (!mbar_wait(&ss->empty[s], ph ^ 1u, ss, p.status)) return;
            // every box counts in full: rows past the matrix arrive as zeros
            mbar_arrive_expect_tx(&ss->full[s], kATileBytes + kBTileBytes);
            // a stage is 128 bytes of every row: 256 FP4 codes or 64 bf16 values
            const int kx = kt * (p.bf16 ? 64 : BKB);
            tma_load_2d(sA + s * kATileBytes, tmap_a, &ss->full[s], kx, mb * BM);
#pragma unroll
            for (int g = 0; g < kBGroups; ++g)
                tma_load_2d(sB + s * kBTileBytes + g * kBBoxRows * BKB, tmap_b, &ss->full[s], kx,
                            nb * BN + g * kBBoxRows);
        }
    }
}

__device__ __forceinline__ void scale_producer_role(const Params& p, SharedState* ss, uint8_t* sSf) {
    const Sched S(p);
    uint32_t it = 0;
    for (int i = 0; i < S.count(); ++i) {
        int mb, nb;
        S.tile(i, p, mb, nb);
        // B's 128-row groups of the tile that exist (the scale buffer has none past them)
        const int ng = min(kBGroups, p.b_groups - kBGroups * nb);
        for (int kt = 0; kt < p.num_k; ++kt, ++it) {
            const int r = it % kSfSlots;
            const uint32_t ph = (it / kSfSlots) & 1u;
            if (!mbar_wait(&ss->sf_free[r], ph ^ 1u, ss, p.status)) return;
            uint8_t* sf = sSf + r * kSfStageBytes;
            mbar_arrive_expect_tx(&ss->sf_in[r], (1 + ng) * kSfRunBytes);
            bulk_load(sf, p.a_scales + ((size_t)mb * p.n_katoms + 4 * kt) * kSfAtomBytes, kSfRunBytes, &ss->sf_in[r]);
            for (int g = 0; g < ng; ++g)
                bulk_load(sf + (1 + g) * kSfRunBytes,
                          p.b_scales + ((size_t)(kBGroups * nb + g) * p.n_katoms + 4 * kt) * kSfAtomBytes,
                          kSfRunBytes, &ss->sf_in[r]);
        }
    }
}

// Operand kinds of the MMA loop.  The loop is instantiated once per kind: a
// run-time choice between the MMA forms inside the loop slowed the issue of
// every MMA (0.40 -> 0.63 ms at 8192x20480x5120).
enum MmaKind { kNvf4 = 0, kMxf4 = 1, kBf16 = 2 };

// One accumulation chain: chain 0 multiplies A by B rows 0-255 of the tile
// into TMEM columns 0-255, chain 1 by rows 256-383 into columns 256-383.  Both
// wait for the same stages and scale slots and commit to the same "empty" and
// "TMEM slot free" barriers (two arrivals each).
template <int kKind>
__device__ __forceinline__ void mma_loop(const Params& p, SharedState* ss, uint8_t* sA, uint8_t* sB,
                                         uint32_t tmem_base, int chain) {
    const Sched S(p);
    const int n = chain ? kChain1N : kChain0N;
    const uint32_t idesc = kKind == kBf16 ? instr_desc_bf16(BM, n) : instr_desc_nvf4(BM, n, kKind == kMxf4);
    const uint32_t d_tmem = tmem_base + (chain ? (uint32_t)kChain0N : 0u);
    const uint32_t b_off = chain ? (uint32_t)(kChain0N * BKB) : 0u;  // the chain's first B row in the stage
    const uint32_t sfb_off = chain ? kSfaCols + kSfb0Cols : kSfaCols;
    const uint32_t sfb_step = chain ? 4u : 8u;                       // scale columns per MMA
    const uint32_t sf_base = tmem_base + kAccCols;
    uint32_t it = 0, tc = 0;
    for (int i = 0; i < S.count(); ++i, ++tc) {
        if (!mbar_wait(&ss->acc_empty[chain], (tc & 1u) ^ 1u, ss, p.status)) return;
        tc_fence_after();
        for (int kt = 0; kt < p.num_k; ++kt, ++it) {
            const int s = it % kStages;
            const uint32_t ph = (it / kStages) & 1u;
            const int ts = it % kTmemSlots;
            if (!mbar_wait(&ss->full[s], ph, ss, p.status) ||
                (kKind != kBf16 && !mbar_wait(&ss->sf_full[ts], (it / kTmemSlots) & 1u, ss, p.status)))
                return;
            tc_fence_after();
            const uint32_t sfa_t = sf_base + ts * kSfColsPerSlot;
            const uint32_t sfb_t = sfa_t + sfb_off;
            const uint32_t a_s = smem_u32(sA + s * kATileBytes);
            const uint32_t b_s = smem_u32(sB + s * kBTileBytes) + b_off;
#pragma unroll
            for (int j = 0; j < kMmaPerStage; ++j) {
                const uint64_t adesc = smem_desc(a_s + 32 * j, 16, 1024, 2);
                const uint64_t bdesc = smem_desc(b_s + 32 * j, 16, 1024, 2);
                const uint32_t acc = (kt > 0 || j > 0) ? 1u : 0u;
                if constexpr (kKind == kBf16)
                    mma_bf16(d_tmem, adesc, bdesc, idesc, acc);
                else if constexpr (kKind == kMxf4)
                    mma_mxf4(d_tmem, adesc, bdesc, idesc, sfa_t + 4 * j, sfb_t + sfb_step * j, acc);
                else
                    mma_nvf4(d_tmem, adesc, bdesc, idesc, sfa_t + 4 * j, sfb_t + sfb_step * j, acc);
            }
            mma_commit(&ss->empty[s]);
            if constexpr (kKind != kBf16) mma_commit(&ss->tmem_free[ts]);
        }
        mma_commit(&ss->acc_full[chain]);
    }
}

__device__ __forceinline__ void mma_role(const Params& p, SharedState* ss, uint8_t* sA, uint8_t* sB,
                                         uint32_t tmem_base, int chain) {
    if (p.bf16) mma_loop<kBf16>(p, ss, sA, sB, tmem_base, chain);
    else if (p.mx) mma_loop<kMxf4>(p, ss, sA, sB, tmem_base, chain);
    else mma_loop<kNvf4>(p, ss, sA, sB, tmem_base, chain);
}

// Scale-factor TMEM layout read by one MMA (measured on the hardware):
//   A (128 rows): row r at lane r, column base + r/32 -- each lane quarter
//     reads only its own rows, so lane r holds only its own row's word;
//   B (N rows): every lane quarter reads all of B: row n at lane
//     32q + n%32, column base + n/32, the same in all four quarters.
// Writer warp q (lanes 32q .. 32q+31 of TMEM), lane l: A row 32q + l, and B
// rows 32c + l of the tile.  Per stage and slot, MMA j reads A words at
// columns 4j..4j+3 (the lane's word is written into all four), chain 0's B
// words (tile rows 0-255) at 16 + 8j .. 16 + 8j + 7 and chain 1's (rows
// 256-383) at 48 + 4j .. 48 + 4j + 3.  In smem, atom j of a 128-row group
// holds row 32c + l's four scales of MMA j at byte 16 l + 4 c, so lane l
// reads A's word with one 4-byte load per MMA and four B words (c = 0..3 of
// a group) with one 16-byte load per group and MMA.
__device__ __forceinline__ void scale_role(const Params& p, SharedState* ss, const uint8_t* sSf, uint32_t tmem_base,
                                           int q, int lane) {
    const Sched S(p);
    const uint32_t sf_base = tmem_base + kAccCols;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    uint32_t it = 0;
    for (int i = 0; i < S.count(); ++i) {
        int mb, nb;
        S.tile(i, p, mb, nb);
        const int ng = min(kBGroups, p.b_groups - kBGroups * nb);  // B groups that exist
        for (int kt = 0; kt < p.num_k; ++kt, ++it) {
            const int r = it % kSfSlots;
            const int ts = it % kTmemSlots;
            if (!warp_wait(&ss->sf_in[r], (it / kSfSlots) & 1u, ss, p.status)) return;
            const uint8_t* sf = sSf + r * kSfStageBytes + lane * 16;
            uint32_t wa[kMmaPerStage];
            uint4 wb[kBGroups][kMmaPerStage];
#pragma unroll
            for (int j = 0; j < kMmaPerStage; ++j) {
                wa[j] = *reinterpret_cast<const uint32_t*>(sf + j * kSfAtomBytes + 4 * q);
#pragma unroll
                for (int g = 0; g < kBGroups; ++g)
                    wb[g][j] = g < ng ? *reinterpret_cast<const uint4*>(sf + (1 + g) * kSfRunBytes + j * kSfAtomBytes)
                                      : make_uint4(0u, 0u, 0u, 0u);
            }
            if (p.mx) {
                // MXFP4 stores each 32-element block's scale in both of its
                // 16-element slots; scale_vec::2X wants the two blocks of an
                // MMA in bytes 0 and 1 of the word
#pragma unroll
                for (int j = 0; j < kMmaPerStage; ++j) {
                    wa[j] = __byte_perm(wa[j], 0u, 0x4420);
#pragma unroll
                    for (int g = 0; g < kBGroups; ++g)
                        wb[g][j] = make_uint4(__byte_perm(wb[g][j].x, 0u, 0x4420), __byte_perm(wb[g][j].y, 0u, 0x4420),
                                              __byte_perm(wb[g][j].z, 0u, 0x4420), __byte_perm(wb[g][j].w, 0u, 0x4420));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ss->sf_free[r]);
            // the TMEM slot is free once both chains' MMAs that read it
            // kTmemSlots stages ago are done
            if (!warp_wait(&ss->tmem_free[ts], ((it / kTmemSlots) & 1u) ^ 1u, ss, p.status)) return;
            tc_fence_after();
            const uint32_t col = lane_addr + sf_base + ts * kSfColsPerSlot;
            const uint32_t va[16] = {wa[0], wa[0], wa[0], wa[0], wa[1], wa[1], wa[1], wa[1],
                                     wa[2], wa[2], wa[2], wa[2], wa[3], wa[3], wa[3], wa[3]};
            tmem_st_x16(col, va);
            // chain 0 (B rows 0-255): 8 columns per MMA, groups 0 and 1
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // MMAs 2h and 2h + 1
                uint32_t vb[16];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint4 lo = wb[0][2 * h + u], hi = wb[1][2 * h + u];
                    vb[8 * u + 0] = lo.x; vb[8 * u + 1] = lo.y; vb[8 * u + 2] = lo.z; vb[8 * u + 3] = lo.w;
                    vb[8 * u + 4] = hi.x; vb[8 * u + 5] = hi.y; vb[8 * u + 6] = hi.z; vb[8 * u + 7] = hi.w;
                }
                tmem_st_x16(col + kSfaCols + 16 * h, vb);
            }
            // chain 1 (B rows 256-383): 4 columns per MMA, group 2
            {
                uint32_t vc[16];
#pragma unroll
                for (int j = 0; j < kMmaPerStage; ++j) {
                    vc[4 * j + 0] = wb[2][j].x; vc[4 * j + 1] = wb[2][j].y;
                    vc[4 * j + 2] = wb[2][j].z; vc[4 * j + 3] = wb[2][j].w;
                }
                tmem_st_x16(col + kSfaCols + kSfb0Cols, vc);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ss->sf_full[ts]);
        }
    }
}

// Stores NC accumulator columns of the lane's row (this warp's 32 rows of
// C, starting at column col0): scale by alpha, convert, and write through
// the warp's two 32 x 32-byte staging tiles (32-byte swizzle: 16-byte chunk
// j of row r at position j ^ ((r/4) % 2)), one TMA store per 32 bytes of
// every row.  Chunks go in pairs, one per tile: both are converted in
// registers, the warp waits until its earlier stores have finished reading
// both tiles, writes them, fences once and commits the two stores as one
// bulk group.  NC / 8 (fp32) and NC / 16 (bf16) are even.
template <int NC>
__device__ __forceinline__ void store_cols(const CUtensorMap* tmap_c, const Params& p, const uint32_t (&acc)[NC],
                                           float alpha, uint8_t* stage, int sw, int lane, int col0, int y,
                                           bool rows_in) {
    constexpr int kPerChunk32 = 8;  // fp32 columns per 32-byte row
    constexpr int kPerChunk16 = 16; // bf16 columns per 32-byte row
    static_assert(kStagingBufs == 2 && (NC / kPerChunk32) % 2 == 0 && (NC / kPerChunk16) % 2 == 0,
                  "chunks are stored in pairs");
    const bool f32 = p.out_fp32 != 0;
    const int per = f32 ? kPerChunk32 : kPerChunk16;
#pragma unroll
    for (int pc = 0; pc < NC / kPerChunk32 / 2; ++pc) {
        const int c2 = 2 * pc;
        if (!f32 && c2 >= NC / kPerChunk16) break;
        uint4 v[2][2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int c = c2 + b;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if (f32) {
                    const uint32_t* a = acc + 8 * c + 4 * j;
                    v[b][j] = make_uint4(__float_as_uint(__fmul_rn(__uint_as_float(a[0]), alpha)),
                                         __float_as_uint(__fmul_rn(__uint_as_float(a[1]), alpha)),
                                         __float_as_uint(__fmul_rn(__uint_as_float(a[2]), alpha)),
                                         __float_as_uint(__fmul_rn(__uint_as_float(a[3]), alpha)));
                } else {
                    const uint32_t* a = acc + (16 * c + 8 * j) % NC;  // c < NC / 16 here
                    v[b][j] = make_uint4(
                        pack_bf16x2(__fmul_rn(__uint_as_float(a[0]), alpha), __fmul_rn(__uint_as_float(a[1]), alpha)),
                        pack_bf16x2(__fmul_rn(__uint_as_float(a[2]), alpha), __fmul_rn(__uint_as_float(a[3]), alpha)),
                        pack_bf16x2(__fmul_rn(__uint_as_float(a[4]), alpha), __fmul_rn(__uint_as_float(a[5]), alpha)),
                        pack_bf16x2(__fmul_rn(__uint_as_float(a[6]), alpha), __fmul_rn(__uint_as_float(a[7]), alpha)));
                }
            }
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            uint8_t* row_base = stage + b * kStagingBytes + lane * 32;
#pragma unroll
            for (int j = 0; j < 2; ++j) *reinterpret_cast<uint4*>(row_base + ((j ^ sw) << 4)) = v[b][j];
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int x = col0 + per * (c2 + b);
                if (rows_in && x < p.N) {
                    if (p.accumulate) tma_add_2d(tmap_c, stage + b * kStagingBytes, x, y);
                    else tma_store_2d(tmap_c, stage + b * kStagingBytes, x, y);
                }
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
    }
}

// Epilogue warp e: lane quarter q = warp % 4, half h = e / 4.  Per tile it
// drains chain 1 first (columns 256 + 64h .. +63, released before they are
// stored), then chain 0 (columns 128h .. +127, 64 at a time, released after
// the second load): at most 64 accumulator words are live at a time, so the
// epilogue needs no spills.
__device__ __forceinline__ void epilogue_role(const CUtensorMap* tmap_c, const Params& p, SharedState* ss,
                                              uint8_t* stage, uint32_t tmem_base, int q, int h, int lane) {
    const Sched S(p);
    const float alpha = p.bf16 ? 1.0f : __fmul_rn(__ldg(p.a_amax + 1), __ldg(p.b_amax + 1));
    const uint32_t t_lane = tmem_base + ((uint32_t)(32 * q) << 16);
    const int sw = (lane >> 2) & 1;
    uint32_t tc = 0;
    for (int i = 0; i < S.count(); ++i, ++tc) {
        int mb, nb;
        S.tile(i, p, mb, nb);
        const int y = mb * BM + 32 * q;
        const bool rows_in = y < p.M;
        {
            if (!warp_wait(&ss->acc_full[1], tc & 1u, ss, p.status)) break;
            tc_fence_after();
            uint32_t acc1[kChain1N / 2];
            static_assert(kChain1N / 2 == 64, "one 64-column load per warp");
            tmem_ld_x64_sync(t_lane + (uint32_t)(kChain0N + (kChain1N / 2) * h), acc1);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ss->acc_empty[1]);
            store_cols<kChain1N / 2>(tmap_c, p, acc1, alpha, stage, sw, lane,
                                     nb * BN + kChain0N + (kChain1N / 2) * h, y, rows_in);
        }
        {
            // chain 0 in two 64-column halves: the first is stored before the
            // second is loaded, so at most 64 accumulator words are live and
            // none has to be spilled
            if (!warp_wait(&ss->acc_full[0], tc & 1u, ss, p.status)) break;
            tc_fence_after();
            constexpr int kHalf = kChain0N / 4;
            static_assert(kHalf == 64, "one 64-column load per half");
            const uint32_t t0 = t_lane + (uint32_t)((kChain0N / 2) * h);
            const int col0 = nb * BN + (kChain0N / 2) * h;
            {
                uint32_t acc0[kHalf];
                tmem_ld_x64_sync(t0, acc0);
                store_cols<kHalf>(tmap_c, p, acc0, alpha, stage, sw, lane, col0, y, rows_in);
            }
            {
                uint32_t acc0[kHalf];
                tmem_ld_x64_sync(t0 + kHalf, acc0);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ss->acc_empty[0]);
                store_cols<kHalf>(tmap_c, p, acc0, alpha, stage, sw, lane, col0 + kHalf, y, rows_in);
            }
        }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

__global__ void __launch_bounds__(kThreads, 1)
    nvf4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_c, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + kStages * kATileBytes;
    uint8_t* sSf = sB + kStages * kBTileBytes;
    uint8_t* sStage = sSf + kSfSlots * kSfStageBytes;
    SharedState* ss = reinterpret_cast<SharedState*>(sStage + kEpiWarps * kStagingBufs * kStagingBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ss->full[s], 1);
            mbar_init(&ss->empty[s], kChains);
        }
        for (int r = 0; r < kSfSlots; ++r) {
            mbar_init(&ss->sf_in[r], 1);
            mbar_init(&ss->sf_free[r], kSfWarps);
        }
        for (int t = 0; t < kTmemSlots; ++t) {
            mbar_init(&ss->sf_full[t], kSfWarps);
            mbar_init(&ss->tmem_free[t], kChains);
        }
        for (int c = 0; c < kChains; ++c) {
            mbar_init(&ss->acc_full[c], 1);
            mbar_init(&ss->acc_empty[c], kEpiWarps);
        }
        ss->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_a) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_b) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_c) : "memory");
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

    if (warp < 8) {
        if (warp == 0) {
            if (lane == 0) producer_role(&tmap_a, &tmap_b, p, ss, sA, sB);
        } else if (warp == 2) {
            if (lane == 0 && !p.bf16) scale_producer_role(p, ss, sSf);
        } else if (warp == 1 || warp == 3) {  // chain 0, chain 1
            if (lane == 0) mma_role(p, ss, sA, sB, tmem_base, warp == 3 ? 1 : 0);
        } else if (warp >= 4) {
            if (!p.bf16) scale_role(p, ss, sSf, tmem_base, warp & 3, lane);
        }
    } else {
        const int e = warp - 8;
        epilogue_role(&tmap_c, p, ss, sStage + e * kStagingBufs * kStagingBytes, tmem_base, warp & 3, e >> 2, lane);
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

// 2D tensor map over a [rows][row_elems] matrix with row stride ld_bytes:
// box box_x x box_y elements, zero fill outside.
int make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, int64_t rows, int64_t row_elems,
             int64_t ld_bytes, int box_x, int box_y, CUtensorMapSwizzle swizzle, const char** msg) {
    cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_x, (cuuint32_t)box_y};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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
    CUtensorMap ta, tb, tcm;
    if (make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.a_codes, g.M, g.K / 2, g.lda, BKB, BM,
                 CU_TENSOR_MAP_SWIZZLE_128B, msg))
        return 1;
    if (make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.b_codes, g.N, g.K / 2, g.ldb, BKB, kBBoxRows,
                 CU_TENSOR_MAP_SWIZZLE_128B, msg))
        return 1;
    if (g.out_fp32) {
        if (make_map(&tcm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.c, g.M, g.N, g.ldc * 4, 8, 32,
                     CU_TENSOR_MAP_SWIZZLE_32B, msg))
            return 1;
    } else {
        if (make_map(&tcm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.c, g.M, g.N, g.ldc * 2, 16, 32,
                     CU_TENSOR_MAP_SWIZZLE_32B, msg))
            return 1;
    }
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
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.num_m = (int)((g.M + BM - 1) / BM);
    p.num_n = (int)((g.N + BN - 1) / BN);
    p.num_k = (int)((g.K + BK - 1) / BK);
    p.n_katoms = 4 * p.num_k;
    p.b_groups = (int)((g.N + 127) / 128);
    p.out_fp32 = g.out_fp32;
    p.accumulate = g.accumulate;
    p.mx = g.mx;
    p.bf16 = 0;
    p.status = g.status;
    // persistent: one CTA per SM, at most one per tile
    const int64_t tiles = (int64_t)p.num_m * p.num_n;
    const int grid = (int)(tiles < g.num_sms ? tiles : g.num_sms);
    nvf4_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(ta, tb, tcm, p);
    return (int)cudaGetLastError();
}

int launch_gemm_bf16(const GemmBf16Args& g, cudaStream_t s, const char** msg) {
    using namespace gemm;
    if (get_encoder(msg)) return 1;
    if (g.M > INT32_MAX || g.N > INT32_MAX || g.K > INT32_MAX) {
        *msg = "dimension exceeds 2^31";
        return -1;
    }
    CUtensorMap ta, tb, tcm;
    if (make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.a, g.M, g.K, g.lda * 2, 64, BM,
                 CU_TENSOR_MAP_SWIZZLE_128B, msg) ||
        make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.b, g.N, g.K, g.ldb * 2, 64, kBBoxRows,
                 CU_TENSOR_MAP_SWIZZLE_128B, msg))
        return 1;
    if (g.out_fp32) {
        if (make_map(&tcm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.c, g.M, g.N, g.ldc * 4, 8, 32,
                     CU_TENSOR_MAP_SWIZZLE_32B, msg))
            return 1;
    } else {
        if (make_map(&tcm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.c, g.M, g.N, g.ldc * 2, 16, 32,
                     CU_TENSOR_MAP_SWIZZLE_32B, msg))
            return 1;
    }
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
    Params p = {};
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.num_m = (int)((g.M + BM - 1) / BM);
    p.num_n = (int)((g.N + BN - 1) / BN);
    p.num_k = (int)((g.K + 63) / 64);
    p.out_fp32 = g.out_fp32;
    p.accumulate = g.accumulate;
    p.bf16 = 1;
    p.status = g.status;
    const int64_t tiles = (int64_t)p.num_m * p.num_n;
    const int grid = (int)(tiles < g.num_sms ? tiles : g.num_sms);
    nvf4_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(ta, tb, tcm, p);
    return (int)cudaGetLastError();
}

}  // namespace nvfp4

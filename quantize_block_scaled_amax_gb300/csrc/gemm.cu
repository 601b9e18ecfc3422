// Block-scaled NVFP4 GEMM on the sm_103a tensor cores (tcgen05 + TMEM), on
// SM pairs (cta_group::2).
//
//   C[m][n] = S_dec(A) S_dec(B) sum_kb sbA[m][kb] sbB[n][kb] sum_16 a[m][k] b[n][k]
//
// The blog "NVFP4 Trains with Precision of 16-Bit..." (Blackwell FP4 tensor
// cores; GEMM speed-up figure) and the paper page ("Pretraining Large
// Language Models with NVFP4", FP4 tensor-core throughput vs FP8 on GB300)
// put the linear layers' Fprop/Dgrad/Wgrad on block-scaled FP4 MMA with FP32
// accumulation; this kernel is that MMA.
//
// What bounds it on this part (measured with MMA-only and load-only loops):
// one M=128 N=256 K=64 block-scaled FP4 MMA occupies an SM's tensor pipe for
// 128 cycles, even back to back into one accumulator from one thread (about
// 9.6 PFLOP/s for the GPU), and TMA delivers at most about 105 bytes per
// cycle into an SM.  A 128 x N tile on one SM needs (128 + N) x 144 bytes
// (codes and scales) per 256 K elements, i.e. 96-108 B/cycle at the MMA
// rate: loads and MMAs would both run at their limits.  A cluster of two
// CTAs on two SMs issues M=256 MMAs (cta_group::2): each SM computes 128
// rows x N, holds its 128 rows of A and half of B, and the pair's MMA reads
// the other half of B from the peer SM, so an SM loads 32 KB of codes per
// 512 MMA cycles (about 74 B/cycle with scales).
//
// Pair tile 256 x 256, K staged 256 at a time (64 bf16 for the BF16 form);
// one persistent cluster per SM pair, working through one GEMM's tiles or
// two GEMMs' (a layer's Dgrad and Wgrad, dealt so that the second fills the
// SM pairs the first's last round leaves idle).  Per CTA, 16 warps:
//   warp 0      code producer: its 128 A rows and its 128 B rows of the
//               stage by TMA (128-byte swizzle), completing on the leader
//               CTA's `full` barrier; 5-stage ring (38 KB per stage).
//   warp 2      scale producer: the stage's scale atoms (its A rows' 2 KB run
//               and both B groups' runs: each SM's MMA reads the scales of
//               all 256 B rows from its own TMEM) by bulk copy into the same
//               stage buffer, completing on its own `sf_in` barrier.
//   warp 1      TMEM owner (512 columns, allocated by the pair); in the leader
//               CTA also the MMA issuer: per stage, one wait on `full` (code
//               tiles and scale slots of both CTAs), four
//               tcgen05.mma.cta_group::2 (M=256 N=256 K=64), one commit
//               multicast to both CTAs' `empty` barrier, which frees the smem
//               stage and the TMEM scale slot at once.
//   warps 4-7   scale writers, one per TMEM lane quarter: read the stage's
//               scale atoms from smem and write them with tcgen05.st into
//               TMEM scale slot s (one slot per ring stage, five slots of 48
//               columns), then arrive on the leader's `full`.
// Per stage the MMAs keep the tensor pipe busy for 512 cycles, so no issuing
// thread may spend more than that per stage: every wait first tests the
// barrier without blocking (a blocking wait costs a few hundred cycles even
// on a completed phase), one lane waits for each warp, the MMA issuer waits
// once per stage, and the copies of a stage are split between two threads.
//   warps 8-15  epilogue: two warps per lane quarter, 128 columns each; each
//               stores its first 64 columns by TMA through a 4 KB smem box,
//               loads the rest, releases the accumulator to the MMA issuer,
//               and stores the rest while the next tile's MMAs run.
// TMEM scale-factor placement (measured with a probe MMA whose scale bytes
// encode their own TMEM address): in both the 1-SM and the pair form, A row
// r of an SM is read from lane r, column base + r / 32; B row n (all N rows,
// in each SM of the pair) from lane 32q + n % 32, column base + n / 32, in
// every lane quarter q.  B rows 0-127 of the pair tile come from the leader
// CTA's shared memory and rows 128-255 from the peer's.
// Every mbarrier wait is bounded (4 s by %globaltimer, adjustable by the
// host for tests): past the limit the waiter records NVFP4_ERR_TIMEOUT, raises
// its CTA's abort flag and the roles drain out; an aborting CTA waits for its
// MMAs to complete and gives copies in flight time to land before TMEM is
// freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <utility>

#include "nvfp4_device.cuh"
#include "nvfp4_launch.h"

namespace nvfp4 {
namespace gemm {

constexpr int BM = 128;             // rows of A per CTA (an SM's share of the pair tile)
constexpr int kPairM = 2 * BM;      // pair tile M
constexpr int BN = 256;             // pair tile N (each CTA loads BN / 2 B rows)
constexpr int kBRows = BN / 2;
constexpr int BK = 256;             // K elements per stage (FP4); bf16: 64
constexpr int BKB = 128;            // bytes per row per stage (the swizzle width)
constexpr int kStages = 5;          // smem ring stages = TMEM scale slots
constexpr int kMmaK = 64;           // K per tcgen05.mma (FP4)
constexpr int kMmaPerStage = BK / kMmaK;
constexpr int kATileBytes = BM * BKB;          // 16 KB
constexpr int kBTileBytes = kBRows * BKB;      // 16 KB
constexpr int kCodeBytes = kATileBytes + kBTileBytes;
constexpr int kSfAtomBytes = 512;              // 128 rows x 4 K blocks (MMA scale layout)
constexpr int kSfRunBytes = 4 * kSfAtomBytes;  // one 128-row group, one stage (16 K blocks)
constexpr int kSfBytes = 3 * kSfRunBytes;      // A's group, then B's two groups
constexpr int kStageBytes = kCodeBytes + kSfBytes;  // 38 KB
constexpr int kThreads = 512;
constexpr int kEpiWarps = 8;
constexpr int kSfWarps = 4;
constexpr int kStagingBytes = 32 * BKB;        // one staging box: 32 rows x 128 bytes
constexpr int kStagingBufs = 1;                // per epilogue warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = BN;              // fp32 accumulator columns
constexpr uint32_t kSfaCols = kMmaPerStage * 4;   // 4 columns per MMA (lane quarter q reads column q)
constexpr uint32_t kSfbCols = kMmaPerStage * 8;   // N = 256: 8 columns per MMA
constexpr uint32_t kSfColsPerSlot = kSfaCols + kSfbCols;
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;  // 4 s per wait
constexpr uint64_t kDrainNs = 100000000ull;            // final wait for the issued MMAs
constexpr uint64_t kGraceNs = 200000ull;               // after an abort: copies in flight land
static_assert(kAccCols + kStages * kSfColsPerSlot <= kTmemCols, "TMEM budget");
static_assert(kSfColsPerSlot % 4 == 0 && kSfaCols % 4 == 0, "TMEM scale columns 4-aligned");
static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte alignment of the 128-byte swizzle");

struct __align__(8) SharedState {
    uint64_t full[kStages];      // leader: the stage is ready for the MMAs: both CTAs' code tiles landed
                                 // (2 producer arrivals + TMA bytes) and both CTAs' scale writers have
                                 // filled the TMEM scale slot (8 arrivals; none for BF16 operands)
    uint64_t sf_in[kStages];     // this CTA's scale atoms of the stage landed (bulk-copy bytes)
    uint64_t empty[kStages];     // MMAs of the stage done: smem stage and TMEM scale slot free
    uint64_t acc_full;           // this tile's MMAs done (commit multicast to both CTAs)
    uint64_t acc_empty;          // leader: accumulator drained by both CTAs' epilogues (16 arrivals)
    uint64_t drain;              // leader: the MMA issuer's last MMAs done (abort path)
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + (size_t)kStages * kStageBytes +
                              (size_t)kEpiWarps * kStagingBufs * kStagingBytes + sizeof(SharedState);
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

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in the leader CTA (rank 0) of the pair.
__device__ __forceinline__ uint32_t leader_addr(const void* p) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(smem_u32(p)));
    return r;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Arrivals on a barrier of the leader CTA (the leader's own barrier when
// called there).  Relaxed: no arrival publishes data written by the arriving
// thread itself.  What a barrier guards is either written by TMA (made
// visible by the barrier's transaction count) or by tcgen05.st / read by
// tcgen05.ld, which the arriving warp has already waited for
// (tcgen05.wait::st / ::ld) and fenced (tcgen05.fence::before_thread_sync).
__device__ __forceinline__ void mbar_arrive_leader(uint32_t leader_bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(leader_bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_leader(uint32_t leader_bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(leader_bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_local(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Non-blocking test of a phase: the fast path of every wait (a blocking wait
// through the bounded loop below costs a few hundred cycles even when the
// phase has long completed, which the MMA issuer cannot afford per stage).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
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

// Bounded wait for the phase with the given parity; false on abort or
// timeout.  Each try_wait blocks for at most a system-dependent short time;
// between them the thread looks at its CTA's abort flag and the clock.  (A
// try_wait with a suspend-time hint woke its thread later after the phase
// completed: the GEMM ran 3-6% slower with it.)
__device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, SharedState* ss, uint32_t* status,
                                            uint64_t limit_ns) {
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int*>(&ss->abort_flag)) return false;
        if (globaltimer() - t0 > limit_ns) {
            atomicOr(status, kStatusTimeout);
            *reinterpret_cast<volatile int*>(&ss->abort_flag) = 1;
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, SharedState* ss, uint32_t* status,
                                          uint64_t limit_ns) {
    return mbar_test(bar, parity) || mbar_wait_slow(bar, parity, ss, status, limit_ns);
}

// TMA tile load into this CTA's shared memory, completing on a barrier of
// the leader CTA (the pair form of the load).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t leader_bar, int x,
                                                 int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(leader_bar), "r"(x), "r"(y)
        : "memory");
}

// Contiguous global -> shared copy (16-byte aligned, size a multiple of 16)
// completing on this CTA's barrier.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start address, leading/stride
// byte offsets (>> 4), descriptor version 1 (bits 46-48), swizzle mode in
// bits 61-63 (2 = 128-byte swizzle).  K-major operand tiles of 128-byte rows:
// 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)(16u >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B (format 1),
// K-major both, N >> 3 at bit 17, scale type at bit 23 (0 = UE4M3 for
// NVFP4, 1 = UE8M0 for MXFP4), M >> 7 at bit 27 (M = 256 for the pair),
// scale-factor data ids 0 (with scale_vec::2X the MMA reads bytes 0 and 1 of
// each scale word).
__host__ __device__ constexpr uint32_t instr_desc_nvf4(int m, int n, bool ue8m0) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((ue8m0 ? 1u : 0u) << 23) |
           ((uint32_t)(m >> 7) << 27);
}

// BF16 operands (the high-precision fallback GEMM): kind::f16, K = 16 per
// instruction, FP32 accumulation.  D = F32 (bits 4-5 = 1), A = B = BF16 (bits
// 7-9 and 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t instr_desc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
        "}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// MXFP4: two UE8M0 scales per row per K = 64 (32-element blocks).
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
        "}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at this shared offset in both CTAs of the pair once
// the MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
}

// A bounded wait on behalf of a whole warp: lane 0 waits, the warp follows
// (the shuffle orders the other lanes after lane 0's wait).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, SharedState* ss, uint32_t* status,
                                          uint64_t limit_ns, int lane) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait(bar, parity, ss, status, limit_ns);
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
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

__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
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

// 32 accumulator columns of the warp's 32 lanes, returned once loaded.
__device__ __forceinline__ void tmem_ld_x32_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// ---- the kernel ----------------------------------------------------------------
// One GEMM problem.
struct Params {
    const uint8_t* a_scales;  // MMA layout (512-byte atoms), rows padded to 128
    const uint8_t* b_scales;
    const float* a_amax;
    const float* b_amax;
    int M, N, K;
    int num_m, num_n, num_k;  // pair tiles along M and N, stages along K
    int group_m;              // M tiles per band of the tile raster
    int n_katoms;             // atoms per 128-row group: 4 * ceil(K / 256)
    int a_groups, b_groups;   // 128-row groups of A and B: ceil(rows / 128)
    int out_fp32;
    int accumulate;           // FP32 output added into C instead of stored
    int mx;                   // MXFP4 operands (UE8M0 scales, 32-element blocks)
    int bf16;                 // BF16 operands: no scales, 64 K elements per stage, alpha = 1
    uint64_t timeout_ns;      // bound of every barrier wait
    uint32_t* status;
};

// The kernel's parameter: one GEMM problem, or two run by one persistent
// launch (a layer's Dgrad and Wgrad), with their operand and output maps.
struct Maps {
    CUtensorMap a, b, c;
};
struct Launch {
    Maps maps[2];
    Params p[2];
    int nprob;  // 1 or 2; both problems have the same operand kind
    int extra;  // problem-1 tiles each lightly loaded cluster takes first (see Sched)
};

// Tile schedule.  Problem 0: cluster c takes pair tiles c, c + C, ... (C
// clusters).  Its last round leaves the clusters from r0 = T0 % C on with one
// tile fewer; with two problems each of those first takes `extra` tiles of
// problem 1 (about one problem-0 tile's worth of work), and the rest of
// problem 1 is dealt round robin, so the two problems' tails even out across
// the clusters.  Within a problem the tiles follow a banded raster: the M
// tiles are cut into bands of `group_m` rows and a band's tiles come one
// after the other, M fastest, so the clusters running at one time share a
// few B panels and the band's A panels, which stay in L2 while the band's B
// panels stream past them once.  (With one band over a long-K operand, say
// 32 A panels of 3 MB, the A panels fell out of L2 between waves and were
// read from DRAM six times over.)
struct Sched {
    int cid, C, r0, e, E, n0, nex, nrr;
    __device__ explicit Sched(const Launch& L) {
        cid = (int)blockIdx.x >> 1;
        C = (int)gridDim.x >> 1;
        const int t0 = L.p[0].num_m * L.p[0].num_n;
        const int t1 = L.nprob > 1 ? L.p[1].num_m * L.p[1].num_n : 0;
        r0 = t0 % C;
        e = (t1 > 0 && r0 > 0) ? L.extra : 0;
        E = min(t1, (C - r0) * e);
        n0 = cid < t0 ? (t0 - cid + C - 1) / C : 0;
        nex = (e > 0 && cid >= r0) ? max(0, min(e, E - (cid - r0) * e)) : 0;
        nrr = cid < t1 - E ? (t1 - E - cid + C - 1) / C : 0;
    }
    __device__ int count() const { return n0 + nex + nrr; }
    // problem g and pair tile (mt, nt) of this cluster's i-th tile
    __device__ void tile(int i, const Launch& L, int& g, int& mt, int& nt) const {
        int t;
        if (i < n0) {
            g = 0;
            t = cid + i * C;
        } else if (i < n0 + nex) {
            g = 1;
            t = (cid - r0) * e + (i - n0);
        } else {
            g = 1;
            t = E + cid + (i - n0 - nex) * C;
        }
        const Params& p = L.p[g];
        const int band_tiles = p.group_m * p.num_n;
        const int band = t / band_tiles;
        const int m0 = band * p.group_m;
        const int rows = min(p.group_m, p.num_m - m0);  // the last band may be shorter
        const int r = t - band * band_tiles;
        nt = r / rows;
        mt = m0 + (r - nt * rows);
    }
};

// Code producer (one lane, both CTAs): this CTA's A rows and B rows of each
// stage, counted on the leader's `full` barrier.  A stage is refilled once
// the MMAs that read it have completed (`empty`, committed to both CTAs).
__device__ __forceinline__ void producer_role(const Launch& L, SharedState* ss, uint8_t* stages, uint32_t rank) {
    const Sched S(L);
    // the leader's `full` barriers (consecutive words of its shared window)
    const uint32_t full_l0 = leader_addr(&ss->full[0]);
    uint32_t it = 0;
    for (int i = 0; i < S.count(); ++i) {
        int g, mt, nt;
        S.tile(i, L, g, mt, nt);
        const Params& p = L.p[g];
        const CUtensorMap* tmap_a = &L.maps[g].a;
        const CUtensorMap* tmap_b = &L.maps[g].b;
        const int ya = mt * kPairM + (int)rank * BM;
        const int yb = nt * BN + (int)rank * kBRows;
        for (int kt = 0; kt < p.num_k; ++kt, ++it) {
            const int s = it % kStages;
            const uint32_t ph = (it / kStages) & 1u;
            if (!mbar_wait(&ss->empty[s], ph ^ 1u, ss, p.status, p.timeout_ns)) return;
            uint8_t* st = stages + s * kStageBytes;
            // every box counts in full: rows past the matrix arrive as zeros
            const uint32_t full_l = full_l0 + 8u * (uint32_t)s;
            if (rank == 0) mbar_arrive_expect_tx(&ss->full[s], kCodeBytes);
            else mbar_arrive_expect_tx_leader(full_l, kCodeBytes);
            const int kx = kt * (p.bf16 ? 64 : BKB);  // a stage is 128 bytes of every row
            tma_load_2d_pair(st, tmap_a, full_l, kx, ya);
            tma_load_2d_pair(st + kATileBytes, tmap_b, full_l, kx, yb);
        }
    }
}

// Scale producer (one lane, both CTAs, NVFP4/MXFP4 only): the stage's scale
// atoms, its A rows' 2 KB run and both B groups' runs, into the stage buffer,
// counted on this CTA's `sf_in` barrier.
__device__ __forceinline__ void scale_producer_role(const Launch& L, SharedState* ss, uint8_t* stages,
                                                    uint32_t rank) {
    const Sched S(L);
    uint32_t it = 0;
    for (int i = 0; i < S.count(); ++i) {
        int g, mt, nt;
        S.tile(i, L, g, mt, nt);
        const Params& p = L.p[g];
        const int ga = 2 * mt + (int)rank;                // this CTA's A group
        const bool a_in = ga < p.a_groups;
        const int nb = min(2, p.b_groups - 2 * nt);       // B groups of the pair tile that exist
        const uint8_t* a_src = p.a_scales + (size_t)ga * p.n_katoms * kSfAtomBytes;
        const uint8_t* b_src = p.b_scales + (size_t)(2 * nt) * p.n_katoms * kSfAtomBytes;
        const size_t b_group = (size_t)p.n_katoms * kSfAtomBytes;
        for (int kt = 0; kt < p.num_k; ++kt, ++it) {
            const int s = it % kStages;
            const uint32_t ph = (it / kStages) & 1u;
            if (!mbar_wait(&ss->empty[s], ph ^ 1u, ss, p.status, p.timeout_ns)) return;
            uint8_t* sf = stages + s * kStageBytes + kCodeBytes;
            const size_t k_off = (size_t)kt * kSfRunBytes;
            // a stage's run lies inside its 128-row group's atoms (checked build)
            const bool k_in = NVFP4_IN_BOUNDS(k_off + kSfRunBytes <= b_group, p.status);
            const bool a_ld = a_in && k_in;
            const int nb_ld = k_in ? nb : 0;
            mbar_arrive_expect_tx(&ss->sf_in[s], (uint32_t)((a_ld ? 1 : 0) + nb_ld) * kSfRunBytes);
            if (a_ld) bulk_load(sf, a_src + k_off, kSfRunBytes, &ss->sf_in[s]);
            for (int g = 0; g < nb_ld; ++g)
                bulk_load(sf + (1 + g) * kSfRunBytes, b_src + g * b_group + k_off, kSfRunBytes, &ss->sf_in[s]);
        }
    }
}

// Operand kinds of the MMA loop.  The loop is instantiated once per kind: a
// run-time choice between the MMA forms inside the loop slowed the issue of
// every MMA.
enum MmaKind { kNvf4 = 0, kMxf4 = 1, kBf16 = 2 };

// The MMA issuer (one thread of the leader CTA).  Per stage: one wait (`full`:
// both CTAs' code tiles and scale slots), four M=256 N=256 MMAs into the
// accumulator (TMEM columns 0-255 of each SM), one commit that frees the
// stage and its scale slot in both CTAs.  Per tile: wait until both
// epilogues have drained the accumulator, commit `acc_full` at the end.  The
// MMAs of a stage keep the tensor pipe busy for 512 cycles; everything this
// thread does per stage has to fit in that.  Returns false on abort.
template <int kKind>
__device__ __forceinline__ bool mma_loop(const Launch& L, SharedState* ss, uint8_t* stages, uint32_t tmem_base) {
    const Sched S(L);
    const Params& p0 = L.p[0];  // operand kind, status and wait bound: the same in both problems
    const uint32_t idesc = kKind == kBf16 ? instr_desc_bf16(kPairM, BN) : instr_desc_nvf4(kPairM, BN, kKind == kMxf4);
    // descriptors of stage 0's tiles; stage s adds s * kStageBytes >> 4 to the
    // start-address field, MMA j adds 32 j >> 4
    const uint64_t adesc0 = smem_desc(smem_u32(stages));
    const uint64_t bdesc0 = smem_desc(smem_u32(stages + kATileBytes));
    int s = 0;            // ring stage of the next MMAs, and its phase parity
    uint32_t ph = 0;
    for (int i = 0; i < S.count(); ++i) {
        int g, mt, nt;
        S.tile(i, L, g, mt, nt);
        const int num_k = L.p[g].num_k;
        if (!mbar_wait(&ss->acc_empty, ((uint32_t)i & 1u) ^ 1u, ss, p0.status, p0.timeout_ns)) return false;
        tc_fence_after();
        for (int kt = 0; kt < num_k; ++kt) {
            if (!mbar_wait(&ss->full[s], ph, ss, p0.status, p0.timeout_ns)) return false;
            tc_fence_after();
            const uint64_t soff = (uint64_t)((uint32_t)(s * kStageBytes) >> 4);
            const uint32_t sf = tmem_base + kAccCols + (uint32_t)s * kSfColsPerSlot;
#pragma unroll
            for (int j = 0; j < kMmaPerStage; ++j) {
                const uint64_t adesc = adesc0 + soff + (uint64_t)(2 * j);
                const uint64_t bdesc = bdesc0 + soff + (uint64_t)(2 * j);
                const uint32_t acc = (kt > 0 || j > 0) ? 1u : 0u;
                if constexpr (kKind == kBf16)
                    mma_bf16(tmem_base, adesc, bdesc, idesc, acc);
                else if constexpr (kKind == kMxf4)
                    mma_mxf4(tmem_base, adesc, bdesc, idesc, sf + 4 * j, sf + kSfaCols + 8 * j, acc);
                else
                    mma_nvf4(tmem_base, adesc, bdesc, idesc, sf + 4 * j, sf + kSfaCols + 8 * j, acc);
            }
            mma_commit_pair(&ss->empty[s]);
            if (++s == kStages) {
                s = 0;
                ph ^= 1u;
            }
        }
        mma_commit_pair(&ss->acc_full);
    }
    return true;
}

// Runs the MMA loop, then waits (bounded) until every MMA it issued has
// completed, on the normal path and after an abort alike, so TMEM and the
// stages are never released under running MMAs.
__device__ __forceinline__ void mma_role(const Launch& L, SharedState* ss, uint8_t* stages, uint32_t tmem_base) {
    if (L.p[0].bf16) mma_loop<kBf16>(L, ss, stages, tmem_base);
    else if (L.p[0].mx) mma_loop<kMxf4>(L, ss, stages, tmem_base);
    else mma_loop<kNvf4>(L, ss, stages, tmem_base);
    mma_commit_pair(&ss->drain);
    // MMAs finish in microseconds; the bound only guards against a fault
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&ss->drain, 0u) && globaltimer() - t0 < kDrainNs) {
    }
}

// Scale writers (warp q = TMEM lane quarter q, both CTAs).  Lane l of the
// stage's scale atoms (MMA layout) holds, in atom j of a 128-row group, the
// four K-block scales of rows 32c + l (c = 0..3) of MMA j at bytes 16 l + 4 c.
// Slot s of TMEM (48 columns from column 256 + 48 s) gets, for MMA j: A's
// word of row 32q + l at column 4j + q (the only one of 4j..4j+3 that lane
// quarter q's part of the MMA reads), and
// B's words of rows 32c + l, c = 0..7 (both 128-row groups of the pair tile),
// at columns 16 + 8j + c, in every lane quarter.  Slot s is free again once
// the MMAs of the stage's previous round have completed: the scale producer
// waited for exactly that (`empty`) before the copies that complete `sf_in`,
// so the writers need no wait of their own for it.
__device__ __forceinline__ void scale_role(const Launch& L, SharedState* ss, const uint8_t* stages,
                                           uint32_t tmem_base, int q, int lane, uint32_t rank) {
    const Sched S(L);
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    // the leader's `full` barriers (consecutive words of its shared window)
    const uint32_t full_l0 = leader_addr(&ss->full[0]);
    uint32_t it = 0;
    for (int i = 0; i < S.count(); ++i) {
        int g, mt, nt;
        S.tile(i, L, g, mt, nt);
        const Params& p = L.p[g];
        const bool a_in = 2 * mt + (int)rank < p.a_groups;
        const int nb = min(2, p.b_groups - 2 * nt);
        for (int kt = 0; kt < p.num_k; ++kt, ++it) {
            const int s = it % kStages;
            const uint32_t ph = (it / kStages) & 1u;
            if (!warp_wait(&ss->sf_in[s], ph, ss, p.status, p.timeout_ns, lane)) return;
            const uint8_t* sf = stages + s * kStageBytes + kCodeBytes + lane * 16;
            uint32_t wa[kMmaPerStage];
            uint4 wb[2][kMmaPerStage];
#pragma unroll
            for (int j = 0; j < kMmaPerStage; ++j) {
                wa[j] = a_in ? *reinterpret_cast<const uint32_t*>(sf + j * kSfAtomBytes + 4 * q) : 0u;
#pragma unroll
                for (int g = 0; g < 2; ++g)
                    wb[g][j] = g < nb ? *reinterpret_cast<const uint4*>(sf + (1 + g) * kSfRunBytes + j * kSfAtomBytes)
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
                    for (int g = 0; g < 2; ++g)
                        wb[g][j] = make_uint4(__byte_perm(wb[g][j].x, 0u, 0x4420), __byte_perm(wb[g][j].y, 0u, 0x4420),
                                              __byte_perm(wb[g][j].z, 0u, 0x4420), __byte_perm(wb[g][j].w, 0u, 0x4420));
                }
            }
            tc_fence_after();
            const uint32_t col = lane_addr + tmem_base + kAccCols + (uint32_t)s * kSfColsPerSlot;
            // A: lane quarter q's part of MMA j reads column 4j + q only, so
            // only that column is written (a quarter of the A-scale bytes a
            // 16-column store would write; about 2% of the GEMM's time)
#pragma unroll
            for (int j = 0; j < kMmaPerStage; ++j) tmem_st_x1(col + 4 * j + q, wa[j]);
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
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) mbar_arrive_local(&ss->full[s]);
                else mbar_arrive_leader(full_l0 + 8u * (uint32_t)s);
            }
        }
    }
}

// The warp waits until its earlier TMA stores have finished reading its
// staging buffer.
__device__ __forceinline__ void staging_free(int lane) {
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncwarp();
}

// Issues the TMA store (or add) of the warp's staging box at column x, row y:
// 32 rows x 128 bytes, the C tensor map's 128-byte swizzle.
__device__ __forceinline__ void store_box(const CUtensorMap* tmap_c, const Params& p, const uint8_t* staging,
                                          int lane, int x, int y, bool rows_in) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        if (rows_in && x < p.N) {
            if (p.accumulate) tma_add_2d(tmap_c, staging, x, y);
            else tma_store_2d(tmap_c, staging, x, y);
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}

// Staging writes of one 32-row box (128 bytes per row, the C tensor map's
// 128-byte swizzle: row r's 16-byte chunk c at chunk position c ^ (r % 8)).
// bf16: 64 columns given as 32 packed words; fp32: 32 columns, scaled here.
__device__ __forceinline__ void stage_bf16(const uint32_t* w, uint8_t* staging, int lane) {
    uint8_t* row = staging + lane * BKB;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2],
                                                                               w[4 * c + 3]);
}

__device__ __forceinline__ void stage_f32(const uint32_t* a, float alpha, uint8_t* staging, int lane) {
    uint8_t* row = staging + lane * BKB;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) =
            make_uint4(__float_as_uint(__fmul_rn(__uint_as_float(a[4 * c]), alpha)),
                       __float_as_uint(__fmul_rn(__uint_as_float(a[4 * c + 1]), alpha)),
                       __float_as_uint(__fmul_rn(__uint_as_float(a[4 * c + 2]), alpha)),
                       __float_as_uint(__fmul_rn(__uint_as_float(a[4 * c + 3]), alpha)));
}

// Epilogue warp (both CTAs): lane quarter q (its TMEM lanes 32q..32q+31, the
// CTA's rows 32q..), column half h (columns 128h..128h+127 of the tile).
// The first 64 columns are loaded, staged and handed to TMA (the staging
// buffer is free: the previous tile's stores have long finished reading
// it), then the last 64 are loaded and the accumulator is released at once;
// their conversion, staging and stores overlap the next tile's MMAs.  At
// most 64 accumulator words are live per thread, so nothing is spilled.
__device__ __forceinline__ void epilogue_role(const Launch& L, SharedState* ss, uint8_t* staging, uint32_t tmem_base,
                                              int q, int h, int lane, uint32_t rank) {
    const Sched S(L);
    // each problem's S_dec,A * S_dec,B
    auto alpha_of = [&](const Params& p) {
        return p.bf16 ? 1.0f : __fmul_rn(__ldg(p.a_amax + 1), __ldg(p.b_amax + 1));
    };
    const float alpha0 = alpha_of(L.p[0]);
    const float alpha1 = L.nprob > 1 ? alpha_of(L.p[1]) : 1.0f;
    const uint32_t t_lane = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(128 * h);
    const uint32_t acc_empty_l = leader_addr(&ss->acc_empty);
    auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            if (rank == 0) mbar_arrive_local(&ss->acc_empty);
            else mbar_arrive_leader(acc_empty_l);
        }
    };
    for (int i = 0; i < S.count(); ++i) {
        int g, mt, nt;
        S.tile(i, L, g, mt, nt);
        const Params& p = L.p[g];
        const CUtensorMap* tmap_c = &L.maps[g].c;
        const float alpha = g ? alpha1 : alpha0;
        if (!warp_wait(&ss->acc_full, (uint32_t)i & 1u, ss, p.status, p.timeout_ns, lane)) break;
        tc_fence_after();
        const int y = mt * kPairM + (int)rank * BM + 32 * q;
        const bool rows_in = y < p.M;
        const int x0 = nt * BN + 128 * h;
        if (!p.out_fp32) {
            // columns 0-63 packed to bf16 and written to staging, 64-127
            // loaded, then the release; the stores follow
            uint32_t a[64];
            tmem_ld_x64_sync(t_lane, a);
            {
                uint32_t w[32];
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    w[k] = pack_bf16x2(__fmul_rn(__uint_as_float(a[2 * k]), alpha),
                                       __fmul_rn(__uint_as_float(a[2 * k + 1]), alpha));
                staging_free(lane);
                stage_bf16(w, staging, lane);
            }
            tmem_ld_x64_sync(t_lane + 64, a);
            release();
            store_box(tmap_c, p, staging, lane, x0, y, rows_in);
            {
                uint32_t w[32];
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    w[k] = pack_bf16x2(__fmul_rn(__uint_as_float(a[2 * k]), alpha),
                                       __fmul_rn(__uint_as_float(a[2 * k + 1]), alpha));
                staging_free(lane);
                stage_bf16(w, staging, lane);
            }
            store_box(tmap_c, p, staging, lane, x0 + 64, y, rows_in);
        } else {
            // columns 0-63 staged and stored, 64-127 loaded, then the release
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                uint32_t a[32];
                tmem_ld_x32_sync(t_lane + 32 * b, a);
                staging_free(lane);
                stage_f32(a, alpha, staging, lane);
                store_box(tmap_c, p, staging, lane, x0 + 32 * b, y, rows_in);
            }
            uint32_t a2[32], a3[32];
            tmem_ld_x32_sync(t_lane + 64, a2);
            tmem_ld_x32_sync(t_lane + 96, a3);
            release();
            staging_free(lane);
            stage_f32(a2, alpha, staging, lane);
            store_box(tmap_c, p, staging, lane, x0 + 64, y, rows_in);
            staging_free(lane);
            stage_f32(a3, alpha, staging, lane);
            store_box(tmap_c, p, staging, lane, x0 + 96, y, rows_in);
        }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

__global__ void __launch_bounds__(kThreads, 1) nvf4_gemm_kernel(const __grid_constant__ Launch L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint8_t* staging = stages + kStages * kStageBytes;
    SharedState* ss = reinterpret_cast<SharedState*>(staging + kEpiWarps * kStagingBufs * kStagingBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // both CTAs' code producers, and both CTAs' scale writers
            mbar_init(&ss->full[s], L.p[0].bf16 ? 2 : 2 + 2 * kSfWarps);
            mbar_init(&ss->sf_in[s], 1);
            mbar_init(&ss->empty[s], 1);              // one commit per stage
        }
        mbar_init(&ss->acc_full, 1);
        mbar_init(&ss->acc_empty, 2 * kEpiWarps);
        mbar_init(&ss->drain, 1);
        ss->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int g = 0; g < L.nprob; ++g) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&L.maps[g].a) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&L.maps[g].b) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&L.maps[g].c) : "memory");
        }
    }
    if (warp == 1) {  // the pair allocates together: the same columns in both SMs
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&ss->tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = ss->tmem_base;

    const bool bf16 = L.p[0].bf16 != 0;
    if (warp == 0) {
        if (lane == 0) producer_role(L, ss, stages, rank);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) mma_role(L, ss, stages, tmem_base);
    } else if (warp == 2) {
        if (lane == 0 && !bf16) scale_producer_role(L, ss, stages, rank);
    } else if (warp >= 4 && warp < 8) {
        if (!bf16) scale_role(L, ss, stages, tmem_base, warp & 3, lane, rank);
    } else if (warp >= 8) {
        const int e = warp - 8;
        epilogue_role(L, ss, staging + e * kStagingBufs * kStagingBytes, tmem_base, warp & 3, e >> 2, lane, rank);
    }

    // Drain.  The MMA issuer has already waited for its MMAs.  Past the first
    // cluster barrier neither CTA issues another copy; after an abort, copies
    // issued earlier (loads that complete on the leader's barriers, stores)
    // may still be in flight, so an aborting CTA waits a while (copies take
    // microseconds) and the second barrier holds both CTAs until it is done.
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (*reinterpret_cast<volatile int*>(&ss->abort_flag)) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < kGraceNs) {
        }
    }
    cluster_sync();  // neither SM frees TMEM while the pair's MMAs may use it
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols));
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
// box box_x x box_y elements, 128-byte swizzle, zero fill outside.
int make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, int64_t rows, int64_t row_elems,
             int64_t ld_bytes, int box_x, int box_y, const char** msg) {
    cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_x, (cuuint32_t)box_y};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *msg = "cuTensorMapEncodeTiled failed";
        return 1;
    }
    return 0;
}

// Per device: the kernel's shared-memory attribute and how many 2-CTA
// clusters fit on the GPU at once (the persistent grid).
struct DeviceLaunch {
    bool ready = false;
    int clusters = 0;
};
DeviceLaunch g_launch[64];
std::mutex g_launch_mu;

int device_launch(int* clusters, const char** msg) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= 64) {
        *msg = "device ordinal out of range";
        return 1;
    }
    std::lock_guard<std::mutex> lk(g_launch_mu);
    DeviceLaunch& d = g_launch[dev];
    if (!d.ready) {
        e = cudaFuncSetAttribute(nvf4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return (int)e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, nvf4_gemm_kernel, &cfg);
        if (e != cudaSuccess) return (int)e;
        if (n < 1) {
            *msg = "no 2-CTA cluster of the GEMM kernel fits on this GPU";
            return 1;
        }
        d.clusters = n;
        d.ready = true;
    }
    *clusters = d.clusters;
    return 0;
}

int launch(const Launch& L, cudaStream_t s, const char** msg) {
    int clusters = 0;
    int e = device_launch(&clusters, msg);
    if (e) return e;
    int64_t tiles = 0;
    for (int g = 0; g < L.nprob; ++g) tiles += (int64_t)L.p[g].num_m * L.p[g].num_n;
    const int64_t grid_clusters = tiles < clusters ? tiles : clusters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * grid_clusters));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, nvf4_gemm_kernel, L);
}

// M tiles per band of the raster (see Sched): as many as keep the band's A
// panels (panel_bytes each: kPairM rows of codes and scales over the whole K)
// within kL2BandBytes, then evened out over the bands.
#ifndef NVFP4_GEMM_L2_BAND_MB
#define NVFP4_GEMM_L2_BAND_MB 32
#endif
constexpr double kL2BandBytes = (double)NVFP4_GEMM_L2_BAND_MB * 1048576.0;

int band_rows(int num_m, double panel_bytes) {
    int gmax = (int)(kL2BandBytes / panel_bytes);
    if (gmax < 1) gmax = 1;
    const int bands = (num_m + gmax - 1) / gmax;
    return (num_m + bands - 1) / bands;
}

int make_c_map(CUtensorMap* tcm, const void* c, int64_t M, int64_t N, int64_t ldc, bool fp32, const char** msg) {
    if (fp32) return make_map(tcm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, c, M, N, ldc * 4, 32, 32, msg);
    return make_map(tcm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c, M, N, ldc * 2, 64, 32, msg);
}

}  // namespace gemm

namespace gemm {
namespace {

// One block-scaled problem's maps and parameters.
int fp4_problem(const GemmArgs& g, Maps* m, Params* pp, const char** msg) {
    if (g.M > INT32_MAX || g.N > INT32_MAX || g.K > INT32_MAX) {
        *msg = "dimension exceeds 2^31";
        return -1;
    }
    if (make_map(&m->a, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.a_codes, g.M, g.K / 2, g.lda, BKB, BM, msg) ||
        make_map(&m->b, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.b_codes, g.N, g.K / 2, g.ldb, BKB, kBRows, msg) ||
        make_c_map(&m->c, g.c, g.M, g.N, g.ldc, g.out_fp32 != 0, msg))
        return 1;
    Params& p = *pp;
    p = {};
    p.a_scales = g.a_scales;
    p.b_scales = g.b_scales;
    p.a_amax = g.a_amax;
    p.b_amax = g.b_amax;
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.num_m = (int)((g.M + kPairM - 1) / kPairM);
    p.num_n = (int)((g.N + BN - 1) / BN);
    p.num_k = (int)((g.K + BK - 1) / BK);
    p.n_katoms = 4 * p.num_k;
    p.group_m = band_rows(p.num_m, (double)kPairM * ((double)g.K / 2 + (double)g.K / 16));
    p.a_groups = (int)((g.M + 127) / 128);
    p.b_groups = (int)((g.N + 127) / 128);
    p.out_fp32 = g.out_fp32;
    p.accumulate = g.accumulate;
    p.mx = g.mx;
    p.bf16 = 0;
    p.timeout_ns = g.timeout_ns ? g.timeout_ns : kDefaultTimeoutNs;
    p.status = g.status;
    return 0;
}

// Relative cost of one pair tile: its K stages plus the epilogue's share
// (about 6 stages' time for bf16 output, 8 for FP32).
double tile_cost(const Params& p) { return (double)p.num_k + (p.out_fp32 ? 8.0 : 6.0); }

}  // namespace
}  // namespace gemm

int launch_gemm(const GemmArgs& g, cudaStream_t s, const char** msg) {
    using namespace gemm;
    if (get_encoder(msg)) return 1;
    Launch L = {};
    L.nprob = 1;
    if (int e = fp4_problem(g, &L.maps[0], &L.p[0], msg)) return e;
    return launch(L, s, msg);
}

int launch_gemm_pair(const GemmArgs& g0, const GemmArgs& g1, cudaStream_t s, const char** msg) {
    using namespace gemm;
    if (get_encoder(msg)) return 1;
    if (g0.mx != g1.mx) {
        *msg = "the two problems of one launch must have the same operand format";
        return -1;
    }
    Launch L = {};
    L.nprob = 2;
    if (int e = fp4_problem(g0, &L.maps[0], &L.p[0], msg)) return e;
    if (int e = fp4_problem(g1, &L.maps[1], &L.p[1], msg)) return e;
    // problem 0 is the one with the costlier tiles: the clusters its last
    // round leaves idle take the cheaper tiles of the other first
    if (tile_cost(L.p[1]) > tile_cost(L.p[0])) {
        std::swap(L.maps[0], L.maps[1]);
        std::swap(L.p[0], L.p[1]);
    }
    const double ratio = tile_cost(L.p[0]) / tile_cost(L.p[1]);
    L.extra = (int)std::min(8.0, std::max(0.0, ratio + 0.5));
    return launch(L, s, msg);
}

int launch_gemm_bf16(const GemmBf16Args& g, cudaStream_t s, const char** msg) {
    using namespace gemm;
    if (get_encoder(msg)) return 1;
    if (g.M > INT32_MAX || g.N > INT32_MAX || g.K > INT32_MAX) {
        *msg = "dimension exceeds 2^31";
        return -1;
    }
    Launch L = {};
    L.nprob = 1;
    if (make_map(&L.maps[0].a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.a, g.M, g.K, g.lda * 2, 64, BM, msg) ||
        make_map(&L.maps[0].b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.b, g.N, g.K, g.ldb * 2, 64, kBRows, msg) ||
        make_c_map(&L.maps[0].c, g.c, g.M, g.N, g.ldc, g.out_fp32 != 0, msg))
        return 1;
    Params& p = L.p[0];
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.num_m = (int)((g.M + kPairM - 1) / kPairM);
    p.num_n = (int)((g.N + BN - 1) / BN);
    p.num_k = (int)((g.K + 63) / 64);
    p.group_m = band_rows(p.num_m, (double)kPairM * 2.0 * (double)g.K);
    p.a_groups = (int)((g.M + 127) / 128);
    p.b_groups = (int)((g.N + 127) / 128);
    p.out_fp32 = g.out_fp32;
    p.accumulate = g.accumulate;
    p.bf16 = 1;
    p.timeout_ns = g.timeout_ns ? g.timeout_ns : kDefaultTimeoutNs;
    p.status = g.status;
    return launch(L, s, msg);
}

}  // namespace nvfp4

// Host-side launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

constexpr int kAmaxThreads = 256;
constexpr int kAmaxUnroll = 8;      // 16-byte loads in flight per amax thread
constexpr int kRhtAmaxThreads = 256;
constexpr int kRowItemBlocks = 64;  // 1x16 blocks per warp item of the rowwise quantizer
constexpr int kQuantThreads = 256;
constexpr int kColThreads = 128;
constexpr int k2dThreads = 256;
constexpr int kMaxPartials = 2048;  // workspace holds one uint32 partial max per amax CTA
// Workspace bytes of one amax pass (what nvfp4_quantize, nvfp4_rht_quantize and
// nvfp4_rht_quantize_rowwise require); nvfp4_quantize_with_rht keeps two sets.
constexpr size_t kSinglePassWorkspaceBytes = (size_t)kMaxPartials * sizeof(uint32_t);

struct ScaleOut;

void launch_amax(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx, uint32_t* partials, int grid,
                 cudaStream_t s);
// partials_plain non-null: the same pass also writes the amax partials of x itself
void launch_rht_amax(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx, uint64_t rht_seed,
                     uint32_t* partials, int grid, cudaStream_t s, uint32_t* partials_plain = nullptr);
void launch_quantize_rowwise(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx,
                             const uint32_t* partials, int npartials, uint8_t* codes, int64_t ld_codes, ScaleOut so,
                             float* amax_out, uint32_t* status, bool sr, bool mx, uint64_t seed, bool rht,
                             uint64_t rht_seed, int grid, cudaStream_t s);
void launch_rht_rows_amax(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx, uint64_t rht_seed,
                          uint32_t* partials, int grid, cudaStream_t s);
void launch_quantize_colwise(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx,
                             const uint32_t* partials, int npartials, uint8_t* codes, int64_t ld_codes, ScaleOut so,
                             float* amax_out, uint32_t* status, bool sr, bool mx, uint64_t seed, bool rht,
                             uint64_t rht_seed, int grid, cudaStream_t s);
void launch_quantize_2d(const void* x, bool fp32, int64_t rows, int64_t cols, int64_t ldx, const uint32_t* partials,
                        int npartials, uint8_t* codes_r, int64_t ld_r, ScaleOut so_r, float* amax_r, uint8_t* codes_c,
                        int64_t ld_c, ScaleOut so_c, float* amax_c, uint32_t* status, int grid, cudaStream_t s);
int64_t colwise_tiles(int64_t rows, int64_t cols);
int quantize_2d_grid(int64_t rows, int64_t cols, bool fp32, int num_sms);
// y[cols][rows] = x^T, bf16; rows, cols % 8 == 0; x, y, ldx, ldy 16-byte granular
void launch_transpose_bf16(const void* x, int64_t rows, int64_t cols, int64_t ldx, void* y, int64_t ldy, int grid,
                           cudaStream_t s);

// GEMM (gemm.cu).  A: [M][K] codes/scales (MMA layout), B: [N][K].
struct GemmArgs {
    const uint8_t* a_codes;
    const uint8_t* a_scales;
    const float* a_amax;
    int64_t lda;  // bytes
    const uint8_t* b_codes;
    const uint8_t* b_scales;
    const float* b_amax;
    int64_t ldb;  // bytes
    void* c;
    int64_t ldc;  // elements
    int64_t M, N, K;
    int out_fp32;
    int accumulate;  // fp32 only: C += result (TMA reduce-add) instead of C = result
    int mx;  // MXFP4 operands: UE8M0 scales per 32 elements, scale_vec::2X
    uint64_t timeout_ns;  // bound of each device-side wait (0: the default, 4 s)
    uint32_t* status;
    int num_sms;
};

// Returns a cudaError_t-like code (0 ok) and fills `msg` on failure.
int launch_gemm(const GemmArgs& args, cudaStream_t s, const char** msg);
// Two block-scaled GEMMs (the same operand format) in one persistent launch,
// their tiles dealt so that the tail of one fills the other's idle clusters;
// each output is bit for bit what launch_gemm gives for it alone.
int launch_gemm_pair(const GemmArgs& a, const GemmArgs& b, cudaStream_t s, const char** msg);

// BF16 GEMM C = A B^T (gemm.cu, the same kernel with kind::f16 MMAs).
struct GemmBf16Args {
    const void* a;  // [M][lda] bf16
    const void* b;  // [N][ldb] bf16
    void* c;        // [M][ldc] bf16 or fp32
    int64_t lda, ldb, ldc;  // elements
    int64_t M, N, K;
    int out_fp32;
    int accumulate;  // fp32 only: C += result
    uint64_t timeout_ns;  // bound of each device-side wait (0: the default, 4 s)
    uint32_t* status;
    int num_sms;
};
int launch_gemm_bf16(const GemmBf16Args& args, cudaStream_t s, const char** msg);

}  // namespace nvfp4

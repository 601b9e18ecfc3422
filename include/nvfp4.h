/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 linear-layer engine.
 *
 * The engine implements the NVFP4 recipe of "Pretraining Large Language
 * Models with NVFP4" (arXiv 2509.25149; summary page, format paragraph,
 * recipe paragraph and limitations paragraph) and of the NVIDIA blog post
 * "NVFP4 Trains with Precision of 16-Bit and Speed and Efficiency of 4-Bit"
 * (technique list):
 *   - a full-tensor amax sets an FP32 tensor scale (S_dec = A/2688,
 *     S_enc = 2688/A, 2688 = 6 * 448);
 *   - 16 consecutive elements share one E4M3 block scale (1x16 blocks for
 *     activations and gradients; one scale per 16x16 tile for weights);
 *   - elements are E2M1 codes {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6},
 *     two per byte, rounded to nearest-even or stochastically (Philox);
 *   - Wgrad inputs first get a 16-point random Hadamard transform along the
 *     token (reduction) dimension;
 *   - Fprop, Dgrad and Wgrad run as block-scaled FP4 GEMMs with FP32
 *     accumulation on the tensor cores.
 *
 * Conventions for every entry point
 *   - All pointers named "device" are CUDA device pointers on the current
 *     device; the caller allocates and owns every buffer.  The library
 *     allocates no device memory.
 *   - Calls are asynchronous on `stream` (cudaStream_t; NULL = legacy
 *     default stream).  Argument errors are detected on the host, return at
 *     once and launch nothing.  Conditions found on the device (non-finite
 *     input, a pipeline wait that ran out) are recorded in a per-device
 *     status word that nvfp4_sync_status() reads and clears.
 *   - Inputs are row-major.  Device pointers must be 16-byte aligned and
 *     row strides (ldx, ld_codes, ldc) multiples of 16 bytes.
 *   - Numerics follow this contract bit for bit (the pages leave the
 *     formulas open; these are the plain readings): FP32 steps are
 *     correctly rounded single operations, in this order:
 *       A = max|x|;  S_dec = fl(A/2688);  S_enc = fl(2688/A) (FLT_MAX if it
 *       overflows; A == 0 gives S_dec = S_enc = 1);
 *       per block: sb = E4M3_rne_satfinite(fl(fl(bamax/6) * S_enc));
 *       r = fl(S_enc/sb) (FLT_MAX if it overflows);  v = fl(x * r);
 *       RTN: nearest E2M1 of clamp(|v|, 6), ties to the even mantissa, sign
 *       kept (a negative value that rounds to 0 gives code 0x8);
 *       SR: u = Philox4x32-10(key = seed, counter = (i/4, 0, 0, 0))[i%4] >> 8,
 *       round |v| up iff u * 2^-24 < (|v| - lo)/(hi - lo), where i is the
 *       element's row-major index in the logical output tensor;
 *       sb == 0: every code of the block is 0.
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* nvfp4_stream_t;

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, bad enum */
    NVFP4_ERR_UNSUPPORTED = 2, /* valid request this build does not implement   */
    NVFP4_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required    */
    NVFP4_ERR_NONFINITE = 4,   /* (device) the input held a NaN or an infinity  */
    NVFP4_ERR_TIMEOUT = 5,     /* (device) a bounded pipeline wait ran out      */
    NVFP4_ERR_CUDA = 6,        /* a CUDA runtime call failed                    */
    NVFP4_ERR_BOUNDS = 7       /* (device, checked build only) an index fell
                                  outside its tensor; the access was skipped   */
} nvfp4_status;

typedef enum { NVFP4_IN_BF16 = 0, NVFP4_IN_FP32 = 1 } nvfp4_in_dtype;
/* GEMM outputs: C = result in bf16 or FP32, or NVFP4_OUT_FP32_ADD: C is an
 * FP32 matrix that the result is added into element by element (one
 * correctly rounded FP32 add per element, C = fl(C + result)), as when a
 * weight gradient is accumulated in FP32 over micro-batches (paper page,
 * recipe paragraph: gradient accumulation stays in FP32). */
typedef enum { NVFP4_OUT_BF16 = 0, NVFP4_OUT_FP32 = 1, NVFP4_OUT_FP32_ADD = 2 } nvfp4_out_dtype;
typedef enum { NVFP4_BLOCK_1x16 = 0, NVFP4_BLOCK_16x16 = 1, NVFP4_BLOCK_MX1x32 = 2 } nvfp4_block;

/*
 * Element formats of a quantized tensor (nvfp4_tensor.format).
 *   NVFP4_FORMAT_NVFP4: E2M1 codes, one E4M3 scale per 16 elements, one FP32
 *     tensor scale (paper page, format paragraph).
 *   NVFP4_FORMAT_MXFP4: the format NVFP4 is compared against (paper page,
 *     format paragraph; explainer page, comparison paragraph): E2M1 codes,
 *     one power-of-two UE8M0 scale per 32 elements (2^(code - 127), the
 *     smallest power of two 2^e with 6 * 2^e >= the block's largest
 *     magnitude, e in [-127, 127]), no tensor scale.  Scale buffers keep one
 *     byte per 16-element slot in either layout, each 32-element block's
 *     code in both of its slots, so their sizes are those of NVFP4; amax
 *     holds {0, 1, 1}.
 */
typedef enum { NVFP4_FORMAT_NVFP4 = 0, NVFP4_FORMAT_MXFP4 = 1 } nvfp4_format;
typedef enum { NVFP4_RTN = 0, NVFP4_SR = 1 } nvfp4_round;

/*
 * Block-scale layouts.
 *   NVFP4_SCALES_LINEAR: byte (r, kb) at r * (cols/16) + kb, where kb = c/16.
 *     For 16x16 blocks the scale of tile (r/16, kb) is repeated on each of
 *     the tile's 16 rows, so both layouts index scales per row.
 *   NVFP4_SCALES_MMA: 512-byte atoms of 128 rows x 4 K blocks (the source
 *     layout of a tcgen05.cp.32x128b.warpx4 scale copy).  This is the layout
 *     nvfp4_gemm reads: the scales of 128 rows x 256 K elements are one
 *     contiguous 2 KB run.  With n_katoms = 4 * ceil(cols/256),
 *       byte (r, kb) = ((r/128) * n_katoms + kb/4) * 512
 *                      + (r%32) * 16 + ((r/32)%4) * 4 + kb%4.
 *     Padding (rows up to a multiple of 128, K blocks up to n_katoms * 4)
 *     is written as zero by the quantize calls.
 *   nvfp4_scales_bytes() gives the buffer size of either layout.
 */
typedef enum { NVFP4_SCALES_LINEAR = 0, NVFP4_SCALES_MMA = 1 } nvfp4_scale_layout;

/*
 * One quantized NVFP4 tensor: the logical [rows][cols] matrix the codes
 * describe, blocks along cols (the GEMM's K).
 *   codes  device, [rows][ld_codes] bytes; element c of a row in byte c/2,
 *          even c in the low nibble.  ld_codes >= cols/2, multiple of 16.
 *   scales device, E4M3 block scales in `scale_layout`.
 *   amax   device float[3] = {A, S_dec, S_enc}, written by quantize calls
 *          and read by the GEMM (alpha = S_dec(A) * S_dec(B)).
 */
typedef struct {
    uint8_t* codes;
    uint8_t* scales;
    float* amax;
    int64_t rows;
    int64_t cols;
    int64_t ld_codes;
    int32_t scale_layout; /* nvfp4_scale_layout */
    int32_t format;       /* nvfp4_format */
} nvfp4_tensor;

/* Bytes of the scale buffer of a [rows][cols] tensor in `scale_layout`
 * (0 for invalid arguments). */
size_t nvfp4_scales_bytes(int64_t rows, int64_t cols, int32_t scale_layout);

/* Workspace bytes that every call taking a workspace accepts, for any
 * shape: the amax pass keeps one partial per CTA there (2048 at most, 8 KB);
 * nvfp4_quantize_with_rht keeps two sets (16 KB), which is what this
 * returns.  nvfp4_quantize, nvfp4_rht_quantize and nvfp4_rht_quantize_rowwise
 * require only 8 KB (NVFP4_ERR_WORKSPACE below that). */
size_t nvfp4_workspace_size(void);

/*
 * nvfp4_quantize -- tensor amax (one full read), then block scales and
 * E2M1 codes (a second read), per the format paragraph of the paper page
 * and the blog's micro-block / 2D-block / stochastic-rounding items.
 *   x            device, [rows][ldx] elements of `dtype` (ldx >= cols).
 *   block        1x16 (activations, gradients) or 16x16 (weights; RTN only,
 *                rows % 16 == 0): NVFP4, outputs with format NVFP4.
 *                MX1x32: MXFP4 (outputs with format MXFP4; RTN or SR;
 *                cols % 32 == 0 for out_rowwise, rows % 32 == 0 for
 *                out_colwise).  MXFP4 has no tensor amax, so it reads x once;
 *                a 32-element block holding a NaN or an infinity flags
 *                NVFP4_ERR_NONFINITE and gets zero codes and scale.
 *   round, seed  rounding mode and the Philox key for SR.
 *   out_rowwise  if non-NULL: describes x, [rows][cols], blocks along cols
 *                (cols % 16 == 0).
 *   out_colwise  if non-NULL: describes x^T, [cols][rows], blocks along rows
 *                (rows % 16 == 0).  At least one output must be given; both
 *                get the same {A, S_dec, S_enc}.
 *   workspace    device, >= 8 KB (half of nvfp4_workspace_size(); any
 *                size from nvfp4_workspace_size() up is accepted), 16-byte
 *                aligned; no initial contents needed.  The call writes it
 *                and its second kernel reads it back, so two calls whose
 *                work can overlap on the GPU (e.g. on unordered streams) must
 *                not share one workspace.
 */
nvfp4_status nvfp4_quantize(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                            nvfp4_block block, nvfp4_round round, uint64_t seed,
                            const nvfp4_tensor* out_rowwise, const nvfp4_tensor* out_colwise,
                            void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_noalloc -- nvfp4_quantize for callers that cannot allocate
 * device memory.  The pages have no counterpart: this is an interface
 * convenience, not part of the method.
 *   Some callers have no way to get the 8 KB workspace nvfp4_quantize asks
 *   for: a plugin or extension whose host framework owns every device
 *   allocation and offers it no allocation hook, or a real-time loop that
 *   must not call cudaMalloc after set-up (cudaMalloc can synchronize the
 *   device and can fail once memory is fragmented).  This entry point keeps
 *   the amax partials in a fixed 8 KB device array inside the library and
 *   allocates nothing; the caller still supplies x and the output buffers.
 *   Arguments, results and errors are those of nvfp4_quantize.
 *   Limit: the array holds 2048 partial maxima, which is what any call needs
 *   whatever the tensor size (the amax pass uses at most 2048 CTAs); the
 *   library checks at compile time that the array covers nvfp4_quantize's
 *   workspace requirement, so no tensor size is refused for lack of scratch.
 *   The first call on a device looks up the array's device address (and
 *   creates the CUDA context if needed); make that first call before any
 *   stream capture.  All calls on a device share the array and it keeps the
 *   previous call's contents (nothing in it needs clearing): calls that can
 *   run at the same time on the GPU, e.g. on unordered streams, race on it.
 */
nvfp4_status nvfp4_quantize_noalloc(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                                    nvfp4_block block, nvfp4_round round, uint64_t seed,
                                    const nvfp4_tensor* out_rowwise, const nvfp4_tensor* out_colwise,
                                    nvfp4_stream_t stream);

/*
 * nvfp4_rht_quantize -- the Wgrad operand path (paper page, limitations
 * paragraph: Hadamard only on Wgrad; blog: Hadamard transforms reshape the
 * distribution).  Every run of 16 consecutive rows (tokens) of each column
 * is transformed y = (1/4) H16 (d . x), H16 Sylvester, d_j = +-1 from bit j
 * of word 0 of Philox4x32-10(key = rht_seed, counter = (0, 0, 1, 0)), the
 * butterfly evaluated stage by stage over index bits 0..3 in FP32.  Then the
 * tensor amax of y, and y^T is quantized with 1x16 blocks along the rows.
 *   out_colwise  describes y^T, [cols][rows]; rows % 16 == 0.  Its format
 *                selects the encoding: NVFP4 (1x16 blocks, the tensor amax
 *                taken over y) or MXFP4 (1x32 blocks, rows % 32 == 0, no
 *                amax pass).
 *   Other arguments as nvfp4_quantize.  Both Wgrad operands must use the
 *   same rht_seed so the transform cancels in the product.
 */
nvfp4_status nvfp4_rht_quantize(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                                nvfp4_round round, uint64_t seed, uint64_t rht_seed,
                                const nvfp4_tensor* out_colwise, void* workspace, size_t workspace_bytes,
                                nvfp4_stream_t stream);

/*
 * nvfp4_quantize_with_rht -- one operand of a linear layer for both of its
 * GEMMs (the paper page's recipe: the Fprop/Dgrad operand without the
 * transform, the Wgrad operand with it along the tokens).  Results are bit
 * for bit those of the two separate calls
 *   nvfp4_quantize(x, block 1x16, round, seed, out_rowwise, NULL)
 *   nvfp4_rht_quantize(x, round, seed, rht_seed, out_colwise)
 * but the two tensor amaxes (of x and of the transformed x) come from one
 * read of x instead of two.
 *   out_rowwise  describes x, [rows][cols], 1x16 blocks along cols.
 *   out_colwise  describes y^T, [cols][rows], y the 16-point RHT of x along
 *                its rows (as nvfp4_rht_quantize); rows % 16 == 0.
 *                Both outputs are required and must have format NVFP4
 *                (MXFP4 has no amax pass to share: use the separate calls).
 *   round, seed  used by both outputs (SR: the same Philox key; each output
 *                indexes the stream by its own logical element index).
 *   workspace    device, >= 2 * 8 KB (nvfp4_workspace_size()), 16-byte
 *                aligned; NVFP4_ERR_WORKSPACE if smaller.
 *   Other arguments as nvfp4_quantize.
 * With SR the rowwise encode runs on the library's second stream of the
 * device (see the linear layer below), forked from `stream` after the amax
 * pass and joined back before the call's work ends, so ordering is that of
 * `stream` alone; a `stream` being captured into a CUDA graph keeps both
 * encodes on itself.
 */
nvfp4_status nvfp4_quantize_with_rht(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                                     nvfp4_round round, uint64_t seed, uint64_t rht_seed,
                                     const nvfp4_tensor* out_rowwise, const nvfp4_tensor* out_colwise,
                                     void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_rht_quantize_rowwise -- the 16-point RHT along each row (the GEMM's
 * K for a rowwise operand: each 1x16 block is one transform chunk), then the
 * tensor amax of the result and rowwise quantization.  The paper page allows
 * the transform on the Fprop and Dgrad inputs too (limitations paragraph:
 * applied to Wgrad only, its effect on the other GEMMs at larger scale left
 * open); both operands of a GEMM transformed with the same rht_seed give the
 * untransformed product, since (1/4) H16 is orthogonal.
 *   out_rowwise  describes y, [rows][cols]; its format selects NVFP4 (1x16)
 *                or MXFP4 (1x32, cols % 32 == 0, no amax pass).
 *   Other arguments as nvfp4_quantize; the transform as nvfp4_rht_quantize.
 */
nvfp4_status nvfp4_rht_quantize_rowwise(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                                        nvfp4_round round, uint64_t seed, uint64_t rht_seed,
                                        const nvfp4_tensor* out_rowwise, void* workspace, size_t workspace_bytes,
                                        nvfp4_stream_t stream);

/*
 * nvfp4_gemm -- C[m][n] = S_dec(A) S_dec(B) sum_kb sbA[m][kb] sbB[n][kb]
 *               sum_{16} e2m1(A[m][k]) e2m1(B[n][k]),
 * a block-scaled FP4 GEMM on the tcgen05 tensor cores with FP32
 * accumulation (blog: Blackwell FP4 tensor cores run the linear layers).
 *   A            [M][K] quantized, B [N][K] quantized, both of the same
 *                format (NVFP4: kind::mxf4nvf4, scale_vec::4X, E4M3 scales,
 *                alpha = S_dec(A) S_dec(B); MXFP4: scale_vec::2X, UE8M0
 *                scales, alpha = 1), both with
 *                NVFP4_SCALES_MMA scales (16-byte aligned buffers of
 *                nvfp4_scales_bytes() bytes), A->cols == B->cols == K,
 *                K % 64 == 0.
 *   C            device, [M][ldc] of out_dtype (bf16 or fp32), written whole;
 *                with NVFP4_OUT_FP32_ADD an FP32 matrix the result is added
 *                into (it must hold finite values or zeros beforehand).
 *   workspace    as nvfp4_quantize (may be NULL with 0 bytes: the GEMM
 *                needs none today).
 * Deterministic: every output element accumulates its K steps in order in
 * one FP32 accumulator, so the same operands give bit-identical C on every
 * launch.
 */
nvfp4_status nvfp4_gemm(const nvfp4_tensor* A, const nvfp4_tensor* B, void* C, nvfp4_out_dtype out_dtype,
                        int64_t ldc, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_gemm_pair -- two independent nvfp4_gemm problems (C0 = A0 B0^T and
 * C1 = A1 B1^T, each argument as nvfp4_gemm's) in one persistent launch,
 * such as a linear layer's Dgrad and Wgrad.  A launch keeps one 256 x 256
 * tile per SM pair at a time; a GEMM alone leaves part of the GPU idle in
 * its last round of tiles, and here the other GEMM's tiles fill that round
 * (the SM pairs with a tile fewer of the costlier problem take the other's
 * tiles first).  Each output is bit for bit what nvfp4_gemm gives for it
 * alone.  Both problems must have the same format (NVFP4 or MXFP4); C0 and
 * C1 must not overlap each other or any operand.
 * Errors: those of nvfp4_gemm for either problem, before any launch.
 */
nvfp4_status nvfp4_gemm_pair(const nvfp4_tensor* A0, const nvfp4_tensor* B0, void* C0, nvfp4_out_dtype out_dtype0,
                             int64_t ldc0, const nvfp4_tensor* A1, const nvfp4_tensor* B1, void* C1,
                             nvfp4_out_dtype out_dtype1, int64_t ldc1, nvfp4_stream_t stream);

/*
 * nvfp4_gemm_bf16 -- C[m][n] = sum_k A[m][k] B[n][k] with bf16 A and B and
 * FP32 accumulation on the tcgen05 tensor cores (kind::f16): the GEMM of the
 * linear layers the recipe keeps in high precision (paper page, recipe
 * paragraph: a few sensitive layers and the final ones stay in BF16).
 *   A            device bf16 [M][lda], B device bf16 [N][ldb] (both K-major,
 *                lda, ldb >= K and multiples of 8), K % 8 == 0.
 *   C            device, [M][ldc] of out_dtype, written whole (or, with
 *                NVFP4_OUT_FP32_ADD, added into).
 *   All pointers 16-byte aligned.  Errors as nvfp4_gemm.
 */
nvfp4_status nvfp4_gemm_bf16(const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                             nvfp4_out_dtype out_dtype, int64_t ldc, int64_t M, int64_t N, int64_t K,
                             nvfp4_stream_t stream);

/*
 * nvfp4_transpose_bf16 -- y = x^T for a bf16 x [rows][ldx] into y
 * [cols][ldy].  Not a step of the method: the BF16 fallback GEMM above takes
 * K-major operands, and a layer kept in (or switched back to) BF16 needs W^T
 * for Dgrad and dY^T, X^T for Wgrad.
 *   rows, cols   positive multiples of 8; ldx >= cols, ldy >= rows, both
 *                multiples of 8 elements; x and y device, 16-byte aligned,
 *                not overlapping.
 *   Errors: NVFP4_ERR_INVALID_ARG for any of the above, before any launch.
 */
nvfp4_status nvfp4_transpose_bf16(const void* x, int64_t rows, int64_t cols, int64_t ldx, void* y, int64_t ldy,
                                  nvfp4_stream_t stream);

/*
 * Linear layer Y = X W^T with NVFP4 GEMMs, following the recipe (paper
 * page: 2D weight scaling keeps Fprop and Dgrad consistent, Hadamard only on
 * Wgrad; blog: stochastic rounding on gradients):
 *   fwd:  X -> xq (1x16 RTN);  W -> wq and wtq (16x16 RTN, both layouts);
 *         Y[M][N] (bf16) = gemm(xq, wq).
 *   bwd:  dY -> dyq (1x16 SR) and, after the RHT along tokens with
 *         rht_seed, dY^T -> dytq (SR), both from one amax read
 *         (nvfp4_quantize_with_rht);  X^T -> xtq (RHT, RTN);
 *         dX[M][K] (bf16) = gemm(dyq, wtq) and dW[N][K] (fp32) =
 *         gemm(dytq, xtq), the two in one launch (nvfp4_gemm_pair).
 * The context holds caller-allocated quantized buffers; every tensor's
 * rows/cols/ld_codes/scale_layout (MMA) must be filled in for the shapes
 * above, and the workspace must have at least nvfp4_workspace_size() bytes
 * (16 KB, for nvfp4_quantize_with_rht; device, 16-byte aligned).  With
 * nvfp4_linear_workspace_size() bytes (24 KB) the forward quantizes W on a
 * second stream while X is quantized on `stream`: the library's one
 * non-blocking stream per device, forked from `stream` and joined back into
 * it by events, so the results and their ordering are those of `stream`
 * alone.  That stream is shared by every forward on the device (concurrent
 * forwards on different streams may wait for one another's W), and a
 * `stream` that is being captured into a CUDA graph gets both quantizations
 * on itself.  X, W, dY are bf16,
 * row-major, contiguous.  Both SR quantizations of dY use sr_seed.
 * M, N, K must be multiples of 64 (16 for the blocks, 64 for the MMA K).
 * X may be NULL in nvfp4_linear_bwd when xtq already holds X^T's codes
 * (nvfp4_linear_fwd_rht below).
 * dw_accumulate = 0: dW = dY^T X (FP32, overwritten); nonzero: the Wgrad
 * GEMM adds into dW (FP32 gradient accumulation across micro-batches, with
 * the GEMM's NVFP4_OUT_FP32_ADD).
 */
typedef struct {
    int64_t M, N, K;
    nvfp4_tensor xq;   /* [M][K]  */
    nvfp4_tensor wq;   /* [N][K]  */
    nvfp4_tensor wtq;  /* [K][N]  */
    nvfp4_tensor dyq;  /* [M][N]  */
    nvfp4_tensor dytq; /* [N][M]  */
    nvfp4_tensor xtq;  /* [K][M]  */
    void* workspace;
    size_t workspace_bytes;
    int32_t dw_accumulate;
} nvfp4_linear_ctx;

/* Workspace bytes with which nvfp4_linear_fwd / nvfp4_linear_fwd_rht
 * quantize X and W on two streams (24 KB; see above). */
size_t nvfp4_linear_workspace_size(void);

nvfp4_status nvfp4_linear_fwd(const void* X, const void* W, void* Y, nvfp4_linear_ctx* ctx, nvfp4_stream_t stream);
nvfp4_status nvfp4_linear_bwd(const void* dY, const void* X, void* dX, float* dW, uint64_t sr_seed,
                              uint64_t rht_seed, nvfp4_linear_ctx* ctx, nvfp4_stream_t stream);

/*
 * nvfp4_linear_fwd_rht -- nvfp4_linear_fwd that also quantizes Wgrad's X
 * operand: X^T -> xtq (the 16-point RHT along the tokens with rht_seed, RTN),
 * from the same read of X that gives xq's tensor scale
 * (nvfp4_quantize_with_rht), so X's full-tensor amax scan runs once per step
 * instead of twice (paper page, limitations paragraph: the tensor scale
 * costs an extra full-tensor amax scan).  xq, xtq, Y are bit for bit what
 * nvfp4_linear_fwd and the backward's own X^T quantization give.
 * nvfp4_linear_bwd then takes X = NULL and reads xtq as it is; its rht_seed
 * must be the one given here (both Wgrad operands share the sign vector).
 * A caller that runs several forwards before their backwards keeps one xtq
 * per forward (xq, wq, wtq may be shared: Dgrad reads only wtq, a function
 * of W).  Errors: as nvfp4_linear_fwd, plus xtq's shape check.
 */
nvfp4_status nvfp4_linear_fwd_rht(const void* X, const void* W, void* Y, uint64_t rht_seed, nvfp4_linear_ctx* ctx,
                                  nvfp4_stream_t stream);

/* Bound, in nanoseconds, of every wait inside the GEMM kernels (a pipeline
 * stage that never fills, a barrier that never completes): past it the
 * kernel records NVFP4_ERR_TIMEOUT in the status word, lets its MMAs and
 * copies in flight finish, and returns, so the context stays usable.  0
 * restores the default (4 s).  Applies to GEMMs launched after the call, in
 * every thread; returns the previous setting.  Meant for tests and
 * diagnostics: a bound far below a GEMM's running time aborts it. */
uint64_t nvfp4_set_wait_limit_ns(uint64_t limit_ns);

/* Synchronize `stream`, then return and clear the device status word of the
 * current device: NVFP4_ERR_BOUNDS (checked build), NVFP4_ERR_TIMEOUT,
 * NVFP4_ERR_NONFINITE or NVFP4_OK, the first that applies (NVFP4_ERR_CUDA if
 * the synchronization itself failed). */
nvfp4_status nvfp4_sync_status(nvfp4_stream_t stream);

/*
 * The checked build.  Compiled with -DNVFP4_CHECKED, every kernel of this
 * library tests the index of each global-memory access it computes itself
 * (input elements, codes, scale bytes, amax partials, scale atoms read by the
 * GEMM) against its tensor's extent; an index outside it skips the access and
 * sets NVFP4_ERR_BOUNDS in the status word.  (Compute sanitizers do not run
 * everywhere this library does; this build answers the same question for the
 * library's own index arithmetic.)  TMA copies are bounded by their tensor
 * maps and are not checked again.
 * nvfp4_checked_build returns 1 in the checked build, 0 otherwise.
 * nvfp4_checked_selftest (checked build) runs one kernel whose single guarded
 * store has an index one past its buffer by construction, so the check must
 * skip it and report it; it returns what nvfp4_sync_status then returns
 * (NVFP4_ERR_BOUNDS when the checks work) after verifying that the buffer's
 * guard word was not written.  In the normal build it returns
 * NVFP4_ERR_UNSUPPORTED without launching anything.
 */
int32_t nvfp4_checked_build(void);
nvfp4_status nvfp4_checked_selftest(nvfp4_stream_t stream);

/* Static English text of a status code. */
const char* nvfp4_status_string(nvfp4_status status);

/* Text of the last error seen by this thread in a call of this library
 * (empty if none); valid until the thread's next call. */
const char* nvfp4_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H_ */

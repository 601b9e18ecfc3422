// C ABI of the NVFP4 engine: argument checks on the host, then kernel
// launches on the caller's stream.  See include/nvfp4.h for the contract.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/nvfp4.h"
#include "nvfp4_device.cuh"
#include "nvfp4_launch.h"

namespace nvfp4 {

// Per-device status word (NVFP4_ERR_NONFINITE / NVFP4_ERR_TIMEOUT bits).
static __device__ uint32_t g_status_word;

#ifdef NVFP4_CHECKED
// nvfp4_checked_selftest: a two-word logical buffer followed by a guard word
// in the same array, and one guarded store whose index is one past the
// logical buffer (so even an unchecked store would land on the guard word).
static __device__ uint32_t g_selftest_words[3];
static __global__ void checked_selftest_kernel(uint32_t* status) {
    const int64_t n = 2;
    const int64_t i = n;  // one past the logical buffer, by construction
    if (NVFP4_IN_BOUNDS(i < n, status)) g_selftest_words[i] = 0xFFFFFFFFu;
}
#endif

namespace {

thread_local char g_err[512];

// Bound of every device-side wait of the GEMM (0: the kernel's default, 4 s).
std::atomic<uint64_t> g_wait_limit_ns{0};

nvfp4_status fail(nvfp4_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    uint32_t* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

nvfp4_status device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word);
        if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        d.ready = true;
    }
    *out = &d;
    return NVFP4_OK;
}

// The second stream: independent work of one call runs there beside the
// caller's stream (W's quantization beside X's in the forward; dY's rowwise
// SR encode beside its colwise one).  One non-blocking stream and two events
// per device, created on first use; g_side_mu is held by a call from its fork
// record to its join wait, so the events are never recorded by one call
// between another call's record and wait (recursive: a call inside a fork may
// fork again, its work then queued behind the outer call's on the second
// stream).
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[kMaxDevices];
std::recursive_mutex g_side_mu;

// The current device's second stream; the caller holds g_side_mu.
nvfp4_status side_stream(SideStream** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_CUDA, "device ordinal %d out of range", dev);
    SideStream& ss = g_side[dev];
    if (!ss.stream) {
        SideStream n;
        e = cudaStreamCreateWithFlags(&n.stream, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            if (n.join) cudaEventDestroy(n.join);
            if (n.fork) cudaEventDestroy(n.fork);
            if (n.stream) cudaStreamDestroy(n.stream);
            return fail(NVFP4_ERR_CUDA, "second stream: %s", cudaGetErrorString(e));
        }
        ss = n;
    }
    *out = &ss;
    return NVFP4_OK;
}

// Runs side_work(stream) and main_work() concurrently: side_work on the
// device's second stream, forked from `s` and joined back into it by events,
// main_work on `s`; results and their ordering are those of `s` alone.  When
// `allowed` is false, or `s` is being captured into a CUDA graph (the shared
// second stream would join the capture; a query that fails, e.g. on the
// legacy stream while another stream is captured, counts as capturing and
// its error is cleared), both run on `s`, side_work first.  Returns the first
// failure; the second stream is joined back whatever fails.
template <class SideFn, class MainFn>
nvfp4_status fork_join(cudaStream_t s, bool allowed, SideFn side_work, MainFn main_work) {
    if (allowed) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
            cudaGetLastError();
            cap = cudaStreamCaptureStatusActive;
        }
        allowed = cap == cudaStreamCaptureStatusNone;
    }
    nvfp4_status st;
    if (!allowed) return (st = side_work(s)) ? st : main_work();
    std::lock_guard<std::recursive_mutex> lk(g_side_mu);
    SideStream* side;
    if ((st = side_stream(&side))) return st;
    cudaError_t e = cudaEventRecord(side->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "fork to the second stream: %s", cudaGetErrorString(e));
    st = side_work(side->stream);
    if (!st) st = main_work();
    e = cudaEventRecord(side->join, side->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, side->join, 0);
    if (st) return st;
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "join of the second stream: %s", cudaGetErrorString(e));
    return NVFP4_OK;
}

nvfp4_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
    return NVFP4_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t n_katoms(int64_t cols) { return 4 * ceil_div(cols, 256); }

size_t scales_bytes(int64_t rows, int64_t cols, int32_t layout) {
    if (rows < 0 || cols < 0 || cols % 16) return 0;
    if (layout == NVFP4_SCALES_LINEAR) return (size_t)(rows * (cols / 16));
    if (layout == NVFP4_SCALES_MMA) return (size_t)(ceil_div(rows, 128) * n_katoms(cols) * 512);
    return 0;
}

ScaleOut scale_out(const nvfp4_tensor& t) {
    ScaleOut s;
    s.p = t.scales;
    s.bytes = (int64_t)scales_bytes(t.rows, t.cols, t.scale_layout);
    s.n_katoms = n_katoms(t.cols);
    s.nkb = t.cols / 16;
    s.mma = t.scale_layout == NVFP4_SCALES_MMA;
    return s;
}

// A quantize output: `rows` x `cols` logical, blocks along cols.
nvfp4_status check_out(const nvfp4_tensor* t, int64_t rows, int64_t cols, const char* name) {
    if (!t->codes || !t->scales || !t->amax) return fail(NVFP4_ERR_INVALID_ARG, "%s: null buffer", name);
    if (t->rows != rows || t->cols != cols)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: shape [%lld][%lld], expected [%lld][%lld]", name, (long long)t->rows,
                    (long long)t->cols, (long long)rows, (long long)cols);
    if (cols % 16) return fail(NVFP4_ERR_INVALID_ARG, "%s: cols %lld not a multiple of 16", name, (long long)cols);
    if (t->ld_codes < cols / 2 || t->ld_codes % 16)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: ld_codes %lld must be >= cols/2 and a multiple of 16", name,
                    (long long)t->ld_codes);
    if (t->scale_layout != NVFP4_SCALES_LINEAR && t->scale_layout != NVFP4_SCALES_MMA)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: bad scale_layout %d", name, t->scale_layout);
    if (t->format != NVFP4_FORMAT_NVFP4 && t->format != NVFP4_FORMAT_MXFP4)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: bad format %d", name, t->format);
    if (!aligned16(t->codes) || !aligned16(t->scales) || (reinterpret_cast<uintptr_t>(t->amax) & 3u))
        return fail(NVFP4_ERR_INVALID_ARG, "%s: codes/scales must be 16-byte aligned, amax 4-byte aligned", name);
    return NVFP4_OK;
}

// Zero the scale buffer when the MMA layout has padding the kernels do not
// visit (rows to a multiple of 128, K blocks to a multiple of 16).
nvfp4_status zero_scale_padding(const nvfp4_tensor* t, cudaStream_t s) {
    if (t->scale_layout != NVFP4_SCALES_MMA) return NVFP4_OK;
    if (t->rows % 128 == 0 && t->cols % 256 == 0) return NVFP4_OK;
    cudaError_t e = cudaMemsetAsync(t->scales, 0, scales_bytes(t->rows, t->cols, NVFP4_SCALES_MMA), s);
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    return NVFP4_OK;
}

nvfp4_status check_input(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx) {
    if (!x) return fail(NVFP4_ERR_INVALID_ARG, "x is null");
    if (dtype != NVFP4_IN_BF16 && dtype != NVFP4_IN_FP32) return fail(NVFP4_ERR_INVALID_ARG, "bad dtype %d", dtype);
    if (rows <= 0 || cols <= 0) return fail(NVFP4_ERR_INVALID_ARG, "empty input [%lld][%lld]", (long long)rows,
                                            (long long)cols);
    if (cols % 16) return fail(NVFP4_ERR_INVALID_ARG, "cols %lld not a multiple of 16", (long long)cols);
    const int esz = dtype == NVFP4_IN_FP32 ? 4 : 2;
    if (ldx < cols || (ldx * esz) % 16)
        return fail(NVFP4_ERR_INVALID_ARG, "ldx %lld must be >= cols and a multiple of 16 bytes", (long long)ldx);
    if (!aligned16(x)) return fail(NVFP4_ERR_INVALID_ARG, "x must be 16-byte aligned");
    if (rows > (int64_t(1) << 40) || cols > (int64_t(1) << 40))
        return fail(NVFP4_ERR_INVALID_ARG, "input too large");
    return NVFP4_OK;
}

nvfp4_status check_workspace(void* ws, size_t bytes) {
    if (!ws || bytes < kSinglePassWorkspaceBytes)
        return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", kSinglePassWorkspaceBytes, bytes);
    if (!aligned16(ws)) return fail(NVFP4_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    return NVFP4_OK;
}

int amax_grid(int64_t rows, int64_t cols, int64_t ldx, bool fp32, int num_sms) {
    // dense: one CTA per chunk of kAmaxThreads * kAmaxUnroll vectors, up to 8
    // CTAs per SM; strided: CTAs walk rows
    const int64_t units = ldx == cols ? ceil_div(rows * cols / (fp32 ? 4 : 8), (int64_t)kAmaxThreads * kAmaxUnroll)
                                      : rows;
    int64_t g = std::min<int64_t>(units, (int64_t)num_sms * 8);
    g = std::min<int64_t>(g, kMaxPartials);
    return (int)std::max<int64_t>(g, 1);
}

// CTAs per SM of the rowwise quantizer.  Every CTA first reduces the amax
// partials and builds its scale table.  With RTN an item is cheap, so that
// start-up dominates a CTA's work: launching only what fits on an SM at once
// (4 CTAs of 256 threads at 64 registers) does it once per resident CTA.
// With SR the items are heavy and many smaller waves balance the SMs better
// (4 CTAs per SM measured slower there).
int row_ctas_per_sm(bool sr) { return sr ? 16 : 4; }

int cap_grid(int64_t units, int per_sm, int num_sms) {
    return (int)std::max<int64_t>(1, std::min<int64_t>(units, (int64_t)num_sms * per_sm));
}

// CTAs of the RHT amax pass: a unit is 16 rows x one 8-byte column vector
int rht_amax_grid(int64_t rows, int64_t cols, bool fp32, int num_sms) {
    const int64_t units = (rows / 16) * (cols / (fp32 ? 2 : 4));
    // one wave of the kernel's 3 CTAs per SM: fewer partials for every
    // encode CTA to reduce than with more, shorter CTAs
    return (int)std::max<int64_t>(1, std::min<int64_t>({ceil_div(units, (int64_t)kRhtAmaxThreads),
                                                       (int64_t)num_sms * 3, (int64_t)kMaxPartials}));
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

size_t nvfp4_scales_bytes(int64_t rows, int64_t cols, int32_t scale_layout) {
    return scales_bytes(rows, cols, scale_layout);
}

size_t nvfp4_workspace_size(void) { return 2 * kSinglePassWorkspaceBytes; }

size_t nvfp4_linear_workspace_size(void) { return 3 * kSinglePassWorkspaceBytes; }

const char* nvfp4_last_error(void) { return g_err; }

const char* nvfp4_status_string(nvfp4_status st) {
    switch (st) {
        case NVFP4_OK: return "ok";
        case NVFP4_ERR_INVALID_ARG: return "invalid argument";
        case NVFP4_ERR_UNSUPPORTED: return "unsupported";
        case NVFP4_ERR_WORKSPACE: return "workspace too small";
        case NVFP4_ERR_NONFINITE: return "non-finite input";
        case NVFP4_ERR_TIMEOUT: return "device wait timed out";
        case NVFP4_ERR_CUDA: return "CUDA error";
        case NVFP4_ERR_BOUNDS: return "device index out of bounds (checked build)";
    }
    return "unknown status";
}

nvfp4_status nvfp4_quantize(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                            nvfp4_block block, nvfp4_round round, uint64_t seed, const nvfp4_tensor* out_rowwise,
                            const nvfp4_tensor* out_colwise, void* workspace, size_t workspace_bytes,
                            nvfp4_stream_t stream) {
    g_err[0] = 0;
    nvfp4_status st = check_input(x, dtype, rows, cols, ldx);
    if (st) return st;
    if (block != NVFP4_BLOCK_1x16 && block != NVFP4_BLOCK_16x16 && block != NVFP4_BLOCK_MX1x32)
        return fail(NVFP4_ERR_INVALID_ARG, "bad block %d", block);
    const bool mx = block == NVFP4_BLOCK_MX1x32;
    const int32_t fmt = mx ? NVFP4_FORMAT_MXFP4 : NVFP4_FORMAT_NVFP4;
    if (round != NVFP4_RTN && round != NVFP4_SR) return fail(NVFP4_ERR_INVALID_ARG, "bad round %d", round);
    if (!out_rowwise && !out_colwise) return fail(NVFP4_ERR_INVALID_ARG, "no output requested");
    if (out_rowwise && (st = check_out(out_rowwise, rows, cols, "out_rowwise"))) return st;
    if (out_colwise) {
        if (rows % 16) return fail(NVFP4_ERR_INVALID_ARG, "colwise output needs rows %% 16 == 0");
        if ((st = check_out(out_colwise, cols, rows, "out_colwise"))) return st;
    }
    if ((out_rowwise && out_rowwise->format != fmt) || (out_colwise && out_colwise->format != fmt))
        return fail(NVFP4_ERR_INVALID_ARG, "output format must be %s for this block", mx ? "MXFP4" : "NVFP4");
    if (mx && ((out_rowwise && cols % 32) || (out_colwise && rows % 32)))
        return fail(NVFP4_ERR_INVALID_ARG, "MXFP4 needs 32-element blocks (cols %% 32 rowwise, rows %% 32 colwise)");
    if (block == NVFP4_BLOCK_16x16) {
        if (rows % 16) return fail(NVFP4_ERR_INVALID_ARG, "16x16 blocks need rows %% 16 == 0");
        if (round != NVFP4_RTN) return fail(NVFP4_ERR_UNSUPPORTED, "16x16 blocks support RTN only");
    }
    if ((st = check_workspace(workspace, workspace_bytes))) return st;
    DeviceInfo* dev;
    if ((st = device_info(&dev))) return st;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool fp32 = dtype == NVFP4_IN_FP32;
    const bool sr = round == NVFP4_SR;
    uint32_t* partials = static_cast<uint32_t*>(workspace);
    if (out_rowwise && (st = zero_scale_padding(out_rowwise, s))) return st;
    if (out_colwise && (st = zero_scale_padding(out_colwise, s))) return st;

    int ag = 0;
    if (!mx) {  // MXFP4 has no tensor scale, hence no amax pass
        ag = amax_grid(rows, cols, ldx, fp32, dev->num_sms);
        launch_amax(x, fp32, rows, cols, ldx, partials, ag, s);
        if ((st = check_launch("amax"))) return st;
    }

    if (block == NVFP4_BLOCK_16x16) {
        const int g = quantize_2d_grid(rows, cols, fp32, dev->num_sms);
        ScaleOut sr_ = out_rowwise ? scale_out(*out_rowwise) : ScaleOut{};
        ScaleOut sc_ = out_colwise ? scale_out(*out_colwise) : ScaleOut{};
        launch_quantize_2d(x, fp32, rows, cols, ldx, partials, ag, out_rowwise ? out_rowwise->codes : nullptr,
                           out_rowwise ? out_rowwise->ld_codes : 0, sr_, out_rowwise ? out_rowwise->amax : nullptr,
                           out_colwise ? out_colwise->codes : nullptr, out_colwise ? out_colwise->ld_codes : 0, sc_,
                           out_colwise ? out_colwise->amax : nullptr, dev->status, g, s);
        return check_launch("quantize_2d");
    }
    if (out_rowwise) {
        const int64_t items = rows * ceil_div(cols / 16, (int64_t)kRowItemBlocks);
        const int g = cap_grid(ceil_div(items, (int64_t)kQuantThreads / 32), row_ctas_per_sm(sr), dev->num_sms);
        launch_quantize_rowwise(x, fp32, rows, cols, ldx, partials, ag, out_rowwise->codes, out_rowwise->ld_codes,
                                scale_out(*out_rowwise), out_rowwise->amax, dev->status, sr, mx, seed, false, 0, g,
                                s);
        if ((st = check_launch("quantize_rowwise"))) return st;
    }
    if (out_colwise) {
        const int g = cap_grid(colwise_tiles(rows, cols), 12, dev->num_sms);
        launch_quantize_colwise(x, fp32, rows, cols, ldx, partials, ag, out_colwise->codes, out_colwise->ld_codes,
                                scale_out(*out_colwise), out_colwise->amax, dev->status, sr, mx, seed, false, 0, g,
                                s);
        if ((st = check_launch("quantize_colwise"))) return st;
    }
    return NVFP4_OK;
}

nvfp4_status nvfp4_rht_quantize(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                                nvfp4_round round, uint64_t seed, uint64_t rht_seed, const nvfp4_tensor* out_colwise,
                                void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
    g_err[0] = 0;
    nvfp4_status st = check_input(x, dtype, rows, cols, ldx);
    if (st) return st;
    if (round != NVFP4_RTN && round != NVFP4_SR) return fail(NVFP4_ERR_INVALID_ARG, "bad round %d", round);
    if (!out_colwise) return fail(NVFP4_ERR_INVALID_ARG, "out_colwise is null");
    if (rows % 16) return fail(NVFP4_ERR_INVALID_ARG, "RHT needs rows %% 16 == 0");
    if ((st = check_out(out_colwise, cols, rows, "out_colwise"))) return st;
    const bool mx = out_colwise->format == NVFP4_FORMAT_MXFP4;
    if (mx && rows % 32) return fail(NVFP4_ERR_INVALID_ARG, "MXFP4 needs rows %% 32 == 0");
    if ((st = check_workspace(workspace, workspace_bytes))) return st;
    DeviceInfo* dev;
    if ((st = device_info(&dev))) return st;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool fp32 = dtype == NVFP4_IN_FP32;
    uint32_t* partials = static_cast<uint32_t*>(workspace);
    if ((st = zero_scale_padding(out_colwise, s))) return st;
    int ag = 0;
    if (!mx) {
        ag = rht_amax_grid(rows, cols, fp32, dev->num_sms);
        launch_rht_amax(x, fp32, rows, cols, ldx, rht_seed, partials, ag, s);
        if ((st = check_launch("rht_amax"))) return st;
    }
    const int g = cap_grid(colwise_tiles(rows, cols), 12, dev->num_sms);
    launch_quantize_colwise(x, fp32, rows, cols, ldx, partials, ag, out_colwise->codes, out_colwise->ld_codes,
                            scale_out(*out_colwise), out_colwise->amax, dev->status, round == NVFP4_SR, mx, seed,
                            true, rht_seed, g, s);
    return check_launch("rht_quantize_colwise");
}

nvfp4_status nvfp4_quantize_with_rht(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                                     nvfp4_round round, uint64_t seed, uint64_t rht_seed,
                                     const nvfp4_tensor* out_rowwise, const nvfp4_tensor* out_colwise,
                                     void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
    g_err[0] = 0;
    nvfp4_status st = check_input(x, dtype, rows, cols, ldx);
    if (st) return st;
    if (round != NVFP4_RTN && round != NVFP4_SR) return fail(NVFP4_ERR_INVALID_ARG, "bad round %d", round);
    if (!out_rowwise || !out_colwise) return fail(NVFP4_ERR_INVALID_ARG, "both outputs are required");
    if (rows % 16) return fail(NVFP4_ERR_INVALID_ARG, "RHT needs rows %% 16 == 0");
    if ((st = check_out(out_rowwise, rows, cols, "out_rowwise")) || (st = check_out(out_colwise, cols, rows, "out_colwise")))
        return st;
    if (out_rowwise->format != NVFP4_FORMAT_NVFP4 || out_colwise->format != NVFP4_FORMAT_NVFP4)
        return fail(NVFP4_ERR_INVALID_ARG, "outputs must have format NVFP4 (MXFP4 has no amax pass to share)");
    if (!workspace || workspace_bytes < 2 * kSinglePassWorkspaceBytes)
        return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", 2 * kSinglePassWorkspaceBytes,
                    workspace_bytes);
    if (!aligned16(workspace)) return fail(NVFP4_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    DeviceInfo* dev;
    if ((st = device_info(&dev))) return st;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool fp32 = dtype == NVFP4_IN_FP32;
    const bool sr = round == NVFP4_SR;
    uint32_t* partials_rht = static_cast<uint32_t*>(workspace);
    uint32_t* partials_plain = partials_rht + kMaxPartials;
    if ((st = zero_scale_padding(out_rowwise, s)) || (st = zero_scale_padding(out_colwise, s))) return st;
    // one read of x for both tensor scales: amax of the transform and of x
    const int ag = rht_amax_grid(rows, cols, fp32, dev->num_sms);
    launch_rht_amax(x, fp32, rows, cols, ldx, rht_seed, partials_rht, ag, s, partials_plain);
    if ((st = check_launch("rht_amax"))) return st;
    const int64_t items = rows * ceil_div(cols / 16, (int64_t)kRowItemBlocks);
    const int gr = cap_grid(ceil_div(items, (int64_t)kQuantThreads / 32), row_ctas_per_sm(sr), dev->num_sms);
    const int gc = cap_grid(colwise_tiles(rows, cols), 12, dev->num_sms);
    // SR: the two encodes are issue-bound; on two streams each fills the
    // other's tail (dY 8192x20480: 0.411 -> 0.394 ms)
    return fork_join(
        s, sr,
        [&](cudaStream_t rs) {
            launch_quantize_rowwise(x, fp32, rows, cols, ldx, partials_plain, ag, out_rowwise->codes,
                                    out_rowwise->ld_codes, scale_out(*out_rowwise), out_rowwise->amax, dev->status, sr,
                                    false, seed, false, 0, gr, rs);
            return check_launch("quantize_rowwise");
        },
        [&]() {
            launch_quantize_colwise(x, fp32, rows, cols, ldx, partials_rht, ag, out_colwise->codes,
                                    out_colwise->ld_codes, scale_out(*out_colwise), out_colwise->amax, dev->status, sr,
                                    false, seed, true, rht_seed, gc, s);
            return check_launch("rht_quantize_colwise");
        });
}

nvfp4_status nvfp4_rht_quantize_rowwise(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                                        nvfp4_round round, uint64_t seed, uint64_t rht_seed,
                                        const nvfp4_tensor* out_rowwise, void* workspace, size_t workspace_bytes,
                                        nvfp4_stream_t stream) {
    g_err[0] = 0;
    nvfp4_status st = check_input(x, dtype, rows, cols, ldx);
    if (st) return st;
    if (round != NVFP4_RTN && round != NVFP4_SR) return fail(NVFP4_ERR_INVALID_ARG, "bad round %d", round);
    if (!out_rowwise) return fail(NVFP4_ERR_INVALID_ARG, "out_rowwise is null");
    if ((st = check_out(out_rowwise, rows, cols, "out_rowwise"))) return st;
    const bool mx = out_rowwise->format == NVFP4_FORMAT_MXFP4;
    if (mx && cols % 32) return fail(NVFP4_ERR_INVALID_ARG, "MXFP4 needs cols %% 32 == 0");
    if ((st = check_workspace(workspace, workspace_bytes))) return st;
    DeviceInfo* dev;
    if ((st = device_info(&dev))) return st;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool fp32 = dtype == NVFP4_IN_FP32;
    uint32_t* partials = static_cast<uint32_t*>(workspace);
    if ((st = zero_scale_padding(out_rowwise, s))) return st;
    const int64_t items = rows * ceil_div(cols / 16, (int64_t)kRowItemBlocks);
    int ag = 0;
    if (!mx) {
        ag = (int)std::max<int64_t>(1, std::min<int64_t>({ceil_div(items, (int64_t)kQuantThreads / 32),
                                                           (int64_t)dev->num_sms * 8, (int64_t)kMaxPartials}));
        launch_rht_rows_amax(x, fp32, rows, cols, ldx, rht_seed, partials, ag, s);
        if ((st = check_launch("rht_rows_amax"))) return st;
    }
    const int g =
        cap_grid(ceil_div(items, (int64_t)kQuantThreads / 32), row_ctas_per_sm(round == NVFP4_SR), dev->num_sms);
    launch_quantize_rowwise(x, fp32, rows, cols, ldx, partials, ag, out_rowwise->codes, out_rowwise->ld_codes,
                            scale_out(*out_rowwise), out_rowwise->amax, dev->status, round == NVFP4_SR, mx, seed,
                            true, rht_seed, g, s);
    return check_launch("rht_quantize_rowwise");
}

namespace {
// Checks one block-scaled GEMM's arguments (host only) and fills its launch
// arguments but the device's (gemm_device).
nvfp4_status gemm_args(const nvfp4_tensor* A, const nvfp4_tensor* B, void* C, nvfp4_out_dtype out_dtype, int64_t ldc,
                       GemmArgs* g) {
    if (!A || !B || !C) return fail(NVFP4_ERR_INVALID_ARG, "null argument");
    nvfp4_status st;
    if ((st = check_out(A, A->rows, A->cols, "A")) || (st = check_out(B, B->rows, B->cols, "B"))) return st;
    if (A->rows <= 0 || B->rows <= 0 || A->cols <= 0) return fail(NVFP4_ERR_INVALID_ARG, "empty GEMM");
    if (A->cols != B->cols)
        return fail(NVFP4_ERR_INVALID_ARG, "K mismatch: %lld vs %lld", (long long)A->cols, (long long)B->cols);
    if (A->cols % 64) return fail(NVFP4_ERR_INVALID_ARG, "K %lld not a multiple of 64", (long long)A->cols);
    if (A->scale_layout != NVFP4_SCALES_MMA || B->scale_layout != NVFP4_SCALES_MMA)
        return fail(NVFP4_ERR_INVALID_ARG, "GEMM operands need NVFP4_SCALES_MMA scales");
    if (!aligned16(A->scales) || !aligned16(B->scales))
        return fail(NVFP4_ERR_INVALID_ARG, "GEMM scale buffers must be 16-byte aligned");
    if (A->format != B->format) return fail(NVFP4_ERR_INVALID_ARG, "GEMM operands must share one format");
    if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32 && out_dtype != NVFP4_OUT_FP32_ADD)
        return fail(NVFP4_ERR_INVALID_ARG, "bad out_dtype %d", out_dtype);
    const int esz = out_dtype == NVFP4_OUT_BF16 ? 2 : 4;
    if (ldc < B->rows || (ldc * esz) % 16 || !aligned16(C))
        return fail(NVFP4_ERR_INVALID_ARG, "C: ldc must be >= N and 16-byte rows, C 16-byte aligned");
    g->a_codes = A->codes;
    g->a_scales = A->scales;
    g->a_amax = A->amax;
    g->lda = A->ld_codes;
    g->b_codes = B->codes;
    g->b_scales = B->scales;
    g->b_amax = B->amax;
    g->ldb = B->ld_codes;
    g->c = C;
    g->ldc = ldc;
    g->M = A->rows;
    g->N = B->rows;
    g->K = A->cols;
    g->out_fp32 = out_dtype != NVFP4_OUT_BF16;
    g->accumulate = out_dtype == NVFP4_OUT_FP32_ADD;
    g->mx = A->format == NVFP4_FORMAT_MXFP4;
    g->timeout_ns = g_wait_limit_ns.load();
    return NVFP4_OK;
}

// The current device's part of a GEMM's launch arguments.
nvfp4_status gemm_device(GemmArgs* g) {
    DeviceInfo* dev;
    nvfp4_status st;
    if ((st = device_info(&dev))) return st;
    g->status = dev->status;
    g->num_sms = dev->num_sms;
    return NVFP4_OK;
}

nvfp4_status gemm_launch_status(int e, const char* msg) {
    if (e == -1) return fail(NVFP4_ERR_UNSUPPORTED, "gemm: %s", msg ? msg : "unsupported");
    if (e) return fail(NVFP4_ERR_CUDA, "gemm: %s", msg ? msg : cudaGetErrorString((cudaError_t)e));
    return check_launch("gemm");
}
}  // namespace

nvfp4_status nvfp4_gemm(const nvfp4_tensor* A, const nvfp4_tensor* B, void* C, nvfp4_out_dtype out_dtype,
                        int64_t ldc, void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    g_err[0] = 0;
    GemmArgs g;
    nvfp4_status st;
    if ((st = gemm_args(A, B, C, out_dtype, ldc, &g)) || (st = gemm_device(&g))) return st;
    const char* msg = nullptr;
    const int e = launch_gemm(g, reinterpret_cast<cudaStream_t>(stream), &msg);
    return gemm_launch_status(e, msg);
}

nvfp4_status nvfp4_gemm_pair(const nvfp4_tensor* A0, const nvfp4_tensor* B0, void* C0, nvfp4_out_dtype out_dtype0,
                             int64_t ldc0, const nvfp4_tensor* A1, const nvfp4_tensor* B1, void* C1,
                             nvfp4_out_dtype out_dtype1, int64_t ldc1, nvfp4_stream_t stream) {
    g_err[0] = 0;
    GemmArgs g0, g1;
    nvfp4_status st;
    if ((st = gemm_args(A0, B0, C0, out_dtype0, ldc0, &g0)) || (st = gemm_args(A1, B1, C1, out_dtype1, ldc1, &g1)))
        return st;
    if (g0.mx != g1.mx) return fail(NVFP4_ERR_INVALID_ARG, "the two GEMMs must share one operand format");
    if ((st = gemm_device(&g0)) || (st = gemm_device(&g1))) return st;
    const char* msg = nullptr;
    const int e = launch_gemm_pair(g0, g1, reinterpret_cast<cudaStream_t>(stream), &msg);
    return gemm_launch_status(e, msg);
}

nvfp4_status nvfp4_gemm_bf16(const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                             nvfp4_out_dtype out_dtype, int64_t ldc, int64_t M, int64_t N, int64_t K,
                             nvfp4_stream_t stream) {
    g_err[0] = 0;
    if (!A || !B || !C) return fail(NVFP4_ERR_INVALID_ARG, "null argument");
    if (M <= 0 || N <= 0 || K <= 0) return fail(NVFP4_ERR_INVALID_ARG, "empty GEMM");
    if (K % 8) return fail(NVFP4_ERR_INVALID_ARG, "K %lld not a multiple of 8", (long long)K);
    if (lda < K || ldb < K || lda % 8 || ldb % 8)
        return fail(NVFP4_ERR_INVALID_ARG, "lda, ldb must be >= K and multiples of 8 elements");
    if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32 && out_dtype != NVFP4_OUT_FP32_ADD)
        return fail(NVFP4_ERR_INVALID_ARG, "bad out_dtype %d", out_dtype);
    const int esz = out_dtype == NVFP4_OUT_BF16 ? 2 : 4;
    if (ldc < N || (ldc * esz) % 16) return fail(NVFP4_ERR_INVALID_ARG, "ldc must be >= N with 16-byte rows");
    if (!aligned16(A) || !aligned16(B) || !aligned16(C))
        return fail(NVFP4_ERR_INVALID_ARG, "A, B, C must be 16-byte aligned");
    DeviceInfo* dev;
    nvfp4_status st;
    if ((st = device_info(&dev))) return st;
    GemmBf16Args g;
    g.a = A;
    g.b = B;
    g.c = C;
    g.lda = lda;
    g.ldb = ldb;
    g.ldc = ldc;
    g.M = M;
    g.N = N;
    g.K = K;
    g.out_fp32 = out_dtype != NVFP4_OUT_BF16;
    g.accumulate = out_dtype == NVFP4_OUT_FP32_ADD;
    g.timeout_ns = g_wait_limit_ns.load();
    g.status = dev->status;
    g.num_sms = dev->num_sms;
    const char* msg = nullptr;
    int e = launch_gemm_bf16(g, reinterpret_cast<cudaStream_t>(stream), &msg);
    if (e == -1) return fail(NVFP4_ERR_UNSUPPORTED, "gemm_bf16: %s", msg ? msg : "unsupported");
    if (e) return fail(NVFP4_ERR_CUDA, "gemm_bf16: %s", msg ? msg : cudaGetErrorString((cudaError_t)e));
    return check_launch("gemm_bf16");
}

static nvfp4_status check_linear_tensor(const nvfp4_tensor* t, int64_t rows, int64_t cols, const char* name) {
    nvfp4_status st = check_out(t, rows, cols, name);
    if (st) return st;
    if (t->scale_layout != NVFP4_SCALES_MMA)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: needs NVFP4_SCALES_MMA", name);
    return NVFP4_OK;
}

nvfp4_status nvfp4_transpose_bf16(const void* x, int64_t rows, int64_t cols, int64_t ldx, void* y, int64_t ldy,
                                  nvfp4_stream_t stream) {
    g_err[0] = 0;
    if (!x || !y) return fail(NVFP4_ERR_INVALID_ARG, "null argument");
    if (rows <= 0 || cols <= 0 || rows % 8 || cols % 8)
        return fail(NVFP4_ERR_INVALID_ARG, "rows and cols must be positive multiples of 8, got %lld x %lld",
                    (long long)rows, (long long)cols);
    if (ldx < cols || ldx % 8 || ldy < rows || ldy % 8)
        return fail(NVFP4_ERR_INVALID_ARG, "ldx (>= cols) and ldy (>= rows) must be multiples of 8 elements");
    if (!aligned16(x) || !aligned16(y)) return fail(NVFP4_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
    DeviceInfo* dev;
    nvfp4_status st;
    if ((st = device_info(&dev))) return st;
    const int64_t units = (rows / 8) * (cols / 8);
    const int grid = cap_grid(ceil_div(units, (int64_t)256), 8, dev->num_sms);
    launch_transpose_bf16(x, rows, cols, ldx, y, ldy, grid, reinterpret_cast<cudaStream_t>(stream));
    return check_launch("transpose_bf16");
}

namespace {
// X's quantization for the forward: xq (1x16 RTN) and, with_rht, X^T's RHT
// codes in xtq from the same amax read; workspace: the first 16 KB.
nvfp4_status linear_quantize_x(const void* X, bool with_rht, uint64_t rht_seed, nvfp4_linear_ctx* ctx,
                               nvfp4_stream_t stream) {
    const int64_t M = ctx->M, K = ctx->K;
    if (with_rht)
        // X 1x16 RTN for Fprop and X^T after the RHT along the tokens, RTN,
        // for Wgrad: both tensor scales from one read of X
        return nvfp4_quantize_with_rht(X, NVFP4_IN_BF16, M, K, K, NVFP4_RTN, 0, rht_seed, &ctx->xq, &ctx->xtq,
                                       ctx->workspace, 2 * kSinglePassWorkspaceBytes, stream);
    return nvfp4_quantize(X, NVFP4_IN_BF16, M, K, K, NVFP4_BLOCK_1x16, NVFP4_RTN, 0, &ctx->xq, nullptr,
                          ctx->workspace, kSinglePassWorkspaceBytes, stream);
}

// The forward pass; with_rht: X^T's RHT codes (xtq) as well, from the same
// amax read of X.  With the larger workspace, W's quantization (its own 8 KB
// of the workspace) runs on the device's second stream, forked from and
// joined back into `stream` by events, while X's runs on `stream`.
nvfp4_status linear_fwd(const void* X, const void* W, void* Y, bool with_rht, uint64_t rht_seed,
                        nvfp4_linear_ctx* ctx, nvfp4_stream_t stream) {
    g_err[0] = 0;
    if (!ctx || !X || !W || !Y) return fail(NVFP4_ERR_INVALID_ARG, "null argument");
    const int64_t M = ctx->M, N = ctx->N, K = ctx->K;
    if (M <= 0 || N <= 0 || K <= 0 || M % 64 || N % 64 || K % 64)
        return fail(NVFP4_ERR_INVALID_ARG, "M, N, K must be positive multiples of 64");
    nvfp4_status st;
    if ((st = check_linear_tensor(&ctx->xq, M, K, "xq")) || (st = check_linear_tensor(&ctx->wq, N, K, "wq")) ||
        (st = check_linear_tensor(&ctx->wtq, K, N, "wtq")))
        return st;
    if (with_rht && (st = check_linear_tensor(&ctx->xtq, K, M, "xtq"))) return st;
    if (!ctx->workspace || ctx->workspace_bytes < nvfp4_workspace_size())
        return fail(NVFP4_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", nvfp4_workspace_size(),
                    ctx->workspace_bytes);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // W's quantization (its own 8 KB of the larger workspace) beside X's
    const bool two_streams = ctx->workspace_bytes >= nvfp4_linear_workspace_size();
    void* ws_w = static_cast<uint8_t*>(ctx->workspace) + (two_streams ? 2 * kSinglePassWorkspaceBytes : 0);
    if ((st = fork_join(
             s, two_streams,
             [&](cudaStream_t ws) {
                 return nvfp4_quantize(W, NVFP4_IN_BF16, N, K, K, NVFP4_BLOCK_16x16, NVFP4_RTN, 0, &ctx->wq, &ctx->wtq,
                                       ws_w, kSinglePassWorkspaceBytes, reinterpret_cast<nvfp4_stream_t>(ws));
             },
             [&]() { return linear_quantize_x(X, with_rht, rht_seed, ctx, stream); })))
        return st;
    return nvfp4_gemm(&ctx->xq, &ctx->wq, Y, NVFP4_OUT_BF16, N, nullptr, 0, stream);
}
}  // namespace

nvfp4_status nvfp4_linear_fwd(const void* X, const void* W, void* Y, nvfp4_linear_ctx* ctx, nvfp4_stream_t stream) {
    return linear_fwd(X, W, Y, false, 0, ctx, stream);
}

nvfp4_status nvfp4_linear_fwd_rht(const void* X, const void* W, void* Y, uint64_t rht_seed, nvfp4_linear_ctx* ctx,
                                  nvfp4_stream_t stream) {
    return linear_fwd(X, W, Y, true, rht_seed, ctx, stream);
}

nvfp4_status nvfp4_linear_bwd(const void* dY, const void* X, void* dX, float* dW, uint64_t sr_seed,
                              uint64_t rht_seed, nvfp4_linear_ctx* ctx, nvfp4_stream_t stream) {
    g_err[0] = 0;
    if (!ctx || !dY || !dX || !dW) return fail(NVFP4_ERR_INVALID_ARG, "null argument");
    const int64_t M = ctx->M, N = ctx->N, K = ctx->K;
    if (M <= 0 || N <= 0 || K <= 0 || M % 64 || N % 64 || K % 64)
        return fail(NVFP4_ERR_INVALID_ARG, "M, N, K must be positive multiples of 64");
    nvfp4_status st;
    if ((st = check_linear_tensor(&ctx->wtq, K, N, "wtq")) || (st = check_linear_tensor(&ctx->dyq, M, N, "dyq")) ||
        (st = check_linear_tensor(&ctx->dytq, N, M, "dytq")) || (st = check_linear_tensor(&ctx->xtq, K, M, "xtq")))
        return st;
    // dY with SR, for both GEMMs from one amax read: rowwise for Dgrad, and
    // transformed along the tokens, transposed, for Wgrad
    if ((st = nvfp4_quantize_with_rht(dY, NVFP4_IN_BF16, M, N, N, NVFP4_SR, sr_seed, rht_seed, &ctx->dyq, &ctx->dytq,
                                      ctx->workspace, ctx->workspace_bytes, stream)))
        return st;
    // Wgrad's X operand: X^T transformed along the tokens (X null: xtq
    // already holds X^T's codes from nvfp4_linear_fwd_rht)
    if (X && (st = nvfp4_rht_quantize(X, NVFP4_IN_BF16, M, K, K, NVFP4_RTN, 0, rht_seed, &ctx->xtq, ctx->workspace,
                                      ctx->workspace_bytes, stream)))
        return st;
    // Dgrad dX = dY W (the 16x16 weight codes of W^T) and Wgrad dW = dY^T X
    // (both operands transformed along the tokens) in one launch
    return nvfp4_gemm_pair(&ctx->dyq, &ctx->wtq, dX, NVFP4_OUT_BF16, K, &ctx->dytq, &ctx->xtq, dW,
                           ctx->dw_accumulate ? NVFP4_OUT_FP32_ADD : NVFP4_OUT_FP32, K, stream);
}

// ---------------------------------------------------------------------------
// Quantize without a caller workspace.
//
// The amax pass of nvfp4_quantize keeps one 32-bit partial maximum per CTA
// (at most kMaxPartials of them) in scratch memory.  nvfp4_quantize_noalloc
// keeps that scratch in the fixed array below instead, so a caller that has
// no way to obtain device memory can still quantize.  The array is 8 KB and
// lives on every device that loads this library until the process exits.
// Every call on a device uses the same array: calls whose work overlaps on
// the GPU (different streams, no ordering between them) race on it.  Nothing
// in it has to start at zero: each call's amax pass writes every slot that
// the same call's encode pass reads.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kMaxPartials];
// nvfp4_quantize's workspace check is what the array must satisfy.
static_assert(sizeof(g_noalloc_scratch) >= kSinglePassWorkspaceBytes,
              "the fixed scratch array must hold one amax pass's partials");

namespace nvfp4 {
namespace {

void* g_noalloc_ptr[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the first call on a device does this).
nvfp4_status noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(NVFP4_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

nvfp4_status nvfp4_quantize_noalloc(const void* x, nvfp4_in_dtype dtype, int64_t rows, int64_t cols, int64_t ldx,
                                    nvfp4_block block, nvfp4_round round, uint64_t seed,
                                    const nvfp4_tensor* out_rowwise, const nvfp4_tensor* out_colwise,
                                    nvfp4_stream_t stream) {
    g_err[0] = 0;
    // the array covers nvfp4_quantize's workspace requirement for any shape
    // (checked at compile time above), so no size can exceed it
    void* scratch = nullptr;
    nvfp4_status st = noalloc_scratch(&scratch);
    if (st) return st;
    return nvfp4_quantize(x, dtype, rows, cols, ldx, block, round, seed, out_rowwise, out_colwise, scratch,
                          sizeof(g_noalloc_scratch), stream);
}

uint64_t nvfp4_set_wait_limit_ns(uint64_t limit_ns) { return g_wait_limit_ns.exchange(limit_ns); }

nvfp4_status nvfp4_sync_status(nvfp4_stream_t stream) {
    g_err[0] = 0;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    uint32_t word = 0;
    e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof word);
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaMemcpyFromSymbol: %s", cudaGetErrorString(e));
    if (word) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero);
        if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaMemcpyToSymbol: %s", cudaGetErrorString(e));
    }
    if (word & kStatusBounds) return fail(NVFP4_ERR_BOUNDS, "a device index fell outside its tensor (checked build)");
    if (word & kStatusTimeout) return fail(NVFP4_ERR_TIMEOUT, "a device wait ran out of iterations");
    if (word & kStatusNonfinite) return fail(NVFP4_ERR_NONFINITE, "input held a NaN or an infinity");
    return NVFP4_OK;
}

int32_t nvfp4_checked_build(void) {
#ifdef NVFP4_CHECKED
    return 1;
#else
    return 0;
#endif
}

nvfp4_status nvfp4_checked_selftest(nvfp4_stream_t stream) {
    g_err[0] = 0;
#ifndef NVFP4_CHECKED
    (void)stream;
    return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_checked_selftest needs the checked build");
#else
    DeviceInfo* dev;
    nvfp4_status st = device_info(&dev);
    if (st) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint32_t zero[3] = {0u, 0u, 0u};
    cudaError_t e = cudaMemcpyToSymbolAsync(g_selftest_words, zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaMemcpyToSymbolAsync: %s", cudaGetErrorString(e));
    checked_selftest_kernel<<<1, 1, 0, s>>>(dev->status);
    if ((st = check_launch("checked_selftest"))) return st;
    st = nvfp4_sync_status(stream);
    uint32_t words[3];
    e = cudaMemcpyFromSymbol(words, g_selftest_words, sizeof words);
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "cudaMemcpyFromSymbol: %s", cudaGetErrorString(e));
    if (words[2] != 0u) return fail(NVFP4_ERR_CUDA, "the guarded store past the buffer was not skipped");
    return st;
#endif
}

}  // extern "C"

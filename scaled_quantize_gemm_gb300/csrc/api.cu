// api.cu -- the extern "C" boundary declared in include/fp8sq.h.
// Validates every argument on the host before anything is enqueued, checks
// that the current device is sm_103, then hands off to the launchers.
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

#include "../../include/fp8sq.h"
#include "internal.h"

namespace {

thread_local char g_msg[512] = "no error";

int fail(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Per-device facts, queried once.  `packed` is 0 until the first query has
// finished, then (major << 24) | (minor << 16) | sms, published with one
// atomic store so concurrent callers see either nothing or all of it.
std::atomic<uint32_t> g_dev[64];

// current device must be sm_103; returns its SM count through *sms
int check_device(int* sms)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fail(FP8SQ_ERR_CUDA, "no usable CUDA device (%s)", cudaGetErrorString(e));
    }
    uint32_t packed = g_dev[dev].load(std::memory_order_acquire);
    if (packed == 0) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return fail(FP8SQ_ERR_CUDA, "cannot query device %d", dev);
        }
        packed = ((uint32_t)major << 24) | ((uint32_t)(minor & 0xFF) << 16) | ((uint32_t)n & 0xFFFFu);
        g_dev[dev].store(packed, std::memory_order_release);
    }
    const int major = (int)(packed >> 24), minor = (int)((packed >> 16) & 0xFF);
    if (!(major == 10 && minor == 3))
        return fail(FP8SQ_ERR_WRONG_ARCH, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
    *sms = (int)(packed & 0xFFFFu);
    return FP8SQ_OK;
}

int cuda_status(cudaError_t e, const char* what)
{
    if (e == cudaSuccess) return FP8SQ_OK;
    cudaGetLastError();
    return fail(FP8SQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool valid_format(int f) { return f == FP8SQ_E4M3 || f == FP8SQ_E5M2; }
bool valid_dtype(int d) { return d == FP8SQ_BF16 || d == FP8SQ_F32; }
bool valid_gran(int g) { return g >= FP8SQ_TENSOR && g <= FP8SQ_MX32_FLOOR_TILED; }
bool column_gran(int g) { return g == FP8SQ_TILE_128x1 || g == FP8SQ_MX32_COL_TILED; }
bool e8m0_tiled(int g)
{
    return g == FP8SQ_MX32_TILED || g == FP8SQ_MX32_COL_TILED || g == FP8SQ_TILE_1x128_POW2 ||
           g == FP8SQ_BLOCK_128x128_POW2 || g == FP8SQ_MX32_FLOOR_TILED;
}

const int64_t kMaxDim = (int64_t)1 << 31;  // GEMM / TMA coordinates are 32-bit

// per-unit layout checks shared by amax and quantize
int check_units(int gran, int64_t rows, int64_t cols)
{
    if (gran == FP8SQ_TILE_1x128 && cols % 128)
        return fail(FP8SQ_ERR_UNSUPPORTED, "1x128 tiles need cols %% 128 == 0 (cols = %lld)", (long long)cols);
    if (gran == FP8SQ_BLOCK_128x128 && (rows % 128 || cols % 128))
        return fail(FP8SQ_ERR_UNSUPPORTED, "128x128 blocks need rows, cols %% 128 == 0 (%lld x %lld)", (long long)rows, (long long)cols);
    if (gran == FP8SQ_MX32 && cols % 32)
        return fail(FP8SQ_ERR_UNSUPPORTED, "MX-32 blocks need cols %% 32 == 0 (cols = %lld)", (long long)cols);
    if (e8m0_tiled(gran) && (rows % 128 || cols % 128))
        return fail(FP8SQ_ERR_UNSUPPORTED, "tiled MX-32 scales need rows, cols %% 128 == 0 (%lld x %lld)", (long long)rows, (long long)cols);
    if (gran == FP8SQ_TILE_128x1 && (rows % 128 || cols % 16))
        return fail(FP8SQ_ERR_UNSUPPORTED, "128x1 column tiles need rows %% 128 == 0 and cols %% 16 == 0 (%lld x %lld)", (long long)rows, (long long)cols);
    return FP8SQ_OK;
}

// workspace layout of the linear layer (offsets in bytes, 256-byte aligned)
struct WsLayout {
    size_t qx = 0, qxT = 0, qw = 0, qwT = 0, qdy = 0, qdyT = 0;
    size_t sx = 0, sxT = 0, sw = 0, swT = 0, sdy = 0, sdyT = 0, scal = 0, total = 0;
};
size_t al256(size_t v) { return (v + 255) & ~size_t(255); }
// TENSOR: codes of x, W, dy + 8 scalars (the backward GEMMs read the codes
//   MN-major, so no transposed copies are kept).
// TILE_1x128: codes and their transposed or column-unit counterparts; x
//   tiles [M][K/128] and column tiles [M/128][K]; W blocks and their
//   transpose; dy tiles [M][N/128] and column tiles [M/128][N].
// MX32: x, W, dy in row blocks and column blocks, tiled E8M0 scales.
// TILE_1x128_POW2: as MX32 in size and layout: x and dy in power-of-two
//   1x128 tiles and 128x1 column tiles, W in power-of-two 128x128 blocks
//   and their transpose, every scale as tiled E8M0 codes.
WsLayout ws_layout(int64_t M, int64_t N, int64_t K, int gran)
{
    WsLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += al256(bytes); return o; };
    L.qx = take((size_t)(M * K));
    L.qw = take((size_t)(N * K));
    L.qdy = take((size_t)(M * N));
    if (gran != FP8SQ_TENSOR) {
        L.qxT = take((size_t)(M * K));
        L.qwT = take((size_t)(N * K));
        L.qdyT = take((size_t)(M * N));
    }
    if (gran == FP8SQ_TENSOR) {
        L.scal = take(8 * sizeof(float));   // sx, sw, sdy, ax, aw, ady
    } else if (gran == FP8SQ_TILE_1x128) {
        L.sx = take((size_t)(M * (K / 128)) * sizeof(float));
        L.sxT = take((size_t)((M / 128) * K) * sizeof(float));
        L.sw = take((size_t)((N / 128) * (K / 128)) * sizeof(float));
        L.swT = take((size_t)((N / 128) * (K / 128)) * sizeof(float));
        L.sdy = take((size_t)(M * (N / 128)) * sizeof(float));
        L.sdyT = take((size_t)((M / 128) * N) * sizeof(float));
    } else {
        L.sx = take((size_t)(M * (K / 32)));
        L.sxT = take((size_t)(M * (K / 32)));
        L.sw = take((size_t)(N * (K / 32)));
        L.swT = take((size_t)(N * (K / 32)));
        L.sdy = take((size_t)(M * (N / 32)));
        L.sdyT = take((size_t)(M * (N / 32)));
    }
    L.total = off;
    return L;
}

// A non-blocking side stream and its fork / join events, one set per host
// thread and device: a caller's stream forks work onto it and waits for it
// again within one call, so no two calls share a set concurrently.  Created
// on first use outside stream capture (while `st` is being captured, a call
// without a set yet gets none and runs serially) and kept for the life of the
// thread.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
int side_stream(cudaStream_t st, SideStream** out)
{
    thread_local SideStream per_dev[64];
    *out = nullptr;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fail(FP8SQ_ERR_CUDA, "no usable CUDA device for the side stream");
    }
    SideStream& ss = per_dev[dev];
    if (!ss.s) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
            cudaGetLastError();
            return FP8SQ_OK;
        }
        if (cs != cudaStreamCaptureStatusNone) return FP8SQ_OK;
        cudaStream_t s = nullptr;
        cudaEvent_t fork = nullptr, join = nullptr;
        if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
            e = cudaGetLastError();
            if (join) cudaEventDestroy(join);
            if (fork) cudaEventDestroy(fork);
            if (s) cudaStreamDestroy(s);
            return fail(FP8SQ_ERR_CUDA, "cannot create the side stream (%s)", cudaGetErrorString(e));
        }
        ss.s = s;
        ss.fork = fork;
        ss.join = join;
    }
    *out = &ss;
    return FP8SQ_OK;
}

}  // namespace

namespace fp8sq {
int api_fail(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return code;
}
int api_check_device(int* sms) { return check_device(sms); }

}  // namespace fp8sq

extern "C" {

FP8SQ_API int fp8_abi_version(void) { return 7; }

FP8SQ_API const char* fp8_last_error(void) { return g_msg; }

FP8SQ_API int fp8_device_status(int clear)
{
    // the GEMM kernels are the ones with device-side waits (the casts have none)
    const int v = fp8sq::read_device_error(clear);
    if (v < 0) return fail(FP8SQ_ERR_CUDA, "cannot read the device error word");
    if (v) return fail(FP8SQ_ERR_TIMEOUT, "a bounded device-side wait ran out");
    return FP8SQ_OK;
}

FP8SQ_API int fp8_selftest_wait_timeout(int limit_us, int* waited_out, void* stream)
{
    if (!waited_out) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_selftest_wait_timeout: null waited_out");
    if (limit_us < 1 || limit_us > 1000000) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_selftest_wait_timeout: limit 1 us .. 1 s");
    if (!aligned4(waited_out)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_selftest_wait_timeout: waited_out alignment");
    int sms, r;
    if ((r = check_device(&sms))) return r;
    return cuda_status(fp8sq::launch_selftest_wait((uint64_t)limit_us * 1000ull, waited_out,
                                                   static_cast<cudaStream_t>(stream)),
                       "fp8_selftest_wait_timeout launch");
}

FP8SQ_API int fp8_amax(const void* x, int x_dtype, int64_t rows, int64_t cols, int gran, float* amax_out,
                       void* stream)
{
    if ((!x && rows * cols != 0) || !amax_out) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_amax: null pointer");
    if (!valid_dtype(x_dtype) || !valid_gran(gran) || gran > FP8SQ_MX32)
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_amax: bad dtype or granularity");
    if (rows < 0 || cols < 0) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_amax: negative size");
    if (!aligned16(x)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_amax: x must be 16-byte aligned");
    if (!aligned4(amax_out)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_amax: amax_out must be 4-byte aligned");
    int r = check_units(gran, rows, cols);
    if (r) return r;
    int sms;
    if ((r = check_device(&sms))) return r;
    fp8sq::QuantArgs a;
    a.x = x;
    a.x_dtype = x_dtype;
    a.rows = rows;
    a.cols = cols;
    a.gran = gran;
    a.amax = amax_out;
    return cuda_status(fp8sq::launch_amax(a, static_cast<cudaStream_t>(stream), sms), "fp8_amax launch");
}

FP8SQ_API int fp8_scale_init(float* states, int n_states, int history_len, void* stream)
{
    if (!states) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_scale_init: null states");
    if (n_states < 0 || history_len < 1 || history_len > 4096)
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_scale_init: bad n_states / history_len");
    if (!aligned4(states)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_scale_init: states must be 4-byte aligned");
    int sms, r;
    if ((r = check_device(&sms))) return r;
    return cuda_status(fp8sq::launch_scale_init(states, n_states, history_len, static_cast<cudaStream_t>(stream)),
                       "fp8_scale_init launch");
}

FP8SQ_API int fp8_update_scale(float* states, int n_states, int history_len, const int* formats, int algo,
                               void* stream)
{
    if (!states || !formats) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_update_scale: null pointer");
    if (n_states < 0 || n_states > 1024 || history_len < 1 || history_len > 4096)
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_update_scale: bad n_states / history_len");
    if (algo != FP8SQ_AMAX_MAX && algo != FP8SQ_AMAX_MOST_RECENT)
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_update_scale: bad algo");
    for (int i = 0; i < n_states; ++i)
        if (!valid_format(formats[i])) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_update_scale: bad format of state %d", i);
    if (!aligned4(states)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_update_scale: states must be 4-byte aligned");
    int sms, r;
    if ((r = check_device(&sms))) return r;
    return cuda_status(
        fp8sq::launch_update_scale(states, n_states, history_len, formats, algo, static_cast<cudaStream_t>(stream)),
        "fp8_update_scale launch");
}

static int validate_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int format, int gran,
                             const float* state, int H, const uint8_t* q, const uint8_t* qT, const void* scales,
                             const float* amax_out)
{
    if ((!x || (!q && !column_gran(gran))) && rows * cols != 0) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize: null x or q");
    if (!valid_dtype(x_dtype) || !valid_format(format) || !valid_gran(gran))
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize: bad dtype, format or granularity");
    if (rows < 0 || cols < 0) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize: negative size");
    if (rows >= kMaxDim || cols >= kMaxDim) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_quantize: dimension too large");
    if (!aligned16(x) || (q && !aligned16(q)) || (qT && !aligned16(qT)))
        return fail(FP8SQ_ERR_MISALIGNED, "fp8_quantize: x, q, qT must be 16-byte aligned");
    if ((scales && !aligned4(scales)) || (amax_out && !aligned4(amax_out)) || (state && !aligned4(state)))
        return fail(FP8SQ_ERR_MISALIGNED, "fp8_quantize: scale / amax / state buffers must be 4-byte aligned");
    int r = check_units(gran, rows, cols);
    if (r) return r;
    if (gran == FP8SQ_TENSOR) {
        if (state && (H < 1 || H > 4096)) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize: bad history_len");
        if (!state && (!amax_out || !scales))
            return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize: current per-tensor scaling needs amax_out and scales_out");
        if (qT && (rows % 16 || cols % 16))
            return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_quantize: a transposed copy needs rows, cols %% 16 == 0");
    } else {
        if (state) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_quantize: delayed scaling is per tensor only");
        if (qT && !(gran == FP8SQ_BLOCK_128x128 || column_gran(gran)))
            return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_quantize: a transposed copy needs TENSOR, BLOCK_128x128 or a column granularity");
        if (!scales) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize: scales_out is required for this granularity");
        if (e8m0_tiled(gran) && !aligned16(scales))
            return fail(FP8SQ_ERR_MISALIGNED, "fp8_quantize: tiled E8M0 scales must be 16-byte aligned");
        if (column_gran(gran)) {
            if (!qT && rows * cols != 0) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize: column granularities need qT");
            if (x_dtype != FP8SQ_BF16) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_quantize: column granularities need bf16 input");
            if (amax_out) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_quantize: no amax output for column granularities");
            if (!aligned16(scales)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_quantize: column-unit scales must be 16-byte aligned");
        }
    }
    return FP8SQ_OK;
}

FP8SQ_API int fp8_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int format, int gran,
                           float* delayed_state, int history_len, uint8_t* q, uint8_t* qT, void* scales_out,
                           float* amax_out, unsigned long long* sat_count, void* stream)
{
    int r = validate_quantize(x, x_dtype, rows, cols, format, gran, delayed_state, history_len, q, qT, scales_out,
                              amax_out);
    if (r) return r;
    if (sat_count && (reinterpret_cast<uintptr_t>(sat_count) & 7u))
        return fail(FP8SQ_ERR_MISALIGNED, "fp8_quantize: sat_count must be 8-byte aligned");
    int sms;
    if ((r = check_device(&sms))) return r;
    fp8sq::QuantArgs a;
    a.x = x;
    a.x_dtype = x_dtype;
    a.rows = rows;
    a.cols = cols;
    a.format = format;
    a.gran = gran;
    a.state = delayed_state;
    a.history_len = history_len;
    a.q = q;
    a.qT = qT;
    a.scales = scales_out;
    a.amax = amax_out;
    a.sat = sat_count;
    return cuda_status(fp8sq::launch_quantize(a, static_cast<cudaStream_t>(stream), sms), "fp8_quantize launch");
}

FP8SQ_API int fp8_quantize_rows_cols(const void* x, int64_t rows, int64_t cols, int format, int unit,
                                     uint8_t* q, void* row_scales, uint8_t* qT, void* col_scales,
                                     unsigned long long* sat_count, void* stream)
{
    if ((!x || !q || !qT || !row_scales || !col_scales) && rows * cols != 0)
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize_rows_cols: null pointer");
    if (!valid_format(format)) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize_rows_cols: bad format");
    if (unit != FP8SQ_TILE_1x128 && unit != FP8SQ_MX32_TILED && unit != FP8SQ_TILE_1x128_POW2)
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize_rows_cols: unit must be TILE_1x128, TILE_1x128_POW2 or MX32_TILED");
    if (rows < 0 || cols < 0) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_quantize_rows_cols: negative size");
    if (rows >= kMaxDim || cols >= kMaxDim) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_quantize_rows_cols: dimension too large");
    if (rows % 128 || cols % 128)
        return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_quantize_rows_cols: rows, cols %% 128 == 0 (%lld x %lld)",
                    (long long)rows, (long long)cols);
    if (!aligned16(x) || !aligned16(q) || !aligned16(qT))
        return fail(FP8SQ_ERR_MISALIGNED, "fp8_quantize_rows_cols: x, q, qT must be 16-byte aligned");
    const bool e8m0 = unit == FP8SQ_MX32_TILED || unit == FP8SQ_TILE_1x128_POW2;
    if (e8m0 ? (!aligned16(row_scales) || !aligned16(col_scales)) : (!aligned4(row_scales) || !aligned4(col_scales)))
        return fail(FP8SQ_ERR_MISALIGNED, "fp8_quantize_rows_cols: scales misaligned");
    if (sat_count && (reinterpret_cast<uintptr_t>(sat_count) & 7u))
        return fail(FP8SQ_ERR_MISALIGNED, "fp8_quantize_rows_cols: sat_count must be 8-byte aligned");
    int sms, r;
    if ((r = check_device(&sms))) return r;
    if (rows * cols == 0) return FP8SQ_OK;
    fp8sq::QuantArgs a;
    a.x = x; a.x_dtype = fp8sq::kBF16; a.rows = rows; a.cols = cols; a.format = format;
    a.gran = unit == FP8SQ_MX32_TILED ? fp8sq::kMXRowCol
             : unit == FP8SQ_TILE_1x128_POW2 ? fp8sq::kTileRowColPow2 : fp8sq::kTileRowCol;
    a.q = q; a.qT = qT; a.scales = row_scales; a.col_scales = col_scales; a.sat = sat_count;
    return cuda_status(fp8sq::launch_quantize(a, static_cast<cudaStream_t>(stream), sms),
                       "fp8_quantize_rows_cols launch");
}

static int validate_gemm(const uint8_t* A, int a_format, const void* a_scale, int a_gran, const uint8_t* B,
                         int b_format, const void* b_scale, int b_gran, int64_t M, int64_t N, int64_t K,
                         const float* bias, const void* D, int d_dtype, int* mode)
{
    // empty operands may come with null pointers (nothing of them is read)
    if ((!A && M * K != 0) || (!B && N * K != 0) || (!D && M * N != 0) ||
        ((!a_scale || !b_scale) && M * N * K != 0))
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_gemm: null pointer");
    if (!valid_format(a_format) || !valid_format(b_format) || !valid_dtype(d_dtype))
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_gemm: bad format or output dtype");
    if (M < 0 || N < 0 || K < 0) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_gemm: negative size");
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm: dimension too large");
    if (!aligned16(A) || !aligned16(B) || !aligned16(D))
        return fail(FP8SQ_ERR_MISALIGNED, "fp8_gemm: A, B, D must be 16-byte aligned");
    if (!aligned4(a_scale) || !aligned4(b_scale) || (bias && !aligned4(bias)))
        return fail(FP8SQ_ERR_MISALIGNED, "fp8_gemm: scales / bias must be 4-byte aligned");
    if (N % 8) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm: N %% 8 != 0");
    if (a_gran == FP8SQ_TENSOR && b_gran == FP8SQ_TENSOR) {
        if (K % 16) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm: K %% 16 != 0");
        *mode = 0;
    } else if (a_gran == FP8SQ_TILE_1x128 && b_gran == FP8SQ_BLOCK_128x128) {
        if (K % 128) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm: 1x128 x 128x128 scaling needs K %% 128 == 0");
        *mode = 1;
    } else if (a_gran == FP8SQ_TILE_128x1 && b_gran == FP8SQ_TILE_128x1) {
        if (K % 128) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm: column-tile scaling needs K %% 128 == 0");
        if (!aligned16(a_scale) || !aligned16(b_scale))
            return fail(FP8SQ_ERR_MISALIGNED, "fp8_gemm: column-tile scales must be 16-byte aligned");
        *mode = 3;
    } else if (e8m0_tiled(a_gran) && e8m0_tiled(b_gran)) {
        if (!aligned16(a_scale) || !aligned16(b_scale))
            return fail(FP8SQ_ERR_MISALIGNED, "fp8_gemm: tiled MX scales must be 16-byte aligned");
        if (M % 128 || N % 128 || K % 128)
            return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm: MX scaling needs M, N, K %% 128 == 0");
        *mode = 2;
    } else {
        return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm: unsupported scale granularity pair (%d, %d)", a_gran, b_gran);
    }
    return FP8SQ_OK;
}

FP8SQ_API int fp8_gemm(const uint8_t* A, int a_format, const void* a_scale, int a_gran, const uint8_t* B,
                       int b_format, const void* b_scale, int b_gran, int64_t M, int64_t N, int64_t K,
                       const float* bias, void* D, int d_dtype, void* stream)
{
    int mode = 0;
    int r = validate_gemm(A, a_format, a_scale, a_gran, B, b_format, b_scale, b_gran, M, N, K, bias, D, d_dtype, &mode);
    if (r) return r;
    int sms;
    if ((r = check_device(&sms))) return r;
    fp8sq::GemmArgs g;
    g.A = A;
    g.B = B;
    g.a_format = a_format;
    g.b_format = b_format;
    g.mode = mode;
    g.a_scale = a_scale;
    g.b_scale = b_scale;
    g.M = M;
    g.N = N;
    g.K = K;
    g.bias = bias;
    g.D = D;
    g.d_dtype = d_dtype;
    const char* why = nullptr;
    cudaError_t e = fp8sq::launch_gemm(g, static_cast<cudaStream_t>(stream), sms, &why);
    if (e == cudaErrorNotSupported) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm: %s", why ? why : "not supported");
    if (e != cudaSuccess && why) {
        cudaGetLastError();
        return fail(FP8SQ_ERR_CUDA, "fp8_gemm: %s", why);
    }
    return cuda_status(e, "fp8_gemm launch");
}

FP8SQ_API int fp8_gemm_layout(const uint8_t* A, int a_format, const void* a_scale, int a_major, const uint8_t* B,
                              int b_format, const void* b_scale, int b_major, int64_t M, int64_t N, int64_t K,
                              const float* bias, void* D, int d_dtype, void* stream)
{
    if ((a_major != FP8SQ_K_MAJOR && a_major != FP8SQ_MN_MAJOR) || (b_major != FP8SQ_K_MAJOR && b_major != FP8SQ_MN_MAJOR))
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_gemm_layout: a_major / b_major must be K_MAJOR or MN_MAJOR");
    int mode = 0;
    int r = validate_gemm(A, a_format, a_scale, FP8SQ_TENSOR, B, b_format, b_scale, FP8SQ_TENSOR, M, N, K, bias, D,
                          d_dtype, &mode);
    if (r) return r;
    if (a_major == FP8SQ_MN_MAJOR && M % 16)
        return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm_layout: an MN-major A needs M %% 16 == 0");
    if (b_major == FP8SQ_MN_MAJOR && N % 16)
        return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm_layout: an MN-major B needs N %% 16 == 0");
    int sms;
    if ((r = check_device(&sms))) return r;
    fp8sq::GemmArgs g;
    g.A = A; g.B = B; g.a_format = a_format; g.b_format = b_format; g.mode = 0;
    g.a_scale = a_scale; g.b_scale = b_scale; g.M = M; g.N = N; g.K = K;
    g.bias = bias; g.D = D; g.d_dtype = d_dtype;
    g.a_mn = a_major == FP8SQ_MN_MAJOR;
    g.b_mn = b_major == FP8SQ_MN_MAJOR;
    const char* why = nullptr;
    cudaError_t e = fp8sq::launch_gemm(g, static_cast<cudaStream_t>(stream), sms, &why);
    if (e == cudaErrorNotSupported) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm_layout: %s", why ? why : "not supported");
    if (e != cudaSuccess && why) {
        cudaGetLastError();
        return fail(FP8SQ_ERR_CUDA, "fp8_gemm_layout: %s", why);
    }
    return cuda_status(e, "fp8_gemm_layout launch");
}

FP8SQ_API int fp8_gemm_cast(const uint8_t* A, int a_format, const void* a_scale, int a_major, const uint8_t* B,
                            int b_format, const void* b_scale, int b_major, int64_t M, int64_t N, int64_t K,
                            const float* bias, void* D, uint8_t* q_out, int q_format, float* q_state,
                            int q_history_len, void* stream)
{
    if ((a_major != FP8SQ_K_MAJOR && a_major != FP8SQ_MN_MAJOR) || (b_major != FP8SQ_K_MAJOR && b_major != FP8SQ_MN_MAJOR))
        return fail(FP8SQ_ERR_INVALID_ARG, "fp8_gemm_cast: a_major / b_major must be K_MAJOR or MN_MAJOR");
    if (!valid_format(q_format)) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_gemm_cast: bad q_format");
    if ((!q_out && M * N != 0) || !q_state) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_gemm_cast: null q_out or q_state");
    if (q_history_len < 1 || q_history_len > 4096) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_gemm_cast: bad q_history_len");
    int mode = 0;
    int r = validate_gemm(A, a_format, a_scale, FP8SQ_TENSOR, B, b_format, b_scale, FP8SQ_TENSOR, M, N, K, bias, D,
                          FP8SQ_BF16, &mode);
    if (r) return r;
    if (K == 0) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm_cast: K == 0");
    if (N % 16) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm_cast: N %% 16 != 0");
    if (a_major == FP8SQ_MN_MAJOR && M % 16)
        return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm_cast: an MN-major A needs M %% 16 == 0");
    if (b_major == FP8SQ_MN_MAJOR && N % 16)
        return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm_cast: an MN-major B needs N %% 16 == 0");
    if (!aligned16(q_out)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_gemm_cast: q_out must be 16-byte aligned");
    if (!aligned4(q_state)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_gemm_cast: q_state must be 4-byte aligned");
    int sms;
    if ((r = check_device(&sms))) return r;
    fp8sq::GemmArgs g;
    g.A = A; g.B = B; g.a_format = a_format; g.b_format = b_format; g.mode = 0;
    g.a_scale = a_scale; g.b_scale = b_scale; g.M = M; g.N = N; g.K = K;
    g.bias = bias; g.D = D; g.d_dtype = fp8sq::kBF16;
    g.a_mn = a_major == FP8SQ_MN_MAJOR;
    g.b_mn = b_major == FP8SQ_MN_MAJOR;
    g.q_out = q_out; g.q_state = q_state; g.q_history_len = q_history_len; g.q_format = q_format;
    const char* why = nullptr;
    cudaError_t e = fp8sq::launch_gemm(g, static_cast<cudaStream_t>(stream), sms, &why);
    if (e == cudaErrorNotSupported) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_gemm_cast: %s", why ? why : "not supported");
    if (e != cudaSuccess && why) {
        cudaGetLastError();
        return fail(FP8SQ_ERR_CUDA, "fp8_gemm_cast: %s", why);
    }
    return cuda_status(e, "fp8_gemm_cast launch");
}

FP8SQ_API size_t fp8_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int gran)
{
    if (M < 0 || N < 0 || K < 0 ||
        !(gran == FP8SQ_TENSOR || gran == FP8SQ_TILE_1x128 || gran == FP8SQ_MX32 || gran == FP8SQ_TILE_1x128_POW2))
        return 0;
    return ws_layout(M, N, K, gran).total;
}

static int check_linear_shape(int64_t M, int64_t N, int64_t K, int gran, const void* ws, size_t ws_bytes)
{
    if (M < 0 || N < 0 || K < 0) return fail(FP8SQ_ERR_INVALID_ARG, "linear: negative size");
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return fail(FP8SQ_ERR_UNSUPPORTED, "linear: dimension too large");
    if (gran == FP8SQ_TENSOR) {
        if (M % 16 || N % 16 || K % 16) return fail(FP8SQ_ERR_UNSUPPORTED, "linear: per-tensor needs M, N, K %% 16 == 0");
    } else if (gran == FP8SQ_TILE_1x128 || gran == FP8SQ_MX32 || gran == FP8SQ_TILE_1x128_POW2) {
        if (M % 128 || N % 128 || K % 128) return fail(FP8SQ_ERR_UNSUPPORTED, "linear: block scaling needs M, N, K %% 128 == 0");
    } else {
        return fail(FP8SQ_ERR_INVALID_ARG, "linear: granularity must be TENSOR, TILE_1x128, TILE_1x128_POW2 or MX32");
    }
    if (!ws) return fail(FP8SQ_ERR_INVALID_ARG, "linear: null workspace");
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(FP8SQ_ERR_MISALIGNED, "linear: workspace must be 256-byte aligned");
    if (ws_bytes < ws_layout(M, N, K, gran).total) return fail(FP8SQ_ERR_INVALID_ARG, "linear: workspace too small");
    return FP8SQ_OK;
}

FP8SQ_API int fp8_linear_fwd(const void* x, const void* w, int64_t M, int64_t N, int64_t K, int gran, int recipe,
                             float* x_state, float* w_state, int history_len, void* workspace, size_t ws_bytes,
                             const float* bias, void* y, int y_dtype, void* stream)
{
    if (!x || !w || !y) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_fwd: null pointer");
    if (recipe != FP8SQ_RECIPE_HYBRID && recipe != FP8SQ_RECIPE_E4M3) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_fwd: bad recipe");
    if (!valid_dtype(y_dtype)) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_fwd: bad y dtype");
    int r = check_linear_shape(M, N, K, gran, workspace, ws_bytes);
    if (r) return r;
    const bool delayed = x_state || w_state;
    if (delayed && (!x_state || !w_state)) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_fwd: give both x_state and w_state, or neither");
    if (delayed && gran != FP8SQ_TENSOR) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_linear_fwd: delayed scaling is per tensor only");
    if (delayed && (history_len < 1 || history_len > 4096)) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_fwd: bad history_len");
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_linear_fwd: x, w, y must be 16-byte aligned");
    if ((bias && !aligned4(bias)) || (x_state && !aligned4(x_state)) || (w_state && !aligned4(w_state)))
        return fail(FP8SQ_ERR_MISALIGNED, "fp8_linear_fwd: bias / states must be 4-byte aligned");
    int sms;
    if ((r = check_device(&sms))) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const WsLayout L = ws_layout(M, N, K, gran);
    const int H = history_len;

    fp8sq::QuantArgs qa;
    qa.x_dtype = fp8sq::kBF16;
    qa.format = fp8sq::kE4M3;
    fp8sq::GemmArgs g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.bias = bias;
    g.D = y;
    g.d_dtype = y_dtype;
    g.A = ws + L.qx;
    g.B = ws + L.qw;
    if (gran == FP8SQ_TENSOR) {
        float* scal = reinterpret_cast<float*>(ws + L.scal);   // sx, sw, sdy, ax, aw, ady
        // x and W in one launch (current scaling: one more for both amaxes);
        // no transposed copies, the backward reads these codes MN-major
        qa.x = x; qa.rows = M; qa.cols = K; qa.gran = fp8sq::kTensor;
        qa.q = ws + L.qx; qa.qT = nullptr;
        qa.state = x_state; qa.history_len = H;
        qa.scales = &scal[0]; qa.amax = delayed ? nullptr : &scal[3];
        fp8sq::QuantArgs qw = qa;
        qw.x = w; qw.rows = N; qw.cols = K;
        qw.q = ws + L.qw; qw.qT = nullptr;
        qw.state = w_state;
        qw.scales = &scal[1]; qw.amax = delayed ? nullptr : &scal[4];
        if ((r = cuda_status(fp8sq::launch_quantize_pair(qa, qw, st, sms), "fp8_linear_fwd: quantize x and w"))) return r;
        // (delayed: each cast writes the dequantisation scale it used into
        // scal[], kept for the backward pass)
        g.mode = 0;
        g.a_scale = &scal[0];
        g.b_scale = &scal[1];
        g.a_format = g.b_format = fp8sq::kE4M3;
    } else if (gran == FP8SQ_TILE_1x128) {
        // x: 1x128 tiles along K (forward) and 128x1 column tiles along M
        // (wgrad), both from one read of x
        qa.x = x; qa.rows = M; qa.cols = K; qa.gran = fp8sq::kTileRowCol;
        qa.q = ws + L.qx; qa.scales = ws + L.sx; qa.qT = ws + L.qxT; qa.col_scales = ws + L.sxT;
        if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_linear_fwd: quantize x"))) return r;
        qa.col_scales = nullptr;
        // W: 128x128 blocks, with the transposed codes and scale grid (dgrad)
        qa.x = w; qa.rows = N; qa.cols = K; qa.gran = fp8sq::kBlock;
        qa.q = ws + L.qw; qa.qT = ws + L.qwT; qa.scales = ws + L.sw;
        qa.scalesT = reinterpret_cast<float*>(ws + L.swT);
        if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_linear_fwd: quantize w"))) return r;
        g.mode = 1;
        g.a_scale = ws + L.sx;
        g.b_scale = ws + L.sw;
    } else if (gran == FP8SQ_TILE_1x128_POW2) {
        // the same units with power-of-two scales, as tiled E8M0 codes: the
        // GEMMs run on the block-scaled MMA with no promotion.  x: 1x128
        // tiles (forward) and 128x1 column tiles (wgrad) from one read.
        qa.x = x; qa.rows = M; qa.cols = K; qa.gran = fp8sq::kTileRowColPow2;
        qa.q = ws + L.qx; qa.scales = ws + L.sx; qa.qT = ws + L.qxT; qa.col_scales = ws + L.sxT;
        if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_linear_fwd: quantize x"))) return r;
        qa.col_scales = nullptr;
        // W: 128x128 blocks, with the transposed codes and W^T's codes (dgrad)
        qa.x = w; qa.rows = N; qa.cols = K; qa.gran = fp8sq::kBlockPow2;
        qa.q = ws + L.qw; qa.qT = ws + L.qwT; qa.scales = ws + L.sw;
        qa.scalesT = reinterpret_cast<float*>(ws + L.swT);
        if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_linear_fwd: quantize w"))) return r;
        g.mode = 2;
        g.a_scale = ws + L.sx;
        g.b_scale = ws + L.sw;
    } else {
        // x and W: MX-32 blocks along K (forward) and along their rows
        // (backward), each from one read of the operand
        qa.x = x; qa.rows = M; qa.cols = K; qa.gran = fp8sq::kMXRowCol;
        qa.q = ws + L.qx; qa.scales = ws + L.sx; qa.qT = ws + L.qxT; qa.col_scales = ws + L.sxT;
        if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_linear_fwd: quantize x"))) return r;
        qa.x = w; qa.rows = N; qa.cols = K;
        qa.q = ws + L.qw; qa.scales = ws + L.sw; qa.qT = ws + L.qwT; qa.col_scales = ws + L.swT;
        if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_linear_fwd: quantize w"))) return r;
        g.mode = 2;
        g.a_scale = ws + L.sx;
        g.b_scale = ws + L.sw;
    }
    const char* why = nullptr;
    cudaError_t e = fp8sq::launch_gemm(g, st, sms, &why);
    if (e == cudaErrorNotSupported) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_linear_fwd: %s", why ? why : "GEMM not supported");
    return cuda_status(e, why ? why : "fp8_linear_fwd: GEMM launch");
}

FP8SQ_API int fp8_linear_bwd(const void* dy, int64_t M, int64_t N, int64_t K, int gran, int recipe,
                             float* dy_state, int history_len, void* workspace, size_t ws_bytes, void* dx, float* dw,
                             void* stream)
{
    if (!dy || !dx || !dw) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_bwd: null pointer");
    if (recipe != FP8SQ_RECIPE_HYBRID && recipe != FP8SQ_RECIPE_E4M3) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_bwd: bad recipe");
    int r = check_linear_shape(M, N, K, gran, workspace, ws_bytes);
    if (r) return r;
    if (dy_state && gran != FP8SQ_TENSOR) return fail(FP8SQ_ERR_UNSUPPORTED, "fp8_linear_bwd: delayed scaling is per tensor only");
    if (dy_state && (history_len < 1 || history_len > 4096)) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_bwd: bad history_len");
    if (!aligned16(dy) || !aligned16(dx) || !aligned16(dw)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_linear_bwd: dy, dx, dw must be 16-byte aligned");
    if (dy_state && !aligned4(dy_state)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_linear_bwd: dy_state must be 4-byte aligned");
    int sms;
    if ((r = check_device(&sms))) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const WsLayout L = ws_layout(M, N, K, gran);
    const int fdy = recipe == FP8SQ_RECIPE_HYBRID ? fp8sq::kE5M2 : fp8sq::kE4M3;
    const char* why = nullptr;

    fp8sq::QuantArgs qa;
    qa.x = dy; qa.x_dtype = fp8sq::kBF16; qa.rows = M; qa.cols = N;
    qa.format = fdy;
    fp8sq::GemmArgs dg, wg;                 // dgrad dx[M][K] = dy W; wgrad dw[N][K] = dy^T x
    dg.M = M; dg.N = K; dg.K = N; dg.D = dx; dg.d_dtype = fp8sq::kBF16;
    dg.A = ws + L.qdy; dg.a_format = fdy; dg.B = ws + L.qwT; dg.b_format = fp8sq::kE4M3;
    wg.M = N; wg.N = K; wg.K = M; wg.D = dw; wg.d_dtype = fp8sq::kF32;
    wg.A = ws + L.qdyT; wg.a_format = fdy; wg.B = ws + L.qxT; wg.b_format = fp8sq::kE4M3;
    if (gran == FP8SQ_TENSOR) {
        float* scal = reinterpret_cast<float*>(ws + L.scal);
        qa.gran = fp8sq::kTensor;
        qa.q = ws + L.qdy; qa.qT = nullptr;
        qa.state = dy_state; qa.history_len = history_len;
        qa.scales = &scal[2]; qa.amax = dy_state ? nullptr : &scal[5];
        if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_linear_bwd: quantize dy"))) return r;
        dg.mode = wg.mode = 0;
        dg.a_scale = &scal[2]; dg.b_scale = &scal[1];
        wg.a_scale = &scal[2]; wg.b_scale = &scal[0];
        // the forward's codes as they are: dgrad's B = W [N][K] and wgrad's
        // A = dy [M][N], B = x [M][K] are MN-major operands
        dg.B = ws + L.qw; dg.b_mn = true;
        wg.A = ws + L.qdy; wg.a_mn = true;
        wg.B = ws + L.qx; wg.b_mn = true;
    } else if (gran == FP8SQ_TILE_1x128) {
        // dy: 1x128 tiles along N (dgrad) and 128x1 column tiles along M
        // (wgrad), both from one read of dy
        qa.gran = fp8sq::kTileRowCol;
        qa.q = ws + L.qdy; qa.scales = ws + L.sdy; qa.qT = ws + L.qdyT; qa.col_scales = ws + L.sdyT;
        if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_linear_bwd: quantize dy"))) return r;
        dg.mode = 1; dg.a_scale = ws + L.sdy; dg.b_scale = ws + L.swT;
        wg.mode = 3; wg.a_scale = ws + L.sdyT; wg.b_scale = ws + L.sxT;
    } else if (gran == FP8SQ_TILE_1x128_POW2) {
        // dy: power-of-two 1x128 tiles along N (dgrad) and 128x1 column tiles
        // along M (wgrad), from one read; both GEMMs on the block-scaled MMA
        qa.gran = fp8sq::kTileRowColPow2;
        qa.q = ws + L.qdy; qa.scales = ws + L.sdy; qa.qT = ws + L.qdyT; qa.col_scales = ws + L.sdyT;
        if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_linear_bwd: quantize dy"))) return r;
        dg.mode = wg.mode = 2;
        dg.a_scale = ws + L.sdy; dg.b_scale = ws + L.swT;
        wg.a_scale = ws + L.sdyT; wg.b_scale = ws + L.sxT;
    } else {
        // dy: MX-32 blocks along N (dgrad) and along M (wgrad), from one read
        qa.gran = fp8sq::kMXRowCol;
        qa.q = ws + L.qdy; qa.scales = ws + L.sdy; qa.qT = ws + L.qdyT; qa.col_scales = ws + L.sdyT;
        if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_linear_bwd: quantize dy"))) return r;
        dg.mode = wg.mode = 2;
        dg.a_scale = ws + L.sdy; dg.b_scale = ws + L.swT;
        wg.a_scale = ws + L.sdyT; wg.b_scale = ws + L.sxT;
    }
    // dgrad and wgrad are independent: wgrad runs on a side stream forked
    // from `st` and joined back into it.  When both persistent grids fit on
    // the device at once (small layers) the two share it; when each fills the
    // device, wgrad's CTAs take the SMs that dgrad's last, partial wave of
    // tiles leaves idle (FFN layers at 16384 tokens: 1.4 % off the step).
    const int cd = fp8sq::gemm_ctas(dg, sms), cw = fp8sq::gemm_ctas(wg, sms);
    SideStream* side = nullptr;
    if (cd > 0 && cw > 0 && (r = side_stream(st, &side))) return r;
    if (side) {
        if ((r = cuda_status(cudaEventRecord(side->fork, st), "fp8_linear_bwd: fork"))) return r;
        if ((r = cuda_status(cudaStreamWaitEvent(side->s, side->fork, 0), "fp8_linear_bwd: fork"))) return r;
        if ((r = cuda_status(fp8sq::launch_gemm(dg, st, sms, &why), why ? why : "fp8_linear_bwd: dgrad"))) return r;
        if ((r = cuda_status(fp8sq::launch_gemm(wg, side->s, sms, &why), why ? why : "fp8_linear_bwd: wgrad"))) return r;
        if ((r = cuda_status(cudaEventRecord(side->join, side->s), "fp8_linear_bwd: join"))) return r;
        return cuda_status(cudaStreamWaitEvent(st, side->join, 0), "fp8_linear_bwd: join");
    }
    if ((r = cuda_status(fp8sq::launch_gemm(dg, st, sms, &why), why ? why : "fp8_linear_bwd: dgrad"))) return r;
    return cuda_status(fp8sq::launch_gemm(wg, st, sms, &why), why ? why : "fp8_linear_bwd: wgrad");
}

static int validate_ln(const void* x, const float* gamma, const float* beta, int64_t M, int64_t K, int format,
                       const float* state, int H, const uint8_t* q, const uint8_t* qT, const float* mu,
                       const float* rstd)
{
    if (!x || !gamma || !q || !state || !mu || !rstd) return fail(FP8SQ_ERR_INVALID_ARG, "layernorm: null pointer");
    if (!valid_format(format)) return fail(FP8SQ_ERR_INVALID_ARG, "layernorm: bad format");
    if (M < 0 || K < 0) return fail(FP8SQ_ERR_INVALID_ARG, "layernorm: negative size");
    if (M >= kMaxDim || K >= kMaxDim) return fail(FP8SQ_ERR_UNSUPPORTED, "layernorm: dimension too large");
    if (M % 16 || K % 16) return fail(FP8SQ_ERR_UNSUPPORTED, "layernorm: needs M, K %% 16 == 0");
    if (H < 1 || H > 4096) return fail(FP8SQ_ERR_INVALID_ARG, "layernorm: bad history_len");
    if (!aligned16(x) || !aligned16(q) || (qT && !aligned16(qT)))
        return fail(FP8SQ_ERR_MISALIGNED, "layernorm: x, q, qT must be 16-byte aligned");
    if (!aligned16(gamma) || (beta && !aligned16(beta)) || !aligned16(mu) || !aligned16(rstd))
        return fail(FP8SQ_ERR_MISALIGNED, "layernorm: gamma, beta, mu, rstd must be 16-byte aligned");
    if (!aligned4(state)) return fail(FP8SQ_ERR_MISALIGNED, "layernorm: state must be 4-byte aligned");
    return FP8SQ_OK;
}

FP8SQ_API int fp8_layernorm_quantize(const void* x, const float* gamma, const float* beta, float eps, int64_t M,
                                     int64_t K, int format, float* delayed_state, int history_len, uint8_t* q,
                                     uint8_t* qT, float* mu_out, float* rstd_out, void* stream)
{
    int r = validate_ln(x, gamma, beta, M, K, format, delayed_state, history_len, q, qT, mu_out, rstd_out);
    if (r) return r;
    int sms;
    if ((r = check_device(&sms))) return r;
    fp8sq::QuantArgs qa;
    qa.x = x; qa.x_dtype = fp8sq::kBF16; qa.rows = M; qa.cols = K; qa.format = format;
    qa.gran = fp8sq::kTensor; qa.state = delayed_state; qa.history_len = history_len; qa.q = q; qa.qT = qT;
    return cuda_status(fp8sq::launch_layernorm_quantize(qa, gamma, beta, eps, mu_out, rstd_out,
                                                        static_cast<cudaStream_t>(stream), sms),
                       "fp8_layernorm_quantize launch");
}

FP8SQ_API int fp8_layernorm_linear_fwd(const void* x, const float* gamma, const float* beta, float eps, const void* w,
                                       int64_t M, int64_t N, int64_t K, float* x_state, float* w_state,
                                       int history_len, void* workspace, size_t ws_bytes, float* mu_out,
                                       float* rstd_out, const float* bias, void* y, int y_dtype, void* stream)
{
    if (!w || !y || !w_state) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_layernorm_linear_fwd: null pointer");
    if (!valid_dtype(y_dtype)) return fail(FP8SQ_ERR_INVALID_ARG, "fp8_layernorm_linear_fwd: bad y dtype");
    int r = check_linear_shape(M, N, K, FP8SQ_TENSOR, workspace, ws_bytes);
    if (r) return r;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const WsLayout L = ws_layout(M, N, K, FP8SQ_TENSOR);
    r = validate_ln(x, gamma, beta, M, K, FP8SQ_E4M3, x_state, history_len, ws + L.qx, nullptr, mu_out, rstd_out);
    if (r) return r;
    if (!aligned16(w) || !aligned16(y)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_layernorm_linear_fwd: w, y must be 16-byte aligned");
    if ((bias && !aligned4(bias)) || !aligned4(w_state)) return fail(FP8SQ_ERR_MISALIGNED, "fp8_layernorm_linear_fwd: bias / w_state alignment");
    int sms;
    if ((r = check_device(&sms))) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int H = history_len;
    float* scal = reinterpret_cast<float*>(ws + L.scal);
    fp8sq::QuantArgs qa;
    qa.x = x; qa.x_dtype = fp8sq::kBF16; qa.rows = M; qa.cols = K; qa.format = fp8sq::kE4M3;
    qa.gran = fp8sq::kTensor; qa.state = x_state; qa.history_len = H; qa.q = ws + L.qx; qa.qT = nullptr;
    qa.scales = &scal[0];       // receives the dequantisation scale the cast used
    if ((r = cuda_status(fp8sq::launch_layernorm_quantize(qa, gamma, beta, eps, mu_out, rstd_out, st, sms),
                         "fp8_layernorm_linear_fwd: layernorm cast")))
        return r;
    qa.x = w; qa.rows = N; qa.cols = K; qa.state = w_state; qa.q = ws + L.qw; qa.qT = nullptr;
    qa.scales = &scal[1];
    if ((r = cuda_status(fp8sq::launch_quantize(qa, st, sms), "fp8_layernorm_linear_fwd: quantize w"))) return r;
    fp8sq::GemmArgs g;
    g.mode = 0; g.M = M; g.N = N; g.K = K; g.bias = bias; g.D = y; g.d_dtype = y_dtype;
    g.A = ws + L.qx; g.B = ws + L.qw; g.a_scale = &scal[0]; g.b_scale = &scal[1];
    g.a_format = g.b_format = fp8sq::kE4M3;
    const char* why = nullptr;
    return cuda_status(fp8sq::launch_gemm(g, st, sms, &why), why ? why : "fp8_layernorm_linear_fwd: GEMM");
}

}  // extern "C"

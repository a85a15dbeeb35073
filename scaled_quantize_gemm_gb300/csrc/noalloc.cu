// noalloc.cu -- fp8_linear_fwd_noalloc: the forward FP8 linear with current
// per-tensor scaling, for callers that cannot allocate device memory.  Its
// scratch (the codes of x and W and four fp32 scalars) lives in a file-scope
// device array instead of a caller-provided workspace.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "../../include/fp8sq.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = FP8SQ_NOALLOC_SCRATCH_BYTES;
constexpr int64_t kMaxDim = (int64_t)1 << 31;

// Held by every GPU that loads this library, until the process exits.  In
// host code `g_noalloc_scratch` only names the symbol; its device address
// comes from cudaGetSymbolAddress, taken once per device.
__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[64] = {};

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

// Device address of the scratch on the current device (first call: set-up).
int scratch_on_current_device(uint8_t** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fp8sq::api_fail(FP8SQ_ERR_CUDA, "fp8_linear_fwd_noalloc: no usable CUDA device");
    }
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return fp8sq::api_fail(FP8SQ_ERR_CUDA, "fp8_linear_fwd_noalloc: cudaGetSymbolAddress failed: %s",
                                   cudaGetErrorString(e));
        }
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
    return FP8SQ_OK;
}

}  // namespace

extern "C" FP8SQ_API int fp8_linear_fwd_noalloc(const void* x, const void* w, int64_t M, int64_t N, int64_t K,
                                                const float* bias, void* y, int y_dtype, void* stream)
{
    using fp8sq::api_fail;
    if (M < 0 || N < 0 || K < 0) return api_fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_fwd_noalloc: negative size");
    // bound each dimension before any product is formed (GEMM / TMA coordinates are 32-bit)
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim)
        return api_fail(FP8SQ_ERR_UNSUPPORTED, "fp8_linear_fwd_noalloc: dimension too large");
    if ((!x && M * K) || (!w && N * K) || (!y && M * N))
        return api_fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_fwd_noalloc: null pointer");
    if (y_dtype != FP8SQ_BF16 && y_dtype != FP8SQ_F32)
        return api_fail(FP8SQ_ERR_INVALID_ARG, "fp8_linear_fwd_noalloc: bad y dtype");
    if (N % 8 || K % 16) return api_fail(FP8SQ_ERR_UNSUPPORTED, "fp8_linear_fwd_noalloc: needs N %% 8 == 0 and K %% 16 == 0");
    const size_t need = round256((size_t)(M * K)) + round256((size_t)(N * K)) + 256;
    if (M * K > (int64_t)kScratchBytes || N * K > (int64_t)kScratchBytes || need > kScratchBytes)
        return api_fail(FP8SQ_ERR_UNSUPPORTED,
                        "fp8_linear_fwd_noalloc: needs %zu bytes of scratch for M=%lld N=%lld K=%lld, "
                        "the static scratch holds %zu (use fp8_linear_fwd with a workspace)",
                        need, (long long)M, (long long)N, (long long)K, kScratchBytes);
    if (((uintptr_t)x | (uintptr_t)w | (uintptr_t)y) & 15u)
        return api_fail(FP8SQ_ERR_MISALIGNED, "fp8_linear_fwd_noalloc: x, w, y must be 16-byte aligned");
    if (bias && ((uintptr_t)bias & 3u))
        return api_fail(FP8SQ_ERR_MISALIGNED, "fp8_linear_fwd_noalloc: bias must be 4-byte aligned");
    int sms, r;
    if ((r = fp8sq::api_check_device(&sms))) return r;
    uint8_t* scratch = nullptr;
    if ((r = scratch_on_current_device(&scratch))) return r;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* qx = scratch;
    uint8_t* qw = scratch + round256((size_t)(M * K));
    float* scal = reinterpret_cast<float*>(qw + round256((size_t)(N * K)));   // s_x, s_w, amax_x, amax_w

    // current per-tensor scaling: each cast zeroes its amax slot first
    fp8sq::QuantArgs qa;
    qa.x = x; qa.x_dtype = fp8sq::kBF16; qa.rows = M; qa.cols = K;
    qa.format = fp8sq::kE4M3; qa.gran = fp8sq::kTensor;
    qa.q = qx; qa.scales = &scal[0]; qa.amax = &scal[2];
    cudaError_t e = fp8sq::launch_quantize(qa, st, sms);
    if (e == cudaSuccess) {
        qa.x = w; qa.rows = N; qa.cols = K;
        qa.q = qw; qa.scales = &scal[1]; qa.amax = &scal[3];
        e = fp8sq::launch_quantize(qa, st, sms);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return api_fail(FP8SQ_ERR_CUDA, "fp8_linear_fwd_noalloc: cast launch: %s", cudaGetErrorString(e));
    }
    fp8sq::GemmArgs g;
    g.mode = 0;
    g.A = qx; g.a_format = fp8sq::kE4M3; g.a_scale = &scal[0];
    g.B = qw; g.b_format = fp8sq::kE4M3; g.b_scale = &scal[1];
    g.M = M; g.N = N; g.K = K;
    g.bias = bias; g.D = y; g.d_dtype = y_dtype;
    const char* why = nullptr;
    e = fp8sq::launch_gemm(g, st, sms, &why);
    if (e == cudaErrorNotSupported)
        return api_fail(FP8SQ_ERR_UNSUPPORTED, "fp8_linear_fwd_noalloc: %s", why ? why : "GEMM not supported");
    if (e != cudaSuccess) {
        cudaGetLastError();
        return api_fail(FP8SQ_ERR_CUDA, "fp8_linear_fwd_noalloc: GEMM launch: %s", why ? why : cudaGetErrorString(e));
    }
    return FP8SQ_OK;
}

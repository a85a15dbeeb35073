// internal.h -- host-side launcher interface between the C-ABI layer
// (api.cu) and the kernel translation units.  Not installed, not part of the ABI.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8sq {

enum { kE4M3 = 0, kE5M2 = 1 };
enum { kBF16 = 0, kF32 = 1 };
enum { kTensor = 0, kTile = 1, kBlock = 2, kMX = 3, kMXTiled = 4, kTileCol = 5, kMXCol = 6,
       kTilePow2 = 7, kBlockPow2 = 8, kMXFloor = 9,
       kTileRowCol = 10, kMXRowCol = 11,     // rows and columns in one pass (fp8_quantize_rows_cols)
       kTileRowColPow2 = 12 };               // the same for power-of-two 1x128 / 128x1 tiles, tiled E8M0 codes

struct QuantArgs {
    const void* x = nullptr;
    int x_dtype = kBF16;
    int64_t rows = 0, cols = 0;
    int format = kE4M3;
    int gran = kTensor;
    float* state = nullptr;          // delayed state block (TENSOR only) or null
    int history_len = 0;
    uint8_t* q = nullptr;            // may be null only for amax-only launches
    uint8_t* qT = nullptr;
    void* scales = nullptr;
    float* scalesT = nullptr;        // 128x128 blocks with qT: the transposed scale grid (power-of-two
                                     // blocks: the tiled E8M0 codes of x^T, as bytes)
    void* col_scales = nullptr;      // rows and columns in one pass: the column-unit scales
    float* amax = nullptr;
    unsigned long long* sat = nullptr;
    const float* amax_in = nullptr;  // current per-tensor: the amax of pass 1
};

// quantize.cu
cudaError_t launch_amax(const QuantArgs& a, cudaStream_t st, int sms);    // writes a.amax per unit
cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st, int sms);
// two per-tensor casts with transposed copies (same dtype, format and
// recipe) in one launch; other argument pairs go through launch_quantize twice
cudaError_t launch_quantize_pair(const QuantArgs& a, const QuantArgs& b, cudaStream_t st, int sms);
cudaError_t launch_scale_init(float* states, int n, int H, cudaStream_t st);
cudaError_t launch_update_scale(float* states, int n, int H, const int* formats, int algo, cudaStream_t st);
// LayerNorm of bf16 x [rows][cols] fused into the delayed per-tensor cast
// (a.state required); writes mu, rstd [rows]
cudaError_t launch_layernorm_quantize(const QuantArgs& a, const float* gamma, const float* beta, float eps,
                                      float* mu, float* rstd, cudaStream_t st, int sms);

struct GemmArgs {
    const uint8_t* A = nullptr;
    const uint8_t* B = nullptr;
    int a_format = kE4M3, b_format = kE4M3;
    int mode = 0;                    // 0 per-tensor, 1 tile x block promotion, 2 MX (tiled E8M0 scales),
                                     // 3 column tiles x column tiles (promotion, scales [K/128][rows])
    const void* a_scale = nullptr;
    const void* b_scale = nullptr;
    int64_t M = 0, N = 0, K = 0;
    const float* bias = nullptr;
    void* D = nullptr;
    int d_dtype = kBF16;
    // operand storage (mode 0 only): K-major A [M][K] / B [N][K], or
    // MN-major A [K][M] / B [K][N]
    bool a_mn = false, b_mn = false;
    // mode 0, bf16 D only: also cast D to FP8 codes q_out [M][N] with the
    // delayed per-tensor state q_state (history q_history_len)
    uint8_t* q_out = nullptr;
    float* q_state = nullptr;
    int q_history_len = 0, q_format = kE4M3;
};

// gemm.cu
cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t st, int sms, const char** why);
// Raises a kernel's dynamic shared-memory limit to `bytes`, once per device.
cudaError_t smem_attr_once(const void* kern, int bytes);
int gemm_ctas(const GemmArgs& g, int sms);   // SMs its persistent grid occupies, -1 if unknown
int read_device_error(int clear);   // 0 or the GEMM kernels' device error word
// launches a kernel whose bounded wait is made to run out (failure-path test)
cudaError_t launch_selftest_wait(uint64_t limit_ns, int* waited_out, cudaStream_t st);
// 2-D tiled TMA map, 128-byte swizzle, zero fill out of bounds; u16 selects
// 2-byte elements (else 1-byte)
bool encode_tmap_2d(CUtensorMap* m, int u16, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_inner,
                    uint32_t box_rows);

// api.cu: the calling thread's error message and the sm_103 device check
int api_fail(int code, const char* fmt, ...);
int api_check_device(int* sms);

}  // namespace fp8sq

/*
 * fp8sq.h -- C ABI of the GB300 (sm_103a) FP8 scaled-linear library.
 *
 * The path: amax -> scale (current or delayed) -> saturating round-to-
 * nearest-even cast to E4M3 / E5M2 -> FP8 GEMM with fp32 accumulation and a
 * dequantising epilogue, for the forward, dgrad and wgrad products of a
 * linear layer y = x W^T.
 *
 * Sources, cited by page title and section:
 *   [TS]  "Transformer Scaling" (lab.mindcaptain.ai, reading 06): Part 01
 *         (scale maps a tensor into FP8's range using amax; delayed vs
 *         current scaling; HYBRID = E4M3 forward, E5M2 gradients), core
 *         vocabulary (amax, delayed scaling), worked example.
 *   [W14] "Week 14. Scaling laws, precision, parallelism": absmax bullet
 *         (x ~ q * scale, scale from max|x|; per tensor / block; 1x128
 *         activation tiles and 128x128 weight blocks; MX blocks of 32), FP8
 *         bullet (E4M3 max 448, E5M2 max 57344; matmuls in FP8), accumulation
 *         precision bullet (wide accumulator, fp32 promotion at intervals).
 *   [TE]  "Accelerating Transformer Training with NVIDIA Transformer Engine":
 *         DelayedScaling(HYBRID, amax_history_len=16, amax_compute_algo=max),
 *         te.Linear, the fp8_meta scale / amax_history dump.
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers are caller-owned device memory; the
 *    library allocates nothing and keeps no state between calls except a
 *    per-device cache of the SM count and a sticky device error word.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *    only enqueues work on it and returns; the caller synchronises.
 *  - Matrices are row-major with row pitch = number of columns.
 *  - Return value: FP8SQ_OK (0) or a negative FP8SQ_ERR_* code.  Arguments
 *    are validated before anything is enqueued, so an error return means
 *    nothing was launched (except FP8SQ_ERR_CUDA from a failed launch).
 *    A pointer to an operand with zero elements may be NULL.
 *    fp8_last_error() gives a message for the calling thread's last error.
 *    Nothing aborts, traps or prints.
 *  - Only sm_103 devices are accepted (FP8SQ_ERR_WRONG_ARCH otherwise).
 */
#ifndef FP8SQ_H
#define FP8SQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FP8SQ_API __attribute__((visibility("default")))
#else
#define FP8SQ_API
#endif

/* ---- status codes ---------------------------------------------------- */
#define FP8SQ_OK 0
#define FP8SQ_ERR_INVALID_ARG -1  /* null pointer, negative size, bad enum */
#define FP8SQ_ERR_UNSUPPORTED -2  /* shape / granularity combination not supported */
#define FP8SQ_ERR_MISALIGNED -3   /* a pointer is not 16-byte aligned */
#define FP8SQ_ERR_WRONG_ARCH -4   /* current device is not sm_103 */
#define FP8SQ_ERR_CUDA -5         /* a CUDA runtime / driver call failed */
#define FP8SQ_ERR_TIMEOUT -6      /* a bounded device-side wait ran out */

/* ---- enumerations ---------------------------------------------------- */
/* [W14] FP8 bullet: E4M3 (max 448, no infinities, S.1111.111 = NaN) and
 * E5M2 (max 57344, IEEE-like with infinities). */
#define FP8SQ_E4M3 0
#define FP8SQ_E5M2 1

/* element types of inputs and outputs */
#define FP8SQ_BF16 0
#define FP8SQ_F32 1

/* scaling units ([W14] absmax bullet) */
#define FP8SQ_TENSOR 0         /* one scale per tensor                          */
#define FP8SQ_TILE_1x128 1     /* one scale per 128 consecutive values of a row */
#define FP8SQ_BLOCK_128x128 2  /* one scale per 128x128 block                   */
#define FP8SQ_MX32 3           /* one power-of-two (E8M0) scale per 32 values   */
#define FP8SQ_MX32_TILED 4     /* MX32 with the scales in the GEMM's tiled layout */
#define FP8SQ_TILE_128x1 5     /* one scale per 128 consecutive values of a column */
#define FP8SQ_MX32_COL_TILED 6 /* one E8M0 scale per 32 values of a column, tiled  */
/* recipe variants with E8M0 scales in the tiled layout (GEMM-ready):       */
#define FP8SQ_TILE_1x128_POW2 7     /* 1x128 tiles, power-of-two scale        */
#define FP8SQ_BLOCK_128x128_POW2 8  /* 128x128 blocks, power-of-two scale     */
#define FP8SQ_MX32_FLOOR_TILED 9    /* MX-32 with the OCP floor exponent rule */

/* Tiled MX scale layout (FP8SQ_MX32_TILED), for a tensor [rows][cols] with
 * rows % 128 == 0 and cols % 128 == 0: the E8M0 code of row r, 32-block
 * t = c / 32 sits at byte
 *     ((r / 128) * (cols / 128) + t / 4) * 512
 *       + (r % 32) * 16 + ((r / 32) % 4) * 4 + (t % 4),
 * i.e. 512-byte chunks of 128 rows x 4 consecutive 32-blocks (128 values
 * along K), in the order the block-scaled tensor-core MMA reads them. */

/* amax history reduction ([TE] amax_compute_algo) */
#define FP8SQ_AMAX_MAX 0
#define FP8SQ_AMAX_MOST_RECENT 1

/* recipes ([TS] Part 01 / [TE] Format.HYBRID; [W14] "E4M3 is enough
 * everywhere" with fine-grained scaling) */
#define FP8SQ_RECIPE_HYBRID 0     /* x, W in E4M3; dY in E5M2 */
#define FP8SQ_RECIPE_E4M3 1       /* everything in E4M3       */

/*
 * Delayed-scaling state of one tensor role ([TS] core vocabulary "Delayed
 * Scaling"; [TE] fp8_meta amax_history and scale): a block of
 * FP8SQ_STATE_FLOATS(H) fp32 values in device memory,
 *     [0 .. H-1]  amax history, newest first (index 0 = the current step)
 *     [H]         m, the multiplier applied before the cast (fmax / a)
 *     [H + 1]     s, the dequantisation step (a / fmax)
 * where a is the history's reduction.  Several states may be packed back to
 * back (state i at offset i * FP8SQ_STATE_FLOATS(H)).
 */
#define FP8SQ_STATE_FLOATS(H) ((H) + 2)

/* ---- 1. amax ------------------------------------------------------------
 * [TS] core vocabulary: amax = the maximum absolute value of a tensor.
 * Computes max|x| of every scaling unit of x[rows][cols] (x: bf16 or fp32).
 *   gran TENSOR:       amax_out[0]
 *   gran TILE_1x128:   amax_out[rows][cols/128]   (cols % 128 == 0)
 *   gran BLOCK_128x128 amax_out[rows/128][cols/128] (rows, cols % 128 == 0)
 *   gran MX32:         amax_out[rows][cols/32]    (cols % 32 == 0)
 * A NaN in a unit gives a NaN amax.  x must be 16-byte aligned; for TENSOR
 * any size is accepted (rows * cols == 0 gives 0).
 */
FP8SQ_API int fp8_amax(const void* x, int x_dtype, int64_t rows, int64_t cols, int gran,
                       float* amax_out, void* stream);

/* ---- 2. scale state -------------------------------------------------------
 * fp8_scale_init: sets n_states packed states to history = 0, m = s = 1.
 * fp8_update_scale: the end-of-step update of delayed scaling ([TS] core
 * vocabulary; [TE] DelayedScaling).  For every state i: a = max over the
 * history (algo MAX) or its newest entry (MOST_RECENT); if a is finite and
 * > 0 then m = fmax/a and s = a/fmax (one fp32 division each, fmax from
 * formats[i]), otherwise m and s are kept; then the history rolls by one
 * (entry j takes entry j-1) and entry 0 becomes 0.
 * formats: HOST array of n_states FP8SQ_E4M3 / FP8SQ_E5M2 (copied at call).
 * n_states <= 1024, 1 <= history_len <= 4096.
 */
FP8SQ_API int fp8_scale_init(float* states, int n_states, int history_len, void* stream);
FP8SQ_API int fp8_update_scale(float* states, int n_states, int history_len, const int* formats,
                               int algo, void* stream);

/* ---- 3. quantize ------------------------------------------------------------
 * q = sat_RNE_fp8(fp32(x) * m) for every element, m taken from the element's
 * scaling unit ([W14] absmax bullet; [TS] worked example: the multiplier
 * 448/240 maps 120 to 224 and a spike of 300 clips at 448).
 *
 *   x         device, bf16 or fp32 [rows][cols], 16-byte aligned
 *   format    FP8SQ_E4M3 / FP8SQ_E5M2 (satfinite: |x*m| >= fmax and +-inf
 *             give +-fmax; NaN gives a NaN code; -0 and negative values that
 *             round to zero give 0x80)
 *   gran, delayed_state:
 *     TENSOR + delayed_state != NULL: delayed scaling.  m = state[H]; the
 *       tensor's amax is max-combined into state[0] (atomic, so several
 *       tensors may share a role).  scales_out, if not NULL (1 float),
 *       receives s = state[H + 1], the dequantisation scale of this cast.
 *     TENSOR + delayed_state == NULL: current scaling, two passes (amax,
 *       then cast).  amax_out (1 float) and scales_out (1 float, receives
 *       s = amax/fmax) are REQUIRED.  m = fmax/amax (amax 0 or non-finite:
 *       m = s = 1).
 *     TILE_1x128 / BLOCK_128x128: current scaling per unit, one pass;
 *       scales_out f32 [rows][cols/128] / [rows/128][cols/128] receives s.
 *     MX32 / MX32_TILED: one pass; scales_out u8 [rows][cols/32] (MX32) or
 *       the tiled layout above (MX32_TILED) receives the E8M0 code
 *       e + 127 of the smallest power of two 2^e with amax <= fmax * 2^e
 *       (clamped to [-127, 127]; amax 0 -> 127; non-finite -> 0xFF with
 *       m = 1); m = 2^-e.
 *     TILE_128x1 / MX32_COL_TILED (column units, for the backward products
 *       that contract over the rows of x): the same rules applied to 128
 *       (or 32) consecutive values of each COLUMN.  Needs bf16 x, rows % 128
 *       == 0 and cols % 16 == 0 (MX: cols % 128 == 0).  qT is required (the
 *       transposed codes are the GEMM operand), q may be NULL.  scales_out:
 *       f32 [rows/128][cols] (TILE_128x1), or the E8M0 codes of qT's 32-value
 *       row blocks in the tiled layout of the [cols][rows] matrix qT
 *       (MX32_COL_TILED).
 *     TILE_1x128_POW2 / BLOCK_128x128_POW2 / MX32_FLOOR_TILED (recipe
 *       variants; rows, cols % 128 == 0): the unit's scale is a power of two,
 *       written as an E8M0 code into the tiled layout above, repeated over
 *       every 32-value block the unit covers, so the codes feed the
 *       block-scaled GEMM.  POW2: the smallest 2^e with amax <= fmax * 2^e
 *       (nothing clips).  FLOOR: e = floor(log2 amax) - emax, the OCP MX
 *       convention, which clips a block whose largest significand exceeds
 *       1.75 (sat_count counts those elements).
 *   q         device u8 [rows][cols], 16-byte aligned
 *   qT        device u8 [cols][rows] (the transposed codes) or NULL; for
 *             TENSOR (same scale; rows, cols % 16 == 0) and BLOCK_128x128
 *             (qT's 128x128 block scales are the transpose of scales_out),
 *             required for the column units
 *   amax_out  device f32 per unit (layout as fp8_amax) or NULL (see above)
 *   sat_count device u64 or NULL: the number of elements with |x*m| > fmax
 *             (they clip) is ADDED to it.
 *   history_len  H of delayed_state (ignored when it is NULL)
 */
FP8SQ_API int fp8_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int format,
                           int gran, float* delayed_state, int history_len, uint8_t* q,
                           uint8_t* qT, void* scales_out, float* amax_out,
                           unsigned long long* sat_count, void* stream);

/* fp8_quantize_rows_cols: both operands of a fine-grained linear layer's
 * products from one read of x ([W14] absmax bullet: 1x128 tiles / 32-value
 * blocks; the column units are the wgrad operands, which contract over the
 * rows of x).  The result is bit-identical to two fp8_quantize calls:
 *   unit TILE_1x128:  q, row_scales      = fp8_quantize(TILE_1x128)
 *                     qT, col_scales     = fp8_quantize(TILE_128x1)
 *   unit MX32_TILED:  q, row_scales      = fp8_quantize(MX32_TILED)
 *                     qT, col_scales     = fp8_quantize(MX32_COL_TILED)
 * with the layouts documented there (f32 [rows][cols/128] and
 * [rows/128][cols]; or the tiled E8M0 layouts of x and of qT).
 *   unit TILE_1x128_POW2: q, row_scales = fp8_quantize(TILE_1x128_POW2)
 *                     (power-of-two 1x128 tiles, tiled E8M0 layout of x);
 *                     qT, col_scales: power-of-two 128x1 column tiles, the
 *                     same rule on 128 consecutive values of a column, each
 *                     code in the four 32-row blocks it covers of the tiled
 *                     E8M0 layout of qT (as MX32_COL_TILED lays them out).
 *   x        device bf16 [rows][cols], 16-byte aligned; rows, cols % 128 == 0
 *   q        device u8 [rows][cols]; qT device u8 [cols][rows]; 16-byte aligned
 *   row_scales, col_scales  device, 4-byte aligned (16 for the E8M0 layouts)
 *   sat_count  device u64 or NULL: the column-unit pass's saturations are
 *              ADDED to it.
 */
FP8SQ_API int fp8_quantize_rows_cols(const void* x, int64_t rows, int64_t cols, int format, int unit,
                                     uint8_t* q, void* row_scales, uint8_t* qT, void* col_scales,
                                     unsigned long long* sat_count, void* stream);

/* ---- 4. GEMM ----------------------------------------------------------------
 * D[m][n] = epi( sum_k Ahat[m][k] * Bhat[n][k] ) with Ahat = dec(qA) * sA,
 * Bhat = dec(qB) * sB ([W14] FP8 bullet: matmuls run in FP8 with a wider
 * accumulator; x ~ q * scale).  Accumulation is fp32 in tensor memory;
 * epi multiplies by the scales, adds bias[n] if given, and rounds to the
 * output type (bf16: round-to-nearest-even).
 *   A  device u8 [M][K] (K contiguous), B device u8 [N][K] (K contiguous);
 *      both 16-byte aligned.  a_format / b_format each E4M3 or E5M2
 *      (E5M2 x E4M3 is the HYBRID dgrad / wgrad pairing).
 *   (a_gran, b_gran) pairs:
 *     (TENSOR, TENSOR): a_scale, b_scale = device f32[1] each (s).
 *     (TILE_1x128, BLOCK_128x128): a_scale f32 [M][K/128], b_scale f32
 *       [N/128][K/128]; partial sums over each 128-wide K block are promoted
 *       to fp32 registers with sA * sB ([W14] accumulation bullet:
 *       promotion to fp32 at fixed intervals); K % 128 == 0.
 *     (TILE_128x1, TILE_128x1): A and B are the transposed codes qT of two
 *       column-tile quantisations (the wgrad operands dy^T and x^T, whose
 *       contraction runs over the original rows): a_scale f32 [K/128][M],
 *       b_scale f32 [K/128][N]; every K block's partial is promoted with
 *       sA[kb][m] * sB[kb][n]; K % 128 == 0.
 *     (any of MX32_TILED, MX32_COL_TILED, TILE_1x128_POW2, BLOCK_128x128_POW2,
 *      MX32_FLOOR_TILED for each operand): a_scale, b_scale u8 E8M0
 *       in the tiled layout of the operand (as written by fp8_quantize
 *       MX32_TILED for q, or MX32_COL_TILED for qT), 16-byte aligned;
 *       D = sum_k dec(qA) 2^(eA - 127) dec(qB) 2^(eB - 127) on the
 *       block-scaled tensor-core path ([W14] absmax bullet: every 32
 *       numbers share a scale); M, N, K % 128 == 0.
 *   D  device [M][N], bf16 or f32, 16-byte aligned; bias device f32 [N] or NULL.
 *   Shapes: M >= 0, N % 8 == 0, K % 16 == 0 (TENSOR) / % 128 (others).
 *   K == 0 writes epi(0).
 */
FP8SQ_API int fp8_gemm(const uint8_t* A, int a_format, const void* a_scale, int a_gran,
                       const uint8_t* B, int b_format, const void* b_scale, int b_gran,
                       int64_t M, int64_t N, int64_t K, const float* bias, void* D, int d_dtype,
                       void* stream);

/* fp8_gemm_layout: fp8_gemm with per-tensor scales (a_gran = b_gran =
 * TENSOR) whose operands may also be stored MN-major:
 *   a_major K_MAJOR: A [M][K] (K contiguous);  MN_MAJOR: A [K][M] (M contiguous)
 *   b_major K_MAJOR: B [N][K] (K contiguous);  MN_MAJOR: B [K][N] (N contiguous)
 * The linear layer's backward products read the forward codes as they are
 * ([W14] FP8 bullet; [TS] core vocabulary: a scaling scheme should not add
 * passes over the tensor): dgrad dx = dy W takes B = the codes of W [N][K]
 * MN-major, wgrad dW = dy^T x takes A = the codes of dy [M][N] and B = the
 * codes of x [M][K], both MN-major, so no transposed copy is written.
 * Needs M % 16 == 0 for an MN-major A and N % 16 == 0 for an MN-major B (row
 * pitch a multiple of 16 bytes), K % 16 == 0; otherwise as fp8_gemm.
 * FP8SQ_ERR_UNSUPPORTED for other granularities with an MN-major operand. */
#define FP8SQ_K_MAJOR 0
#define FP8SQ_MN_MAJOR 1
FP8SQ_API int fp8_gemm_layout(const uint8_t* A, int a_format, const void* a_scale, int a_major,
                              const uint8_t* B, int b_format, const void* b_scale, int b_major,
                              int64_t M, int64_t N, int64_t K, const float* bias, void* D, int d_dtype,
                              void* stream);

/* fp8_gemm_cast: fp8_gemm_layout with a bf16 output D that also casts D, as
 * stored, to FP8 in the GEMM's epilogue with delayed per-tensor scaling
 * ([TS] delayed scaling; [W14] FP8 bullet): the result is the same as
 *   fp8_gemm_layout(..., D, FP8SQ_BF16, ...);
 *   fp8_quantize(D, FP8SQ_BF16, M, N, q_format, FP8SQ_TENSOR, q_state,
 *                q_history_len, q_out, NULL, NULL, NULL, NULL, stream);
 * (q_out[m][n] = sat_rne(fp32(D[m][n]) * q_state[H]), max|D| max-combined
 * into q_state[0]) without reading D back: the next linear layer's input
 * cast (or the previous layer's output-gradient cast) rides on this GEMM.
 *   q_out     device u8 [M][N], 16-byte aligned; q_state device f32 state
 *             block of q_history_len; q_format E4M3 or E5M2.
 *   Needs K > 0, N % 16 == 0 (and the fp8_gemm_layout shape rules).
 *   Saturations are not counted. */
FP8SQ_API int fp8_gemm_cast(const uint8_t* A, int a_format, const void* a_scale, int a_major,
                            const uint8_t* B, int b_format, const void* b_scale, int b_major,
                            int64_t M, int64_t N, int64_t K, const float* bias, void* D,
                            uint8_t* q_out, int q_format, float* q_state, int q_history_len,
                            void* stream);

/* ---- 5. linear layer ---------------------------------------------------------
 * [TE] te.Linear under fp8_autocast; [TS] Part 01 (HYBRID).
 * Forward  y[M][N]  = x[M][K] W[N][K]^T      (x, W quantised in E4M3)
 * Backward dx[M][K] = dy[M][N] W             (dy in E5M2 under HYBRID)
 *          dW[N][K] = dy^T x                 (fp32 output, the master-weight
 *                                              precision of [W14] FP8 bullet)
 * x, w, dy: device bf16.  y: bf16 or f32.  dx: bf16.  dw: f32.
 * gran TENSOR: delayed scaling when x_state / w_state / dy_state are given
 *   (each a state block of history_len), current scaling when all are NULL.
 *   The forward keeps the codes of x and W in the workspace; the backward
 *   adds dy's codes and reads all three as they are (dgrad and wgrad take
 *   them as MN-major operands, see fp8_gemm_layout): no transposed copy.
 * gran TILE_1x128: x in 1x128 tiles, W in 128x128 blocks, current scaling
 *   ([W14] absmax bullet, the DeepSeek-V3 granularity).  Backward: dy in
 *   1x128 tiles along N for dgrad (B = W^T codes, its blocks transposed); dy
 *   and x in 128x1 column tiles along M for wgrad (both operands promoted per
 *   128 tokens).  The forward also casts x in column tiles for the backward.
 * gran TILE_1x128_POW2: the units of TILE_1x128 with power-of-two scales
 *   (the MX rule on each 1x128 tile, 128x128 block and 128x1 column tile,
 *   stored as tiled E8M0 codes): every GEMM runs on the block-scaled MMA,
 *   with no promotion.  dgrad's B is W^T with W's blocks transposed.
 * gran MX32: every operand in MX-32 blocks along its contraction dimension:
 *   x, W along K (forward), dy along N and W along N (dgrad), dy and x along
 *   M (wgrad); the forward also writes the column-block codes of x and W.
 * workspace: device, >= fp8_linear_workspace_bytes(M, N, K, gran), 256-byte
 *   aligned; the same workspace must be passed to the matching backward.
 * Shapes: M, N, K % 128 == 0 (TENSOR: M % 16, N % 16, K % 16).
 * fp8_linear_bwd takes the forward's gran and workspace.  Under the HYBRID
 * recipe dy is cast to E5M2, under RECIPE_E4M3 to E4M3.
 * Streams: all work is ordered on `stream`.  fp8_linear_bwd runs wgrad on a
 *   library-owned non-blocking stream (one per host thread and device, kept
 *   for the thread's life) beside dgrad, forked from `stream` by an event and
 *   joined back into it by another before the call returns; work queued on
 *   `stream` after the call sees both results.  (Small layers' two grids
 *   share the device; large layers' wgrad takes the SMs that dgrad's last
 *   wave of tiles leaves idle.)  Under stream capture this records two
 *   parallel branches; the library's stream is created only outside capture
 *   (a call captured before one exists runs both GEMMs on `stream`).
 */
FP8SQ_API size_t fp8_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int gran);
FP8SQ_API int fp8_linear_fwd(const void* x, const void* w, int64_t M, int64_t N, int64_t K,
                             int gran, int recipe, float* x_state, float* w_state,
                             int history_len, void* workspace, size_t ws_bytes,
                             const float* bias, void* y, int y_dtype, void* stream);
FP8SQ_API int fp8_linear_bwd(const void* dy, int64_t M, int64_t N, int64_t K, int gran, int recipe,
                             float* dy_state, int history_len, void* workspace, size_t ws_bytes,
                             void* dx, float* dw, void* stream);

/* ---- 5a. LayerNorm fused into the cast ---------------------------------
 * [TE] te.LayerNorm / te.LayerNormLinear: the normalisation in front of a
 * linear layer, fused here with the amax and the FP8 cast so the bf16
 * LayerNorm output never goes to HBM.  Per row r of x [M][K] (bf16):
 *   mu[r] = sum(x)/K, var = sum((x - mu)^2)/K, rstd[r] = 1/sqrt(var + eps),
 *   y = (x - mu[r]) * rstd[r] * gamma[c] + beta[c]      (fp32 arithmetic)
 * then q = sat_RNE_fp8(y * m) with delayed per-tensor scaling: m = state[H],
 * amax(|y|) max-combined into state[0] (as fp8_quantize TENSOR + delayed).
 *   gamma, beta  device f32 [K], 16-byte aligned (beta may be NULL)
 *   q            device u8 [M][K]; qT device u8 [K][M] or NULL
 *   mu_out, rstd_out  device f32 [M], 16-byte aligned, required (the LayerNorm
 *                     backward needs them)
 *   M % 16 == 0, K % 16 == 0; x, q, qT 16-byte aligned.
 * The row statistics are fp32 reductions whose order is this library's; the
 * codes equal those of the exact LayerNorm except where y * m lies within the
 * reductions' rounding error of a midpoint between two codes.
 * fp8_layernorm_linear_fwd: the same cast of x, then the per-tensor delayed
 * linear forward of fp8_linear_fwd (W cast, GEMM) with the TENSOR workspace
 * layout, so fp8_linear_bwd (gran TENSOR) runs the backward of the linear.
 */
FP8SQ_API int fp8_layernorm_quantize(const void* x, const float* gamma, const float* beta, float eps,
                                     int64_t M, int64_t K, int format, float* delayed_state, int history_len,
                                     uint8_t* q, uint8_t* qT, float* mu_out, float* rstd_out, void* stream);
FP8SQ_API int fp8_layernorm_linear_fwd(const void* x, const float* gamma, const float* beta, float eps,
                                       const void* w, int64_t M, int64_t N, int64_t K, float* x_state,
                                       float* w_state, int history_len, void* workspace, size_t ws_bytes,
                                       float* mu_out, float* rstd_out, const float* bias, void* y, int y_dtype,
                                       void* stream);

/* ---- 5b. forward linear without allocation --------------------------------
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc or hand over a workspace -- code running inside
 * a framework that owns every byte of device memory through its own pool, or
 * a plugin called where allocating (which can synchronise the device) is not
 * allowed.
 *
 * Computes y = x W^T like fp8_linear_fwd with gran TENSOR and current
 * per-tensor scaling (x, W cast to E4M3 with m = 448/amax; y = acc * s_x *
 * s_w + bias).  Its scratch -- the codes of x and W and four fp32 scalars --
 * is a file-scope device array of FP8SQ_NOALLOC_SCRATCH_BYTES (32 MiB) that
 * every GPU on which this library's device code is loaded holds until the
 * process exits.  The call allocates nothing itself (no cudaMalloc, cudaFree
 * or allocating library routine).
 *   M, N, K must each be below 2^31 (checked before any product is formed).
 *   x  device bf16 [M][K], w device bf16 [N][K], y device bf16 / f32 [M][N],
 *      bias device f32 [N] or NULL; x, w, y 16-byte aligned.
 *   Needs N % 8 == 0, K % 16 == 0 and round256(M*K) + round256(N*K) + 256 <=
 *   FP8SQ_NOALLOC_SCRATCH_BYTES; larger sizes return FP8SQ_ERR_UNSUPPORTED
 *   with a message giving the bytes needed.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) for that device.  Under CUDA's lazy module loading
 * (the default) that lookup may be what loads the library's device code onto
 * the device and places the array there, so the first call can reserve the
 * 32 MiB and can fail with FP8SQ_ERR_CUDA (out of memory).  Make that first
 * call at set-up time, before any stream capture; later calls on the device
 * reserve nothing.  All calls share the one array and it keeps the last
 * call's contents (the amax slots are cleared by every call), so calls whose
 * work overlaps on the GPU -- on different streams, or from several threads
 * -- race on it and must be serialised by the caller.
 */
#define FP8SQ_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
FP8SQ_API int fp8_linear_fwd_noalloc(const void* x, const void* w, int64_t M, int64_t N, int64_t K,
                                     const float* bias, void* y, int y_dtype, void* stream);

/* ---- 6. diagnostics --------------------------------------------------------
 * fp8_device_status: synchronises the current device and returns
 *   FP8SQ_ERR_TIMEOUT if any bounded device-side wait of this library ran out
 *   since the last clear (the kernel that hit it wrote nothing further and
 *   returned), FP8SQ_OK otherwise.  clear != 0 resets the word.  While the
 *   word is set, GEMM kernels return early without computing.
 * fp8_selftest_wait_timeout: exercises that failure path on purpose, with
 *   no fault and no hang: one thread waits, through the library's bounded
 *   wait, on an mbarrier phase nothing completes, gives up after limit_us
 *   (1 .. 1e6), sets the device error word and returns; *waited_out (device
 *   int) receives 1.  fp8_device_status then reports FP8SQ_ERR_TIMEOUT until
 *   cleared.
 * fp8_last_error: message for the calling thread's last non-zero status
 *   (static thread-local storage; never NULL).
 * fp8_abi_version: 7.  Changes from 6: fp8_linear_fwd / fp8_linear_bwd,
 *   fp8_linear_workspace_bytes and fp8_quantize_rows_cols accept
 *   TILE_1x128_POW2 (the fine-grained units with power-of-two scales).
 *   Changes from 5 to 6: fp8_gemm_cast added (the GEMM's
 *   epilogue casts its bf16 output to FP8 with delayed scaling).
 *   Changes from 4 to 5: fp8_gemm_layout added (MN-major
 *   operands); the per-tensor linear layer keeps no transposed codes (its
 *   backward reads the forward's codes MN-major), so
 *   fp8_linear_workspace_bytes(TENSOR) is smaller.
 *   Changes from 3 to 4: fp8_quantize_rows_cols added.
 *   Changes from 2 to 3: fp8_selftest_wait_timeout added;
 *   the LayerNorm entry points need 16-byte aligned gamma, beta, mu, rstd;
 *   a delayed per-tensor fp8_quantize writes s to a non-NULL scales_out.
 *   Every kernel is launched with programmatic stream serialisation (the
 *   next kernel's launch overlaps; memory order on the stream is kept).
 */
FP8SQ_API int fp8_device_status(int clear);
FP8SQ_API int fp8_selftest_wait_timeout(int limit_us, int* waited_out, void* stream);
FP8SQ_API const char* fp8_last_error(void);
FP8SQ_API int fp8_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FP8SQ_H */

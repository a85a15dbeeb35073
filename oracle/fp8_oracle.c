/*
 * fp8_oracle.c -- plain, slow, obviously-correct CPU oracle for the FP8
 * scaled-linear path.  TEST INFRASTRUCTURE ONLY: it is loaded by the tests,
 * by __graft_entry__.smoke() and by bench.py's CPU-baseline leg, never by the
 * product library.  It shares no code, header or table with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [TS]  "Transformer Scaling" (lab.mindcaptain.ai, reading 06):
 *         "Part 01 - Low precision starts with range management",
 *         "Core vocabulary" (amax, Delayed Scaling), "Worked example".
 *   [W14] "Week 14. Scaling laws, precision, parallelism" (snula course):
 *         absmax bullet, FP8 bullet, "Accumulation precision" bullet,
 *         bf16-vs-fp16 "In plain terms" paragraph.
 *   [TE]  "Accelerating Transformer Training with NVIDIA Transformer Engine"
 *         (JuicyTalk): DelayedScaling(HYBRID, amax_history_len=16,
 *         amax_compute_algo="max") recipe and the fp8_meta dump.
 *
 * Every float operation below that decides a result is a single IEEE
 * operation rounded to nearest (compile with -ffp-contract=off, no fast-math).
 * Readings of points the pages leave open are stated where they are used.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_E4M3 0
#define ORC_E5M2 1

#define ORC_ALGO_MAX 0
#define ORC_ALGO_MOST_RECENT 1

/* ------------------------------------------------------------------------
 * 1. Codec.
 * [W14] FP8 bullet: E4M3 = 4 exponent bits, 3 mantissa bits, max 448;
 * E5M2 = 5 exponent bits, 2 mantissa bits, max 57344.  Max 448 fixes the
 * E4M3 variant without infinities (exponent bias 7, only S.1111.111 is NaN);
 * E5M2 keeps the IEEE layout (bias 15, exponent 31 = inf/NaN).
 * ---------------------------------------------------------------------- */
double orc_decode(int fmt, uint8_t c)
{
    int s = c >> 7;
    double v;
    if (fmt == ORC_E4M3) {
        int e = (c >> 3) & 15, m = c & 7;
        if (e == 15 && m == 7) return NAN;
        v = (e == 0) ? ldexp((double)m / 8.0, 1 - 7) : ldexp(1.0 + (double)m / 8.0, e - 7);
    } else {
        int e = (c >> 2) & 31, m = c & 3;
        if (e == 31) return m ? NAN : (s ? -INFINITY : INFINITY);
        v = (e == 0) ? ldexp((double)m / 4.0, 1 - 15) : ldexp(1.0 + (double)m / 4.0, e - 15);
    }
    return s ? -v : v;
}

/* Largest finite code (positive half): E4M3 0x7E = 448, E5M2 0x7B = 57344. */
int orc_max_code(int fmt) { return fmt == ORC_E4M3 ? 0x7E : 0x7B; }
double orc_fmax(int fmt) { return orc_decode(fmt, (uint8_t)orc_max_code(fmt)); }

/* Encode by definition: the representable value nearest to v.  The
 * non-negative finite codes 0..maxcode decode to strictly increasing values,
 * so a binary search over the decoded values finds the two neighbours of
 * |v|.  On an exact tie the code with an even last bit (= even mantissa)
 * wins: round-to-nearest-even, which the [W14] accumulation example pins
 * (promotion every 8 terms gives exactly 300 only under ties-to-even).
 * |v| at or beyond the largest finite value saturates to it, and so does
 * infinity ([TS] worked example: "clips at 448").  The sign is copied, so a
 * negative value that rounds to zero gives -0 (0x80).  NaN gives 0x7F. */
uint8_t orc_encode(int fmt, float v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    int maxc = orc_max_code(fmt);
    if (a >= orc_decode(fmt, (uint8_t)maxc)) return (uint8_t)(sign | maxc);
    int lo = 0, hi = maxc;              /* invariant: dec(lo) <= a < dec(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_decode(fmt, (uint8_t)mid) <= a) lo = mid; else hi = mid;
    }
    double dlo = orc_decode(fmt, (uint8_t)lo), dhi = orc_decode(fmt, (uint8_t)hi);
    double half = (dlo + dhi) / 2.0;    /* exact in double */
    int c;
    if (a < half) c = lo;
    else if (a > half) c = hi;
    else c = (lo % 2 == 0) ? lo : hi;
    return (uint8_t)(sign | c);
}

/* bf16 = the upper 16 bits of an fp32 with round-to-nearest-even on the
 * dropped 16 bits.  [W14] bf16 paragraph: 8 significant bits, 257 rounds to
 * 256 (a tie between 256 and 258, resolved to the even significand). */
uint16_t orc_bf16_from_f32(float v)
{
    uint32_t b;
    memcpy(&b, &v, 4);
    if (isnan(v)) return (uint16_t)((b >> 16) | 0x0040);
    uint32_t upper = b >> 16, lower = b & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

float orc_f32_from_bf16(uint16_t h)
{
    uint32_t b = (uint32_t)h << 16;
    float v;
    memcpy(&v, &b, 4);
    return v;
}

/* ------------------------------------------------------------------------
 * 2. amax ([TS] core vocabulary: "the maximum absolute value in a tensor or
 * history window").  Exact; any NaN makes the result NaN.
 * ---------------------------------------------------------------------- */
float orc_amax(const float* x, int64_t n)
{
    float m = 0.0f;
    int any_nan = 0;
    #pragma omp parallel for reduction(max:m) reduction(|:any_nan) schedule(static) if(n > 65536)
    for (int64_t i = 0; i < n; ++i) {
        if (isnan(x[i])) any_nan = 1;
        else if (fabsf(x[i]) > m) m = fabsf(x[i]);
    }
    return any_nan ? NAN : m;
}

/* max of two amaxes with NaN propagation */
static float amax2(float a, float b)
{
    if (isnan(a) || isnan(b)) return NAN;
    return a > b ? a : b;
}

/* ------------------------------------------------------------------------
 * 3. Current scaling of one unit.
 * [W14] absmax bullet: the grid step is max|x| / qmax and x ~ q * step; the
 * step comes from the current block ("online"), not from earlier steps.
 * [TS] worked example uses the multiplier form: 448 / 240 multiplies the
 * value before the cast.  Both are kept: m = fmax / amax (multiplier applied
 * before the cast) and s = amax / fmax (dequantisation step), each one IEEE
 * fp32 division.  amax zero or non-finite: m = s = 1 (reading; pages silent).
 * ---------------------------------------------------------------------- */
void orc_current_scale(float amax, int fmt, float* m, float* s)
{
    float fmax = (float)orc_fmax(fmt);
    if (isfinite(amax) && amax > 0.0f) {
        *m = fmax / amax;
        *s = amax / fmax;
    } else {
        *m = 1.0f;
        *s = 1.0f;
    }
}

/* Quantize a run of values with a multiplier: q = enc(fp32(x * m)).  One
 * fp32 multiply, then the saturating round-to-nearest-even cast.  Counts
 * the elements whose scaled magnitude exceeds fmax (they clip). */
static int64_t quant_run(const float* x, int64_t n, int64_t stride, float m, int fmt,
                         uint8_t* q, int64_t qstride)
{
    float fmax = (float)orc_fmax(fmt);
    int64_t sat = 0;
    #pragma omp parallel for reduction(+:sat) schedule(static) if(n > 65536)
    for (int64_t i = 0; i < n; ++i) {
        float p = x[i * stride] * m;
        if (fabsf(p) > fmax) ++sat;
        q[i * qstride] = orc_encode(fmt, p);
    }
    return sat;
}

/* ------------------------------------------------------------------------
 * 4. Per-tensor current scaling: amax of the whole tensor, m and s, cast.
 * Returns the number of clipped elements.
 * ---------------------------------------------------------------------- */
int64_t orc_quantize_tensor_current(const float* x, int64_t n, int fmt, uint8_t* q,
                                    float* amax_out, float* s_out)
{
    float a = orc_amax(x, n), m, s;
    orc_current_scale(a, fmt, &m, &s);
    *amax_out = a;
    *s_out = s;
    return quant_run(x, n, 1, m, fmt, q, 1);
}

/* Cast with a given multiplier (used by the delayed path and by tests). */
int64_t orc_quantize_with_multiplier(const float* x, int64_t n, float m, int fmt, uint8_t* q)
{
    return quant_run(x, n, 1, m, fmt, q, 1);
}

/* ------------------------------------------------------------------------
 * 5. 1x128 activation tiles ([W14] absmax bullet: DeepSeek-V3 gave "every 128
 * activation values" their own scale).  Reading: the 128 values run along
 * the contiguous (last) dimension of x[R][C]; C % 128 == 0.
 * s[R][C/128], amax[R][C/128].
 * ---------------------------------------------------------------------- */
int64_t orc_quantize_tile1x128(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q,
                               float* s_out, float* amax_out)
{
    int64_t T = C / 128, sat = 0;
    #pragma omp parallel for reduction(+:sat) schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t t = 0; t < T; ++t) {
            const float* u = x + r * C + t * 128;
            float a = orc_amax(u, 128), m, s;
            orc_current_scale(a, fmt, &m, &s);
            s_out[r * T + t] = s;
            if (amax_out) amax_out[r * T + t] = a;
            sat += quant_run(u, 128, 1, m, fmt, q + r * C + t * 128, 1);
        }
    }
    return sat;
}

/* ------------------------------------------------------------------------
 * 6. 128x128 weight blocks ([W14] absmax bullet: "each 128x128 block of
 * weights").  R % 128 == 0, C % 128 == 0.  s[R/128][C/128].
 * ---------------------------------------------------------------------- */
int64_t orc_quantize_block128(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q,
                              float* s_out, float* amax_out)
{
    int64_t BR = R / 128, BC = C / 128, sat = 0;
    #pragma omp parallel for reduction(+:sat) schedule(static)
    for (int64_t bi = 0; bi < BR; ++bi) {
        for (int64_t bj = 0; bj < BC; ++bj) {
            float a = 0.0f;
            for (int64_t r = 0; r < 128; ++r)
                a = amax2(a, orc_amax(x + (bi * 128 + r) * C + bj * 128, 128));
            float m, s;
            orc_current_scale(a, fmt, &m, &s);
            s_out[bi * BC + bj] = s;
            if (amax_out) amax_out[bi * BC + bj] = a;
            for (int64_t r = 0; r < 128; ++r) {
                int64_t off = (bi * 128 + r) * C + bj * 128;
                sat += quant_run(x + off, 128, 1, m, fmt, q + off, 1);
            }
        }
    }
    return sat;
}

/* ------------------------------------------------------------------------
 * 7. MX blocks of 32 with a power-of-two (E8M0) scale.
 * [W14] absmax bullet: "MX formats give every 32 numbers a shared scale".
 * Reading (pages give no exponent rule): the absmax rule restricted to powers
 * of two -- the smallest 2^e with amax <= fmax * 2^e, so no element clips.
 * With amax = f * 2^E, 1 <= f < 2, and fmax = 1.75 * 2^emax (both formats):
 * e = E - emax, plus one when f > 1.75.  e is clamped to [-127, 127]; the
 * E8M0 code is e + 127.  amax == 0 gives e = 0 (code 127); non-finite amax
 * gives code 0xFF (the E8M0 NaN) and the cast uses m = 1.
 * m = 2^-e and s = 2^e are exact in fp32.
 * ---------------------------------------------------------------------- */
uint8_t orc_mx_scale_code(float amax, int fmt)
{
    if (!isfinite(amax)) return 0xFF;
    if (amax == 0.0f) return 127;
    int emax = (fmt == ORC_E4M3) ? 8 : 15;
    int E;
    double f = frexp((double)amax, &E);  /* amax = f * 2^E, 0.5 <= f < 1 */
    f *= 2.0;
    E -= 1;                              /* amax = f * 2^E, 1 <= f < 2 */
    int e = E - emax + (f > 1.75 ? 1 : 0);
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint8_t)(e + 127);
}

/* The OCP MX convention's exponent (a recipe variant, not the pages'):
 * e = floor(log2(amax)) - emax, so a block whose largest significand
 * exceeds 1.75 clips at fmax.  Same clamping and special codes as above. */
uint8_t orc_mx_scale_code_floor(float amax, int fmt)
{
    if (!isfinite(amax)) return 0xFF;
    if (amax == 0.0f) return 127;
    int emax = (fmt == ORC_E4M3) ? 8 : 15;
    int E;
    frexp((double)amax, &E);
    int e = (E - 1) - emax;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint8_t)(e + 127);
}

int64_t orc_quantize_mx32_floor(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q,
                                uint8_t* e8m0_out)
{
    int64_t T = C / 32, sat = 0;
    #pragma omp parallel for reduction(+:sat) schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t t = 0; t < T; ++t) {
            const float* u = x + r * C + t * 32;
            uint8_t code = orc_mx_scale_code_floor(orc_amax(u, 32), fmt);
            float m = (code == 0xFF) ? 1.0f : (float)ldexp(1.0, -((int)code - 127));
            e8m0_out[r * T + t] = code;
            sat += quant_run(u, 32, 1, m, fmt, q + r * C + t * 32, 1);
        }
    }
    return sat;
}

/* Power-of-two scales for 1x128 tiles and 128x128 blocks (a recipe variant:
 * the scale of each unit restricted to a power of two, by the same rule as
 * the MX blocks -- the smallest 2^e with amax <= fmax * 2^e).  Output: E8M0
 * codes, e_tile[R][C/128] / e_block[R/128][C/128]. */
int64_t orc_quantize_tile1x128_pow2(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q,
                                    uint8_t* e_out)
{
    int64_t T = C / 128, sat = 0;
    #pragma omp parallel for reduction(+:sat) schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t t = 0; t < T; ++t) {
            const float* u = x + r * C + t * 128;
            uint8_t code = orc_mx_scale_code(orc_amax(u, 128), fmt);
            float m = (code == 0xFF) ? 1.0f : (float)ldexp(1.0, -((int)code - 127));
            e_out[r * T + t] = code;
            sat += quant_run(u, 128, 1, m, fmt, q + r * C + t * 128, 1);
        }
    }
    return sat;
}

int64_t orc_quantize_block128_pow2(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q,
                                   uint8_t* e_out)
{
    int64_t BR = R / 128, BC = C / 128, sat = 0;
    #pragma omp parallel for reduction(+:sat) schedule(static)
    for (int64_t bi = 0; bi < BR; ++bi) {
        for (int64_t bj = 0; bj < BC; ++bj) {
            float a = 0.0f;
            for (int64_t r = 0; r < 128; ++r)
                a = amax2(a, orc_amax(x + (bi * 128 + r) * C + bj * 128, 128));
            uint8_t code = orc_mx_scale_code(a, fmt);
            float m = (code == 0xFF) ? 1.0f : (float)ldexp(1.0, -((int)code - 127));
            e_out[bi * BC + bj] = code;
            for (int64_t r = 0; r < 128; ++r) {
                int64_t off = (bi * 128 + r) * C + bj * 128;
                sat += quant_run(x + off, 128, 1, m, fmt, q + off, 1);
            }
        }
    }
    return sat;
}

int64_t orc_quantize_mx32(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q,
                          uint8_t* e8m0_out, float* amax_out)
{
    int64_t T = C / 32, sat = 0;
    #pragma omp parallel for reduction(+:sat) schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t t = 0; t < T; ++t) {
            const float* u = x + r * C + t * 32;
            float a = orc_amax(u, 32);
            uint8_t code = orc_mx_scale_code(a, fmt);
            float m = (code == 0xFF) ? 1.0f : (float)ldexp(1.0, -((int)code - 127));
            e8m0_out[r * T + t] = code;
            if (amax_out) amax_out[r * T + t] = a;
            sat += quant_run(u, 32, 1, m, fmt, q + r * C + t * 32, 1);
        }
    }
    return sat;
}

/* ------------------------------------------------------------------------
 * 7b. Column units, for the backward products that contract over the other
 * dimension (dgrad over the output features, wgrad over the tokens): the
 * same 1x128 / MX-32 rules applied to 128 (or 32) consecutive values of a
 * COLUMN of x[R][C].  By definition these are the row units of x^T.
 *   tile128x1: s[R/128][C] (column c, row block rb at rb*C + c)
 *   mx32_col:  e8m0[R/32][C]
 * Codes keep x's layout: q[r][c].
 * ---------------------------------------------------------------------- */
int64_t orc_quantize_tile128x1(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q,
                               float* s_out, float* amax_out)
{
    int64_t RB = R / 128, sat = 0;
    #pragma omp parallel for reduction(+:sat) schedule(static)
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t rb = 0; rb < RB; ++rb) {
            float a = 0.0f;
            for (int64_t r = rb * 128; r < rb * 128 + 128; ++r)
                a = amax2(a, fabsf(x[r * C + c]));
            float m, s;
            orc_current_scale(a, fmt, &m, &s);
            s_out[rb * C + c] = s;
            if (amax_out) amax_out[rb * C + c] = a;
            sat += quant_run(x + rb * 128 * C + c, 128, C, m, fmt, q + rb * 128 * C + c, C);
        }
    }
    return sat;
}

/* Power-of-two column tiles (the recipe variant of tile128x1): the MX rule's
 * power of two for each 128 consecutive values of a column; E8M0 codes
 * e[R/128][C]. */
int64_t orc_quantize_tile128x1_pow2(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q, uint8_t* e_out)
{
    int64_t RB = R / 128, sat = 0;
    #pragma omp parallel for reduction(+:sat) schedule(static)
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t rb = 0; rb < RB; ++rb) {
            float a = 0.0f;
            for (int64_t r = rb * 128; r < rb * 128 + 128; ++r)
                a = amax2(a, fabsf(x[r * C + c]));
            uint8_t code = orc_mx_scale_code(a, fmt);
            float m = (code == 0xFF) ? 1.0f : (float)ldexp(1.0, -((int)code - 127));
            e_out[rb * C + c] = code;
            sat += quant_run(x + rb * 128 * C + c, 128, C, m, fmt, q + rb * 128 * C + c, C);
        }
    }
    return sat;
}

int64_t orc_quantize_mx32_col(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q,
                              uint8_t* e8m0_out, float* amax_out)
{
    int64_t RB = R / 32, sat = 0;
    #pragma omp parallel for reduction(+:sat) schedule(static)
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t rb = 0; rb < RB; ++rb) {
            float a = 0.0f;
            for (int64_t r = rb * 32; r < rb * 32 + 32; ++r)
                a = amax2(a, fabsf(x[r * C + c]));
            uint8_t code = orc_mx_scale_code(a, fmt);
            float m = (code == 0xFF) ? 1.0f : (float)ldexp(1.0, -((int)code - 127));
            e8m0_out[rb * C + c] = code;
            if (amax_out) amax_out[rb * C + c] = a;
            sat += quant_run(x + rb * 32 * C + c, 32, C, m, fmt, q + rb * 32 * C + c, C);
        }
    }
    return sat;
}

/* ------------------------------------------------------------------------
 * 7c. LayerNorm in front of a linear layer (the Transformer Engine
 * tutorial's te.LayerNormLinear / te.LayerNorm; the pages give no formula,
 * so the standard one): per row, mean = sum(x)/K, var = sum((x-mean)^2)/K,
 * rstd = 1/sqrt(var + eps), y = (x - mean) * rstd * gamma + beta.  Computed
 * in double; y_out is double [R][K], mu / rstd double [R].
 * ---------------------------------------------------------------------- */
void orc_layernorm(const float* x, int64_t R, int64_t K, const float* gamma, const float* beta, double eps,
                   double* y_out, double* mu_out, double* rstd_out)
{
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        const float* row = x + r * K;
        double sum = 0.0;
        for (int64_t k = 0; k < K; ++k) sum += row[k];
        double mean = sum / (double)K;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) ss += (row[k] - mean) * (row[k] - mean);
        double rstd = 1.0 / sqrt(ss / (double)K + eps);
        mu_out[r] = mean;
        rstd_out[r] = rstd;
        for (int64_t k = 0; k < K; ++k)
            y_out[r * K + k] = (row[k] - mean) * rstd * (double)gamma[k] + (beta ? (double)beta[k] : 0.0);
    }
}

/* ------------------------------------------------------------------------
 * 8. Delayed scaling with an amax history.
 * [TS] core vocabulary: delayed scaling "uses historical amax" to set the
 * scale, avoiding a read of the tensor before the cast, at the cost of lag;
 * the worked example shows the stale scale clipping a spike.
 * [TE] recipe: amax_history_len = 16, amax_compute_algo = "max"; the
 * fp8_meta dump shows amax_history[0, :] and scale per tensor role.
 * State per tensor role: hist[H], then m (qscale), then s (dscale).
 * Readings: the current step's amax does not affect its own cast; the newest
 * amax sits at hist[0]; init is hist = 0, m = s = 1; no margin.
 * ---------------------------------------------------------------------- */
void orc_state_init(float* state, int H)
{
    for (int i = 0; i < H; ++i) state[i] = 0.0f;
    state[H] = 1.0f;
    state[H + 1] = 1.0f;
}

/* cast with the state's current multiplier; record this tensor's amax in
 * hist[0] (max with what is there, so two tensors sharing a role combine) */
int64_t orc_quantize_delayed(const float* x, int64_t n, int fmt, float* state, int H, uint8_t* q)
{
    float m = state[H];
    int64_t sat = quant_run(x, n, 1, m, fmt, q, 1);
    state[0] = amax2(state[0], orc_amax(x, n));
    return sat;
}

/* end-of-step update: a = max over the history (or the newest entry);
 * finite positive a sets m = fmax/a, s = a/fmax, otherwise m, s are kept;
 * then the history rolls by one and hist[0] starts the next step at 0. */
void orc_update_scale(float* state, int H, int fmt, int algo)
{
    float a = state[0];
    if (algo == ORC_ALGO_MAX)
        for (int i = 1; i < H; ++i) a = amax2(a, state[i]);
    if (isfinite(a) && a > 0.0f) {
        float fmax = (float)orc_fmax(fmt);
        state[H] = fmax / a;
        state[H + 1] = a / fmax;
    }
    for (int i = H - 1; i >= 1; --i) state[i] = state[i - 1];
    state[0] = 0.0f;
}

/* ------------------------------------------------------------------------
 * 9. Dequantisation to exact doubles: xhat = dec(q) * s(unit).  dec(q) has
 * at most 4 significant bits and s is an fp32, so the product is exact.
 * gran: 0 tensor (s[0]), 1 tile 1x128 (s[R][C/128]), 2 block 128x128
 * (s[R/128][C/128]), 3 MX-32 (E8M0 codes u8[R][C/32]), 4 column tile 128x1
 * (s[R/128][C]), 5 column MX-32 (E8M0 codes u8[R/32][C]), 6 power-of-two 1x128
 * tiles (E8M0 codes u8[R][C/128]), 7 power-of-two 128x128 blocks (E8M0 codes
 * u8[R/128][C/128]), 8 power-of-two 128x1 column tiles (E8M0 codes
 * u8[R/128][C]).
 * ---------------------------------------------------------------------- */
void orc_dequantize(const uint8_t* q, int64_t R, int64_t C, int fmt, int gran,
                    const void* scales, double* out)
{
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t c = 0; c < C; ++c) {
            double s;
            if (gran == 0) s = ((const float*)scales)[0];
            else if (gran == 1) s = ((const float*)scales)[r * (C / 128) + c / 128];
            else if (gran == 2) s = ((const float*)scales)[(r / 128) * (C / 128) + c / 128];
            else if (gran == 4) s = ((const float*)scales)[(r / 128) * C + c];
            else if (gran == 5 || gran == 8) {
                uint8_t code = (gran == 5) ? ((const uint8_t*)scales)[(r / 32) * C + c]
                                           : ((const uint8_t*)scales)[(r / 128) * C + c];
                s = (code == 0xFF) ? NAN : ldexp(1.0, (int)code - 127);
            } else if (gran == 6 || gran == 7) {
                uint8_t code = (gran == 6) ? ((const uint8_t*)scales)[r * (C / 128) + c / 128]
                                           : ((const uint8_t*)scales)[(r / 128) * (C / 128) + c / 128];
                s = (code == 0xFF) ? NAN : ldexp(1.0, (int)code - 127);
            } else {
                uint8_t code = ((const uint8_t*)scales)[r * (C / 32) + c / 32];
                s = (code == 0xFF) ? NAN : ldexp(1.0, (int)code - 127);
            }
            out[r * C + c] = orc_decode(fmt, q[r * C + c]) * s;
        }
    }
}

/* ------------------------------------------------------------------------
 * 10. Unit-check helpers for the [W14] worked examples.
 * ---------------------------------------------------------------------- */

/* int8 symmetric absmax ([W14] absmax bullet): step = amax / (2^(b-1) - 1)
 * with b = 8, q = round(x / step) to nearest even, clamped to +-127. */
void orc_int8_absmax(const float* x, int64_t n, int8_t* q, float* step_out)
{
    float a = orc_amax(x, n);
    float step = a / 127.0f;
    *step_out = step;
    for (int64_t i = 0; i < n; ++i) {
        float r = (step > 0.0f) ? nearbyintf(x[i] / step) : 0.0f;  /* default FE_TONEAREST */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
}

/* [W14] accumulation-precision example: add `n` copies of `term`, rounding
 * the running sum to the format after every addition; every `promote`
 * terms (0 = never) the rounded partial sum is added into an fp32 total
 * and the partial restarts from zero.  Returns the final sum. */
float orc_fp8_running_sum(int fmt, float term, int n, int promote, int* first_stall_step)
{
    float total = 0.0f, part = 0.0f;
    int cnt = 0;
    if (first_stall_step) *first_stall_step = -1;
    for (int i = 1; i <= n; ++i) {
        float next = (float)orc_decode(fmt, orc_encode(fmt, part + term));
        if (first_stall_step && *first_stall_step < 0 && promote == 0 && next == part) *first_stall_step = i - 1;
        part = next;
        if (promote > 0 && ++cnt == promote) {
            total += part;
            part = 0.0f;
            cnt = 0;
        }
    }
    return total + part;
}

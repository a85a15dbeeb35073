// quantize.cu -- amax, scale rules and the saturating FP8 cast on sm_103a.
//
// All of this is HBM-bound (2 B read + 1 B written per bf16 element, +1 B for
// a transposed copy), so the kernels are built around coalesced 128-bit
// loads, 64-bit code stores, an in-register amax (packed bf16 absolute
// values reduced with a 2-way unsigned max), warp shuffles and one atomic per
// CTA.  No shared-memory staging is needed: every scaling unit lives in the
// registers of one thread group.
//
// Arithmetic follows the pages' statement of the method:
//  * amax = max|x| ("Transformer Scaling", core vocabulary), taken on the
//    IEEE bit patterns of |x| so that a NaN propagates;
//  * current scale m = fmax / amax, s = amax / fmax, each one IEEE fp32
//    division ("Week 14", absmax bullet: the step comes from the current
//    block; "Transformer Scaling" worked example: the multiplier form);
//  * cast q = cvt.rn.satfinite(fp32(x) * m) ("Transformer Scaling" worked
//    example: a value past the range clips at 448);
//  * MX: one power-of-two scale per 32 values ("Week 14", absmax bullet),
//    the smallest 2^e with amax <= fmax * 2^e;
//  * delayed: m from the state, the tensor's amax max-combined into the
//    newest history slot; the end-of-step update takes the history max
//    ("Transformer Scaling", delayed scaling; the Transformer Engine
//    tutorial's DelayedScaling recipe).
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8sq {

template <int FMT>
struct Fmt;
template <>
struct Fmt<kE4M3> {
    static constexpr float fmax = 448.0f;
    static constexpr int emax = 8;
};
template <>
struct Fmt<kE5M2> {
    static constexpr float fmax = 57344.0f;
    static constexpr int emax = 15;
};

// ------------------------------------------------------------------ loads
__device__ __forceinline__ uint4 ld_nc_v4(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 8 consecutive input elements held in registers.
template <int DT>
struct Vec8;

template <>
struct Vec8<kBF16> {
    uint4 w;
    static constexpr int bytes = 16;
    __device__ __forceinline__ void load(const void* base, int64_t elem) { w = ld_nc_v4(static_cast<const uint16_t*>(base) + elem); }
    __device__ __forceinline__ void zero() { w = make_uint4(0, 0, 0, 0); }
    // fp32 bit pattern of max|x_i| (NaN-propagating: NaN bits sort above inf)
    __device__ __forceinline__ uint32_t absmax_bits() const
    {
        const uint32_t k = 0x7FFF7FFFu;
        uint32_t u = __vmaxu2(__vmaxu2(w.x & k, w.y & k), __vmaxu2(w.z & k, w.w & k));
        return max(u & 0xFFFFu, u >> 16) << 16;
    }
    __device__ __forceinline__ void get(float (&f)[8]) const
    {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(ws[i] << 16);
            f[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
        }
    }
};

template <>
struct Vec8<kF32> {
    uint4 a, b;
    static constexpr int bytes = 32;
    __device__ __forceinline__ void load(const void* base, int64_t elem)
    {
        const float* p = static_cast<const float*>(base) + elem;
        a = ld_nc_v4(p);
        b = ld_nc_v4(p + 4);
    }
    __device__ __forceinline__ void zero() { a = b = make_uint4(0, 0, 0, 0); }
    __device__ __forceinline__ uint32_t absmax_bits() const
    {
        const uint32_t k = 0x7FFFFFFFu;
        uint32_t m0 = max(max(a.x & k, a.y & k), max(a.z & k, a.w & k));
        uint32_t m1 = max(max(b.x & k, b.y & k), max(b.z & k, b.w & k));
        return max(m0, m1);
    }
    __device__ __forceinline__ void get(float (&f)[8]) const
    {
        f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
        f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
        f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
        f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
    }
};

// ------------------------------------------------------------------ scale rules
// current scaling: m = fmax/amax, s = amax/fmax; amax 0 or non-finite -> 1, 1
template <int FMT>
__device__ __forceinline__ void current_scale(uint32_t amax_bits, float& m, float& s)
{
    float a = __uint_as_float(amax_bits);
    if (amax_bits != 0u && amax_bits < 0x7F800000u) {
        m = __fdiv_rn(Fmt<FMT>::fmax, a);
        s = __fdiv_rn(a, Fmt<FMT>::fmax);
    } else {
        m = 1.0f;
        s = 1.0f;
    }
}

// MX: E8M0 code of the smallest 2^e with amax <= fmax * 2^e, and m = 2^-e
template <int FMT>
__device__ __forceinline__ uint32_t mx_scale(uint32_t amax_bits, float& m)
{
    if (amax_bits >= 0x7F800000u) { m = 1.0f; return 0xFFu; }
    if (amax_bits == 0u) { m = 1.0f; return 127u; }
    int E;
    uint32_t frac;
    uint32_t ef = amax_bits >> 23;
    if (ef == 0u) {                      // subnormal: normalise
        uint32_t mant = amax_bits & 0x7FFFFFu;
        int p = 31 - __clz(mant);        // leading one position, 0..22
        E = p - 149;
        frac = (mant << (23 - p)) & 0x7FFFFFu;
    } else {
        E = (int)ef - 127;
        frac = amax_bits & 0x7FFFFFu;
    }
    int e = E - Fmt<FMT>::emax + (frac > 0x600000u ? 1 : 0);   // 1.f > 1.75
    e = max(-127, min(127, e));
    m = (e <= 126) ? __uint_as_float((uint32_t)(127 - e) << 23) : __uint_as_float(0x00400000u);
    return (uint32_t)(e + 127);
}

// MX by the OCP floor rule: e = floor(log2 amax) - emax (can clip)
template <int FMT>
__device__ __forceinline__ uint32_t mx_scale_floor(uint32_t amax_bits, float& m)
{
    if (amax_bits >= 0x7F800000u) { m = 1.0f; return 0xFFu; }
    if (amax_bits == 0u) { m = 1.0f; return 127u; }
    uint32_t ef = amax_bits >> 23;
    const int E = (ef == 0u) ? (31 - __clz(amax_bits & 0x7FFFFFu)) - 149 : (int)ef - 127;
    int e = E - Fmt<FMT>::emax;
    e = max(-127, min(127, e));
    m = (e <= 126) ? __uint_as_float((uint32_t)(127 - e) << 23) : __uint_as_float(0x00400000u);
    return (uint32_t)(e + 127);
}

// cast 8 values with multiplier m; returns 8 codes packed little-endian
template <int FMT>
__device__ __forceinline__ uint2 cast8(const float (&f)[8], float m, uint32_t absbits, uint32_t& nsat)
{
    // absbits: fp32 bit pattern of max |f_i|.  rn(|x| m) is monotone in |x|
    // (m > 0), so no element saturates unless the scaled maximum does; the
    // elements are counted one by one only then, or when the chunk holds an
    // inf or NaN (whose bit pattern says nothing about the other elements).
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = __fmul_rn(f[i], m);
    if (absbits >= 0x7F800000u || __fmul_rn(__uint_as_float(absbits), m) > Fmt<FMT>::fmax) {
#pragma unroll
        for (int i = 0; i < 8; ++i) nsat += (fabsf(p[i]) > Fmt<FMT>::fmax) ? 1u : 0u;
    }
    uint32_t lo = cvt_fp8x2<FMT>(p[0], p[1]) | (cvt_fp8x2<FMT>(p[2], p[3]) << 16);
    uint32_t hi = cvt_fp8x2<FMT>(p[4], p[5]) | (cvt_fp8x2<FMT>(p[6], p[7]) << 16);
    return make_uint2(lo, hi);
}

__device__ __forceinline__ void atomic_max_bits(float* dst, uint32_t bits)
{
    // |x| bit patterns order like the values (NaN above inf); skip the atomic
    // when the stored value already covers ours.
    unsigned int* p = reinterpret_cast<unsigned int*>(dst);
    if (bits > *reinterpret_cast<volatile unsigned int*>(p)) atomicMax(p, bits);
}

__device__ __forceinline__ void add_sat(unsigned long long* sat, uint32_t n)
{
    n = __reduce_add_sync(0xFFFFFFFFu, n);
    if ((threadIdx.x & 31) == 0 && n) atomicAdd(sat, (unsigned long long)n);
}

// block-wide max of the fp32 bit patterns; result valid in every thread
template <int NWARPS>
__device__ __forceinline__ uint32_t block_max_bits(uint32_t v, uint32_t* red)
{
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t r = red[0];
#pragma unroll
    for (int i = 1; i < NWARPS; ++i) r = max(r, red[i]);
    return r;
}

// ================================================================== per-tensor
// Pass 1 of current per-tensor scaling (and fp8_amax TENSOR): grid-stride
// over 8-element chunks, 4 independent 128-bit loads in flight per thread.
constexpr int kFlatThreads = 256;
constexpr int kFlatUnroll = 4;
// 16-element groups per thread per pass of the row-unit kernels: two for
// 1x128 tiles, four for MX-32 blocks.  Measured on the GB300 (interleaved,
// L2 flushed): 1x128 at 16384 x 14336 110.6 -> 108.2-108.5 us with two
// against four; MX-32 with two was faster at 4096 x 4096 but slower at
// 8192 x 8192 (34.8 against 34.1 us); eight was slower at every size.
template <int UNIT>
__host__ __device__ constexpr int row_unroll()
{
    return UNIT == 32 ? 4 : 2;
}

// amax of one tensor over blocks [bid, bid + nblk, ...) of a grid-stride loop
template <int DT>
__device__ __forceinline__ void amax_tensor_body(const void* __restrict__ x, int64_t n, float* __restrict__ amax_out,
                                                 int64_t bid, int64_t nblk, uint32_t* red)
{
    const int64_t nch = n / 8;
    uint32_t mx = 0;
    const int64_t stride = nblk * kFlatThreads * kFlatUnroll;
    for (int64_t c0 = bid * kFlatThreads * kFlatUnroll; c0 < nch; c0 += stride) {
        Vec8<DT> v[kFlatUnroll];
#pragma unroll
        for (int u = 0; u < kFlatUnroll; ++u) {
            int64_t c = c0 + u * kFlatThreads + threadIdx.x;
            if (c < nch) v[u].load(x, c * 8); else v[u].zero();
        }
#pragma unroll
        for (int u = 0; u < kFlatUnroll; ++u) mx = max(mx, v[u].absmax_bits());
    }
    // ragged tail (n % 8 elements): the job's first block, first threads
    if (bid == 0 && threadIdx.x < (n & 7)) {
        int64_t i = nch * 8 + threadIdx.x;
        uint32_t b = (DT == kBF16) ? ((uint32_t)(static_cast<const uint16_t*>(x)[i] & 0x7FFFu) << 16)
                                   : (__float_as_uint(static_cast<const float*>(x)[i]) & 0x7FFFFFFFu);
        mx = max(mx, b);
    }
    uint32_t r = block_max_bits<kFlatThreads / 32>(mx, red);
    if (threadIdx.x == 0) atomic_max_bits(amax_out, r);
}

template <int DT>
__global__ void __launch_bounds__(kFlatThreads) k_amax_tensor(const void* __restrict__ x, int64_t n,
                                                              float* __restrict__ amax_out)
{
    pdl_enter();
    __shared__ uint32_t red[kFlatThreads / 32];
    amax_tensor_body<DT>(x, n, amax_out, blockIdx.x, gridDim.x, red);
}

// The amaxes of two tensors in one launch: blocks [0, blocks_a) reduce a,
// the rest reduce b (a linear layer's x and W under current scaling).
struct AmaxJob {
    const void* x;
    int64_t n;
    float* amax;
};
template <int DT>
__global__ void __launch_bounds__(kFlatThreads) k_amax_tensor2(AmaxJob a, AmaxJob b, int blocks_a)
{
    pdl_enter();
    __shared__ uint32_t red[kFlatThreads / 32];
    if ((int)blockIdx.x < blocks_a)
        amax_tensor_body<DT>(a.x, a.n, a.amax, blockIdx.x, blocks_a, red);
    else
        amax_tensor_body<DT>(b.x, b.n, b.amax, blockIdx.x - blocks_a, gridDim.x - blocks_a, red);
}

// Cast pass of per-tensor scaling without a transposed copy, over blocks
// [bid, bid + nblk, ...) of a grid-stride loop.
//   DELAYED: m = state[H]; the tensor's amax is max-combined into state[0]
//            (and into amax_out if given).
//   current: m, s from *amax_in; the job's block 0 writes s.
template <int DT, int FMT, bool DELAYED>
__device__ __forceinline__ void cast_tensor_body(const void* __restrict__ x, int64_t n, uint8_t* __restrict__ q,
                                                 float* state, int H, const float* amax_in, float* s_out,
                                                 float* amax_out, unsigned long long* sat, int64_t bid,
                                                 int64_t nblk, uint32_t* red)
{
    float m, s;
    if (DELAYED) {
        m = state[H];
        s = 0.0f;
        // the dequantisation scale this cast uses (the state's s is updated
        // only at the end of the step)
        if (bid == 0 && threadIdx.x == 0 && s_out) *s_out = state[H + 1];
    } else {
        current_scale<FMT>(__float_as_uint(*amax_in), m, s);
        if (bid == 0 && threadIdx.x == 0 && s_out) *s_out = s;
    }
    const int64_t nch = n / 8;
    uint32_t mx = 0, nsat = 0;
    const int64_t stride = nblk * kFlatThreads * kFlatUnroll;
    for (int64_t c0 = bid * kFlatThreads * kFlatUnroll; c0 < nch; c0 += stride) {
        Vec8<DT> v[kFlatUnroll];
#pragma unroll
        for (int u = 0; u < kFlatUnroll; ++u) {
            int64_t c = c0 + u * kFlatThreads + threadIdx.x;
            if (c < nch) v[u].load(x, c * 8); else v[u].zero();
        }
#pragma unroll
        for (int u = 0; u < kFlatUnroll; ++u) {
            int64_t c = c0 + u * kFlatThreads + threadIdx.x;
            const uint32_t ab = v[u].absmax_bits();
            if (DELAYED) mx = max(mx, ab);
            float f[8];
            v[u].get(f);
            uint2 codes = cast8<FMT>(f, m, ab, nsat);
            if (c < nch) *reinterpret_cast<uint2*>(q + c * 8) = codes;
        }
    }
    if (bid == 0 && threadIdx.x < (n & 7)) {
        int64_t i = nch * 8 + threadIdx.x;
        float f = (DT == kBF16) ? __uint_as_float((uint32_t)static_cast<const uint16_t*>(x)[i] << 16)
                                : static_cast<const float*>(x)[i];
        float p = __fmul_rn(f, m);
        nsat += fabsf(p) > Fmt<FMT>::fmax ? 1u : 0u;
        q[i] = (uint8_t)(cvt_fp8x2<FMT>(p, 0.0f) & 0xFFu);
        mx = max(mx, __float_as_uint(f) & 0x7FFFFFFFu);
    }
    if (sat) add_sat(sat, nsat);
    if (DELAYED) {
        uint32_t r = block_max_bits<kFlatThreads / 32>(mx, red);
        if (threadIdx.x == 0) {
            atomic_max_bits(&state[0], r);
            if (amax_out) atomic_max_bits(amax_out, r);
        }
    }
}

template <int DT, int FMT, bool DELAYED>
__global__ void __launch_bounds__(kFlatThreads) k_cast_tensor(const void* __restrict__ x, int64_t n,
                                                              uint8_t* __restrict__ q, float* state, int H,
                                                              const float* amax_in, float* s_out,
                                                              float* amax_out, unsigned long long* sat)
{
    pdl_enter();
    __shared__ uint32_t red[kFlatThreads / 32];
    cast_tensor_body<DT, FMT, DELAYED>(x, n, q, state, H, amax_in, s_out, amax_out, sat, blockIdx.x, gridDim.x, red);
}

// Two per-tensor casts without transposed copies in one launch (a linear
// layer's x and W): blocks [0, blocks_a) cast a, the rest cast b.
struct FlatCastJob {
    const void* x;
    int64_t n;
    uint8_t* q;
    float* state;
    const float* amax_in;
    float* s_out;
    float* amax_out;
};
template <int DT, int FMT, bool DELAYED>
__global__ void __launch_bounds__(kFlatThreads) k_cast_tensor2(FlatCastJob a, FlatCastJob b, int blocks_a, int H,
                                                               unsigned long long* sat)
{
    pdl_enter();
    __shared__ uint32_t red[kFlatThreads / 32];
    if ((int)blockIdx.x < blocks_a)
        cast_tensor_body<DT, FMT, DELAYED>(a.x, a.n, a.q, a.state, H, a.amax_in, a.s_out, a.amax_out, sat, blockIdx.x,
                                           blocks_a, red);
    else
        cast_tensor_body<DT, FMT, DELAYED>(b.x, b.n, b.q, b.state, H, b.amax_in, b.s_out, b.amax_out, sat,
                                           blockIdx.x - blocks_a, gridDim.x - blocks_a, red);
}

// 8x8 byte transpose: in[i] holds row i (bytes = columns 0..7); out[j] holds
// column j (bytes = rows 0..7).  Four 4x4 transposes with byte permutes.
__device__ __forceinline__ void transpose4x4(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                             uint32_t& c0, uint32_t& c1, uint32_t& c2, uint32_t& c3)
{
    uint32_t t0 = __byte_perm(w0, w1, 0x5140);  // w0.b0 w1.b0 w0.b1 w1.b1
    uint32_t t1 = __byte_perm(w2, w3, 0x5140);
    uint32_t t2 = __byte_perm(w0, w1, 0x7362);  // w0.b2 w1.b2 w0.b3 w1.b3
    uint32_t t3 = __byte_perm(w2, w3, 0x7362);
    c0 = __byte_perm(t0, t1, 0x5410);
    c1 = __byte_perm(t0, t1, 0x7632);
    c2 = __byte_perm(t2, t3, 0x5410);
    c3 = __byte_perm(t2, t3, 0x7632);
}
__device__ __forceinline__ void transpose8x8(const uint2 (&in)[8], uint2 (&out)[8])
{
    uint32_t a[4], b[4], c[4], d[4];
    // rows 0-3 cols 0-3 -> cols 0-3 rows 0-3 (low words of out[0..3])
    transpose4x4(in[0].x, in[1].x, in[2].x, in[3].x, a[0], a[1], a[2], a[3]);
    // rows 4-7 cols 0-3 -> high words of out[0..3]
    transpose4x4(in[4].x, in[5].x, in[6].x, in[7].x, b[0], b[1], b[2], b[3]);
    // rows 0-3 cols 4-7 -> low words of out[4..7]
    transpose4x4(in[0].y, in[1].y, in[2].y, in[3].y, c[0], c[1], c[2], c[3]);
    transpose4x4(in[4].y, in[5].y, in[6].y, in[7].y, d[0], d[1], d[2], d[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        out[j] = make_uint2(a[j], b[j]);
        out[4 + j] = make_uint2(c[j], d[j]);
    }
}

// Row-wise LayerNorm folded into the cast (LN = true): x is replaced by
// y = (x - mu[r]) * rstd[r] * gamma[c] + beta[c] before the multiplier, the
// amax is taken over y, and the bf16 LayerNorm output never leaves the SM.
struct LnParams {
    const float* mu = nullptr;
    const float* rstd = nullptr;
    const float* gamma = nullptr;
    const float* beta = nullptr;
};

// Per-tensor cast with a transposed copy: one 128x128 tile per 256-thread
// CTA, each thread an 8x8 sub-block (8 rows x one 128-bit load), all loads
// in flight at once.  Warp layout: 4 column groups x 8 row groups, so every
// load instruction reads 64-byte row segments and every code store writes
// whole 32-byte sectors, in both q and qT.  Requires rows, cols % 8 == 0
// (% 16 for the LayerNorm mode).  Three CTAs (24 warps) per SM keep enough
// loads in flight: measured on the GB300 at 16384 x 14336 (delayed E5M2,
// identical codes), 144.2 us = 6.5 TB/s against 168.2 us for a persistent
// TMA-fed ring with 8 consumer warps per SM.
// One 128 x 128 tile (tile_c, tile_r) of the cast; red: 8 words of shared memory.
template <int DT, int FMT, bool DELAYED, bool LN>
__device__ __forceinline__ void cast_tile_T(const void* __restrict__ x, int64_t R, int64_t C,
                                            uint8_t* __restrict__ q, uint8_t* __restrict__ qT, float* state, int H,
                                            const float* amax_in, float* s_out, float* amax_out,
                                            unsigned long long* sat, const LnParams& ln, int64_t tile_c,
                                            int64_t tile_r, uint32_t* red)
{
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int64_t c0 = tile_c * 128 + ((w & 3) * 4 + (l & 3)) * 8;
    const int64_t r0 = tile_r * 128 + ((w >> 2) * 8 + (l >> 2)) * 8;
    float m, s;
    if (DELAYED) {
        m = state[H];
        s = 0.0f;
        // the dequantisation scale this cast uses (the state's s is updated
        // only at the end of the step)
        if (tile_c == 0 && tile_r == 0 && threadIdx.x == 0 && s_out) *s_out = state[H + 1];
    } else {
        current_scale<FMT>(__float_as_uint(*amax_in), m, s);
        if (tile_c == 0 && tile_r == 0 && threadIdx.x == 0 && s_out) *s_out = s;
    }
    const bool ok = (r0 < R) && (c0 < C);    // rows, cols % 16 == 0: whole 8 x 8 groups
    Vec8<DT> v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (ok) v[i].load(x, (r0 + i) * C + c0); else v[i].zero();
    }
    float g[8], be[8], mu[8], rs[8];
    if (LN) {
        // this thread's 8 columns of gamma / beta and 8 rows of mean / rstd as
        // 128-bit loads (16-byte aligned buffers)
        const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        const float4* g4 = reinterpret_cast<const float4*>(ln.gamma + c0);
        const float4* b4 = reinterpret_cast<const float4*>(ln.beta + c0);
        const float4* m4 = reinterpret_cast<const float4*>(ln.mu + r0);
        const float4* r4 = reinterpret_cast<const float4*>(ln.rstd + r0);
        const float4 ga = ok ? __ldg(g4) : z4, gb = ok ? __ldg(g4 + 1) : z4;
        const float4 ba = (ok && ln.beta) ? __ldg(b4) : z4, bb = (ok && ln.beta) ? __ldg(b4 + 1) : z4;
        const float4 ma = ok ? __ldg(m4) : z4, mb = ok ? __ldg(m4 + 1) : z4;
        const float4 ra = ok ? __ldg(r4) : z4, rb = ok ? __ldg(r4 + 1) : z4;
        g[0] = ga.x; g[1] = ga.y; g[2] = ga.z; g[3] = ga.w; g[4] = gb.x; g[5] = gb.y; g[6] = gb.z; g[7] = gb.w;
        be[0] = ba.x; be[1] = ba.y; be[2] = ba.z; be[3] = ba.w; be[4] = bb.x; be[5] = bb.y; be[6] = bb.z; be[7] = bb.w;
        mu[0] = ma.x; mu[1] = ma.y; mu[2] = ma.z; mu[3] = ma.w; mu[4] = mb.x; mu[5] = mb.y; mu[6] = mb.z; mu[7] = mb.w;
        rs[0] = ra.x; rs[1] = ra.y; rs[2] = ra.z; rs[3] = ra.w; rs[4] = rb.x; rs[5] = rb.y; rs[6] = rb.z; rs[7] = rb.w;
    }
    uint32_t mx = 0, nsat = 0;
    uint2 rows[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float f[8];
        v[i].get(f);
        uint32_t ab;
        if (LN) {
            ab = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                f[j] = __fmaf_rn(__fmul_rn(__fsub_rn(f[j], mu[i]), rs[i]), g[j], be[j]);
                ab = max(ab, __float_as_uint(f[j]) & 0x7FFFFFFFu);
            }
        } else {
            ab = v[i].absmax_bits();
        }
        if (DELAYED) mx = max(mx, ab);
        rows[i] = cast8<FMT>(f, m, ab, nsat);
    }
    if (ok) {
#pragma unroll
        for (int i = 0; i < 8; ++i) *reinterpret_cast<uint2*>(q + (r0 + i) * C + c0) = rows[i];
        if (qT) {
            uint2 cols[8];
            transpose8x8(rows, cols);
#pragma unroll
            for (int j = 0; j < 8; ++j) *reinterpret_cast<uint2*>(qT + (c0 + j) * R + r0) = cols[j];
        }
    } else {
        nsat = 0;
    }
    if (sat) add_sat(sat, nsat);
    if (DELAYED) {
        uint32_t r = block_max_bits<8>(mx, red);
        if (threadIdx.x == 0) {
            atomic_max_bits(&state[0], r);
            if (amax_out) atomic_max_bits(amax_out, r);
        }
    }
}

template <int DT, int FMT, bool DELAYED, bool LN = false>
__global__ void __launch_bounds__(256) k_cast_tensor_T(const void* __restrict__ x, int64_t R, int64_t C,
                                                       uint8_t* __restrict__ q, uint8_t* __restrict__ qT,
                                                       float* state, int H, const float* amax_in,
                                                       float* s_out, float* amax_out,
                                                       unsigned long long* sat, LnParams ln)
{
    pdl_enter();
    __shared__ uint32_t red[8];
    cast_tile_T<DT, FMT, DELAYED, LN>(x, R, C, q, qT, state, H, amax_in, s_out, amax_out, sat, ln, blockIdx.x,
                                      blockIdx.y, red);
}

// Two per-tensor casts of the same kind in one launch (a linear layer's x
// and W): blocks [0, tiles_a) take a's tiles in row-major tile order, the
// rest b's.  At small layers each cast alone is one partial wave; one launch
// saves a kernel's prologue and tail.
struct CastJob {
    const void* x;
    int64_t R, C;
    uint8_t* q;
    uint8_t* qT;
    float* state;          // delayed
    const float* amax_in;  // current
    float* s_out;
    float* amax_out;
};
template <int DT, int FMT, bool DELAYED>
__global__ void __launch_bounds__(256) k_cast_tensor_T2(CastJob a, CastJob b, int64_t tiles_a, int H,
                                                        unsigned long long* sat)
{
    pdl_enter();
    __shared__ uint32_t red[8];
    // field by field, so the parameters are read in place
    const bool first = (int64_t)blockIdx.x < tiles_a;
    const int64_t t = first ? (int64_t)blockIdx.x : (int64_t)blockIdx.x - tiles_a;
    const int64_t R = first ? a.R : b.R, C = first ? a.C : b.C;
    const int64_t tiles_c = (C + 127) / 128;
    cast_tile_T<DT, FMT, DELAYED, false>(first ? a.x : b.x, R, C, first ? a.q : b.q, first ? a.qT : b.qT,
                                         first ? a.state : b.state, H, first ? a.amax_in : b.amax_in,
                                         first ? a.s_out : b.s_out, first ? a.amax_out : b.amax_out, sat, LnParams(),
                                         t % tiles_c, t / tiles_c, red);
}

// MX scales: the canonical layout is u8 [rows][cols/32]; the tiled layout
// (TILED = true) is the one the block-scaled GEMM copies straight into tensor
// memory: 512-byte chunks of 128 rows x 4 consecutive 32-blocks, chunk
// (r/128, t/4) at ((r/128) * (cols/128) + t/4) * 512, inside it
// (r % 32) * 16 + ((r / 32) % 4) * 4 + t % 4.
__device__ __forceinline__ int64_t mx_tiled_offset(int64_t r, int64_t t, int64_t cols)
{
    return ((r >> 7) * (cols >> 7) + (t >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (t & 3);
}

// ================================================================== column units
// Column tiles of 128 rows (UNIT = 128, scales f32 [R/128][C]) and column MX
// blocks of 32 rows (UNIT = 32, E8M0 scales in the tiled layout of the
// transposed matrix [C][R]): the operands of products that contract over
// the rows of x.  One 128 x 128 tile per 256-thread CTA with the lane map of
// k_cast_tensor_T: thread (w, l) holds rows r0..r0+7 x columns c0..c0+7,
// c0 = ((w & 3) * 4 + (l & 3)) * 8 and r0 = ((w >> 2) * 8 + (l >> 2)) * 8.
// A column's 32 rows are four row groups of one warp (a shuffle over lanes
// l ^ 4, l ^ 8); its 128 rows are the eight row groups of warps w and w + 4
// (shuffles, then one exchange through shared memory), after which thread
// c < 128 computes column c's scale once for the CTA and writes it.  Writes
// the transposed codes qT and, when q is given, the codes in x's layout.
// ROWQ: the same pass also quantises the rows in their own units (UNIT = 128:
// 1x128 tiles, f32 scales [R][C/128] into rscales; UNIT = 32: MX-32 blocks,
// E8M0 codes in the tiled layout of x [R][C]) and writes q with those row
// codes: both operands of a fine-grained linear's products from one read of
// x.  A row's 32 columns are four lanes of one warp; its 128 columns are four
// warps (shuffles over l ^ 1, l ^ 2, then shared memory), and thread
// 128 + r computes row r's 1x128 scale.  For MX-32 units the four lanes that
// share a unit's maxima each compute two of its eight E8M0 scales and pass
// the multipliers on by shuffles (16384 x 14336: column blocks 133 -> 117 us,
// rows + columns 226 -> 167 us, against every lane computing all sixteen).
// The CTA's loads are all issued at its start and nothing is loaded while it
// reduces and casts, so the SM's memory pipe needs several CTAs: four per SM
// (64 registers; 128-row column tiles at three, 80 registers, took 131.5
// against 117.3 us), except MX-32 rows + columns, three (80 registers; at
// four they spill).
// POW2 (UNIT = 128): power-of-two tiles by the MX rule; each tile's E8M0
// code fills the four 32-blocks it covers in the tiled layouts (rows: of x,
// columns: of x^T), the layouts the block-scaled GEMM reads.
template <int FMT, int UNIT, bool ROWQ = false, bool POW2 = false>
__global__ void __launch_bounds__(256, UNIT == 32 && ROWQ ? 3 : 4) k_quant_col_block(const void* __restrict__ x, int64_t R, int64_t C,
                                                         uint8_t* __restrict__ q, uint8_t* __restrict__ qT,
                                                         void* scales, void* rscales, unsigned long long* sat)
{
    pdl_enter();
    __shared__ uint32_t colred[2][128];              // column maxima of the two 64-row halves
    __shared__ __align__(16) float colm[128];        // column multipliers (128-row tiles)
    __shared__ __align__(16) uint8_t colflag[128];   // column may saturate (128-row tiles)
    __shared__ uint32_t rowred[ROWQ && UNIT == 128 ? 4 : 1][128];   // row maxima of the four 32-column warps
    __shared__ __align__(16) float rowm[ROWQ && UNIT == 128 ? 128 : 4];
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int cl = ((w & 3) * 4 + (l & 3)) * 8;      // columns of this thread within the tile
    const int rl = ((w >> 2) * 8 + (l >> 2)) * 8;    // rows of this thread within the tile
    const int64_t tr0 = (int64_t)blockIdx.y * 128, tc0 = (int64_t)blockIdx.x * 128;
    const int64_t r0 = tr0 + rl, c0 = tc0 + cl;
    const bool ok = r0 < R && c0 < C;                // rows % 128 == 0, cols % 16 == 0
    Vec8<kBF16> v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (ok) v[i].load(x, (r0 + i) * C + c0); else v[i].zero();
    }
    // column maxima of the |x| bit patterns, kept packed: word k holds columns
    // 2k (low half) and 2k + 1 (high half) as bf16 patterns (NaN sorts above
    // inf, so it propagates).  This thread's 8 rows, then the row groups of
    // the unit (lanes that share l & 3).  Packing keeps the registers low
    // enough for three CTAs per SM.
    uint32_t pm[4] = {0u, 0u, 0u, 0u};
    const uint32_t k7 = 0x7FFF7FFFu;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        pm[0] = __vmaxu2(pm[0], v[i].w.x & k7);
        pm[1] = __vmaxu2(pm[1], v[i].w.y & k7);
        pm[2] = __vmaxu2(pm[2], v[i].w.z & k7);
        pm[3] = __vmaxu2(pm[3], v[i].w.w & k7);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        pm[k] = __vmaxu2(pm[k], __shfl_xor_sync(0xFFFFFFFFu, pm[k], 4));
        pm[k] = __vmaxu2(pm[k], __shfl_xor_sync(0xFFFFFFFFu, pm[k], 8));
        if (UNIT == 128) pm[k] = __vmaxu2(pm[k], __shfl_xor_sync(0xFFFFFFFFu, pm[k], 16));
    }
    uint32_t cm[8];                                  // fp32 bit patterns of the column maxima
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        cm[2 * k] = pm[k] << 16;
        cm[2 * k + 1] = pm[k] & 0xFFFF0000u;
    }
    // row maxima (ROWQ): this thread's 8 columns of each of its rows, then the
    // four lanes of the warp that cover 32 columns (l ^ 1, l ^ 2)
    uint32_t rmax[8];
    if (ROWQ) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t a = v[i].absmax_bits();
            a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
            a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
            rmax[i] = a;
        }
    }
    float m[8], rm[8];
    bool maysat = false;      // some column's scaled maximum may exceed fmax
    if (UNIT == 128) {
        if ((l >> 2) == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) colred[w >> 2][cl + j] = cm[j];
        }
        if (ROWQ && (l & 3) == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) rowred[w & 3][rl + i] = rmax[i];
        }
        __syncthreads();
        if (threadIdx.x < 128) {
            const int c = threadIdx.x;
            const uint32_t a = max(colred[0][c], colred[1][c]);
            float mm, ss;
            if (POW2) {
                // power-of-two column tile: its E8M0 code fills the four
                // 32-row blocks it covers in the tiled layout of x^T
                const uint32_t code = mx_scale<FMT>(a, mm);
                if (tc0 + c < C) {
                    uint8_t* e = static_cast<uint8_t*>(scales);
#pragma unroll
                    for (int k = 0; k < 4; ++k) e[mx_tiled_offset(tc0 + c, tr0 / 32 + k, R)] = (uint8_t)code;
                }
            } else {
                current_scale<FMT>(a, mm, ss);
                if (tc0 + c < C) static_cast<float*>(scales)[(tr0 / 128) * C + tc0 + c] = ss;
            }
            colm[c] = mm;
            colflag[c] = (a >= 0x7F800000u || __fmul_rn(__uint_as_float(a), mm) > Fmt<FMT>::fmax) ? 1 : 0;
        } else if (ROWQ) {
            const int r = threadIdx.x - 128;
            const uint32_t a = max(max(rowred[0][r], rowred[1][r]), max(rowred[2][r], rowred[3][r]));
            float mm, ss;
            if (POW2) {
                // power-of-two 1x128 tile: its code fills the four 32-column
                // blocks it covers in the tiled layout of x
                const uint32_t code = mx_scale<FMT>(a, mm);
                if (tr0 + r < R) {
                    uint8_t* e = static_cast<uint8_t*>(rscales);
#pragma unroll
                    for (int k = 0; k < 4; ++k) e[mx_tiled_offset(tr0 + r, tc0 / 32 + k, C)] = (uint8_t)code;
                }
            } else {
                current_scale<FMT>(a, mm, ss);
                if (tr0 + r < R) static_cast<float*>(rscales)[(tr0 + r) * (C / 128) + blockIdx.x] = ss;
            }
            rowm[r] = mm;
        }
        __syncthreads();
        const float4 m0 = *reinterpret_cast<const float4*>(&colm[cl]);
        const float4 m1 = *reinterpret_cast<const float4*>(&colm[cl + 4]);
        m[0] = m0.x; m[1] = m0.y; m[2] = m0.z; m[3] = m0.w;
        m[4] = m1.x; m[5] = m1.y; m[6] = m1.z; m[7] = m1.w;
        const uint2 fl = *reinterpret_cast<const uint2*>(&colflag[cl]);   // the 8 columns' flags
        maysat = (fl.x | fl.y) != 0u;
    } else {
        // The four lanes that share a unit's maxima split its scale work:
        // lane g of the column group (l bits 2-3) takes columns 2g, 2g + 1,
        // lane h of the row group (l bits 0-1) rows 2h, 2h + 1; the
        // multipliers reach the other lanes by shuffles, and each lane stores
        // its own two E8M0 codes at once.
        const int g = (l >> 2) & 3, h = l & 3;
        const uint32_t ca = g == 0 ? cm[0] : g == 1 ? cm[2] : g == 2 ? cm[4] : cm[6];
        const uint32_t cb = g == 0 ? cm[1] : g == 1 ? cm[3] : g == 2 ? cm[5] : cm[7];
        float ma, mb;
        const uint32_t ka = mx_scale<FMT>(ca, ma), kb = mx_scale<FMT>(cb, mb);
        int flag = (ca >= 0x7F800000u || __fmul_rn(__uint_as_float(ca), ma) > Fmt<FMT>::fmax ||
                    cb >= 0x7F800000u || __fmul_rn(__uint_as_float(cb), mb) > Fmt<FMT>::fmax) ? 1 : 0;
        flag |= __shfl_xor_sync(0xFFFFFFFFu, flag, 4);
        flag |= __shfl_xor_sync(0xFFFFFFFFu, flag, 8);
        maysat = flag != 0;
        const int cbase = l & ~12;
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            m[j] = __shfl_sync(0xFFFFFFFFu, ma, cbase | ((j >> 1) << 2));
            m[j + 1] = __shfl_sync(0xFFFFFFFFu, mb, cbase | ((j >> 1) << 2));
        }
        if (ok) {
            uint8_t* e = static_cast<uint8_t*>(scales);
            e[mx_tiled_offset(c0 + 2 * g, r0 / 32, R)] = (uint8_t)ka;
            e[mx_tiled_offset(c0 + 2 * g + 1, r0 / 32, R)] = (uint8_t)kb;
        }
        if (ROWQ) {
            const uint32_t ra = h == 0 ? rmax[0] : h == 1 ? rmax[2] : h == 2 ? rmax[4] : rmax[6];
            const uint32_t rb = h == 0 ? rmax[1] : h == 1 ? rmax[3] : h == 2 ? rmax[5] : rmax[7];
            float rma, rmb;
            const uint32_t qa = mx_scale<FMT>(ra, rma), qb = mx_scale<FMT>(rb, rmb);
            const int rbase = l & ~3;
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                rm[i] = __shfl_sync(0xFFFFFFFFu, rma, rbase | (i >> 1));
                rm[i + 1] = __shfl_sync(0xFFFFFFFFu, rmb, rbase | (i >> 1));
            }
            if (ok) {
                uint8_t* e = static_cast<uint8_t*>(rscales);
                e[mx_tiled_offset(r0 + 2 * h, c0 / 32, C)] = (uint8_t)qa;
                e[mx_tiled_offset(r0 + 2 * h + 1, c0 / 32, C)] = (uint8_t)qb;
            }
        }
    }
    uint2 rows[8];
    uint32_t nsat = 0, nsat_r = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float f[8], p[8];
        v[i].get(f);
#pragma unroll
        for (int j = 0; j < 8; ++j) p[j] = __fmul_rn(f[j], m[j]);
        if (maysat) {
#pragma unroll
            for (int j = 0; j < 8; ++j) nsat += (fabsf(p[j]) > Fmt<FMT>::fmax) ? 1u : 0u;
        }
        rows[i].x = cvt_fp8x2<FMT>(p[0], p[1]) | (cvt_fp8x2<FMT>(p[2], p[3]) << 16);
        rows[i].y = cvt_fp8x2<FMT>(p[4], p[5]) | (cvt_fp8x2<FMT>(p[6], p[7]) << 16);
        if (ROWQ && ok) {
            // the row-unit codes of this row go to q (their saturations are
            // counted separately: sat counts the column-unit pass); 1x128
            // tiles read the row's multiplier from shared memory row by row,
            // which keeps the kernel within three CTAs' registers
            const float rmi = UNIT == 128 ? rowm[rl + i] : rm[i];
            *reinterpret_cast<uint2*>(q + (r0 + i) * C + c0) = cast8<FMT>(f, rmi, v[i].absmax_bits(), nsat_r);
        }
    }
    (void)nsat_r;
    if (ok) {
        if (q && !ROWQ) {
#pragma unroll
            for (int i = 0; i < 8; ++i) *reinterpret_cast<uint2*>(q + (r0 + i) * C + c0) = rows[i];
        }
        uint2 cols[8];
        transpose8x8(rows, cols);
#pragma unroll
        for (int j = 0; j < 8; ++j) *reinterpret_cast<uint2*>(qT + (c0 + j) * R + r0) = cols[j];
    } else {
        nsat = 0;
    }
    if (sat) add_sat(sat, nsat);
}

// LayerNorm statistics: mean = sum(x) / K and var = sum((x - mean)^2) / K in
// fp32, rstd = 1 / sqrt(var + eps) with IEEE division and square root.  The
// reduction order is a function of the row width alone, so the statistics
// (and hence the codes) do not depend on whether the one-pass or the
// two-pass path produced them.  Rows of up to 4096 elements: one warp per
// row (k_ln_warp).  Longer rows (two passes only): a 256-thread CTA takes
// LN_RB rows at a time, thread t owns the 8-element chunks t, t + 256, ...
// of every row and sums them in that order (each chunk as a tree of (even,
// odd) element pairs; the pair's two partials added last), then the warp
// reduction of warp_sum4, then the eight warps' partials in a fixed tree;
// one lane per row divides, and broadcasts the result.
constexpr int LN_RB = 4;         // rows per CTA iteration of the long-row kernel

// The arithmetic below works on (even, odd) element pairs with the packed
// fp32x2 instructions; each lane of a pair is an IEEE round-to-nearest fp32
// operation, so the pairing changes only how many instructions run.
__device__ __forceinline__ void bf16x8_pairs(const uint4& w, float2 (&p)[4])
{
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) p[k] = make_float2(__uint_as_float(ws[k] << 16), __uint_as_float(ws[k] & 0xFFFF0000u));
}
// acc + the chunk's sum, as (even, odd) partials: ((p0 + p1) + (p2 + p3))
__device__ __forceinline__ float2 ln_sum8(const float2 (&p)[4], float2 acc)
{
    return __fadd2_rn(acc, __fadd2_rn(__fadd2_rn(p[0], p[1]), __fadd2_rn(p[2], p[3])));
}
// acc + the chunk's squared deviations from the mean (nm = -mean), in order
__device__ __forceinline__ float2 ln_sq8(const float2 (&p)[4], float2 nm, float2 acc)
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 d = __fadd2_rn(p[k], nm);
        acc = __ffma2_rn(d, d, acc);
    }
    return acc;
}
// (even, odd) bf16 elements of w, each widened exactly and added to its half
// of c with one fp32 rounding (the mixed-precision add): the value of
// widening first and then adding, in one instruction per element.
__device__ __forceinline__ float2 bf16x2_add(uint32_t w, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %4;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "r"(w), "f"(c.x), "f"(c.y));
    return d;
}
// The chunk's elements minus the mean (nm = -mean), as (even, odd) pairs.
__device__ __forceinline__ void ln_dev8(const uint4& w, float2 nm, float2 (&d)[4])
{
    d[0] = bf16x2_add(w.x, nm);
    d[1] = bf16x2_add(w.y, nm);
    d[2] = bf16x2_add(w.z, nm);
    d[3] = bf16x2_add(w.w, nm);
}
// NaN-propagating max of a and |b| (|x| orders like its fp32 bit pattern,
// and every NaN an fp32 operation returns is the canonical 0x7FFFFFFF, the
// largest |x| pattern: the same result as the integer max of the patterns)
__device__ __forceinline__ float max_abs_nan(float a, float b)
{
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(fabsf(b)));
    return d;
}
// The LayerNorm of a chunk, y = (x - mean) rstd gamma + beta, its |y| max
// into amax, and its codes under the multiplier m (the arithmetic of cast8).
// d: the chunk's deviations from the mean (x - mean, rounded once).
template <int FMT>
__device__ __forceinline__ uint2 ln_cast8(const float2 (&d)[4], float2 rs, const float2 (&g)[4],
                                          const float2 (&be)[4], float m, float& amax, uint32_t& nsat)
{
    float2 y[4];
    float a = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        y[k] = __ffma2_rn(__fmul2_rn(d[k], rs), g[k], be[k]);
        a = max_abs_nan(max_abs_nan(a, y[k].x), y[k].y);
    }
    amax = max_abs_nan(amax, a);
    const float2 m2 = make_float2(m, m);
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = __fmul2_rn(y[k], m2);
    if (__float_as_uint(a) >= 0x7F800000u || __fmul_rn(a, m) > Fmt<FMT>::fmax) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            nsat += (fabsf(y[k].x) > Fmt<FMT>::fmax ? 1u : 0u) + (fabsf(y[k].y) > Fmt<FMT>::fmax ? 1u : 0u);
    }
    return make_uint2(cvt_fp8x2<FMT>(y[0].x, y[0].y) | (cvt_fp8x2<FMT>(y[1].x, y[1].y) << 16),
                      cvt_fp8x2<FMT>(y[2].x, y[2].y) | (cvt_fp8x2<FMT>(y[3].x, y[3].y) << 16));
}

// The warp sums of LN_RB = 4 per-lane values (one per row) in six shuffles:
// a reduce-scatter over lane bits 4 and 3 (lanes 0-15 keep rows 0-1, lanes
// 8-15 and 24-31 then keep the odd row), then a butterfly over bits 2-0.
// Lane l returns the sum of row l >> 3, the same value in all eight lanes of
// its group.
__device__ __forceinline__ float warp_sum4(const float (&s)[LN_RB], int lane)
{
    const bool b4 = lane & 16, b3 = lane & 8;
    const float u0 = __fadd_rn(b4 ? s[2] : s[0], __shfl_xor_sync(0xFFFFFFFFu, b4 ? s[0] : s[2], 16));
    const float u1 = __fadd_rn(b4 ? s[3] : s[1], __shfl_xor_sync(0xFFFFFFFFu, b4 ? s[1] : s[3], 16));
    float v = __fadd_rn(b3 ? u1 : u0, __shfl_xor_sync(0xFFFFFFFFu, b3 ? u0 : u1, 8));
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
// The eight warps' partials of row j, in a fixed tree.
__device__ __forceinline__ float ln_tree8(const float (*p)[LN_RB], int j)
{
    return __fadd_rn(__fadd_rn(__fadd_rn(p[0][j], p[1][j]), __fadd_rn(p[2][j], p[3][j])),
                     __fadd_rn(__fadd_rn(p[4][j], p[5][j]), __fadd_rn(p[6][j], p[7][j])));
}
// One reduction of the LN_RB rows over the CTA: the warp sums (lanes 0, 8,
// 16, 24 store theirs), a barrier, then every lane takes the CTA total of
// row lane % LN_RB.  The caller must not write p again before every warp has
// passed a later barrier.
__device__ __forceinline__ float cta_rows_sum(const float (&s)[LN_RB], float (*p)[LN_RB], int warp, int lane)
{
    const float v = warp_sum4(s, lane);
    if ((lane & 7) == 0) p[warp][lane >> 3] = v;
    __syncthreads();
    return ln_tree8(p, lane & (LN_RB - 1));
}

// The statistics of rows longer than 4096 elements (the CTA-wide order
// above), streaming each row twice (through L2) instead of holding it.
__global__ void __launch_bounds__(256) k_ln_stats_long(const uint16_t* __restrict__ x, int64_t R, int K, float eps,
                                                       float* __restrict__ mu, float* __restrict__ rstd)
{
    pdl_enter();
    __shared__ float part[2][8][LN_RB];
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int nch = K / 8;
    const int64_t r0 = (int64_t)blockIdx.x * LN_RB;
    float s[LN_RB];
#pragma unroll
    for (int j = 0; j < LN_RB; ++j) {
        const bool live = r0 + j < R;
        const uint16_t* row = x + (live ? r0 + j : 0) * (int64_t)K;
        float2 acc = make_float2(0.0f, 0.0f);
        for (int c = t; live && c < nch; c += 256) {
            Vec8<kBF16> v;
            v.load(row, c * 8);
            float2 p[4];
            bf16x8_pairs(v.w, p);
            acc = ln_sum8(p, acc);
        }
        s[j] = __fadd_rn(acc.x, acc.y);
    }
    const float mean_l = __fdiv_rn(cta_rows_sum(s, part[0], warp, lane), (float)K);
#pragma unroll
    for (int j = 0; j < LN_RB; ++j) {
        const float mean = __shfl_sync(0xFFFFFFFFu, mean_l, j);
        const bool live = r0 + j < R;
        const uint16_t* row = x + (live ? r0 + j : 0) * (int64_t)K;
        float2 acc = make_float2(0.0f, 0.0f);
        for (int c = t; live && c < nch; c += 256) {
            Vec8<kBF16> v;
            v.load(row, c * 8);
            float2 p[4];
            bf16x8_pairs(v.w, p);
            acc = ln_sq8(p, make_float2(-mean, -mean), acc);
        }
        s[j] = __fadd_rn(acc.x, acc.y);
    }
    const float var_l = __fdiv_rn(cta_rows_sum(s, part[1], warp, lane), (float)K);
    if (warp == 0 && lane < LN_RB && r0 + lane < R) {
        mu[r0 + lane] = mean_l;
        rstd[r0 + lane] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var_l, eps)));
    }
}

// Rows of up to 32 x 8 x CT elements (CT = 4: 1024, CT = 8: 2048, CT = 16:
// 4096), one warp per RBW rows at a time: lane l owns the 8-element chunks
// l, l + 32, ... of its rows and sums them in that order into eight
// partials, one per element position of a chunk (mixed-precision adds, no
// separate widening), which it combines as ((p0 + p1) + (p2 + p3)) over the
// (even, odd) pairs and then even + odd; the squared deviations take the
// (even, odd) pairs as above.  A warp butterfly (the same sum in every lane)
// completes the row; no barrier and no shared memory reduction.  Each lane copies its chunks of the
// warp's next rows into the warp's shared-memory stage (cp.async) once its
// sums have consumed the current ones, so the next rows' loads are in flight
// while the current rows are reduced, normalised and cast (no barrier guards
// the stage: a lane reads back only what it copied).  CAST = true: the
// LayerNorm fused into the delayed per-tensor cast, x read once, 3 B moved
// per element (gamma and beta staged once per CTA as four arrays of 16-byte
// halves, so a warp's reads of a chunk's halves are consecutive 16-byte
// words); CAST = false: the statistics alone, which serve the two-pass cast
// at these widths, so both paths share the reduction order.
__device__ __forceinline__ float ln_warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
template <bool CAST, int CT, int RBW>
__host__ __device__ constexpr int ln_warp_smem(int K)
{
    return (CAST ? 2 * K * 4 : 0) + 8 * RBW * CT * 32 * 16;   // gamma and beta (fp32), then eight warps' stages
}
template <bool CAST, int FMT, int CT, int RBW>
__global__ void __launch_bounds__(256, CT >= 16 ? 2 : 3) k_ln_warp(const uint16_t* __restrict__ x, int64_t R, int K, float eps,
                                                    const float* __restrict__ gamma, const float* __restrict__ beta,
                                                    float* __restrict__ mu, float* __restrict__ rstd,
                                                    uint8_t* __restrict__ q, float* state, int H, float* s_out,
                                                    unsigned long long* sat)
{
    pdl_enter();
    extern __shared__ __align__(16) uint8_t ln_smem[];
    __shared__ uint32_t red[8];
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int nch = K / 8;
    float4* gb4 = reinterpret_cast<float4*>(ln_smem);          // CAST: gamma lo, gamma hi, beta lo, beta hi [nch]
    // this warp's stage: [RBW rows][CT chunks][32 lanes] of 16 bytes
    uint4* xs = reinterpret_cast<uint4*>(ln_smem + (CAST ? 2 * K * 4 : 0)) + warp * (RBW * CT * 32);
    const int64_t stride = (int64_t)gridDim.x * 8 * RBW;
    auto stage = [&](int64_t r0) {
#pragma unroll
        for (int j = 0; j < RBW; ++j) {
            if (r0 + j >= R) continue;
            const uint16_t* row = x + (r0 + j) * (int64_t)K;
#pragma unroll
            for (int i = 0; i < CT; ++i) {
                const int c = lane + 32 * i;
                if (c < nch) cp_async16(&xs[(j * CT + i) * 32 + lane], row + c * 8);
            }
        }
        cp_async_commit();
    };
    stage(((int64_t)blockIdx.x * 8 + warp) * RBW);
    float m = 0.0f;
    if (CAST) {
        const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int c = t; c < nch; c += 256) {
            const float4* g = reinterpret_cast<const float4*>(gamma) + 2 * c;
            const float4* b = reinterpret_cast<const float4*>(beta) + 2 * c;
            gb4[c] = g[0];
            gb4[nch + c] = g[1];
            gb4[2 * nch + c] = beta ? b[0] : z4;
            gb4[3 * nch + c] = beta ? b[1] : z4;
        }
        __syncthreads();
        m = state[H];
        if (blockIdx.x == 0 && t == 0 && s_out) *s_out = state[H + 1];
    }
    float amax = 0.0f;
    uint32_t nsat = 0;
    for (int64_t r0 = ((int64_t)blockIdx.x * 8 + warp) * RBW; r0 < R; r0 += stride) {
        cp_async_wait_all();
        Vec8<kBF16> v[RBW][CT];
#pragma unroll
        for (int j = 0; j < RBW; ++j) {
#pragma unroll
            for (int i = 0; i < CT; ++i) {
                const int c = lane + 32 * i;
                if (r0 + j < R && c < nch) v[j][i].w = xs[(j * CT + i) * 32 + lane]; else v[j][i].zero();
            }
        }
        float mean[RBW], rs[RBW];
        float s0[RBW];
#pragma unroll
        for (int j = 0; j < RBW; ++j) {
            float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                             make_float2(0.0f, 0.0f)};
#pragma unroll
            for (int i = 0; i < CT; ++i) {
                if (lane + 32 * i >= nch) continue;
                acc[0] = bf16x2_add(v[j][i].w.x, acc[0]);
                acc[1] = bf16x2_add(v[j][i].w.y, acc[1]);
                acc[2] = bf16x2_add(v[j][i].w.z, acc[2]);
                acc[3] = bf16x2_add(v[j][i].w.w, acc[3]);
            }
            const float2 t = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
            s0[j] = __fadd_rn(t.x, t.y);
        }
        // the sums have consumed this warp's stage: start the next rows'
        stage(r0 + stride);
#pragma unroll
        for (int j = 0; j < RBW; ++j) mean[j] = __fdiv_rn(ln_warp_sum(s0[j]), (float)K);
#pragma unroll
        for (int j = 0; j < RBW; ++j) {
            float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < CT; ++i) {
                if (lane + 32 * i >= nch) continue;
                float2 d[4];
                ln_dev8(v[j][i].w, make_float2(-mean[j], -mean[j]), d);
#pragma unroll
                for (int k = 0; k < 4; ++k) acc = __ffma2_rn(d[k], d[k], acc);
            }
            const float var = __fdiv_rn(ln_warp_sum(__fadd_rn(acc.x, acc.y)), (float)K);
            rs[j] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
            if (lane == 0 && r0 + j < R) {
                mu[r0 + j] = mean[j];
                rstd[r0 + j] = rs[j];
            }
        }
        if (CAST) {
#pragma unroll
            for (int i = 0; i < CT; ++i) {
                const int c = lane + 32 * i;
                if (c >= nch) continue;
                const float4 ga = gb4[c], gh = gb4[nch + c], ba = gb4[2 * nch + c], bh = gb4[3 * nch + c];
                const float2 g[4] = {make_float2(ga.x, ga.y), make_float2(ga.z, ga.w), make_float2(gh.x, gh.y),
                                     make_float2(gh.z, gh.w)};
                const float2 be[4] = {make_float2(ba.x, ba.y), make_float2(ba.z, ba.w), make_float2(bh.x, bh.y),
                                      make_float2(bh.z, bh.w)};
#pragma unroll
                for (int j = 0; j < RBW; ++j) {
                    if (r0 + j >= R) continue;
                    float2 d[4];
                    ln_dev8(v[j][i].w, make_float2(-mean[j], -mean[j]), d);
                    *reinterpret_cast<uint2*>(q + (r0 + j) * (int64_t)K + c * 8) =
                        ln_cast8<FMT>(d, make_float2(rs[j], rs[j]), g, be, m, amax, nsat);
                }
            }
        }
    }
    if (CAST) {
        if (sat) add_sat(sat, nsat);
        const uint32_t b = block_max_bits<8>(__float_as_uint(amax), red);
        if (t == 0) atomic_max_bits(&state[0], b);
    }
}

// One LayerNorm-kernel launch: KERN is a k_ln_warp instantiation,
// `rows_per_cta` the rows one CTA takes per iteration;
// CAST launches pass the codes and state.
template <typename Kern>
static void launch_ln(Kern kern, int rows_per_cta, int smem, const QuantArgs& a, const float* gamma,
                      const float* beta, float eps, float* mu, float* rstd, cudaStream_t st, int sms, bool cast)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    const int64_t groups = (a.rows + rows_per_cta - 1) / rows_per_cta;
    const int64_t cap = (int64_t)sms * per_sm;
    const unsigned grid = (unsigned)(groups < cap ? groups : cap);
    launch_k(kern, grid, 256, smem, st, static_cast<const uint16_t*>(a.x), a.rows, (int)a.cols, eps, gamma, beta, mu,
             rstd, cast ? a.q : (uint8_t*)nullptr, cast ? a.state : (float*)nullptr, cast ? a.history_len : 0,
             cast ? static_cast<float*>(a.scales) : (float*)nullptr, cast ? a.sat : (unsigned long long*)nullptr);
}

// A k_ln_warp launch: its shared memory (gamma and beta for CAST, the warps'
// stages) allowed once at the largest width it serves.
template <bool CAST, int FMT, int CT, int RBW>
static cudaError_t launch_ln_warp(const QuantArgs& a, const float* gamma, const float* beta, float eps, float* mu,
                                  float* rstd, cudaStream_t st, int sms)
{
    auto kern = k_ln_warp<CAST, FMT, CT, RBW>;
    cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(kern), ln_warp_smem<CAST, CT, RBW>(32 * 8 * CT));
    if (e != cudaSuccess) return e;
    launch_ln(kern, 8 * RBW, ln_warp_smem<CAST, CT, RBW>((int)a.cols), a, gamma, beta, eps, mu, rstd, st, sms, CAST);
    return cudaGetLastError();
}

cudaError_t launch_layernorm_quantize(const QuantArgs& a, const float* gamma, const float* beta, float eps,
                                      float* mu, float* rstd, cudaStream_t st, int sms)
{
    if (a.rows == 0 || a.cols == 0) return cudaSuccess;
    const int K = (int)a.cols;
    // row width -> kernel: up to 1024 a warp per two rows, up to 4096 a warp
    // per row (all held in registers); wider rows stream their statistics and
    // always take two passes
    const int width = K <= 1024 ? 0 : K <= 2048 ? 1 : K <= 4096 ? 2 : 3;
    const bool one_pass = !a.qT && !a.amax && width < 3;
    const bool e4 = a.format == kE4M3;
    cudaError_t e = cudaSuccess;
    if (width == 0) {
        if (one_pass) return e4 ? launch_ln_warp<true, kE4M3, 4, 2>(a, gamma, beta, eps, mu, rstd, st, sms)
                                : launch_ln_warp<true, kE5M2, 4, 2>(a, gamma, beta, eps, mu, rstd, st, sms);
        e = launch_ln_warp<false, kE4M3, 4, 2>(a, gamma, beta, eps, mu, rstd, st, sms);
    } else if (width == 1) {
        if (one_pass) return e4 ? launch_ln_warp<true, kE4M3, 8, 1>(a, gamma, beta, eps, mu, rstd, st, sms)
                                : launch_ln_warp<true, kE5M2, 8, 1>(a, gamma, beta, eps, mu, rstd, st, sms);
        e = launch_ln_warp<false, kE4M3, 8, 1>(a, gamma, beta, eps, mu, rstd, st, sms);
    } else if (width == 2) {
        if (one_pass) return e4 ? launch_ln_warp<true, kE4M3, 16, 1>(a, gamma, beta, eps, mu, rstd, st, sms)
                                : launch_ln_warp<true, kE5M2, 16, 1>(a, gamma, beta, eps, mu, rstd, st, sms);
        e = launch_ln_warp<false, kE4M3, 16, 1>(a, gamma, beta, eps, mu, rstd, st, sms);
    } else {
        launch_k(k_ln_stats_long, (unsigned)((a.rows + LN_RB - 1) / LN_RB), 256, 0, st,
                 static_cast<const uint16_t*>(a.x), a.rows, K, eps, mu, rstd);
    }
    if (e != cudaSuccess) return e;
    // two passes: the statistics above, then the tiled cast in its LayerNorm
    // mode (which also writes the transposed copy)
    LnParams ln;
    ln.mu = mu;
    ln.rstd = rstd;
    ln.gamma = gamma;
    ln.beta = beta;
    const dim3 grid((unsigned)((a.cols + 127) / 128), (unsigned)((a.rows + 127) / 128));
    auto kern = e4 ? k_cast_tensor_T<kBF16, kE4M3, true, true> : k_cast_tensor_T<kBF16, kE5M2, true, true>;
    launch_k(kern, grid, 256, 0, st, a.x, a.rows, a.cols, a.q, a.qT, a.state, a.history_len, nullptr,
             static_cast<float*>(a.scales), a.amax, a.sat, ln);
    return cudaGetLastError();
}

// ================================================================== row units
// 1x128 tiles (UNIT = 128) and MX-32 blocks (UNIT = 32).  Each lane holds 16
// consecutive elements (two 128-bit chunks) and a unit is UNIT/16 consecutive
// lanes; units never straddle a row because cols % UNIT == 0, so the tensor is
// treated as flat.  Sixteen elements per lane halve the per-element cost of
// the unit's shuffles and scale computation against eight.
// WRITE_Q = false computes the unit amaxes only (fp8_amax).
// RULE: 0 = current fp32 scale (1x128 tiles); 1 = E8M0, smallest power of two
// that fits (MX-32 blocks, and power-of-two 1x128 tiles); 2 = E8M0 by the
// OCP floor rule (MX-32 blocks).  A power-of-two 1x128 tile writes its code
// into all four 32-blocks it covers in the tiled layout.
template <int DT, int FMT, int UNIT, bool WRITE_Q, bool TILED = false, int RULE = (UNIT == 32 ? 1 : 0)>
__global__ void __launch_bounds__(kFlatThreads) k_quant_rowunits(const void* __restrict__ x, int64_t n,
                                                                 uint8_t* __restrict__ q, void* scales,
                                                                 float* amax_out, unsigned long long* sat,
                                                                 int64_t cols = 0)
{
    pdl_enter();
    constexpr int TPU = UNIT / 16;  // lanes per unit
    constexpr int U = row_unroll<UNIT>();
    const int64_t ng = n / 16;      // 16-element groups
    uint32_t nsat = 0;
    const int64_t stride = (int64_t)gridDim.x * kFlatThreads * U;
    for (int64_t g0 = (int64_t)blockIdx.x * kFlatThreads * U; g0 < ng; g0 += stride) {
        Vec8<DT> v[U][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t g = g0 + u * kFlatThreads + threadIdx.x;
            if (g < ng) {
                v[u][0].load(x, g * 16);
                v[u][1].load(x, g * 16 + 8);
            } else {
                v[u][0].zero();
                v[u][1].zero();
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t g = g0 + u * kFlatThreads + threadIdx.x;
            const uint32_t b0 = v[u][0].absmax_bits(), b1 = v[u][1].absmax_bits();
            uint32_t a = max(b0, b1);
#pragma unroll
            for (int o = TPU / 2; o >= 1; o >>= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
            const bool valid = g < ng;             // uniform over a unit's lanes
            const bool leader = (threadIdx.x % TPU) == 0;
            const int64_t unit = g / TPU;
            if (valid && leader && amax_out) amax_out[unit] = __uint_as_float(a);
            if (WRITE_Q) {
                float m, s = 0.0f;
                uint32_t code = 0;
                if (RULE == 1) code = mx_scale<FMT>(a, m);
                else if (RULE == 2) code = mx_scale_floor<FMT>(a, m);
                else current_scale<FMT>(a, m, s);
                float f[8];
                v[u][0].get(f);
                const uint2 c0 = cast8<FMT>(f, m, b0, nsat);
                v[u][1].get(f);
                const uint2 c1 = cast8<FMT>(f, m, b1, nsat);
                if (valid) {
                    *reinterpret_cast<uint4*>(q + g * 16) = make_uint4(c0.x, c0.y, c1.x, c1.y);
                    if (leader) {
                        if (RULE == 0) {
                            static_cast<float*>(scales)[unit] = s;
                        } else if (TILED) {
                            constexpr int SUB = UNIT / 32;      // 32-blocks per unit
                            const int64_t per_row = cols / UNIT;
                            int64_t r, t;
                            if ((uint64_t)unit < (1ull << 32)) {     // 32-bit division where it fits
                                r = (uint32_t)unit / (uint32_t)per_row;
                                t = (uint32_t)unit - (uint32_t)r * (uint32_t)per_row;
                            } else {
                                r = unit / per_row;
                                t = unit % per_row;
                            }
#pragma unroll
                            for (int i = 0; i < SUB; ++i)
                                static_cast<uint8_t*>(scales)[mx_tiled_offset(r, t * SUB + i, cols)] = (uint8_t)code;
                        } else {
                            static_cast<uint8_t*>(scales)[unit] = (uint8_t)code;
                        }
                    }
                }
            }
        }
    }
    if (WRITE_Q && sat) add_sat(sat, nsat);
}

// ================================================================== 128x128 blocks
// One CTA per block, 256 threads, 8x8 elements per thread (same warp layout
// as k_cast_tensor_T); block amax through shared memory, then the cast.
// With qT, the block's transposed codes go to qT [C][R] and its scale to
// sT[C/128][R/128] (the 128x128 blocks of x^T are x's blocks transposed).
// POW2: the block scale is the smallest power of two that fits (E8M0); its
// code fills the block's whole 512-byte chunk of the tiled MX layout (all 128
// rows x four 32-blocks), so the block feeds the block-scaled GEMM directly.
// Four CTAs per SM (64 registers, no spills): measured on the GB300 against
// three (80 registers), L2 flushed, identical codes: 16384 x 14336 106.5 ->
// 100.4 us (with qT 141.6 -> 139.3), 8192 x 8192 32.3 -> 28.7 us.
template <int DT, int FMT, bool WRITE_Q, bool POW2 = false>
__global__ void __launch_bounds__(256, 4) k_quant_block128(const void* __restrict__ x, int64_t R, int64_t C,
                                                        uint8_t* __restrict__ q, float* s_out,
                                                        float* amax_out, unsigned long long* sat,
                                                        uint8_t* __restrict__ qT = nullptr, float* sT = nullptr,
                                                        uint8_t* e_tiled = nullptr, uint8_t* eT_tiled = nullptr)
{
    pdl_enter();
    __shared__ uint32_t red[8];
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int64_t c0 = (int64_t)blockIdx.x * 128 + ((w & 3) * 4 + (l & 3)) * 8;
    const int64_t r0 = (int64_t)blockIdx.y * 128 + ((w >> 2) * 8 + (l >> 2)) * 8;
    Vec8<DT> v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i].load(x, (r0 + i) * C + c0);
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mx = max(mx, v[i].absmax_bits());
    const uint32_t a = block_max_bits<8>(mx, red);
    const int64_t unit = (int64_t)blockIdx.y * gridDim.x + blockIdx.x;
    float m, s = 0.0f;
    if (POW2) {
        const uint32_t code = mx_scale<FMT>(a, m);
        if (WRITE_Q) {
            const uint16_t two = (uint16_t)(code | (code << 8));
            reinterpret_cast<uint16_t*>(e_tiled + unit * 512)[threadIdx.x] = two;
            // the same block of x^T: chunk (column block, row block) of its layout
            if (eT_tiled)
                reinterpret_cast<uint16_t*>(eT_tiled + ((int64_t)blockIdx.x * gridDim.y + blockIdx.y) * 512)[threadIdx.x] =
                    two;
        }
    } else {
        current_scale<FMT>(a, m, s);
    }
    if (threadIdx.x == 0) {
        if (amax_out) amax_out[unit] = __uint_as_float(a);
        if (WRITE_Q && !POW2) s_out[unit] = s;
        if (WRITE_Q && !POW2 && sT) sT[(int64_t)blockIdx.x * gridDim.y + blockIdx.y] = s;
    }
    if (!WRITE_Q) return;
    uint32_t nsat = 0;
    uint2 rows[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float f[8];
        v[i].get(f);
        rows[i] = cast8<FMT>(f, m, v[i].absmax_bits(), nsat);
        *reinterpret_cast<uint2*>(q + (r0 + i) * C + c0) = rows[i];
    }
    if (qT) {
        uint2 cols[8];
        transpose8x8(rows, cols);
#pragma unroll
        for (int j = 0; j < 8; ++j) *reinterpret_cast<uint2*>(qT + (c0 + j) * R + r0) = cols[j];
    }
    if (sat) add_sat(sat, nsat);
}

// ================================================================== state
__global__ void k_scale_init(float* states, int n, int H)
{
    pdl_enter();
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t total = (int64_t)n * (H + 2);
    if (i < total) {
        int64_t j = i % (H + 2);
        states[i] = (j < H) ? 0.0f : 1.0f;
    }
}

struct FormatList {
    uint8_t f[1024];
};

__global__ void k_update_scale(float* states, int n, int H, FormatList fl, int algo)
{
    pdl_enter();
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float* st = states + (int64_t)i * (H + 2);
    uint32_t a = __float_as_uint(st[0]) & 0x7FFFFFFFu;
    if (algo == 0)
        for (int j = 1; j < H; ++j) a = max(a, __float_as_uint(st[j]) & 0x7FFFFFFFu);
    if (a != 0u && a < 0x7F800000u) {
        float fm = fl.f[i] == kE4M3 ? Fmt<kE4M3>::fmax : Fmt<kE5M2>::fmax;
        float af = __uint_as_float(a);
        st[H] = __fdiv_rn(fm, af);
        st[H + 1] = __fdiv_rn(af, fm);
    }
    for (int j = H - 1; j >= 1; --j) st[j] = st[j - 1];
    st[0] = 0.0f;
}

// ================================================================== launchers
// CTAs of a flat kernel (kFlatThreads threads, no dynamic shared memory)
// that fit on one SM at once, queried once per kernel and device.
static int resident_per_sm(const void* kern)
{
    static std::mutex mu;
    static const void* keys[128];
    static int devs[128], vals[128];
    static int n = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (keys[i] == kern && devs[i] == dev) return vals[i];
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kFlatThreads, 0) != cudaSuccess || b < 1) {
        cudaGetLastError();
        b = 1;
    }
    if (n < 128) {
        keys[n] = kern;
        devs[n] = dev;
        vals[n] = b;
        ++n;
    }
    return b;
}

// CTAs a grid-stride flat kernel is launched with per SM: a whole number of
// the CTAs that fit at once, about eight.  A grid that is not a whole
// number of resident waves runs its last CTAs as a partial wave (a 16384 x
// 14336 cast ran at 0.80 of HBM with 8 CTAs per SM requested and 6
// resident, 0.91 with 6); two full waves of 4 (the 64-register row-unit
// casts) time slightly better than one.
static int64_t flat_cap(const void* kern, int sms)
{
    const int per_sm = resident_per_sm(kern);
    const int waves = per_sm >= 8 ? 1 : 8 / per_sm;
    return (int64_t)sms * per_sm * waves;
}

// Grid of a grid-stride flat kernel over nch work items (kFlatUnroll per
// thread per pass).
template <typename K>
static int flat_grid(K kern, int64_t nch, int sms)
{
    const int64_t per_block = (int64_t)kFlatThreads * kFlatUnroll;
    const int64_t need = (nch + per_block - 1) / per_block;
    const int64_t cap = flat_cap(reinterpret_cast<const void*>(kern), sms);
    const int64_t g = need < cap ? need : cap;
    return g < 1 ? 1 : (int)g;
}

// The same for the row-unit kernels (U groups per thread per pass).
template <int U, typename K>
static int flat_grid_u(K kern, int64_t nch, int sms)
{
    const int64_t per_block = (int64_t)kFlatThreads * U;
    const int64_t need = (nch + per_block - 1) / per_block;
    const int64_t cap = flat_cap(reinterpret_cast<const void*>(kern), sms);
    const int64_t g = need < cap ? need : cap;
    return g < 1 ? 1 : (int)g;
}

// The grids of the two jobs of a two-tensor flat kernel: each job's own need
// when both fit at once, else the resident capacity split in proportion to
// the jobs' sizes (at least one CTA each).
template <typename K>
static void flat_grid2(K kern, int64_t na, int64_t nb, int sms, int& ga, int& gb)
{
    const int64_t per_block = (int64_t)kFlatThreads * kFlatUnroll;
    const int64_t need_a = (na + per_block - 1) / per_block, need_b = (nb + per_block - 1) / per_block;
    const int64_t cap = flat_cap(reinterpret_cast<const void*>(kern), sms);
    int64_t a = need_a < 1 ? 1 : need_a, b = need_b < 1 ? 1 : need_b;
    if (a + b > cap) {
        a = (int64_t)((double)cap * (double)na / (double)(na + nb) + 0.5);
        a = a < 1 ? 1 : (a > cap - 1 ? cap - 1 : a);
        b = cap - a < 1 ? 1 : cap - a;
    }
    ga = (int)a;
    gb = (int)b;
}

template <int DT>
static cudaError_t amax_dt(const QuantArgs& a, cudaStream_t st, int sms)
{
    const int64_t n = a.rows * a.cols;
    switch (a.gran) {
    case kTensor:
        if (cudaMemsetAsync(a.amax, 0, sizeof(float), st) != cudaSuccess) return cudaGetLastError();
        if (n > 0) launch_k(k_amax_tensor<DT>, flat_grid(k_amax_tensor<DT>, n / 8, sms), kFlatThreads, 0, st, a.x, n, a.amax);
        break;
    case kTile:
        if (n > 0) launch_k(k_quant_rowunits<DT, kE4M3, 128, false>, flat_grid_u<row_unroll<128>()>(k_quant_rowunits<DT, kE4M3, 128, false>, n / 16, sms), kFlatThreads, 0, st, a.x, n, nullptr, nullptr, a.amax, nullptr, (int64_t)0);
        break;
    case kMX:
        if (n > 0) launch_k(k_quant_rowunits<DT, kE4M3, 32, false>, flat_grid_u<row_unroll<32>()>(k_quant_rowunits<DT, kE4M3, 32, false>, n / 16, sms), kFlatThreads, 0, st, a.x, n, nullptr, nullptr, a.amax, nullptr, (int64_t)0);
        break;
    case kBlock:
        if (n > 0) launch_k(k_quant_block128<DT, kE4M3, false>, dim3((unsigned)(a.cols / 128), (unsigned)(a.rows / 128)), 256, 0, st, a.x, a.rows, a.cols, nullptr, nullptr, a.amax, nullptr,
                            nullptr, nullptr, nullptr, nullptr);
        break;
    }
    return cudaGetLastError();
}

cudaError_t launch_amax(const QuantArgs& a, cudaStream_t st, int sms)
{
    return a.x_dtype == kBF16 ? amax_dt<kBF16>(a, st, sms) : amax_dt<kF32>(a, st, sms);
}

template <int DT, int FMT>
static cudaError_t quant_dt_fmt(const QuantArgs& a, cudaStream_t st, int sms)
{
    const int64_t n = a.rows * a.cols;
    const int H = a.history_len;
    if (a.gran == kTensor) {
        const bool delayed = a.state != nullptr;
        if (!delayed) {
            // pass 1: amax into a.amax (required), pass 2 reads it
            QuantArgs p = a;
            p.gran = kTensor;
            cudaError_t e = amax_dt<DT>(p, st, sms);
            if (e != cudaSuccess) return e;
        } else if (a.amax) {
            if (cudaMemsetAsync(a.amax, 0, sizeof(float), st) != cudaSuccess) return cudaGetLastError();
        }
        float* s_out = static_cast<float*>(a.scales);
        if (a.qT) {
            if (n == 0) {
                if (!delayed) launch_k(k_cast_tensor<DT, FMT, false>, 1, kFlatThreads, 0, st, a.x, 0, a.q, nullptr, 0, a.amax, s_out, nullptr, nullptr);
                else if (s_out) launch_k(k_cast_tensor<DT, FMT, true>, 1, kFlatThreads, 0, st, a.x, 0, a.q, a.state, H, nullptr, s_out, a.amax, nullptr);
                return cudaGetLastError();
            }
            dim3 grid((unsigned)((a.cols + 127) / 128), (unsigned)((a.rows + 127) / 128));
            if (delayed)
                launch_k(k_cast_tensor_T<DT, FMT, true>, grid, 256, 0, st, a.x, a.rows, a.cols, a.q, a.qT, a.state, H, nullptr, s_out,
                         a.amax, a.sat, LnParams());
            else
                launch_k(k_cast_tensor_T<DT, FMT, false>, grid, 256, 0, st, a.x, a.rows, a.cols, a.q, a.qT, nullptr, 0, a.amax, s_out,
                         nullptr, a.sat, LnParams());
        } else {
            int g = delayed ? flat_grid(k_cast_tensor<DT, FMT, true>, n / 8, sms)
                            : flat_grid(k_cast_tensor<DT, FMT, false>, n / 8, sms);
            if (delayed)
                launch_k(k_cast_tensor<DT, FMT, true>, g, kFlatThreads, 0, st, a.x, n, a.q, a.state, H, nullptr, s_out, a.amax, a.sat);
            else
                launch_k(k_cast_tensor<DT, FMT, false>, g, kFlatThreads, 0, st, a.x, n, a.q, nullptr, 0, a.amax, s_out, nullptr, a.sat);
        }
        return cudaGetLastError();
    }
    if (n == 0) return cudaSuccess;
    switch (a.gran) {
    case kTile:
        launch_k(k_quant_rowunits<DT, FMT, 128, true>, flat_grid_u<row_unroll<128>()>(k_quant_rowunits<DT, FMT, 128, true>, n / 16, sms), kFlatThreads, 0, st, a.x, n, a.q, a.scales, a.amax, a.sat,
                 (int64_t)0);
        break;
    case kMX:
        launch_k(k_quant_rowunits<DT, FMT, 32, true>, flat_grid_u<row_unroll<32>()>(k_quant_rowunits<DT, FMT, 32, true>, n / 16, sms), kFlatThreads, 0, st, a.x, n, a.q, a.scales, a.amax, a.sat,
                 (int64_t)0);
        break;
    case kMXTiled:
        launch_k(k_quant_rowunits<DT, FMT, 32, true, true>, flat_grid_u<row_unroll<32>()>(k_quant_rowunits<DT, FMT, 32, true, true>, n / 16, sms), kFlatThreads, 0, st, a.x, n, a.q, a.scales, a.amax, a.sat, a.cols);
        break;
    case kTilePow2:
        launch_k(k_quant_rowunits<DT, FMT, 128, true, true, 1>, flat_grid_u<row_unroll<128>()>(k_quant_rowunits<DT, FMT, 128, true, true, 1>, n / 16, sms), kFlatThreads, 0, st, a.x, n, a.q, a.scales, a.amax, a.sat, a.cols);
        break;
    case kMXFloor:
        launch_k(k_quant_rowunits<DT, FMT, 32, true, true, 2>, flat_grid_u<row_unroll<32>()>(k_quant_rowunits<DT, FMT, 32, true, true, 2>, n / 16, sms), kFlatThreads, 0, st, a.x, n, a.q, a.scales, a.amax, a.sat, a.cols);
        break;
    case kBlockPow2:
        // (qT and scalesT: the transposed codes and the tiled E8M0 codes of
        // x^T, for a linear layer's dgrad)
        launch_k(k_quant_block128<DT, FMT, true, true>, dim3((unsigned)(a.cols / 128), (unsigned)(a.rows / 128)), 256, 0, st, a.x, a.rows, a.cols, a.q, nullptr, a.amax, a.sat, a.qT, nullptr, static_cast<uint8_t*>(a.scales),
                 reinterpret_cast<uint8_t*>(a.scalesT));
        break;
    case kTileCol:
    case kMXCol: {
        const dim3 grid((unsigned)((a.cols + 127) / 128), (unsigned)(a.rows / 128));
        auto kern = a.gran == kTileCol ? k_quant_col_block<FMT, 128> : k_quant_col_block<FMT, 32>;
        launch_k(kern, grid, 256, 0, st, a.x, a.rows, a.cols, a.q, a.qT, a.scales, nullptr, a.sat);
        break;
    }
    case kTileRowCol:
    case kTileRowColPow2:
    case kMXRowCol: {
        // rows in their own units into q / scales, columns into qT / col_scales
        const dim3 grid((unsigned)(a.cols / 128), (unsigned)(a.rows / 128));
        auto kern = a.gran == kTileRowCol       ? k_quant_col_block<FMT, 128, true>
                    : a.gran == kTileRowColPow2 ? k_quant_col_block<FMT, 128, true, true>
                                                : k_quant_col_block<FMT, 32, true>;
        launch_k(kern, grid, 256, 0, st, a.x, a.rows, a.cols, a.q, a.qT, a.col_scales, a.scales, a.sat);
        break;
    }
    case kBlock:
        launch_k(k_quant_block128<DT, FMT, true>, dim3((unsigned)(a.cols / 128), (unsigned)(a.rows / 128)), 256, 0, st, a.x, a.rows, a.cols, a.q, static_cast<float*>(a.scales), a.amax, a.sat, a.qT, a.scalesT,
                 nullptr, nullptr);
        break;
    }
    return cudaGetLastError();
}

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st, int sms)
{
    if (a.x_dtype == kBF16)
        return a.format == kE4M3 ? quant_dt_fmt<kBF16, kE4M3>(a, st, sms) : quant_dt_fmt<kBF16, kE5M2>(a, st, sms);
    return a.format == kE4M3 ? quant_dt_fmt<kF32, kE4M3>(a, st, sms) : quant_dt_fmt<kF32, kE5M2>(a, st, sms);
}

// Two per-tensor casts with transposed copies in one launch (plus, for
// current scaling, one launch for both amaxes): a linear layer's x and W.
template <int DT, int FMT>
static cudaError_t quant_pair_dt_fmt(const QuantArgs& a, const QuantArgs& b, cudaStream_t st, int sms)
{
    const bool delayed = a.state != nullptr;
    // the amax slots start at zero (one memset when they are adjacent)
    auto clear = [&](float* pa, float* pb) -> cudaError_t {
        if (pa && pb && pb == pa + 1) return cudaMemsetAsync(pa, 0, 2 * sizeof(float), st);
        if (pa && cudaMemsetAsync(pa, 0, sizeof(float), st) != cudaSuccess) return cudaGetLastError();
        if (pb && cudaMemsetAsync(pb, 0, sizeof(float), st) != cudaSuccess) return cudaGetLastError();
        return cudaSuccess;
    };
    if (clear(a.amax, b.amax) != cudaSuccess) return cudaGetLastError();
    const int64_t na = a.rows * a.cols, nb = b.rows * b.cols;
    if (!delayed) {
        int ga, gb;
        flat_grid2(k_amax_tensor2<DT>, na / 8, nb / 8, sms, ga, gb);
        launch_k(k_amax_tensor2<DT>, ga + gb, kFlatThreads, 0, st, AmaxJob{a.x, na, a.amax}, AmaxJob{b.x, nb, b.amax}, ga);
    }
    const int64_t tiles_a = ((a.cols + 127) / 128) * ((a.rows + 127) / 128);
    const int64_t tiles_b = ((b.cols + 127) / 128) * ((b.rows + 127) / 128);
    const CastJob ja{a.x, a.rows, a.cols, a.q, a.qT, a.state, delayed ? nullptr : a.amax, static_cast<float*>(a.scales),
                     delayed ? a.amax : nullptr};
    const CastJob jb{b.x, b.rows, b.cols, b.q, b.qT, b.state, delayed ? nullptr : b.amax, static_cast<float*>(b.scales),
                     delayed ? b.amax : nullptr};
    const unsigned grid = (unsigned)(tiles_a + tiles_b);
    if (delayed)
        launch_k(k_cast_tensor_T2<DT, FMT, true>, grid, 256, 0, st, ja, jb, tiles_a, a.history_len, a.sat);
    else
        launch_k(k_cast_tensor_T2<DT, FMT, false>, grid, 256, 0, st, ja, jb, tiles_a, 0, a.sat);
    return cudaGetLastError();
}

// The same without transposed copies: the flat cast over both tensors.
template <int DT, int FMT>
static cudaError_t quant_pair_flat_dt_fmt(const QuantArgs& a, const QuantArgs& b, cudaStream_t st, int sms)
{
    const bool delayed = a.state != nullptr;
    const int64_t na = a.rows * a.cols, nb = b.rows * b.cols;
    if (a.amax && b.amax && b.amax == a.amax + 1) {
        if (cudaMemsetAsync(a.amax, 0, 2 * sizeof(float), st) != cudaSuccess) return cudaGetLastError();
    } else {
        if (a.amax && cudaMemsetAsync(a.amax, 0, sizeof(float), st) != cudaSuccess) return cudaGetLastError();
        if (b.amax && cudaMemsetAsync(b.amax, 0, sizeof(float), st) != cudaSuccess) return cudaGetLastError();
    }
    if (!delayed) {
        int ga, gb;
        flat_grid2(k_amax_tensor2<DT>, na / 8, nb / 8, sms, ga, gb);
        launch_k(k_amax_tensor2<DT>, ga + gb, kFlatThreads, 0, st, AmaxJob{a.x, na, a.amax}, AmaxJob{b.x, nb, b.amax}, ga);
    }
    int ga, gb;
    if (delayed) flat_grid2(k_cast_tensor2<DT, FMT, true>, na / 8, nb / 8, sms, ga, gb);
    else flat_grid2(k_cast_tensor2<DT, FMT, false>, na / 8, nb / 8, sms, ga, gb);
    const FlatCastJob ja{a.x, na, a.q, a.state, delayed ? nullptr : a.amax, static_cast<float*>(a.scales),
                         delayed ? a.amax : nullptr};
    const FlatCastJob jb{b.x, nb, b.q, b.state, delayed ? nullptr : b.amax, static_cast<float*>(b.scales),
                         delayed ? b.amax : nullptr};
    if (delayed)
        launch_k(k_cast_tensor2<DT, FMT, true>, ga + gb, kFlatThreads, 0, st, ja, jb, ga, a.history_len, a.sat);
    else
        launch_k(k_cast_tensor2<DT, FMT, false>, ga + gb, kFlatThreads, 0, st, ja, jb, ga, 0, a.sat);
    return cudaGetLastError();
}

cudaError_t launch_quantize_pair(const QuantArgs& a, const QuantArgs& b, cudaStream_t st, int sms)
{
    const bool same = a.gran == kTensor && b.gran == kTensor && a.x_dtype == b.x_dtype && a.format == b.format &&
                      (a.qT != nullptr) == (b.qT != nullptr) && (a.state != nullptr) == (b.state != nullptr) &&
                      (!a.state || a.history_len == b.history_len) && (a.state || (a.amax && b.amax)) &&
                      a.sat == b.sat;
    if (!same || a.rows * a.cols == 0 || b.rows * b.cols == 0 || a.rows % 8 || a.cols % 8 || b.rows % 8 || b.cols % 8) {
        cudaError_t e = launch_quantize(a, st, sms);
        return e != cudaSuccess ? e : launch_quantize(b, st, sms);
    }
    if (!a.qT) {
        if (a.x_dtype == kBF16)
            return a.format == kE4M3 ? quant_pair_flat_dt_fmt<kBF16, kE4M3>(a, b, st, sms)
                                     : quant_pair_flat_dt_fmt<kBF16, kE5M2>(a, b, st, sms);
        return a.format == kE4M3 ? quant_pair_flat_dt_fmt<kF32, kE4M3>(a, b, st, sms)
                                 : quant_pair_flat_dt_fmt<kF32, kE5M2>(a, b, st, sms);
    }
    if (a.x_dtype == kBF16)
        return a.format == kE4M3 ? quant_pair_dt_fmt<kBF16, kE4M3>(a, b, st, sms) : quant_pair_dt_fmt<kBF16, kE5M2>(a, b, st, sms);
    return a.format == kE4M3 ? quant_pair_dt_fmt<kF32, kE4M3>(a, b, st, sms) : quant_pair_dt_fmt<kF32, kE5M2>(a, b, st, sms);
}

cudaError_t launch_scale_init(float* states, int n, int H, cudaStream_t st)
{
    int64_t total = (int64_t)n * (H + 2);
    if (total > 0) launch_k(k_scale_init, (unsigned)((total + 255) / 256), 256, 0, st, states, n, H);
    return cudaGetLastError();
}

cudaError_t launch_update_scale(float* states, int n, int H, const int* formats, int algo, cudaStream_t st)
{
    FormatList fl;
    for (int i = 0; i < n; ++i) fl.f[i] = (uint8_t)formats[i];
    if (n > 0) launch_k(k_update_scale, (n + 127) / 128, 128, 0, st, states, n, H, fl, algo);
    return cudaGetLastError();
}

}  // namespace fp8sq

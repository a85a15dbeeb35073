// gemm.cu -- FP8 GEMM on the sm_103a 5th-generation tensor cores.
//
// D[m][n] = epi(sum_k dec(A[m][k]) sA * dec(B[n][k]) sB): the "matmuls run in
// FP8" with a wider accumulator of the week-14 page (FP8 bullet,
// accumulation-precision bullet); x ~ q * scale from its absmax bullet.
//
// One persistent CTA per SM, warp-specialised:
//   warp 0     TMA producer: 128x128 A and BNx128 B tiles (K-major, 128-byte
//              swizzle) into a STAGES-deep shared-memory ring
//   warp 1     allocates tensor memory; one thread issues tcgen05.mma
//              (kind::f8f6f4, M=128, N=BN, K=32 per instruction) and
//              tcgen05.commit to release ring slots / publish accumulators
//   warps 2..  epilogue: tcgen05.ld the fp32 accumulator, multiply by the
//              dequantisation scales, round, store
// Mode 0 (per-tensor scales): two TMEM accumulators of BN columns, so the
// epilogue of tile i overlaps the MMAs of tile i+1.
// Mode 1 (1x128 activation tiles x 128x128 weight blocks): the MMAs of each
// 128-wide K block write a fresh partial into one of two TMEM buffers and
// the epilogue warps promote it into fp32 registers with sA[m][kb] *
// sB[nb][kb] (the fixed-interval fp32 promotion of the week-14 page,
// interval = the 128-wide scale block).
// Every mbarrier wait is bounded (1 s): on expiry the kernel sets a device
// error word, stops issuing work, drains what it issued and frees its
// tensor memory before returning.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace fp8sq {

__device__ int g_dev_error = 0;

// Every wait of this file reports into g_dev_error.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity)
{
    return wait_bounded_err(bar, parity, &g_dev_error);
}

// Raises a kernel's dynamic shared-memory limit once per device.  Setting a
// function attribute on every launch puts a driver call on the launch path
// that held back back-to-back calls (a fine-grained backward took 279 us in
// a loop of calls against 238 us replayed from a CUDA graph).
cudaError_t smem_attr_once(const void* kern, int bytes)
{
    static std::mutex mu;
    static const void* done_kern[128];
    static int done_dev[128];
    static int n_done = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done_kern[i] == kern && done_dev[i] == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && n_done < 128) {
        done_kern[n_done] = kern;
        done_dev[n_done] = dev;
        ++n_done;
    }
    return e;
}

struct TileSched {
    int num_m, num_n, group;
    __device__ __forceinline__ void coords(int t, int& mb, int& nb) const
    {
        const int per_group = group * num_n;
        const int g = t / per_group;
        const int first = g * group;
        const int gs = min(num_m - first, group);
        const int r = t - g * per_group;
        mb = first + r % gs;
        nb = r / gs;
    }
};

// M-tiles per group of the rasterisation.  The concurrent tiles of one wave
// cover `group` M-tiles and about concurrent / group N-tiles, so they hold
// (group x tile_m + concurrent / group x tile_n) rows of K bytes in L2, and
// B is read from DRAM num_m / group times.  The largest group of 32, 16, 8
// whose wave stays within 48 MB (about a third of L2) is taken; 8 otherwise.
// Measured on the GB300 (per-tensor pair kernel, 16384 x 14336 x 4096 / 8192^3
// / 16384 x 4096 x 14336, us): group 8: 533.5 / 302.0 / 529.7; 16: 524.5 /
// 297.5 / 532.3; 32: 522.0 / 307.8 / 552.5.  The MX kernel at 8192^3: 16:
// 355.8, 32: 353.4, 64: 379.2.
static int raster_group(int64_t K, int tile_m, int tile_n, int concurrent)
{
    for (int g = 32; g > 8; g /= 2) {
        const int64_t rows = (int64_t)g * tile_m + (int64_t)((concurrent + g - 1) / g) * tile_n;
        if (rows * K <= (int64_t)48 << 20) return g;
    }
    return 8;
}

struct EpiParams {
    int M, N, K;
    const float* sA;     // mode 0: 1 float; mode 1: [M][K/128]
    const float* sB;     // mode 0: 1 float; mode 1: [N/128][K/128]
    const float* bias;   // [N] or null
    void* D;
    // mode 0 with the output cast (QOUT): codes of D as stored, delayed
    // per-tensor scaling with the state qstate (m = qstate[qH], max|D| into
    // qstate[0])
    uint8_t* Q = nullptr;
    float* qstate = nullptr;
    int qH = 0, qfmt = 0;
};

constexpr int BM = 128;
constexpr int BK = 128;  // bytes = elements for 8-bit operands
constexpr int A_BYTES = BM * BK;

// ------------------------------------------------------------------ epilogue store
// 32 consecutive columns of one row: v[j] is column col0 + j.
template <bool OUT_BF16>
__device__ __forceinline__ void store_row32(const EpiParams& p, int row, int col0, const float (&v)[32])
{
    if (row >= p.M) return;
    if (OUT_BF16) {
        __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.D) + (int64_t)row * p.N + col0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (col0 + 8 * c + 8 <= p.N) {
                uint4 w;
                __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * c + 0], v[8 * c + 1]);
                __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * c + 2], v[8 * c + 3]);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * c + 4], v[8 * c + 5]);
                __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * c + 6], v[8 * c + 7]);
                w.x = *reinterpret_cast<uint32_t*>(&h0);
                w.y = *reinterpret_cast<uint32_t*>(&h1);
                w.z = *reinterpret_cast<uint32_t*>(&h2);
                w.w = *reinterpret_cast<uint32_t*>(&h3);
                *reinterpret_cast<uint4*>(d + 8 * c) = w;
            }
        }
    } else {
        float* d = static_cast<float*>(p.D) + (int64_t)row * p.N + col0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (col0 + 8 * c + 8 <= p.N) {
                *reinterpret_cast<float4*>(d + 8 * c) = make_float4(v[8 * c], v[8 * c + 1], v[8 * c + 2], v[8 * c + 3]);
                *reinterpret_cast<float4*>(d + 8 * c + 4) =
                    make_float4(v[8 * c + 4], v[8 * c + 5], v[8 * c + 6], v[8 * c + 7]);
            }
        }
    }
}

// Staged TMA store of one warp's 32 rows x SC columns (SC = 32 bytes of the
// output type: 16 bf16 or 8 fp32).  Each lane writes its row's 32 bytes into
// the warp's 1 KB shared buffer, then lane 0 issues a bulk tensor store; the
// tensor map clips rows and columns past the matrix.  The buffer is reused
// only after the previous store has read it (wait_group.read 0), so skipping
// a fully out-of-range store never lets a pending one be overwritten.  Writing
// whole 32-byte row segments through the TMA instead of 16-byte per-lane
// stores halves the L2 write requests and takes the stores off the LSU.
constexpr int kStageBytes = 1024;   // per epilogue warp

template <bool OUT_BF16>
__device__ __forceinline__ void stage_store(uint8_t* buf, const CUtensorMap* tmD, const float* v, int col0, int row0,
                                            int M, int N, int lane)
{
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncwarp();
    uint8_t* rowp = buf + lane * 32;
    if (OUT_BF16) {
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
            uint4 w4;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q4 + 0], v[8 * q4 + 1]);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q4 + 2], v[8 * q4 + 3]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q4 + 4], v[8 * q4 + 5]);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q4 + 6], v[8 * q4 + 7]);
            w4.x = *reinterpret_cast<uint32_t*>(&h0);
            w4.y = *reinterpret_cast<uint32_t*>(&h1);
            w4.z = *reinterpret_cast<uint32_t*>(&h2);
            w4.w = *reinterpret_cast<uint32_t*>(&h3);
            *reinterpret_cast<uint4*>(rowp + 16 * q4) = w4;
        }
    } else {
        *reinterpret_cast<float4*>(rowp) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(rowp + 16) = make_float4(v[4], v[5], v[6], v[7]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && col0 < N && row0 < M) {
        asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                         reinterpret_cast<uint64_t>(tmD)),
                     "r"(col0), "r"(row0), "r"(smem_addr(buf))
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}
// One lane's 32-byte staging row: 16 bf16 or 8 fp32 outputs.
template <bool OUT_BF16>
__device__ __forceinline__ void stage_row(uint8_t* rowp, const float* v)
{
    if (OUT_BF16) {
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
            uint4 w4;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q4 + 0], v[8 * q4 + 1]);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q4 + 2], v[8 * q4 + 3]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q4 + 4], v[8 * q4 + 5]);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q4 + 6], v[8 * q4 + 7]);
            w4.x = *reinterpret_cast<uint32_t*>(&h0);
            w4.y = *reinterpret_cast<uint32_t*>(&h1);
            w4.z = *reinterpret_cast<uint32_t*>(&h2);
            w4.w = *reinterpret_cast<uint32_t*>(&h3);
            *reinterpret_cast<uint4*>(rowp + 16 * q4) = w4;
        }
    } else {
        *reinterpret_cast<float4*>(rowp) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(rowp + 16) = make_float4(v[4], v[5], v[6], v[7]);
    }
}
// Bulk tensor store of a 32 x 32-byte staging buffer (one bulk group per call
// site's commit).
__device__ __forceinline__ void bulk_store_2d(const CUtensorMap* m, int x, int y, const uint8_t* buf)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(x), "r"(y), "r"(smem_addr(buf))
                 : "memory");
}

__device__ __forceinline__ void stage_store_drain(int lane)
{
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

// ------------------------------------------------------------------ shared layout
template <int BN, int STAGES, int NACC, int EPI_STAGE_WARPS = 0>
struct Smem {
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int BAR_OFF = STAGES * STAGE;
    static constexpr int NBARS = 2 * STAGES + 2 * NACC + 1;
    static constexpr int STG_OFF = BAR_OFF + 512;                      // epilogue staging (1 KB per warp)
    static constexpr int BYTES = STG_OFF + EPI_STAGE_WARPS * kStageBytes + 1024;   // + alignment slack
    static_assert(NBARS * 8 + 16 <= 512, "barriers and the TMEM holder fit before the staging area");
};

// Common prologue: barriers, tensor memory, early exit if the error word is set.
template <int STAGES, int NACC, int EPI_WARPS>
__device__ __forceinline__ bool gemm_setup(uint8_t* smem, int bar_off, uint32_t tmem_cols,
                                           const CUtensorMap* tmA, const CUtensorMap* tmB, uint32_t& tmem_base)
{
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + bar_off);
    uint32_t* holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2 * NACC + 1);
    __shared__ int s_skip;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        s_skip = *reinterpret_cast<volatile int*>(&g_dev_error);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars[s], 1);            // full
            mbar_init(&bars[STAGES + s], 1);   // empty
        }
        for (int b = 0; b < NACC; ++b) {
            mbar_init(&bars[2 * STAGES + b], 1);                 // accumulator full
            mbar_init(&bars[2 * STAGES + NACC + b], EPI_WARPS);  // accumulator empty
        }
        mbar_init(&bars[2 * STAGES + 2 * NACC], 1);              // drain
        fence_mbar_init();
        prefetch_tmap(tmA);
        prefetch_tmap(tmB);
    }
    __syncthreads();
    if (s_skip) return false;
    if (warp == 1) {
        tmem_alloc(holder, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem_base = *holder;
    return true;
}

// ------------------------------------------------------------------ producer
template <int BN, int STAGES>
__device__ __forceinline__ void producer_loop(uint8_t* smem, uint64_t* full, uint64_t* empty,
                                              const CUtensorMap* tmA, const CUtensorMap* tmB,
                                              const TileSched& sched, int num_tiles, int nkb)
{
    constexpr int STAGE = A_BYTES + BN * BK;
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    bool aborted = false;
    for (int t = blockIdx.x; t < num_tiles && !aborted; t += gridDim.x) {
        int mb, nb;
        sched.coords(t, mb, nb);
        for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bounded(&empty[stage], phase ^ 1u)) {
                aborted = true;
                break;
            }
            uint8_t* sa = smem + stage * STAGE;
            mbar_arrive_expect_tx(&full[stage], STAGE);
            tma_load_2d(sa, tmA, kb * BK, mb * BM, &full[stage]);
            tma_load_2d(sa + A_BYTES, tmB, kb * BK, nb * BN, &full[stage]);
            ++issued;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (aborted) {
        // wait for the copies still in flight before the CTA can exit
        int n = issued < STAGES ? issued : STAGES;
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < n; ++i) {
            if (--s < 0) {
                s = STAGES - 1;
                ph ^= 1u;
            }
            wait_drain(&full[s], ph);
        }
    }
}

// ================================================================== mode 0
// Per-tensor scales on CTA pairs (tcgen05 .cta_group::2).  A cluster of two
// CTAs computes 256 x 256 output tiles: CTA r holds A rows [128 r, 128 r + 128)
// and B rows [128 r, 128 r + 128) of the tile in its own shared memory; the
// even CTA (the leader) issues the M = 256 MMAs, which read both CTAs' shared
// memory and accumulate each CTA's 128 rows into that CTA's TMEM.  Each SM
// thus loads half of the B tile it multiplies with, which halves the B reads
// from shared memory per FLOP against one CTA per tile.
//   warp 0 (both CTAs): TMA producer into a 6-stage ring (32 KB per stage);
//     the loads of both CTAs complete on the leader's full barrier, for
//     which the leader's producer alone declares the pair's bytes.
//   warp 1: pair-wide TMEM allocation (512 columns: two 256-column
//     accumulators); in the leader one thread issues the MMAs and commits,
//     multicast to both CTAs, the ring's empty and the accumulators' full
//     barriers.
//   warps 2-5 (both CTAs): epilogue of the CTA's 128 rows, through 1 KB
//     per-warp shared-memory buffers and bulk tensor stores; each warp
//     releases an accumulator by arriving on the leader's barrier.
// Every thread of both CTAs reaches both cluster barriers: the skip decision
// taken from the error word is the leader's, read by the peer, and no role
// leaves before the final one.  Before a CTA may leave, its producer waits
// for the last release of every ring stage and the leader's MMA thread for
// the last release of both accumulators, so no multicast commit or remote
// arrival is still in flight into a CTA that has exited.
// Measured against one CTA per 128 x 224 tile, bit-identical output and
// 3503 against 3321 TFLOP/s at 16384 x 14336 x 4096, 3494 against 3283 at
// 8192^3; a 256 x 224 pair tile with 7 stages ran at 3362.
constexpr int kPairBN = 256;
constexpr int kPairStages = 6;
using PairSmem = Smem<kPairBN / 2, kPairStages, 2, 16>;  // per epilogue warp: four 1 KB staging buffers

__device__ __forceinline__ bool wait_bounded_cluster(uint64_t* bar, uint32_t parity)
{
    return wait_bounded_err_cluster(bar, parity, &g_dev_error);
}

// LAYOUT bit 0: A MN-major, bit 1: B MN-major (compile-time, so the
// K-major instantiation issues its MMAs from hoisted descriptors).
// QOUT (bf16 output only): the epilogue also casts the output, as stored in
// bf16, to FP8 with the delayed per-tensor scale of p.qstate -- the codes
// fp8_quantize would produce from D -- and max-combines max|D| into
// p.qstate[0], so the next layer's cast never reads D back.
template <bool OUT_BF16, int LAYOUT, bool QOUT = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    k_gemm_tensor_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       EpiParams p, uint32_t idesc, TileSched sched, const __grid_constant__ CUtensorMap tmD,
                       const __grid_constant__ CUtensorMap tmQ)
{
    pdl_enter();
    constexpr int BN = kPairBN, BH = BN / 2, STAGES = kPairStages;
    using L = PairSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* afull = empty + STAGES;
    uint64_t* aempty = afull + 2;
    uint64_t* drain = aempty + 2;
    uint32_t* holder = reinterpret_cast<uint32_t*>(drain + 1);
    constexpr uint32_t TMEM_COLS = 2 * BN;
    static_assert(TMEM_COLS <= 512, "two accumulators must fit in tensor memory");
    __shared__ int s_skip;
    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool a_mn = (LAYOUT & 1) != 0, b_mn = (LAYOUT & 2) != 0;   // MN-major operands

    if (threadIdx.x == 0) {
        s_skip = rank == 0 ? *reinterpret_cast<volatile int*>(&g_dev_error) : 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);            // the leader's expect_tx arrival (both CTAs' bytes)
            mbar_init(&empty[s], 1);           // the leader's multicast commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&afull[b], 1);           // the leader's multicast commit
            mbar_init(&aempty[b], 8);          // four epilogue warps of each CTA (used in the leader)
        }
        mbar_init(drain, 1);
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    __syncthreads();
    cluster_sync_all();                        // both CTAs' barriers initialised, the leader's flag written
    int skip = s_skip;
    if (rank != 0) skip = (int)ld_shared_cluster_u32(cluster_map(smem_addr(&s_skip), 0));
    cluster_sync_all();                        // the flag is read before either CTA may leave
    if (skip) return;                          // the same decision in both CTAs
    if (warp == 1) {
        tmem_alloc_pair(holder, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *holder;

    const int num_tiles = sched.num_m * sched.num_n;
    const int nkb = (p.K + BK - 1) / BK;
    const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

    if (warp == 0) {
        if (lane == 0) {
            constexpr uint32_t PAIR_TX = 2u * (uint32_t)L::STAGE;   // bytes landing per stage in the pair
            const uint32_t full0 = cluster_map(smem_addr(full), 0);
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            bool aborted = false;
            for (int t = cid; t < num_tiles && !aborted; t += ncl) {
                int mb, nb;
                sched.coords(t, mb, nb);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!wait_bounded_cluster(&empty[stage], phase ^ 1u)) {
                        aborted = true;
                        break;
                    }
                    uint8_t* sa = smem + stage * L::STAGE;
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], PAIR_TX);
                    const int ar = mb * 2 * BM + (int)rank * BM, br = nb * BN + (int)rank * BH;
                    // K-major boxes are (k, row); MN-major ones (row, k)
                    tma_load_2d_pair(sa, &tmA, a_mn ? ar : kb * BK, a_mn ? kb * BK : ar, full0 + 8u * stage);
                    tma_load_2d_pair(sa + A_BYTES, &tmB, b_mn ? br : kb * BK, b_mn ? kb * BK : br,
                                     full0 + 8u * stage);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!aborted) {
                for (int i = 0; i < STAGES; ++i) {     // every stage's last release has landed
                    if (!wait_bounded_cluster(&empty[stage], phase ^ 1u)) break;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            } else if (rank == 0) {
                // the pair's copies still in flight complete on the leader's barriers
                int n = issued < STAGES ? issued : STAGES;
                int s = stage;
                uint32_t ph = phase;
                for (int i = 0; i < n; ++i) {
                    if (--s < 0) {
                        s = STAGES - 1;
                        ph ^= 1u;
                    }
                    wait_drain(&full[s], ph);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            int stage = 0, lt = 0;
            uint32_t phase = 0;
            bool aborted = false;
            for (int t = cid; t < num_tiles && !aborted; t += ncl, ++lt) {
                const int b = lt & 1;
                const uint32_t u = (uint32_t)(lt >> 1);
                if (!wait_bounded_cluster(&aempty[b], (u & 1u) ^ 1u)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(b * BN);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!wait_bounded_cluster(&full[stage], phase)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(smem + stage * L::STAGE);
                    // K = 32 slice k: 32 bytes further along a K-major row, or
                    // 32 rows (4 atoms, 4 KB) further down an MN-major tile
                    // (start address in 16-byte units: +2 or +256)
                    const uint64_t da = a_mn ? sdesc_mn_sw128(sa) : sdesc_kmajor_sw128(sa);
                    const uint64_t db = b_mn ? sdesc_mn_sw128(sa + A_BYTES) : sdesc_kmajor_sw128(sa + A_BYTES);
                    constexpr uint64_t sta = a_mn ? 256 : 2, stb = b_mn ? 256 : 2;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_pair_f8f6f4(d, da + sta * k, db + stb * k, idesc, (kb | k) != 0 ? 1u : 0u);
                    mma_pair_commit(&empty[stage], 3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!aborted) mma_pair_commit(&afull[b], 3);
            }
            if (!aborted) {
                for (int j = 0; j < 2; ++j) {           // both accumulators' last releases have landed
                    const int l2 = lt + j;
                    if (!wait_bounded_cluster(&aempty[l2 & 1], ((uint32_t)(l2 >> 1) & 1u) ^ 1u)) break;
                }
            } else {
                mma_pair_commit(drain, 1);              // completes once every issued MMA is done
                wait_drain(drain, 0);
            }
        }
    } else {
        const int quarter = warp & 3;       // the TMEM lane quarter this warp may read
        const float scale = __ldg(p.sA) * __ldg(p.sB);
        // four 1 KB staging buffers per warp: a chunk's 32 output columns (two
        // bf16 or four fp32 row segments of 32 bytes) and, with QOUT, its codes
        uint8_t* stg = smem + L::STG_OFF + (warp - 2) * 4 * kStageBytes;
        uint8_t* qstg = stg + 2 * kStageBytes;
        constexpr int SC = OUT_BF16 ? 16 : 8;   // columns per 32-byte staged row segment
        const uint32_t aempty0 = cluster_map(smem_addr(aempty), 0);
        static_assert(!QOUT || OUT_BF16, "the output cast takes the bf16 output");
        float qm = 1.0f;
        uint32_t qmax = 0;                  // packed pair of |bf16| maxima
        if constexpr (QOUT) qm = p.qstate[p.qH];
        int lt = 0;
        for (int t = cid; t < num_tiles; t += ncl, ++lt) {
            const int b = lt & 1;
            const uint32_t u = (uint32_t)(lt >> 1);
            const bool ok = wait_bounded_cluster(&afull[b], u & 1u);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            int mb, nb;
            sched.coords(t, mb, nb);
            const int row0 = mb * 2 * BM + (int)rank * BM + quarter * 32;
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * BN);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + (uint32_t)c, r);
                tmem_ld_wait();
                float v[32];
                const int colc = nb * BN + c;
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * scale;
                if (p.bias) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (colc + j < p.N) v[j] += __ldg(p.bias + colc + j);
                }
                // the previous chunk's bulk stores have read their buffers
                // (one wait per chunk: they had the whole chunk to do so)
                if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                __syncwarp();
#pragma unroll
                for (int h = 0; h < 32 / SC; ++h) stage_row<OUT_BF16>(stg + h * kStageBytes + 32 * lane, v + h * SC);
                if constexpr (QOUT) {
                    // the codes of this lane's 32 outputs as rounded to bf16:
                    // q = sat_rne(fp32(bf16(v)) * m), as the cast of D would
                    uint32_t w[8];
                    const int row = row0 + lane;
                    // only outputs inside the matrix enter the maximum (a row
                    // past M holds the bias; columns past N hold zeros)
                    const uint32_t keep = row < p.M ? 0x7FFF7FFFu : 0u;
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        __nv_bfloat162 h0 = __floats2bfloat162_rn(v[j], v[j + 1]);
                        __nv_bfloat162 h1 = __floats2bfloat162_rn(v[j + 2], v[j + 3]);
                        const uint32_t b0 = *reinterpret_cast<uint32_t*>(&h0), b1 = *reinterpret_cast<uint32_t*>(&h1);
                        qmax = __vmaxu2(qmax, __vmaxu2(b0 & keep, b1 & keep));
                        const float f0 = __fmul_rn(__uint_as_float(b0 << 16), qm);
                        const float f1 = __fmul_rn(__uint_as_float(b0 & 0xFFFF0000u), qm);
                        const float f2 = __fmul_rn(__uint_as_float(b1 << 16), qm);
                        const float f3 = __fmul_rn(__uint_as_float(b1 & 0xFFFF0000u), qm);
                        w[j / 4] = p.qfmt == kE4M3 ? (cvt_e4m3x2(f0, f1) | (cvt_e4m3x2(f2, f3) << 16))
                                                   : (cvt_e5m2x2(f0, f1) | (cvt_e5m2x2(f2, f3) << 16));
                    }
                    // the warp's 32 rows x 32 codes: whole 32-byte rows
                    *reinterpret_cast<uint4*>(qstg + 32 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4*>(qstg + 32 * lane + 16) = make_uint4(w[4], w[5], w[6], w[7]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                // one lane issues the chunk's bulk tensor stores (the tensor
                // maps clip rows past M and columns past N)
                if (lane == 0 && row0 < p.M) {
#pragma unroll
                    for (int h = 0; h < 32 / SC; ++h)
                        if (colc + h * SC < p.N) bulk_store_2d(&tmD, colc + h * SC, row0, stg + h * kStageBytes);
                    if (QOUT && colc < p.N) bulk_store_2d(&tmQ, colc, row0, qstg);
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(aempty0 + 8u * b);
        }
        stage_store_drain(lane);
        if constexpr (QOUT) {
            uint32_t a = max(qmax & 0xFFFFu, qmax >> 16) << 16;
            a = __reduce_max_sync(0xFFFFFFFFu, a);
            if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(p.qstate), a);
        }
    }
    __syncthreads();
    cluster_sync_all();                        // nothing is pending into either CTA any more
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ================================================================== mode 1
// Fine-grained scales with per-K-block promotion.  One CTA per 128 x 256
// tile; the MMAs of each 128-wide K block write a fresh fp32 partial into one
// of two 256-column TMEM buffers, and eight epilogue warps promote it into
// fp32 registers (acc += partial x scale) while the MMAs of the next K block
// run into the other buffer.
//   warp 0: TMA producer (48 KB per stage, 4 stages);
//   warp 1: TMEM allocation (512 columns); one thread issues the MMAs and
//     one commit per K block, on the buffer's full barrier;
//   warp 2: stage releaser.  The buffer's full barrier fires only after the
//     MMAs that read the K block's shared-memory stage have completed, so
//     one thread waits on it and frees the stage for the producer; the MMA
//     thread then needs a single commit per K block.  It also counts in the
//     buffer's release, so the MMAs never run two phases ahead of it;
//   warp 3: idle (it completes warpgroup 0);
//   warps 4 .. 11: warp w reads TMEM lane quarter w % 4 and owns the 128
//     columns (w - 4) / 4 of the tile.  Per K block it copies them out in two
//     waits of two 32-column chunks, releases the buffer after the second
//     wait, then does the FMAs (two columns per packed f32x2 FMA).
// With two buffers the MMAs run one K block ahead of the promotion, so the
// promotion of a K block (wake-up, the two waits, the release) and the MMA
// thread's turnaround between K blocks both have to fit in one K block of
// MMAs.  128 accumulators plus 64 copied registers a thread exceed the 168
// registers of a 12-warp CTA, so the warpgroups re-split the register file
// (setmaxnreg): warpgroup 0 drops to kPromoCtlRegs, the two epilogue
// warpgroups rise to kPromoEpiRegs.
// SM selects the scale layouts:
//   1: A in 1x128 tiles sA[M][K/128], B in 128x128 blocks sB[ceil(N/128)][K/128]:
//      a warp's 128 columns are one weight block, so its scale is one number
//      per K block, sA[row][kb] * sB[block][kb];
//   3: both operands in tiles along K with K-block-major scales sA[K/128][M],
//      sB[K/128][N] (the transposed codes of column-tile quantisation): per
//      element sA[kb][row] * sB[kb][col]; the warp's column scales reach its
//      lanes through a double-buffered shared-memory slot.
// Measured, per-row scales, bf16 out, TFLOP/s at 4096^3 / 16384 x 14336 x
// 4096 / 8192^3, outputs bit-identical throughout.  This kernel, through the
// library: 1848-1871 / 2080-2133 / 2270-2351.  Timed side by side in one
// process (the first row is this design while an epilogue warp still freed
// the stages):
//   one CTA per 128 x 256 tile                               1832 2188 2421
//   the same on CTA pairs (256 x 256, cluster-wide handshake) 1716 2115 2348
//   128 x 192 tiles, all 96 columns copied in one wait       1651 1902 1985
// From separate runs:
//   256 x 128 CTA-pair tiles, four 128-column buffers        1335 1440 1525
//   ten warps, 168 registers, four serial 32-column copies   1633-1676 1961-2002 2103-2182
// The epilogue's waits stay at CTA scope; with the same handshake across a
// CTA pair, a release arrival at cluster scope on every K block put a fence
// behind each K block's scale loads (ncu: membar the dominant stall, 12 %
// tensor-pipe activity).
constexpr int kPromoBN = 256;
constexpr int kPromoStages = 4;
constexpr int kPromoEpi0 = 4;                        // first epilogue warp (warpgroup 1)
constexpr int kPromoEpi = 8;                         // epilogue warps
constexpr int kPromoThreads = 32 * (kPromoEpi0 + kPromoEpi);
constexpr int kPromoCtlRegs = 48;                    // warpgroup 0 after the re-split
constexpr int kPromoEpiRegs = 224;                   // epilogue warpgroups after the re-split
// registers a thread must be launched with for the re-split to fit
constexpr int kPromoLaunchRegs = (128 * kPromoCtlRegs + 32 * kPromoEpi * kPromoEpiRegs + kPromoThreads - 1) / kPromoThreads;
using PromoSmem = Smem<kPromoBN, kPromoStages, 2>;

// acc[0..1] += x[0..1] * s[0..1], both lanes rounded once (the packed
// f32x2 FMA: bit-identical to two fmaf calls, half the issue slots)
__device__ __forceinline__ void fma2(float& a0, float& a1, float x0, float x1, float s0, float s1)
{
    const float2 r = __ffma2_rn(make_float2(x0, x1), make_float2(s0, s1), make_float2(a0, a1));
    a0 = r.x;
    a1 = r.y;
}

// warpgroup register re-split (every thread of the warpgroup executes it)
template <int N>
__device__ __forceinline__ void regs_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <bool OUT_BF16, int SM>
__global__ void __launch_bounds__(kPromoThreads, 1)
    k_gemm_promote(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   EpiParams p, uint32_t idesc, TileSched sched)
{
    pdl_enter();
    constexpr int BN = kPromoBN, STAGES = kPromoStages, NB = 2, EPI = kPromoEpi;
    constexpr int COLS = 4 * BN / EPI;       // columns per epilogue warp (128)
    constexpr int NLD = COLS / 32;           // 32-column copies per K block
    constexpr int CPL = COLS / 32;           // column scales per lane (SM 3)
    static_assert(SM == 1 || SM == 3, "scale layout");
    static_assert(COLS == 128, "a warp's columns are one weight block");
    using L = PromoSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* afull = empty + STAGES;
    uint64_t* aempty = afull + NB;
    uint64_t* drain = aempty + NB;
    constexpr uint32_t TMEM_COLS = 512;
    __shared__ __align__(16) float colbuf[SM == 3 ? EPI : 1][2][SM == 3 ? COLS : 4];

    uint32_t tmem_base;
    // a buffer is released by the epilogue warps and the stage releaser
    if (!gemm_setup<STAGES, NB, EPI + 1>(smem, L::BAR_OFF, TMEM_COLS, &tmA, &tmB, tmem_base)) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_tiles = sched.num_m * sched.num_n;
    const int nkb = p.K / BK;

    if (warp < kPromoEpi0) regs_dec<kPromoCtlRegs>();
    if (warp == 0) {
        if (lane == 0) producer_loop<BN, STAGES>(smem, full, empty, &tmA, &tmB, sched, num_tiles, nkb);
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool aborted = false;
            for (int t = blockIdx.x; t < num_tiles && !aborted; t += gridDim.x) {
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int b = it % NB;
                    const uint32_t u = (uint32_t)(it / NB);
                    if (!wait_bounded(&aempty[b], (u & 1u) ^ 1u) || !wait_bounded(&full[stage], phase)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + (uint32_t)(b * BN);
                    const uint32_t sa = smem_addr(smem + stage * L::STAGE);
                    const uint64_t da = sdesc_kmajor_sw128(sa);
                    const uint64_t db = sdesc_kmajor_sw128(sa + A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k) mma_f8f6f4(d, da + 2 * k, db + 2 * k, idesc, k != 0 ? 1u : 0u);
                    mma_commit(&afull[b]);   // also releases the stage (through warp 2)
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (aborted) {
                mma_commit(drain);
                wait_drain(drain, 0);
            }
        }
    } else if (warp == 2) {
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int b = it % NB;
                    if (!wait_bounded(&afull[b], (uint32_t)(it / NB) & 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive(&empty[it % STAGES]);
                    mbar_arrive(&aempty[b]);
                }
            }
        }
    } else if (warp >= kPromoEpi0) {
        regs_inc<kPromoEpiRegs>();
        const int quarter = warp & 3;
        const int part = (warp - kPromoEpi0) >> 2;  // column half of the tile
        const int ew = warp - kPromoEpi0;
        const int ksb = p.K / BK;                   // scale blocks along K
        const int nblk = (p.N + 127) / 128;         // weight blocks along N
        int it = 0;
        bool ok_all = true;
        for (int t = blockIdx.x; t < num_tiles && ok_all; t += gridDim.x) {
            int mb, nb;
            sched.coords(t, mb, nb);
            const int row = mb * BM + quarter * 32 + lane;
            const int rowc = row < p.M ? row : p.M - 1;   // clamp for the scale reads
            const int col0 = nb * BN + part * COLS;
            float acc[COLS];
#pragma unroll
            for (int j = 0; j < COLS; ++j) acc[j] = 0.0f;
            // SM 1: sc = the K block's combined scale (one weight block per warp).
            // SM 3: ra = the row's scale, cb = this lane's CPL column scales.
            const float* sa_row = p.sA + (int64_t)rowc * ksb;
            int wblk = nb * (BN / 128) + part;
            wblk = wblk < nblk ? wblk : nblk - 1;
            const float* sb_row = p.sB + (int64_t)wblk * ksb;
            int cl = col0 + CPL * lane;
            cl = cl < p.N - CPL ? cl : p.N - CPL;
            float sc = 0.0f, ra = 0.0f;
            float cb[CPL];
            if constexpr (SM == 1) {
                sc = __ldg(sa_row) * __ldg(sb_row);
            } else {
                ra = __ldg(p.sA + rowc);
#pragma unroll
                for (int j = 0; j < CPL; ++j) cb[j] = __ldg(p.sB + cl + j);
            }
            for (int kb = 0; kb < nkb; ++kb) {
                const int kn = kb + 1 < nkb ? kb + 1 : kb;
                float na = 0.0f, nbv = 0.0f;
                float ncb[CPL];
                [[maybe_unused]] const float* cbuf = nullptr;
                if constexpr (SM == 1) {
                    na = __ldg(sa_row + kn);
                    nbv = __ldg(sb_row + kn);
                } else {
                    na = __ldg(p.sA + (int64_t)kn * p.M + rowc);
#pragma unroll
                    for (int j = 0; j < CPL; ++j) ncb[j] = __ldg(p.sB + (int64_t)kn * p.N + cl + j);
                    float* w = colbuf[ew][kb & 1];
#pragma unroll
                    for (int j = 0; j < CPL; ++j) w[CPL * lane + j] = cb[j];
                    __syncwarp();
                    cbuf = w;
                }
                const int b = it % NB;
                const uint32_t u = (uint32_t)(it / NB);
                ++it;
                const bool ok = wait_bounded(&afull[b], u & 1u);
                if (!__all_sync(0xFFFFFFFFu, ok)) {
                    ok_all = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * BN + part * COLS);
                // Per-column scales (SM 3): the four 32-column copies are
                // pipelined with the FMAs -- the copy of chunk g + 1 is in
                // flight while chunk g is promoted, and the buffer is released
                // right after the last copy lands (two 32-register copy
                // buffers beside the 128 accumulators): 3 % faster at 8192^3
                // and 14336 x 4096 x 16384.
                auto promote32 = [&](float* a, const uint32_t (&r)[32], int chunk) {
                    if constexpr (SM == 1) {
#pragma unroll
                        for (int c = 0; c < 32; c += 2)
                            fma2(a[c], a[c + 1], __uint_as_float(r[c]), __uint_as_float(r[c + 1]), sc, sc);
                    } else {
                        // ra x column scale, two columns per packed f32x2 multiply
                        const float* s32 = cbuf + 32 * chunk;
                        const float2 ra2 = make_float2(ra, ra);
#pragma unroll
                        for (int c = 0; c < 32; c += 4) {
                            const float4 s4 = *reinterpret_cast<const float4*>(s32 + c);
                            const float2 s01 = __fmul2_rn(ra2, make_float2(s4.x, s4.y));
                            const float2 s23 = __fmul2_rn(ra2, make_float2(s4.z, s4.w));
                            fma2(a[c], a[c + 1], __uint_as_float(r[c]), __uint_as_float(r[c + 1]), s01.x, s01.y);
                            fma2(a[c + 2], a[c + 3], __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]), s23.x,
                                 s23.y);
                        }
                    }
                };
                if constexpr (SM == 3) {
                    uint32_t ra_[32], rb_[32];
                    tmem_ld_32x32b_x32(taddr, ra_);
                    tmem_ld_wait();
#pragma unroll
                    for (int g = 0; g < NLD; ++g) {
                        if (g + 1 < NLD) tmem_ld_32x32b_x32(taddr + 32 * (g + 1), (g & 1) ? ra_ : rb_);
                        promote32(acc + 32 * g, (g & 1) ? rb_ : ra_, g);
                        if (g + 1 < NLD) tmem_ld_wait();
                        if (g + 2 == NLD) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&aempty[b]);
                        }
                    }
                } else {
                    // per-row scales: two copies per wait, then their FMAs
                    // (the pipelined order above measured 1.5 % slower here)
#pragma unroll
                    for (int g = 0; g < NLD / 2; ++g) {
                        uint32_t r[2][32];
                        tmem_ld_32x32b_x32(taddr + 64 * g, r[0]);
                        tmem_ld_32x32b_x32(taddr + 64 * g + 32, r[1]);
                        tmem_ld_wait();
                        if (g == NLD / 2 - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&aempty[b]);
                        }
                        promote32(acc + 64 * g, r[0], 2 * g);
                        promote32(acc + 64 * g + 32, r[1], 2 * g + 1);
                    }
                }
                if constexpr (SM == 1) {
                    sc = na * nbv;
                } else {
                    ra = na;
#pragma unroll
                    for (int j = 0; j < CPL; ++j) cb[j] = ncb[j];
                }
            }
            if (!ok_all) break;
#pragma unroll
            for (int h = 0; h < NLD; ++h) {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    v[j] = acc[32 * h + j];
                    if (p.bias && col0 + 32 * h + j < p.N) v[j] += __ldg(p.bias + col0 + 32 * h + j);
                }
                store_row32<OUT_BF16>(p, row, col0 + 32 * h, v);
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// Registers a thread of `kern` is launched with (the compiled count, in the
// allocation unit of 8), queried once per kernel.
static cudaError_t launch_regs(const void* kern, int* regs)
{
    static std::mutex mu;
    static const void* done_kern[16];
    static int done_regs[16];
    static int n_done = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done_kern[i] == kern) {
            *regs = done_regs[i];
            return cudaSuccess;
        }
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    *regs = (fa.numRegs + 7) & ~7;
    if (n_done < 16) {
        done_kern[n_done] = kern;
        done_regs[n_done] = *regs;
        ++n_done;
    }
    return cudaSuccess;
}

// launches the promotion kernel for scale layout SM (1 or 3)
template <int SM>
static cudaError_t launch_promote(const GemmArgs& g, const EpiParams& p, cudaStream_t st, int sms, const char** why)
{
    constexpr int BN = kPromoBN;
    CUtensorMap ta, tb;
    if (!encode_tmap_2d(&ta, 0, g.A, g.K, g.M, 128u, BM) || !encode_tmap_2d(&tb, 0, g.B, g.K, g.N, 128u, BN)) {
        *why = "cuTensorMapEncodeTiled failed";
        return cudaErrorInvalidValue;
    }
    TileSched sched{(int)((g.M + BM - 1) / BM), (int)((g.N + BN - 1) / BN), 16};
    const int tiles = sched.num_m * sched.num_n;
    uint32_t idesc = 0;
    idesc |= 1u << 4;
    idesc |= (uint32_t)g.a_format << 7;
    idesc |= (uint32_t)g.b_format << 10;
    idesc |= (uint32_t)(BN >> 3) << 17;
    idesc |= (uint32_t)(BM >> 4) << 24;
    const int smem = PromoSmem::BYTES;
    auto kern = g.d_dtype == kBF16 ? k_gemm_promote<true, SM> : k_gemm_promote<false, SM>;
    // the warpgroups' setmaxnreg shares must fit in what the CTA is launched
    // with, or the raising warpgroups would wait for registers forever
    int regs = 0;
    cudaError_t e = launch_regs(reinterpret_cast<const void*>(kern), &regs);
    if (e != cudaSuccess) return e;
    if (regs < kPromoLaunchRegs) {
        *why = "promotion kernel compiled with fewer registers than its warpgroup split needs";
        return cudaErrorInvalidConfiguration;
    }
    e = smem_attr_once(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    const int grid = tiles < sms ? tiles : sms;
    launch_k(kern, grid, kPromoThreads, smem, st, ta, tb, p, idesc, sched);
    return cudaGetLastError();
}

// ================================================================== mode 2
// MX-32 block scaling on the block-scaled tensor-core path
// (tcgen05.mma kind::mxf8f6f4.block_scale, E8M0 scale factors).  The ring
// stages carry only the A and B tiles.  The scale factors reach tensor
// memory on their own path: a warpgroup of writers (one warp per TMEM lane
// quarter) reads the 512-byte scale chunks of eight K blocks at a time (one
// per 128 rows x 128 K of A, and of each 128 rows of B; contiguous in the
// tiled scale layout of fp8_quantize) from global memory into registers and
// writes them with tcgen05.st into one of two scale-factor slots, each
// quarter the same 32 lanes x 4 columns per chunk (the layout the
// replicating 32x128b.warpx4 copy gives).  A slot is rewritten only after
// the MMAs that read it have completed (one commit per group), so the MMA
// queue holds MMAs only and the writers run up to a group ahead.  MMA j
// (K = 32 slice j of a K block) selects byte j of each scale word through
// the descriptor's scale-factor ids.
template <int BN, int STAGES, int NACC>
struct MxLayout {
    static constexpr int CH = BN / 128;                  // 128-row scale chunks of B
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int BAR_OFF = STAGES * STAGE;
    static constexpr int SFBAR_OFF = BAR_OFF + 256;      // scale-factor slot full[2], empty[2]
    static constexpr int STG_OFF = BAR_OFF + 512;        // epilogue staging, 1 KB per warp
    static constexpr int BYTES = STG_OFF + 8 * kStageBytes + 1024;
    static constexpr int SF_G = 8;                       // K blocks per scale-factor group
    static constexpr int SF_KB_COLS = 16;                // TMEM columns per K block: A 4, B 4 per chunk, padding
    static constexpr int SF_COL0 = NACC * BN;            // first scale-factor TMEM column
    static constexpr int SF_SLOT_COLS = SF_G * SF_KB_COLS;
    static_assert(4 * (1 + CH) <= SF_KB_COLS, "scale columns of a K block");
    static_assert(SF_COL0 + 2 * SF_SLOT_COLS <= 512, "tensor memory budget");
    static_assert(2 * STAGES + 2 * NACC + 2 <= 32, "barriers below the scale-factor barriers");
};

struct MxParams {
    const uint8_t* sfa;   // tiled E8M0 scales of A
    const uint8_t* sfb;   // tiled E8M0 scales of B
    int kb128;            // K / 128
    int nchunks_b;        // N / 128
};

// warpgroups: 0 producer / MMA (two idle warps), 1-2 epilogue (two warps per
// lane quarter), 3 scale-factor writers.  Registers are re-split with
// setmaxnreg: 56 / 184 / 80 of the 128 a thread is launched with.
constexpr int kMxThreads = 512;
constexpr int kMxCtlRegs = 56, kMxEpiRegs = 184, kMxSfRegs = 80;
constexpr int kMxLaunchRegs = (128 * kMxCtlRegs + 256 * kMxEpiRegs + 128 * kMxSfRegs + kMxThreads - 1) / kMxThreads;

template <int BN, int STAGES, int NACC, bool OUT_BF16>
__global__ void __launch_bounds__(kMxThreads, 1)
    k_gemm_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, EpiParams p,
              uint32_t idesc, TileSched sched, MxParams mx, const __grid_constant__ CUtensorMap tmD)
{
    pdl_enter();
    constexpr int EPI = 8;
    using L = MxLayout<BN, STAGES, NACC>;
    constexpr int G = L::SF_G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* afull = empty + STAGES;
    uint64_t* aempty = afull + NACC;
    uint64_t* drain = aempty + NACC;
    uint64_t* sf_full = reinterpret_cast<uint64_t*>(smem + L::SFBAR_OFF);
    uint64_t* sf_empty = sf_full + 2;
    constexpr uint32_t TMEM_COLS = 512;

    if (threadIdx.x == 0) {
        // initialised before gemm_setup's fence and barrier
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sf_full[s], 4);     // the four writer warps
            mbar_init(&sf_empty[s], 1);    // the MMA thread's commit
        }
    }
    uint32_t tmem_base;
    if (!gemm_setup<STAGES, NACC, EPI>(smem, L::BAR_OFF, TMEM_COLS, &tmA, &tmB, tmem_base)) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_tiles = sched.num_m * sched.num_n;
    const int nkb = p.K / BK;

    if (warp < 4) {
        regs_dec<kMxCtlRegs>();
        if (warp == 0 && lane == 0) {
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            bool aborted = false;
            for (int t = blockIdx.x; t < num_tiles && !aborted; t += gridDim.x) {
                int mb, nb;
                sched.coords(t, mb, nb);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!wait_bounded(&empty[stage], phase ^ 1u)) {
                        aborted = true;
                        break;
                    }
                    uint8_t* sa = smem + stage * L::STAGE;
                    mbar_arrive_expect_tx(&full[stage], (uint32_t)L::STAGE);
                    tma_load_2d(sa, &tmA, kb * BK, mb * BM, &full[stage]);
                    tma_load_2d(sa + A_BYTES, &tmB, kb * BK, nb * BN, &full[stage]);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (aborted) {
                int n = issued < STAGES ? issued : STAGES;
                int s = stage;
                uint32_t ph = phase;
                for (int i = 0; i < n; ++i) {
                    if (--s < 0) {
                        s = STAGES - 1;
                        ph ^= 1u;
                    }
                    wait_drain(&full[s], ph);
                }
            }
        } else if (warp == 1 && lane == 0) {
            int stage = 0, lt = 0, cw = 0;
            uint32_t phase = 0;
            bool aborted = false;
            for (int t = blockIdx.x; t < num_tiles && !aborted; t += gridDim.x, ++lt) {
                const int b = lt % NACC;
                const uint32_t u = (uint32_t)(lt / NACC);
                if (!wait_bounded(&aempty[b], (u & 1u) ^ 1u)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(b * BN);
                uint32_t sf0 = 0;
                for (int kb = 0; kb < nkb; ++kb) {
                    const int j = kb % G;
                    if (j == 0) {
                        if (!wait_bounded(&sf_full[cw & 1], (uint32_t)(cw >> 1) & 1u)) {
                            aborted = true;
                            break;
                        }
                        tc_fence_after();
                        sf0 = tmem_base + (uint32_t)(L::SF_COL0 + (cw & 1) * L::SF_SLOT_COLS);
                    }
                    if (!wait_bounded(&full[stage], phase)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(smem + stage * L::STAGE);
                    const uint32_t sfa_t = sf0 + (uint32_t)(j * L::SF_KB_COLS);
                    const uint32_t sfb_t = sfa_t + 4;
                    const uint64_t da = sdesc_kmajor_sw128(sa);
                    const uint64_t db = sdesc_kmajor_sw128(sa + A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_mxf8f6f4(d, da + 2 * k, db + 2 * k, idesc | ((uint32_t)k << 29) | ((uint32_t)k << 4),
                                     sfa_t, sfb_t, (kb | k) != 0 ? 1u : 0u);
                    mma_commit(&empty[stage]);
                    if (j == G - 1 || kb == nkb - 1) {
                        mma_commit(&sf_empty[cw & 1]);   // the group's MMAs have read its slot
                        ++cw;
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!aborted) mma_commit(&afull[b]);
            }
            if (aborted) {
                mma_commit(drain);
                wait_drain(drain, 0);
            }
        }
    } else if (warp < 12) {
        regs_inc<kMxEpiRegs>();
        // two warps per TMEM lane quarter split the BN columns
        constexpr int COLS = BN / 2;
        const int quarter = warp & 3;
        const int part = (warp - 4) >> 2;
        uint8_t* stg = smem + L::STG_OFF + (warp - 4) * kStageBytes;
        constexpr int SC = OUT_BF16 ? 16 : 8;
        int lt = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++lt) {
            const int b = lt % NACC;
            const uint32_t u = (uint32_t)(lt / NACC);
            const bool ok = wait_bounded(&afull[b], u & 1u);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            int mb, nb;
            sched.coords(t, mb, nb);
            const int row0 = mb * BM + quarter * 32;
            const uint32_t taddr =
                tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * BN + part * COLS);
            // The whole slice comes out in one wait and the accumulator is
            // released before any conversion or store: with one accumulator
            // the next tile's MMAs wait for this release, not for the stores.
            uint32_t r[COLS / 32][32];
#pragma unroll
            for (int c = 0; c < COLS / 32; ++c) tmem_ld_32x32b_x32(taddr + (uint32_t)(32 * c), r[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&aempty[b]);
#pragma unroll
            for (int c = 0; c < COLS / 32; ++c) {
                float v[32];
                const int col0 = nb * BN + part * COLS + 32 * c;
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[c][j]);
                if (p.bias) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j < p.N) v[j] += __ldg(p.bias + col0 + j);
                }
#pragma unroll
                for (int h = 0; h < 32 / SC; ++h)
                    stage_store<OUT_BF16>(stg, &tmD, v + h * SC, col0 + h * SC, row0, p.M, p.N, lane);
            }
        }
        stage_store_drain(lane);
    } else {
        regs_dec<kMxSfRegs>();
        // scale-factor writers: warp (12 + q) fills lane quarter q of every
        // group's slot, four K blocks per round of loads
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int cpt = (nkb + G - 1) / G;                   // groups per tile
        int wi = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            int mb, nb;
            sched.coords(t, mb, nb);
            int nch = mx.nchunks_b - nb * L::CH;
            nch = nch < L::CH ? nch : L::CH;
            for (int g = 0; g < cpt; ++g, ++wi) {
                const int slot = wi & 1;
                const bool okw = wait_bounded(&sf_empty[slot], ((uint32_t)(wi >> 1) & 1u) ^ 1u);
                if (!__all_sync(0xFFFFFFFFu, okw)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col0 = tmem_base + lane_base + (uint32_t)(L::SF_COL0 + slot * L::SF_SLOT_COLS);
#pragma unroll
                for (int h = 0; h < G / 4; ++h) {
                    uint32_t r[4][16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int kb = g * G + h * 4 + i;
#pragma unroll
                        for (int c = 0; c < 16; ++c) r[i][c] = 0u;
                        if (kb < nkb) {
                            const uint4 a = __ldg(reinterpret_cast<const uint4*>(
                                mx.sfa + ((int64_t)mb * mx.kb128 + kb) * 512 + 16 * lane));
                            r[i][0] = a.x;
                            r[i][1] = a.y;
                            r[i][2] = a.z;
                            r[i][3] = a.w;
#pragma unroll
                            for (int c = 0; c < L::CH; ++c)
                                if (c < nch) {
                                    const uint4 q = __ldg(reinterpret_cast<const uint4*>(
                                        mx.sfb + ((int64_t)(nb * L::CH + c) * mx.kb128 + kb) * 512 + 16 * lane));
                                    r[i][4 + 4 * c] = q.x;
                                    r[i][5 + 4 * c] = q.y;
                                    r[i][6 + 4 * c] = q.z;
                                    r[i][7 + 4 * c] = q.w;
                                }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (g * G + h * 4 + i < nkb)
                            tmem_st_32x32b_x16(col0 + (uint32_t)((h * 4 + i) * L::SF_KB_COLS), r[i]);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_full[slot]);
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ================================================================== self-test
// One thread waits, through the same bounded wait the GEMM kernels use, on
// an mbarrier phase that nothing completes; the wait gives up after
// limit_ns, sets the device error word and the kernel returns.  Lets the
// failure path be exercised without faulting or hanging the GPU.
__global__ void k_selftest_wait(uint64_t limit_ns, int* waited_out)
{
    pdl_enter();
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        const bool ok = wait_bounded_err(&bar, 0, &g_dev_error, limit_ns);
        *waited_out = ok ? 0 : 1;
    }
}

cudaError_t launch_selftest_wait(uint64_t limit_ns, int* waited_out, cudaStream_t st)
{
    launch_k(k_selftest_wait, 1, 32, 0, st, limit_ns, waited_out);
    return cudaGetLastError();
}

// ================================================================== K == 0
template <bool OUT_BF16>
__global__ void k_fill_bias(void* D, int64_t M, int64_t N, const float* bias)
{
    pdl_enter();
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= M * N) return;
    float v = bias ? bias[i % N] : 0.0f;
    if (OUT_BF16) static_cast<__nv_bfloat16*>(D)[i] = __float2bfloat16_rn(v);
    else static_cast<float*>(D)[i] = v;
}

// ================================================================== host
// the driver's tensor-map encoder, resolved once (thread-safe static
// initialisation); null if the driver does not provide it
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
        return nullptr;
    }();
    return fn;
}

bool encode_tmap_2d(CUtensorMap* m, int u16, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_inner,
                    uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t esz = u16 ? 2 : 1;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * esz};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(m, u16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr),
                    dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D u8 tensor [rows][inner] (inner contiguous), box box_rows x 128 bytes, 128-byte swizzle
static bool make_tmap(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows)
{
    return encode_tmap_2d(m, 0, ptr, inner, rows, 128u, box_rows);
}

// instruction descriptor, kind::f8f6f4: D fp32, A/B format, both K-major, N, M = 128
static uint32_t make_idesc(int a_fmt, int b_fmt, int n)
{
    uint32_t d = 0;
    d |= 1u << 4;                       // D format: F32
    d |= (uint32_t)a_fmt << 7;          // 0 = E4M3, 1 = E5M2
    d |= (uint32_t)b_fmt << 10;
    d |= (uint32_t)(n >> 3) << 17;      // N / 8
    d |= (uint32_t)(BM >> 4) << 24;     // M / 16
    return d;
}

// instruction descriptor, kind::mxf8f6f4.block_scale: A/B format, both
// K-major, N, E8M0 scale factors, M = 128; the scale-factor byte ids
// (bits 4-5 for B, 29-30 for A) are or-ed in per MMA
static uint32_t make_idesc_mx(int a_fmt, int b_fmt, int n)
{
    uint32_t d = 0;
    d |= (uint32_t)a_fmt << 7;
    d |= (uint32_t)b_fmt << 10;
    d |= (uint32_t)(n >> 3) << 17;
    d |= 1u << 23;                      // scale factors: UE8M0
    d |= (uint32_t)(BM >> 4) << 24;
    return d;
}

// 2-D tensor map of the output D [M][N] for the staged epilogue stores: box
// 32 rows x 32 bytes, no swizzle (stores clip at the matrix edge)
// 2-D tensor map of 8-bit codes Q [M][N] for the staged code stores: box
// 32 rows x 32 bytes, no swizzle
static bool make_tmap_codes(CUtensorMap* m, void* Q, int64_t M, int64_t N)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)N};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, Q, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

static bool make_tmap_out(CUtensorMap* m, void* D, int64_t M, int64_t N, bool bf16)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t esz = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(N * esz)};
    cuuint32_t box[2] = {(cuuint32_t)(32 / esz), 32u};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, D, dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Co-resident CTA pairs of the pair kernel on the current device (queried
// once per device and output type; the kernel's resources never change).
// The cache entries are atomics: concurrent first calls may both query and
// store, always the same value.
template <typename KernelT>
static cudaError_t pair_clusters(KernelT kern, int variant, int smem, int* clusters)
{
    static std::atomic<int> cache[2][64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) {
        const int c = cache[variant][dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *clusters = c;
            return cudaSuccess;
        }
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) cache[variant][dev].store(n, std::memory_order_relaxed);
    *clusters = n;
    return cudaSuccess;
}

// SMs a launch of g occupies (its persistent grid: one CTA per SM), -1 if
// that cannot be determined.  Lets a caller run two independent GEMMs side by
// side when both grids fit on the device at once.
int gemm_ctas(const GemmArgs& g, int sms)
{
    if (g.M == 0 || g.N == 0 || g.K == 0) return 0;
    const bool pair = g.mode == 0;   // the per-tensor kernel runs on CTA pairs
    if (pair) {
        const int64_t tiles = ((g.M + 2 * BM - 1) / (2 * BM)) * ((g.N + kPairBN - 1) / kPairBN);
        const bool bf16 = g.d_dtype == kBF16;
        int clusters = 0;
        if (pair_clusters(bf16 ? k_gemm_tensor_pair<true, 0> : k_gemm_tensor_pair<false, 0>, bf16 ? 1 : 0,
                          PairSmem::BYTES, &clusters) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            return -1;
        }
        return 2 * (int)(tiles < clusters ? tiles : clusters);
    }
    // the promotion and MX kernels: one CTA per 128 x 256 tile
    const int64_t tiles = ((g.M + BM - 1) / BM) * ((g.N + 255) / 256);
    return (int)(tiles < sms ? tiles : sms);
}

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t st, int sms, const char** why)
{
    *why = nullptr;
    if (g.M == 0 || g.N == 0) return cudaSuccess;
    const bool bf16 = g.d_dtype == kBF16;
    if (g.K == 0) {
        int64_t n = g.M * g.N;
        if (bf16) launch_k(k_fill_bias<true>, (unsigned)((n + 255) / 256), 256, 0, st, g.D, g.M, g.N, g.bias);
        else launch_k(k_fill_bias<false>, (unsigned)((n + 255) / 256), 256, 0, st, g.D, g.M, g.N, g.bias);
        return cudaGetLastError();
    }
    EpiParams p;
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.sA = static_cast<const float*>(g.a_scale);
    p.sB = static_cast<const float*>(g.b_scale);
    p.bias = g.bias;
    p.D = g.D;
    CUtensorMap ta, tb;
    if (g.mode == 0) {
        constexpr int BN = kPairBN;
        // K-major: [rows][K] in boxes of 128 rows x 128 K; MN-major: [K][rows]
        // in boxes of 128 K rows x 128 along M / N
        const bool ok_a = g.a_mn ? make_tmap(&ta, g.A, g.M, g.K, BK) : make_tmap(&ta, g.A, g.K, g.M, BM);
        const bool ok_b = g.b_mn ? make_tmap(&tb, g.B, g.N, g.K, BK) : make_tmap(&tb, g.B, g.K, g.N, BN / 2);
        if (!ok_a || !ok_b) {
            *why = "cuTensorMapEncodeTiled failed";
            return cudaErrorInvalidValue;
        }
        CUtensorMap td;
        if (!make_tmap_out(&td, g.D, g.M, g.N, bf16)) {
            *why = "cuTensorMapEncodeTiled failed (output)";
            return cudaErrorInvalidValue;
        }
        TileSched sched{(int)((g.M + 2 * BM - 1) / (2 * BM)), (int)((g.N + BN - 1) / BN), 8};
        const int tiles = sched.num_m * sched.num_n;
        uint32_t idesc = make_idesc(g.a_format, g.b_format, BN);
        idesc = (idesc & ~(0x1Fu << 24)) | ((uint32_t)((2 * BM) >> 4) << 24);   // M = 256 over the pair
        if (g.a_mn) idesc |= 1u << 15;          // A MN-major
        if (g.b_mn) idesc |= 1u << 16;          // B MN-major
        const int smem = PairSmem::BYTES;
        const int layout = (g.a_mn ? 1 : 0) | (g.b_mn ? 2 : 0);
        using PairKern = decltype(&k_gemm_tensor_pair<true, 0>);
        static const PairKern kerns[3][4] = {
            {k_gemm_tensor_pair<false, 0>, k_gemm_tensor_pair<false, 1>, k_gemm_tensor_pair<false, 2>,
             k_gemm_tensor_pair<false, 3>},
            {k_gemm_tensor_pair<true, 0>, k_gemm_tensor_pair<true, 1>, k_gemm_tensor_pair<true, 2>,
             k_gemm_tensor_pair<true, 3>},
            {k_gemm_tensor_pair<true, 0, true>, k_gemm_tensor_pair<true, 1, true>,
             k_gemm_tensor_pair<true, 2, true>, k_gemm_tensor_pair<true, 3, true>}};
        if (g.q_out && !bf16) {
            *why = "the fused output cast takes a bf16 output";
            return cudaErrorNotSupported;
        }
        CUtensorMap tq = td;                   // unused unless the epilogue casts
        if (g.q_out && !make_tmap_codes(&tq, g.q_out, g.M, g.N)) {
            *why = "cuTensorMapEncodeTiled failed (codes)";
            return cudaErrorInvalidValue;
        }
        p.Q = g.q_out;
        p.qstate = g.q_state;
        p.qH = g.q_history_len;
        p.qfmt = g.q_format;
        auto kern = kerns[g.q_out ? 2 : (bf16 ? 1 : 0)][layout];
        int clusters = 0;
        // every layout instantiation has the same resources: one cached query
        // per output type (and the shared-memory attribute set for this one)
        cudaError_t e = pair_clusters(kern, bf16 ? 1 : 0, smem, &clusters);
        if (e == cudaSuccess) e = smem_attr_once(reinterpret_cast<const void*>(kern), smem);
        if (e != cudaSuccess) {
            *why = "cluster occupancy query failed";
            return e;
        }
        if (clusters < 1) {
            *why = "no CTA pair of this kernel fits on the device";
            return cudaErrorNotSupported;
        }
        const int grid = 2 * (tiles < clusters ? tiles : clusters);
        sched.group = raster_group(g.K, 2 * BM, BN, grid / 2);
        launch_k(kern, grid, 192, smem, st, ta, tb, p, idesc, sched, td, tq);
        return cudaGetLastError();
    }
    if (g.mode == 1) return launch_promote<1>(g, p, st, sms, why);
    if (g.mode == 3) return launch_promote<3>(g, p, st, sms, why);
    if (g.mode == 2) {
        constexpr int BN = 256, ST = 4, NACC = 1;
        using L = MxLayout<BN, ST, NACC>;
        if (!make_tmap(&ta, g.A, g.K, g.M, BM) || !make_tmap(&tb, g.B, g.K, g.N, BN)) {
            *why = "cuTensorMapEncodeTiled failed";
            return cudaErrorInvalidValue;
        }
        TileSched sched{(int)(g.M / BM), (int)((g.N + BN - 1) / BN), 16};
        const int tiles = sched.num_m * sched.num_n;
        MxParams mx{static_cast<const uint8_t*>(g.a_scale), static_cast<const uint8_t*>(g.b_scale), (int)(g.K / 128),
                    (int)(g.N / 128)};
        const uint32_t idesc = make_idesc_mx(g.a_format, g.b_format, BN);
        auto kern = bf16 ? k_gemm_mx<BN, ST, NACC, true> : k_gemm_mx<BN, ST, NACC, false>;
        // the warpgroups' setmaxnreg shares must fit in what the CTA is
        // launched with, or the raising warpgroup would wait forever
        int regs = 0;
        cudaError_t e = launch_regs(reinterpret_cast<const void*>(kern), &regs);
        if (e != cudaSuccess) return e;
        if (regs < kMxLaunchRegs) {
            *why = "MX kernel compiled with fewer registers than its warpgroup split needs";
            return cudaErrorInvalidConfiguration;
        }
        e = smem_attr_once(reinterpret_cast<const void*>(kern), L::BYTES);
        if (e != cudaSuccess) return e;
        CUtensorMap td;
        if (!make_tmap_out(&td, g.D, g.M, g.N, bf16)) {
            *why = "cuTensorMapEncodeTiled failed (output)";
            return cudaErrorInvalidValue;
        }
        const int grid = tiles < sms ? tiles : sms;
        sched.group = raster_group(g.K, BM, BN, grid);
        launch_k(kern, grid, kMxThreads, L::BYTES, st, ta, tb, p, idesc, sched, mx, td);
        return cudaGetLastError();
    }
    *why = "GEMM mode not built";
    return cudaErrorNotSupported;
}

int read_device_error(int clear)
{
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(&v, g_dev_error, sizeof(int)) != cudaSuccess) return -1;
    if (clear) {
        int z = 0;
        if (cudaMemcpyToSymbol(g_dev_error, &z, sizeof(int)) != cudaSuccess) return -1;
    }
    return v;
}

}  // namespace fp8sq

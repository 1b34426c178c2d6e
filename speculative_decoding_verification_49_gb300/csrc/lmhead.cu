// lmhead.cu -- the verifier's LM-head GEMM on the tcgen05 tensor cores of
// sm_103a: logits[r, v] = sum_k hidden[r, k] * weight[v, k] (bf16 in, f32
// accumulated in tensor memory).
//
// "Speculative decoding -- draft, verify, repeat" (factory.pai-world.com,
// lesson 07-16), section "Core algorithm": the verifier scores the N drafts
// in one forward pass, whose last step is this product of the final hidden
// states with the LM head; the draft model ends in the same product.
//
// A persistent grid walks the output in blocks of 256 columns and, when the
// product has at least two 128-row tiles, 256 rows: a cluster of two CTAs on
// neighbouring SMs acts as one MMA unit (tcgen05 cta_group::2).  Each CTA's
// warp 0 streams its 128 x 64 tile of the hidden states and its 128 x 64 half
// of the weight tile with 2-D TMA copies (128-byte swizzle) into a 6-stage
// shared-memory ring, across tile boundaries, and both CTAs' copies are
// counted on the even CTA's barrier.  One thread of the even CTA's warp 1
// issues tcgen05.mma with M = 256, N = 256, K = 16 (four per 64-wide stage):
// each SM stages and reads 32 KiB per 4.2 MFLOP of its share, where one CTA
// computing 128 x 256 alone would stage and read 48 KiB.  The commits free a
// stage in both CTAs.  The accumulator is one of two 128 x 256 f32 halves in
// each CTA's tensor memory (all 512 columns), so warps 4-7 of both CTAs read a
// finished tile back (tcgen05.ld, one TMEM lane = one row per thread) while
// the next tile accumulates into the other one.  A product with a single row
// tile runs on single CTAs (M = 128, the whole weight tile, 4 stages).  The
// epilogue either writes the logits as f32 (32 x 32 blocks staged in shared
// memory and written by TMA tensor stores), or (the fused verify path) each
// row's statistics over the tile -- max and sum of exp2((z - max) *
// log2(e)/T), or max and argmax for greedy rows, and the logit at the row's
// draft token -- and, when given a buffer, the f32 logits as well (the verify
// then reads back only the rows it samples from; without one the logits never
// reach HBM).  The blocks of one
// 256-column weight slab come next to each other so that the units working at
// the same time share that slab through L2.
// Every mbarrier wait is bounded (2 s); a CTA that gives up sets the status
// word, lets the copies its barriers count land and frees its tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cfloat>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "lmhead.h"
#include "spec_verify.h"
#include "sv_tc.cuh"

namespace {

constexpr int kBM = 128;  // tile rows per CTA (TMEM lanes)
constexpr int kBN = 256;  // tile columns (TMEM columns)
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int kTileA = kBM * kBK * 2;
constexpr int kTileB = kBN * kBK * 2;
constexpr int kGemmThreads = 256;
constexpr uint32_t kTmemCols = 512;  // two 128 x 256 f32 accumulators
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kErrTimeout = 4;
constexpr int kMaxStagesG = 6;

// A single CTA stages its 128 x 64 hidden tile and the whole 256 x 64 weight
// tile per step (48 KiB, 4 stages); a CTA of a pair stages its 128 hidden rows
// and its 128-column half of the weight tile (32 KiB, 6 stages).
template <bool PAIR> struct GemmCfg {
    static constexpr int kStages = PAIR ? 6 : 4;
    static constexpr int kTileBh = PAIR ? kTileB / 2 : kTileB;
    static constexpr int kStage = kTileA + kTileBh;
};

struct GemmCtl {
    uint64_t full[kMaxStagesG];     // the stage's copies have landed (a pair: both CTAs', on the even CTA's)
    uint64_t empty[kMaxStagesG];    // the MMAs have read the stage (commit, multicast to both CTAs of a pair)
    uint64_t acc_full[2];   // an accumulator holds a finished tile (MMA commit)
    uint64_t acc_empty[2];  // the epilogue has read it (one arrival per epilogue warp, of both CTAs of a pair)
    int last_kb[kMaxStagesG];  // last k-block (counted over all tiles) issued into each stage
    uint32_t tmem_base;
    int abort;
};

// Logits epilogue, staged in shared memory 32 rows x 32 columns at a time.
// With a tensor map of the output (V a multiple of 4): each epilogue warp
// writes its block into one of two 4 KiB buffers in the 128-byte-swizzled
// layout of the map and one lane stores it with a single TMA tensor store.
// Otherwise the warp turns the block around (row stride 33: no bank
// conflicts) so that every warp store writes 128 contiguous bytes of one row.
constexpr int kEpiStride = 33;
constexpr int kEpiBuf = 32 * 32 * 4;                   // one staged block, bytes
constexpr size_t kEpiBytes = 4 * 2 * (size_t)kEpiBuf;  // 4 warps x 2 buffers
static_assert(4 * 32 * kEpiStride * 4 <= (int)kEpiBytes, "the transpose fits in the staging area");

template <bool PAIR> __host__ __device__ constexpr size_t smem_ring() { return (size_t)GemmCfg<PAIR>::kStages * GemmCfg<PAIR>::kStage; }
static_assert(smem_ring<true>() % 1024 == 0 && smem_ring<false>() % 1024 == 0, "the staging area stays 1024-aligned");

template <bool PAIR> constexpr size_t smem_bytes()
{
    return 1024 + smem_ring<PAIR>() + kEpiBytes + sizeof(GemmCtl);
}
static_assert(smem_bytes<true>() <= 232448 && smem_bytes<false>() <= 232448, "227 KiB of shared memory per CTA");

constexpr double kLog2e = 1.4426950408889634074;

struct LmParams {
    int M, N, K;
    float *logits;  // [M, N] f32 (logits epilogue)
    int tma_store;  // the logits go out through the output tensor map
    int *status;    // error bits, may be null
    svlm::StatsArgs st;  // statistics epilogue
};

// The statistics of one row over one tile, in one pass over two chunks of 128
// columns (four tcgen05.ld in flight per chunk, one wait): the chunk maximum
// as a tree, then for sampled rows the running sum of exp2((z - max) * cf),
// rescaled when the maximum grows, over eight independent partial sums; for
// greedy rows the lowest column holding the maximum.  Columns past the
// vocabulary count as -inf; NaN never becomes the maximum.  A thread whose row
// is past M still issues the warp-collective loads but writes nothing.
__device__ __forceinline__ void row_stats(uint32_t taddr, int n0, const LmParams &p, int row_in)
{
    constexpr int kChunk = 128;
    const svlm::StatsArgs &a = p.st;
    const bool valid = row_in < p.M;
    const int row = valid ? row_in : 0;
    const int b = row / a.rows_per_seq;
    const int i = row - b * a.rows_per_seq;
    float T = a.greedy || !a.T ? 0.0f : a.T[b];
    const bool sampled = T > 0.0f && T != INFINITY && T >= FLT_MIN;  // NaN compares false
    const float cf = sampled ? (float)(kLog2e / (double)T) : 0.0f;
    const int d = (i < a.N) ? a.tokens[(size_t)b * a.N + i] : -1;
    const int dl = d - n0;  // the draft token's column in this tile, if in range
    float m = -INFINITY, s = 0.0f;
    int arg = INT_MAX;
#pragma unroll 1
    for (int c0 = 0; c0 < kBN; c0 += kChunk) {
        uint32_t r[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk / 32; ++j)
            sv::tmem_ld32_nowait(taddr + (uint32_t)(c0 + 32 * j), r + 32 * j);
        sv::tmem_wait_ld();
        const int lim = p.N - n0 - c0;  // columns of this chunk inside the vocabulary
        float v[kChunk];
#pragma unroll
        for (int k = 0; k < kChunk; ++k)
            v[k] = (k < lim) ? __uint_as_float(r[k]) : -INFINITY;
        if (valid && (unsigned)(dl - c0) < (unsigned)kChunk && dl - c0 < lim) {
#pragma unroll
            for (int k = 0; k < kChunk; ++k)
                if (k == dl - c0)
                    a.zgat[row] = v[k];
        }
        float mx[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
            mx[k] = v[k];
#pragma unroll
        for (int k = 16; k < kChunk; ++k)
            mx[k & 15] = fmaxf(mx[k & 15], v[k]);
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
            for (int k = 0; k < w; ++k)
                mx[k] = fmaxf(mx[k], mx[k + w]);
        const float mc = mx[0];
        if (sampled) {
            const float mn = fmaxf(m, mc);
            if (mn != -INFINITY) {
                s = __fmul_rn(s, sv::ex2(__fmul_rn(__fsub_rn(m, mn), cf)));
                float acc[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    acc[k] = 0.0f;
#pragma unroll
                for (int k = 0; k < kChunk; ++k)
                    acc[k & 7] = __fadd_rn(acc[k & 7], sv::ex2(__fmul_rn(__fsub_rn(v[k], mn), cf)));
#pragma unroll
                for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
                    for (int k = 0; k < w; ++k)
                        acc[k] = __fadd_rn(acc[k], acc[k + w]);
                s = __fadd_rn(s, acc[0]);
            }
            m = mn;
        } else if (mc > m) {
            m = mc;
            int idx = 0;
#pragma unroll
            for (int k = kChunk - 1; k >= 0; --k)
                if (v[k] == mc)
                    idx = k;
            arg = n0 + c0 + idx;
        }
    }
    if (valid) {
        float *out = a.part + ((size_t)row * ((p.N + kBN - 1) / kBN) + n0 / kBN) * 2;
        out[0] = m;
        out[1] = sampled ? s : __int_as_float(arg);
    }
}

// One epilogue warp's 32 rows of a finished tile (row r0 + lane for lane) out
// as f32 logits: 32-column blocks through one of the warp's two staging
// buffers in the 128-byte-swizzled layout of the output map, each written by
// one TMA tensor store (blocks past M or N are clipped by the map).
__device__ __forceinline__ void store_tile(uint32_t taddr, unsigned char *epi_raw, int q, int lane, int r0, int n0,
                                           uint32_t &nstore, const CUtensorMap *tmC, const LmParams &p)
{
    for (int c0 = 0; c0 < kBN; c0 += 32, ++nstore) {
        float v[32];
        sv::tmem_ld32(taddr + (uint32_t)c0, v);
        unsigned char *buf = epi_raw + (size_t)(q * 2 + (nstore & 1)) * kEpiBuf;
        if (lane == 0)
            sv::bulk_wait_read<1>();  // the store that last read this buffer is done with it
        __syncwarp();
        // row `lane`: 16-byte chunk j at chunk j ^ (row % 8) (128-byte swizzle)
        float4 *rowp = reinterpret_cast<float4 *>(buf + lane * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            rowp[j ^ (lane & 7)] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        sv::fence_async_shared();
        __syncwarp();
        if (lane == 0) {
            if (r0 < p.M && n0 + c0 < p.N)
                sv::tma_store_2d(tmC, n0 + c0, r0, buf);
            sv::bulk_commit();  // one group per block, empty when nothing was stored
        }
    }
}

template <bool STATS, bool PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1)
    sv_lmhead_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, LmParams p)
{
    using Cfg = GemmCfg<PAIR>;
    constexpr int kStages = Cfg::kStages;
    constexpr int P = PAIR ? 2 : 1;  // CTAs per MMA unit
    extern __shared__ unsigned char smem_raw[];
    // 128-byte-swizzled tiles want 1024-byte alignment
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *epi_raw = smem + smem_ring<PAIR>();  // 1024-aligned staging area
    float *epi = reinterpret_cast<float *>(epi_raw);
    GemmCtl &ctl = *reinterpret_cast<GemmCtl *>(epi_raw + kEpiBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? sv::cluster_ctarank() : 0u;
    const bool leader = rank == 0;  // the CTA whose thread issues the MMAs
    const int unit = blockIdx.x / P, nunits = gridDim.x / P;
    const int Mt = (p.M + kBM - 1) / kBM;
    const int Mp = (Mt + P - 1) / P;  // blocks of P row tiles
    const int nblock = Mp * ((p.N + kBN - 1) / kBN);
    const int nk = (p.K + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            sv::mbar_init(&ctl.full[s], 1);  // the even CTA's expect-tx arrival
            sv::mbar_init(&ctl.empty[s], 1);
            ctl.last_kb[s] = -1;
        }
        for (int b = 0; b < 2; ++b) {
            sv::mbar_init(&ctl.acc_full[b], 1);
            sv::mbar_init(&ctl.acc_empty[b], 4u * P);
        }
        ctl.abort = 0;
        sv::fence_mbar_init();
    }
    if constexpr (PAIR) {
        sv::cluster_sync();  // the peer is running before the collective allocation
        if (warp == 2) {
            sv::tmem_alloc_pair(&ctl.tmem_base, kTmemCols);
            sv::tmem_relinquish_pair();
        }
    } else if (warp == 2) {
        sv::tmem_alloc(&ctl.tmem_base, kTmemCols);
        sv::tmem_relinquish();
    }
    sv::tc_fence_before();
    if constexpr (PAIR)
        sv::cluster_sync();  // both CTAs' barriers exist before any copy, arrival or commit reaches them
    else
        __syncthreads();
    sv::tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            sv::tma_prefetch_desc(&tmA);
            sv::tma_prefetch_desc(&tmB);
            uint32_t g = 0;  // k-blocks issued so far, over all tiles
            for (int blk = unit; blk < nblock && !ctl.abort; blk += nunits) {
                const int m0 = ((blk % Mp) * P + (int)rank) * kBM, n0 = (blk / Mp) * kBN;
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = (int)(g % kStages);
                    const uint32_t ph = (g / kStages) & 1u;
                    if (!sv::mbar_wait_bounded(&ctl.empty[s], ph ^ 1u, &ctl.abort, kWaitNs)) {
                        ctl.abort = 1;
                        break;
                    }
                    unsigned char *a = smem + (size_t)s * Cfg::kStage;
                    if constexpr (PAIR) {
                        // this CTA's hidden rows and weight half, counted on the even CTA's barrier, which
                        // alone posts the bytes of both CTAs (the odd CTA's may land first: the phase
                        // cannot complete before that arrival)
                        const uint32_t full_cl = sv::dsmem_addr(&ctl.full[s], 0);
                        if (leader)
                            sv::mbar_arrive_expect_tx(&ctl.full[s], 2u * Cfg::kStage);
                        sv::tma_load_2d_pair(a, &tmA, kb * kBK, m0, full_cl);
                        sv::tma_load_2d_pair(a + kTileA, &tmB, kb * kBK, n0 + (int)rank * (kBN / 2), full_cl);
                    } else {
                        sv::mbar_arrive_expect_tx(&ctl.full[s], Cfg::kStage);
                        sv::tma_load_2d(a, &tmA, kb * kBK, m0, &ctl.full[s]);
                        sv::tma_load_2d(a + kTileA, &tmB, kb * kBK, n0, &ctl.full[s]);
                    }
                    ctl.last_kb[s] = (int)g;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = sv::idesc_bf16_f32(kBM * P, kBN);
            uint32_t g = 0;
            int t = 0;
            for (int blk = unit; blk < nblock && !ctl.abort; blk += nunits, ++t) {
                const int buf = t & 1;
                const uint32_t use = (uint32_t)(t >> 1);
                // the epilogue (of both CTAs) has finished with this accumulator's previous tile
                if (!sv::mbar_wait_bounded(&ctl.acc_empty[buf], (use & 1u) ^ 1u, &ctl.abort, kWaitNs)) {
                    ctl.abort = 1;
                    break;
                }
                sv::tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * kBN);
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = (int)(g % kStages);
                    const uint32_t ph = (g / kStages) & 1u;
                    if (!sv::mbar_wait_bounded(&ctl.full[s], ph, &ctl.abort, kWaitNs)) {
                        ctl.abort = 1;
                        break;
                    }
                    sv::tc_fence_after();
                    const unsigned char *a = smem + (size_t)s * Cfg::kStage;
                    const uint64_t da = sv::smem_desc_k128(a), db = sv::smem_desc_k128(a + kTileA);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {  // K = 16 per MMA: 32 bytes along the swizzled row
                        if constexpr (PAIR)
                            sv::tc_mma_bf16_pair(d, da + 2u * kk, db + 2u * kk, idesc, (kb | kk) != 0);
                        else
                            sv::tc_mma_bf16(d, da + 2u * kk, db + 2u * kk, idesc, (kb | kk) != 0);
                    }
                    // the stage may be refilled once these MMAs have read it
                    if constexpr (PAIR)
                        sv::tc_commit_pair_multicast(&ctl.empty[s], 3);
                    else
                        sv::tc_commit(&ctl.empty[s]);
                }
                if constexpr (PAIR)
                    sv::tc_commit_pair_multicast(&ctl.acc_full[buf], 3);  // the tile is complete
                else
                    sv::tc_commit(&ctl.acc_full[buf]);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        const int q = warp - 4;  // TMEM lanes 32q .. 32q+31
        int t = 0;
        uint32_t nstore = 0;  // staged blocks so far (TMA-store epilogue): alternates the buffers
        for (int blk = unit; blk < nblock; blk += nunits, ++t) {
            const int buf = t & 1;
            const uint32_t use = (uint32_t)(t >> 1);
            const bool ok = sv::mbar_wait_bounded(&ctl.acc_full[buf], use & 1u, &ctl.abort, kWaitNs);
            if (!__all_sync(0xffffffffu, ok && !ctl.abort)) {  // tcgen05.ld is warp-collective
                if (lane == 0 && p.status)
                    atomicOr(p.status, kErrTimeout);
                break;
            }
            sv::tc_fence_after();
            const int m0 = ((blk % Mp) * P + (int)rank) * kBM, n0 = (blk / Mp) * kBN;
            const int row = m0 + 32 * q + lane;
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kBN);
            if constexpr (STATS) {
                row_stats(taddr, n0, p, row);
                if (p.tma_store)  // the logits too, from the same accumulator
                    store_tile(taddr, epi_raw, q, lane, m0 + 32 * q, n0, nstore, &tmC, p);
            } else if (p.tma_store) {
                store_tile(taddr, epi_raw, q, lane, m0 + 32 * q, n0, nstore, &tmC, p);
            } else {
                float *stg = epi + q * 32 * kEpiStride;
                const int r0 = m0 + 32 * q;  // the warp's first row
                for (int c0 = 0; c0 < kBN; c0 += 32) {
                    float v[32];
                    sv::tmem_ld32(taddr + (uint32_t)c0, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        stg[lane * kEpiStride + i] = v[i];
                    __syncwarp();
                    const int col = n0 + c0 + lane;
                    const int rows = min(32, p.M - r0);
                    if (col < p.N)
                        for (int r = 0; r < rows; ++r)
                            p.logits[(size_t)(r0 + r) * p.N + col] = stg[r * kEpiStride + lane];
                    __syncwarp();
                }
            }
            sv::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    sv::mbar_arrive_cl(sv::dsmem_addr(&ctl.acc_empty[buf], 0));
                else
                    sv::mbar_arrive(&ctl.acc_empty[buf]);
            }
        }
        if (lane == 0)
            sv::bulk_wait_all();  // every tensor store has read its buffer and completed
        __syncwarp();
    }
    sv::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && ctl.abort) {
        // let the copies this CTA's barriers count land before it exits (a pair's
        // odd CTA counts on the even CTA's barriers, which drains them)
        if (leader)
            for (int s = 0; s < kStages; ++s)
                if (ctl.last_kb[s] >= 0) {
                    int never = 0;
                    sv::mbar_wait_bounded(&ctl.full[s], (uint32_t)(ctl.last_kb[s] / kStages) & 1u, &never, kWaitNs / 4);
                }
        if (p.status)
            atomicOr(p.status, kErrTimeout);
    }
    if constexpr (PAIR) {
        sv::cluster_sync();  // the peer no longer writes into this CTA's stages, barriers or tensor memory
        if (warp == 2)
            sv::tmem_dealloc_pair(tmem, kTmemCols);
    } else if (warp == 2) {
        sv::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- host side -----------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load();
    if (!f) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        f = reinterpret_cast<EncodeTiledFn>(ptr);
        fn.store(f);
    }
    return f;
}

// Row-major bf16 matrix [rows, K] as a TMA map with boxes of box_rows x 64.
bool make_map(CUtensorMap *m, const void *base, int rows, int K, int box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major f32 logits [rows, cols] as a TMA map with 32 x 32 boxes in the
// 128-byte-swizzled layout (the epilogue's tensor stores); cols * 4 must be a
// multiple of 16 and base 16-byte aligned.
bool make_map_out(CUtensorMap *m, const float *base, int rows, int cols)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

std::once_flag g_attr_once;
cudaError_t g_attr_err = cudaSuccess;

template <bool STATS, bool PAIR> cudaError_t set_smem_attr()
{
    return cudaFuncSetAttribute(sv_lmhead_kernel<STATS, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes<PAIR>());
}

// Clusters (CTAs, or CTA pairs) of the kernel that fit on the device at once,
// queried once per device and kind; SMs / P if the query fails.
template <bool STATS>
int resident_units(bool pair, int dev, int sms, const cudaLaunchConfig_t &cfg)
{
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev][2];
    const int P = pair ? 2 : 1;
    if (dev < 0 || dev >= kMaxDev)
        return sms / P;
    int n = cache[dev][pair].load();
    if (n <= 0) {
        n = 0;
        const cudaError_t e = pair ? cudaOccupancyMaxActiveClusters(&n, sv_lmhead_kernel<STATS, true>, &cfg)
                                   : cudaOccupancyMaxActiveClusters(&n, sv_lmhead_kernel<STATS, false>, &cfg);
        if (e != cudaSuccess || n <= 0) {
            cudaGetLastError();
            return sms / P;
        }
        n = n < sms / P ? n : sms / P;
        cache[dev][pair].store(n);
    }
    return n;
}

template <bool STATS>
sv_status launch(const void *hidden, const void *weight, int M, int V, int K, const LmParams &p, cudaStream_t st)
{
    if (M < 0 || V < 0 || K < 1 || K % 8 != 0)
        return SV_ERR_INVALID_ARG;
    if (M == 0 || V == 0)
        return SV_OK;
    if (!hidden || !weight || (reinterpret_cast<uintptr_t>(hidden) & 15u) || (reinterpret_cast<uintptr_t>(weight) & 15u))
        return SV_ERR_INVALID_ARG;
    std::call_once(g_attr_once, [] {
        cudaError_t e = set_smem_attr<false, false>();
        if (e == cudaSuccess)
            e = set_smem_attr<false, true>();
        if (e == cudaSuccess)
            e = set_smem_attr<true, false>();
        if (e == cudaSuccess)
            e = set_smem_attr<true, true>();
        g_attr_err = e;
    });
    if (g_attr_err != cudaSuccess)
        return SV_ERR_CUDA;
    CUtensorMap ta, tb, tc;
    // the logits go out by tensor stores when their rows are 16-byte multiples
    // (the statistics epilogue writes them only that way)
    LmParams q = p;
    q.tma_store = 0;
    if (p.logits && V % 4 == 0 && (reinterpret_cast<uintptr_t>(p.logits) & 15u) == 0 &&
        make_map_out(&tc, p.logits, M, V))
        q.tma_store = 1;
    if (STATS && p.logits && !q.tma_store)
        return SV_ERR_INVALID_ARG;
    // CTA pairs (one 256-row MMA) when there are two row tiles to pair
    const bool pair = (M + kBM - 1) / kBM >= 2;
    const int P = pair ? 2 : 1;
    if (!make_map(&ta, hidden, M, K, kBM) || !make_map(&tb, weight, V, K, kBN / P))
        return SV_ERR_CUDA;
    if (!q.tma_store)
        tc = ta;  // not read
    const long long nblock = (long long)((M + kBM * P - 1) / (kBM * P)) * ((V + kBN - 1) / kBN);
    if (nblock > INT_MAX / P)
        return SV_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SV_ERR_CUDA;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((sms / P) * P));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = pair ? smem_bytes<true>() : smem_bytes<false>();
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // one CTA per SM walks the blocks: as many units as can be resident at once
    const int fit = resident_units<STATS>(pair, dev, sms, cfg);
    const long long units = nblock < fit ? nblock : fit;
    cfg.gridDim = dim3((unsigned)(units * P));
    const cudaError_t e = pair ? cudaLaunchKernelEx(&cfg, sv_lmhead_kernel<STATS, true>, ta, tb, tc, q)
                               : cudaLaunchKernelEx(&cfg, sv_lmhead_kernel<STATS, false>, ta, tb, tc, q);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

} // namespace

namespace svlm {

sv_status launch_logits(const void *hidden, const void *weight, int M, int V, int K, float *logits,
                        cudaStream_t stream)
{
    if (M > 0 && V > 0 && !logits)
        return SV_ERR_INVALID_ARG;
    LmParams p{};
    p.M = M;
    p.N = V;
    p.K = K;
    p.logits = logits;
    return launch<false>(hidden, weight, M, V, K, p, stream);
}

sv_status launch_stats(const void *hidden, const void *weight, int M, int V, int K, const StatsArgs &a,
                       cudaStream_t stream, float *logits)
{
    if (M > 0 && V > 0 && (!a.part || !a.zgat || a.rows_per_seq < 1 || (a.N > 0 && !a.tokens)))
        return SV_ERR_INVALID_ARG;
    LmParams p{};
    p.M = M;
    p.N = V;
    p.K = K;
    p.logits = logits;
    p.st = a;
    return launch<true>(hidden, weight, M, V, K, p, stream);
}

} // namespace svlm

extern "C" sv_status spec_verify_lm_head_logits(const void *hidden, const void *weight, int M, int V, int K,
                                                float *logits, void *stream)
{
    return svlm::launch_logits(hidden, weight, M, V, K, logits, static_cast<cudaStream_t>(stream));
}

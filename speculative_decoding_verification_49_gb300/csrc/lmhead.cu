// lmhead.cu -- the verifier's LM-head GEMM on the tcgen05 tensor cores of
// sm_103a: logits[r, v] = sum_k hidden[r, k] * weight[v, k] (bf16 in, f32
// accumulated in tensor memory).
//
// "Speculative decoding -- draft, verify, repeat" (factory.pai-world.com,
// lesson 07-16), section "Core algorithm": the verifier scores the N drafts
// in one forward pass, whose last step is this product of the final hidden
// states with the LM head; the draft model ends in the same product.
//
// A persistent grid of CTA pairs (clusters of 2, one CTA per SM; single CTAs
// when the product has only one 128-row tile) walks the output in 256 x 256
// blocks: the two CTAs of a pair take the two 128-row
// tiles of one block, and the blocks of one 256-column weight slab come next
// to each other so that the pairs working at the same time share that slab
// through L2.  In each CTA warp 0 streams its 128 x 64 tile of the hidden
// states and half of the 256 x 64 weight tile with 2-D TMA copies (128-byte
// swizzle) into a 4-stage shared-memory ring, across tile boundaries; the
// weight half is multicast into both CTAs, so each SM stages 32 KiB per 64-wide
// step instead of 48 KiB, and a stage is refilled only when the MMAs of both
// CTAs have read it.  One thread of warp 1 issues tcgen05.mma (M = 128, N = 256,
// K = 16, four per 64-wide stage) into one of two 128 x 256 f32 accumulators
// in tensor memory (all 512 columns) and frees each stage with
// tcgen05.commit; warps 4-7 read a finished accumulator back (tcgen05.ld, one
// TMEM lane = one row per thread) while the next tile accumulates into the
// other one, and run the epilogue: either the logits go out as f32, or (the
// fused verify path) only each row's statistics over the tile do -- max and
// sum of exp2((z - max) * log2(e)/T), or max and argmax for greedy rows, and
// the logit at the row's draft token -- so the logits never reach HBM.
// Every mbarrier wait is bounded (2 s); a CTA that gives up sets the status
// word, lets its copies land and frees its tensor memory.
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

constexpr int kBM = 128;  // tile rows (TMEM lanes)
constexpr int kBN = 256;  // tile columns (TMEM columns)
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int kStagesG = 4;
constexpr int kTileA = kBM * kBK * 2;
constexpr int kTileB = kBN * kBK * 2;
constexpr int kStageBytes = kTileA + kTileB;
constexpr int kGemmThreads = 256;
constexpr int kMaxPair = 2;  // CTAs of a cluster sharing one weight tile (1 when there is one row tile)
constexpr uint32_t kTmemCols = 512;  // two 128 x 256 f32 accumulators
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kErrTimeout = 4;

struct GemmCtl {
    uint64_t full[kStagesG];
    uint64_t empty[kStagesG];  // both CTAs of the pair have read the stage (one MMA commit each)
    uint64_t acc_full[2];   // an accumulator holds a finished tile (MMA commit)
    uint64_t acc_empty[2];  // the epilogue has read it (one arrival per epilogue warp)
    int last_kb[kStagesG];  // last k-block (counted over all tiles) issued into each stage
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemG = 1024 + (size_t)kStagesG * kStageBytes + sizeof(GemmCtl);

constexpr double kLog2e = 1.4426950408889634074;

struct LmParams {
    int M, N, K;
    float *logits;  // [M, N] f32 (logits epilogue)
    int *status;    // error bits, may be null
    svlm::StatsArgs st;  // statistics epilogue
};

// The statistics of one row over one tile (32 columns per tcgen05.ld).  A
// thread whose row is past M still issues the warp-collective loads but
// writes nothing.
__device__ __forceinline__ void row_stats(uint32_t taddr, int n0, const LmParams &p, int row_in)
{
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
    float m = -INFINITY;
    int arg = INT_MAX;
    for (int c0 = 0; c0 < kBN; c0 += 32) {
        float v[32];
        sv::tmem_ld32(taddr + (uint32_t)c0, v);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const int c = c0 + k;
            if (n0 + c < p.N) {
                if (v[k] > m) {
                    m = v[k];
                    arg = n0 + c;
                }
                if (c == dl && valid)
                    a.zgat[row] = v[k];
            }
        }
    }
    float s = 0.0f;
    // tcgen05.ld is warp-collective and the rows of one warp may belong to
    // greedy and sampled sequences alike: the whole warp loads, the sampled
    // rows accumulate
    if (__any_sync(0xffffffffu, sampled)) {
        for (int c0 = 0; c0 < kBN; c0 += 32) {
            float v[32];
            sv::tmem_ld32(taddr + (uint32_t)c0, v);
            if (sampled) {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if (n0 + c0 + k < p.N)
                        s = __fadd_rn(s, sv::ex2(__fmul_rn(__fsub_rn(v[k], m), cf)));
            }
        }
    }
    if (valid) {
        float *out = a.part + ((size_t)row * ((p.N + kBN - 1) / kBN) + n0 / kBN) * 2;
        out[0] = m;
        out[1] = sampled ? s : __int_as_float(arg);
    }
}

template <bool STATS>
__global__ void __launch_bounds__(kGemmThreads, 1)
    sv_lmhead_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, LmParams p)
{
    extern __shared__ unsigned char smem_raw[];
    // 128-byte-swizzled tiles want 1024-byte alignment
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GemmCtl &ctl = *reinterpret_cast<GemmCtl *>(smem + (size_t)kStagesG * kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = sv::cluster_ctarank();
    const int P = (int)sv::cluster_nctarank();  // CTAs sharing a weight tile: 1 or 2
    const int pair = blockIdx.x / P, npairs_grid = gridDim.x / P;
    const int Mt = (p.M + kBM - 1) / kBM;
    const int Mp = (Mt + P - 1) / P;  // blocks of P row tiles
    const int nblock = Mp * ((p.N + kBN - 1) / kBN);
    const int nk = (p.K + kBK - 1) / kBK;
    const uint16_t all = (uint16_t)((1u << P) - 1u);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesG; ++s) {
            sv::mbar_init(&ctl.full[s], 1);
            sv::mbar_init(&ctl.empty[s], (uint32_t)P);
            ctl.last_kb[s] = -1;
        }
        for (int b = 0; b < 2; ++b) {
            sv::mbar_init(&ctl.acc_full[b], 1);
            sv::mbar_init(&ctl.acc_empty[b], 4);
        }
        ctl.abort = 0;
        sv::fence_mbar_init();
    }
    if (warp == 2) {
        sv::tmem_alloc(&ctl.tmem_base, kTmemCols);
        sv::tmem_relinquish();
    }
    sv::tc_fence_before();
    sv::cluster_sync();  // both CTAs' barriers exist before any copy or commit reaches them
    sv::tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            sv::tma_prefetch_desc(&tmA);
            sv::tma_prefetch_desc(&tmB);
            uint32_t g = 0;  // k-blocks issued so far, over all tiles
            for (int blk = pair; blk < nblock && !ctl.abort; blk += npairs_grid) {
                const int m0 = ((blk % Mp) * P + (int)rank) * kBM, n0 = (blk / Mp) * kBN;
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = (int)(g % kStagesG);
                    const uint32_t ph = (g / kStagesG) & 1u;
                    if (!sv::mbar_wait_bounded(&ctl.empty[s], ph ^ 1u, &ctl.abort, kWaitNs)) {
                        ctl.abort = 1;
                        break;
                    }
                    unsigned char *a = smem + (size_t)s * kStageBytes;
                    sv::mbar_arrive_expect_tx(&ctl.full[s], kStageBytes);
                    sv::tma_load_2d(a, &tmA, kb * kBK, m0, &ctl.full[s]);
                    // this CTA's share of the weight tile, into every CTA of the cluster
                    sv::tma_load_2d_multicast(a + kTileA + rank * (kTileB / P), &tmB, kb * kBK, n0 + (int)rank * (kBN / P),
                                              &ctl.full[s], all);
                    ctl.last_kb[s] = (int)g;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = sv::idesc_bf16_f32(kBM, kBN);
            uint32_t g = 0;
            int t = 0;
            for (int blk = pair; blk < nblock && !ctl.abort; blk += npairs_grid, ++t) {
                const int buf = t & 1;
                const uint32_t use = (uint32_t)(t >> 1);
                // the epilogue has finished with this accumulator's previous tile
                if (!sv::mbar_wait_bounded(&ctl.acc_empty[buf], (use & 1u) ^ 1u, &ctl.abort, kWaitNs)) {
                    ctl.abort = 1;
                    break;
                }
                sv::tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * kBN);
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = (int)(g % kStagesG);
                    const uint32_t ph = (g / kStagesG) & 1u;
                    if (!sv::mbar_wait_bounded(&ctl.full[s], ph, &ctl.abort, kWaitNs)) {
                        ctl.abort = 1;
                        break;
                    }
                    sv::tc_fence_after();
                    const unsigned char *a = smem + (size_t)s * kStageBytes;
                    const uint64_t da = sv::smem_desc_k128(a), db = sv::smem_desc_k128(a + kTileA);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)  // K = 16 per MMA: 32 bytes along the swizzled row
                        sv::tc_mma_bf16(d, da + 2u * kk, db + 2u * kk, idesc, (kb | kk) != 0);
                    sv::tc_commit_multicast(&ctl.empty[s], all);  // this CTA's MMAs have read the stage
                }
                sv::tc_commit(&ctl.acc_full[buf]);  // the tile is complete
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        const int q = warp - 4;  // TMEM lanes 32q .. 32q+31
        int t = 0;
        for (int blk = pair; blk < nblock; blk += npairs_grid, ++t) {
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
            } else {
                for (int c0 = 0; c0 < kBN; c0 += 32) {
                    float v[32];
                    sv::tmem_ld32(taddr + (uint32_t)c0, v);
                    if (row < p.M) {
                        float *dst = p.logits + (size_t)row * p.N + n0 + c0;
                        for (int i = 0; i < 32; ++i)
                            if (n0 + c0 + i < p.N)
                                dst[i] = v[i];
                    }
                }
            }
            sv::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                sv::mbar_arrive(&ctl.acc_empty[buf]);
        }
    }
    sv::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && ctl.abort) {
        // let every copy issued into this CTA's shared memory land before it exits
        for (int s = 0; s < kStagesG; ++s)
            if (ctl.last_kb[s] >= 0) {
                int never = 0;
                sv::mbar_wait_bounded(&ctl.full[s], (uint32_t)(ctl.last_kb[s] / kStagesG) & 1u, &never, kWaitNs / 4);
            }
        if (p.status)
            atomicOr(p.status, kErrTimeout);
    }
    sv::cluster_sync();  // the peer no longer writes into this CTA's stages or barriers
    if (warp == 2)
        sv::tmem_dealloc(tmem, kTmemCols);
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

std::once_flag g_attr_once;
cudaError_t g_attr_err = cudaSuccess;

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
        g_attr_err = cudaFuncSetAttribute(sv_lmhead_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)kSmemG);
        if (g_attr_err == cudaSuccess)
            g_attr_err = cudaFuncSetAttribute(sv_lmhead_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)kSmemG);
    });
    if (g_attr_err != cudaSuccess)
        return SV_ERR_CUDA;
    CUtensorMap ta, tb;
    // pairs of CTAs share each weight tile when there are two row tiles to pair
    const int P = (M + kBM - 1) / kBM >= kMaxPair ? kMaxPair : 1;
    if (!make_map(&ta, hidden, M, K, kBM) || !make_map(&tb, weight, V, K, kBN / P))
        return SV_ERR_CUDA;
    const long long nblock = (long long)((M + kBM * P - 1) / (kBM * P)) * ((V + kBN - 1) / kBN);
    if (nblock > INT_MAX / P)
        return SV_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SV_ERR_CUDA;
    const long long pairs = nblock < sms / P ? nblock : sms / P;  // one CTA per SM walks the blocks
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(pairs * P));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kSmemG;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, sv_lmhead_kernel<STATS>, ta, tb, p) != cudaSuccess) {
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
                       cudaStream_t stream)
{
    if (M > 0 && V > 0 && (!a.part || !a.zgat || a.rows_per_seq < 1 || (a.N > 0 && !a.tokens)))
        return SV_ERR_INVALID_ARG;
    LmParams p{};
    p.M = M;
    p.N = V;
    p.K = K;
    p.st = a;
    return launch<true>(hidden, weight, M, V, K, p, stream);
}

} // namespace svlm

extern "C" sv_status spec_verify_lm_head_logits(const void *hidden, const void *weight, int M, int V, int K,
                                                float *logits, void *stream)
{
    return svlm::launch_logits(hidden, weight, M, V, K, logits, static_cast<cudaStream_t>(stream));
}

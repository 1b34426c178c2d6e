// kv_commit.cu -- KV-cache commit/rollback after a verify step, for sm_103a.
//
// "Speculative decoding -- draft, verify, repeat" (factory.pai-world.com,
// lesson 07-16), section "KV cache dance": the verifier's forward over the N
// drafts writes their N KV entries into a scratch buffer; once the verify step
// has fixed num_accepted, the first num_accepted entries are appended to the
// cache and the others are dropped.  The lesson's exercise 4 states the check
// (prefix + the accepted drafts is what the next iteration reads).
//
// The work is a plain byte copy: per (plane, sequence) segment, the first
// a*row_bytes bytes of its scratch rows go to the cache at row cache_len[b].
// Two kernels, both stream-ordered after whatever produced num_accepted:
//   sv_kv_copy_kernel  one warp per 4 KiB unit of a segment's scratch rows
//                      (grid: x = plane and unit, y = sequence, so the index
//                      arithmetic stays in 32 bits); the warp moves the
//                      accepted part of its unit with coalesced 16-byte loads
//                      and stores, four per lane in flight (a warp whose unit
//                      holds no accepted row exits at once);
//   sv_kv_len_kernel   advances cache_len and reports bad counts / overflow.
// The length update needs its own launch: every copying warp reads cache_len.
// The copy is HBM-bound on the accepted bytes (each read once, written once).
// A sequence typically accepts one or two of its N rows, so the work is small
// and most units are empty.  Measured alternatives that were no faster on
// such a commit: a TMA-staged copy (bulk load into shared memory, bulk store
// out; the stage must be sized for all N rows), a persistent grid, one CTA
// per (sequence, split) striping all planes, larger or smaller units, deeper
// unrolling, and one warp serving the same unit of 2, 4 or 8 planes with all
// their loads in flight, 1-4 loads per lane and plane (12.6-16.5 us against
// 12.55 us per commit).
#include <climits>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "spec_verify.h"
#include "sv_device.cuh"

namespace {

using namespace sv;

constexpr int kKvWarps = 4;                 // warps per CTA of the copy kernel
constexpr uint32_t kKvUnit = 4096u;         // bytes of a segment one warp owns
constexpr int kKvUnroll = 4;                // 16-byte vectors per lane in flight
constexpr int kKvLenThreads = 256;
constexpr int kKvMaxGridY = 65535;          // sequences per launch row; larger batches loop

struct KvParams {
    const unsigned char *scratch;  // [P][B][N][row_bytes]
    unsigned char *cache;          // [P][B][max_len][row_bytes]
    int32_t *cache_len;            // [B]
    const int32_t *nacc;           // [B]
    int32_t *status;               // error bits, may be null
    int P, B, N, max_len;
    unsigned long long row_bytes;
    unsigned long long seg_bytes;  // N * row_bytes: one sequence's scratch rows in one plane
    int nunit;                     // units per segment
};

// Rows of a sequence to commit, and the error bits its counts raise.
__device__ __forceinline__ int kv_rows(int a, int len, int N, int max_len, int &bits)
{
    bits = 0;
    if (a < 0)  // the verify step flagged the sequence invalid: nothing to commit
        return 0;
    if (a > N) {
        bits = SV_KV_BAD_COUNT;
        return 0;
    }
    if (len < 0 || (long long)len + a > max_len) {
        bits = SV_KV_OVERFLOW;
        return 0;
    }
    return a;
}

__global__ void __launch_bounds__(kKvWarps * 32) sv_kv_copy_kernel(KvParams k)
{
    grid_dependency_wait();
    // blockIdx.y walks the sequences, blockIdx.x the (plane, unit) pairs of one
    // sequence; every warp of a CTA serves the same sequence
    const unsigned lane = threadIdx.x & 31u;
    const unsigned u = blockIdx.x * kKvWarps + (threadIdx.x >> 5);
    if (u >= (unsigned)k.P * (unsigned)k.nunit)
        return;
    const unsigned p = k.nunit == 1 ? u : u / (unsigned)k.nunit;
    const unsigned long long off = (unsigned long long)(u - p * (unsigned)k.nunit) * kKvUnit;
    for (int b = blockIdx.y; b < k.B; b += gridDim.y) {
        const int len = __ldg(&k.cache_len[b]);
        int bits;
        const unsigned long long total =
            (unsigned long long)kv_rows(__ldg(&k.nacc[b]), len, k.N, k.max_len, bits) * k.row_bytes;
        if (total <= off)
            continue;
        const unsigned long long left = total - off;
        const unsigned n = (unsigned)((left < kKvUnit ? left : kKvUnit) / 16);  // 16-byte vectors
        const unsigned long long seg = (unsigned long long)p * k.B + b;
        const int4 *src = reinterpret_cast<const int4 *>(k.scratch + seg * k.seg_bytes + off);
        int4 *dst = reinterpret_cast<int4 *>(k.cache + (seg * k.max_len + len) * k.row_bytes + off);
        for (unsigned v = lane; v < n; v += 32u * kKvUnroll) {
            int4 x[kKvUnroll];
#pragma unroll
            for (int j = 0; j < kKvUnroll; ++j)
                if (v + 32u * j < n)
                    x[j] = __ldcs(src + v + 32u * j);  // read once: evict first
#pragma unroll
            for (int j = 0; j < kKvUnroll; ++j)
                if (v + 32u * j < n)
                    dst[v + 32u * j] = x[j];
        }
    }
}

__global__ void __launch_bounds__(kKvLenThreads) sv_kv_len_kernel(KvParams k)
{
    grid_dependency_wait();  // every copy of this commit has read cache_len
    const int b = blockIdx.x * kKvLenThreads + threadIdx.x;
    if (b >= k.B)
        return;
    const int len = k.cache_len[b];
    int bits;
    const int rows = kv_rows(k.nacc[b], len, k.N, k.max_len, bits);
    if (bits) {
        if (k.status)
            atomicOr(k.status, bits);
        return;
    }
    k.cache_len[b] = len + rows;
}

cudaLaunchConfig_t kv_launch(unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                             cudaLaunchAttribute *attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

} // namespace

extern "C" sv_status spec_verify_kv_commit(const void *scratch, void *cache, int32_t *cache_len,
                                           const int32_t *num_accepted, int32_t *status, int planes,
                                           int B, int N, int max_len, size_t row_bytes, void *stream)
{
    if (B < 0 || N < 0 || planes < 1 || max_len < 0 || row_bytes == 0 || row_bytes % 16 != 0)
        return SV_ERR_INVALID_ARG;
    if (B == 0)
        return SV_OK;
    if (!cache_len || !num_accepted || (N > 0 && (!scratch || !cache)))
        return SV_ERR_INVALID_ARG;
    if (!aligned16(scratch) || !aligned16(cache))
        return SV_ERR_INVALID_ARG;
    // every byte offset the kernels form must fit in 62 bits
    const unsigned long long rows_max = (unsigned long long)(max_len > N ? max_len : N);
    const unsigned long long segs = (unsigned long long)planes * (unsigned long long)B;
    if (rows_max > 0 && row_bytes > (1ull << 62) / rows_max / segs)
        return SV_ERR_TOO_LARGE;

    KvParams k;
    k.scratch = static_cast<const unsigned char *>(scratch);
    k.cache = static_cast<unsigned char *>(cache);
    k.cache_len = cache_len;
    k.nacc = num_accepted;
    k.status = status;
    k.P = planes;
    k.B = B;
    k.N = N;
    k.max_len = max_len;
    k.row_bytes = row_bytes;
    k.seg_bytes = (unsigned long long)N * row_bytes;
    const unsigned long long nunit = (k.seg_bytes + kKvUnit - 1) / kKvUnit;
    if (nunit > (unsigned long long)INT_MAX)
        return SV_ERR_TOO_LARGE;
    k.nunit = (int)nunit;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (N > 0 && max_len > 0) {
        const unsigned long long per_seq = (unsigned long long)planes * k.nunit;  // warps per sequence
        if (per_seq > (unsigned long long)UINT_MAX - kKvWarps)
            return SV_ERR_TOO_LARGE;
        cudaLaunchConfig_t cfg = kv_launch((unsigned)((per_seq + kKvWarps - 1) / kKvWarps), kKvWarps * 32, 0, st,
                                           attr);
        cfg.gridDim.y = (unsigned)(B < kKvMaxGridY ? B : kKvMaxGridY);
        if (cudaLaunchKernelEx(&cfg, sv_kv_copy_kernel, k) != cudaSuccess) {
            cudaGetLastError();
            return SV_ERR_CUDA;
        }
    }
    cudaLaunchConfig_t cfg = kv_launch((unsigned)((B + kKvLenThreads - 1) / kKvLenThreads), kKvLenThreads, 0, st,
                                       attr);
    if (cudaLaunchKernelEx(&cfg, sv_kv_len_kernel, k) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

// lmhead.h -- internal interface of the tensor-core LM-head product
// (lmhead.cu) for the fused verify path in spec_verify.cu.  Not part of the
// C ABI.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "spec_verify.h"

namespace svlm {

constexpr int kTileN = 256;  // vocabulary columns per output tile

// Row statistics of logits = hidden @ weight^T, per (row, 256-column tile):
// part[(r * tiles + t) * 2 + {0, 1}] = (m, s) with m the tile's largest logit
// and s = sum exp2((z - m) * cf), cf = log2(e)/T of the row's sequence; for a
// greedy sequence (greedy flag, or T <= 0, or an invalid T) = (largest logit,
// its lowest column, as int bits).  zgat[r] = the logit at the row's draft
// token, when it has one.  Row r belongs to sequence r / rows_per_seq at
// position r % rows_per_seq; its draft token is tokens[b * N + i] for i < N.
struct StatsArgs {
    const int32_t *tokens;  // [B, N]
    const float *T;         // [B], or null when greedy
    int greedy;
    int N;
    int rows_per_seq;  // N + 1 for the verifier's rows, N for the draft's
    float *part;       // [M, tiles, 2]
    float *zgat;       // [M]
};

inline int tiles(int V) { return (V + kTileN - 1) / kTileN; }

// logits [M, V] f32
sv_status launch_logits(const void *hidden, const void *weight, int M, int V, int K, float *logits,
                        cudaStream_t stream);
// statistics; with `logits` ([M, V] f32, 16-byte aligned, V % 4 == 0) the
// logits as well, from the same accumulators; without it they never leave
// tensor memory
sv_status launch_stats(const void *hidden, const void *weight, int M, int V, int K, const StatsArgs &a,
                       cudaStream_t stream, float *logits = nullptr);

} // namespace svlm

// spec_verify.cu -- GB300 (sm_103a) speculative-sampling verify step.
//
// Three kernel launches per call.
//
// Kernel A (sv_rows_kernel): one verified position (sequence b, position i)
// per thread-block cluster of C CTAs; CTA r owns the r-th contiguous column
// chunk of target row i and, for i < N, draft row i.  Per CTA (8 consumer
// warps + 1 producer warp) the producer streams the chunk through a ring of
// shared-memory stages with 1-D TMA bulk copies (mbarrier complete_tx) and the
// consumers keep an online (max, sum of exp) per row, or (max, argmax) for
// greedy sequences.  The partials are merged over distributed shared memory,
// and position i is decided from the two gathered logits:
//     accept iff p(d) == 0 or u_i < min(1, q(d)/p(d)),
//     q(d) = exp((zq_d - mq)/T)/Sq, p(d) = exp((zp_d - mp)/T)/Sp.
// A rejection lowers the sequence's first-rejection slot (atomicMin); the row
// statistics (mq, Sq, mp, Sp) go to the workspace.
//
// Kernels B (sv_mass_kernel) and C (sv_pick_kernel) sample the emitted token
// at the first rejection j (N if none) from normalise(max(0, q_j - p_j)) (or
// the bonus token from q_N) by inverse CDF: B sums the residual mass of every
// slice of those row pairs with a balanced persistent grid, C finds the slice,
// the thread and the element, writes out_tokens and num_accepted, and resets
// the workspace for the next call, so no memset is ever enqueued.  Only one
// row pair per sequence is read a second time.
//
// Method: "Speculative decoding -- draft, verify, repeat"
// (factory.pai-world.com lesson 07-16), section "Core algorithm", steps 3-6;
// build section Step 1 (rejection step) and Step 2 (residual distribution).
#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cuda_runtime.h>
#include <mutex>

#include "spec_verify.h"
#include "lmhead.h"
#include "sv_device.cuh"

namespace {

constexpr int kConsWarps = 8;
constexpr int kConsThreads = kConsWarps * 32;
constexpr int kThreads = kConsThreads + 32;  // + one producer warp
constexpr int kProducerWarp = kConsWarps;
constexpr int kVPT = 2;                      // 16-byte vectors per consumer thread, row and stage
constexpr int kSliceVecs = kConsThreads;     // one vector per consumer thread: the scan unit
constexpr int kTileVecs = kVPT * kSliceVecs; // vectors per row and stage
constexpr int kTileBytes = kTileVecs * 16;
constexpr int kStagesA = 3;                  // ring depth of the row kernel
__host__ __device__ constexpr int ring_bytes(int stages) { return stages * 2 * kTileBytes; }
constexpr int kMaxSlices = 128;              // slices per chunk (512 KiB of one row)
constexpr int kMaxCluster = 16;
constexpr int kPackMaxB = 1024;              // sequences whose sampled flags one warp holds (32 per lane)
constexpr int kProfRuns = 4096;  // runs whose kernel times one profiling session keeps
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait, then give up

constexpr int kNoReject = 0x7f7f7f7f;        // byte pattern 0x7f: memset-able
constexpr int kErrBadToken = 1;
constexpr int kErrBadValue = 2;
constexpr int kErrTimeout = 4;
constexpr int kErrBadTree = 8;

enum { MODE_INVALID = 0, MODE_GREEDY = 1, MODE_SAMPLED = 2 };
enum { RES_DIFF = 0, RES_Q = 1 };

constexpr double kLog2e = 1.4426950408889634074;

struct SvParams {
    const void *target;
    const void *draft;
    const int32_t *tokens;
    const float *u;
    const float *T;
    int32_t *out;
    int32_t *nacc;
    float *q_at;
    float *p_at;
    float *tstats;
    float *dstats;
    float *ratio_at;  // debug: the ratio each accept test compared u with (NaN where none)
    int *ws_first;    // [max_B] first rejected position, kNoReject if none
    int *ws_err;      // [max_B] error bits of the sequence
    int *ws_tok;      // [max_B*(max_N+1)] greedy argmax of each position
    unsigned long long *ws_xc;  // [max_B*(max_N+1)] (m, S) of a position's first normalised row (one-row units), 0 between calls
    float *ws_stats;  // [max_B*(max_N+1)][4] (mq, Sq, mp, Sp) of each position
    float *ws_slice;  // [max_B*slices][8] residual mass of each warp's share of a slice
    int *status;      // sticky error bits of the context
    unsigned long long *hist;          // [N+1] sequences by accepted drafts (may be NULL)
    unsigned long long *hist_invalid;  // sequences that were invalid
    // tree verification (N is then the node count M; rows are per node)
    const int32_t *parent;  // [B][M+1]
    int32_t *path;          // [B][M+1] accepted node ids
    // fused LM-head path: the sampling kernels read row b of a compact
    // [B, V] buffer instead of the rows (b, j) of the full logits (target
    // and draft rows separately)
    int compact_t, compact_d;
    int B, N, V, greedy;
};

// Rows the sampling kernels read for sequence b stopping at position j.
__device__ __forceinline__ size_t sample_trow(const SvParams &p, int b, int j)
{
    return p.compact_t ? (size_t)b : (size_t)b * (p.N + 1) + j;
}

__device__ __forceinline__ size_t sample_drow(const SvParams &p, int b, int j)
{
    return p.compact_d ? (size_t)b : (size_t)b * p.N + j;
}

// Producer/consumer ring state in shared memory.
template <int S> struct Ring {
    static constexpr int kStages = S;
    uint64_t full[S];
    uint64_t empty[S];
    int last_g[S];  // last ring position issued into each stage
    int abort;
};

// Shared-memory control blocks (after the ring).  Fields read by peer CTAs
// over DSMEM are written before a cluster barrier and not rewritten after it.
struct CtlA {
    Ring<kStagesA> ring;
    double cfd;                    // log2(e) / T
    float cf;                      // the same, rounded to float
    float pm_t, ps_t, pm_d, ps_d;  // sampled partials (target, draft)
    float gv;                      // greedy partial
    int gi, gnan;
    float zq_d, zp_d, u_i;         // the decision's inputs
    int has_child;                 // tree: the node has children (its draft row is read)
    float red_m[kConsWarps], red_s[kConsWarps], red_m2[kConsWarps], red_s2[kConsWarps];
    int red_i[kConsWarps], red_n[kConsWarps];
};

constexpr size_t kSmemA = ring_bytes(kStagesA) + sizeof(CtlA);

template <int DT> struct Elt;
template <> struct Elt<SV_F32> {
    static constexpr int kPerVec = 4;  // elements per 16-byte vector
};
template <> struct Elt<SV_BF16> {
    static constexpr int kPerVec = 8;
};

template <int DT>
__device__ __forceinline__ void unpack(const uint4 v, float *z)
{
    if constexpr (DT == SV_BF16) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            z[2 * k] = __uint_as_float(w[k] << 16);
            z[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    } else {
        z[0] = __uint_as_float(v.x);
        z[1] = __uint_as_float(v.y);
        z[2] = __uint_as_float(v.z);
        z[3] = __uint_as_float(v.w);
    }
}

template <int DT>
__device__ __forceinline__ float logit_at(const void *base, size_t idx)
{
    if constexpr (DT == SV_BF16) {
        const unsigned short bits = __ldg(static_cast<const unsigned short *>(base) + idx);
        return __uint_as_float(static_cast<uint32_t>(bits) << 16);
    } else {
        return __ldg(static_cast<const float *>(base) + idx);
    }
}

// ---- online softmax normaliser: m = running max, s = sum exp2((z - m) c) ----
struct Online {
    float m, s;
};

__device__ __forceinline__ Online online_merge(Online a, Online b, float cf)
{
    const float m = fmaxf(a.m, b.m);
    const float sa = (a.m == m) ? a.s : a.s * sv::ex2((a.m - m) * cf);
    const float sb = (b.m == m) ? b.s : b.s * sv::ex2((b.m - m) * cf);
    return {m, sa + sb};
}

__device__ __forceinline__ Online warp_merge(Online o, float cf)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Online p;
        p.m = __shfl_xor_sync(0xffffffffu, o.m, off);
        p.s = __shfl_xor_sync(0xffffffffu, o.s, off);
        o = online_merge(o, p, cf);
    }
    return o;
}

// K 16-byte vectors of logits (one ring tile's share of a thread) into its
// running normaliser, without branches: M = max(m, tile max) (the tile max on
// bf16x2 words for bf16, exact; NaN never the max), the sums are scaled by
// exp2((m - M) c) when the max moved (else by 1), and every element adds
// exp2((z - M) c), the arguments and the sums on f32x2 pairs so that the
// thread keeps two partial sums (even and odd elements).  While only -inf has
// been seen M is -inf and the arguments are taken against 0 instead, so the
// sums stay 0; a NaN element makes them NaN.  Elements past the row's end are
// passed as -inf.
//
// For bf16 the argument is z c - K in one rounding (fma), K = fl(M c).  That
// shifts every term by the same e = M c - K (the rounding error of M c, up to
// half an ulp of M c: about 1e-6 in log2 units at |M c| = 50), so the sum is
// 2^e times sum exp2((z - M) c).  The rescale when the max moves is
// exp2(K_old - K_new), which keeps one common shift e of the final M in the
// whole sum, and online_fold removes it: e = fma(M, c, -K) exactly, and the
// sum is multiplied by 2^-e = 1 - e ln 2 (to within e^2).
struct Online2 {
    float m;
    unsigned long long s;  // (even, odd) partial sums
};

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int DT, int K>
__device__ __forceinline__ void online_add_tile(Online2 &o, const uint4 (&v)[K], float cf)
{
    constexpr int NP = (DT == SV_BF16) ? 4 : 2;  // f32x2 pairs per vector
    float vmax;
    if constexpr (DT == SV_BF16) {
        uint32_t mx = sv::bmax2(sv::bmax2(v[0].x, v[0].y), sv::bmax2(v[0].z, v[0].w));
#pragma unroll
        for (int k = 1; k < K; ++k)
            mx = sv::bmax2(mx, sv::bmax2(sv::bmax2(v[k].x, v[k].y), sv::bmax2(v[k].z, v[k].w)));
        vmax = fmaxf(lo_bf16(mx), hi_bf16(mx));
    } else {
        vmax = -INFINITY;
#pragma unroll
        for (int k = 0; k < K; ++k)
            vmax = fmaxf(vmax, fmaxf(fmaxf(__uint_as_float(v[k].x), __uint_as_float(v[k].y)),
                                     fmaxf(__uint_as_float(v[k].z), __uint_as_float(v[k].w))));
    }
    const float M = fmaxf(o.m, vmax);
    const float Ms = (M == -INFINITY) ? 0.0f : M;
    // the arguments' shift, new and so far (bf16; -inf before any finite max),
    // each rounded once and never contracted
    const float Kn = __fmul_rn(Ms, cf), Ko = __fmul_rn(o.m, cf);
    float r;
    if constexpr (DT == SV_BF16)
        r = (vmax > o.m) ? sv::ex2(__fsub_rn(Ko, Kn)) : 1.0f;
    else
        r = (vmax > o.m) ? sv::ex2((o.m - vmax) * cf) : 1.0f;
    const unsigned long long Cf = sv::pack2(cf, cf);
    unsigned long long e[K * NP];
    if constexpr (DT == SV_BF16) {
        const float nmc = -Kn;
        const unsigned long long Nmc = sv::pack2(nmc, nmc);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float a0, a1;
                sv::unpack2(sv::fma2(sv::pack2(lo_bf16(w[q]), hi_bf16(w[q])), Cf, Nmc), a0, a1);
                e[k * NP + q] = sv::pack2(sv::ex2(a0), sv::ex2(a1));
            }
        }
    } else {
        const unsigned long long Mp = sv::pack2(Ms, Ms);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const unsigned long long z[2] = {sv::pack2(__uint_as_float(v[k].x), __uint_as_float(v[k].y)),
                                             sv::pack2(__uint_as_float(v[k].z), __uint_as_float(v[k].w))};
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float a0, a1;
                sv::unpack2(sv::mul2(sv::sub2(z[q], Mp), Cf), a0, a1);
                e[k * NP + q] = sv::pack2(sv::ex2(a0), sv::ex2(a1));
            }
        }
    }
    // pairwise sum of the K * NP pairs
#pragma unroll
    for (int w = 1; w < K * NP; w *= 2)
#pragma unroll
        for (int q = 0; q + w < K * NP; q += 2 * w)
            e[q] = sv::add2(e[q], e[q + w]);
    o.s = sv::fma2(o.s, sv::pack2(r, r), e[0]);
    o.m = M;
}

// Elements past a row's end: -inf in every lane of a vector.
template <int DT> __device__ __forceinline__ uint4 neg_inf_vec()
{
    constexpr uint32_t w = (DT == SV_BF16) ? 0xff80ff80u : 0xff800000u;
    return make_uint4(w, w, w, w);
}

// A thread's (m, s) from its running state.  For bf16 the common shift
// e = m c - fl(m c) of every term is taken out: s * 2^-e = s - s e ln 2.
template <int DT>
__device__ __forceinline__ Online online_fold(const Online2 &o, float cf)
{
    float a, b;
    sv::unpack2(o.s, a, b);
    float s = a + b;
    if constexpr (DT == SV_BF16) {
        if (isfinite(o.m)) {
            const float e = fmaf(o.m, cf, -__fmul_rn(o.m, cf));
            s = fmaf(s, -(e * 0.6931471805599453f), s);
        }
    }
    return {o.m, s};
}

// ---- greedy: max, lowest index of the max, NaN seen --------------------------
struct ArgMax {
    float v;
    int i;
    int nan;
};

// One 16-byte vector of logits into a thread's running argmax: the vector max
// (and a NaN test) on bf16x2 words or pairs of floats, NaN never the max; when
// it exceeds the running max, the lowest column of the vector holding it.
template <int DT>
__device__ __forceinline__ void argmax_add2(ArgMax &a, const uint4 v, int col0)
{
    constexpr int NE = Elt<DT>::kPerVec;
    float vmax;
    int nan;
    if constexpr (DT == SV_BF16) {
        const uint32_t mx = sv::bmax2(sv::bmax2(v.x, v.y), sv::bmax2(v.z, v.w));
        const uint32_t mn = sv::bmax2_nan(sv::bmax2_nan(v.x, v.y), sv::bmax2_nan(v.z, v.w));
        vmax = fmaxf(lo_bf16(mx), hi_bf16(mx));
        nan = mx != mn;
    } else {
        const float x = __uint_as_float(v.x), y = __uint_as_float(v.y);
        const float zz = __uint_as_float(v.z), w = __uint_as_float(v.w);
        vmax = fmaxf(fmaxf(x, y), fmaxf(zz, w));
        const float vn = sv::fmax_nan(sv::fmax_nan(x, y), sv::fmax_nan(zz, w));
        nan = vn != vn;
    }
    a.nan |= nan;
    if (vmax > a.v) {
        float z[NE];
        unpack<DT>(v, z);
        int best = NE - 1;
#pragma unroll
        for (int k = NE - 1; k >= 0; --k)
            if (z[k] == vmax)
                best = k;
        a.v = vmax;
        a.i = col0 + best;
    }
}

__device__ __forceinline__ ArgMax argmax_merge(ArgMax a, ArgMax b)
{
    ArgMax r = (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
    r.nan = a.nan | b.nan;
    return r;
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ArgMax p;
        p.v = __shfl_xor_sync(0xffffffffu, a.v, off);
        p.i = __shfl_xor_sync(0xffffffffu, a.i, off);
        p.nan = __shfl_xor_sync(0xffffffffu, a.nan, off);
        a = argmax_merge(a, p);
    }
    return a;
}

// ---- residual mass of one 16-byte vector --------------------------------------
// r_k = max(0, q_k - p_k) (RES_DIFF) or q_k (RES_Q), with
// q_k = 2^((zq_k - mq) c) / Sq evaluated as 2^(zq_k c - Kq) * Iq: the argument
// in one rounding against the shift Kq = fl(mq c), whose rounding error e is
// folded into the row's scale, Iq = (1 - e ln 2) / Sq (residual_shift below),
// and q_k - p_k = fma(2^(..) , Iq, -p_k) in one rounding.  Adjacent elements
// k, k+1 travel as one f32x2 pair (they come out of one bf16x2 word, or two
// neighbouring floats).  Every operation rounds to nearest and nothing is
// contracted, so the result is bit-identical wherever it is recomputed
// (kernels B and C).
template <int DT>
__device__ __forceinline__ void residual_vec(const uint4 vt, const uint4 vd, int res_mode, float Kq,
                                             float Iq_, float Kp, float Ip_, float cf, float *r)
{
    constexpr int NE = Elt<DT>::kPerVec;
    constexpr int NP = NE / 2;
    unsigned long long zt[NP], zd[NP];
    const uint32_t wt[4] = {vt.x, vt.y, vt.z, vt.w};
    const uint32_t wd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        if constexpr (DT == SV_BF16) {
            zt[k] = sv::pack2(__uint_as_float(wt[k] << 16), __uint_as_float(wt[k] & 0xffff0000u));
            zd[k] = sv::pack2(__uint_as_float(wd[k] << 16), __uint_as_float(wd[k] & 0xffff0000u));
        } else {
            zt[k] = sv::pack2(__uint_as_float(wt[2 * k]), __uint_as_float(wt[2 * k + 1]));
            zd[k] = sv::pack2(__uint_as_float(wd[2 * k]), __uint_as_float(wd[2 * k + 1]));
        }
    }
    const unsigned long long Cf = sv::pack2(cf, cf);
    const unsigned long long NKq = sv::pack2(-Kq, -Kq), Iq = sv::pack2(Iq_, Iq_);
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        float a0, a1;
        sv::unpack2(sv::fma2(zt[k], Cf, NKq), a0, a1);
        const unsigned long long eq = sv::pack2(sv::ex2(a0), sv::ex2(a1));
        if (res_mode == RES_DIFF) {
            const unsigned long long NKp = sv::pack2(-Kp, -Kp), NIp = sv::pack2(-Ip_, -Ip_);
            sv::unpack2(sv::fma2(zd[k], Cf, NKp), a0, a1);
            const unsigned long long npk = sv::mul2(sv::pack2(sv::ex2(a0), sv::ex2(a1)), NIp);  // -p
            float d0, d1;
            sv::unpack2(sv::fma2(eq, Iq, npk), d0, d1);
            r[2 * k] = fmaxf(d0, 0.0f);
            r[2 * k + 1] = fmaxf(d1, 0.0f);
        } else {
            sv::unpack2(sv::mul2(eq, Iq), r[2 * k], r[2 * k + 1]);
        }
    }
}

// The shift and scale of a row for residual_vec from its statistics (m, S):
// K = fl(m c), e = m c - K exactly (fma), I = (1 - e ln 2) / S.
__device__ __forceinline__ void residual_shift(float m, float S, float cf, float &K, float &I)
{
    K = __fmul_rn(m, cf);
    const float e = fmaf(m, cf, -K);
    I = __fmul_rn(1.0f / S, fmaf(-e, 0.6931471805599453f, 1.0f));
}

__device__ __forceinline__ float warp_incl_scan(float x, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x = __fadd_rn(x, y);
    }
    return x;
}

// The warp's total of x, in every lane, by a xor butterfly.  Bit for bit the
// value warp_incl_scan leaves in lane 31: at step o both add to lane 31's
// partial the partial of lane 31 - o (= 31 xor o), which in both covers the
// same o lanes summed by the same tree, so every addition has the same
// operands in the same order.
__device__ __forceinline__ float warp_total(float x)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1)
        x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// ---- ring of shared-memory stages fed by TMA bulk copies --------------------
// Issues ring tiles [t_begin, t_end) of the chunk into ring positions g, g+1,
// ...  Runs on one lane of the producer warp.
template <typename RingT>
__device__ __forceinline__ void produce(RingT &rg, unsigned char *ring, const uint4 *tsrc, const uint4 *dsrc,
                                        int nvec_chunk, int t_begin, int t_end, uint32_t g)
{
    constexpr int kStages = RingT::kStages;
    for (int t = t_begin; t < t_end; ++t, ++g) {
        const uint32_t s = g % kStages;
        const uint32_t ph = (g / kStages) & 1u;
        if (!sv::mbar_wait_bounded(&rg.empty[s], ph ^ 1u, &rg.abort, kWaitLimitNs)) {
            rg.abort = 1;
            return;
        }
        const int nvec = min(kTileVecs, nvec_chunk - t * kTileVecs);
        const uint32_t bytes = static_cast<uint32_t>(nvec) * 16u;
        sv::mbar_arrive_expect_tx(&rg.full[s], dsrc ? 2u * bytes : bytes);
        unsigned char *stage = ring + s * (2 * kTileBytes);
        sv::bulk_g2s(stage, tsrc + (size_t)t * kTileVecs, bytes, &rg.full[s]);
        if (dsrc)
            sv::bulk_g2s(stage + kTileBytes, dsrc + (size_t)t * kTileVecs, bytes, &rg.full[s]);
        rg.last_g[s] = static_cast<int>(g);
    }
}

// Consumer side: wait until ring position g is filled.
template <typename RingT>
__device__ __forceinline__ bool consume_wait(RingT &rg, uint32_t g)
{
    constexpr int kStages = RingT::kStages;
    const uint32_t s = g % kStages;
    return sv::mbar_wait_bounded(&rg.full[s], (g / kStages) & 1u, &rg.abort, kWaitLimitNs);
}

template <typename RingT>
__device__ __forceinline__ void consume_release(RingT &rg, uint32_t g, int lane)
{
    __syncwarp();
    if (lane == 0)
        sv::mbar_arrive(&rg.empty[g % RingT::kStages]);
}

// Called by thread 0 before the first __syncthreads of a kernel.
template <typename RingT>
__device__ __forceinline__ void ring_init(RingT &rg)
{
    for (int s = 0; s < RingT::kStages; ++s) {
        sv::mbar_init(&rg.full[s], 1);
        sv::mbar_init(&rg.empty[s], kConsWarps);
        rg.last_g[s] = -1;
    }
    rg.abort = 0;
    sv::fence_mbar_init();
}

// After an abort: never leave with a bulk copy still writing into this CTA's
// shared memory (bounded wait on the last copy issued into each stage).
template <typename RingT>
__device__ __forceinline__ void ring_drain(RingT &rg)
{
    for (int s = 0; s < RingT::kStages; ++s) {
        const int lg = rg.last_g[s];
        if (lg >= 0) {
            int never = 0;
            sv::mbar_wait_bounded(&rg.full[s], ((uint32_t)lg / RingT::kStages) & 1u, &never, kWaitLimitNs / 4);
        }
    }
}

__device__ __forceinline__ int sequence_mode(const SvParams &p, int b, float &T)
{
    T = 0.0f;
    if (p.greedy)
        return MODE_GREEDY;
    T = p.T[b];
    if (T != T)
        return MODE_INVALID;
    if (T <= 0.0f)
        return MODE_GREEDY;
    if (T == INFINITY || T < FLT_MIN)
        return MODE_INVALID;
    return MODE_SAMPLED;
}

// Column chunk of CTA `rank` of `C`, in 16-byte vectors.
struct Chunk {
    int v0, nvec, ntiles, nslices;
};

__device__ __forceinline__ Chunk chunk_of(int NV, uint32_t rank, uint32_t C)
{
    Chunk c;
    c.v0 = (int)((long long)NV * rank / C);
    const int v1 = (int)((long long)NV * (rank + 1) / C);
    c.nvec = v1 - c.v0;
    c.ntiles = (c.nvec + kTileVecs - 1) / kTileVecs;
    c.nslices = (c.nvec + kSliceVecs - 1) / kSliceVecs;
    return c;
}

// The ratio q(x)/p(x) of the accept test of a draft token x, evaluated in the
// log domain.  cfd = log2(e)/T in double; with lq = (zq - mq) cfd and
// lp = (zp - mp) cfd (both exact differences, one rounding each), the ratio is
// 2^(lq - lp) * Sp/Sq: the integer part of lq - lp goes to the exponent and the
// fractional part through ex2, so no double-precision exp or division is on
// the common path.  Only when an argument nears double underflow are q(x) and
// p(x) evaluated as the definition does.  p(x) == 0 gives +inf; q(x) == 0
// gives 0.
__device__ __forceinline__ double decision_ratio(float zq, float zp, float mq, float Sq, float mp, float Sp,
                                                 double cfd)
{
    if (zp == -INFINITY)
        return INFINITY;
    if (zq == -INFINITY)
        return 0.0;
    const double lq = ((double)zq - (double)mq) * cfd;
    const double lp = ((double)zp - (double)mp) * cfd;
    if (lq < -1000.0 || lp < -1000.0) {
        const double qd = exp2(lq) / (double)Sq, pd = exp2(lp) / (double)Sp;
        return (pd == 0.0) ? INFINITY : qd / pd;
    }
    const double L = lq - lp;
    const double fl = floor(L);
    const float frac = (float)(L - fl);
    return ldexp((double)(sv::ex2(frac) * (Sp / Sq)), (int)fl);
}

// u < min(1, ratio); an infinite ratio (p(x) == 0) accepts whatever u is, and
// a zero ratio (q(x) == 0) never does (u < 0 never holds).
__device__ __forceinline__ bool accept_by_ratio(double ratio, double u)
{
    return ratio == INFINITY || u < fmin(1.0, ratio);
}


// =============================================================================
// Kernel A: row normalisers and accept decisions, one cluster per position
// =============================================================================
//
// Positions are taken in descending order (all sequences at position N, then
// N-1, ..., then 0) so that position 0, where most first rejections happen,
// is read last and is still in L2 when kernel B samples there.
template <int DT, bool TREE>
__global__ void __launch_bounds__(kThreads, 4) sv_rows_kernel(const SvParams p)
{
    constexpr int VE = Elt<DT>::kPerVec;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    constexpr int kStages = kStagesA;
    CtlA &ctl = *reinterpret_cast<CtlA *>(smem + ring_bytes(kStages));

    if constexpr (TREE)
        sv::grid_launch_dependents();  // the walk's clusters may start on SMs as this grid's CTAs retire
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t C = sv::cluster_nctarank();
    const uint32_t rank = sv::cluster_ctarank();
    const int N = p.N, V = p.V;
    const int unit = blockIdx.x / C;
    const int pos = unit / p.B;
    const int i = N - pos;
    const int b = unit - pos * p.B;

    float T;
    const int mode = sequence_mode(p, b, T);
    const size_t trow = (size_t)b * (N + 1) + i;
    const size_t drow = TREE ? trow : (size_t)b * N + i;
    int d = 0;
    bool bad_d = false, bad_tree = false;
    if constexpr (TREE) {
        // node i: its token (i >= 1) and its parent must be valid
        if (i > 0) {
            d = p.tokens[trow];
            bad_d = d < 0 || d >= V;
        }
        const int par = p.parent[trow];
        bad_tree = (i == 0) ? (par != -1) : (par < 0 || par >= i);
    } else {
        d = (i < N) ? p.tokens[(size_t)b * N + i] : 0;
        bad_d = (i < N) && (d < 0 || d >= V);
    }

    const Chunk ch = chunk_of(V / VE, rank, C);
    const size_t row_vecs = (size_t)(V / VE);
    const uint4 *tsrc = static_cast<const uint4 *>(p.target) + trow * row_vecs + ch.v0;

    if (tid == 0) {
        ring_init(ctl.ring);
        const double cfd = (mode == MODE_SAMPLED) ? kLog2e / (double)T : 0.0;
        ctl.cfd = cfd;
        ctl.cf = (float)cfd;
    }
    if constexpr (TREE) {
        // a node's draft row is read only when the node has children
        if (warp == kProducerWarp) {
            bool any = false;
            for (int c = i + 1 + lane; c <= N; c += 32)
                any |= p.parent[(size_t)b * (N + 1) + c] == i;
            any = __any_sync(0xffffffffu, any);
            if (lane == 0)
                ctl.has_child = any ? 1 : 0;
        }
    }
    // The decision's inputs are loaded by an idle lane of the producer warp at
    // the start and parked in shared memory after pass 1.
    const bool prefetcher = !TREE && rank == 0 && tid == 32 * kProducerWarp + 1;
    float pre_zq = 0.0f, pre_zp = 0.0f, pre_u = 0.0f;
    if (prefetcher && mode == MODE_SAMPLED && i < N && !bad_d) {
        pre_zq = logit_at<DT>(p.target, trow * (size_t)V + d);
        pre_zp = logit_at<DT>(p.draft, drow * (size_t)V + d);
        pre_u = p.u[trow];
    }
    __syncthreads();
    const float cf = ctl.cf;
    const bool has_draft = (mode == MODE_SAMPLED) && (TREE ? ctl.has_child != 0 : i < N);
    const uint4 *dsrc = has_draft ? static_cast<const uint4 *>(p.draft) + drow * row_vecs + ch.v0 : nullptr;

    // ---- pass 1: stream the chunk of both rows once
    Online2 ot2{-INFINITY, 0ull}, od2{-INFINITY, 0ull};  // 0ull = (+0.0f, +0.0f)
    ArgMax ga{-INFINITY, INT_MAX, 0};
    if (mode != MODE_INVALID) {
        if (warp == kProducerWarp) {
            if (lane == 0)
                produce(ctl.ring, ring, tsrc, dsrc, ch.nvec, 0, ch.ntiles, 0);
            __syncwarp();
        } else {
            for (int t = 0; t < ch.ntiles; ++t) {
                if (consume_wait(ctl.ring, t)) {
                    const unsigned char *stage = ring + (t % kStages) * (2 * kTileBytes);
                    if (mode == MODE_GREEDY) {
#pragma unroll
                        for (int k = 0; k < kVPT; ++k) {
                            const int sv_ = k * kSliceVecs + tid;  // vector within the stage
                            const int vec = t * kTileVecs + sv_;
                            if (vec < ch.nvec)
                                argmax_add2<DT>(ga, reinterpret_cast<const uint4 *>(stage)[sv_], (ch.v0 + vec) * VE);
                        }
                    } else {
                        uint4 vt[kVPT], vd[kVPT];
#pragma unroll
                        for (int k = 0; k < kVPT; ++k) {
                            const int sv_ = k * kSliceVecs + tid;
                            const bool in = t * kTileVecs + sv_ < ch.nvec;
                            vt[k] = in ? reinterpret_cast<const uint4 *>(stage)[sv_] : neg_inf_vec<DT>();
                            vd[k] = (in && has_draft) ? reinterpret_cast<const uint4 *>(stage + kTileBytes)[sv_]
                                                      : neg_inf_vec<DT>();
                        }
                        online_add_tile<DT, kVPT>(ot2, vt, cf);
                        if (has_draft)
                            online_add_tile<DT, kVPT>(od2, vd, cf);
                    }
                } else {
                    ctl.ring.abort = 1;
                }
                consume_release(ctl.ring, t, lane);
            }
        }
    }

    if (prefetcher) {
        ctl.zq_d = pre_zq;
        ctl.zp_d = pre_zp;
        ctl.u_i = pre_u;
    }

    // ---- CTA partial
    Online ot = online_fold<DT>(ot2, cf), od = online_fold<DT>(od2, cf);
    if (warp < kConsWarps) {
        if (mode == MODE_GREEDY) {
            ga = warp_argmax(ga);
            if (lane == 0) {
                ctl.red_m[warp] = ga.v;
                ctl.red_i[warp] = ga.i;
                ctl.red_n[warp] = ga.nan;
            }
        } else if (mode == MODE_SAMPLED) {
            ot = warp_merge(ot, cf);
            od = warp_merge(od, cf);
            if (lane == 0) {
                ctl.red_m[warp] = ot.m;
                ctl.red_s[warp] = ot.s;
                ctl.red_m2[warp] = od.m;
                ctl.red_s2[warp] = od.s;
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        if (mode == MODE_GREEDY) {
            ArgMax a{ctl.red_m[0], ctl.red_i[0], ctl.red_n[0]};
            for (int w = 1; w < kConsWarps; ++w)
                a = argmax_merge(a, ArgMax{ctl.red_m[w], ctl.red_i[w], ctl.red_n[w]});
            ctl.gv = a.v;
            ctl.gi = a.i;
            ctl.gnan = a.nan;
        } else if (mode == MODE_SAMPLED) {
            Online a{ctl.red_m[0], ctl.red_s[0]}, e{ctl.red_m2[0], ctl.red_s2[0]};
            for (int w = 1; w < kConsWarps; ++w) {
                a = online_merge(a, Online{ctl.red_m[w], ctl.red_s[w]}, cf);
                e = online_merge(e, Online{ctl.red_m2[w], ctl.red_s2[w]}, cf);
            }
            ctl.pm_t = a.m;
            ctl.ps_t = a.s;
            ctl.pm_d = e.m;
            ctl.ps_d = e.s;
        }
    }
    if (C > 1)
        sv::cluster_sync();  // partials visible cluster-wide
    else
        __syncthreads();

    // ---- merge over the cluster and decide (rank 0 only: the others are done)
    // Warp 0 merges the C partials (lane r reads CTA r over DSMEM); lane 0
    // decides position i and records the outcome for kernel B.
    if (rank == 0 && warp == 0) {
        if (mode == MODE_GREEDY) {
            ArgMax a{-INFINITY, INT_MAX, 0};
            if (lane < (int)C) {
                a.v = sv::ld_dsmem_f32(sv::dsmem_addr(&ctl.gv, lane));
                a.i = sv::ld_dsmem_s32(sv::dsmem_addr(&ctl.gi, lane));
                a.nan = sv::ld_dsmem_s32(sv::dsmem_addr(&ctl.gnan, lane));
            }
            a = warp_argmax(a);
            if (lane == 0) {
                int errb = (bad_d ? kErrBadToken : 0) | (bad_tree ? kErrBadTree : 0);
                if (a.nan || a.v == INFINITY || a.v == -INFINITY)
                    errb |= kErrBadValue;
                p.ws_tok[trow] = a.i;
                if (!TREE && i < N && d != a.i)
                    atomicMin(&p.ws_first[b], i);
                if (errb)
                    atomicOr(&p.ws_err[b], errb);
                if (p.tstats) {
                    p.tstats[trow * 2 + 0] = a.v;
                    p.tstats[trow * 2 + 1] = NAN;
                }
                if (!TREE && i < N) {
                    if (p.q_at)
                        p.q_at[drow] = NAN;
                    if (p.p_at)
                        p.p_at[drow] = NAN;
                    if (p.ratio_at)
                        p.ratio_at[drow] = NAN;
                    if (p.dstats) {
                        p.dstats[drow * 2 + 0] = NAN;
                        p.dstats[drow * 2 + 1] = NAN;
                    }
                }
            }
        } else if (mode == MODE_SAMPLED) {
            Online t{-INFINITY, 0.0f}, e{-INFINITY, 0.0f};
            if (lane < (int)C) {
                t.m = sv::ld_dsmem_f32(sv::dsmem_addr(&ctl.pm_t, lane));
                t.s = sv::ld_dsmem_f32(sv::dsmem_addr(&ctl.ps_t, lane));
                if (has_draft) {
                    e.m = sv::ld_dsmem_f32(sv::dsmem_addr(&ctl.pm_d, lane));
                    e.s = sv::ld_dsmem_f32(sv::dsmem_addr(&ctl.ps_d, lane));
                }
            }
            t = warp_merge(t, cf);
            e = warp_merge(e, cf);
            if (lane == 0) {
                int errb = (bad_d ? kErrBadToken : 0) | (bad_tree ? kErrBadTree : 0);
                const float mq = t.m, Sq = t.s, mp = e.m, Sp = e.s;
                bool valid = isfinite(mq) && isfinite(Sq) && Sq > 0.0f;
                if (has_draft)
                    valid = valid && isfinite(mp) && isfinite(Sp) && Sp > 0.0f;
                if (!TREE && i < N && p.ratio_at)
                    p.ratio_at[drow] = NAN;
                if (!valid) {
                    errb |= kErrBadValue;
                } else if (!TREE && i < N && !bad_d) {
                    const float zq = ctl.zq_d, zp = ctl.zp_d;
                    const double cfd = ctl.cfd;
                    const double ratio = decision_ratio(zq, zp, mq, Sq, mp, Sp, cfd);
                    if (!accept_by_ratio(ratio, (double)ctl.u_i))
                        atomicMin(&p.ws_first[b], i);
                    if (p.ratio_at)
                        p.ratio_at[drow] = (float)ratio;
                    if (p.q_at)
                        p.q_at[drow] = (float)(exp2(((double)zq - (double)mq) * cfd) / (double)Sq);
                    if (p.p_at)
                        p.p_at[drow] = (float)(exp2(((double)zp - (double)mp) * cfd) / (double)Sp);
                }
                float *st = p.ws_stats + trow * 4;
                st[0] = mq;
                st[1] = Sq;
                st[2] = mp;
                st[3] = Sp;
                if (errb)
                    atomicOr(&p.ws_err[b], errb);
                if (p.tstats) {
                    p.tstats[trow * 2 + 0] = mq;
                    p.tstats[trow * 2 + 1] = Sq;
                }
                if (p.dstats && has_draft) {
                    p.dstats[drow * 2 + 0] = mp;
                    p.dstats[drow * 2 + 1] = Sp;
                }
            }
        } else if (lane == 0) {
            atomicOr(&p.ws_err[b], kErrBadValue | (bad_d ? kErrBadToken : 0) | (bad_tree ? kErrBadTree : 0));
            if (!TREE && i < N && p.ratio_at)
                p.ratio_at[drow] = NAN;
        }
    }
    if (tid == 0 && ctl.ring.abort)
        atomicOr(&p.ws_err[b], kErrTimeout);
    if (C > 1)
        sv::cluster_sync();  // no peer reads this CTA's shared memory any more
    if (tid == 0 && ctl.ring.abort)
        ring_drain(ctl.ring);
}

// =============================================================================
// Kernel A1: one logit row per CTA (batches with a CTA per position)
// =============================================================================
//
// Where kernel A would run one CTA per position (no cluster), the units are
// single rows instead: a sampled position's target and draft rows are two
// CTAs, a greedy or bonus position's target row one.  Every unit then streams
// the same number of bytes, so one-wave batches (a mixed batch whose greedy
// positions read half as much) and the last wave of large ones do not end on
// a tail of two-row units.  Each ring stage holds two consecutive 8 KiB tiles
// of the one row (the same 16 KiB in flight per stage, the same 32 elements
// per thread and stage).  A position's two rows meet in one 64-bit workspace
// cell: each CTA swaps its row's (m, S) in, and the one that finds the other
// row's pair there decides with kernel A's arithmetic.  Units run position by position in
// descending order (position 0 last, as in kernel A), a sequence's two rows
// next to each other; a draft-row unit of a greedy sequence (or of a tree node
// without children) reads nothing and leaves.  PACKED (chains of at most
// kPackMaxB sequences): the rows that are read take the front of the grid,
// and no block is spent on a draft row that is not read.
template <int DT, bool TREE, bool PACKED = false>
__global__ void __launch_bounds__(kThreads, 4) sv_row_kernel(const SvParams p)
{
    constexpr int VE = Elt<DT>::kPerVec;
    constexpr int kStageVecs = 2 * kTileVecs;  // vectors of the row per ring stage
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    constexpr int kStages = kStagesA;
    CtlA &ctl = *reinterpret_cast<CtlA *>(smem + ring_bytes(kStages));

    // The next grid (the tree walk, or the chain's mass kernel) may start its
    // CTAs on SMs as this grid's retire; they wait for its results on the
    // device (mixed batch 47.75 -> 47.34 us per call, headline 202.4 -> 202.2
    // us; the same trigger in kernel A cost the small batches ~2 us).
    sv::grid_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N = p.N, V = p.V, B = p.B;
    int i, b, is_draft;
    {
        const int u = blockIdx.x;
        if (TREE) {  // every node may have a draft row
            const int pos = u / (2 * B), w = u - pos * (2 * B);
            i = N - pos;
            b = w >> 1;
            is_draft = w & 1;
        } else if (u < B) {  // position N: target rows only
            i = N;
            b = u;
            is_draft = 0;
        } else if (PACKED) {
            // The B(N+1) target rows first (positions in descending order),
            // then the draft rows of the nS sampled sequences at positions
            // N-1 .. 0; blocks past the last of them leave.  A draft block's
            // warps each read the sampled flags of all sequences (lane w holds
            // those of sequences 32w .. 32w + 31) and map the block themselves.
            if (u < B * (N + 1)) {
                const int pos = u / B;
                i = N - pos;
                b = u - pos * B;
                is_draft = 0;
            } else {
                uint32_t word = 0;
                if (lane * 32 < B) {
                    float Tb;
#pragma unroll 8
                    for (int k = 0; k < 32; ++k) {
                        const int bb = lane * 32 + k;
                        if (bb < B && sequence_mode(p, bb, Tb) == MODE_SAMPLED)
                            word |= 1u << k;
                    }
                }
                int cum = __popc(word);  // inclusive prefix over lanes
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int o = __shfl_up_sync(0xffffffffu, cum, off);
                    if (lane >= off)
                        cum += o;
                }
                const int nS = __shfl_sync(0xffffffffu, cum, 31);
                const int v = u - B * (N + 1);
                if (v >= N * nS)
                    return;  // uniform over the CTA
                const int pos = v / nS, k = v - pos * nS;  // k-th sampled sequence
                i = N - 1 - pos;
                const int w = __ffs(__ballot_sync(0xffffffffu, cum > k)) - 1;  // its word
                uint32_t m = __shfl_sync(0xffffffffu, word, w);
                for (int rem = k - (__shfl_sync(0xffffffffu, cum, w) - __popc(m)); rem > 0; --rem)
                    m &= m - 1;
                b = w * 32 + __ffs(m) - 1;
                is_draft = 1;
            }
        } else {
            const int v = u - B, pos = v / (2 * B), w = v - pos * (2 * B);
            i = N - 1 - pos;
            b = w >> 1;
            is_draft = w & 1;
        }
    }

    float T;
    const int mode = sequence_mode(p, b, T);
    const size_t trow = (size_t)b * (N + 1) + i;
    const size_t drow = TREE ? trow : (size_t)b * N + i;
    int d = 0;
    bool bad_d = false, bad_tree = false;
    if constexpr (TREE) {
        if (i > 0) {
            d = p.tokens[trow];
            bad_d = d < 0 || d >= V;
        }
        const int par = p.parent[trow];
        bad_tree = (i == 0) ? (par != -1) : (par < 0 || par >= i);
    } else {
        d = (i < N) ? p.tokens[(size_t)b * N + i] : 0;
        bad_d = (i < N) && (d < 0 || d >= V);
    }
    if (tid == 0) {
        ring_init(ctl.ring);
        const double cfd = (mode == MODE_SAMPLED) ? kLog2e / (double)T : 0.0;
        ctl.cfd = cfd;
        ctl.cf = (float)cfd;
        if (!TREE)
            ctl.has_child = 1;  // (a tree node's is set by the producer warp below)
    }
    if constexpr (TREE) {
        if (warp == kProducerWarp) {
            bool any = false;
            for (int c = i + 1 + lane; c <= N; c += 32)
                any |= p.parent[(size_t)b * (N + 1) + c] == i;
            any = __any_sync(0xffffffffu, any);
            __syncwarp();
            if (lane == 0)
                ctl.has_child = any ? 1 : 0;
        }
    }
    const bool decides = !TREE && mode == MODE_SAMPLED && i < N;  // a two-row position of the chain
    // The decision's inputs, loaded by an idle lane of the producer warp and
    // parked in shared memory after the stream.  In a packed (one-wave) grid
    // they are loaded while the row streams, so that no block starts its
    // stream late; in larger grids a block's late start is covered by the
    // others on its SM, and loading them before the stream measured 0.4 %
    // faster (headline kernel A 173.1 -> 172.4 us).
    const bool prefetcher = tid == 32 * kProducerWarp + 1;
    const bool prefetch = prefetcher && decides && !bad_d;
    float pre_zq = 0.0f, pre_zp = 0.0f, pre_u = 0.0f;
    if (prefetch && !PACKED) {
        pre_zq = logit_at<DT>(p.target, trow * (size_t)V + d);
        pre_zp = logit_at<DT>(p.draft, drow * (size_t)V + d);
        pre_u = p.u[trow];
    }
    __syncthreads();
    if (is_draft && (mode != MODE_SAMPLED || !ctl.has_child))
        return;  // no draft row is read (uniform over the CTA)
    if (prefetch && PACKED) {
        pre_zq = logit_at<DT>(p.target, trow * (size_t)V + d);
        pre_zp = logit_at<DT>(p.draft, drow * (size_t)V + d);
        pre_u = p.u[trow];
    }
    const float cf = ctl.cf;
    const int NV = V / VE;
    const uint4 *src = static_cast<const uint4 *>(is_draft ? p.draft : p.target) + (is_draft ? drow : trow) * (size_t)NV;
    const int nst = (NV + kStageVecs - 1) / kStageVecs;

    // ---- stream the row once
    Online2 o2{-INFINITY, 0ull};
    ArgMax ga{-INFINITY, INT_MAX, 0};
    if (mode != MODE_INVALID) {
        if (warp == kProducerWarp) {
            if (lane == 0) {
                for (int t = 0; t < nst; ++t) {
                    const uint32_t s = (uint32_t)t % kStages;
                    if (!sv::mbar_wait_bounded(&ctl.ring.empty[s], (((uint32_t)t / kStages) & 1u) ^ 1u, &ctl.ring.abort,
                                               kWaitLimitNs)) {
                        ctl.ring.abort = 1;
                        break;
                    }
                    const int nvec = min(kStageVecs, NV - t * kStageVecs);
                    const uint32_t bytes = static_cast<uint32_t>(nvec) * 16u;
                    sv::mbar_arrive_expect_tx(&ctl.ring.full[s], bytes);
                    sv::bulk_g2s(ring + s * (2 * kTileBytes), src + (size_t)t * kStageVecs, bytes, &ctl.ring.full[s]);
                    ctl.ring.last_g[s] = t;
                }
            }
            __syncwarp();
        } else {
            // Each thread takes its vectors of the stage into registers and the
            // stage is released before the arithmetic, so that the next copy
            // into it overlaps the arithmetic on this one (headline kernel A1
            // 175.1 -> 174.6 us with the unchecked loads of full stages).
            for (int t = 0; t < nst; ++t) {
                const bool ok = consume_wait(ctl.ring, t);
                const uint4 *stage = reinterpret_cast<const uint4 *>(ring + (t % kStages) * (2 * kTileBytes));
                uint4 v[2 * kVPT];
                if (ok && (t + 1) * kStageVecs <= NV) {  // a full stage
#pragma unroll
                    for (int k = 0; k < 2 * kVPT; ++k)
                        v[k] = stage[k * kSliceVecs + tid];
                } else {
#pragma unroll
                    for (int k = 0; k < 2 * kVPT; ++k) {
                        const int sv_ = k * kSliceVecs + tid;
                        v[k] = (ok && t * kStageVecs + sv_ < NV) ? stage[sv_] : neg_inf_vec<DT>();
                    }
                }
                consume_release(ctl.ring, t, lane);
                if (!ok) {
                    ctl.ring.abort = 1;
                } else if (mode == MODE_GREEDY) {
#pragma unroll
                    for (int k = 0; k < 2 * kVPT; ++k) {
                        const int vec = t * kStageVecs + k * kSliceVecs + tid;
                        if (vec < NV)
                            argmax_add2<DT>(ga, v[k], vec * VE);
                    }
                } else {
                    online_add_tile<DT, 2 * kVPT>(o2, v, cf);
                }
            }
        }
    }
    if (prefetcher) {
        ctl.zq_d = pre_zq;
        ctl.zp_d = pre_zp;
        ctl.u_i = pre_u;
    }

    // ---- the CTA's result
    Online o = online_fold<DT>(o2, cf);
    if (warp < kConsWarps) {
        if (mode == MODE_GREEDY) {
            ga = warp_argmax(ga);
            if (lane == 0) {
                ctl.red_m[warp] = ga.v;
                ctl.red_i[warp] = ga.i;
                ctl.red_n[warp] = ga.nan;
            }
        } else if (mode == MODE_SAMPLED) {
            o = warp_merge(o, cf);
            if (lane == 0) {
                ctl.red_m[warp] = o.m;
                ctl.red_s[warp] = o.s;
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        int errb = (bad_d ? kErrBadToken : 0) | (bad_tree ? kErrBadTree : 0);
        if (mode == MODE_GREEDY) {
            ArgMax a{ctl.red_m[0], ctl.red_i[0], ctl.red_n[0]};
            for (int w = 1; w < kConsWarps; ++w)
                a = argmax_merge(a, ArgMax{ctl.red_m[w], ctl.red_i[w], ctl.red_n[w]});
            if (a.nan || a.v == INFINITY || a.v == -INFINITY)
                errb |= kErrBadValue;
            p.ws_tok[trow] = a.i;
            if (!TREE && i < N && d != a.i)
                atomicMin(&p.ws_first[b], i);
            if (p.tstats) {
                p.tstats[trow * 2 + 0] = a.v;
                p.tstats[trow * 2 + 1] = NAN;
            }
            if (!TREE && i < N) {
                if (p.q_at)
                    p.q_at[drow] = NAN;
                if (p.p_at)
                    p.p_at[drow] = NAN;
                if (p.ratio_at)
                    p.ratio_at[drow] = NAN;
                if (p.dstats) {
                    p.dstats[drow * 2 + 0] = NAN;
                    p.dstats[drow * 2 + 1] = NAN;
                }
            }
        } else if (mode == MODE_SAMPLED) {
            Online a{ctl.red_m[0], ctl.red_s[0]};
            for (int w = 1; w < kConsWarps; ++w)
                a = online_merge(a, Online{ctl.red_m[w], ctl.red_s[w]}, cf);
            if (!(isfinite(a.m) && isfinite(a.s) && a.s > 0.0f))
                errb |= kErrBadValue;
            float *st = p.ws_stats + trow * 4 + (is_draft ? 2 : 0);
            st[0] = a.m;
            st[1] = a.s;
            if (!is_draft && p.tstats) {
                p.tstats[trow * 2 + 0] = a.m;
                p.tstats[trow * 2 + 1] = a.s;
            }
            if (is_draft && p.dstats) {
                p.dstats[drow * 2 + 0] = a.m;
                p.dstats[drow * 2 + 1] = a.s;
            }
            if (decides) {
                // The position's two rows meet in one 64-bit exchange: each
                // swaps its (m, S) into the position's cell, and the row that
                // finds the other's pair there is the second and decides.  The
                // pair travels in the atomic, so no fence and no reload.
                unsigned long long mine =
                    ((unsigned long long)__float_as_uint(a.s) << 32) | (unsigned long long)__float_as_uint(a.m);
                if (mine == 0ull)
                    mine = 0x7fffffff7fffffffull;  // (0, 0) is not a valid pair either; 0 marks an empty cell
                const unsigned long long other = atomicExch(&p.ws_xc[trow], mine);
                if (other != 0ull) {
                    p.ws_xc[trow] = 0ull;
                    const float om = __uint_as_float((unsigned)(other & 0xffffffffull));
                    const float os = __uint_as_float((unsigned)(other >> 32));
                    const float mq = is_draft ? om : a.m, Sq = is_draft ? os : a.s;
                    const float mp = is_draft ? a.m : om, Sp = is_draft ? a.s : os;
                    float *sq = p.ws_stats + trow * 4;  // both rows' statistics, for the residual pass
                    sq[0] = mq;
                    sq[1] = Sq;
                    sq[2] = mp;
                    sq[3] = Sp;
                    const bool valid = isfinite(mq) && isfinite(Sq) && Sq > 0.0f && isfinite(mp) && isfinite(Sp) &&
                                       Sp > 0.0f;
                    if (p.ratio_at)
                        p.ratio_at[drow] = NAN;
                    if (valid && !bad_d) {
                        const float zq = ctl.zq_d, zp = ctl.zp_d;
                        const double cfd = ctl.cfd;
                        const double ratio = decision_ratio(zq, zp, mq, Sq, mp, Sp, cfd);
                        if (!accept_by_ratio(ratio, (double)ctl.u_i))
                            atomicMin(&p.ws_first[b], i);
                        if (p.ratio_at)
                            p.ratio_at[drow] = (float)ratio;
                        if (p.q_at)
                            p.q_at[drow] = (float)(exp2(((double)zq - (double)mq) * cfd) / (double)Sq);
                        if (p.p_at)
                            p.p_at[drow] = (float)(exp2(((double)zp - (double)mp) * cfd) / (double)Sp);
                    }
                }
            }
        } else if (!is_draft) {
            errb |= kErrBadValue;
            if (!TREE && i < N && p.ratio_at)
                p.ratio_at[drow] = NAN;
        }
        if (ctl.ring.abort)
            errb |= kErrTimeout;
        if (errb)
            atomicOr(&p.ws_err[b], errb);
        if (ctl.ring.abort)
            ring_drain(ctl.ring);
    }
}

// =============================================================================
// Kernels B and C: the emitted token of each sequence
// =============================================================================
//
// j = first rejected position (N if none).  Sampled sequences draw the token
// at j from normalise(max(0, q_j - p_j)) (or the bonus token from q_N) by
// inverse CDF in ascending token order.
//
// Kernel B (sv_mass_kernel) sums the residual mass of every slice of 256
// 16-byte vectors of those row pairs.  Its grid is a fixed number of CTAs;
// each takes an equal contiguous share of all ring tiles of all sampled
// sequences and streams them through its TMA ring, so the work is balanced
// to one tile.  Thread t takes vector t of a slice; a slice's mass is the sum
// of its 8 warp totals (warp-inclusive scans), added in warp order.
//
// Kernel C (sv_pick_kernel), one CTA per sequence, finds the slice where the
// cumulative mass first exceeds u_N * R, recomputes that slice with the same
// rounded arithmetic (so its warp totals equal kernel B's), finds the warp,
// lane and element, writes out_tokens / num_accepted and returns the
// workspace slots to their idle state.

constexpr int kPickThreads = kSliceVecs;  // one vector of a slice per thread

// Ring of the mass kernel: kVPTM slices per tile, kStagesM stages.
constexpr int kVPTM = 2;
constexpr int kStagesM = 3;
constexpr int kTileVecsM = kVPTM * kSliceVecs;
constexpr int kTileBytesM = kTileVecsM * 16;
constexpr int kRingBytesM = kStagesM * 2 * kTileBytesM;

// Per-stage description of the tile the producer put there.
struct alignas(16) TileMeta {
    int b;         // sequence, or -1: no more tiles
    int slice;     // first slice of the tile within the sequence's row
    int res_mode;
    float mq, isq, mp, isp, cf;
};

struct CtlM {
    Ring<kStagesM> ring;
    TileMeta meta[kStagesM];
};

constexpr size_t kSmemM = kRingBytesM + sizeof(CtlM);

// Residual-mode parameters of a sampled sequence: j, the residual mode, and
// (mq, isq, mp, isp) as the raw statistics (m, S) of position j's rows until
// sample_shifts turns them into residual_vec's shifts and scales.
struct SeqSample {
    int j, res_mode;
    float mq, isq, mp, isp, cf, uN;
};

// The row statistics of position j as residual_vec's shifts and scales.
__device__ __forceinline__ void sample_shifts(SeqSample &s, float cf)
{
    s.cf = cf;
    residual_shift(s.mq, s.isq, cf, s.mq, s.isq);
    if (s.res_mode == RES_DIFF)
        residual_shift(s.mp, s.isp, cf, s.mp, s.isp);
}

// Sequence b's first rejection j, its residual mode and whether it is sampled
// (T in s.cf); the rows to read are known from here on.
__device__ __forceinline__ bool sequence_head(const SvParams &p, int b, SeqSample &s)
{
    float T;
    const int mode = sequence_mode(p, b, T);
    int j = __ldcg(&p.ws_first[b]);
    j = j > p.N ? p.N : j;
    const int err = __ldcg(&p.ws_err[b]);
    s.j = j;
    s.cf = T;
    s.res_mode = (j < p.N) ? RES_DIFF : RES_Q;
    return !err && mode == MODE_SAMPLED;
}

// The second half: position j's raw statistics (m, S) ...
__device__ __forceinline__ void sequence_stats(const SvParams &p, int b, SeqSample &s)
{
    const int j = s.j;
    const float *st = p.ws_stats + ((size_t)b * (p.N + 1) + j) * 4;
    s.mq = __ldcg(st + 0);
    s.isq = __ldcg(st + 1);
    s.mp = (j < p.N) ? __ldcg(st + 2) : 0.0f;
    s.isp = (j < p.N) ? __ldcg(st + 3) : 1.0f;
}

// ... and as residual_vec's shifts and scales (T in s.cf on entry).
__device__ __forceinline__ void sequence_tail(const SvParams &p, int b, SeqSample &s)
{
    sequence_stats(p, b, s);
    sample_shifts(s, (float)(kLog2e / (double)s.cf));
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 4) sv_mass_kernel(const SvParams p)
{
    constexpr int VE = Elt<DT>::kPerVec;
    constexpr int kStages = kStagesM;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    CtlM &ctl = *reinterpret_cast<CtlM *>(smem + kRingBytesM);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NV = p.V / VE;
    const int T = (NV + kTileVecsM - 1) / kTileVecsM;  // ring tiles per row
    const int S = (NV + kSliceVecs - 1) / kSliceVecs;  // slices per row
    const long long total = (long long)p.B * T;
    const long long t_begin = total * blockIdx.x / gridDim.x;
    const long long t_end = total * (blockIdx.x + 1) / gridDim.x;

    if (tid == 0)
        ring_init(ctl.ring);
    sv::grid_dependency_wait();  // kernel A's results
    __syncthreads();

    if (warp == kProducerWarp) {
        if (lane == 0) {
            uint32_t g = 0;
            int cur_b = -1;
            bool cur_ok = false, have_stats = false;
            SeqSample sq{};
            for (long long tt = t_begin; tt < t_end && !ctl.ring.abort; ++tt) {
                const int b = (int)(tt / T);
                const int t = (int)(tt - (long long)b * T);
                if (b != cur_b) {
                    cur_b = b;
                    cur_ok = sequence_head(p, b, sq);
                    have_stats = false;
                }
                if (!cur_ok)
                    continue;
                const uint32_t s = g % kStages;
                if (!sv::mbar_wait_bounded(&ctl.ring.empty[s], ((g / kStages) & 1u) ^ 1u, &ctl.ring.abort,
                                           kWaitLimitNs)) {
                    ctl.ring.abort = 1;
                    break;
                }
                // the copies first (the rows are known from j), then the
                // statistics they are summed with, loaded while the copies fly,
                // then the producer's arrival
                const uint4 *tsrc = static_cast<const uint4 *>(p.target) + sample_trow(p, b, sq.j) * (size_t)NV;
                const uint4 *dsrc = (sq.res_mode == RES_DIFF)
                                        ? static_cast<const uint4 *>(p.draft) + sample_drow(p, b, sq.j) * (size_t)NV
                                        : nullptr;
                const int nvec = min(kTileVecsM, NV - t * kTileVecsM);
                const uint32_t bytes = static_cast<uint32_t>(nvec) * 16u;
                sv::mbar_expect_tx(&ctl.ring.full[s], dsrc ? 2u * bytes : bytes);
                unsigned char *stage = ring + s * (2 * kTileBytesM);
                sv::bulk_g2s(stage, tsrc + (size_t)t * kTileVecsM, bytes, &ctl.ring.full[s]);
                if (dsrc)
                    sv::bulk_g2s(stage + kTileBytesM, dsrc + (size_t)t * kTileVecsM, bytes, &ctl.ring.full[s]);
                ctl.ring.last_g[s] = static_cast<int>(g);
                if (!have_stats) {
                    sequence_tail(p, b, sq);
                    have_stats = true;
                }
                TileMeta &m = ctl.meta[s];
                m.b = b;
                m.slice = t * kVPTM;
                m.res_mode = sq.res_mode;
                m.mq = sq.mq;
                m.isq = sq.isq;
                m.mp = sq.mp;
                m.isp = sq.isp;
                m.cf = sq.cf;
                sv::mbar_arrive(&ctl.ring.full[s]);
                ++g;
            }
            // end marker (no bytes): consumers stop at it
            const uint32_t s = g % kStages;
            if (!ctl.ring.abort &&
                sv::mbar_wait_bounded(&ctl.ring.empty[s], ((g / kStages) & 1u) ^ 1u, &ctl.ring.abort, kWaitLimitNs)) {
                ctl.meta[s].b = -1;
                sv::mbar_arrive_expect_tx(&ctl.ring.full[s], 0);
            } else {
                ctl.ring.abort = 1;
            }
        }
        __syncwarp();
    } else {
        for (uint32_t g = 0;; ++g) {
            const uint32_t s = g % kStages;
            if (!consume_wait(ctl.ring, g)) {
                ctl.ring.abort = 1;
                break;
            }
            const TileMeta m = ctl.meta[s];
            if (m.b < 0)
                break;
            const unsigned char *stage = ring + s * (2 * kTileBytesM);
#pragma unroll
            for (int k = 0; k < kVPTM; ++k) {
                const int sv_ = k * kSliceVecs + tid;
                const int vec = m.slice * kSliceVecs + sv_;
                float part = 0.0f;
                if (vec < NV) {
                    float r[VE];
                    const uint4 vd = (m.res_mode == RES_DIFF) ? reinterpret_cast<const uint4 *>(stage + kTileBytesM)[sv_]
                                                              : make_uint4(0, 0, 0, 0);
                    residual_vec<DT>(reinterpret_cast<const uint4 *>(stage)[sv_], vd, m.res_mode, m.mq, m.isq, m.mp,
                                     m.isp, m.cf, r);
#pragma unroll
                    for (int e = 0; e < VE; ++e)
                        part = __fadd_rn(part, r[e]);
                }
                const float tot = warp_total(part);  // = the inclusive scan's lane 31
                const int sl = m.slice + k;
                if (lane == 31 && sl < S)
                    p.ws_slice[((size_t)m.b * S + sl) * kConsWarps + warp] = tot;  // this warp's share
            }
            consume_release(ctl.ring, g, lane);
        }
    }
    if (tid == 0 && ctl.ring.abort) {
        atomicOr(p.status, kErrTimeout);
        ring_drain(ctl.ring);
    }
}

// Mass of one slice of the residual at thread granularity: thread t's share
// (vector t of the slice) and its warp-inclusive prefix; identical to the
// arithmetic of sv_mass_kernel.
template <int DT>
__device__ __forceinline__ float slice_thread_mass(const uint4 *tsrc, const uint4 *dsrc, int slice, int NV, int tid,
                                                   const SeqSample &s, float *r)
{
    constexpr int VE = Elt<DT>::kPerVec;
    const int vec = slice * kSliceVecs + tid;
    float part = 0.0f;
    if (vec < NV) {
        const uint4 vd = (s.res_mode == RES_DIFF) ? __ldcg(dsrc + vec) : make_uint4(0, 0, 0, 0);
        residual_vec<DT>(__ldcg(tsrc + vec), vd, s.res_mode, s.mq, s.isq, s.mp, s.isp, s.cf, r);
#pragma unroll
        for (int e = 0; e < VE; ++e)
            part = __fadd_rn(part, r[e]);
    } else {
#pragma unroll
        for (int e = 0; e < VE; ++e)
            r[e] = 0.0f;
    }
    return part;
}

constexpr int kMaxRowSlices = kMaxCluster * kMaxSlices;  // slices of the longest supported row

// ---- inverse CDF over slice masses (kernel C and the tree walk) ---------------
// Above the slice level the search runs in 64-bit fixed point: every float
// warp share x (a mass in [0, 1]) is the integer floor(x 2^62), exact for
// x >= 2^-38, so slice masses, their prefix sums and the total R are exact
// integer sums, and the target floor(u R) is one 64 x 64-bit high product.
// Where a token falls is then resolved to the float precision of one warp's
// share of one slice, not of the running total (in float the cumulative mass
// near R/2 resolves only about 3e-8 R, coarser than many tail tokens of a
// 150 000-token vocabulary), and with integer additions, not the narrow FP64
// pipe.
typedef unsigned long long fx_t;
constexpr fx_t kFxNone = ~0ull;  // no remainder: rounding fell back to the last slice with mass

__device__ __forceinline__ fx_t fx_of(float x)
{
    const uint32_t bits = __float_as_uint(x);
    int e = (int)((bits >> 23) & 0xffu);
    if ((bits >> 31) || e == 0)  // -0, or below 2^-126: nothing at this scale
        return 0ull;
    e = e > 127 ? 127 : e;       // masses stay below 2 (a share is at most R <= 1 plus rounding)
    const fx_t m = (fx_t)((bits & 0x7fffffu) | 0x800000u);
    const int sh = e - 88;       // x = m 2^(e - 150), so x 2^62 = m 2^(e - 88)
    return sh >= 0 ? (m << sh) : (sh > -24 ? (m >> -sh) : 0ull);
}

__device__ __forceinline__ float fx_to_float(fx_t v) { return __ull2float_rn(v) * 0x1p-62f; }

// floor(u R) for u in [0, 1): u as the exact integer u 2^64 (for u >= 2^-40),
// times R, high 64 bits of the product.
__device__ __forceinline__ fx_t fx_scale(float u, fx_t R)
{
    const uint32_t bits = __float_as_uint(u);
    const int e = (int)((bits >> 23) & 0xffu);
    if ((bits >> 31) || e == 0)
        return 0ull;
    const fx_t m = (fx_t)((bits & 0x7fffffu) | 0x800000u);
    const int sh = e - 86;  // u 2^64 = m 2^(e - 86); e <= 126 since u < 1
    const fx_t ux = sh >= 0 ? (m << (sh > 40 ? 40 : sh)) : (sh > -24 ? (m >> -sh) : 0ull);
    return __umul64hi(ux, R);
}

__device__ __forceinline__ fx_t warp_incl_scan_fx(fx_t x, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const fx_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    return x;
}

// Total of a slice: its eight warp shares, in fixed point.
__device__ __forceinline__ fx_t slice_total_fx(const float *w8)
{
    fx_t t = 0ull;
#pragma unroll
    for (int q = 0; q < kConsWarps; ++q)
        t += fx_of(w8[q]);
    return t;
}

// Warp 0: the total of S slice masses.
__device__ __forceinline__ fx_t warp_total_slices(const fx_t *slice, int S, int lane)
{
    fx_t carry = 0ull;
    for (int c0 = 0; c0 < S; c0 += 32) {
        const int c = c0 + lane;
        const fx_t m = (c < S) ? slice[c] : 0ull;
        carry = __shfl_sync(0xffffffffu, warp_incl_scan_fx(m, lane) + carry, 31);
    }
    return carry;
}

// Warp-wide: the first slice whose cumulative mass exceeds x, and x1 = x minus
// the mass before it.  x < R always (u < 1), so a slice is always found; the
// fallback (the last slice with mass, x1 = kFxNone) guards only an empty total.
__device__ __forceinline__ void warp_find_slice(const fx_t *slice, int S, fx_t x, int lane, int &cs, fx_t &x1)
{
    cs = -1;
    x1 = kFxNone;
    fx_t run = 0ull;
    for (int c0 = 0; c0 < S && cs < 0; c0 += 32) {
        const int c = c0 + lane;
        const fx_t m = (c < S) ? slice[c] : 0ull;
        const fx_t inc = warp_incl_scan_fx(m, lane) + run;
        const unsigned hit = __ballot_sync(0xffffffffu, c < S && x < inc);
        if (hit) {
            const int l = __ffs(hit) - 1;
            const fx_t prev = __shfl_sync(0xffffffffu, inc, l > 0 ? l - 1 : 0);
            cs = c0 + l;
            x1 = x - (l > 0 ? prev : run);
        }
        run = __shfl_sync(0xffffffffu, inc, 31);
    }
    if (cs < 0) {  // no mass at all: the last slice that has mass, else the last
        for (int c0 = ((S - 1) / 32) * 32; c0 >= 0 && cs < 0; c0 -= 32) {
            const int c = c0 + lane;
            const unsigned m = __ballot_sync(0xffffffffu, c < S && slice[c] > 0ull);
            if (m)
                cs = c0 + 31 - __clz(m);
        }
        if (cs < 0)
            cs = S - 1;
        x1 = kFxNone;
    }
}

// Element search inside slice ss, whose masses thread t holds for vector t
// (r[VE] and their sum `part`; threads past the 256 of a slice pass zeros):
// warp totals in warp order (a fixed-point running sum, as the slice total was
// formed), then the lane, then the element where the cumulative mass first
// exceeds x1; rounding falls back to the last element with mass.  Every thread
// of the block calls it (it synchronises the block).
struct PickState {
    float incl[kConsThreads];
    int sel, token;
    float xl;
};

template <int VE>
__device__ int pick_in_slice(PickState &ps, int ss, float part, const float *r, fx_t x1, int NV)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float incl = warp_incl_scan(part, lane);
    if (tid < kConsThreads)
        ps.incl[tid] = incl;
    __syncthreads();
    if (warp == 0) {
        int sel = -1;
        float xl = 0.0f;
        if (x1 != kFxNone) {
            const fx_t wt = (lane < kConsWarps) ? fx_of(ps.incl[lane * 32 + 31]) : 0ull;
            fx_t wc = 0ull, wprev = 0ull;
            int ws = -1;
            for (int w = 0; w < kConsWarps; ++w) {
                const fx_t next = wc + __shfl_sync(0xffffffffu, wt, w);
                if (ws < 0 && x1 < next) {
                    ws = w;
                    wprev = wc;
                }
                wc = next;
            }
            if (ws >= 0) {
                const float xw = fx_to_float(x1 - wprev);
                const float li = ps.incl[ws * 32 + lane];
                const unsigned ml = __ballot_sync(0xffffffffu, xw < li);
                if (ml) {
                    const int ls = __ffs(ml) - 1;
                    const float lprev = __shfl_sync(0xffffffffu, li, ls > 0 ? ls - 1 : 0);
                    sel = ws * 32 + ls;
                    xl = __fsub_rn(xw, ls > 0 ? lprev : 0.0f);
                }
            }
        }
        if (lane == 0) {
            ps.sel = sel;
            ps.xl = xl;
            ps.token = -1;
        }
    }
    __syncthreads();
    if (ps.sel >= 0 && tid == ps.sel) {
        float acc = 0.0f;
        for (int e = 0; e < VE; ++e) {
            acc = __fadd_rn(acc, r[e]);
            if (ps.xl < acc) {
                ps.token = (ss * kSliceVecs + tid) * VE + e;
                break;
            }
        }
    }
    __syncthreads();
    if (ps.token < 0) {
        if (tid == 0)
            ps.sel = -1;
        __syncthreads();
        if (tid < kConsThreads)
            for (int e = VE - 1; e >= 0; --e)
                if (r[e] > 0.0f) {
                    atomicMax(&ps.sel, (ss * kSliceVecs + tid) * VE + e);
                    break;
                }
        __syncthreads();
        if (tid == 0)
            ps.token = ps.sel >= 0 ? ps.sel : min(NV, (ss + 1) * kSliceVecs) * VE - 1;
        __syncthreads();
    }
    return ps.token;
}

struct PickShared {
    fx_t slice[kMaxRowSlices];  // the sequence's slice masses
    float wtot[kConsWarps];
    PickState ps;
    int sstar, retry;
    fx_t x1;
    float cf;                   // log2(e)/T
};

// Outputs of sequence b, written by every thread of the block in parallel:
// slot k < j the accepted draft, slot j `last`, the rest -1 (every slot -1
// for an invalid sequence).  my_tok is this thread's draft token
// (tokens[b][tid] for tid < N), loaded when the kernel started so that no
// load is left on the way out.  Then thread 0 writes num_accepted, counts the
// telemetry and returns the sequence's slots to idle (after the barrier: every
// thread has read them).
__device__ void emit_outputs(const SvParams &p, int b, int j, int last, bool invalid, int my_tok)
{
    const int N = p.N, tid = threadIdx.x;
    int32_t *out = p.out + (size_t)b * (N + 1);
    for (int k = tid; k <= N; k += blockDim.x) {
        int v = -1;
        if (!invalid) {
            if (k < j)
                v = (k == tid) ? my_tok : p.tokens[(size_t)b * N + k];
            else if (k == j)
                v = last;
        }
        out[k] = v;
    }
    __syncthreads();
    if (tid == 0) {
        if (invalid) {
            p.nacc[b] = -1;
            atomicOr(p.status, __ldcg(&p.ws_err[b]));
            if (p.hist)
                atomicAdd(p.hist_invalid, 1ull);
        } else {
            p.nacc[b] = j;
            if (p.hist)
                atomicAdd(&p.hist[j], 1ull);
        }
        p.ws_first[b] = kNoReject;
        p.ws_err[b] = 0;
    }
}

// A sequence that is not sampled: invalid (its error bits go to the status
// word) or greedy (the argmax at j).  Every thread of the block.
__device__ void emit_unsampled(const SvParams &p, int b, int j, int my_tok)
{
    const bool invalid = __ldcg(&p.ws_err[b]) != 0;
    const int last = invalid ? -1 : __ldcg(&p.ws_tok[(size_t)b * (p.N + 1) + j]);
    emit_outputs(p, b, j, last, invalid, my_tok);
}

// The token of a sampled sequence, from the slice masses of its residual in
// sh.slice: the slice where the cumulative mass first exceeds u_N * R, then
// (recomputing that slice with the masses' arithmetic) the warp, lane and
// element.  A residual without mass (q_j == p_j) is replaced by q_j, whose
// slice masses are recomputed here.  Every thread of the block calls it;
// threads past the first 256 only take part in the barriers.
template <int DT>
__device__ int draw_token(PickShared &sh, SeqSample &sq, const uint4 *tsrc, const uint4 *dsrc, int NV, int S)
{
    constexpr int VE = Elt<DT>::kPerVec;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool cons = tid < kConsThreads;
    float r[VE];
    bool shifted = false;  // sq holds the raw statistics until the first residual needs them
    for (int attempt = 0; attempt < 2; ++attempt) {
        if (attempt == 1) {
            sample_shifts(sq, sh.cf);
            shifted = true;
            sq.res_mode = RES_Q;
            for (int sl = 0; sl < S; ++sl) {
                const float part = cons ? slice_thread_mass<DT>(tsrc, nullptr, sl, NV, tid, sq, r) : 0.0f;
                const float incl = warp_incl_scan(part, lane);
                if (lane == 31 && cons)
                    sh.wtot[warp] = incl;
                __syncthreads();
                if (tid == 0)
                    sh.slice[sl] = slice_total_fx(sh.wtot);
                __syncthreads();
            }
        }
        if (warp == 0) {
            const fx_t Rt = warp_total_slices(sh.slice, S, lane);
            int cs;
            fx_t x1;
            warp_find_slice(sh.slice, S, fx_scale(sq.uN, Rt), lane, cs, x1);
            if (lane == 0) {
                sh.retry = (Rt == 0ull && sq.res_mode == RES_DIFF) ? 1 : 0;
                sh.sstar = cs;
                sh.x1 = x1;
            }
        }
        __syncthreads();
        if (!sh.retry)
            break;
        __syncthreads();
    }
    const int ss = sh.sstar;
    // the chosen slice's vectors are loaded before the statistics are first used
    const int vec = ss * kSliceVecs + tid;
    const bool in = cons && vec < NV;
    uint4 vt = make_uint4(0, 0, 0, 0), vd = make_uint4(0, 0, 0, 0);
    if (in) {
        vt = __ldcg(tsrc + vec);
        if (sq.res_mode == RES_DIFF)
            vd = __ldcg(dsrc + vec);
    }
    if (!shifted)
        sample_shifts(sq, sh.cf);
    float part = 0.0f;
    if (in) {
        residual_vec<DT>(vt, vd, sq.res_mode, sq.mq, sq.isq, sq.mp, sq.isp, sq.cf, r);
#pragma unroll
        for (int e = 0; e < VE; ++e)
            part = __fadd_rn(part, r[e]);
    } else {
#pragma unroll
        for (int e = 0; e < VE; ++e)
            r[e] = 0.0f;
    }
    return pick_in_slice<VE>(sh.ps, ss, part, r, sh.x1, NV);
}

// Slice sl's mass: its 8 warp shares (left by kernel B), in fixed point.
__device__ __forceinline__ fx_t slice_share_total(const float *shares, int sl)
{
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(shares + (size_t)sl * kConsWarps));
    const float4 c = __ldcg(reinterpret_cast<const float4 *>(shares + (size_t)sl * kConsWarps + 4));
    const float w8[kConsWarps] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
    return slice_total_fx(w8);
}

template <int DT>
__global__ void __launch_bounds__(kPickThreads) sv_pick_kernel(const SvParams p)
{
    constexpr int VE = Elt<DT>::kPerVec;
    __shared__ PickShared sh;
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    const int N = p.N;
    const int NV = p.V / VE;
    const int S = (NV + kSliceVecs - 1) / kSliceVecs;

    sv::grid_dependency_wait();  // kernel B's slice masses
    const int my_tok = (tid < N) ? p.tokens[(size_t)b * N + tid] : -1;  // for the outputs
    // slice tid's mass, loaded alongside the sequence's statistics (used only if it is sampled)
    const float *shares = p.ws_slice + (size_t)b * S * kConsWarps;
    const fx_t my_mass = (tid < S) ? slice_share_total(shares, tid) : 0ull;
    SeqSample sq{};
    // u is read only where it is required ([B, N+1] unless the whole call is greedy)
    sq.uN = (!p.greedy && p.u) ? p.u[(size_t)b * (N + 1) + N] : 0.0f;
    const bool sampled = sequence_head(p, b, sq);  // sq.cf holds T
    if (tid == 0)
        sh.cf = sampled ? (float)(kLog2e / (double)sq.cf) : 0.0f;  // log2(e)/T, once
    if (sampled)
        sequence_stats(p, b, sq);  // in flight until the chosen slice's vectors are loaded (draw_token)
    __syncthreads();
    const int j = sq.j;
    if (!sampled) {
        emit_unsampled(p, b, j, my_tok);
        return;
    }

    const uint4 *tsrc = static_cast<const uint4 *>(p.target) + sample_trow(p, b, j) * (size_t)NV;
    const uint4 *dsrc = (j < N) ? static_cast<const uint4 *>(p.draft) + sample_drow(p, b, j) * (size_t)NV : nullptr;
    if (tid < S)
        sh.slice[tid] = my_mass;
    for (int sl = tid + kPickThreads; sl < S; sl += kPickThreads)
        sh.slice[sl] = slice_share_total(shares, sl);
    __syncthreads();
    const int token = draw_token<DT>(sh, sq, tsrc, dsrc, NV, S);
    emit_outputs(p, b, j, token, false, my_tok);
}

// =============================================================================
// Tree verification: the walk (kernel W), one CTA per sequence
// =============================================================================
//
// Kernel A (TREE) has left, per node, the row statistics (mq, Sq, mp, Sp), or
// the argmax for greedy sequences, and the error bits.  The walk starts at the
// root; at node n it tries n's children in index order.  With r_0 = q_n and
// r_{k+1} = (r_k - p_n)+ / R_{k+1}, R_{k+1} = sum (r_k - p_n)+, child c (the
// (k+1)-th tried) passes iff p_n(x) == 0 or u_c < min(1, r_k(x) / p_n(x)),
// x = its token.  A pass moves the walk to c; a rejection costs one pass over
// the row pair of n through the TMA ring, which yields the slice masses of
// (r_k - p_n)+ and so R_{k+1} (when it is 0, r_k stays).  When no child
// passes, the token is drawn from r_k by inverse CDF at u[0]: the slice masses
// of the last rejection pass are r_k's up to the factor R_k, otherwise one
// more pass computes them.  The element arithmetic is explicitly rounded and
// identical in every pass and in the recomputation of the chosen slice.
// A pass is bound by the arithmetic of one SM (two exp2 per element pair plus
// the residual chain), so the CTA has several groups of 8 consumer warps; the
// group that consumes a tile maps thread t to vector t of each slice, exactly
// as the recomputation does.

constexpr int kWalkGroups = 3;              // consumer groups of 8 warps; group g takes pass tiles g, g+3, ...
constexpr int kStagesG = 3;                 // ring stages of one consumer group
constexpr int kStagesW = kWalkGroups * kStagesG;  // 144 KiB of row pairs in flight
constexpr int kWalkThreads = kWalkGroups * kConsThreads + 32;  // + the producer warp
constexpr int kWalkProducerWarp = kWalkGroups * kConsWarps;
static_assert(kWalkThreads <= 1024, "a CTA holds at most 1024 threads");
constexpr int kMaxTreeNodes = 1024;         // nodes per tree (root included)
constexpr int kMaxWalkSlices = 512;         // slices of one row: V*elt <= 2 MiB
constexpr int kMaxWalkCluster = 4;          // CTAs (SMs) that share one tree's passes

// Each consumer group owns kStagesG stages of the ring (group g: stages
// g*kStagesG .. g*kStagesG + kStagesG - 1), which it alone consumes and the
// producer alone fills, in the order of the group's own tiles.  So every wait
// of a group is on the next phase of a stage whose previous phase that group
// consumed itself: an mbarrier parity wait cannot be satisfied by a phase two
// steps back.  (With one ring shared by groups that each take every third
// position, a group would wait on stages whose previous phase belonged to
// another group and might not have completed yet; the parity of that wait
// would then match the phase before it, and the wait would return early.)
struct CtlW {
    Ring<kStagesW> ring;
    float shares[kMaxWalkSlices * kConsWarps];  // warp shares of every slice of the current pass
    fx_t slice[kMaxWalkSlices];                 // slice masses (fixed-point sums of their shares): this
                                                // CTA's slices after a pass, every slice in the pick
    fx_t rsum[3];                               // a pass's total, added up by every CTA of the
                                                // cluster into each CTA's copy; slot = pass % 3
    PickState ps;
    int kids[kMaxTreeNodes];
    int nkids, accept, sstar;
    fx_t x1;                                    // the pick's remainder
    float cf;
    double cfd;                                 // log2(e) / T in double
    // the tree, fetched once: every decision of the walk reads shared memory
    int par[kMaxTreeNodes], tok[kMaxTreeNodes];
    int amax[kMaxTreeNodes];                    // greedy: the argmax of each node's verifier row
    float u[kMaxTreeNodes];
    float zq[kMaxTreeNodes], zp[kMaxTreeNodes];  // logits at node c's token in its parent's rows
    float st[kMaxTreeNodes * 4];                // (mq, Sq, mp, Sp) of each node
    unsigned char acc0[kMaxTreeNodes];          // node c's test against q of its parent (no rejection yet)
    float ratio0[kMaxTreeNodes];                // that test's ratio (kept for the debug output only)
    int err;                                    // the sequence's error bits, read once
};

constexpr size_t kSmemW = ring_bytes(kStagesW) + sizeof(CtlW);
static_assert(kSmemW <= 232448, "227 KiB of shared memory per CTA");

// (q - c p)+ (use_p) or q for the VE elements of one 16-byte vector, with
// q = 2^(zq cf - Kq) * Iq and p = 2^(zp cf - Kp) * Ip in residual_vec's form
// (shifts and scales from residual_shift), and q - c p = fma(2^(..), Iq,
// 2^(..) * (-c Ip)) in one rounding: at c = 1, -c Ip = -Ip exactly and this is
// kernel B's q - p bit for bit, so a chain-shaped tree samples as the chain
// does.  Pairs of adjacent elements travel as one f32x2; every operation
// rounds to nearest, so the walk's passes and the recomputation of the chosen
// slice agree bit for bit.
template <int DT>
__device__ __forceinline__ void tree_vec(const uint4 vt, const uint4 vd, bool use_p, float Kq, float Iq_, float Kp,
                                         float Ip_, float c, float cf, float *r)
{
    constexpr int NE = Elt<DT>::kPerVec;
    constexpr int NP = NE / 2;
    const uint32_t wt[4] = {vt.x, vt.y, vt.z, vt.w};
    const uint32_t wd[4] = {vd.x, vd.y, vd.z, vd.w};
    const unsigned long long Cf = sv::pack2(cf, cf);
    const unsigned long long NKq = sv::pack2(-Kq, -Kq), Iq = sv::pack2(Iq_, Iq_);
    const float ncp = -__fmul_rn(c, Ip_);  // -c / Sp' (exactly -Ip_ at c = 1)
    const unsigned long long NKp = sv::pack2(-Kp, -Kp), NcIp = sv::pack2(ncp, ncp);
#pragma unroll
    for (int e = 0; e < NP; ++e) {
        unsigned long long zt, zd;
        if constexpr (DT == SV_BF16) {
            zt = sv::pack2(__uint_as_float(wt[e] << 16), __uint_as_float(wt[e] & 0xffff0000u));
            zd = sv::pack2(__uint_as_float(wd[e] << 16), __uint_as_float(wd[e] & 0xffff0000u));
        } else {
            zt = sv::pack2(__uint_as_float(wt[2 * e]), __uint_as_float(wt[2 * e + 1]));
            zd = sv::pack2(__uint_as_float(wd[2 * e]), __uint_as_float(wd[2 * e + 1]));
        }
        float a0, a1;
        sv::unpack2(sv::fma2(zt, Cf, NKq), a0, a1);
        const unsigned long long eq = sv::pack2(sv::ex2(a0), sv::ex2(a1));
        if (use_p) {
            sv::unpack2(sv::fma2(zd, Cf, NKp), a0, a1);
            const unsigned long long ncp_k = sv::mul2(sv::pack2(sv::ex2(a0), sv::ex2(a1)), NcIp);  // -c p
            float d0, d1;
            sv::unpack2(sv::fma2(eq, Iq, ncp_k), d0, d1);
            r[2 * e] = fmaxf(d0, 0.0f);
            r[2 * e + 1] = fmaxf(d1, 0.0f);
        } else {
            sv::unpack2(sv::mul2(eq, Iq), r[2 * e], r[2 * e + 1]);
        }
    }
}

// Ring tile of the i-th tile this CTA streams in a pass: a cluster of C CTAs
// splits the row pair's tiles in blocks of kWalkGroups (one per consumer group).
__device__ __forceinline__ int walk_tile(int i, uint32_t rank, uint32_t C)
{
    return (int)(((uint32_t)(i / kWalkGroups) * C + rank) * kWalkGroups) + i % kWalkGroups;
}

// gcount[grp] without indexing a register array by a run-time value.
__device__ __forceinline__ uint32_t group_count(const uint32_t (&gcount)[kWalkGroups], int grp)
{
    static_assert(kWalkGroups == 3, "one select per group");
    return grp == 0 ? gcount[0] : (grp == 1 ? gcount[1] : gcount[2]);
}

// The CTA of the cluster that streams slice sl (in tile sl / kVPT).
__device__ __forceinline__ uint32_t walk_slice_owner(int sl, uint32_t C)
{
    return (uint32_t)((sl / kVPT) / kWalkGroups) % C;
}

// One pass over the row pair of a node: the slice masses of (q - c p)+
// (use_p) or q; returns their total.  Every thread of every CTA of the
// cluster calls it.  Each CTA streams its share of the tiles, writes the warp
// shares of those slices into its own shared memory, totals its own slices
// into w.slice (fixed point) and their sum into w.rpart; after a cluster
// barrier every CTA adds up the C partials, so all of them return the same
// total (the pick gathers the peers' slices once, at the end).
// Ring stage and phase parity of the k-th tile (counted over every pass) of
// consumer group grp.
__device__ __forceinline__ uint32_t walk_stage(int grp, uint32_t k) { return (uint32_t)grp * kStagesG + k % kStagesG; }
__device__ __forceinline__ uint32_t walk_parity(uint32_t k) { return (k / kStagesG) & 1u; }

template <int DT>
__device__ fx_t walk_mass_pass(CtlW &w, unsigned char *ring, const uint4 *tsrc, const uint4 *dsrc, int NV,
                               float Kq, float Iq, float Kp, float Ip, float c, float cf,
                               uint32_t (&gcount)[kWalkGroups], int &npass)
{
    constexpr int VE = Elt<DT>::kPerVec;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t C = sv::cluster_nctarank(), rank = sv::cluster_ctarank();
    const int NT = (NV + kTileVecs - 1) / kTileVecs;
    const int S = (NV + kSliceVecs - 1) / kSliceVecs;
    int n_own = 0;  // tiles this CTA streams: a prefix i = 0 .. n_own-1 of its sequence
    while (walk_tile(n_own, rank, C) < NT)
        ++n_own;
    // The pass's total goes to slot npass % 3 of every CTA's rsum; the slot
    // of the pass after next, read two barriers ago, is cleared here for it.
    const int slot = npass % 3;
    if (tid == 0)
        w.rsum[(npass + 1) % 3] = 0ull;
    // pass tile i belongs to group i % kWalkGroups, as that group's tile
    // gcount[grp] + i / kWalkGroups; lane grp of the producer warp fills that
    // group's stages, so a slower group never holds up the others' copies
    if (warp == kWalkProducerWarp) {
        if (lane < kWalkGroups) {
            const int grp = lane;
            for (int i = grp; i < n_own; i += kWalkGroups) {
                const uint32_t k = group_count(gcount, grp) + (uint32_t)(i / kWalkGroups);
                const uint32_t st = walk_stage(grp, k);
                if (!sv::mbar_wait_bounded(&w.ring.empty[st], walk_parity(k) ^ 1u, &w.ring.abort, kWaitLimitNs)) {
                    w.ring.abort = 1;
                    break;
                }
                const int t = walk_tile(i, rank, C);
                const int nvec = min(kTileVecs, NV - t * kTileVecs);
                const uint32_t bytes = static_cast<uint32_t>(nvec) * 16u;
                sv::mbar_arrive_expect_tx(&w.ring.full[st], dsrc ? 2u * bytes : bytes);
                unsigned char *stage = ring + st * (2 * kTileBytes);
                sv::bulk_g2s(stage, tsrc + (size_t)t * kTileVecs, bytes, &w.ring.full[st]);
                if (dsrc)
                    sv::bulk_g2s(stage + kTileBytes, dsrc + (size_t)t * kTileVecs, bytes, &w.ring.full[st]);
                w.ring.last_g[st] = static_cast<int>(k);
            }
        }
        __syncwarp();
    } else {
        const int grp = warp / kConsWarps, lt = tid - grp * kConsThreads, lw = warp - grp * kConsWarps;
        const uint32_t gbase = group_count(gcount, grp);
        for (int i = grp; i < n_own; i += kWalkGroups) {
            const uint32_t k = gbase + (uint32_t)(i / kWalkGroups);
            const uint32_t st = walk_stage(grp, k);
            const int t = walk_tile(i, rank, C);
            if (sv::mbar_wait_bounded(&w.ring.full[st], walk_parity(k), &w.ring.abort, kWaitLimitNs)) {
                const unsigned char *stage = ring + st * (2 * kTileBytes);
#pragma unroll
                for (int q = 0; q < kVPT; ++q) {
                    const int sv_ = q * kSliceVecs + lt;
                    const int vec = t * kTileVecs + sv_;
                    float part = 0.0f;
                    if (vec < NV) {
                        float r[VE];
                        const uint4 vd = dsrc ? reinterpret_cast<const uint4 *>(stage + kTileBytes)[sv_]
                                              : make_uint4(0, 0, 0, 0);
                        tree_vec<DT>(reinterpret_cast<const uint4 *>(stage)[sv_], vd, dsrc != nullptr, Kq, Iq, Kp,
                                     Ip, c, cf, r);
#pragma unroll
                        for (int e = 0; e < VE; ++e)
                            part = __fadd_rn(part, r[e]);
                    }
                    const float tot = warp_total(part);  // = the inclusive scan's lane 31
                    const int sl = t * kVPT + q;
                    if (lane == 31 && sl < S)
                        w.shares[sl * kConsWarps + lw] = tot;
                }
            } else {
                w.ring.abort = 1;
            }
            __syncwarp();
            if (lane == 0)
                sv::mbar_arrive(&w.ring.empty[st]);
        }
        // The warp's shares of this pass in fixed point, one per lane (the
        // j-th share the warp wrote: tile j / kVPT of its group, slot j %
        // kVPT).  Fixed-point sums are exact: whatever the order of these
        // additions, every CTA ends with the same total, the sum of all
        // slice masses.
        __syncwarp();
        fx_t acc = 0ull;
        for (int j = lane; j < ((n_own - grp + kWalkGroups - 1) / kWalkGroups) * kVPT; j += 32) {
            const int sl = walk_tile(grp + (j / kVPT) * kWalkGroups, rank, C) * kVPT + j % kVPT;
            if (sl < S)
                acc += fx_of(w.shares[sl * kConsWarps + lw]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0 && acc != 0ull) {
            if (C > 1)
                for (uint32_t r = 0; r < C; ++r)
                    sv::red_add_dsmem_u64(sv::dsmem_addr(&w.rsum[slot], r), acc);
            else
                atomicAdd(&w.rsum[slot], acc);
        }
    }
    for (int grp = 0; grp < kWalkGroups; ++grp)  // every thread keeps the counts
        gcount[grp] += (n_own > grp) ? (uint32_t)((n_own - grp + kWalkGroups - 1) / kWalkGroups) : 0u;
    if (C > 1)
        sv::cluster_sync();  // the additions into every CTA's slot are complete and visible
    else
        __syncthreads();
    ++npass;
    return w.rsum[slot];
}

// Inverse CDF over the slice masses in w.slice (total w.Rt) at u: the slice,
// then (recomputing that slice with the pass's arithmetic: (q - c p)+ when
// dsrc is given, else q) the warp, lane and element.  Every thread calls it;
// returns the token.
template <int DT>
__device__ int walk_pick(CtlW &w, const uint4 *tsrc, const uint4 *dsrc, int NV, float Kq, float Iq, float Kp,
                         float Ip, float c, float cf, float u, fx_t Rt)
{
    constexpr int VE = Elt<DT>::kPerVec;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t C = sv::cluster_nctarank(), rank = sv::cluster_ctarank();
    const int S = (NV + kSliceVecs - 1) / kSliceVecs;
    // The slice masses of the last pass: each CTA totals its own slices from
    // its warp shares, then reads the peers' (after the barrier that makes
    // them visible; after the second no CTA reads another's memory).
    for (int sl = tid; sl < S; sl += kWalkThreads)
        if (walk_slice_owner(sl, C) == rank)
            w.slice[sl] = slice_total_fx(&w.shares[sl * kConsWarps]);
    if (C > 1) {
        sv::cluster_sync();
        for (int sl = tid; sl < S; sl += kWalkThreads) {
            const uint32_t owner = walk_slice_owner(sl, C);
            if (owner != rank)
                w.slice[sl] = sv::ld_dsmem_u64(sv::dsmem_addr(&w.slice[sl], owner));
        }
        sv::cluster_sync();
    } else {
        __syncthreads();
    }
    if (warp == 0) {
        int cs;
        fx_t x1;
        warp_find_slice(w.slice, S, fx_scale(u, Rt), lane, cs, x1);
        if (lane == 0) {
            w.sstar = cs;
            w.x1 = x1;
        }
    }
    __syncthreads();
    const int ss = w.sstar;
    float r[VE];
#pragma unroll
    for (int e = 0; e < VE; ++e)
        r[e] = 0.0f;
    float part = 0.0f;
    const int vec = ss * kSliceVecs + tid;
    if (tid < kConsThreads && vec < NV) {
        const uint4 vd = dsrc ? __ldcg(dsrc + vec) : make_uint4(0, 0, 0, 0);
        tree_vec<DT>(__ldcg(tsrc + vec), vd, dsrc != nullptr, Kq, Iq, Kp, Ip, c, cf, r);
#pragma unroll
        for (int e = 0; e < VE; ++e)
            part = __fadd_rn(part, r[e]);
    }
    return pick_in_slice<VE>(w.ps, ss, part, r, w.x1, NV);
}

template <int DT>
__global__ void __launch_bounds__(kWalkThreads, 1) sv_tree_walk_kernel(const SvParams p)
{
    constexpr int VE = Elt<DT>::kPerVec;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    CtlW &w = *reinterpret_cast<CtlW *>(smem + ring_bytes(kStagesW));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t C = sv::cluster_nctarank(), rank = sv::cluster_ctarank();
    const int b = blockIdx.x / (int)C, M = p.N, V = p.V, NV = V / VE;
    const bool leader = rank == 0;  // every CTA of the cluster walks the tree; the leader writes
    const size_t row0 = (size_t)b * (M + 1);
    const int32_t *par = p.parent + row0;
    const int32_t *tok = p.tokens + row0;
    int32_t *out = p.out + row0;
    int32_t *path = p.path + row0;

    float T;
    const int mode = sequence_mode(p, b, T);
    if (tid == 0) {
        ring_init(w.ring);
        for (int k = 0; k < 3; ++k)
            w.rsum[k] = 0ull;
        w.cfd = (mode == MODE_SAMPLED) ? kLog2e / (double)T : 0.0;
        w.cf = (float)w.cfd;
    }
    // The tree's inputs (kernel A does not write them, so before the wait):
    // topology, tokens, uniforms and, for sampled trees, the two logits each
    // child's test reads in its parent's rows (checked indices: a bad tree or
    // token is caught by kernel A and ends the walk below).
    for (int c = tid; c <= M; c += kWalkThreads) {
        const int pc = par[c], x = tok[c];
        w.par[c] = pc;
        w.tok[c] = x;
        w.u[c] = p.greedy ? 0.0f : p.u[row0 + c];
        float zq = NAN, zp = NAN;
        if (mode == MODE_SAMPLED && c >= 1 && pc >= 0 && pc < c && x >= 0 && x < V) {
            zq = logit_at<DT>(p.target, (row0 + pc) * (size_t)V + x);
            zp = logit_at<DT>(p.draft, (row0 + pc) * (size_t)V + x);
        }
        w.zq[c] = zq;
        w.zp[c] = zp;
        if (p.ratio_at && leader)
            p.ratio_at[row0 + c] = NAN;  // nodes the walk does not test
    }
    sv::grid_dependency_wait();  // kernel A's statistics
    for (int i = tid; i < (M + 1) * 4; i += kWalkThreads)
        w.st[i] = __ldcg(p.ws_stats + row0 * 4 + i);
    if (mode == MODE_GREEDY)
        for (int c = tid; c <= M; c += kWalkThreads)
            w.amax[c] = __ldcg(&p.ws_tok[row0 + c]);
    if (tid == 0)
        w.err = __ldcg(&p.ws_err[b]);
    __syncthreads();
    // Every child's test before any rejection at its parent (r_0 = q), in
    // parallel and off the walk's serial path.
    if (mode == MODE_SAMPLED) {
        for (int c = 1 + tid; c <= M; c += kWalkThreads) {
            const int pc = w.par[c];
            bool a = false;
            double ratio = 0.0;
            if (pc >= 0 && pc < c) {
                const float *s = w.st + pc * 4;
                ratio = decision_ratio(w.zq[c], w.zp[c], s[0], s[1], s[2], s[3], w.cfd);
                a = accept_by_ratio(ratio, (double)w.u[c]);
            }
            w.acc0[c] = a ? 1 : 0;
            w.ratio0[c] = (float)ratio;
        }
        __syncthreads();
    }
    const int err = w.err;
    // The leader resets the error word for the next call: every CTA of the
    // cluster has read it first, so all of them take the same branch below (a
    // CTA that missed the error would wait for the exited leader at a pass's
    // cluster barrier).
    if (C > 1)
        sv::cluster_sync();
    if (err || mode == MODE_INVALID) {
        if (tid == 0 && leader) {
            for (int q = 0; q <= M; ++q) {
                out[q] = -1;
                path[q] = -1;
            }
            p.nacc[b] = -1;
            atomicOr(p.status, err ? err : kErrBadValue);
            if (p.hist)
                atomicAdd(p.hist_invalid, 1ull);
            p.ws_err[b] = 0;
        }
        return;
    }
    int depth = 0;
    if (mode == MODE_GREEDY) {
        if (!leader)
            return;
        if (tid == 0) {
            int n = 0;
            for (;;) {
                const int an = w.amax[n];
                int next = -1;
                for (int c = n + 1; c <= M && next < 0; ++c)
                    if (w.par[c] == n && w.tok[c] == an)
                        next = c;
                if (next < 0) {
                    out[depth] = an;
                    break;
                }
                out[depth] = w.tok[next];
                path[depth] = next;
                ++depth;
                n = next;
            }
        }
    } else {
        const float cf = w.cf;
        const float u0 = w.u[0];
        int n = 0, npass = 0;                      // node; passes so far
        uint32_t gcount[kWalkGroups] = {0u, 0u, 0u};  // tiles each consumer group has consumed
        for (;;) {
            const float *st = w.st + n * 4;
            const float mq = st[0], Sq = st[1], mp = st[2], Sp = st[3];
            const float isq = 1.0f / Sq;
            float Kq, Iq, Kp = 0.0f, Ip = 0.0f;  // the passes' shifts and scales (residual_shift)
            residual_shift(mq, Sq, cf, Kq, Iq);
            const uint4 *tsrc = static_cast<const uint4 *>(p.target) + (row0 + n) * (size_t)NV;
            const uint4 *dsrc = static_cast<const uint4 *>(p.draft) + (row0 + n) * (size_t)NV;
            // children of n, in index order
            if (warp == 0) {
                int cnt = 0;
                for (int c0 = n + 1; c0 <= M; c0 += 32) {
                    const int c = c0 + lane;
                    const bool is = c <= M && w.par[c] == n;
                    const unsigned m = __ballot_sync(0xffffffffu, is);
                    if (is)
                        w.kids[cnt + __popc(m & ((1u << lane) - 1u))] = c;
                    cnt += __popc(m);
                }
                if (lane == 0)
                    w.nkids = cnt;
            }
            __syncthreads();
            const int nk = w.nkids;
            const float isp = nk ? 1.0f / Sp : 0.0f;
            if (nk)
                residual_shift(mp, Sp, cf, Kp, Ip);
            // After k rejections with a non-empty residual, r_k = (q - c p)+ / Z:
            // r_0 = q (c = 0, Z = 1), and (r_k - p)+ = (q - (c + Z) p)+ / Z, so a
            // rejection moves c to c + Z and Z to the new pass's total (both
            // unchanged when that total is 0: r_k stays).
            float c = 0.0f, Z = 1.0f;
            int accepted = -1;
            bool masses_ready = false;  // w.slice holds the masses of (q - c p)+, Rlast their total
            fx_t Rlast = 0ull;
            for (int ci = 0; ci < nk; ++ci) {
                const int ch = w.kids[ci];
                if (tid == 0) {
                    const float zq = w.zq[ch], zp = w.zp[ch];  // at ch's token in n's rows
                    const double uc = (double)w.u[ch];
                    bool acc;
                    double ratio;  // for the debug output only
                    if (c == 0.0f) {
                        acc = w.acc0[ch] != 0;
                        ratio = w.ratio0[ch];
                    } else {
                        const float qx = __fmul_rn(sv::ex2(__fmul_rn(__fsub_rn(zq, mq), cf)), isq);
                        const float px = __fmul_rn(sv::ex2(__fmul_rn(__fsub_rn(zp, mp), cf)), isp);
                        const float rk = __fdiv_rn(fmaxf(__fmaf_rn(px, -c, qx), 0.0f), Z);
                        // u < min(1, rk/px) with px > 0, compared exactly: u px < rk
                        acc = (zp == -INFINITY) || (px == 0.0f) || (uc < 1.0 && uc * (double)px < (double)rk);
                        ratio = (zp == -INFINITY || px == 0.0f) ? (double)INFINITY : (double)rk / (double)px;
                    }
                    w.accept = acc ? 1 : 0;
                    if (p.ratio_at && leader)
                        p.ratio_at[row0 + ch] = (float)ratio;
                }
                __syncthreads();
                if (w.accept) {
                    accepted = ch;
                    break;
                }
                const float c1 = __fadd_rn(c, Z);
                const fx_t Rt = walk_mass_pass<DT>(w, ring, tsrc, dsrc, NV, Kq, Iq, Kp, Ip, c1, cf, gcount, npass);
                const float R = fx_to_float(Rt);
                if (R > 0.0f) {
                    Rlast = Rt;
                    c = c1;
                    Z = R;
                    masses_ready = true;
                } else {
                    masses_ready = false;  // the residual is empty: r_k stays
                }
            }
            if (accepted >= 0) {
                if (tid == 0 && leader) {
                    out[depth] = w.tok[accepted];
                    path[depth] = accepted;
                }
                ++depth;
                n = accepted;
                __syncthreads();
                continue;
            }
            // the token: from r_k = (q - c p)+ / Z, by inverse CDF over its slice masses
            const uint4 *dk = (c > 0.0f) ? dsrc : nullptr;
            if (!masses_ready)
                Rlast = walk_mass_pass<DT>(w, ring, tsrc, dk, NV, Kq, Iq, Kp, Ip, c, cf, gcount, npass);
            const int t = walk_pick<DT>(w, tsrc, dk, NV, Kq, Iq, Kp, Ip, c, cf, u0, Rlast);
            if (tid == 0 && leader)
                out[depth] = t;
            break;
        }
    }
    if (tid == 0 && leader) {
        for (int q = depth + 1; q <= M; ++q)
            out[q] = -1;
        for (int q = depth; q <= M; ++q)
            path[q] = -1;
        p.nacc[b] = depth;
        if (p.hist)
            atomicAdd(&p.hist[depth], 1ull);
        p.ws_err[b] = 0;
    }
    if (tid == 0 && w.ring.abort) {
        atomicOr(p.status, kErrTimeout);
        // never leave with a bulk copy still writing into this CTA's shared
        // memory: a bounded wait on the last tile issued into each stage
        for (int st = 0; st < kStagesW; ++st) {
            const int lk = w.ring.last_g[st];
            if (lk >= 0) {
                int never = 0;
                sv::mbar_wait_bounded(&w.ring.full[st], walk_parity((uint32_t)lk), &never, kWaitLimitNs / 4);
            }
        }
    }
}

// =============================================================================
// Fused LM-head path: decisions from the GEMM epilogue's tile statistics
// =============================================================================
//
// The tensor-core product of the hidden states with the LM head leaves, per
// row and 256-column tile, (m, s) or (max, argmax), and the logit at the
// row's draft token (lmhead.cu).  One warp per position merges the tiles of
// the target row and of the draft row in tile order, then decides position i
// exactly as kernel A does.  A gather kernel then copies, per sequence, the
// hidden states of the rows at the first rejection j; their logits are
// recomputed on the tensor cores into compact [B, V] buffers, which kernels B
// and C sample from.

struct FusedArgs {
    const float *part_t, *part_d;  // [rows, tiles, 2]
    const float *zgat_t, *zgat_d;  // [rows]
    int tiles;
    const unsigned char *hid_t, *hid_d;  // hidden states, rows of row_bytes_t / row_bytes_d
    unsigned char *hc_t, *hc_d;          // [B] gathered rows
    int row_bytes_t, row_bytes_d;
};

__device__ __forceinline__ void merge_tiles(const float *part, int tiles, bool sampled, float cf, int lane, float &m,
                                            float &s, int &arg)
{
    if (sampled) {
        Online o{-INFINITY, 0.0f};
        for (int t = lane; t < tiles; t += 32)
            o = online_merge(o, Online{part[2 * t], part[2 * t + 1]}, cf);
        o = warp_merge(o, cf);
        m = o.m;
        s = o.s;
        arg = 0;
    } else {
        ArgMax a{-INFINITY, INT_MAX, 0};
        for (int t = lane; t < tiles; t += 32)
            a = argmax_merge(a, ArgMax{part[2 * t], __float_as_int(part[2 * t + 1]), 0});
        a = warp_argmax(a);
        m = a.v;
        s = 0.0f;
        arg = a.i;
    }
}

__global__ void __launch_bounds__(256) sv_fused_decide_kernel(const SvParams p, const FusedArgs f)
{
    sv::grid_dependency_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x * 8 + warp;
    const int N = p.N;
    if (unit >= p.B * (N + 1))
        return;
    const int b = unit / (N + 1), i = unit - b * (N + 1);
    float T;
    const int mode = sequence_mode(p, b, T);
    if (mode == MODE_INVALID) {
        if (lane == 0) {
            atomicOr(&p.ws_err[b], kErrBadValue);
            if (p.ratio_at && i < N)
                p.ratio_at[(size_t)b * N + i] = NAN;
        }
        return;
    }
    const bool sampled = mode == MODE_SAMPLED;
    const double cfd = sampled ? kLog2e / (double)T : 0.0;
    const float cf = (float)cfd;
    const size_t trow = (size_t)b * (N + 1) + i, drow = (size_t)b * N + i;
    float mq, Sq, mp = -INFINITY, Sp = 0.0f;
    int aq, ap;
    merge_tiles(f.part_t + trow * f.tiles * 2, f.tiles, sampled, cf, lane, mq, Sq, aq);
    if (sampled && i < N)
        merge_tiles(f.part_d + drow * f.tiles * 2, f.tiles, true, cf, lane, mp, Sp, ap);
    if (lane != 0)
        return;
    const int d = (i < N) ? p.tokens[drow] : 0;
    const bool bad_d = (i < N) && (d < 0 || d >= p.V);
    int errb = bad_d ? kErrBadToken : 0;
    if (!isfinite(mq) || (sampled && !(isfinite(Sq) && Sq > 0.0f)) ||
        (sampled && i < N && !(isfinite(mp) && isfinite(Sp) && Sp > 0.0f)))
        errb |= kErrBadValue;
    if (p.ratio_at && i < N)
        p.ratio_at[drow] = NAN;
    if (!sampled) {
        p.ws_tok[trow] = aq;
        if (i < N && d != aq)
            atomicMin(&p.ws_first[b], i);
        if (p.tstats) {
            p.tstats[trow * 2 + 0] = mq;
            p.tstats[trow * 2 + 1] = NAN;
        }
    } else {
        if (!errb && i < N) {
            const double ratio = decision_ratio(__ldcg(&f.zgat_t[trow]), __ldcg(&f.zgat_d[drow]), mq, Sq, mp, Sp, cfd);
            if (!accept_by_ratio(ratio, (double)p.u[trow]))
                atomicMin(&p.ws_first[b], i);
            if (p.ratio_at)
                p.ratio_at[drow] = (float)ratio;
        }
        float *st = p.ws_stats + trow * 4;
        st[0] = mq;
        st[1] = Sq;
        st[2] = mp;
        st[3] = Sp;
        if (p.tstats) {
            p.tstats[trow * 2 + 0] = mq;
            p.tstats[trow * 2 + 1] = Sq;
        }
        if (p.dstats && i < N) {
            p.dstats[drow * 2 + 0] = mp;
            p.dstats[drow * 2 + 1] = Sp;
        }
    }
    if (errb)
        atomicOr(&p.ws_err[b], errb);
}

// Hidden states of the rows at the first rejection j of every sequence into
// the compact buffers: the draft row, and the verifier row when its logits
// were not kept.
__global__ void __launch_bounds__(256) sv_fused_gather_kernel(const SvParams p, const FusedArgs f)
{
    sv::grid_dependency_wait();
    const int b = blockIdx.x, N = p.N;
    int j = __ldcg(&p.ws_first[b]);
    j = j > N ? N : j;
    if (f.hid_t) {
        const uint4 *src = reinterpret_cast<const uint4 *>(f.hid_t + ((size_t)b * (N + 1) + j) * f.row_bytes_t);
        uint4 *dst = reinterpret_cast<uint4 *>(f.hc_t + (size_t)b * f.row_bytes_t);
        for (int v = threadIdx.x; v < f.row_bytes_t / 16; v += blockDim.x)
            dst[v] = __ldg(src + v);
    }
    if (j < N && f.hid_d) {
        const uint4 *sd = reinterpret_cast<const uint4 *>(f.hid_d + ((size_t)b * N + j) * f.row_bytes_d);
        uint4 *dd = reinterpret_cast<uint4 *>(f.hc_d + (size_t)b * f.row_bytes_d);
        for (int v = threadIdx.x; v < f.row_bytes_d / 16; v += blockDim.x)
            dd[v] = __ldg(sd + v);
    }
}

// =============================================================================
// Self-test of the bounded waits
// =============================================================================
//
// Every mbarrier wait in the library gives up after a time limit and reports
// it.  This kernel waits on a barrier that nothing ever arrives at, with the
// same bounded wait, and records whether it gave up.
__device__ int g_sv_timeout_probe;

__global__ void sv_timeout_probe_kernel(uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int never;
    if (threadIdx.x == 0) {
        never = 0;
        sv::mbar_init(&bar, 1);
        sv::fence_mbar_init();
        const bool completed = sv::mbar_wait_bounded(&bar, 0, &never, limit_ns);
        g_sv_timeout_probe = completed ? 1 : 2;
    }
}

} // namespace

// =============================================================================
// host side
// =============================================================================

struct spec_verify_ctx {
    int device;
    int max_B, max_N, V;
    sv_dtype dtype;
    int num_sms;
    int cluster_override;                // kernel A cluster size, 0 = automatic
    int clusters_a[kMaxCluster + 1];     // co-resident clusters of kernel A per size, 0 = none
    int clusters_tree[kMaxCluster + 1];  // the same for kernel A over tree nodes
    void *ws;
    int mass_ctas;                       // resident CTAs of the mass kernel (all SMs)
    int *ws_first, *ws_err, *ws_tok, *status;
    unsigned long long *ws_xc;
    float *ws_stats, *ws_slice;
    unsigned long long *hist;  // [max_N + 2]: accepted-draft histogram, then invalid
    // fused LM-head path: scratch allocated on its first call (and when K grows)
    void *fz;
    int fz_Kt, fz_Kd;
    int fz_keep;        // the statistics products also write every row's logits (else the rejected rows are recomputed)
    int fz_keep_alloc;  // the mode the scratch was allocated for
    float *fz_part_t, *fz_part_d, *fz_zgat_t, *fz_zgat_d, *fz_lt, *fz_ld;
    unsigned char *fz_hc_t, *fz_hc_d;
    // profiling: events before kernel A, between the kernels and after kernel B
    int prof_on, prof_runs;
    cudaEvent_t *prof_ev;  // [kProfRuns][3]
};

namespace {

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess)
            return;
        ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev)
            cudaSetDevice(prev);
    }
};

int elt_bytes(sv_dtype dt) { return dt == SV_BF16 ? 2 : 4; }

template <typename K> cudaError_t set_kernel_attrs(K kernel, size_t smem)
{
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int DT> cudaError_t set_attrs()
{
    cudaError_t e = set_kernel_attrs(sv_rows_kernel<DT, false>, kSmemA);
    if (e == cudaSuccess)
        e = set_kernel_attrs(sv_row_kernel<DT, false>, kSmemA);
    if (e == cudaSuccess)
        e = set_kernel_attrs(sv_row_kernel<DT, false, true>, kSmemA);
    if (e == cudaSuccess)
        e = set_kernel_attrs(sv_row_kernel<DT, true>, kSmemA);
    if (e == cudaSuccess)
        e = set_kernel_attrs(sv_rows_kernel<DT, true>, kSmemA);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(sv_mass_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(sv_tree_walk_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemW);
    return e;
}

// Resident CTAs of the mass kernel on the whole device.
template <int DT> int mass_ctas(int num_sms)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sv_mass_kernel<DT>, kThreads, kSmemM) != cudaSuccess) {
        cudaGetLastError();
        n = 1;
    }
    return (n > 0 ? n : 1) * num_sms;
}

// Slices of 256 vectors per row.
int residual_slices(int V, sv_dtype dt)
{
    const int nv = V * (dt == SV_BF16 ? 2 : 4) / 16;
    return (nv + kSliceVecs - 1) / kSliceVecs;
}

// attr must hold two entries; `dependent` lets the launch overlap the tail of
// the previous kernel on the stream (the kernel waits for it on the device).
cudaLaunchConfig_t launch_config(unsigned grid, int C, size_t smem, cudaStream_t stream,
                                 cudaLaunchAttribute *attr, bool dependent = false)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dependent) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    return cfg;
}

template <typename K> int active_clusters(K kernel, int C, size_t smem)
{
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config((unsigned)(C * 1024), C, smem, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// Co-resident clusters of kernel A for every cluster size.
template <int DT, bool TREE = false> void query_clusters(int *a)
{
    for (int k = 1; k <= kMaxCluster; ++k)
        a[k] = active_clusters(sv_rows_kernel<DT, TREE>, k, kSmemA);
    a[1] = a[1] > 0 ? a[1] : 1;
}

// Smallest cluster that keeps each chunk within kMaxSlices slices.
int min_cluster(int nv) { return (nv + kMaxSlices * kSliceVecs - 1) / (kMaxSlices * kSliceVecs); }

int clamp_cluster(int C, int nv, const int *fits)
{
    const int cmin = min_cluster(nv);
    if (C < cmin)
        C = cmin;
    if (C > 8 && cmin <= 8)
        C = 8;
    if (C > nv)
        C = nv;
    if (C < 1)
        C = 1;
    while (C > 1 && C > cmin && fits[C] == 0)
        --C;
    return C;
}

// Kernel A: one CTA per position once there are at least two positions per
// SM, else split the rows over a cluster for parallelism (about two waves of
// four CTAs per SM), down to 4 KiB of a row per CTA.  Measured on GB300: 384
// positions (mixed batch) 56.4 us with one CTA per position against 59.5 us in
// clusters of 4; 1024 tree nodes 137.5 us against 139.3 us in clusters of 2;
// 5 positions of 4 KiB rows 17.7 us per call unsplit against 18.7 us in
// clusters of 8.
int cluster_a(const spec_verify_ctx *c, int B, int N, bool tree = false)
{
    if (c->cluster_override > 0)
        return c->cluster_override;
    const int nv = c->V * elt_bytes(c->dtype) / 16;
    const int *fits = tree ? c->clusters_tree : c->clusters_a;
    const long long units = (long long)B * (N + 1);
    if (units >= 2LL * c->num_sms)
        return clamp_cluster(1, nv, fits);
    const long long want = 8LL * c->num_sms;
    int C = (int)((want + units - 1) / (units > 0 ? units : 1));
    // a CTA's share of a row stays at least 4 KiB: shorter rows are not split
    // (tiny rows gain nothing from a cluster but its launch and barriers)
    const long long by_len = (long long)nv * 16 / 4096;
    if (C > by_len)
        C = by_len > 1 ? (int)by_len : 1;
    return clamp_cluster(C < 8 ? C : 8, nv, fits);
}

sv_status run_impl(spec_verify_ctx *ctx, const void *target, const void *draft, const int32_t *tokens,
                   const float *u, const float *T, int greedy, int B, int N, int32_t *out,
                   int32_t *nacc, void *stream, float *q_at, float *p_at, float *tstats, float *dstats,
                   float *ratio_at)
{
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    if (B < 0 || B > ctx->max_B || N < 0 || N > ctx->max_N)
        return SV_ERR_INVALID_ARG;
    if (B == 0)
        return SV_OK;
    if (!target || !out || !nacc)
        return SV_ERR_INVALID_ARG;
    if (N > 0 && !tokens)
        return SV_ERR_INVALID_ARG;
    if (!greedy && (!T || !u || (N > 0 && !draft)))
        return SV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(target) & 15u) || (draft && (reinterpret_cast<uintptr_t>(draft) & 15u)))
        return SV_ERR_INVALID_ARG;
    const int CA = cluster_a(ctx, B, N);
    const int nv = ctx->V * elt_bytes(ctx->dtype) / 16;
    if ((nv + CA - 1) / CA > kMaxSlices * kSliceVecs)
        return SV_ERR_SHAPE;
    const long long units = (long long)B * (N + 1);
    if (units * CA > INT_MAX)
        return SV_ERR_INVALID_ARG;
    const long long tiles = (long long)B * ((nv + kTileVecsM - 1) / kTileVecsM);
    const int grid_m = (int)(tiles < ctx->mass_ctas ? tiles : ctx->mass_ctas);

    if (reinterpret_cast<uintptr_t>(ctx->ws_slice) & 15u)  // kernel C reads it as float4
        return SV_ERR_CUDA;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return SV_ERR_CUDA;

    SvParams prm{};
    prm.target = target;
    prm.draft = greedy ? nullptr : draft;
    prm.tokens = tokens;
    prm.u = u;
    prm.T = T;
    prm.out = out;
    prm.nacc = nacc;
    prm.q_at = q_at;
    prm.p_at = p_at;
    prm.tstats = tstats;
    prm.dstats = dstats;
    prm.ratio_at = ratio_at;
    prm.ws_first = ctx->ws_first;
    prm.ws_err = ctx->ws_err;
    prm.ws_tok = ctx->ws_tok;
    prm.ws_xc = ctx->ws_xc;
    prm.ws_stats = ctx->ws_stats;
    prm.ws_slice = ctx->ws_slice;
    prm.hist = ctx->hist;
    prm.hist_invalid = ctx->hist ? ctx->hist + ctx->max_N + 1 : nullptr;
    prm.status = ctx->status;
    prm.parent = nullptr;
    prm.path = nullptr;
    prm.compact_t = 0;
    prm.compact_d = 0;
    prm.B = B;
    prm.N = N;
    prm.V = ctx->V;
    prm.greedy = greedy ? 1 : 0;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaEvent_t *ev = nullptr;
    if (ctx->prof_on && ctx->prof_runs < kProfRuns)
        ev = ctx->prof_ev + 3 * ctx->prof_runs++;
    if (ev)
        cudaEventRecord(ev[0], st);
    cudaLaunchAttribute attr[2];
    cudaError_t e;
    const bool wave = CA == 1 && units >= ctx->clusters_a[1];
    const bool packed = CA == 1 && !wave && units >= 2LL * ctx->num_sms && B <= kPackMaxB;
    if (wave || packed) {
        // One CTA per logit row (B target rows at position N, two rows at the
        // others).  Measured on GB300: headline 212.3 -> 209.1 us per call,
        // stress 682.3 -> 672.4 us.  Below a wave of positions the rows that
        // are read are packed at the front of the grid, target rows first, so
        // that they all start in the first wave and without a dependent load
        // (mixed batch, 384 positions: 38.4 -> 35.5 us against kernel A's CTA
        // per position; batches of tiny rows keep kernel A, 10.5 against 12.5 us).
        cudaLaunchConfig_t cfg = launch_config((unsigned)(B * (2LL * N + 1)), 1, kSmemA, st, attr);
        if (packed)
            e = (ctx->dtype == SV_BF16) ? cudaLaunchKernelEx(&cfg, sv_row_kernel<SV_BF16, false, true>, prm)
                                        : cudaLaunchKernelEx(&cfg, sv_row_kernel<SV_F32, false, true>, prm);
        else
            e = (ctx->dtype == SV_BF16) ? cudaLaunchKernelEx(&cfg, sv_row_kernel<SV_BF16, false>, prm)
                                        : cudaLaunchKernelEx(&cfg, sv_row_kernel<SV_F32, false>, prm);
    } else {
        cudaLaunchConfig_t cfg = launch_config((unsigned)(units * CA), CA, kSmemA, st, attr);
        e = (ctx->dtype == SV_BF16) ? cudaLaunchKernelEx(&cfg, sv_rows_kernel<SV_BF16, false>, prm)
                                    : cudaLaunchKernelEx(&cfg, sv_rows_kernel<SV_F32, false>, prm);
    }
    if (e == cudaSuccess) {
        if (ev)
            cudaEventRecord(ev[1], st);
        // B and C are dependent launches (their start overlaps the previous
        // kernel's tail), except between the profiling events
        cudaLaunchAttribute pdl[1];
        pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pdl[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfgm = {};
        cfgm.gridDim = dim3((unsigned)(grid_m > 0 ? grid_m : 1));
        cfgm.blockDim = dim3(kThreads);
        cfgm.dynamicSmemBytes = kSmemM;
        cfgm.stream = st;
        cfgm.attrs = pdl;
        cfgm.numAttrs = ev == nullptr ? 1 : 0;
        e = (ctx->dtype == SV_BF16) ? cudaLaunchKernelEx(&cfgm, sv_mass_kernel<SV_BF16>, prm)
                                    : cudaLaunchKernelEx(&cfgm, sv_mass_kernel<SV_F32>, prm);
        if (e == cudaSuccess) {
            cudaLaunchConfig_t cfgp = {};
            cfgp.gridDim = dim3((unsigned)B);
            cfgp.blockDim = dim3(kPickThreads);
            cfgp.stream = st;
            cfgp.attrs = pdl;
            cfgp.numAttrs = 1;
            e = (ctx->dtype == SV_BF16) ? cudaLaunchKernelEx(&cfgp, sv_pick_kernel<SV_BF16>, prm)
                                        : cudaLaunchKernelEx(&cfgp, sv_pick_kernel<SV_F32>, prm);
        }
        if (ev && e == cudaSuccess)
            cudaEventRecord(ev[2], st);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

sv_status tree_run_impl(spec_verify_ctx *ctx, const void *target, const void *draft, const int32_t *parent,
                        const int32_t *tokens, const float *u, const float *T, int greedy, int B, int M,
                        int32_t *out, int32_t *path, int32_t *nacc, float *tstats, float *dstats, float *ratio_at,
                        void *stream)
{
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    if (B < 0 || B > ctx->max_B || M < 0 || M > ctx->max_N || M + 1 > kMaxTreeNodes)
        return SV_ERR_INVALID_ARG;
    if (B == 0)
        return SV_OK;
    if (!target || !parent || !tokens || !out || !path || !nacc)
        return SV_ERR_INVALID_ARG;
    if (!greedy && (!T || !u || (M > 0 && !draft)))
        return SV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(target) & 15u) || (draft && (reinterpret_cast<uintptr_t>(draft) & 15u)))
        return SV_ERR_INVALID_ARG;
    const int nv = ctx->V * elt_bytes(ctx->dtype) / 16;
    if ((nv + kSliceVecs - 1) / kSliceVecs > kMaxWalkSlices)
        return SV_ERR_SHAPE;
    const int CA = cluster_a(ctx, B, M, /*tree=*/true);
    if ((nv + CA - 1) / CA > kMaxSlices * kSliceVecs)
        return SV_ERR_SHAPE;
    const long long units = (long long)B * (M + 1);
    if (units * CA > INT_MAX)
        return SV_ERR_INVALID_ARG;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return SV_ERR_CUDA;

    SvParams prm{};
    memset(&prm, 0, sizeof prm);
    prm.target = target;
    prm.draft = greedy ? nullptr : draft;
    prm.tokens = tokens;
    prm.u = u;
    prm.T = T;
    prm.out = out;
    prm.nacc = nacc;
    prm.tstats = tstats;
    prm.dstats = dstats;
    prm.ratio_at = ratio_at;
    prm.ws_first = ctx->ws_first;
    prm.ws_err = ctx->ws_err;
    prm.ws_tok = ctx->ws_tok;
    prm.ws_xc = ctx->ws_xc;
    prm.ws_stats = ctx->ws_stats;
    prm.ws_slice = ctx->ws_slice;
    prm.hist = ctx->hist;
    prm.hist_invalid = ctx->hist ? ctx->hist + ctx->max_N + 1 : nullptr;
    prm.status = ctx->status;
    prm.parent = parent;
    prm.path = path;
    prm.B = B;
    prm.N = M;
    prm.V = ctx->V;
    prm.greedy = greedy ? 1 : 0;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    cudaError_t e;
    if (CA == 1 && units >= ctx->clusters_tree[1]) {
        // one CTA per logit row: each node's target row and, if it has
        // children, its draft row (64-tree call 132.1 -> 125.4 us)
        cudaLaunchConfig_t cfg = launch_config((unsigned)(2LL * units), 1, kSmemA, st, attr);
        e = (ctx->dtype == SV_BF16) ? cudaLaunchKernelEx(&cfg, sv_row_kernel<SV_BF16, true>, prm)
                                    : cudaLaunchKernelEx(&cfg, sv_row_kernel<SV_F32, true>, prm);
    } else {
        cudaLaunchConfig_t cfg = launch_config((unsigned)(units * CA), CA, kSmemA, st, attr);
        e = (ctx->dtype == SV_BF16) ? cudaLaunchKernelEx(&cfg, sv_rows_kernel<SV_BF16, true>, prm)
                                    : cudaLaunchKernelEx(&cfg, sv_rows_kernel<SV_F32, true>, prm);
    }
    if (e == cudaSuccess) {
        cudaLaunchAttribute pdl[1];
        pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pdl[0].val.programmaticStreamSerializationAllowed = 1;
        // a cluster of CW CTAs per tree splits each residual pass (one CTA per SM)
        int CW = ctx->num_sms / B;
        CW = CW < 1 ? 1 : CW > kMaxWalkCluster ? kMaxWalkCluster : CW;
        cudaLaunchAttribute wattr[2];
        wattr[0] = pdl[0];
        wattr[1].id = cudaLaunchAttributeClusterDimension;
        wattr[1].val.clusterDim.x = (unsigned)CW;
        wattr[1].val.clusterDim.y = 1;
        wattr[1].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfgw = {};
        cfgw.gridDim = dim3((unsigned)(B * CW));
        cfgw.blockDim = dim3(kWalkThreads);
        cfgw.dynamicSmemBytes = kSmemW;
        cfgw.stream = st;
        cfgw.attrs = wattr;
        cfgw.numAttrs = 2;
        e = (ctx->dtype == SV_BF16) ? cudaLaunchKernelEx(&cfgw, sv_tree_walk_kernel<SV_BF16>, prm)
                                    : cudaLaunchKernelEx(&cfgw, sv_tree_walk_kernel<SV_F32>, prm);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return SV_OK;
}

// Scratch of the fused path, sized for the context's limits and the widest
// hidden states seen so far.
// Scratch of the fused path: tile statistics and draft-token logits of every
// row; the logits of every verifier row (kept) or, for the recomputation, of
// one verifier row per sequence and its hidden state; the logits and hidden
// state of one draft row per sequence (always recomputed).
sv_status fused_scratch(spec_verify_ctx *ctx, int Kt, int Kd)
{
    if (ctx->fz && Kt <= ctx->fz_Kt && Kd <= ctx->fz_Kd && ctx->fz_keep == ctx->fz_keep_alloc)
        return SV_OK;
    Kt = Kt > ctx->fz_Kt ? Kt : ctx->fz_Kt;
    Kd = Kd > ctx->fz_Kd ? Kd : ctx->fz_Kd;
    const bool keep = ctx->fz_keep != 0;
    const size_t nb = (size_t)(ctx->max_B > 0 ? ctx->max_B : 1);
    const size_t rows_t = nb * (size_t)(ctx->max_N + 1), rows_d = nb * (size_t)(ctx->max_N > 0 ? ctx->max_N : 1);
    const size_t tiles = (size_t)svlm::tiles(ctx->V);
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t lt_rows = keep ? rows_t : nb;
    const size_t o_pt = 0, o_pd = o_pt + up(rows_t * tiles * 8), o_zt = o_pd + up(rows_d * tiles * 8);
    const size_t o_zd = o_zt + up(rows_t * 4), o_lt = o_zd + up(rows_d * 4), o_ld = o_lt + up(lt_rows * ctx->V * 4);
    const size_t o_ht = o_ld + up(nb * ctx->V * 4);
    const size_t o_hd = o_ht + (keep ? 0 : up(nb * (size_t)Kt * 2));
    const size_t bytes = o_hd + up(nb * (size_t)(Kd > 0 ? Kd : 8) * 2);
    cudaFree(ctx->fz);
    ctx->fz = nullptr;
    if (cudaMalloc(&ctx->fz, bytes) != cudaSuccess) {
        cudaGetLastError();
        ctx->fz = nullptr;
        return SV_ERR_OOM;
    }
    unsigned char *z = static_cast<unsigned char *>(ctx->fz);
    ctx->fz_part_t = reinterpret_cast<float *>(z + o_pt);
    ctx->fz_part_d = reinterpret_cast<float *>(z + o_pd);
    ctx->fz_zgat_t = reinterpret_cast<float *>(z + o_zt);
    ctx->fz_zgat_d = reinterpret_cast<float *>(z + o_zd);
    ctx->fz_lt = reinterpret_cast<float *>(z + o_lt);
    ctx->fz_ld = reinterpret_cast<float *>(z + o_ld);
    ctx->fz_hc_t = keep ? nullptr : z + o_ht;
    ctx->fz_hc_d = z + o_hd;
    ctx->fz_Kt = Kt;
    ctx->fz_Kd = Kd;
    ctx->fz_keep_alloc = ctx->fz_keep;
    return SV_OK;
}

sv_status fused_run_impl(spec_verify_ctx *ctx, const void *ht, const void *wt, int Kt, const void *hd, const void *wd,
                         int Kd, const int32_t *tokens, const float *u, const float *T, int greedy, int B, int N,
                         int32_t *out, int32_t *nacc, float *tstats, float *dstats, float *ratio_at, void *stream)
{
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    if (ctx->dtype != SV_F32)
        return SV_ERR_DTYPE;  // the recomputed logits are float32
    if (B < 0 || B > ctx->max_B || N < 0 || N > ctx->max_N || Kt < 8 || Kt % 8 != 0)
        return SV_ERR_INVALID_ARG;
    if (B == 0)
        return SV_OK;
    const bool need_draft = !greedy && N > 0;
    if (!ht || !wt || !out || !nacc || (N > 0 && !tokens) || (!greedy && (!T || !u)))
        return SV_ERR_INVALID_ARG;
    if (need_draft && (!hd || !wd || Kd < 8 || Kd % 8 != 0))
        return SV_ERR_INVALID_ARG;
    for (const void *q : {ht, wt, hd, wd})
        if (reinterpret_cast<uintptr_t>(q) & 15u)
            return SV_ERR_INVALID_ARG;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return SV_ERR_CUDA;
    sv_status r = fused_scratch(ctx, Kt, need_draft ? Kd : 8);
    if (r != SV_OK)
        return r;
    const int V = ctx->V;
    const bool keep = ctx->fz_keep != 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // 1. tile statistics of every verifier row and every draft row (and, when
    //    kept, the verifier rows' logits: that product is bound by its MMAs,
    //    while the draft's, at its short K, would be bound by the stores)
    svlm::StatsArgs a{tokens, greedy ? nullptr : T, greedy ? 1 : 0, N, N + 1, ctx->fz_part_t, ctx->fz_zgat_t};
    if ((r = svlm::launch_stats(ht, wt, B * (N + 1), V, Kt, a, st, keep ? ctx->fz_lt : nullptr)) != SV_OK)
        return r;
    if (need_draft) {
        svlm::StatsArgs ad{tokens, T, 0, N, N, ctx->fz_part_d, ctx->fz_zgat_d};
        if ((r = svlm::launch_stats(hd, wd, B * N, V, Kd, ad, st)) != SV_OK)
            return r;
    }

    SvParams prm{};
    memset(&prm, 0, sizeof prm);
    prm.target = ctx->fz_lt;
    prm.draft = ctx->fz_ld;
    prm.tokens = tokens;
    prm.u = u;
    prm.T = T;
    prm.out = out;
    prm.nacc = nacc;
    prm.tstats = tstats;
    prm.dstats = dstats;
    prm.ratio_at = ratio_at;
    prm.ws_first = ctx->ws_first;
    prm.ws_err = ctx->ws_err;
    prm.ws_tok = ctx->ws_tok;
    prm.ws_xc = ctx->ws_xc;
    prm.ws_stats = ctx->ws_stats;
    prm.ws_slice = ctx->ws_slice;
    prm.hist = ctx->hist;
    prm.hist_invalid = ctx->hist ? ctx->hist + ctx->max_N + 1 : nullptr;
    prm.status = ctx->status;
    prm.compact_t = keep ? 0 : 1;  // kept: the rows (b, j) of the full verifier logits
    prm.compact_d = 1;
    prm.B = B;
    prm.N = N;
    prm.V = V;
    prm.greedy = greedy ? 1 : 0;
    FusedArgs f;
    f.part_t = ctx->fz_part_t;
    f.part_d = ctx->fz_part_d;
    f.zgat_t = ctx->fz_zgat_t;
    f.zgat_d = ctx->fz_zgat_d;
    f.tiles = svlm::tiles(V);
    f.hid_t = keep ? nullptr : static_cast<const unsigned char *>(ht);
    f.hid_d = need_draft ? static_cast<const unsigned char *>(hd) : nullptr;
    f.hc_t = ctx->fz_hc_t;
    f.hc_d = ctx->fz_hc_d;
    f.row_bytes_t = Kt * 2;
    f.row_bytes_d = need_draft ? Kd * 2 : 0;

    // 2. decisions
    const long long units = (long long)B * (N + 1);
    sv_fused_decide_kernel<<<(unsigned)((units + 7) / 8), 256, 0, st>>>(prm, f);
    if (cudaGetLastError() != cudaSuccess)
        return SV_ERR_CUDA;
    // 3. the hidden rows at the first rejection; 4. their logits, recomputed
    //    (the draft row always, the verifier row when not kept)
    if (!keep || need_draft) {
        sv_fused_gather_kernel<<<(unsigned)B, 256, 0, st>>>(prm, f);
        if (cudaGetLastError() != cudaSuccess)
            return SV_ERR_CUDA;
    }
    if (!keep && (r = svlm::launch_logits(ctx->fz_hc_t, wt, B, V, Kt, ctx->fz_lt, st)) != SV_OK)
        return r;
    if (need_draft && (r = svlm::launch_logits(ctx->fz_hc_d, wd, B, V, Kd, ctx->fz_ld, st)) != SV_OK)
        return r;
    // 5. residual masses and the token, as in spec_verify_run
    const int nv = V * 4 / 16;
    const long long tiles_m = (long long)B * ((nv + kTileVecsM - 1) / kTileVecsM);
    const int grid_m = (int)(tiles_m < ctx->mass_ctas ? tiles_m : ctx->mass_ctas);
    sv_mass_kernel<SV_F32><<<(unsigned)(grid_m > 0 ? grid_m : 1), kThreads, kSmemM, st>>>(prm);
    sv_pick_kernel<SV_F32><<<(unsigned)B, kPickThreads, 0, st>>>(prm);
    if (cudaGetLastError() != cudaSuccess)
        return SV_ERR_CUDA;
    return SV_OK;
}

} // namespace

extern "C" {

sv_status spec_verify_create(spec_verify_ctx **out, int device, int max_B, int max_N, int V, sv_dtype dtype)
{
    if (!out)
        return SV_ERR_INVALID_ARG;
    *out = nullptr;
    if (dtype != SV_F32 && dtype != SV_BF16)
        return SV_ERR_DTYPE;
    if (max_B < 0 || max_N < 0 || device < 0)
        return SV_ERR_INVALID_ARG;
    if (V < 1 || ((long long)V * elt_bytes(dtype)) % 16 != 0)
        return SV_ERR_SHAPE;
    if ((long long)V * elt_bytes(dtype) / 16 > (long long)kMaxCluster * kMaxSlices * kSliceVecs)
        return SV_ERR_SHAPE;

    DeviceGuard guard(device);
    if (!guard.ok)
        return SV_ERR_CUDA;
    spec_verify_ctx *c = static_cast<spec_verify_ctx *>(calloc(1, sizeof(spec_verify_ctx)));
    if (!c)
        return SV_ERR_OOM;
    c->device = device;
    c->max_B = max_B;
    c->max_N = max_N;
    c->V = V;
    c->dtype = dtype;
    if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        free(c);
        return SV_ERR_CUDA;
    }
    cudaError_t e = (dtype == SV_BF16) ? set_attrs<SV_BF16>() : set_attrs<SV_F32>();
    if (e != cudaSuccess) {
        cudaGetLastError();
        free(c);
        return SV_ERR_CUDA;
    }
    if (dtype == SV_BF16) {
        query_clusters<SV_BF16>(c->clusters_a);
        query_clusters<SV_BF16, true>(c->clusters_tree);
    } else {
        query_clusters<SV_F32>(c->clusters_a);
        query_clusters<SV_F32, true>(c->clusters_tree);
    }

    c->mass_ctas = (dtype == SV_BF16) ? mass_ctas<SV_BF16>(c->num_sms) : mass_ctas<SV_F32>(c->num_sms);
    c->fz_keep = 1;  // the fused path keeps every row's logits unless told otherwise

    // workspace: hist[max_N+2] (u64) | first[nb] err[nb] tok[ntok] stats[4*ntok] | xc[ntok] (u64) |
    // slice[nb*S*8] status;
    // the slice shares start on a 256-byte boundary (kernel C reads them as float4)
    const size_t nb = (size_t)(max_B > 0 ? max_B : 1);
    const size_t ntok = nb * (size_t)(max_N + 1);
    const size_t nslice = nb * (size_t)residual_slices(V, dtype) * kConsWarps;
    const size_t hist_ints = ((size_t)(max_N + 2) * 2 + 63) / 64 * 64;
    const size_t xc_off = (hist_ints + 2 * nb + 5 * ntok + 1) / 2 * 2;  // 8-byte aligned
    const size_t slice_off = (xc_off + 2 * ntok + 63) / 64 * 64;
    const size_t bytes = sizeof(int) * (slice_off + nslice + 1);
    if (cudaMalloc(&c->ws, bytes) != cudaSuccess) {
        cudaGetLastError();
        free(c);
        return SV_ERR_OOM;
    }
    c->hist = static_cast<unsigned long long *>(c->ws);
    int *w = static_cast<int *>(c->ws) + hist_ints;
    c->ws_first = w;
    c->ws_err = w + nb;
    c->ws_tok = w + 2 * nb;
    c->ws_stats = reinterpret_cast<float *>(w + 2 * nb + ntok);
    c->ws_xc = reinterpret_cast<unsigned long long *>(static_cast<int *>(c->ws) + xc_off);
    c->ws_slice = reinterpret_cast<float *>(static_cast<int *>(c->ws) + slice_off);
    c->status = static_cast<int *>(c->ws) + slice_off + nslice;
    if (cudaMemset(c->ws, 0, bytes) != cudaSuccess || cudaMemset(c->ws_first, 0x7f, sizeof(int) * nb) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        cudaFree(c->ws);
        free(c);
        return SV_ERR_CUDA;
    }
    *out = c;
    return SV_OK;
}

sv_status spec_verify_run(spec_verify_ctx *ctx, const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *uniforms, const float *temperature,
                          int greedy, int B, int N, int32_t *out_tokens, int32_t *num_accepted, void *stream)
{
    return run_impl(ctx, target_logits, draft_logits, draft_tokens, uniforms, temperature, greedy, B, N,
                    out_tokens, num_accepted, stream, nullptr, nullptr, nullptr, nullptr, nullptr);
}

sv_status spec_verify_run_debug(spec_verify_ctx *ctx, const void *target_logits, const void *draft_logits,
                                const int32_t *draft_tokens, const float *uniforms, const float *temperature,
                                int greedy, int B, int N, int32_t *out_tokens, int32_t *num_accepted,
                                void *stream, float *q_at_draft, float *p_at_draft, float *target_row_stats,
                                float *draft_row_stats, float *ratio_at_draft)
{
    return run_impl(ctx, target_logits, draft_logits, draft_tokens, uniforms, temperature, greedy, B, N,
                    out_tokens, num_accepted, stream, q_at_draft, p_at_draft, target_row_stats,
                    draft_row_stats, ratio_at_draft);
}

sv_status spec_verify_tree_run(spec_verify_ctx *ctx, const void *target_logits, const void *draft_logits,
                               const int32_t *parent, const int32_t *draft_tokens, const float *uniforms,
                               const float *temperature, int greedy, int B, int M, int32_t *out_tokens,
                               int32_t *path_nodes, int32_t *num_accepted, float *target_row_stats,
                               float *draft_row_stats, float *ratio_at_node, void *stream)
{
    return tree_run_impl(ctx, target_logits, draft_logits, parent, draft_tokens, uniforms, temperature, greedy, B,
                         M, out_tokens, path_nodes, num_accepted, target_row_stats, draft_row_stats, ratio_at_node,
                         stream);
}

sv_status spec_verify_run_fused(spec_verify_ctx *ctx, const void *target_hidden, const void *target_weight,
                                int Kt, const void *draft_hidden, const void *draft_weight, int Kd,
                                const int32_t *draft_tokens, const float *uniforms, const float *temperature,
                                int greedy, int B, int N, int32_t *out_tokens, int32_t *num_accepted,
                                float *target_row_stats, float *draft_row_stats, float *ratio_at_draft,
                                void *stream)
{
    return fused_run_impl(ctx, target_hidden, target_weight, Kt, draft_hidden, draft_weight, Kd, draft_tokens,
                          uniforms, temperature, greedy, B, N, out_tokens, num_accepted, target_row_stats,
                          draft_row_stats, ratio_at_draft, stream);
}

sv_status spec_verify_selftest_timeout(int limit_us, int *gave_up, void *stream)
{
    if (limit_us < 1 || limit_us > 10000000 || !gave_up)
        return SV_ERR_INVALID_ARG;
    *gave_up = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int zero = 0;
    int flag = 0;
    if (cudaMemcpyToSymbolAsync(g_sv_timeout_probe, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st) !=
        cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    sv_timeout_probe_kernel<<<1, 32, 0, st>>>((uint64_t)limit_us * 1000ull);
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&flag, g_sv_timeout_probe, sizeof flag, 0, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    *gave_up = flag == 2 ? 1 : 0;
    return SV_OK;
}

sv_status spec_verify_get_status(spec_verify_ctx *ctx)
{
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return SV_ERR_CUDA;
    int bits = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&bits, ctx->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    if (bits) {
        const int zero = 0;
        if (cudaMemcpy(ctx->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            return SV_ERR_CUDA;
        }
    }
    if (bits & kErrTimeout)
        return SV_ERR_TIMEOUT;
    if (bits & kErrBadTree)
        return SV_ERR_BAD_TREE;
    if (bits & kErrBadToken)
        return SV_ERR_BAD_TOKEN;
    if (bits & kErrBadValue)
        return SV_ERR_BAD_VALUE;
    return SV_OK;
}

sv_status spec_verify_acceptance_counts(spec_verify_ctx *ctx, uint64_t *counts, int ncounts, int reset)
{
    if (!ctx || !counts || ncounts < ctx->max_N + 2)
        return SV_ERR_INVALID_ARG;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return SV_ERR_CUDA;
    const size_t bytes = sizeof(unsigned long long) * (size_t)(ctx->max_N + 2);
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(counts, ctx->hist, bytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
        (reset && cudaMemset(ctx->hist, 0, bytes) != cudaSuccess) || (reset && cudaDeviceSynchronize() != cudaSuccess)) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    for (int k = ctx->max_N + 2; k < ncounts; ++k)
        counts[k] = 0;
    return SV_OK;
}

sv_status spec_verify_set_cluster_size(spec_verify_ctx *ctx, int cluster_size)
{
    if (!ctx || cluster_size < 0 || cluster_size > kMaxCluster)
        return SV_ERR_INVALID_ARG;
    if (cluster_size > 1 && ctx->clusters_a[cluster_size] == 0)
        return SV_ERR_INVALID_ARG;
    const int nv = ctx->V * elt_bytes(ctx->dtype) / 16;
    if (cluster_size > nv)
        return SV_ERR_INVALID_ARG;
    ctx->cluster_override = cluster_size;
    return SV_OK;
}

sv_status spec_verify_set_fused_logits(spec_verify_ctx *ctx, int keep)
{
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    ctx->fz_keep = keep ? 1 : 0;
    return SV_OK;
}

int spec_verify_cluster_size(spec_verify_ctx *ctx, int B, int N)
{
    if (!ctx)
        return 0;
    return cluster_a(ctx, B, N);
}

const char *spec_verify_error_string(sv_status s)
{
    switch (s) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: bad pointer, alignment, batch or draft count";
    case SV_ERR_SHAPE: return "SV_ERR_SHAPE: unsupported vocabulary size";
    case SV_ERR_DTYPE: return "SV_ERR_DTYPE: unknown logit dtype";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: a CUDA runtime call failed";
    case SV_ERR_OOM: return "SV_ERR_OOM: workspace allocation failed";
    case SV_ERR_BAD_TOKEN: return "SV_ERR_BAD_TOKEN: a draft token was outside [0, V)";
    case SV_ERR_BAD_VALUE: return "SV_ERR_BAD_VALUE: non-finite logits or temperature";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: a bounded wait in the kernel gave up";
    case SV_ERR_BAD_TREE: return "SV_ERR_BAD_TREE: a parent array broke parent[0] = -1, 0 <= parent[n] < n";
    case SV_ERR_TOO_LARGE:
        return "SV_ERR_TOO_LARGE: batch exceeds the fixed scratch of spec_verify_run_noalloc "
               "(B <= 2048, B*(N+1) <= 16384, B*ceil(V*elt/4KiB) <= 32768)";
    }
    return "unknown sv_status";
}

namespace {
void prof_free(spec_verify_ctx *ctx)
{
    if (ctx->prof_ev) {
        for (int k = 0; k < 3 * kProfRuns; ++k)
            cudaEventDestroy(ctx->prof_ev[k]);
        free(ctx->prof_ev);
        ctx->prof_ev = nullptr;
    }
    ctx->prof_on = 0;
    ctx->prof_runs = 0;
}
} // namespace

sv_status spec_verify_profile(spec_verify_ctx *ctx, int enable)
{
    if (!ctx)
        return SV_ERR_INVALID_ARG;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return SV_ERR_CUDA;
    if (!enable) {
        prof_free(ctx);
        return SV_OK;
    }
    if (!ctx->prof_ev) {
        ctx->prof_ev = static_cast<cudaEvent_t *>(calloc(3 * kProfRuns, sizeof(cudaEvent_t)));
        if (!ctx->prof_ev)
            return SV_ERR_OOM;
        for (int k = 0; k < 3 * kProfRuns; ++k)
            if (cudaEventCreate(&ctx->prof_ev[k]) != cudaSuccess) {
                cudaGetLastError();
                for (int m = 0; m < k; ++m)
                    cudaEventDestroy(ctx->prof_ev[m]);
                free(ctx->prof_ev);
                ctx->prof_ev = nullptr;
                return SV_ERR_CUDA;
            }
    }
    ctx->prof_on = 1;
    ctx->prof_runs = 0;
    return SV_OK;
}

sv_status spec_verify_profile_read(spec_verify_ctx *ctx, double *ms_rows, double *ms_sample, int *runs)
{
    if (!ctx || !ctx->prof_ev)
        return SV_ERR_INVALID_ARG;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return SV_ERR_CUDA;
    double a = 0.0, b = 0.0;
    for (int k = 0; k < ctx->prof_runs; ++k) {
        cudaEvent_t *ev = ctx->prof_ev + 3 * k;
        float t1 = 0.0f, t2 = 0.0f;
        if (cudaEventSynchronize(ev[2]) != cudaSuccess || cudaEventElapsedTime(&t1, ev[0], ev[1]) != cudaSuccess ||
            cudaEventElapsedTime(&t2, ev[1], ev[2]) != cudaSuccess) {
            cudaGetLastError();
            return SV_ERR_CUDA;
        }
        a += t1;
        b += t2;
    }
    if (ms_rows)
        *ms_rows = a;
    if (ms_sample)
        *ms_sample = b;
    if (runs)
        *runs = ctx->prof_runs;
    return SV_OK;
}

void spec_verify_destroy(spec_verify_ctx *ctx)
{
    if (!ctx)
        return;
    {
        DeviceGuard guard(ctx->device);
        prof_free(ctx);
        cudaFree(ctx->ws);
        cudaFree(ctx->fz);
    }
    free(ctx);
}

} // extern "C"

// =============================================================================
// entry point for callers that cannot allocate device memory
// =============================================================================
//
// spec_verify_run_noalloc runs the same kernels as spec_verify_run, but its
// scratch lives in the file-scope array below instead of a context
// workspace: per sequence the first-rejection slot and the error bits, per
// verified position the greedy argmax, the row statistics (mq, Sq, mp, Sp)
// and the 64-bit cell that pairs the position's two row CTAs, per 4 KiB slice of
// a sampled row pair the eight warp shares of its residual mass, and one
// status word.  The array is part of the module image: every GPU that
// loads this library holds it until the process exits, and nothing is ever
// allocated for it.  Host code only sees a stand-in symbol for it, so the
// device address is looked up once per device with cudaGetSymbolAddress.

namespace {
constexpr int kNoAllocMaxB = 2048;        // sequences per call
constexpr int kNoAllocMaxUnits = 16384;   // B*(N+1) verified positions per call
constexpr int kNoAllocMaxSlices = 32768;  // B*ceil(V*elt/4 KiB) residual slices per call
constexpr int kNoAllocXcOff = 2 * kNoAllocMaxB + 5 * kNoAllocMaxUnits;  // even: 8-byte aligned
constexpr int kNoAllocSliceOff = kNoAllocXcOff + 2 * kNoAllocMaxUnits;  // a multiple of 64 ints
static_assert(kNoAllocSliceOff % 64 == 0, "slice shares must start on a 256-byte boundary");
constexpr int kNoAllocInts = kNoAllocSliceOff + 8 * kNoAllocMaxSlices + 1;  // about 1.45 MiB
// the 256-sequence Qwen-vocabulary batch (V = 151936 bf16: 75 slices a row) fits
static_assert(256 * 75 <= kNoAllocMaxSlices, "the scratch holds a 256 x 151936 bf16 batch");
constexpr int kNoAllocMaxDevices = 64;
} // namespace

static __device__ __align__(256) int g_sv_noalloc_scratch[kNoAllocInts];

namespace {

struct NoAllocDevice {
    bool ready;
    int *scratch;     // device address of g_sv_noalloc_scratch on this device
    int num_sms;
    int mass_bf16, mass_f32;
    int clusters_bf16[kMaxCluster + 1];  // co-resident clusters of the row kernel per size
    int clusters_f32[kMaxCluster + 1];
};

std::mutex g_noalloc_mutex;
NoAllocDevice g_noalloc[kNoAllocMaxDevices];

// One-time set-up on `device` (which the caller has made current): resolve
// the scratch address, put it in its idle state, set the kernel attributes and
// record how many clusters of each size fit.  Synchronous.
sv_status noalloc_setup(int device, NoAllocDevice &nd)
{
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_sv_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    int *w = static_cast<int *>(ptr);
    if (cudaMemset(w, 0, sizeof(int) * kNoAllocInts) != cudaSuccess ||
        cudaMemset(w, 0x7f, sizeof(int) * kNoAllocMaxB) != cudaSuccess ||
        cudaDeviceGetAttribute(&nd.num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        set_attrs<SV_BF16>() != cudaSuccess || set_attrs<SV_F32>() != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    query_clusters<SV_BF16>(nd.clusters_bf16);
    query_clusters<SV_F32>(nd.clusters_f32);
    nd.mass_bf16 = mass_ctas<SV_BF16>(nd.num_sms);
    nd.mass_f32 = mass_ctas<SV_F32>(nd.num_sms);
    nd.scratch = w;
    nd.ready = true;
    return SV_OK;
}

} // namespace

extern "C" sv_status spec_verify_run_noalloc(const void *target_logits, const void *draft_logits,
                                            const int32_t *draft_tokens, const float *uniforms,
                                            const float *temperature, int greedy, int B, int N, int V,
                                            sv_dtype dtype, int32_t *out_tokens, int32_t *num_accepted,
                                            void *stream)
{
    if (dtype != SV_F32 && dtype != SV_BF16)
        return SV_ERR_DTYPE;
    if (B < 0 || N < 0)
        return SV_ERR_INVALID_ARG;
    if (V < 1 || ((long long)V * elt_bytes(dtype)) % 16 != 0 ||
        (long long)V * elt_bytes(dtype) / 16 > (long long)kMaxCluster * kMaxSlices * kSliceVecs)
        return SV_ERR_SHAPE;
    if (B > kNoAllocMaxB || (long long)B * (N + 1) > kNoAllocMaxUnits ||
        (long long)B * residual_slices(V, dtype) > kNoAllocMaxSlices)
        return SV_ERR_TOO_LARGE;
    if (B == 0)
        return SV_OK;

    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kNoAllocMaxDevices) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    NoAllocDevice *nd = &g_noalloc[device];
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (!nd->ready) {
            const sv_status st = noalloc_setup(device, *nd);
            if (st != SV_OK)
                return st;
        }
    }

    // A context on the stack that points into the static scratch.
    spec_verify_ctx c;
    memset(&c, 0, sizeof c);
    c.device = device;
    c.max_B = kNoAllocMaxB;
    c.max_N = kNoAllocMaxUnits;
    c.V = V;
    c.dtype = dtype;
    c.num_sms = nd->num_sms;
    memcpy(c.clusters_a, dtype == SV_BF16 ? nd->clusters_bf16 : nd->clusters_f32, sizeof c.clusters_a);
    c.mass_ctas = dtype == SV_BF16 ? nd->mass_bf16 : nd->mass_f32;
    int *w = nd->scratch;
    c.ws = w;
    c.ws_first = w;
    c.ws_err = w + kNoAllocMaxB;
    c.ws_tok = w + 2 * kNoAllocMaxB;
    c.ws_stats = reinterpret_cast<float *>(w + 2 * kNoAllocMaxB + kNoAllocMaxUnits);
    c.ws_xc = reinterpret_cast<unsigned long long *>(w + kNoAllocXcOff);
    c.ws_slice = reinterpret_cast<float *>(w + kNoAllocSliceOff);
    c.status = w + kNoAllocSliceOff + 8 * kNoAllocMaxSlices;

    // The scratch keeps whatever the previous call left in it: put the slots
    // this call uses into their starting state first (on the same stream, so
    // calls issued in stream order never see each other's values).
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(c.ws_first, 0x7f, sizeof(int) * B, st) != cudaSuccess ||
        cudaMemsetAsync(c.ws_err, 0, sizeof(int) * B, st) != cudaSuccess ||
        cudaMemsetAsync(c.status, 0, sizeof(int), st) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    return run_impl(&c, target_logits, draft_logits, draft_tokens, uniforms, temperature, greedy, B, N,
                    out_tokens, num_accepted, stream, nullptr, nullptr, nullptr, nullptr, nullptr);
}

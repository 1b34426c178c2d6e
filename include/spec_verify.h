/*
 * spec_verify.h -- C ABI of the GB300 speculative-sampling verify step.
 *
 * The operation (per sequence b, positions i = 0..N, tokens k = 0..V-1) is the
 * verify half of one speculative step as stated in "Speculative decoding --
 * draft, verify, repeat" (factory.pai-world.com, lesson 07-16), section
 * "Core algorithm", steps 3-6, with its build section's Step 1 (rejection
 * step) and Step 2 (residual distribution):
 *
 *   q_i = softmax(target_logits[b,i,:] / T_b)    i = 0..N     (verifier)
 *   p_i = softmax(draft_logits[b,i,:]  / T_b)    i = 0..N-1   (draft)
 *   scan i = 0..N-1: accept draft d_i iff p_i(d_i) == 0 or
 *                    u[b,i] < min(1, q_i(d_i) / p_i(d_i))
 *   first rejection j: token ~ normalise(max(0, q_j - p_j))
 *   no rejection:      bonus token ~ q_N
 *   emit d_0..d_{j-1} and that token; num_accepted = j.
 *
 * The final token is drawn by inverse CDF in ascending token order from the
 * single uniform u[b,N]: the smallest k with u*R < r_0+...+r_k, R the total
 * mass.  A residual of total mass 0 (q_j == p_j) draws from q_j instead.
 * Greedy sequences (greedy != 0, or T_b <= 0): a_i = argmax_k target[b,i,k]
 * (lowest index on ties); accept d_i iff d_i == a_i; emit a_j at the first
 * mismatch, else a_N.  Draft logits and uniforms are then not read.
 *
 * All tensors are caller-owned device memory, C-contiguous, row-major.  The
 * library never allocates or synchronises inside spec_verify_run; the run (three
 * kernel launches) is enqueued on the caller's stream and completes
 * asynchronously.  Further entry points below: tree verification, the verify
 * fused into the LM-head products, the LM-head product alone, the KV-cache
 * commit, acceptance counters, kernel timing and an allocation-free variant.
 *
 * Thread-safety: a context holds a small workspace that every run updates;
 * use one context per stream (runs on one stream are serialised by it).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spec_verify_ctx spec_verify_ctx;

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1, /* NULL/misaligned pointer, B or N outside the context's limits */
    SV_ERR_SHAPE = 2,       /* V unsupported (V*elt not a multiple of 16 bytes, or too large) */
    SV_ERR_DTYPE = 3,       /* unknown sv_dtype */
    SV_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, attribute, copy) */
    SV_ERR_OOM = 5,         /* workspace allocation failed at create */
    SV_ERR_BAD_TOKEN = 6,   /* device: some draft token was outside [0, V) */
    SV_ERR_BAD_VALUE = 7,   /* device: NaN/+inf/all -inf logits, or NaN/+inf/subnormal temperature */
    SV_ERR_TIMEOUT = 8,     /* device: a bounded wait inside the kernel gave up */
    SV_ERR_TOO_LARGE = 9,   /* spec_verify_run_noalloc: batch beyond its fixed scratch */
    SV_ERR_BAD_TREE = 10    /* device: a parent array broke parent[0] = -1, 0 <= parent[n] < n */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/*
 * Create a context on `device` for batches of up to max_B sequences with up
 * to max_N draft tokens over a vocabulary of V tokens stored as `dtype`.
 * Allocates a workspace of about 8*(max_N+2) + 8*max_B + 28*max_B*(max_N+1) +
 * 32*max_B*ceil(V*elt/4 KiB) bytes (per-sequence first-rejection slots and
 * error flags; per-position argmax, row statistics and the 64-bit cell that
 * pairs a position's two rows; per-slice residual masses, the acceptance counters)
 * and one status word.  spec_verify_run and
 * spec_verify_tree_run allocate nothing later; spec_verify_run_fused adds its
 * own scratch on its first call.
 * Requires V >= 1 and V*sizeof(dtype) a multiple of 16 (V % 8 == 0 for bf16,
 * V % 4 == 0 for f32).  Returns SV_ERR_SHAPE otherwise, SV_ERR_OOM if the
 * workspace cannot be allocated, SV_ERR_CUDA if the device cannot be used.
 * On failure *out is set to NULL.
 */
sv_status spec_verify_create(spec_verify_ctx **out, int device, int max_B, int max_N, int V,
                             sv_dtype dtype);

/*
 * Enqueue one verify step on `stream` (a cudaStream_t; NULL = legacy default
 * stream).
 *   target_logits  device [B, N+1, V] of dtype, 16-byte aligned base
 *   draft_logits   device [B, N, V] of dtype, 16-byte aligned base; may be
 *                  NULL when greedy != 0 or N == 0
 *   draft_tokens   device int32 [B, N]; may be NULL when N == 0
 *   uniforms       device float [B, N+1]: columns 0..N-1 feed the accept
 *                  tests, column N the residual/bonus sample; values in
 *                  [0,1); may be NULL when greedy != 0
 *   temperature    device float [B]; T <= 0 makes that sequence greedy;
 *                  may be NULL when greedy != 0
 *   greedy         nonzero: every sequence is greedy
 *   out_tokens     device int32 [B, N+1]: emitted tokens, unused slots -1
 *   num_accepted   device int32 [B]: accepted drafts, 0..N
 * A sequence whose inputs are invalid (a draft token outside [0,V), a row
 * the method reads with a NaN or +inf logit or with only -inf logits, a NaN,
 * +inf or subnormal positive temperature) gets out_tokens = -1 in every slot
 * and num_accepted = -1, and sets a sticky device status that
 * spec_verify_get_status reports.  Host-side errors return a code and
 * enqueue nothing.  B == 0 enqueues nothing and returns SV_OK.
 */
sv_status spec_verify_run(spec_verify_ctx *ctx, const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *uniforms,
                          const float *temperature, int greedy, int B, int N,
                          int32_t *out_tokens, int32_t *num_accepted, void *stream);

/*
 * Same as spec_verify_run, and also writes, for every position, the
 * quantities the decisions were made from (any of these may be NULL):
 *   q_at_draft        float [B, N]: q_i(d_i), evaluated in double from the
 *                     row statistics (a check of the normalisers)
 *   p_at_draft        float [B, N]: p_i(d_i), likewise
 *   target_row_stats  float [B, N+1, 2]: (max_k z, sum_k exp((z_k - max)/T))
 *   draft_row_stats   float [B, N, 2]:   the same for the draft rows
 *   ratio_at_draft    float [B, N]: the ratio q_i(d_i)/p_i(d_i) that the
 *                     accept test of position i compared u[b,i] with (the
 *                     test is u < min(1, ratio)), rounded to float; +inf
 *                     where p_i(d_i) == 0
 * Greedy and invalid sequences report (max, NaN) and NaN probabilities and
 * ratios.
 */
sv_status spec_verify_run_debug(spec_verify_ctx *ctx, const void *target_logits,
                                const void *draft_logits, const int32_t *draft_tokens,
                                const float *uniforms, const float *temperature, int greedy,
                                int B, int N, int32_t *out_tokens, int32_t *num_accepted,
                                void *stream, float *q_at_draft, float *p_at_draft,
                                float *target_row_stats, float *draft_row_stats,
                                float *ratio_at_draft);

/*
 * Synchronise the device, read and clear the sticky device status of this
 * context: SV_OK, or the first of SV_ERR_TIMEOUT, SV_ERR_BAD_TOKEN,
 * SV_ERR_BAD_VALUE raised by a run since the last call.  SV_ERR_CUDA if the
 * read fails.
 */
sv_status spec_verify_get_status(spec_verify_ctx *ctx);

/*
 * Tree verification: B candidate trees of M+1 nodes each, node 0 being the
 * committed context (the pages name candidate trees: "Speculative decoding --
 * draft, verify, repeat", sections on Medusa, with its tree attention, and on
 * EAGLE, with EAGLE-2's dynamic draft trees; they state no rule for a node
 * with several candidates, so this follows the plainest one that keeps the
 * output distributed as the verifier's: the children of a node are taken to
 * be independent draws from the draft distribution at that node and are tried
 * in index order, each rejection replacing the current verifier distribution
 * by the normalised residual max(0, r - p) / sum max(0, r - p); an accepted
 * child becomes the current node; when no child passes, the token is drawn
 * from the last residual (from q of the node at a leaf).  A tree whose nodes
 * form one chain gives exactly spec_verify_run's result.
 *
 * Arguments (device memory, caller-owned, contiguous; per sequence b, node n):
 *   target_logits [B, M+1, V]  verifier logits after node n's path
 *   draft_logits  [B, M+1, V]  draft logits at node n (the distribution its
 *                              children were drawn from); rows of leaves are
 *                              not read; may be NULL when greedy or M == 0
 *   parent        int32 [B, M+1]  parent[b][0] = -1, 0 <= parent[b][n] < n
 *   draft_tokens  int32 [B, M+1]  the token of node n (entry 0 unused)
 *   uniforms      float [B, M+1]  entry n >= 1: the accept test of node n;
 *                                 entry 0: the final sample
 *   temperature   float [B]; T <= 0 (or greedy != 0) selects greedy: accept
 *                 the first child whose token is the verifier's argmax
 *                 (lowest index on ties), emit the argmax where none is
 *   out_tokens    int32 [B, M+1]  the accepted path's tokens, then the drawn
 *                                 token, then -1
 *   path_nodes    int32 [B, M+1]  the accepted path's node ids, then -1
 *   num_accepted  int32 [B]       path length (-1 for an invalid sequence)
 *   target_row_stats, draft_row_stats  float [B, M+1, 2] (m, S) per node, or
 *                 NULL; written for every node (draft: nodes with children)
 *   ratio_at_node float [B, M+1] or NULL: for every child the walk tested,
 *                 the ratio r(x)/p(x) its uniform was compared with (r the
 *                 verifier distribution or residual at that point, x its
 *                 token; +inf where p(x) == 0), NaN for nodes not tested
 * Requires B <= max_B, M <= max_N of the context, M + 1 <= 1024 and
 * V*elt <= 2 MiB.  Invalid sequences (a bad token, a bad parent array, a row
 * with NaN/+inf or only -inf among those read, a bad temperature) emit -1
 * everywhere and set the context's status (SV_ERR_BAD_TREE for the parent
 * array).  Two launches on `stream`; nothing is allocated.  The acceptance
 * counters count path lengths.
 */
sv_status spec_verify_tree_run(spec_verify_ctx *ctx, const void *target_logits, const void *draft_logits,
                               const int32_t *parent, const int32_t *draft_tokens, const float *uniforms,
                               const float *temperature, int greedy, int B, int M, int32_t *out_tokens,
                               int32_t *path_nodes, int32_t *num_accepted, float *target_row_stats,
                               float *draft_row_stats, float *ratio_at_node, void *stream);

/*
 * The LM-head product on the tensor cores: logits[r][v] = sum_k hidden[r][k] *
 * weight[v][k], bf16 inputs, f32 accumulation ("Speculative decoding -- draft,
 * verify, repeat", section "Core algorithm": the verifier's forward ends in
 * this product; so does the draft's).  hidden: device [M, K] bf16 row-major,
 * weight: device [V, K] bf16 row-major (each row a vocabulary entry), logits:
 * device [M, V] f32.  K must be a multiple of 8 and both inputs 16-byte
 * aligned, else SV_ERR_INVALID_ARG; SV_ERR_CUDA if the TMA descriptors cannot
 * be built or the launch fails.  Asynchronous on `stream`, current device.
 */
sv_status spec_verify_lm_head_logits(const void *hidden, const void *weight, int M, int V, int K, float *logits,
                                     void *stream);

/*
 * The verify step fused into the LM-head products: the inputs are the final
 * hidden states and the LM-head weights of both models instead of logits
 * (the verifier's forward and the draft's both end in this product: "Speculative
 * decoding -- draft, verify, repeat", section "Core algorithm").  The logits
 * are computed on the tensor cores and reduced in the product's epilogue to
 * the row statistics the method needs (max, sum of exp((z - max)/T), or the
 * argmax for greedy sequences, and the logit at each draft token), so no pass
 * over the logits reads them back.  To draw the token, the row pair at each
 * sampled sequence's first rejection is needed: by default the verifier
 * product's epilogue also writes every verifier row's float32 logits into the
 * context's scratch, the draw reads back only the rows it needs, and the
 * draft row is recomputed on the tensor cores (a second read of the draft
 * head); with spec_verify_set_fused_logits(ctx, 0) no logits reach HBM and
 * both rows are recomputed (a second read of both heads).  The result equals
 * spec_verify_run on the float32 logits hidden @ weight^T.
 *
 *   target_hidden [B*(N+1), Kt] bf16, row b*(N+1)+i for position i
 *   target_weight [V, Kt] bf16 (row v: vocabulary entry v)
 *   draft_hidden  [B*N, Kd] bf16, draft_weight [V, Kd] bf16 (NULL when greedy)
 *   the other arguments as spec_verify_run; target_row_stats [B, N+1, 2] and
 *   draft_row_stats [B, N, 2] (m, S) and ratio_at_draft [B, N] (the ratio
 *   each accept test compared its uniform with, as in spec_verify_run_debug)
 *   may be NULL.
 * Requires a context created with SV_F32 (SV_ERR_DTYPE otherwise; its V is the
 * vocabulary size), Kt and Kd multiples of 8, 16-byte aligned inputs.  The
 * first call (and a call with larger Kt or Kd, or after the mode changed)
 * allocates its scratch and therefore synchronises: about
 * 8*(2*max_N+1)*max_B*ceil(V/256) bytes of tile statistics, 4*max_B*V +
 * 2*max_B*Kd bytes for the draft rows' recomputation, plus
 * 4*(max_N+1)*max_B*V bytes of kept verifier logits, or 4*max_B*V +
 * 2*max_B*Kt bytes when the verifier rows are recomputed too.  Later calls
 * enqueue seven launches on `stream` when the verifier logits are kept (four
 * when greedy: no draft product), eight when they are recomputed (six when
 * greedy), and allocate nothing.
 */
sv_status spec_verify_run_fused(spec_verify_ctx *ctx, const void *target_hidden, const void *target_weight,
                                int Kt, const void *draft_hidden, const void *draft_weight, int Kd,
                                const int32_t *draft_tokens, const float *uniforms, const float *temperature,
                                int greedy, int B, int N, int32_t *out_tokens, int32_t *num_accepted,
                                float *target_row_stats, float *draft_row_stats, float *ratio_at_draft,
                                void *stream);

/*
 * The fused path's handling of the verifier logits (spec_verify_run_fused):
 * keep != 0 (the default) writes every verifier row's float32 logits from the
 * statistics epilogue and reads back the rows it samples from; keep == 0
 * keeps them out of HBM and recomputes the sampled rows (the draft rows are
 * recomputed either way).  Takes effect at the next fused call, which then
 * reallocates the scratch.  SV_ERR_INVALID_ARG for a null context.
 */
sv_status spec_verify_set_fused_logits(spec_verify_ctx *ctx, int keep);

/*
 * Acceptance telemetry (how many drafts each verify accepted, the quantity
 * the pages tell users to watch: mean accepted length and acceptance rate).
 * Every run adds each sequence to counts[k], k = its num_accepted (0..N), or
 * to counts[max_N + 1] when it was invalid.  Copies the max_N + 2 counters
 * into `counts` (ncounts >= max_N + 2; further entries are zeroed), after
 * synchronising the device; reset != 0 then clears them.
 */
sv_status spec_verify_acceptance_counts(spec_verify_ctx *ctx, uint64_t *counts, int ncounts, int reset);

/*
 * Cluster size used by the next runs: the number of CTAs (1..16) that share
 * one verified position in the normalising pass; 0 restores the automatic
 * choice (the sampling pass always chooses its own).  Returns
 * SV_ERR_INVALID_ARG for a size the device cannot co-schedule.
 */
sv_status spec_verify_set_cluster_size(spec_verify_ctx *ctx, int cluster_size);

/* The cluster size the next run will use for B sequences of N drafts. */
int spec_verify_cluster_size(spec_verify_ctx *ctx, int B, int N);

/* Static string naming a status code. */
const char *spec_verify_error_string(sv_status s);

/*
 * Kernel timing for benchmarks.  While enabled, every run records CUDA events
 * before its first kernel (row normalisers and accept tests), after it, and
 * after the last (sampling and output), up to 4096 runs; enabling again
 * restarts the count.  The sampling kernels then start only after the first
 * kernel has finished.  spec_verify_profile_read waits for the recorded runs
 * and returns the summed device time of the two parts in milliseconds and the
 * number of runs.  Disabling frees the events.
 */
sv_status spec_verify_profile(spec_verify_ctx *ctx, int enable);
sv_status spec_verify_profile_read(spec_verify_ctx *ctx, double *ms_rows, double *ms_sample, int *runs);

/*
 * Self-test of the library's failure detection (the pages have no
 * counterpart).  Every wait inside the kernels is bounded: it gives up after
 * a time limit (2 s in the verify kernels), reports SV_ERR_TIMEOUT through the
 * status word, lets its copies in flight land and returns, so a stalled
 * producer never hangs the GPU.  This call launches one block whose barrier
 * wait nothing ever satisfies, with a limit of limit_us microseconds
 * (1 .. 10^7), synchronises `stream` and sets *gave_up = 1 if the block gave
 * up and reported it, 0 otherwise.  Returns SV_ERR_INVALID_ARG for a bad
 * limit or a NULL gave_up, SV_ERR_CUDA if the launch or copies fail.
 */
sv_status spec_verify_selftest_timeout(int limit_us, int *gave_up, void *stream);

/* Free the workspace and the context.  NULL is ignored. */
void spec_verify_destroy(spec_verify_ctx *ctx);

/*
 * Allocation-free variant of spec_verify_run (the pages have no counterpart:
 * this is a deployment convenience, not part of the method).
 *
 * Some callers must not allocate device memory once they are running: an
 * inference engine that reserved all free memory for its KV cache at start-up,
 * a plug-in whose host framework owns every allocation, or a decode loop that
 * cannot afford the implicit device synchronisation and possible failure of a
 * cudaMalloc.  This entry point needs no context and allocates nothing: its
 * scratch is a fixed array of about 1.45 MiB compiled into the library, which
 * every GPU that loads the library holds until the process exits.
 *
 * Arguments are those of spec_verify_run, with the vocabulary size V and the
 * logit dtype given per call; it runs on the current device.  Limits: B <= 2048,
 * B*(N+1) <= 16384 and B*ceil(V*elt/4 KiB) <= 32768 (so 256 sequences of
 * N = 7 drafts over a 151936-token bf16 vocabulary fit, and 1024 sequences of
 * 128256 float32 logits do not), else SV_ERR_TOO_LARGE and nothing is
 * enqueued.
 * Invalid sequences are reported through out_tokens = -1 and
 * num_accepted = -1 only (there is no status word to query).
 *
 * The first call on a device does a one-time, synchronous set-up (it looks up
 * the scratch address, clears it and sets kernel attributes); make that first
 * call before any stream capture.  Every later call enqueues three small
 * memsets of the scratch slots it uses and the three kernels, on `stream`, and
 * nothing else.  All calls on a device share the one scratch array: calls
 * that can overlap on the GPU (different streams without ordering between
 * them, or several host threads) race and corrupt each other's results.
 */
sv_status spec_verify_run_noalloc(const void *target_logits, const void *draft_logits,
                                  const int32_t *draft_tokens, const float *uniforms,
                                  const float *temperature, int greedy, int B, int N, int V,
                                  sv_dtype dtype, int32_t *out_tokens, int32_t *num_accepted,
                                  void *stream);

/*
 * KV-cache commit and rollback after a verify step: "Speculative decoding --
 * draft, verify, repeat" (factory.pai-world.com, lesson 07-16), section "KV
 * cache dance" and its exercise 4.  The verifier's forward over the N drafts
 * wrote their KV entries to a scratch buffer; this appends each sequence's
 * first num_accepted[b] entries to its cache and advances cache_len[b], so
 * the next iteration reads the prefix plus the accepted drafts.  The rejected
 * entries are never copied (the rollback).
 *
 * Layout (device memory, caller-owned, byte rows of any content):
 *   scratch   [planes][B][N][row_bytes]        may be NULL when N == 0
 *   cache     [planes][B][max_len][row_bytes]  rows cache_len[b] .. + a - 1 written
 *   cache_len int32 [B], read and advanced in place
 *   num_accepted int32 [B], as written by spec_verify_run (-1 = invalid sequence)
 * A plane is any slab that shares the sequence's length, e.g. the K or the V
 * half of one layer; row_bytes is one token's entry in one plane.
 *
 * Per sequence: num_accepted < 0 commits nothing; num_accepted > N commits
 * nothing and sets SV_KV_BAD_COUNT; cache_len < 0 or cache_len + num_accepted
 * > max_len commits nothing and sets SV_KV_OVERFLOW.  The bits are OR-ed into
 * *status (device int32, may be NULL); the caller clears it.
 *
 * Host errors: SV_ERR_INVALID_ARG for negative sizes, planes < 1,
 * row_bytes == 0 or not a multiple of 16, a NULL pointer that is needed, or
 * scratch / cache not 16-byte aligned; SV_ERR_TOO_LARGE when the byte offsets
 * would pass 2^62; SV_ERR_CUDA when a launch fails.  Asynchronous on
 * `stream` (cudaStream_t, NULL = legacy default stream), on the current
 * device; allocates nothing; two kernel launches (one when N == 0), ordered
 * after the work already on the stream.
 */
enum {
    SV_KV_OVERFLOW = 1,   /* cache_len + num_accepted > max_len, or cache_len < 0 */
    SV_KV_BAD_COUNT = 2   /* num_accepted > N */
};

sv_status spec_verify_kv_commit(const void *scratch, void *cache, int32_t *cache_len,
                                const int32_t *num_accepted, int32_t *status, int planes, int B,
                                int N, int max_len, size_t row_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */

/*
 * sv_oracle.c -- float64 CPU oracle of the speculative-sampling verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * CUDA path is checked against.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference legs may load it.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes (per sequence b), following
 *   "Speculative decoding -- draft, verify, repeat" (factory.pai-world.com,
 *    lesson 07-16), section "Core algorithm", steps 2-6, and its build
 *    section, Step 1 (rejection step), Step 2 (residual distribution) and
 *    Step 3 (one speculative step):
 *
 *   q_i = softmax(zq[b,i,:] / T)   verifier distribution, i = 0..N
 *   p_i = softmax(zp[b,i,:] / T)   draft distribution,    i = 0..N-1
 *   for i = 0..N-1 (left to right):
 *       accept d_i  iff  p_i(d_i) == 0  or  u[b,i] < min(1, q_i(d_i)/p_i(d_i))
 *   first rejection at j: sample t from normalise(max(0, q_j - p_j))
 *   no rejection (j = N):  sample the bonus token t from q_N
 *   emit d_0..d_{j-1}, t ;  num_accepted = j
 *
 * Readings taken where the pages are silent (none of the four pages fixes
 * these points; each is the plainest form the rest of the pages support):
 *   - softmax is evaluated in its max-subtracted form, with plain
 *     left-to-right summation in double;
 *   - temperature divides both the target and the draft logits;
 *   - the comparison is strict (u < ratio), and p_i(d_i) == 0 accepts
 *     (the rejection-step listing maps a zero draft probability to an
 *     infinite ratio);
 *   - `sample` is the inverse CDF in ascending token order against one
 *     uniform u[b,N]: t = smallest k with u*R < C_k, C_k = r_0+...+r_k,
 *     R = C_{V-1}; if rounding leaves no such k, t = largest k with r_k > 0;
 *   - a residual of total mass 0 (q_j == p_j) samples from q_j instead;
 *   - greedy sequences (greedy flag, or T <= 0): a_i = argmax_k zq[b,i,k]
 *     with the lowest index on ties; accept d_i iff d_i == a_i; emit a_j at
 *     the first mismatch, else the bonus a_N;
 *   - a row is invalid if it holds a NaN or +inf logit or only -inf logits;
 *     a temperature that is NaN, +inf or in (0, FLT_MIN) is invalid; a draft
 *     token outside [0, V) is invalid.  An invalid sequence emits -1 in every
 *     slot and num_accepted = -1.  Every row the method reads is checked:
 *     all 2N+1 rows of a sampled sequence, the N+1 target rows of a greedy
 *     one.
 *
 * Decision margins (reported so that tests can tell rounding-sensitive
 * decisions apart): for an accept test the margin is |u_i - ratio|, the
 * distance the ratio would have to move to change the decision (below 1 the
 * threshold is the ratio itself; at or above 1 the threshold is 1 and the
 * decision changes only once the ratio falls to u_i, which is ratio - u_i
 * away); a zero draft probability accepts with margin +inf.  For the final
 * sample it is the distance from u[b,N] to the nearer edge of the chosen
 * token's CDF interval, min(|u - C_{t-1}/R|, |u - C_t/R|).  Greedy decisions
 * have margin +inf.  The ratio q_i(d_i)/p_i(d_i) itself is reported too
 * (+inf where p_i(d_i) == 0).
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F64 2

#define ORC_SEQ_BAD_TOKEN 1
#define ORC_SEQ_BAD_VALUE 2

/* One logit, upcast exactly to double.  bf16 is the top half of an IEEE
 * binary32 word, so shifting its 16 bits up by 16 gives the same value. */
static double orc_logit(const void *base, int dtype, size_t idx)
{
    if (dtype == ORC_F64)
        return ((const double *)base)[idx];
    if (dtype == ORC_F32)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Row validity as defined above: no NaN, no +inf, at least one finite value
 * (a row of only -inf has no distribution). */
static int orc_row_valid(const void *base, int dtype, size_t off, int V)
{
    int any_finite = 0;
    for (int k = 0; k < V; k++) {
        double z = orc_logit(base, dtype, off + (size_t)k);
        if (isnan(z) || z == INFINITY)
            return 0;
        if (z != -INFINITY)
            any_finite = 1;
    }
    return any_finite;
}

/* Normaliser of softmax(z / T): m = max_k z_k and S = sum_k exp((z_k - m)/T),
 * summed left to right.  Then softmax(z/T)_k = exp((z_k - m)/T) / S. */
static void orc_row_normaliser(const void *base, int dtype, size_t off, int V,
                               double T, double *m_out, double *S_out)
{
    double m = -INFINITY;
    for (int k = 0; k < V; k++) {
        double z = orc_logit(base, dtype, off + (size_t)k);
        if (z > m)
            m = z;
    }
    double S = 0.0;
    for (int k = 0; k < V; k++) {
        double z = orc_logit(base, dtype, off + (size_t)k);
        S += exp((z - m) / T);
    }
    *m_out = m;
    *S_out = S;
}

static double orc_prob(double z, double m, double S, double T)
{
    return exp((z - m) / T) / S;
}

/* argmax with the lowest index on ties, compared on the stored values. */
static int orc_argmax(const void *base, int dtype, size_t off, int V)
{
    int best = 0;
    double best_z = orc_logit(base, dtype, off);
    for (int k = 1; k < V; k++) {
        double z = orc_logit(base, dtype, off + (size_t)k);
        if (z > best_z) {
            best_z = z;
            best = k;
        }
    }
    return best;
}

/* Inverse CDF of the (unnormalised) mass r[0..V-1] against u in [0,1):
 * t = smallest k with u*R < C_k where C_k = r_0 + ... + r_k, R = C_{V-1}.
 * Writes the margin min(|u - C_{t-1}/R|, |u - C_t/R|). */
static int orc_inverse_cdf(const double *r, int V, double u, double *margin)
{
    double R = 0.0;
    for (int k = 0; k < V; k++)
        R += r[k];
    double x = u * R;
    double C_prev = 0.0, C = 0.0;
    int t = -1;
    for (int k = 0; k < V; k++) {
        C_prev = C;
        C += r[k];
        if (x < C) {
            t = k;
            break;
        }
    }
    if (t < 0) {
        /* rounding left u*R at or above the last cumulative value: take the
         * last token that carries mass, and report the distance to 1. */
        for (int k = V - 1; k >= 0; k--) {
            if (r[k] > 0.0) {
                t = k;
                break;
            }
        }
        if (t < 0)
            t = V - 1; /* all-zero mass: cannot happen for a valid row */
        *margin = fabs(u - 1.0);
        return t;
    }
    double lo = fabs(u - C_prev / R), hi = fabs(u - C / R);
    *margin = lo < hi ? lo : hi;
    return t;
}

typedef struct {
    const void *target;          /* [B, N+1, V] */
    const void *draft;           /* [B, N, V], may be NULL when greedy != 0 */
    int dtype;
    const int32_t *draft_tokens; /* [B, N] */
    const double *u;             /* [B, N+1]: 0..N-1 accept tests, N sample */
    const double *T;             /* [B], may be NULL when greedy != 0 */
    int greedy;
    int B, N, V;
    int32_t *out_tokens;   /* [B, N+1] */
    int32_t *num_accepted; /* [B] */
    /* optional diagnostics (NULL to skip) */
    double *q_at_d;        /* [B, N]   q_i(d_i) */
    double *p_at_d;        /* [B, N]   p_i(d_i) */
    double *tstats;        /* [B, N+1, 2]  (m, S) of target rows */
    double *dstats;        /* [B, N, 2]    (m, S) of draft rows */
    double *accept_margin; /* [B, N]   NaN where not evaluated */
    double *sample_margin; /* [B] */
    int32_t *seq_status;   /* [B]  0, or ORC_SEQ_* bits */
    double *ratio_at_d;    /* [B, N]   q_i(d_i)/p_i(d_i) of every test made, NaN elsewhere */
} orc_args;

static void orc_fill_invalid(const orc_args *a, int b)
{
    for (int i = 0; i <= a->N; i++)
        a->out_tokens[(size_t)b * (a->N + 1) + i] = -1;
    a->num_accepted[b] = -1;
}

static void orc_verify_sequence(const orc_args *a, int b, double *r)
{
    const int N = a->N, V = a->V;
    const size_t trow0 = (size_t)b * (N + 1); /* first target row of b */
    const size_t drow0 = (size_t)b * N;       /* first draft row of b  */
    int status = 0;

    if (a->accept_margin)
        for (int i = 0; i < N; i++)
            a->accept_margin[drow0 + i] = NAN;
    if (a->ratio_at_d)
        for (int i = 0; i < N; i++)
            a->ratio_at_d[drow0 + i] = NAN;
    if (a->sample_margin)
        a->sample_margin[b] = NAN;

    for (int i = 0; i < N; i++) {
        int32_t d = a->draft_tokens[drow0 + i];
        if (d < 0 || d >= V)
            status |= ORC_SEQ_BAD_TOKEN;
    }

    int greedy = a->greedy != 0;
    double T = 0.0;
    if (!greedy) {
        T = a->T[b];
        if (isnan(T))
            status |= ORC_SEQ_BAD_VALUE;
        else if (T <= 0.0)
            greedy = 1;
        else if (T == INFINITY || T < (double)FLT_MIN)
            status |= ORC_SEQ_BAD_VALUE;
    }

    for (int i = 0; i <= N; i++)
        if (!orc_row_valid(a->target, a->dtype, (trow0 + i) * (size_t)V, V))
            status |= ORC_SEQ_BAD_VALUE;
    if (!greedy)
        for (int i = 0; i < N; i++)
            if (!orc_row_valid(a->draft, a->dtype, (drow0 + i) * (size_t)V, V))
                status |= ORC_SEQ_BAD_VALUE;

    if (a->seq_status)
        a->seq_status[b] = status;
    if (status) {
        orc_fill_invalid(a, b);
        return;
    }

    int32_t *out = a->out_tokens + trow0;
    for (int i = 0; i <= N; i++)
        out[i] = -1;

    if (greedy) {
        int j = N;
        for (int i = 0; i < N; i++) {
            int ai = orc_argmax(a->target, a->dtype, (trow0 + i) * (size_t)V, V);
            if (a->draft_tokens[drow0 + i] != ai) {
                j = i;
                out[i] = ai;
                break;
            }
            out[i] = a->draft_tokens[drow0 + i];
            if (a->accept_margin)
                a->accept_margin[drow0 + i] = INFINITY;
        }
        if (j < N && a->accept_margin)
            a->accept_margin[drow0 + j] = INFINITY;
        if (j == N)
            out[N] = orc_argmax(a->target, a->dtype, (trow0 + N) * (size_t)V, V);
        a->num_accepted[b] = j;
        if (a->sample_margin)
            a->sample_margin[b] = INFINITY;
        return;
    }

    /* Normalisers of every row the method reads. */
    double *mq = (double *)malloc(sizeof(double) * 2 * (size_t)(N + 1));
    double *Sq = mq + (N + 1);
    double *mp = (double *)malloc(sizeof(double) * 2 * (size_t)(N + 1));
    double *Sp = mp + (N + 1);
    for (int i = 0; i <= N; i++) {
        orc_row_normaliser(a->target, a->dtype, (trow0 + i) * (size_t)V, V, T, &mq[i], &Sq[i]);
        if (a->tstats) {
            a->tstats[(trow0 + i) * 2 + 0] = mq[i];
            a->tstats[(trow0 + i) * 2 + 1] = Sq[i];
        }
    }
    for (int i = 0; i < N; i++) {
        orc_row_normaliser(a->draft, a->dtype, (drow0 + i) * (size_t)V, V, T, &mp[i], &Sp[i]);
        if (a->dstats) {
            a->dstats[(drow0 + i) * 2 + 0] = mp[i];
            a->dstats[(drow0 + i) * 2 + 1] = Sp[i];
        }
    }

    /* q_i(d_i) and p_i(d_i) at every draft position. */
    for (int i = 0; i < N; i++) {
        int32_t d = a->draft_tokens[drow0 + i];
        double qd = orc_prob(orc_logit(a->target, a->dtype, (trow0 + i) * (size_t)V + d), mq[i], Sq[i], T);
        double pd = orc_prob(orc_logit(a->draft, a->dtype, (drow0 + i) * (size_t)V + d), mp[i], Sp[i], T);
        if (a->q_at_d)
            a->q_at_d[drow0 + i] = qd;
        if (a->p_at_d)
            a->p_at_d[drow0 + i] = pd;
    }

    /* Left-to-right accept scan; stop at the first rejection j. */
    int j = N;
    for (int i = 0; i < N; i++) {
        int32_t d = a->draft_tokens[drow0 + i];
        double qd = orc_prob(orc_logit(a->target, a->dtype, (trow0 + i) * (size_t)V + d), mq[i], Sq[i], T);
        double pd = orc_prob(orc_logit(a->draft, a->dtype, (drow0 + i) * (size_t)V + d), mp[i], Sp[i], T);
        double ui = a->u[trow0 + i];
        int accept;
        double margin = INFINITY, ratio = INFINITY;
        if (pd == 0.0) {
            accept = 1;
        } else {
            ratio = qd / pd;
            double thresh = ratio < 1.0 ? ratio : 1.0;
            accept = ui < thresh;
            margin = fabs(ui - ratio);
        }
        if (a->accept_margin)
            a->accept_margin[drow0 + i] = margin;
        if (a->ratio_at_d)
            a->ratio_at_d[drow0 + i] = ratio;
        if (!accept) {
            j = i;
            break;
        }
        out[i] = d;
    }

    /* Mass to sample from: the residual (q_j - p_j)_+ at a rejection, q_N
     * for the bonus token. */
    if (j < N) {
        size_t toff = (trow0 + j) * (size_t)V, doff = (drow0 + j) * (size_t)V;
        double R = 0.0;
        for (int k = 0; k < V; k++) {
            double qk = orc_prob(orc_logit(a->target, a->dtype, toff + k), mq[j], Sq[j], T);
            double pk = orc_prob(orc_logit(a->draft, a->dtype, doff + k), mp[j], Sp[j], T);
            double diff = qk - pk;
            r[k] = diff > 0.0 ? diff : 0.0;
            R += r[k];
        }
        if (R == 0.0) /* q_j == p_j: the rejection had probability 0 */
            for (int k = 0; k < V; k++)
                r[k] = orc_prob(orc_logit(a->target, a->dtype, toff + k), mq[j], Sq[j], T);
    } else {
        size_t toff = (trow0 + N) * (size_t)V;
        for (int k = 0; k < V; k++)
            r[k] = orc_prob(orc_logit(a->target, a->dtype, toff + k), mq[N], Sq[N], T);
    }
    double smargin;
    out[j] = orc_inverse_cdf(r, V, a->u[trow0 + N], &smargin);
    if (a->sample_margin)
        a->sample_margin[b] = smargin;
    a->num_accepted[b] = j;

    free(mq);
    free(mp);
}

typedef struct {
    const orc_args *a;
    int b0, b1;
} orc_range;

static void *orc_worker(void *arg)
{
    orc_range *rg = (orc_range *)arg;
    double *r = (double *)malloc(sizeof(double) * (size_t)rg->a->V);
    for (int b = rg->b0; b < rg->b1; b++)
        orc_verify_sequence(rg->a, b, r);
    free(r);
    return NULL;
}

/*
 * Batched entry point.  Returns 0, or -1 on a bad argument.  nthreads <= 1
 * runs on the calling thread; otherwise sequences are split into nthreads
 * contiguous ranges, one POSIX thread each.
 */
int orc_verify(const void *target, const void *draft, int dtype,
               const int32_t *draft_tokens, const double *u, const double *T,
               int greedy, int B, int N, int V,
               int32_t *out_tokens, int32_t *num_accepted,
               double *q_at_d, double *p_at_d, double *tstats, double *dstats,
               double *accept_margin, double *sample_margin,
               int32_t *seq_status, double *ratio_at_d, int nthreads)
{
    if (B < 0 || N < 0 || V < 1 || !target || !out_tokens || !num_accepted || !u)
        return -1;
    if (N > 0 && !draft_tokens)
        return -1;
    if (!greedy && (!T || (N > 0 && !draft)))
        return -1;
    if (dtype != ORC_F32 && dtype != ORC_BF16 && dtype != ORC_F64)
        return -1;
    orc_args a = {target, draft, dtype, draft_tokens, u, T, greedy, B, N, V,
                  out_tokens, num_accepted, q_at_d, p_at_d, tstats, dstats,
                  accept_margin, sample_margin, seq_status, ratio_at_d};
    if (nthreads <= 1 || B <= 1) {
        orc_range rg = {&a, 0, B};
        orc_worker(&rg);
        return 0;
    }
    if (nthreads > B)
        nthreads = B;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    orc_range *rg = (orc_range *)malloc(sizeof(orc_range) * (size_t)nthreads);
    for (int t = 0; t < nthreads; t++) {
        rg[t].a = &a;
        rg[t].b0 = (int)((long long)B * t / nthreads);
        rg[t].b1 = (int)((long long)B * (t + 1) / nthreads);
        pthread_create(&th[t], NULL, orc_worker, &rg[t]);
    }
    for (int t = 0; t < nthreads; t++)
        pthread_join(th[t], NULL);
    free(th);
    free(rg);
    return 0;
}

/* Softmax(z/T) of one row, for the tests that pin the normaliser against a
 * library routine. */
int orc_softmax_row(const void *row, int dtype, int V, double T, double *probs,
                    double *m_out, double *S_out)
{
    if (V < 1 || T <= 0.0)
        return -1;
    double m, S;
    orc_row_normaliser(row, dtype, 0, V, T, &m, &S);
    for (int k = 0; k < V; k++)
        probs[k] = orc_prob(orc_logit(row, dtype, (size_t)k), m, S, T);
    *m_out = m;
    *S_out = S;
    return 0;
}

/*
 * KV-cache commit after a verify step, following the same lesson's section
 * "KV cache dance": the verifier's forward over the N drafts writes their N
 * KV entries into a scratch buffer; once the verify step has fixed how many
 * drafts were accepted, the first num_accepted of those entries are appended
 * to the cache and the rest are dropped (the rollback).  Exercise 4 of the
 * lesson states the check: a 10-token prefix, 5 drafts, a rejection at the
 * third draft, and the cache then reads prefix + the first 2 drafts.
 *
 * Layout (bytes, row-major): scratch [P][B][N][row_bytes], cache
 * [P][B][max_len][row_bytes]; P planes (for example K and V of every layer)
 * share one length per sequence, cache_len[b].  Per sequence b:
 *   a = num_accepted[b]
 *   a < 0 (an invalid verify):          nothing is committed
 *   a > N:                              nothing; status |= 2
 *   cache_len[b] < 0 or
 *   cache_len[b] + a > max_len:         nothing; status |= 1
 *   otherwise, for every plane p and k < a:
 *       cache[p][b][cache_len[b] + k] = scratch[p][b][k];  cache_len[b] += a
 * Returns the status bits.
 */
int orc_kv_commit(const unsigned char *scratch, unsigned char *cache, int32_t *cache_len,
                  const int32_t *num_accepted, int P, int B, int N, int max_len,
                  size_t row_bytes)
{
    int status = 0;
    for (int b = 0; b < B; ++b) {
        const int a = num_accepted[b];
        if (a < 0)
            continue;
        if (a > N) {
            status |= 2;
            continue;
        }
        const int len = cache_len[b];
        if (len < 0 || (long long)len + a > max_len) {
            status |= 1;
            continue;
        }
        for (int p = 0; p < P; ++p)
            for (int k = 0; k < a; ++k) {
                const size_t src = (((size_t)p * B + b) * N + k) * row_bytes;
                const size_t dst = (((size_t)p * B + b) * max_len + len + k) * row_bytes;
                memcpy(cache + dst, scratch + src, row_bytes);
            }
        cache_len[b] = len + a;
    }
    return status;
}

/*
 * Tree verification.  The pages name candidate trees (the lesson's "Medusa"
 * section: candidates from every head verified in one forward with tree
 * attention; its "EAGLE" section and the reading list: EAGLE-2's dynamic draft
 * trees) and require that the output keep the verifier's distribution
 * ("A friend writes first and the teacher grades", section "The guarantee that
 * the answer does not change"), but give no rule for a node with several
 * candidates.  The plainest rule that keeps the guarantee, taken here: the
 * children of a node are independent draws from the draft distribution at
 * that node, and they are tried in ascending node order with the same accept
 * test, each rejection replacing the current verifier distribution by the
 * normalised residual (current - draft)+; an accepted child becomes the new
 * node; when every child is rejected, the token is drawn from the last
 * residual; a leaf draws the bonus token from its verifier distribution.
 * A tree whose nodes form one chain is exactly the chain verify above.
 *
 * Per sequence b, nodes n = 0..M (node 0 = the committed context):
 *   parent[b][n]: -1 for n = 0, in [0, n) otherwise (siblings in index order)
 *   tokens[b][n]: the draft token of node n (n >= 1)
 *   target row n: logits of the verifier after node n's path, q_n = softmax(./T)
 *   draft row n:  logits of the draft at node n, p_n = softmax(./T), from which
 *                 n's children were drawn (read only for nodes with children)
 *   u[b][n], n >= 1: the accept test of node n;  u[b][0]: the final sample
 * Walk: n = 0, r = q_0.  For each child c of n in order: x = tokens[c];
 *   accept iff p_n(x) == 0 or u[c] < min(1, r(x)/p_n(x)); on accept the path
 *   gains c, n = c, r = q_c and the walk goes on; on reject
 *   r <- (r - p_n)+ / sum (r - p_n)+, or r unchanged if that sum is 0.
 *   No child accepted (or none at all): t = inverse CDF of r at u[b][0].
 * Outputs: out_tokens = the path's tokens then t, -1 after; path_nodes = the
 * path's node ids, -1 after; num_accepted = path length.  Greedy sequences:
 * accept the first child whose token is argmax q_n; emit argmax q_n at the
 * end.  Invalid sequences (as in the chain verify, plus a parent array that
 * breaks the rules above: status bit 4) emit -1 everywhere.
 */
#define ORC_SEQ_BAD_TREE 4

typedef struct {
    const void *target, *draft;
    int dtype;
    const int32_t *parent, *tokens;
    const double *u, *T;
    int greedy, B, M, V;
    int32_t *out_tokens, *path_nodes, *num_accepted;
    double *tstats, *dstats, *accept_margin, *sample_margin;
    int32_t *seq_status;
    double *ratio_at; /* [B, M+1] r(x)/p_n(x) of every child tested, NaN elsewhere */
} orc_tree_args;

static void orc_tree_sequence(const orc_tree_args *a, int b, double *r, double *p)
{
    const int M = a->M, V = a->V;
    const size_t row0 = (size_t)b * (M + 1); /* node n of b is row row0 + n */
    const int32_t *par = a->parent + row0;
    const int32_t *tok = a->tokens + row0;
    int32_t *out = a->out_tokens + row0, *path = a->path_nodes + row0;
    int status = 0;

    for (int n = 0; n <= M; n++) {
        out[n] = -1;
        path[n] = -1;
        if (a->accept_margin)
            a->accept_margin[row0 + n] = NAN;
        if (a->ratio_at)
            a->ratio_at[row0 + n] = NAN;
    }
    if (a->sample_margin)
        a->sample_margin[b] = NAN;

    if (par[0] != -1)
        status |= ORC_SEQ_BAD_TREE;
    for (int n = 1; n <= M; n++) {
        if (par[n] < 0 || par[n] >= n)
            status |= ORC_SEQ_BAD_TREE;
        if (tok[n] < 0 || tok[n] >= V)
            status |= ORC_SEQ_BAD_TOKEN;
    }
    int greedy = a->greedy != 0;
    double T = 0.0;
    if (!greedy) {
        T = a->T[b];
        if (isnan(T))
            status |= ORC_SEQ_BAD_VALUE;
        else if (T <= 0.0)
            greedy = 1;
        else if (T == INFINITY || T < (double)FLT_MIN)
            status |= ORC_SEQ_BAD_VALUE;
    }
    for (int n = 0; n <= M; n++) {
        if (!orc_row_valid(a->target, a->dtype, (row0 + n) * (size_t)V, V))
            status |= ORC_SEQ_BAD_VALUE;
        int has_child = 0;
        for (int c = n + 1; c <= M; c++)
            if (par[c] == n)
                has_child = 1;
        if (!greedy && has_child && !(status & ORC_SEQ_BAD_TREE) &&
            !orc_row_valid(a->draft, a->dtype, (row0 + n) * (size_t)V, V))
            status |= ORC_SEQ_BAD_VALUE;
    }
    if (a->seq_status)
        a->seq_status[b] = status;
    if (status) {
        a->num_accepted[b] = -1;
        return;
    }

    int n = 0, depth = 0;
    if (greedy) {
        for (;;) {
            int an = orc_argmax(a->target, a->dtype, (row0 + n) * (size_t)V, V);
            int next = -1;
            for (int c = n + 1; c <= M && next < 0; c++) {
                if (par[c] != n)
                    continue;
                if (a->accept_margin)
                    a->accept_margin[row0 + c] = INFINITY;
                if (tok[c] == an)
                    next = c;
            }
            if (next < 0) {
                out[depth] = an;
                break;
            }
            out[depth] = tok[next];
            path[depth] = next;
            depth++;
            n = next;
        }
        a->num_accepted[b] = depth;
        if (a->sample_margin)
            a->sample_margin[b] = INFINITY;
        return;
    }

    for (;;) {
        double mq, Sq;
        orc_row_normaliser(a->target, a->dtype, (row0 + n) * (size_t)V, V, T, &mq, &Sq);
        if (a->tstats) {
            a->tstats[(row0 + n) * 2 + 0] = mq;
            a->tstats[(row0 + n) * 2 + 1] = Sq;
        }
        for (int k = 0; k < V; k++)
            r[k] = orc_prob(orc_logit(a->target, a->dtype, (row0 + n) * (size_t)V + k), mq, Sq, T);
        int has_child = 0;
        for (int c = n + 1; c <= M; c++)
            if (par[c] == n)
                has_child = 1;
        if (has_child) {
            double mp, Sp;
            orc_row_normaliser(a->draft, a->dtype, (row0 + n) * (size_t)V, V, T, &mp, &Sp);
            if (a->dstats) {
                a->dstats[(row0 + n) * 2 + 0] = mp;
                a->dstats[(row0 + n) * 2 + 1] = Sp;
            }
            for (int k = 0; k < V; k++)
                p[k] = orc_prob(orc_logit(a->draft, a->dtype, (row0 + n) * (size_t)V + k), mp, Sp, T);
        }
        int next = -1;
        for (int c = n + 1; c <= M && next < 0; c++) {
            if (par[c] != n)
                continue;
            const int x = tok[c];
            int accept;
            double margin = INFINITY, ratio = INFINITY;
            if (p[x] == 0.0) {
                accept = 1;
            } else {
                ratio = r[x] / p[x];
                double thresh = ratio < 1.0 ? ratio : 1.0;
                accept = a->u[row0 + c] < thresh;
                margin = fabs(a->u[row0 + c] - ratio);
            }
            if (a->accept_margin)
                a->accept_margin[row0 + c] = margin;
            if (a->ratio_at)
                a->ratio_at[row0 + c] = ratio;
            if (accept) {
                next = c;
                break;
            }
            /* rejected: the next sibling is tested against the residual */
            double R = 0.0;
            for (int k = 0; k < V; k++) {
                double diff = r[k] - p[k];
                R += diff > 0.0 ? diff : 0.0;
            }
            if (R > 0.0)
                for (int k = 0; k < V; k++) {
                    double diff = r[k] - p[k];
                    r[k] = (diff > 0.0 ? diff : 0.0) / R;
                }
        }
        if (next < 0) {
            double smargin;
            out[depth] = orc_inverse_cdf(r, V, a->u[row0], &smargin);
            if (a->sample_margin)
                a->sample_margin[b] = smargin;
            break;
        }
        out[depth] = tok[next];
        path[depth] = next;
        depth++;
        n = next;
    }
    a->num_accepted[b] = depth;
}

typedef struct {
    const orc_tree_args *a;
    int b0, b1;
} orc_tree_range;

static void *orc_tree_worker(void *arg)
{
    orc_tree_range *rg = (orc_tree_range *)arg;
    double *r = (double *)malloc(sizeof(double) * 2 * (size_t)rg->a->V);
    for (int b = rg->b0; b < rg->b1; b++)
        orc_tree_sequence(rg->a, b, r, r + rg->a->V);
    free(r);
    return NULL;
}

/* Batched tree verification; returns 0, or -1 on a bad argument. */
int orc_tree_verify(const void *target, const void *draft, int dtype, const int32_t *parent,
                    const int32_t *tokens, const double *u, const double *T, int greedy,
                    int B, int M, int V, int32_t *out_tokens, int32_t *path_nodes,
                    int32_t *num_accepted, double *tstats, double *dstats,
                    double *accept_margin, double *sample_margin, int32_t *seq_status,
                    double *ratio_at, int nthreads)
{
    if (B < 0 || M < 0 || V < 1 || !target || !parent || !tokens || !u || !out_tokens ||
        !path_nodes || !num_accepted)
        return -1;
    if (!greedy && (!T || (M > 0 && !draft)))
        return -1;
    if (dtype != ORC_F32 && dtype != ORC_BF16 && dtype != ORC_F64)
        return -1;
    orc_tree_args a = {target, draft, dtype, parent, tokens, u, T, greedy, B, M, V,
                       out_tokens, path_nodes, num_accepted, tstats, dstats,
                       accept_margin, sample_margin, seq_status, ratio_at};
    if (nthreads <= 1 || B <= 1) {
        orc_tree_range rg = {&a, 0, B};
        orc_tree_worker(&rg);
        return 0;
    }
    if (nthreads > B)
        nthreads = B;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    orc_tree_range *rg = (orc_tree_range *)malloc(sizeof(orc_tree_range) * (size_t)nthreads);
    for (int t = 0; t < nthreads; t++) {
        rg[t].a = &a;
        rg[t].b0 = (int)((long long)B * t / nthreads);
        rg[t].b1 = (int)((long long)B * (t + 1) / nthreads);
        pthread_create(&th[t], NULL, orc_tree_worker, &rg[t]);
    }
    for (int t = 0; t < nthreads; t++)
        pthread_join(th[t], NULL);
    free(th);
    free(rg);
    return 0;
}

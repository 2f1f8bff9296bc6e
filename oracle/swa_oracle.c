/*
 * swa_oracle.c -- the oracle for causal sliding-window softmax attention with attention sinks.
 *
 * TEST INFRASTRUCTURE. This is the plain, slow, obviously-correct CPU statement of what the GPU
 * library computes, in fp64. Only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark load it. The GPU library never calls it, links it or includes it, and the two share no
 * code: no headers, no helpers, no tables.
 *
 * What it follows:
 *  - Causal softmax attention, O = softmax(Q K^T / sqrt(D) + M) V with M the causal mask:
 *    page "模糊窗口注意力" (Blurry Window Attention, arXiv 2606.09862), section 2.1, equation (1).
 *  - The sliding-window formula x_t = sum_{i=max(1,t-w+1)}^{t} exp(q_t k_i^T/sqrt d) v_i / sum(...):
 *    page "hyper.ai summary of arXiv 2608.28444" (SWA with sinks vs. linear attention), section
 *    "带 Sink 的滑动窗口注意力", SWA formula.  The window holds w keys, the query's own key included.
 *  - Sinks: the first s = 4 tokens are always attended, in addition to the w - 4 window tokens
 *    (same page and section).  So with m = w - s recent keys, query t (0-indexed) attends
 *        K(t) = { i <= t : i < s  or  i >= t - m + 1 }.
 *  - The softmax normalisation a_ij = exp(q_i.k_j/sqrt d) / sum_l exp(q_i.k_l/sqrt d), sum_j a_ij = 1:
 *    page "滑窗与固定稀疏" (sliding window and fixed sparsity), eq attn-fixed-softmax-sink.
 *  - The streaming cache = sink block KV[0:k] + recent block KV[t-m:t], k + m slots:
 *    page "滑窗与固定稀疏", section "StreamingLLM 怎么用 4 个 sink token 撑住流式生成？",
 *    eq attn-fixed-streaming; rolling buffer cache_slot(i) = i mod W, eq attn-fixed-rolling.
 *
 * Every floating-point step is fp64.  The key set is found by brute force: every provided key is
 * tested against the membership predicate.  The softmax subtracts the row maximum before
 * exponentiating (mathematically neutral; it only keeps exp() finite).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Membership of key position i in the key set of query position t (0-indexed positions).
 * Causal (eq (1) of the BLA page), sinks i < s, and the recent window of m = w - s keys ending at
 * t (the SWA-with-sinks page). */
int swa_oracle_is_key(int64_t t, int64_t i, int64_t w, int64_t s)
{
    if (i < 0 || i > t) return 0;
    if (i < s) return 1;
    return i >= t - (w - s) + 1;
}

/* Membership of n key positions in the key set of query position t: out[j] = is_key(t, pos[j]). */
void swa_oracle_is_key_many(int64_t t, const int64_t *pos, int64_t n, int64_t w, int64_t s, uint8_t *out)
{
    for (int64_t j = 0; j < n; ++j) out[j] = (uint8_t)swa_oracle_is_key(t, pos[j], w, s);
}

/* Dense 0/1 mask of an L x L problem: mask[t*L + i] = 1 iff key i is attended by query t.
 * This is the picture of the "StreamingLLM recent band + sink left bar" pattern (page
 * "滑窗与固定稀疏", figure fig-attn-four-mask-compare). */
void swa_oracle_mask(int64_t L, int64_t w, int64_t s, uint8_t *mask)
{
    for (int64_t t = 0; t < L; ++t)
        for (int64_t i = 0; i < L; ++i)
            mask[t * L + i] = (uint8_t)swa_oracle_is_key(t, i, w, s);
}

/* One query row against a set of provided keys, each carrying its absolute position.
 * The keys may come in any order (the output of softmax attention does not depend on the order of
 * the keys: page "模糊窗口注意力", section 3 introduction, permutation invariance). */
static void attend_one(const double *q, int64_t qpos,
                       const double *k, const double *v, const int64_t *kpos, int64_t nk,
                       int64_t d, int64_t w, int64_t s, double scale,
                       double *o, double *lse, double *x, unsigned char *in)
{
    double mx = -INFINITY;
    for (int64_t j = 0; j < nk; ++j) {
        in[j] = (unsigned char)swa_oracle_is_key(qpos, kpos[j], w, s);
        if (!in[j]) continue;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += q[c] * k[j * d + c];
        x[j] = scale * dot;
        if (x[j] > mx) mx = x[j];
    }
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    double den = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
        if (!in[j]) continue;
        double e = exp(x[j] - mx);
        den += e;
        for (int64_t c = 0; c < d; ++c) o[c] += e * v[j * d + c];
    }
    if (den > 0.0) {
        for (int64_t c = 0; c < d; ++c) o[c] /= den;
        if (lse) *lse = mx + log(den);
    } else {
        /* no key at all (cannot happen for a query that sees its own key) */
        for (int64_t c = 0; c < d; ++c) o[c] = NAN;
        if (lse) *lse = NAN;
    }
}

typedef struct {
    const double *q, *k, *v;
    const int64_t *qpos, *kpos;
    int64_t nh, nq, nk, d, w, s;
    double scale;
    double *o, *lse;
    int64_t first, last; /* flat (head, row) range [first, last) */
} job_t;

static void *run_job(void *arg)
{
    job_t *jb = (job_t *)arg;
    double *x = (double *)malloc((size_t)(jb->nk > 0 ? jb->nk : 1) * sizeof(double));
    unsigned char *in = (unsigned char *)malloc((size_t)(jb->nk > 0 ? jb->nk : 1));
    for (int64_t f = jb->first; f < jb->last; ++f) {
        int64_t h = f / jb->nq, r = f % jb->nq;
        attend_one(jb->q + (h * jb->nq + r) * jb->d, jb->qpos[r],
                   jb->k + h * jb->nk * jb->d, jb->v + h * jb->nk * jb->d, jb->kpos, jb->nk,
                   jb->d, jb->w, jb->s, jb->scale,
                   jb->o + (h * jb->nq + r) * jb->d, jb->lse ? jb->lse + h * jb->nq + r : NULL,
                   x, in);
    }
    free(x);
    free(in);
    return NULL;
}

/* For each of nh independent heads: queries q[h] (nq x d, positions qpos) against keys/values
 * k[h], v[h] (nk x d, positions kpos).  o: nh x nq x d, lse (optional): nh x nq, natural log of
 * sum_{i in K(t)} exp(scale * q_t.k_i).  Work is split over nthreads POSIX threads by (head, row). */
void swa_oracle_attend(const double *q, const int64_t *qpos,
                       const double *k, const double *v, const int64_t *kpos,
                       int64_t nh, int64_t nq, int64_t nk, int64_t d, int64_t w, int64_t s,
                       double scale, double *o, double *lse, int nthreads)
{
    int64_t total = nh * nq;
    if (total <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = (int)total;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        job_t jb = {q, k, v, qpos, kpos, nh, nq, nk, d, w, s, scale, o, lse,
                    total * i / nthreads, total * (i + 1) / nthreads};
        jobs[i] = jb;
    }
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, run_job, &jobs[i]);
    run_job(&jobs[0]);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(jobs);
    free(th);
}

/* Replay of the streaming-cache writes, one position after another: position p goes to slot p when
 * p < s (the sink block) and to slot s + ((p - s) mod m) otherwise (the recent ring of m = w - s
 * slots), overwriting whatever the slot held.  After npos writes, holder[j] is the position slot j
 * holds, or -1 when it was never written.  With s = 0 this is the rolling buffer cache_slot(i) =
 * i mod W of page "滑窗与固定稀疏", eq attn-fixed-rolling. */
void swa_oracle_cache_replay(int64_t w, int64_t s, int64_t npos, int64_t *holder)
{
    int64_t m = w - s;
    for (int64_t j = 0; j < w; ++j) holder[j] = -1;
    for (int64_t p = 0; p < npos; ++p) {
        int64_t slot = (p < s) ? p : s + (p - s) % m;
        holder[slot] = p;
    }
}

/*
 * attn_oracle.c -- fp64 CPU oracle for exact attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * What it computes is the plain definition that the tiled online-softmax
 * method reaches up to rounding order, written out row by row in double
 * precision, following the dense reference of aiml.sh "verify-tiled-attention"
 * (function standard_attention, steps "1. Compute S = Q K^T * scale",
 * "2. Row-wise softmax", "3. Output O = P V") and the naive_attention of
 * deepnotes "flash-attention-implemented-verified-and-measured" (section
 * "The reference implementation, in full").  For one query row i of one
 * (batch, head) slice:
 *
 *   s_j   = scale * sum_c q[i,c] * k[j,c]        for every visible key j
 *   m     = max_j s_j        (0 when subtract_max == 0: the unshifted softmax
 *                             that the same page's overflow test exercises)
 *   e_j   = exp(s_j - m)
 *   Z     = sum_j e_j
 *   o[i,:] = sum_j (e_j / Z) * v[j,:]
 *   lse_i = m + ln Z
 *
 * Visible keys: all Skv keys when causal == 0.  When causal != 0, key j is
 * visible to query i iff j <= i + (Skv - Sq); for Sq == Skv this is the page's
 * "limit = i + 1".  The pages only use Sq == Skv; bottom-right alignment for
 * Sq != Skv is this library's reading.  A row with no visible key (possible
 * only when causal and Sq > Skv) has o = 0 and lse = -inf: the
 * huhohoo "tiled-online-softmax" page ("Online normalization") says such
 * rows need separate handling, and these are the values chosen for them.
 *
 * The log-sum-exp output is not on the pages; lse = m + ln Z in natural log
 * of the scaled scores is this library's definition of it.
 *
 * Layout: q [BH, Sq, d], k and v [BH, Skv, d], o [BH, Sq, d], lse [BH, Sq],
 * all contiguous row-major doubles.  Work is split over rows across
 * nthreads POSIX threads; each row is computed independently with the same
 * loop order, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int64_t bh_count, sq, skv, d;
    int causal, subtract_max;
    double scale;
    /* rows to compute: either all rows (rows == NULL) or a list of
     * (bh, i) pairs, written packed into o/lse in list order */
    const int64_t *rows;
    int64_t nrows;
    int64_t begin, end; /* range of row slots for this thread */
    int status;
} oracle_job;

static int64_t visible_keys(int64_t i, int64_t sq, int64_t skv, int causal)
{
    if (!causal)
        return skv;
    int64_t lim = i + 1 + (skv - sq);
    if (lim < 0)
        lim = 0;
    if (lim > skv)
        lim = skv;
    return lim;
}

/* One query row, straight from the definition above.  s is scratch of at
 * least skv doubles. */
static void oracle_row(const double *qi, const double *k, const double *v,
                       int64_t n_vis, int64_t d, double scale,
                       int subtract_max, double *s, double *oi, double *lsei)
{
    int64_t j, c;
    for (c = 0; c < d; ++c)
        oi[c] = 0.0;
    if (n_vis == 0) {
        *lsei = -INFINITY;
        return;
    }
    /* 1. scores */
    for (j = 0; j < n_vis; ++j) {
        const double *kj = k + j * d;
        double acc = 0.0;
        for (c = 0; c < d; ++c)
            acc += qi[c] * kj[c];
        s[j] = acc * scale;
    }
    /* 2. row maximum */
    double m = 0.0;
    if (subtract_max) {
        m = s[0];
        for (j = 1; j < n_vis; ++j)
            if (s[j] > m)
                m = s[j];
    }
    /* 3. exponentials and their sum */
    double z = 0.0;
    for (j = 0; j < n_vis; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    /* 4. probabilities times values */
    for (j = 0; j < n_vis; ++j) {
        const double p = s[j] / z;
        const double *vj = v + j * d;
        for (c = 0; c < d; ++c)
            oi[c] += p * vj[c];
    }
    /* 5. log-sum-exp of the scaled scores */
    *lsei = m + log(z);
}

static void *oracle_worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    double *s = (double *)malloc((size_t)(job->skv > 0 ? job->skv : 1) * sizeof(double));
    if (!s) {
        job->status = 2;
        return NULL;
    }
    for (int64_t r = job->begin; r < job->end; ++r) {
        int64_t bh, i, slot_o, slot_l;
        if (job->rows) {
            bh = job->rows[2 * r];
            i = job->rows[2 * r + 1];
            slot_o = r * job->d;
            slot_l = r;
        } else {
            bh = r / job->sq;
            i = r % job->sq;
            slot_o = r * job->d;
            slot_l = r;
        }
        const double *qi = job->q + (bh * job->sq + i) * job->d;
        const double *kb = job->k + bh * job->skv * job->d;
        const double *vb = job->v + bh * job->skv * job->d;
        int64_t n_vis = visible_keys(i, job->sq, job->skv, job->causal);
        double lse_val;
        oracle_row(qi, kb, vb, n_vis, job->d, job->scale, job->subtract_max, s,
                   job->o + slot_o, &lse_val);
        if (job->lse)
            job->lse[slot_l] = lse_val;
    }
    free(s);
    return NULL;
}

static int run_jobs(oracle_job *tmpl, int64_t total, int nthreads)
{
    enum { MAX_THREADS = 256 };
    oracle_job jobs[MAX_THREADS];
    pthread_t th[MAX_THREADS];
    int started[MAX_THREADS];
    int status = 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > MAX_THREADS)
        nthreads = MAX_THREADS;
    if ((int64_t)nthreads > total)
        nthreads = total > 0 ? (int)total : 1;
    int64_t per = (total + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *tmpl;
        jobs[t].begin = t * per;
        jobs[t].end = (t + 1) * per < total ? (t + 1) * per : total;
        jobs[t].status = 0;
        started[t] = 0;
        if (jobs[t].begin >= jobs[t].end)
            continue;
        if (nthreads > 1 && pthread_create(&th[t], NULL, oracle_worker, &jobs[t]) == 0)
            started[t] = 1;
        else
            oracle_worker(&jobs[t]); /* single thread, or a thread could not start */
    }
    for (int t = 0; t < nthreads; ++t) {
        if (started[t])
            pthread_join(th[t], NULL);
        status |= jobs[t].status;
    }
    return status;
}

/* All rows of all (batch, head) slices.  Returns 0 on success. */
int oracle_attn_fwd(const double *q, const double *k, const double *v,
                    double *o, double *lse, int64_t bh_count, int64_t sq,
                    int64_t skv, int64_t d, int causal, double scale,
                    int subtract_max, int nthreads)
{
    if (bh_count < 0 || sq < 0 || skv < 0 || d < 1)
        return 1;
    oracle_job tmpl;
    memset(&tmpl, 0, sizeof(tmpl));
    tmpl.q = q; tmpl.k = k; tmpl.v = v; tmpl.o = o; tmpl.lse = lse;
    tmpl.bh_count = bh_count; tmpl.sq = sq; tmpl.skv = skv; tmpl.d = d;
    tmpl.causal = causal; tmpl.subtract_max = subtract_max; tmpl.scale = scale;
    tmpl.rows = NULL;
    return run_jobs(&tmpl, bh_count * sq, nthreads);
}

/* Only the listed rows: rows holds nrows pairs (bh, i).  o receives nrows*d
 * values and lse nrows values, in list order. */
int oracle_attn_rows(const double *q, const double *k, const double *v,
                     double *o, double *lse, int64_t bh_count, int64_t sq,
                     int64_t skv, int64_t d, int causal, double scale,
                     const int64_t *rows, int64_t nrows, int nthreads)
{
    if (bh_count < 0 || sq < 0 || skv < 0 || d < 1 || nrows < 0)
        return 1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[2 * r] < 0 || rows[2 * r] >= bh_count || rows[2 * r + 1] < 0 ||
            rows[2 * r + 1] >= sq)
            return 1;
    oracle_job tmpl;
    memset(&tmpl, 0, sizeof(tmpl));
    tmpl.q = q; tmpl.k = k; tmpl.v = v; tmpl.o = o; tmpl.lse = lse;
    tmpl.bh_count = bh_count; tmpl.sq = sq; tmpl.skv = skv; tmpl.d = d;
    tmpl.causal = causal; tmpl.subtract_max = 1; tmpl.scale = scale;
    tmpl.rows = rows; tmpl.nrows = nrows;
    return run_jobs(&tmpl, nrows, nthreads);
}

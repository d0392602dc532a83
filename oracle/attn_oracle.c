/*
 * attn_oracle.c -- fp64 CPU oracle for scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link or call this file.  Only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark use it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes is the plain definition, written out row by row:
 *
 *   "Optimizing Attention on GPUs by Exploiting GPU Architectural NUMA
 *   Effects" (detail page), section 4, equation "S = QK^T, P = softmax(S/sqrt d),
 *   O = PV", with Q, K, V in R^{N x d} per head (section 4, notation table).
 *
 * For one query row q_i and the attended key set J_i:
 *   s_j  = scale * sum_k q_{i,k} k_{j,k}          (j in J_i)
 *   M    = max_j s_j
 *   p_j  = exp(s_j - M)
 *   l    = sum_j p_j
 *   o_i  = (sum_j p_j v_j) / l
 *   lse_i = M + log(l)      (natural log of sum_j exp(s_j))
 *
 * Subtracting M is only for range; it does not change o or lse.
 * J_i is the key range [k_lo, k_hi), further limited to j <= qpos_i when
 * causal is set.  An empty J_i gives o_i = 0 and lse_i = -inf (the pages
 * are silent on this case; this is the reading the CUDA path also follows).
 *
 * The log-sum-exp merge of partial states follows "kernbench2 ... Fused
 * Grouped-Query Attention", section "Inference with Long-Context Length",
 * Case 4 (two-phase reduction of the running softmax state (m, l, O)).
 *
 * Everything is computed in double precision.  Rows are spread over POSIX
 * threads; each row's arithmetic is sequential and independent of the
 * thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v;
    const int64_t *qpos;
    int64_t nq, nk, d, k_lo, k_hi;
    double scale;
    int causal;
    double *o, *lse;
    double *scratch; /* nk doubles per thread */
    int64_t row_begin, row_end;
} row_job;

/* One query row: scores, max, exponentials, normaliser, weighted sum of V. */
static void attend_one_row(const row_job *jb, int64_t i, double *s) {
    const int64_t d = jb->d;
    const double *qi = jb->q + i * d;
    double *oi = jb->o + i * d;
    int64_t hi = jb->k_hi;
    if (jb->causal) {
        int64_t last = jb->qpos[i] + 1; /* keys j <= qpos_i */
        if (last < hi) hi = last;
    }
    int64_t lo = jb->k_lo;
    for (int64_t c = 0; c < d; ++c) oi[c] = 0.0;
    if (hi <= lo) {
        jb->lse[i] = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = lo; j < hi; ++j) {
        const double *kj = jb->k + j * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += qi[c] * kj[c];
        s[j - lo] = jb->scale * dot;
        if (s[j - lo] > m) m = s[j - lo];
    }
    double l = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        double p = exp(s[j - lo] - m);
        s[j - lo] = p;
        l += p;
    }
    for (int64_t j = lo; j < hi; ++j) {
        const double *vj = jb->v + j * d;
        const double p = s[j - lo];
        for (int64_t c = 0; c < d; ++c) oi[c] += p * vj[c];
    }
    for (int64_t c = 0; c < d; ++c) oi[c] /= l;
    jb->lse[i] = m + log(l);
}

static void *row_worker(void *arg) {
    row_job *jb = (row_job *)arg;
    for (int64_t i = jb->row_begin; i < jb->row_end; ++i) attend_one_row(jb, i, jb->scratch);
    return NULL;
}

/* Number of worker threads the oracle uses when the caller passes 0. */
int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Attention for one head.
 *   q    [nq, d]   query rows
 *   qpos [nq]      absolute position of each query row (used only when causal)
 *   k, v [nk, d]   keys and values of the head (row j = key position j)
 *   keys attended: [k_lo, k_hi) and, if causal, j <= qpos[i]
 *   o    [nq, d]   output rows;  lse [nq] natural-log log-sum-exp of the scaled scores
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attention_head(const double *q, const double *k, const double *v, const int64_t *qpos,
                          int64_t nq, int64_t nk, int64_t d, double scale, int causal,
                          int64_t k_lo, int64_t k_hi, double *o, double *lse, int nthreads) {
    if (nq < 0 || nk < 0 || d <= 0 || k_lo < 0 || k_hi > nk) return -1;
    if (causal && !qpos) return -1;
    if (nq == 0) return 0;
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > nq) nthreads = (int)nq;
    int64_t span = nk > 0 ? nk : 1;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)span * (size_t)nthreads);
    row_job *jobs = (row_job *)malloc(sizeof(row_job) * (size_t)nthreads);
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!scratch || !jobs || !tids) {
        free(scratch); free(jobs); free(tids);
        return -1;
    }
    int64_t per = (nq + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        row_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->qpos = qpos;
        jb->nq = nq; jb->nk = nk; jb->d = d; jb->k_lo = k_lo; jb->k_hi = k_hi;
        jb->scale = scale; jb->causal = causal; jb->o = o; jb->lse = lse;
        jb->scratch = scratch + (size_t)t * (size_t)span;
        jb->row_begin = (int64_t)t * per;
        jb->row_end = jb->row_begin + per < nq ? jb->row_begin + per : nq;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, row_worker, &jobs[t]) != 0) break;
        started = t;
    }
    row_worker(&jobs[0]);
    /* rows of threads that could not be started run here */
    for (int t = started + 1; t < nthreads; ++t) row_worker(&jobs[t]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    free(scratch); free(jobs); free(tids);
    return 0;
}

/*
 * Log-sum-exp merge of S partial states of one query row.
 *   o_parts [S, d]  each partial output already normalised by its own l_s
 *   lse_parts [S]   each partial's log-sum-exp (-inf for an empty partial)
 * Result: L = max_s lse_s, w_s = exp(lse_s - L),
 *         o = sum_s w_s o_s / sum_s w_s,  lse = L + log(sum_s w_s).
 * All partials empty: o = 0, lse = -inf.
 */
int oracle_lse_merge(const double *o_parts, const double *lse_parts, int64_t S, int64_t d,
                     double *o, double *lse) {
    if (S < 0 || d <= 0) return -1;
    double L = -INFINITY;
    for (int64_t s = 0; s < S; ++s)
        if (lse_parts[s] > L) L = lse_parts[s];
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    if (L == -INFINITY) {
        *lse = -INFINITY;
        return 0;
    }
    double wsum = 0.0;
    for (int64_t s = 0; s < S; ++s) {
        if (lse_parts[s] == -INFINITY) continue;
        double w = exp(lse_parts[s] - L);
        wsum += w;
        for (int64_t c = 0; c < d; ++c) o[c] += w * o_parts[s * d + c];
    }
    for (int64_t c = 0; c < d; ++c) o[c] /= wsum;
    *lse = L + log(wsum);
    return 0;
}

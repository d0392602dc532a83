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
 *
 * The backward pass (oracle_attention_bwd_head) is the gradient of the same
 * definition by the chain rule, for a loss whose gradient with respect to the
 * output is dO (the pages measure an FA2 backward pass but print no formula
 * for it; the gradient of the section-4 equation is fixed by the mathematics):
 *   dv_j += p_j dO_i                              (O = P V)
 *   dp_j  = <dO_i, v_j>
 *   D_i   = <dO_i, o_i> = sum_j p_j dp_j
 *   ds_j  = p_j (dp_j - D_i)                      (softmax Jacobian)
 *   dq_i  = scale * sum_j ds_j k_j                (s_j = scale <q_i, k_j>)
 *   dk_j += scale * ds_j q_i
 * with p the normalised probabilities of row i over its attended keys.
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

/* ------------------------------------------------------------------ backward */

typedef struct {
    const double *q, *k, *v, *dout;
    const int64_t *qpos;
    int64_t nq, nk, d;
    double scale;
    int causal;
    double *dq;      /* [nq, d], rows of this job only */
    double *dk, *dv; /* [nk, d], this job's private sums */
    double *p;       /* nk doubles of scratch */
    int64_t row_begin, row_end;
} grad_job;

/* Gradient contributions of one query row (see the file comment). */
static void grad_one_row(const grad_job *jb, int64_t i) {
    const int64_t d = jb->d;
    const double *qi = jb->q + i * d;
    const double *gi = jb->dout + i * d;
    double *dqi = jb->dq + i * d;
    for (int64_t c = 0; c < d; ++c) dqi[c] = 0.0;
    int64_t hi = jb->nk;
    if (jb->causal && jb->qpos[i] + 1 < hi) hi = jb->qpos[i] + 1;
    if (hi <= 0) return; /* no attended key: the output is the constant 0 */
    double *p = jb->p;
    double m = -INFINITY;
    for (int64_t j = 0; j < hi; ++j) {
        const double *krow = jb->k + j * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += qi[c] * krow[c];
        p[j] = jb->scale * dot;
        if (p[j] > m) m = p[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < hi; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (int64_t j = 0; j < hi; ++j) p[j] /= l;
    /* D_i = <dO_i, o_i> with o_i = sum_j p_j v_j */
    double D = 0.0;
    for (int64_t c = 0; c < d; ++c) {
        double oc = 0.0;
        for (int64_t j = 0; j < hi; ++j) oc += p[j] * jb->v[j * d + c];
        D += gi[c] * oc;
    }
    for (int64_t j = 0; j < hi; ++j) {
        const double *krow = jb->k + j * d;
        const double *vrow = jb->v + j * d;
        double dp = 0.0;
        for (int64_t c = 0; c < d; ++c) dp += gi[c] * vrow[c];
        const double ds = p[j] * (dp - D);
        double *dkj = jb->dk + j * d;
        double *dvj = jb->dv + j * d;
        for (int64_t c = 0; c < d; ++c) {
            dqi[c] += jb->scale * ds * krow[c];
            dkj[c] += jb->scale * ds * qi[c];
            dvj[c] += p[j] * gi[c];
        }
    }
}

static void *grad_worker(void *arg) {
    grad_job *jb = (grad_job *)arg;
    for (int64_t i = jb->row_begin; i < jb->row_end; ++i) grad_one_row(jb, i);
    return NULL;
}

/*
 * Gradients of one head.
 *   q, dout [nq, d]; k, v [nk, d]; qpos [nq] (used only when causal: key j is
 *   attended by row i when j <= qpos[i])
 *   dq [nq, d]; dk, dv [nk, d]   outputs (overwritten)
 * dk and dv are the sums of the rows' contributions; each thread sums its own
 * rows and the threads' sums are added in thread order.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attention_bwd_head(const double *q, const double *k, const double *v,
                              const double *dout, const int64_t *qpos, int64_t nq, int64_t nk,
                              int64_t d, double scale, int causal, double *dq, double *dk,
                              double *dv, int nthreads) {
    if (nq < 0 || nk < 0 || d <= 0) return -1;
    if (causal && !qpos) return -1;
    for (int64_t x = 0; x < nk * d; ++x) dk[x] = dv[x] = 0.0;
    if (nq == 0) return 0;
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > nq) nthreads = (int)nq;
    const size_t span = (size_t)(nk > 0 ? nk : 1);
    const size_t kd = (size_t)nk * (size_t)d;
    double *scratch = (double *)malloc(sizeof(double) * span * (size_t)nthreads);
    double *acc = (double *)calloc(2 * kd * (size_t)nthreads + 1, sizeof(double));
    grad_job *jobs = (grad_job *)malloc(sizeof(grad_job) * (size_t)nthreads);
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!scratch || !acc || !jobs || !tids) {
        free(scratch); free(acc); free(jobs); free(tids);
        return -1;
    }
    int64_t per = (nq + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        grad_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->dout = dout; jb->qpos = qpos;
        jb->nq = nq; jb->nk = nk; jb->d = d; jb->scale = scale; jb->causal = causal;
        jb->dq = dq;
        jb->dk = acc + 2 * kd * (size_t)t;
        jb->dv = jb->dk + kd;
        jb->p = scratch + span * (size_t)t;
        jb->row_begin = (int64_t)t * per;
        jb->row_end = jb->row_begin + per < nq ? jb->row_begin + per : nq;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, grad_worker, &jobs[t]) != 0) break;
        started = t;
    }
    grad_worker(&jobs[0]);
    for (int t = started + 1; t < nthreads; ++t) grad_worker(&jobs[t]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = 0; t < nthreads; ++t)
        for (size_t x = 0; x < kd; ++x) {
            dk[x] += jobs[t].dk[x];
            dv[x] += jobs[t].dv[x];
        }
    free(scratch); free(acc); free(jobs); free(tids);
    return 0;
}

/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for batched
 * speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the test-suite, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes follows the "spec-verify" page (Hugging Face kernels page
 * phanerozoic/spec-verify), section "Method":
 *   - greedy: accept draft token t_i while it equals argmax(target_i); at the
 *     first miss emit argmax(target_i) and stop; when all K match emit
 *     argmax(target_K) as the bonus token;
 *   - speculative sampling (Leviathan et al. / Chen et al.): accept t_i with
 *     probability min(1, p_i(t_i)/q_i(t_i)) using an explicit uniform; on a
 *     rejection resample from norm(max(0, p_i - q_i)); when all K are accepted
 *     sample the bonus from p_K.
 * and section "Correctness": probabilities need not be normalised and masses
 * are summed exactly -- read here as fp64 sums taken in ascending token order.
 *
 * Readings of points the page leaves open (each listed in the design notes):
 *   - argmax ties go to the lowest index (strict '>' while scanning upward);
 *   - the accept test is  (double)u * (double)q(t) < (double)p(t); the fp64
 *     product of two fp32 values is exact, so the decision is exact;
 *   - the inverse CDF returns the smallest v whose running fp64 sum C_v
 *     exceeds T = u * R (R = total mass), so zero-mass tokens are never drawn;
 *     if rounding makes T reach R, the last token with non-zero mass is drawn;
 *   - the bonus draw and the resample draw use the same per-sequence uniform
 *     u_resample[b] (exactly one of the two happens in a round);
 *   - a rejection whose residual has zero total mass (possible only with
 *     unnormalised rows) falls back to sampling from p_i; if that mass is zero
 *     too, next_token = -1 and the ZERO_MASS status bit is set;
 *   - a draft id outside [0, V) makes the whole sequence invalid: (0, -1) and
 *     the BAD_TOKEN status bit;
 *   - round mode values other than 0 (greedy) and 1 (sampling) give (0, -1)
 *     and the BAD_MODE status bit.
 *
 * Layout: p row (b, i), i in [0, K], starts at p + (b*(K+1) + i) * p_stride;
 * q row (b, i), i in [0, K), starts at q + (b*K + i) * q_stride; t, u_accept
 * are [B][K]; u_resample is [B]; mode is [B].
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#define ORC_STATUS_BAD_TOKEN 1u
#define ORC_STATUS_ZERO_MASS 2u
#define ORC_STATUS_OVERFLOW 4u
#define ORC_STATUS_BAD_MODE 8u

/* Index of the largest element of row[0..V), the lowest index among equals. */
int64_t orc_argmax_lowest(const float *row, int64_t V)
{
    float best = row[0];
    int64_t idx = 0;
    for (int64_t v = 1; v < V; ++v) {
        if (row[v] > best) {
            best = row[v];
            idx = v;
        }
    }
    return idx;
}

/* Inverse CDF over non-negative fp64 masses r[0..V) with uniform u in [0,1).
 * Returns the smallest v with C_v = r_0 + ... + r_v > u * R, R = C_{V-1};
 * -1 if R is zero.  Sums run in fp64, ascending v. */
int64_t orc_icdf(const double *r, int64_t V, double u)
{
    double R = 0.0;
    for (int64_t v = 0; v < V; ++v)
        R += r[v];
    if (!(R > 0.0))
        return -1;
    double T = u * R;
    double C = 0.0;
    int64_t last_nonzero = -1;
    for (int64_t v = 0; v < V; ++v) {
        C += r[v];
        if (r[v] > 0.0)
            last_nonzero = v;
        if (C > T)
            return v;
    }
    return last_nonzero; /* u * R rounded up to R */
}

/* Residual masses r_v = max(0, p_v - q_v) formed in fp64; with q == NULL the
 * masses are p_v themselves (the bonus draw and the zero-residual fallback). */
static void residual_row(const float *p, const float *q, int64_t V, double *r)
{
    for (int64_t v = 0; v < V; ++v) {
        if (q) {
            double d = (double)p[v] - (double)q[v];
            r[v] = d > 0.0 ? d : 0.0;
        } else {
            r[v] = (double)p[v];
        }
    }
}

/* Running fp64 sums C_v of the residual (or of p when q == NULL); returns the
 * total.  Used by the tests to locate inverse-CDF boundaries. */
double orc_residual_cumsum(const float *p, const float *q, int64_t V, double *C)
{
    double acc = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double m;
        if (q) {
            double d = (double)p[v] - (double)q[v];
            m = d > 0.0 ? d : 0.0;
        } else {
            m = (double)p[v];
        }
        acc += m;
        C[v] = acc;
    }
    return acc;
}

static int tokens_in_range(const int32_t *t, int K, int64_t V)
{
    for (int i = 0; i < K; ++i)
        if (t[i] < 0 || (int64_t)t[i] >= V)
            return 0;
    return 1;
}

static void greedy_one(const float *p, int64_t p_stride, const int32_t *t,
                       int K, int64_t V, int32_t *n_out, int32_t *next_out,
                       uint32_t *status)
{
    if (!tokens_in_range(t, K, V)) {
        *n_out = 0;
        *next_out = -1;
        *status |= ORC_STATUS_BAD_TOKEN;
        return;
    }
    for (int i = 0; i < K; ++i) {
        int64_t a = orc_argmax_lowest(p + (int64_t)i * p_stride, V);
        if ((int64_t)t[i] != a) {
            *n_out = i;
            *next_out = (int32_t)a;
            return;
        }
    }
    *n_out = K;
    *next_out = (int32_t)orc_argmax_lowest(p + (int64_t)K * p_stride, V);
}

static void sample_one(const float *p, int64_t p_stride, const float *q,
                       int64_t q_stride, const int32_t *t, const float *u_acc,
                       double u_res, int K, int64_t V, double *r,
                       int32_t *n_out, int32_t *next_out, uint32_t *status)
{
    if (!tokens_in_range(t, K, V)) {
        *n_out = 0;
        *next_out = -1;
        *status |= ORC_STATUS_BAD_TOKEN;
        return;
    }
    for (int i = 0; i < K; ++i) {
        const float *pi = p + (int64_t)i * p_stride;
        const float *qi = q + (int64_t)i * q_stride;
        int32_t x = t[i];
        int accept = (double)u_acc[i] * (double)qi[x] < (double)pi[x];
        if (!accept) {
            residual_row(pi, qi, V, r);
            int64_t j = orc_icdf(r, V, u_res);
            if (j < 0) {
                residual_row(pi, NULL, V, r);
                j = orc_icdf(r, V, u_res);
            }
            if (j < 0)
                *status |= ORC_STATUS_ZERO_MASS;
            *n_out = i;
            *next_out = (int32_t)j;
            return;
        }
    }
    residual_row(p + (int64_t)K * p_stride, NULL, V, r);
    int64_t j = orc_icdf(r, V, u_res);
    if (j < 0)
        *status |= ORC_STATUS_ZERO_MASS;
    *n_out = K;
    *next_out = (int32_t)j;
}

/* One batch of sequences [b0, b1): mode == NULL means all greedy when
 * q == NULL and all sampling otherwise. */
typedef struct {
    const uint8_t *mode;
    const float *p;
    int64_t p_stride;
    const float *q;
    int64_t q_stride;
    const int32_t *t;
    const float *u_acc;
    const double *u_res;
    int K;
    int64_t V;
    int32_t *n_out;
    int32_t *next_out;
    int b0, b1;
    uint32_t status;
    int oom;
} orc_job;

static void run_job(orc_job *j)
{
    double *r = NULL;
    if (j->q) {
        r = (double *)malloc((size_t)j->V * sizeof(double));
        if (!r) {
            j->oom = 1;
            return;
        }
    }
    for (int b = j->b0; b < j->b1; ++b) {
        const float *pb = j->p + (int64_t)b * (j->K + 1) * j->p_stride;
        const int32_t *tb = j->t + (int64_t)b * j->K;
        int m = j->mode ? (int)j->mode[b] : (j->q ? 1 : 0);
        if (m == 0) {
            greedy_one(pb, j->p_stride, tb, j->K, j->V, &j->n_out[b],
                       &j->next_out[b], &j->status);
        } else if (m == 1 && j->q) {
            const float *qb = j->q + (int64_t)b * j->K * j->q_stride;
            sample_one(pb, j->p_stride, qb, j->q_stride, tb,
                       j->u_acc + (int64_t)b * j->K, j->u_res[b], j->K, j->V,
                       r, &j->n_out[b], &j->next_out[b], &j->status);
        } else {
            j->n_out[b] = 0;
            j->next_out[b] = -1;
            j->status |= ORC_STATUS_BAD_MODE;
        }
    }
    free(r);
}

static void *job_thread(void *arg)
{
    run_job((orc_job *)arg);
    return NULL;
}

/* Splits sequences into nthreads contiguous blocks, one pthread each. */
static int run_batched(const uint8_t *mode, const float *p, int64_t p_stride,
                       const float *q, int64_t q_stride, const int32_t *t,
                       const float *u_acc, const double *u_res, int B, int K,
                       int64_t V, int32_t *n_out, int32_t *next_out,
                       uint32_t *status, int nthreads)
{
    if (B <= 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > B)
        nthreads = B;
    orc_job *jobs = (orc_job *)calloc((size_t)nthreads, sizeof(orc_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -1;
    }
    for (int k = 0; k < nthreads; ++k) {
        orc_job *j = &jobs[k];
        j->mode = mode;
        j->p = p;
        j->p_stride = p_stride;
        j->q = q;
        j->q_stride = q_stride;
        j->t = t;
        j->u_acc = u_acc;
        j->u_res = u_res;
        j->K = K;
        j->V = V;
        j->n_out = n_out;
        j->next_out = next_out;
        j->b0 = (int)((int64_t)B * k / nthreads);
        j->b1 = (int)((int64_t)B * (k + 1) / nthreads);
    }
    char *spawned = (char *)calloc((size_t)nthreads, 1);
    for (int k = 1; k < nthreads; ++k) {
        if (spawned && pthread_create(&th[k], NULL, job_thread, &jobs[k]) == 0)
            spawned[k] = 1;
        else
            run_job(&jobs[k]); /* run inline if a thread cannot start */
    }
    run_job(&jobs[0]);
    int rc = 0;
    for (int k = 0; k < nthreads; ++k) {
        if (spawned && spawned[k])
            pthread_join(th[k], NULL);
        if (jobs[k].oom)
            rc = -1;
        *status |= jobs[k].status;
    }
    free(spawned);
    free(jobs);
    free(th);
    return rc;
}

int orc_verify_greedy(const float *p, int64_t p_stride, const int32_t *t,
                      int B, int K, int64_t V, int32_t *n_out,
                      int32_t *next_out, uint32_t *status, int nthreads)
{
    return run_batched(NULL, p, p_stride, NULL, 0, t, NULL, NULL, B, K, V,
                       n_out, next_out, status, nthreads);
}

int orc_verify_sample(const float *p, int64_t p_stride, const float *q,
                      int64_t q_stride, const int32_t *t, const float *u_acc,
                      const double *u_res, int B, int K, int64_t V,
                      int32_t *n_out, int32_t *next_out, uint32_t *status,
                      int nthreads)
{
    return run_batched(NULL, p, p_stride, q, q_stride, t, u_acc, u_res, B, K,
                       V, n_out, next_out, status, nthreads);
}

int orc_verify_round(const uint8_t *mode, const float *p, int64_t p_stride,
                     const float *q, int64_t q_stride, const int32_t *t,
                     const float *u_acc, const double *u_res, int B, int K,
                     int64_t V, int32_t *n_out, int32_t *next_out,
                     uint32_t *status, int nthreads)
{
    return run_batched(mode, p, p_stride, q, q_stride, t, u_acc, u_res, B, K,
                       V, n_out, next_out, status, nthreads);
}

/* Commit step of a round ("keep draft_tokens[:n_accepted], append
 * next_token", spec-verify page, section "Usage"): appends t[b][0..n) and
 * next to tokens[b][lengths[b]..] and advances lengths[b].  A sequence whose
 * next token is -1 is left untouched; one that would pass max_len is left
 * untouched and sets the OVERFLOW status bit. */
void orc_commit(const int32_t *t, int B, int K, const int32_t *n_acc,
                const int32_t *next, int32_t *tokens, int32_t *lengths,
                int max_len, uint32_t *status)
{
    for (int b = 0; b < B; ++b) {
        if (next[b] < 0)
            continue;
        int len = lengths[b];
        int n = n_acc[b];
        if (len < 0 || (int64_t)len + n + 1 > max_len) {
            *status |= ORC_STATUS_OVERFLOW;
            continue;
        }
        int32_t *row = tokens + (int64_t)b * max_len;
        for (int i = 0; i < n; ++i)
            row[len + i] = t[(int64_t)b * K + i];
        row[len + n] = next[b];
        lengths[b] = len + n + 1;
    }
}

/* Per-position acceptance rate of the sampling rule, the quantity behind the
 * page's analytic accepted-length law ("spec-verify" page, section
 * "Measured"; the law itself is the rejection-sampling theorem of Leviathan
 * et al. / Chen et al.).  For each sequence b and draft position i < K:
 *     alpha[b][i] = sum_v min(p_i(v) / P_i, q_i(v) / Q_i),
 * P_i and Q_i the fp64 row totals (rows need not be normalised; a row with
 * zero total gives alpha = 0), and, when expected != NULL,
 *     expected[b] = sum_{m=1..K} prod_{j<m} alpha[b][j],
 * the mean number of accepted draft tokens of a round.  Sums run in fp64 in
 * ascending v. */
void orc_alpha(const float *p, int64_t p_stride, const float *q,
               int64_t q_stride, int B, int K, int64_t V, double *alpha,
               double *expected)
{
    for (int b = 0; b < B; ++b) {
        double mean = 0.0, reach = 1.0;
        for (int i = 0; i < K; ++i) {
            const float *pr = p + ((int64_t)b * (K + 1) + i) * p_stride;
            const float *qr = q + ((int64_t)b * K + i) * q_stride;
            double P = 0.0, Q = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                P += (double)pr[v];
                Q += (double)qr[v];
            }
            double a = 0.0;
            if (P > 0.0 && Q > 0.0) {
                for (int64_t v = 0; v < V; ++v) {
                    const double x = (double)pr[v] / P;
                    const double y = (double)qr[v] / Q;
                    a += x < y ? x : y;
                }
            }
            alpha[(int64_t)b * K + i] = a;
            reach *= a;    /* P(n > i) = prod_{j <= i} alpha_j */
            mean += reach;
        }
        if (expected)
            expected[b] = mean;
    }
}

/* Temperature softmax of one row of logits in fp64:
 *     out_v = exp((z_v - max_w z_w) / tau) / sum_w exp((z_w - max_w z_w) / tau),
 * the warp the "spec-verify" page requires both distributions to share
 * (section "Requirements and limits").  Sums run in ascending v. */
void orc_softmax(const float *z, int64_t V, double tau, double *out)
{
    double m = (double)z[0];
    for (int64_t v = 1; v < V; ++v)
        if ((double)z[v] > m)
            m = (double)z[v];
    double S = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        out[v] = exp(((double)z[v] - m) / tau);
        S += out[v];
    }
    for (int64_t v = 0; v < V; ++v)
        out[v] /= S;
}

/* Sampling verification of one sequence from logits: p_i = softmax(zp_i/tau),
 * q_i = softmax(zq_i/tau) in fp64, then the rule of section "Method" on those
 * rows -- accept t_i iff u_acc[i] * q_i(t_i) < p_i(t_i) (fp64), on a rejection
 * draw from max(0, p_i - q_i) with u_res, after all K the bonus from p_K. */
static void sample_logits_one(const float *zp, int64_t zp_stride, const float *zq,
                              int64_t zq_stride, const int32_t *t,
                              const float *u_acc, double u_res, int K,
                              int64_t V, double tau, double *pr, double *qr,
                              int32_t *n_out, int32_t *next_out,
                              uint32_t *status)
{
    if (!tokens_in_range(t, K, V)) {
        *n_out = 0;
        *next_out = -1;
        *status |= ORC_STATUS_BAD_TOKEN;
        return;
    }
    for (int i = 0; i < K; ++i) {
        orc_softmax(zp + (int64_t)i * zp_stride, V, tau, pr);
        orc_softmax(zq + (int64_t)i * zq_stride, V, tau, qr);
        int32_t x = t[i];
        if (!((double)u_acc[i] * qr[x] < pr[x])) {
            for (int64_t v = 0; v < V; ++v) {
                const double d = pr[v] - qr[v];
                pr[v] = (d > 0.0) ? d : 0.0;
            }
            int64_t j = orc_icdf(pr, V, u_res);
            if (j < 0) { /* p_i == q_i: the residual has no mass; draw from p_i */
                orc_softmax(zp + (int64_t)i * zp_stride, V, tau, pr);
                j = orc_icdf(pr, V, u_res);
            }
            *next_out = (int32_t)j;
            *n_out = i;
            return;
        }
    }
    orc_softmax(zp + (int64_t)K * zp_stride, V, tau, pr);
    *n_out = K;
    *next_out = (int32_t)orc_icdf(pr, V, u_res);
}

/* Batched form over B sequences (layout as the probability entry points,
 * logits in place of probabilities).  Returns -1 for a temperature that is
 * not a positive finite number, -2 when out of memory, 0 otherwise. */
int orc_verify_sample_logits(const float *zp, int64_t zp_stride,
                             const float *zq, int64_t zq_stride,
                             const int32_t *t, const float *u_acc,
                             const double *u_res, int B, int K, int64_t V,
                             double tau, int32_t *n_out, int32_t *next_out,
                             uint32_t *status)
{
    if (!(tau > 0.0) || !isfinite(tau))
        return -1;
    double *pr = malloc((size_t)V * sizeof(double));
    double *qr = malloc((size_t)V * sizeof(double));
    if (!pr || !qr) {
        free(pr);
        free(qr);
        return -2;
    }
    for (int b = 0; b < B; ++b)
        sample_logits_one(zp + (int64_t)b * (K + 1) * zp_stride, zp_stride,
                          zq + (int64_t)b * K * zq_stride, zq_stride,
                          t + (int64_t)b * K, u_acc + (int64_t)b * K, u_res[b],
                          K, V, tau, pr, qr, n_out + b, next_out + b, status);
    free(pr);
    free(qr);
    return 0;
}

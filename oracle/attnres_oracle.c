/*
 * attnres_oracle.c -- plain, slow FP64 CPU oracle for the Attention Residuals
 * (AttnRes) read operator.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the benchmark's CPU-baseline leg call it; the product path never
 * does.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (per token n, independently -- "Fast Attention Residuals",
 * section "Equation"):
 *
 *   t_s     = v_s[n, ko : ko+R]                 (the implicit key slice)
 *   r_s     = 1 / sqrt(mean_j(t_s[j]^2) + eps)  (mean over the R key channels)
 *   k_s     = r_s * t_s
 *   z_s     = scale * <k_s, q>                  (routing logit)
 *   a_s     = softmax over s of z               (routing weight, "alpha")
 *   o       = sum_s a_s * v_s[n, 0:D]           (full-width read)
 *
 * The page places the key in the final R coordinates (ko = D-R); the caller
 * passes ko explicitly so that ko = 0 (the first R channels) is also covered.
 *
 * Optional output RMSNorm ("[Perf] Parallelize AttnRes long-sequence
 * reduction", Summary: the forward saves the output-RMSNorm reciprocal
 * standard deviation o_rstd for backward reuse, next to o_pre and the
 * output RMS weight).  The pages do not print its formula; the plain reading
 * used here is the standard weighted RMSNorm over D with the same eps:
 *
 *   rho = 1 / sqrt(mean_j(o[j]^2) + eps),  yhat = rho * o,  y = yhat * w_o
 *
 * Without the flag, y = o.
 *
 * First-order backward for an upstream gradient dy[n, 0:D] (derived by the
 * chain rule from the equation above; the pages state that ordinary
 * first-order autograd flows through keys, query and shared sources):
 *
 *   out-norm:  dw_o += dy * yhat (summed over n),  g = dy * w_o,
 *              do = rho * (g - yhat * <g, yhat> / D);   else do = dy
 *   da_s  = <do, v_s>
 *   delta = sum_s a_s * da_s
 *   dz_s  = a_s * (da_s - delta)                  (softmax backward)
 *   dq   += scale * sum_s dz_s * k_s              (summed over n)
 *   dt_s  = r_s * dz_s * (scale * q - (z_s / R) * k_s)   (RMSNorm backward)
 *   dv_s  = a_s * do, plus dt_s added on channels [ko, ko+R)
 *
 * Everything is IEEE double.  bf16 inputs are widened exactly (a bf16 value
 * is the top 16 bits of an IEEE single).  Tokens are independent, so a token
 * range may be split across threads; the sums over n (dq, dw_o) are formed
 * per thread in token order and then added in thread order.
 *
 * Parity status: every function here is pinned by the CPU tests (closed-form
 * special cases, invariants, central finite differences, and an independent
 * float64 autograd derivation of the gradients).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Widen one bf16 bit pattern to double (exact). */
static double bf16_to_double(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------------------
 * One token, all quantities in double.
 *   v      [S][D]   the token's S source rows
 *   q      [R]      query
 *   w_o    [D]      output-norm weight (used only when out_norm != 0)
 * Forward outputs (any may be NULL):
 *   y [D], alpha [S], rstd [S], logit [S], o_rstd [1]
 * Backward (performed when dy != NULL):
 *   dv [S][D] written; dq_acc [R] and dw_acc [D] accumulated (+=).
 * work: scratch of at least 4*S + 3*D doubles.
 * ------------------------------------------------------------------------- */
static void token_oracle(int S, int D, int R, int ko, double eps, double scale,
                         int out_norm, const double *v, const double *q,
                         const double *w_o, double *y, double *alpha,
                         double *rstd, double *logit, double *o_rstd,
                         const double *dy, double *dv, double *dq_acc,
                         double *dw_acc, double *work) {
    double *r = work;           /* [S] key reciprocal RMS  */
    double *z = r + S;          /* [S] logits              */
    double *a = z + S;          /* [S] softmax weights     */
    double *o = a + S;          /* [D] mixture             */
    double *yhat = o + D;       /* [D] normalised mixture  */
    double *dout = yhat + D;    /* [D] gradient wrt o      */

    /* key statistics and logits */
    for (int s = 0; s < S; ++s) {
        const double *t = v + (size_t)s * D + ko;
        double sumsq = 0.0;
        for (int j = 0; j < R; ++j) sumsq += t[j] * t[j];
        r[s] = 1.0 / sqrt(sumsq / (double)R + eps);
        double dot = 0.0;
        for (int j = 0; j < R; ++j) dot += (r[s] * t[j]) * q[j];
        z[s] = scale * dot;
    }
    /* softmax over sources (max subtracted for range, which leaves it unchanged) */
    double zmax = z[0];
    for (int s = 1; s < S; ++s)
        if (z[s] > zmax) zmax = z[s];
    double denom = 0.0;
    for (int s = 0; s < S; ++s) {
        a[s] = exp(z[s] - zmax);
        denom += a[s];
    }
    for (int s = 0; s < S; ++s) a[s] /= denom;

    /* weighted sum of full-width rows */
    for (int j = 0; j < D; ++j) {
        double acc = 0.0;
        for (int s = 0; s < S; ++s) acc += a[s] * v[(size_t)s * D + j];
        o[j] = acc;
    }
    /* optional output RMSNorm */
    double rho = 1.0;
    if (out_norm) {
        double ms = 0.0;
        for (int j = 0; j < D; ++j) ms += o[j] * o[j];
        rho = 1.0 / sqrt(ms / (double)D + eps);
        for (int j = 0; j < D; ++j) yhat[j] = rho * o[j];
    }
    if (y)
        for (int j = 0; j < D; ++j) y[j] = out_norm ? yhat[j] * w_o[j] : o[j];
    if (alpha)
        for (int s = 0; s < S; ++s) alpha[s] = a[s];
    if (rstd)
        for (int s = 0; s < S; ++s) rstd[s] = r[s];
    if (logit)
        for (int s = 0; s < S; ++s) logit[s] = z[s];
    if (o_rstd) *o_rstd = rho;

    if (!dy) return;

    /* gradient wrt the mixture o */
    if (out_norm) {
        double gy = 0.0;
        for (int j = 0; j < D; ++j) {
            dw_acc[j] += dy[j] * yhat[j];
            gy += dy[j] * w_o[j] * yhat[j];
        }
        for (int j = 0; j < D; ++j)
            dout[j] = rho * (dy[j] * w_o[j] - yhat[j] * gy / (double)D);
    } else {
        for (int j = 0; j < D; ++j) dout[j] = dy[j];
    }
    /* softmax backward */
    double delta = 0.0;
    double *da = work + 3 * S + 3 * D; /* [S] */
    for (int s = 0; s < S; ++s) {
        double d = 0.0;
        for (int j = 0; j < D; ++j) d += dout[j] * v[(size_t)s * D + j];
        da[s] = d;
        delta += a[s] * d;
    }
    for (int s = 0; s < S; ++s) {
        double dz = a[s] * (da[s] - delta);
        const double *t = v + (size_t)s * D + ko;
        double *g = dv + (size_t)s * D;
        for (int j = 0; j < D; ++j) g[j] = a[s] * dout[j];
        for (int j = 0; j < R; ++j) {
            double k = r[s] * t[j];
            dq_acc[j] += scale * dz * k;
            g[ko + j] += r[s] * dz * (scale * q[j] - (z[s] / (double)R) * k);
        }
    }
}

/* ---------------------------------------------------------------------------
 * Multi-token drivers.  Sources are packed [S][N][D]; element (s, n, j) sits
 * at src[(s*N + n)*D + j].  Per-token outputs: y [N][D], alpha/rstd/logit
 * [N][S], o_rstd [N], dsrc [S][N][D].  dq [R] and dw_o [D] are overwritten.
 * ------------------------------------------------------------------------- */
typedef struct {
    int S, D, R, ko, out_norm, bf16;
    long N, n0, n1;
    double eps, scale;
    const void *src, *q, *w_o, *dy;
    double *y, *alpha, *rstd, *logit, *o_rstd, *dsrc;
    double *dq, *dw_o; /* this worker's partial sums */
    int status;
} job_t;

static double load_elem(const void *base, int bf16, size_t idx) {
    return bf16 ? bf16_to_double(((const uint16_t *)base)[idx])
                : ((const double *)base)[idx];
}

static void *run_range(void *arg) {
    job_t *jb = (job_t *)arg;
    const int S = jb->S, D = jb->D, R = jb->R;
    const long N = jb->N;
    double *v = malloc(sizeof(double) * (size_t)S * D);
    double *q = malloc(sizeof(double) * (size_t)R);
    double *w = malloc(sizeof(double) * (size_t)D);
    double *dy = malloc(sizeof(double) * (size_t)D);
    double *dv = malloc(sizeof(double) * (size_t)S * D);
    double *work = malloc(sizeof(double) * (size_t)(4 * S + 3 * D));
    if (!v || !q || !w || !dy || !dv || !work) {
        jb->status = -1;
        goto done;
    }
    for (int j = 0; j < R; ++j) q[j] = load_elem(jb->q, jb->bf16, (size_t)j);
    for (int j = 0; j < D; ++j)
        w[j] = (jb->out_norm && jb->w_o) ? load_elem(jb->w_o, jb->bf16, (size_t)j) : 1.0;
    for (long n = jb->n0; n < jb->n1; ++n) {
        for (int s = 0; s < S; ++s)
            for (int j = 0; j < D; ++j)
                v[(size_t)s * D + j] =
                    load_elem(jb->src, jb->bf16, ((size_t)s * N + n) * D + j);
        const int want_bwd = jb->dy != NULL;
        if (want_bwd)
            for (int j = 0; j < D; ++j)
                dy[j] = load_elem(jb->dy, jb->bf16, (size_t)n * D + j);
        token_oracle(S, D, R, jb->ko, jb->eps, jb->scale, jb->out_norm, v, q, w,
                     jb->y ? jb->y + (size_t)n * D : NULL,
                     jb->alpha ? jb->alpha + (size_t)n * S : NULL,
                     jb->rstd ? jb->rstd + (size_t)n * S : NULL,
                     jb->logit ? jb->logit + (size_t)n * S : NULL,
                     jb->o_rstd ? jb->o_rstd + n : NULL, want_bwd ? dy : NULL,
                     dv, jb->dq, jb->dw_o, work);
        if (want_bwd && jb->dsrc)
            for (int s = 0; s < S; ++s)
                memcpy(jb->dsrc + ((size_t)s * N + n) * D, dv + (size_t)s * D,
                       sizeof(double) * (size_t)D);
    }
    jb->status = 0;
done:
    free(v); free(q); free(w); free(dy); free(dv); free(work);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments or allocation failure. */
static int run_all(int S, long N, int D, int R, int ko, double eps, double scale,
                   int out_norm, int bf16, const void *src, const void *q,
                   const void *w_o, const void *dy, double *y, double *alpha,
                   double *rstd, double *logit, double *o_rstd, double *dsrc,
                   double *dq, double *dw_o, int nthreads) {
    if (S < 1 || N < 0 || D < 1 || R < 1 || R > D || ko < 0 || ko + R > D) return -1;
    if (!src || !q || (out_norm && !w_o)) return -1;
    if (nthreads < 1) nthreads = 1;
    if ((long)nthreads > N) nthreads = N > 0 ? (int)N : 1;
    job_t *jobs = calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = calloc((size_t)nthreads, sizeof(pthread_t));
    double *part = calloc((size_t)nthreads * (size_t)(R + D), sizeof(double));
    if (!jobs || !th || !part) {
        free(jobs); free(th); free(part);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        job_t *jb = &jobs[t];
        jb->S = S; jb->D = D; jb->R = R; jb->ko = ko; jb->out_norm = out_norm;
        jb->bf16 = bf16; jb->N = N; jb->eps = eps; jb->scale = scale;
        jb->n0 = N * t / nthreads;
        jb->n1 = N * (t + 1) / nthreads;
        jb->src = src; jb->q = q; jb->w_o = w_o; jb->dy = dy;
        jb->y = y; jb->alpha = alpha; jb->rstd = rstd; jb->logit = logit;
        jb->o_rstd = o_rstd; jb->dsrc = dsrc;
        jb->dq = part + (size_t)t * (R + D);
        jb->dw_o = jb->dq + R;
        jb->status = -1;
    }
    int spawned = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, run_range, &jobs[t]) == 0) spawned = t;
        else break;
    run_range(&jobs[0]);
    for (int t = 1; t <= spawned; ++t) pthread_join(th[t], NULL);
    /* threads that failed to spawn run here, in order */
    for (int t = spawned + 1; t < nthreads; ++t) run_range(&jobs[t]);
    int rc = 0;
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != 0) rc = -1;
    if (dy) {
        if (dq)
            for (int j = 0; j < R; ++j) {
                double acc = 0.0;
                for (int t = 0; t < nthreads; ++t) acc += part[(size_t)t * (R + D) + j];
                dq[j] = acc;
            }
        if (dw_o)
            for (int j = 0; j < D; ++j) {
                double acc = 0.0;
                for (int t = 0; t < nthreads; ++t) acc += part[(size_t)t * (R + D) + R + j];
                dw_o[j] = acc;
            }
    }
    free(jobs); free(th); free(part);
    return rc;
}

/* Public entry points (C ABI, host memory only).
 *   *_bf16: src [S][N][D], q [R], w_o [D], dy [N][D] are bf16 bit patterns.
 *   *_f64 : the same arrays in double (used for finite differences).
 * Pass dy = NULL for forward only.  Any output pointer may be NULL. */
int attnres_oracle_bf16(int S, long N, int D, int R, int key_offset, double eps,
                        double scale, int out_norm, const uint16_t *src,
                        const uint16_t *q, const uint16_t *w_o, const uint16_t *dy,
                        double *y, double *alpha, double *rstd, double *logit,
                        double *o_rstd, double *dsrc, double *dq, double *dw_o,
                        int nthreads) {
    return run_all(S, N, D, R, key_offset, eps, scale, out_norm, 1, src, q, w_o, dy,
                   y, alpha, rstd, logit, o_rstd, dsrc, dq, dw_o, nthreads);
}

int attnres_oracle_f64(int S, long N, int D, int R, int key_offset, double eps,
                       double scale, int out_norm, const double *src, const double *q,
                       const double *w_o, const double *dy, double *y, double *alpha,
                       double *rstd, double *logit, double *o_rstd, double *dsrc,
                       double *dq, double *dw_o, int nthreads) {
    return run_all(S, N, D, R, key_offset, eps, scale, out_norm, 0, src, q, w_o, dy,
                   y, alpha, rstd, logit, o_rstd, dsrc, dq, dw_o, nthreads);
}

/*
 * attn_oracle.c -- plain, slow fp64 CPU reference for exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library may link, load
 * or call this file; only the test suite, the bench's cpu_baseline leg and
 * the smoke check use it, to judge the CUDA kernels.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * Sources (cited below by these short names):
 *   [hyper] hyper.ai story on FlashAttention-4 (German), single paragraph:
 *           FA4 speeds attention up "without touching the mathematical
 *           accuracy", i.e. the result is exact softmax attention.
 *   [nl]    "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
 *           Asymmetric Hardware Scaling" (gist.science/nl), section
 *           "Technische samenvatting": Probleemstelling (attention is the
 *           bottleneck), Methodologie §1 (O accumulated from softmax(S) V),
 *           Methodologie §3 (backward pass: gradients, dQ reduced by atomic
 *           additions).
 *
 * What is computed is the textbook definition, written out:
 *   forward, per head and query row i, visible keys V_i = {j : j <= i} when
 *   causal, all j otherwise:
 *       s_ij  = scale * sum_d Q[i,d] K[j,d]
 *       m_i   = max_{j in V_i} s_ij
 *       Z_i   = sum_{j in V_i} exp(s_ij - m_i)
 *       P_ij  = exp(s_ij - m_i) / Z_i             (0 for j not in V_i)
 *       O_i   = sum_j P_ij V_j
 *       LSE_i = m_i + ln Z_i                      (natural log, scaled scores)
 *   backward, for the loss whose gradient w.r.t. O is dO:
 *       dV_j  = sum_i P_ij dO_i
 *       dP_ij = dO_i . V_j
 *       Delta_i = sum_j P_ij dP_ij                (softmax Jacobian term)
 *       dS_ij = P_ij (dP_ij - Delta_i)
 *       dQ_i  = scale * sum_j dS_ij K_j
 *       dK_j  = scale * sum_i dS_ij Q_i
 *
 * Each row of S is formed explicitly and the softmax is the explicit two-pass
 * form (max, then exponentials and their sum); nothing is computed online.
 * All arrays are one head, row-major: Q/K/V/dO/O are [S][D], LSE/Delta [S].
 * Parallelism (OpenMP) is over independent rows or columns only and does not
 * change any summation order: every sum runs over its index in natural order.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* 1 when key j is visible to query i. */
static int visible(long i, long j, int causal) { return !causal || j <= i; }

/* number of keys visible to query i */
static long n_visible(long i, long S, int causal) { return causal ? i + 1 : S; }

/* kt[d*S + j] = k[j*D + d]: a transposed copy so the score row below is a
 * loop over contiguous memory.  Pure data movement. */
static double *transpose(const double *k, long S, long D) {
    double *kt = (double *)malloc(sizeof(double) * (size_t)S * (size_t)D);
    if (!kt) return NULL;
    for (long j = 0; j < S; ++j)
        for (long d = 0; d < D; ++d) kt[d * S + j] = k[j * D + d];
    return kt;
}

/* s[j] = scale * sum_d q_i[d] k[j,d] for the n visible keys j < n.
 * The sum over d runs in order d = 0..D-1 for every j. */
static void score_row(const double *qi, const double *kt, long S, long D, long n,
                      double scale, double *s) {
    for (long j = 0; j < n; ++j) s[j] = 0.0;
    for (long d = 0; d < D; ++d) {
        const double qd = qi[d];
        const double *kd = kt + d * S;
        for (long j = 0; j < n; ++j) s[j] += qd * kd[j];
    }
    for (long j = 0; j < n; ++j) s[j] *= scale;
}

/* Explicit two-pass softmax of one score row: p[j] = exp(s[j]-m)/Z, and
 * returns LSE = m + ln Z. */
static double softmax_row(const double *s, long n, double *p) {
    double m = -INFINITY;
    for (long j = 0; j < n; ++j) if (s[j] > m) m = s[j];
    double z = 0.0;
    for (long j = 0; j < n; ++j) { p[j] = exp(s[j] - m); z += p[j]; }
    for (long j = 0; j < n; ++j) p[j] /= z;
    return m + log(z);
}

/*
 * Forward for a list of query rows (rows == NULL means all S rows, in order).
 * o_rows [nrows][D], lse_rows [nrows].  Returns 0, or -1 on allocation failure.
 */
int fa_oracle_fwd(const double *q, const double *k, const double *v, long S, long D,
                  int causal, double scale, const long *rows, long nrows,
                  double *o_rows, double *lse_rows) {
    if (rows == NULL) nrows = S;
    double *kt = transpose(k, S, D);
    if (!kt) return -1;
    int fail = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S);
        double *p = (double *)malloc(sizeof(double) * (size_t)S);
        if (!s || !p) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long r = 0; r < nrows; ++r) {
                const long i = rows ? rows[r] : r;
                const long n = n_visible(i, S, causal);
                score_row(q + i * D, kt, S, D, n, scale, s);
                lse_rows[r] = softmax_row(s, n, p);
                double *o = o_rows + r * D;
                for (long d = 0; d < D; ++d) o[d] = 0.0;
                for (long j = 0; j < n; ++j) {
                    const double pj = p[j];
                    const double *vj = v + j * D;
                    for (long d = 0; d < D; ++d) o[d] += pj * vj[d];
                }
            }
        }
        free(s);
        free(p);
    }
    free(kt);
    return fail ? -1 : 0;
}

/*
 * Row statistics for the backward pass, for the listed rows (rows == NULL:
 * every row i of the head, in order):
 *   lse[r]   = LSE_i (as in the forward),
 *   delta[r] = Delta_i = sum_j P_ij dP_ij with dP_ij = dO_i . V_j,
 *   o (optional, may be NULL) row r = O_i, the exact forward output.
 */
int fa_oracle_bwd_stats(const double *q, const double *k, const double *v,
                        const double *dout, long S, long D, int causal, double scale,
                        const long *rows, long nrows, double *lse, double *delta, double *o) {
    if (rows == NULL) nrows = S;
    double *kt = transpose(k, S, D);
    double *vt = transpose(v, S, D);
    if (!kt || !vt) { free(kt); free(vt); return -1; }
    int fail = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S);
        double *p = (double *)malloc(sizeof(double) * (size_t)S);
        double *dp = (double *)malloc(sizeof(double) * (size_t)S);
        if (!s || !p || !dp) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long r = 0; r < nrows; ++r) {
                const long i = rows ? rows[r] : r;
                const long n = n_visible(i, S, causal);
                score_row(q + i * D, kt, S, D, n, scale, s);
                lse[r] = softmax_row(s, n, p);
                /* dP_ij = dO_i . V_j (no scale: dP is the gradient w.r.t. P) */
                score_row(dout + i * D, vt, S, D, n, 1.0, dp);
                double acc = 0.0;
                for (long j = 0; j < n; ++j) acc += p[j] * dp[j];
                delta[r] = acc;
                if (o) {
                    double *oi = o + r * D;
                    for (long d = 0; d < D; ++d) oi[d] = 0.0;
                    for (long j = 0; j < n; ++j)
                        for (long d = 0; d < D; ++d) oi[d] += p[j] * v[j * D + d];
                }
            }
        }
        free(s);
        free(p);
        free(dp);
    }
    free(kt);
    free(vt);
    return fail ? -1 : 0;
}

/*
 * dQ for a list of rows (NULL = all rows), given the oracle's own lse/delta
 * from fa_oracle_bwd_stats.  P_ij = exp(s_ij - LSE_i) is the softmax of the
 * row (exp(s - m)/Z == exp(s - (m + ln Z))).
 */
int fa_oracle_bwd_dq(const double *q, const double *k, const double *v,
                     const double *dout, const double *lse, const double *delta,
                     long S, long D, int causal, double scale,
                     const long *rows, long nrows, double *dq_rows) {
    if (rows == NULL) nrows = S;
    double *kt = transpose(k, S, D);
    double *vt = transpose(v, S, D);
    if (!kt || !vt) { free(kt); free(vt); return -1; }
    int fail = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S);
        double *dp = (double *)malloc(sizeof(double) * (size_t)S);
        if (!s || !dp) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long r = 0; r < nrows; ++r) {
                const long i = rows ? rows[r] : r;
                const long n = n_visible(i, S, causal);
                score_row(q + i * D, kt, S, D, n, scale, s);
                score_row(dout + i * D, vt, S, D, n, 1.0, dp);
                double *g = dq_rows + r * D;
                for (long d = 0; d < D; ++d) g[d] = 0.0;
                for (long j = 0; j < n; ++j) {
                    const double pij = exp(s[j] - lse[i]);
                    const double dsij = pij * (dp[j] - delta[i]);
                    const double *kj = k + j * D;
                    for (long d = 0; d < D; ++d) g[d] += dsij * kj[d];
                }
                for (long d = 0; d < D; ++d) g[d] *= scale;
            }
        }
        free(s);
        free(dp);
    }
    free(kt);
    free(vt);
    return fail ? -1 : 0;
}

/*
 * dK and dV for a list of key columns (NULL = all), given the oracle's own
 * lse/delta.  For column j the sums run over the queries i that see key j.
 */
int fa_oracle_bwd_dkdv(const double *q, const double *k, const double *v,
                       const double *dout, const double *lse, const double *delta,
                       long S, long D, int causal, double scale,
                       const long *cols, long ncols, double *dk_cols, double *dv_cols) {
    if (cols == NULL) ncols = S;
    int fail = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S);
        double *dp = (double *)malloc(sizeof(double) * (size_t)S);
        if (!s || !dp) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long c = 0; c < ncols; ++c) {
                const long j = cols ? cols[c] : c;
                const double *kj = k + j * D;
                const double *vj = v + j * D;
                double *gk = dk_cols + c * D;
                double *gv = dv_cols + c * D;
                for (long d = 0; d < D; ++d) { gk[d] = 0.0; gv[d] = 0.0; }
                for (long i = 0; i < S; ++i) {
                    if (!visible(i, j, causal)) continue;
                    const double *qi = q + i * D;
                    const double *doi = dout + i * D;
                    double sij = 0.0, dpij = 0.0;
                    for (long d = 0; d < D; ++d) sij += qi[d] * kj[d];
                    for (long d = 0; d < D; ++d) dpij += doi[d] * vj[d];
                    sij *= scale;
                    const double pij = exp(sij - lse[i]);
                    const double dsij = pij * (dpij - delta[i]);
                    for (long d = 0; d < D; ++d) {
                        gv[d] += pij * doi[d];
                        gk[d] += dsij * qi[d];
                    }
                }
                for (long d = 0; d < D; ++d) gk[d] *= scale;
            }
        }
        free(s);
        free(dp);
    }
    return fail ? -1 : 0;
}

/* Reference 2^x for the exp2 approximation checks: the C library's exp2 in
 * double precision, elementwise. */
void fa_oracle_exp2(const double *x, double *y, long n) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) y[i] = exp2(x[i]);
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int fa_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

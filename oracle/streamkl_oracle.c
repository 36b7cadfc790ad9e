/*
 * streamkl_oracle.c -- float64 CPU oracle for the attention KL divergence.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this library.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Source: "StreamKL: Fast and Memory-Efficient KL Divergence for Boosting
 * Attention Distillation" (gist.science/paper/2606.20005, technical summary).
 * Each function names the section it follows.  The method is an exact
 * reformulation, so the oracle is the plain definition, written row by row
 * in float64 with nothing fused or blocked:
 *
 *   S_t[i,j] = scale * <Q_t[i,:], K_t[j,:]>           t = 1 (teacher), 2 (student)
 *   P_t[i,:] = softmax over the visible keys of row i
 *   KL[i]    = sum_j P1[i,j] * (log P1[i,j] - log P2[i,j])
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - natural logarithm throughout; LSE_t[i] = log sum_j exp(S_t[i,j]);
 *   - causal rows are aligned bottom-right: row i sees keys j <= i + Nk - Nq;
 *   - gradients are the true derivatives of sum_i g[i]*KL[i], including the
 *     softmax scale (chain rule through S = scale * Q K^T).
 *
 * Layout of every tensor: contiguous [B, H, N, d] (d fastest), float64.
 * Outputs KL/LSE are [B, H, Nq]; dQ is [B, H, Nq, d]; dK is [B, H, Nk, d].
 * Every entry point returns 0 on success and a negative value on bad
 * arguments (it never aborts).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Small helpers: nothing here is specific to the method.                    */
/* ------------------------------------------------------------------------ */

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

static double dot(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int k = 0; k < d; ++k) s += a[k] * b[k];
    return s;
}

/* Number of keys row i may attend to (keys 0 .. n-1).  Non-causal: all Nk.
 * Causal, bottom-right aligned: keys j <= i + (Nk - Nq). */
static int64_t visible_keys(int64_t i, int64_t Nq, int64_t Nk, int causal) {
    if (!causal) return Nk;
    int64_t n = i + (Nk - Nq) + 1;
    if (n < 0) n = 0;
    if (n > Nk) n = Nk;
    return n;
}

static int check_dims(int B, int H, int64_t Nq, int64_t Nk, int d, int causal) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return -1;
    if (causal && Nq > Nk) return -2;  /* a row would see no key at all */
    return 0;
}

/* ------------------------------------------------------------------------ */
/* One query row, by definition (Problem Statement: row-wise KL of two        */
/* attention distributions; Methodology 1: LSE_t = log sum exp S_t).          */
/* ------------------------------------------------------------------------ */

typedef struct {
    double lse1, lse2, kl;
} row_stats;

/* Scores of row i against its n visible keys, for one head. */
static void row_scores(const double* q1, const double* K1h, const double* q2, const double* K2h,
                       int64_t n, int d, double scale, double* S1, double* S2) {
    for (int64_t j = 0; j < n; ++j) {
        S1[j] = scale * dot(q1, K1h + j * d, d);
        S2[j] = scale * dot(q2, K2h + j * d, d);
    }
}

/* log sum_j exp(S[j]) in two passes: the maximum first, then the shifted sum. */
static double log_sum_exp(const double* S, int64_t n) {
    double M = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (S[j] > M) M = S[j];
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) sum += exp(S[j] - M);
    return M + log(sum);
}

/* KL(P1 || P2) for one row with log P_t = S_t - LSE_t. */
static row_stats row_kl(const double* S1, const double* S2, int64_t n) {
    row_stats r;
    r.lse1 = log_sum_exp(S1, n);
    r.lse2 = log_sum_exp(S2, n);
    double kl = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double logp1 = S1[j] - r.lse1;
        double logp2 = S2[j] - r.lse2;
        kl += exp(logp1) * (logp1 - logp2);
    }
    r.kl = kl;
    return r;
}

/* Row statistics of flat row index r in [0, B*H*Nq). */
static row_stats compute_row(int H, int64_t Nq, int64_t Nk, int d, const double* Q1, const double* K1,
                             const double* Q2, const double* K2, double scale, int causal, int64_t r,
                             double* S1, double* S2) {
    int64_t bh = r / Nq, i = r % Nq;
    (void)H;
    const double* q1 = Q1 + r * d;
    const double* q2 = Q2 + r * d;
    const double* K1h = K1 + bh * Nk * d;
    const double* K2h = K2 + bh * Nk * d;
    int64_t n = visible_keys(i, Nq, Nk, causal);
    row_scores(q1, K1h, q2, K2h, n, d, scale, S1, S2);
    return row_kl(S1, S2, n);
}

/* ------------------------------------------------------------------------ */
/* Forward: KL, LSE1, LSE2 per row (Methodology 2: only these are saved).    */
/* ------------------------------------------------------------------------ */

/* All rows.  nthreads <= 0 keeps the OpenMP default. */
int oracle_fwd(int B, int H, int64_t Nq, int64_t Nk, int d, const double* Q1, const double* K1,
               const double* Q2, const double* K2, double scale, int causal, double* KL, double* LSE1,
               double* LSE2, int nthreads) {
    int rc = check_dims(B, H, Nq, Nk, d, causal);
    if (rc) return rc;
    set_threads(nthreads);
    int64_t rows = (int64_t)B * H * Nq;
    int failed = 0;
#pragma omp parallel
    {
        double* S1 = (double*)malloc(sizeof(double) * Nk);
        double* S2 = (double*)malloc(sizeof(double) * Nk);
        if (!S1 || !S2) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < rows; ++r) {
                row_stats s = compute_row(H, Nq, Nk, d, Q1, K1, Q2, K2, scale, causal, r, S1, S2);
                KL[r] = s.kl;
                LSE1[r] = s.lse1;
                LSE2[r] = s.lse2;
            }
        }
        free(S1);
        free(S2);
    }
    return failed ? -3 : 0;
}

/* Selected rows only: rows[k] is a flat index into [B, H, Nq]; outputs are
 * packed in the order of rows[]. */
int oracle_fwd_rows(int B, int H, int64_t Nq, int64_t Nk, int d, const double* Q1, const double* K1,
                    const double* Q2, const double* K2, double scale, int causal, int64_t nrows,
                    const int64_t* rows, double* KL, double* LSE1, double* LSE2, int nthreads) {
    int rc = check_dims(B, H, Nq, Nk, d, causal);
    if (rc) return rc;
    int64_t total = (int64_t)B * H * Nq;
    for (int64_t k = 0; k < nrows; ++k)
        if (rows[k] < 0 || rows[k] >= total) return -4;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        double* S1 = (double*)malloc(sizeof(double) * Nk);
        double* S2 = (double*)malloc(sizeof(double) * Nk);
        if (!S1 || !S2) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t k = 0; k < nrows; ++k) {
                row_stats s = compute_row(H, Nq, Nk, d, Q1, K1, Q2, K2, scale, causal, rows[k], S1, S2);
                KL[k] = s.kl;
                LSE1[k] = s.lse1;
                LSE2[k] = s.lse2;
            }
        }
        free(S1);
        free(S2);
    }
    return failed ? -3 : 0;
}

/* ------------------------------------------------------------------------ */
/* Online recurrence (Methodology 1, "Online Formulation").  Five running    */
/* scalars per row -- m1, m2, l1, l2, acc -- updated one key tile of width    */
/* BK at a time; acc is rescaled with the teacher maximum only.  Finish:      */
/* KL = acc / l1 + LSE2 - LSE1 with LSE_t = m_t + log l_t.  The oracle uses   */
/* this only to check that the recurrence reproduces the definition.          */
/* ------------------------------------------------------------------------ */

int oracle_online_fwd(int B, int H, int64_t Nq, int64_t Nk, int d, const double* Q1, const double* K1,
                      const double* Q2, const double* K2, double scale, int causal, int64_t BK, double* KL,
                      double* LSE1, double* LSE2, int nthreads) {
    int rc = check_dims(B, H, Nq, Nk, d, causal);
    if (rc) return rc;
    if (BK < 1) return -5;
    set_threads(nthreads);
    int64_t rows = (int64_t)B * H * Nq;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t bh = r / Nq, i = r % Nq;
        const double* q1 = Q1 + r * d;
        const double* q2 = Q2 + r * d;
        const double* K1h = K1 + bh * Nk * d;
        const double* K2h = K2 + bh * Nk * d;
        int64_t n = visible_keys(i, Nq, Nk, causal);
        double m1 = -INFINITY, m2 = -INFINITY, l1 = 0.0, l2 = 0.0, acc = 0.0;
        for (int64_t j0 = 0; j0 < n; j0 += BK) {
            int64_t j1 = j0 + BK < n ? j0 + BK : n;
            /* new maxima over the tile */
            double t1 = -INFINITY, t2 = -INFINITY;
            for (int64_t j = j0; j < j1; ++j) {
                double s1 = scale * dot(q1, K1h + j * d, d);
                double s2 = scale * dot(q2, K2h + j * d, d);
                if (s1 > t1) t1 = s1;
                if (s2 > t2) t2 = s2;
            }
            double m1n = m1 > t1 ? m1 : t1;
            double m2n = m2 > t2 ? m2 : t2;
            double a1 = exp(m1 - m1n); /* exp(-inf) = 0 on the first tile */
            double a2 = exp(m2 - m2n);
            double sum1 = 0.0, sum2 = 0.0, sumacc = 0.0;
            for (int64_t j = j0; j < j1; ++j) {
                double s1 = scale * dot(q1, K1h + j * d, d);
                double s2 = scale * dot(q2, K2h + j * d, d);
                double e1 = exp(s1 - m1n);
                sum1 += e1;
                sum2 += exp(s2 - m2n);
                sumacc += e1 * (s1 - s2);
            }
            l1 = a1 * l1 + sum1;
            l2 = a2 * l2 + sum2;
            acc = a1 * acc + sumacc;
            m1 = m1n;
            m2 = m2n;
        }
        double lse1 = m1 + log(l1), lse2 = m2 + log(l2);
        LSE1[r] = lse1;
        LSE2[r] = lse2;
        KL[r] = acc / l1 + lse2 - lse1;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward (Methodology 2, "Recomputation Strategy", two settings).         */
/*   setting 1: P1 fixed, gradients to the student (Q2, K2):                 */
/*              dS2[i,j] = g[i] * (P2[i,j] - P1[i,j])                         */
/*   setting 2: P2 fixed, gradients to the teacher (Q1, K1):                 */
/*              dS1[i,j] = g[i] * P1[i,j] * (log P1 - log P2 - KL[i])         */
/*              with log P_t = S_t - LSE_t (logit differences, never log P).  */
/*   dQ[i] = scale * sum_j dS[i,j] K[j],  dK[j] = scale * sum_i dS[i,j] Q[i]  */
/* ------------------------------------------------------------------------ */

static double dscore(int setting, double g, double s1, double s2, row_stats st) {
    double logp1 = s1 - st.lse1, logp2 = s2 - st.lse2;
    double p1 = exp(logp1);
    if (setting == 1) return g * (exp(logp2) - p1);
    return g * p1 * (logp1 - logp2 - st.kl);
}

/* dQ of the trainable side for the query rows listed (flat into [B,H,Nq]);
 * output packed [nrows, d]. */
static int bwd_dq_rows(int setting, int B, int H, int64_t Nq, int64_t Nk, int d, const double* g,
                       const double* Q1, const double* K1, const double* Q2, const double* K2, double scale,
                       int causal, int64_t nrows, const int64_t* rows, double* dQ) {
    const double* Kt = setting == 1 ? K2 : K1;
    int failed = 0;
    (void)B;
#pragma omp parallel
    {
        double* S1 = (double*)malloc(sizeof(double) * Nk);
        double* S2 = (double*)malloc(sizeof(double) * Nk);
        if (!S1 || !S2) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t k = 0; k < nrows; ++k) {
                int64_t r = rows[k], bh = r / Nq, i = r % Nq;
                row_stats st = compute_row(H, Nq, Nk, d, Q1, K1, Q2, K2, scale, causal, r, S1, S2);
                int64_t n = visible_keys(i, Nq, Nk, causal);
                double* out = dQ + k * d;
                for (int c = 0; c < d; ++c) out[c] = 0.0;
                for (int64_t j = 0; j < n; ++j) {
                    double ds = dscore(setting, g[r], S1[j], S2[j], st);
                    const double* kj = Kt + (bh * Nk + j) * d;
                    for (int c = 0; c < d; ++c) out[c] += scale * ds * kj[c];
                }
            }
        }
        free(S1);
        free(S2);
    }
    return failed ? -3 : 0;
}

/* dK of the trainable side for the key rows listed (flat into [B,H,Nk]);
 * output packed [nkeys, d].  Row statistics (LSE1, LSE2, KL) are computed,
 * by definition, for every query row that sees one of the listed keys. */
static int bwd_dk_keys(int setting, int B, int H, int64_t Nq, int64_t Nk, int d, const double* g,
                       const double* Q1, const double* K1, const double* Q2, const double* K2, double scale,
                       int causal, int64_t nkeys, const int64_t* keys, double* dK) {
    const double* Qt = setting == 1 ? Q2 : Q1;
    int64_t BH = (int64_t)B * H;
    /* lowest key index listed per head, so that only the rows that can see a
     * listed key get their statistics computed */
    int64_t* jmin = (int64_t*)malloc(sizeof(int64_t) * BH);
    row_stats* st = (row_stats*)malloc(sizeof(row_stats) * BH * Nq);
    if (!jmin || !st) {
        free(jmin);
        free(st);
        return -3;
    }
    for (int64_t h = 0; h < BH; ++h) jmin[h] = Nk;
    for (int64_t k = 0; k < nkeys; ++k) {
        int64_t bh = keys[k] / Nk, j = keys[k] % Nk;
        if (j < jmin[bh]) jmin[bh] = j;
    }
    int failed = 0;
#pragma omp parallel
    {
        double* S1 = (double*)malloc(sizeof(double) * Nk);
        double* S2 = (double*)malloc(sizeof(double) * Nk);
        if (!S1 || !S2) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < BH * Nq; ++r) {
                int64_t bh = r / Nq, i = r % Nq;
                if (jmin[bh] >= Nk || visible_keys(i, Nq, Nk, causal) <= jmin[bh]) continue;
                st[r] = compute_row(H, Nq, Nk, d, Q1, K1, Q2, K2, scale, causal, r, S1, S2);
            }
        }
        free(S1);
        free(S2);
    }
    if (!failed) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t k = 0; k < nkeys; ++k) {
            int64_t bh = keys[k] / Nk, j = keys[k] % Nk;
            double* out = dK + k * d;
            for (int c = 0; c < d; ++c) out[c] = 0.0;
            const double* k1 = K1 + (bh * Nk + j) * d;
            const double* k2 = K2 + (bh * Nk + j) * d;
            for (int64_t i = 0; i < Nq; ++i) {
                if (visible_keys(i, Nq, Nk, causal) <= j) continue; /* row i does not see key j */
                int64_t r = bh * Nq + i;
                double s1 = scale * dot(Q1 + r * d, k1, d);
                double s2 = scale * dot(Q2 + r * d, k2, d);
                double ds = dscore(setting, g[r], s1, s2, st[r]);
                const double* qi = Qt + r * d;
                for (int c = 0; c < d; ++c) out[c] += scale * ds * qi[c];
            }
        }
    }
    free(jmin);
    free(st);
    return failed ? -3 : 0;
}

/* Full backward: dQ [B,H,Nq,d] and dK [B,H,Nk,d] of the trainable side.
 * g is the upstream gradient dL/dKL, one value per row [B,H,Nq]. */
int oracle_bwd(int setting, int B, int H, int64_t Nq, int64_t Nk, int d, const double* g, const double* Q1,
               const double* K1, const double* Q2, const double* K2, double scale, int causal, double* dQ,
               double* dK, int nthreads) {
    int rc = check_dims(B, H, Nq, Nk, d, causal);
    if (rc) return rc;
    if (setting != 1 && setting != 2) return -6;
    set_threads(nthreads);
    int64_t nr = (int64_t)B * H * Nq, nk = (int64_t)B * H * Nk;
    int64_t* idx = (int64_t*)malloc(sizeof(int64_t) * (nr > nk ? nr : nk));
    if (!idx) return -3;
    for (int64_t k = 0; k < nr; ++k) idx[k] = k;
    rc = bwd_dq_rows(setting, B, H, Nq, Nk, d, g, Q1, K1, Q2, K2, scale, causal, nr, idx, dQ);
    if (!rc) {
        for (int64_t k = 0; k < nk; ++k) idx[k] = k;
        rc = bwd_dk_keys(setting, B, H, Nq, Nk, d, g, Q1, K1, Q2, K2, scale, causal, nk, idx, dK);
    }
    free(idx);
    return rc;
}

/* dQ for selected query rows (flat into [B,H,Nq]); output packed [nrows, d]. */
int oracle_bwd_dq_rows(int setting, int B, int H, int64_t Nq, int64_t Nk, int d, const double* g,
                       const double* Q1, const double* K1, const double* Q2, const double* K2, double scale,
                       int causal, int64_t nrows, const int64_t* rows, double* dQ, int nthreads) {
    int rc = check_dims(B, H, Nq, Nk, d, causal);
    if (rc) return rc;
    if (setting != 1 && setting != 2) return -6;
    int64_t total = (int64_t)B * H * Nq;
    for (int64_t k = 0; k < nrows; ++k)
        if (rows[k] < 0 || rows[k] >= total) return -4;
    set_threads(nthreads);
    return bwd_dq_rows(setting, B, H, Nq, Nk, d, g, Q1, K1, Q2, K2, scale, causal, nrows, rows, dQ);
}

/* dK for selected key rows (flat into [B,H,Nk]); output packed [nkeys, d]. */
int oracle_bwd_dk_keys(int setting, int B, int H, int64_t Nq, int64_t Nk, int d, const double* g,
                       const double* Q1, const double* K1, const double* Q2, const double* K2, double scale,
                       int causal, int64_t nkeys, const int64_t* keys, double* dK, int nthreads) {
    int rc = check_dims(B, H, Nq, Nk, d, causal);
    if (rc) return rc;
    if (setting != 1 && setting != 2) return -6;
    int64_t total = (int64_t)B * H * Nk;
    for (int64_t k = 0; k < nkeys; ++k)
        if (keys[k] < 0 || keys[k] >= total) return -4;
    set_threads(nthreads);
    return bwd_dk_keys(setting, B, H, Nq, Nk, d, g, Q1, K1, Q2, K2, scale, causal, nkeys, keys, dK);
}

/* Threads the OpenMP runtime will use (for reporting the baseline's cores). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

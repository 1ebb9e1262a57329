/*
 * Oracle for exact multi-head scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, fp64 CPU statement of what the
 * GPU path computes.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may build, load or call it; the library under self_attention_gb300/ never does, and the
 * two share no code.
 *
 * Source: "Self-attention, CUDA kernels and FlashAttention" (2026-11-15), section 1
 * "How self-attention works mathematically in a Vision Transformer":
 *   scores   S = Q K^T / sqrt(d_k)               (the "Scores" formula)
 *   weights  P = softmax(S), taken row by row     (each row of probabilities sums to one)
 *   output   O = P V                              (the "Attention(Q,K,V)" formula)
 *   heads    the same computation, independently, for every head (e.g. 12 heads).
 * Section 3 of the same article ("Recomputation in backpropagation") says the backward pass
 * keeps only small per-row normalisation statistics; here that statistic is the natural-log
 * log-sum-exp of each row of S, LSE_i = log sum_j exp(S_ij).
 * The article prints no backward formulas; the gradients below are the chain rule applied to
 * the three formulas above (with L a scalar loss and dO = dL/dO):
 *   dV = P^T dO
 *   dP = dO V^T
 *   dS = P o (dP - D 1^T),  D_i = sum_j P_ij dP_ij = sum_c dO_ic O_ic
 *   dQ = scale * dS K,      dK = scale * dS^T Q       (scale = 1/sqrt(d_k), inside S)
 *
 * Every tensor is [BH, N, d] row-major fp64 (BH = batch x heads).  The score matrix is
 * materialised in full, N x N per head, exactly as the definition reads; heads are processed
 * one after another and rows of one head in parallel (OpenMP), which changes nothing but the
 * wall time.  The caller widens bf16 inputs to fp64 before the call; `scale` is the same
 * fp32 value the GPU path receives, widened to fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* exp of every score minus the row maximum, then divided by their sum: the row softmax of
 * section 1 ("Softmax weighting and aggregation"), written the numerically safe way (the
 * common factor exp(-max) cancels).  Returns the row's log-sum-exp. */
static double softmax_row(const double *s, double *p, int64_t n)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (s[j] > m) m = s[j];
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        p[j] = exp(s[j] - m);
        sum += p[j];
    }
    for (int64_t j = 0; j < n; ++j) p[j] /= sum;
    return m + log(sum);
}

static double dot(const double *a, const double *b, int64_t d)
{
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += a[c] * b[c];
    return acc;
}

/* S = scale * Q K^T for one head (the "Scores" formula), into an N x N buffer. */
static void scores(const double *q, const double *k, double *s, int64_t n, int64_t d, double scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j)
            s[i * n + j] = scale * dot(q + i * d, k + j * d, d);
}

/* P (in place over S) and LSE, row by row. */
static void softmax_rows(double *s_to_p, double *lse, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double *row = s_to_p + i * n;
        lse[i] = softmax_row(row, row, n);
    }
}

/* O = P V: O_i = sum_j P_ij V_j (the "Attention(Q,K,V)" formula). */
static void weighted_values(const double *p, const double *v, double *o, int64_t n, int64_t d)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double *oi = o + i * d;
        for (int64_t c = 0; c < d; ++c) oi[c] = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            const double pij = p[i * n + j];
            const double *vj = v + j * d;
            for (int64_t c = 0; c < d; ++c) oi[c] += pij * vj[c];
        }
    }
}

/* Forward for all heads: o [BH,N,d], lse [BH,N]. Returns 0, or -1 if memory ran out. */
int oracle_attn_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
                    int64_t bh, int64_t n, int64_t d, double scale)
{
    double *s = (double *)malloc((size_t)(n * n) * sizeof(double));
    if (!s) return -1;
    for (int64_t h = 0; h < bh; ++h) {
        const int64_t off = h * n * d;
        scores(q + off, k + off, s, n, d, scale);
        softmax_rows(s, lse + h * n, n);
        weighted_values(s, v + off, o + off, n, d);
    }
    free(s);
    return 0;
}

/* Forward and backward for all heads.  Outputs: dq, dk, dv [BH,N,d]; o [BH,N,d] and lse [BH,N]
 * (the oracle's own fp64 forward); dvec [BH,N] = rowsum(dO o O); dprime [BH,N] = rowsum(P o dP),
 * the same quantity by its other definition, returned so that callers can check the two agree.
 * Returns 0, or -1 if memory ran out. */
int oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                    double *dq, double *dk, double *dv, double *o, double *lse, double *dvec,
                    double *dprime, int64_t bh, int64_t n, int64_t d, double scale)
{
    double *p = (double *)malloc((size_t)(n * n) * sizeof(double));
    double *ds = (double *)malloc((size_t)(n * n) * sizeof(double));
    if (!p || !ds) {
        free(p);
        free(ds);
        return -1;
    }
    for (int64_t h = 0; h < bh; ++h) {
        const int64_t off = h * n * d;
        const double *qh = q + off, *kh = k + off, *vh = v + off, *doh = dout + off;
        double *oh = o + off, *dqh = dq + off, *dkh = dk + off, *dvh = dv + off;
        double *lh = lse + h * n, *dh = dvec + h * n, *dph = dprime + h * n;

        scores(qh, kh, p, n, d, scale);
        softmax_rows(p, lh, n);
        weighted_values(p, vh, oh, n, d);

        /* D_i = sum_c dO_ic O_ic */
        for (int64_t i = 0; i < n; ++i) dh[i] = dot(doh + i * d, oh + i * d, d);

        /* dP_ij = dO_i . V_j ; D'_i = sum_j P_ij dP_ij ; dS_ij = P_ij (dP_ij - D_i) */
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                const double dpij = dot(doh + i * d, vh + j * d, d);
                acc += p[i * n + j] * dpij;
                ds[i * n + j] = p[i * n + j] * (dpij - dh[i]);
            }
            dph[i] = acc;
        }

        /* dQ_i = scale * sum_j dS_ij K_j */
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            double *row = dqh + i * d;
            for (int64_t c = 0; c < d; ++c) row[c] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                const double w = ds[i * n + j];
                for (int64_t c = 0; c < d; ++c) row[c] += w * kh[j * d + c];
            }
            for (int64_t c = 0; c < d; ++c) row[c] *= scale;
        }

        /* dK_j = scale * sum_i dS_ij Q_i ;  dV_j = sum_i P_ij dO_i */
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < n; ++j) {
            double *rk = dkh + j * d, *rv = dvh + j * d;
            for (int64_t c = 0; c < d; ++c) rk[c] = rv[c] = 0.0;
            for (int64_t i = 0; i < n; ++i) {
                const double wk = ds[i * n + j], wv = p[i * n + j];
                for (int64_t c = 0; c < d; ++c) {
                    rk[c] += wk * qh[i * d + c];
                    rv[c] += wv * doh[i * d + c];
                }
            }
            for (int64_t c = 0; c < d; ++c) rk[c] *= scale;
        }
    }
    free(p);
    free(ds);
    return 0;
}

/* Forward for selected query rows of ONE head (q, k, v point at that head's [N,d] block):
 * o_rows [nrows,d], lse_rows [nrows].  Each row of the definition is independent of the
 * others, so this is the same formula evaluated at fewer indices.  Returns 0 or -1. */
int oracle_attn_fwd_rows(const double *q, const double *k, const double *v, const int64_t *rows,
                         int64_t nrows, double *o_rows, double *lse_rows, int64_t n, int64_t d,
                         double scale)
{
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)n * sizeof(double));
        if (!s) {
#pragma omp atomic write
            err = -1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s) continue;
            const int64_t i = rows[r];
            for (int64_t j = 0; j < n; ++j) s[j] = scale * dot(q + i * d, k + j * d, d);
            lse_rows[r] = softmax_row(s, s, n);
            double *oi = o_rows + r * d;
            for (int64_t c = 0; c < d; ++c) oi[c] = 0.0;
            for (int64_t j = 0; j < n; ++j)
                for (int64_t c = 0; c < d; ++c) oi[c] += s[j] * v[j * d + c];
        }
        free(s);
    }
    return err;
}

/* Backward for selected rows of ONE head: dq_rows [nq,d] for query rows qrows, dk_rows and
 * dv_rows [nk,d] for key rows krows.  A key row's gradient sums over every query, so the
 * whole head's forward (P row by row, O, D) is evaluated first; nothing N x N is kept.
 * Returns 0 or -1. */
int oracle_attn_bwd_rows(const double *q, const double *k, const double *v, const double *dout,
                         const int64_t *qrows, int64_t nq, const int64_t *krows, int64_t nk,
                         double *dq_rows, double *dk_rows, double *dv_rows, int64_t n, int64_t d,
                         double scale)
{
    double *lse = (double *)malloc((size_t)n * sizeof(double));
    double *dvec = (double *)malloc((size_t)n * sizeof(double));
    int err = (!lse || !dvec) ? -1 : 0;

    /* LSE_i and D_i = dO_i . O_i for every query row i */
    if (!err) {
#pragma omp parallel
        {
            double *s = (double *)malloc((size_t)n * sizeof(double));
            double *oi = (double *)malloc((size_t)d * sizeof(double));
            if (!s || !oi) {
#pragma omp atomic write
                err = -1;
            }
#pragma omp for schedule(static)
            for (int64_t i = 0; i < n; ++i) {
                if (!s || !oi) continue;
                for (int64_t j = 0; j < n; ++j) s[j] = scale * dot(q + i * d, k + j * d, d);
                lse[i] = softmax_row(s, s, n);
                for (int64_t c = 0; c < d; ++c) oi[c] = 0.0;
                for (int64_t j = 0; j < n; ++j)
                    for (int64_t c = 0; c < d; ++c) oi[c] += s[j] * v[j * d + c];
                dvec[i] = dot(dout + i * d, oi, d);
            }
            free(s);
            free(oi);
        }
    }

    /* dQ_i = scale * sum_j P_ij (dP_ij - D_i) K_j */
    if (!err) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t r = 0; r < nq; ++r) {
            const int64_t i = qrows[r];
            double *row = dq_rows + r * d;
            for (int64_t c = 0; c < d; ++c) row[c] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                const double pij = exp(scale * dot(q + i * d, k + j * d, d) - lse[i]);
                const double dsij = pij * (dot(dout + i * d, v + j * d, d) - dvec[i]);
                for (int64_t c = 0; c < d; ++c) row[c] += dsij * k[j * d + c];
            }
            for (int64_t c = 0; c < d; ++c) row[c] *= scale;
        }
    }

    /* dK_j = scale * sum_i dS_ij Q_i ;  dV_j = sum_i P_ij dO_i */
    if (!err) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t r = 0; r < nk; ++r) {
            const int64_t j = krows[r];
            double *rk = dk_rows + r * d, *rv = dv_rows + r * d;
            for (int64_t c = 0; c < d; ++c) rk[c] = rv[c] = 0.0;
            for (int64_t i = 0; i < n; ++i) {
                const double pij = exp(scale * dot(q + i * d, k + j * d, d) - lse[i]);
                const double dsij = pij * (dot(dout + i * d, v + j * d, d) - dvec[i]);
                for (int64_t c = 0; c < d; ++c) {
                    rk[c] += dsij * q[i * d + c];
                    rv[c] += pij * dout[i * d + c];
                }
            }
            for (int64_t c = 0; c < d; ++c) rk[c] *= scale;
        }
    }
    free(lse);
    free(dvec);
    return err;
}

/* Element-wise fp32 addition c = a + b ("Self-attention, CUDA kernels and FlashAttention",
 * section 2: the vector_add_cuda kernel computes C[idx] = A[idx] + B[idx] for idx < N).  One
 * fp32 addition per element, rounded to nearest even as IEEE 754 prescribes. */
void oracle_vector_add(const float *a, const float *b, float *c, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) c[i] = a[i] + b[i];
}

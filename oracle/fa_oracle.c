/*
 * fa_oracle.c -- fp64 reference for exact attention.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this code.  It shares no source, header, helper or constant with
 * the CUDA library, and the CUDA library never calls it.
 *
 * What it computes (the plain definition, no blocking, no online softmax):
 *
 *   S_ij  = scale * sum_d Q_id K_jd                       standard attention,
 *           ("FlashAttention from scratch" walkthrough, l189.com, sec. 1.1;
 *            "FlashAttention 深入", section on the standard attention problem)
 *   S_ij  = -inf for j > i when causal                    query i sees keys j <= i
 *           (l189.com walkthrough, sec. 5.3, causal mask)
 *   S_ij  = -inf unless i - left <= j <= i + right        sliding window, each
 *           bound absent when negative (claire-chang.com FlashAttention
 *           introduction, flash_attn_func window_size)
 *   S_ij += -slope * |i - j|                              ALiBi bias on the
 *           scaled score (same page, alibi_slopes)
 *   S_ij  = -inf unless mask[i / T][j / T] != 0           block-sparse
 *           attention over T x T blocks (FlashAttention paper's block-sparse
 *           extension, as the "FlashAttention 深入" and l189.com pages report it)
 *   m_i   = max_j S_ij
 *   P_ij  = exp(S_ij - m_i) / sum_k exp(S_ik - m_i)       max-shifted softmax
 *           (l189.com walkthrough, sec. 2.2 and sec. 5.2)
 *   O_i   = sum_j P_ij V_j
 *   LSE_i = m_i + ln sum_j exp(S_ij - m_i)                natural log of the
 *           scaled scores (the per-row statistic the forward saves, sec. 3.1/3.3)
 *
 * and, for an upstream gradient dO (softmax Jacobian, l189.com sec. 3.3):
 *
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   Di    = sum_j P_ij dP_ij          (full-row sum; equals dO_i . O_i)
 *   dS_ij = P_ij (dP_ij - Di)
 *   dQ_i  = scale sum_j dS_ij K_j
 *   dK_j  = scale sum_i dS_ij Q_i
 *
 * All arithmetic is in double.  The S and P rows of every requested query row
 * are materialised.  Asking for every row gives the full N x N matrices; asking
 * for a subset runs the same code on fewer rows.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "fa_oracle.h"

int fa_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void fa_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* One query row: materialise the score row S_i. and probability row P_i.,
 * then O_i, LSE_i and (if dout != NULL) dP_i., Di, dS_i. and dQ_i. */
/* The block mask of one call: NULL, or one byte per (query block, key
 * block) of `tile` x `tile` scores, n_kb key blocks per row of blocks. */
typedef struct {
    const unsigned char* mask;
    long tile, n_kb;
} block_mask;

/* Is key j visible to query i? */
static int visible(long i, long j, int causal, long left, long right,
                   const block_mask* bm) {
    if (causal && j > i) return 0;
    if (left >= 0 && j < i - left) return 0;
    if (right >= 0 && j > i + right) return 0;
    if (bm->mask && !bm->mask[(i / bm->tile) * bm->n_kb + j / bm->tile]) return 0;
    return 1;
}

static void one_row(const double* q, const double* k, const double* v,
                    const double* dout, long N, long D, double scale,
                    int causal, long left, long right, double slope,
                    const block_mask* bm, long i,
                    double* s_row, double* p_row, double* ds_row, double* o_i,
                    double* lse_i, double* dq_i, double* di_i) {
    const double* qi = q + i * D;

    /* scores S_ij = scale * Q_i . K_j - slope * |i - j|, -inf where masked */
    for (long j = 0; j < N; ++j) {
        if (!visible(i, j, causal, left, right, bm)) {
            s_row[j] = -INFINITY;
            continue;
        }
        const double* kj = k + j * D;
        double acc = 0.0;
        for (long d = 0; d < D; ++d) acc += qi[d] * kj[d];
        s_row[j] = scale * acc - slope * (double)labs(i - j);
    }

    /* row maximum over visible keys */
    double m = -INFINITY;
    for (long j = 0; j < N; ++j)
        if (s_row[j] > m) m = s_row[j];

    /* softmax with the maximum subtracted; a row that sees no key has
     * O = 0 and LSE = -inf */
    double denom = 0.0;
    for (long j = 0; j < N; ++j) {
        double e = (s_row[j] == -INFINITY) ? 0.0 : exp(s_row[j] - m);
        p_row[j] = e;
        denom += e;
    }
    if (denom > 0.0)
        for (long j = 0; j < N; ++j) p_row[j] /= denom;
    *lse_i = denom > 0.0 ? m + log(denom) : -INFINITY;

    /* O_i = sum_j P_ij V_j */
    for (long d = 0; d < D; ++d) o_i[d] = 0.0;
    for (long j = 0; j < N; ++j) {
        double p = p_row[j];
        if (p == 0.0) continue;
        const double* vj = v + j * D;
        for (long d = 0; d < D; ++d) o_i[d] += p * vj[d];
    }

    if (!dout) return;

    /* dP_ij = dO_i . V_j, kept in ds_row until dS is formed */
    const double* doi = dout + i * D;
    for (long j = 0; j < N; ++j) {
        const double* vj = v + j * D;
        double acc = 0.0;
        for (long d = 0; d < D; ++d) acc += doi[d] * vj[d];
        ds_row[j] = acc;
    }
    double di = 0.0;
    for (long j = 0; j < N; ++j) di += p_row[j] * ds_row[j];
    *di_i = di;
    for (long j = 0; j < N; ++j) ds_row[j] = p_row[j] * (ds_row[j] - di);

    if (dq_i) {
        for (long d = 0; d < D; ++d) dq_i[d] = 0.0;
        for (long j = 0; j < N; ++j) {
            double g = ds_row[j];
            if (g == 0.0) continue;
            const double* kj = k + j * D;
            for (long d = 0; d < D; ++d) dq_i[d] += g * kj[d];
        }
        for (long d = 0; d < D; ++d) dq_i[d] *= scale;
    }
}

int fa_oracle_rows(const double* q, const double* k, const double* v,
                   const double* dout, long N, long D, double scale,
                   int causal, const long* rows, long nrows, double* o,
                   double* lse, double* dq, double* di, long kv_begin,
                   long kv_end, double* dk, double* dv) {
    return fa_oracle_rows_ex(q, k, v, dout, N, D, scale, causal, -1, -1, 0.0,
                             rows, nrows, o, lse, dq, di, kv_begin, kv_end, dk,
                             dv);
}

int fa_oracle_rows_ex(const double* q, const double* k, const double* v,
                      const double* dout, long N, long D, double scale,
                      int causal, long left, long right, double slope,
                      const long* rows, long nrows, double* o, double* lse,
                      double* dq, double* di, long kv_begin, long kv_end,
                      double* dk, double* dv) {
    return fa_oracle_rows_bs(q, k, v, dout, N, D, scale, causal, left, right,
                             slope, NULL, 1, rows, nrows, o, lse, dq, di,
                             kv_begin, kv_end, dk, dv);
}

int fa_oracle_rows_bs(const double* q, const double* k, const double* v,
                      const double* dout, long N, long D, double scale,
                      int causal, long left, long right, double slope,
                      const unsigned char* mask, long tile,
                      const long* rows, long nrows, double* o, double* lse,
                      double* dq, double* di, long kv_begin, long kv_end,
                      double* dk, double* dv) {
    return fa_oracle_rows_p(q, k, v, dout, N, D, scale, causal, left, right,
                            slope, mask, tile, rows, nrows, o, lse, dq, di,
                            kv_begin, kv_end, dk, dv, NULL);
}

int fa_oracle_rows_p(const double* q, const double* k, const double* v,
                     const double* dout, long N, long D, double scale,
                     int causal, long left, long right, double slope,
                     const unsigned char* mask, long tile,
                     const long* rows, long nrows, double* o, double* lse,
                     double* dq, double* di, long kv_begin, long kv_end,
                     double* dk, double* dv, double* p) {
    if (!q || !k || !v || !o || !lse || N < 1 || D < 1 || nrows < 0)
        return 1;
    if (left < -1 || right < -1 || !isfinite(slope)) return 1;
    if (mask && tile < 1) return 1;
    block_mask bm = {mask, tile, (N + tile - 1) / tile};
    if ((dq || di || dk || dv) && !dout) return 1;
    int want_cols = (dk != NULL) || (dv != NULL);
    if (want_cols && (kv_begin < 0 || kv_end > N || kv_begin > kv_end))
        return 1;
    if (rows) {
        for (long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= N) return 1;
    }

    /* materialised P and dS rows for the requested query rows */
    double* p_all = (double*)malloc(sizeof(double) * (size_t)nrows * (size_t)N);
    double* ds_all = dout ? (double*)malloc(sizeof(double) * (size_t)nrows * (size_t)N) : NULL;
    double* s_all = (double*)malloc(sizeof(double) * (size_t)nrows * (size_t)N);
    if (!p_all || !s_all || (dout && !ds_all)) {
        free(p_all);
        free(ds_all);
        free(s_all);
        return 2;
    }
    double* di_tmp = (double*)malloc(sizeof(double) * (size_t)(nrows > 0 ? nrows : 1));
    if (!di_tmp) {
        free(p_all);
        free(ds_all);
        free(s_all);
        return 2;
    }

#pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < nrows; ++r) {
        long i = rows ? rows[r] : r;
        one_row(q, k, v, dout, N, D, scale, causal, left, right, slope, &bm, i,
                s_all + (size_t)r * N,
                p_all + (size_t)r * N, dout ? ds_all + (size_t)r * N : NULL,
                o + (size_t)r * D, lse + r, dq ? dq + (size_t)r * D : NULL,
                di_tmp + r);
    }
    if (di && dout) memcpy(di, di_tmp, sizeof(double) * (size_t)nrows);

    /* column sums over the requested rows: dV_j = sum_i P_ij dO_i and
     * dK_j = scale * sum_i dS_ij Q_i, for keys kv_begin <= j < kv_end */
    if (want_cols) {
        long ncols = kv_end - kv_begin;
#pragma omp parallel for schedule(static)
        for (long c = 0; c < ncols; ++c) {
            long j = kv_begin + c;
            double* dvj = dv ? dv + (size_t)c * D : NULL;
            double* dkj = dk ? dk + (size_t)c * D : NULL;
            if (dvj)
                for (long d = 0; d < D; ++d) dvj[d] = 0.0;
            if (dkj)
                for (long d = 0; d < D; ++d) dkj[d] = 0.0;
            for (long r = 0; r < nrows; ++r) {
                long i = rows ? rows[r] : r;
                double p = p_all[(size_t)r * N + j];
                double g = ds_all[(size_t)r * N + j];
                if (dvj && p != 0.0) {
                    const double* doi = dout + i * D;
                    for (long d = 0; d < D; ++d) dvj[d] += p * doi[d];
                }
                if (dkj && g != 0.0) {
                    const double* qi = q + i * D;
                    for (long d = 0; d < D; ++d) dkj[d] += g * qi[d];
                }
            }
            if (dkj)
                for (long d = 0; d < D; ++d) dkj[d] *= scale;
        }
    }

    if (p) memcpy(p, p_all, sizeof(double) * (size_t)nrows * (size_t)N);
    free(p_all);
    free(ds_all);
    free(s_all);
    free(di_tmp);
    return 0;
}

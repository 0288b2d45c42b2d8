/*
 * fa_oracle.h -- fp64 reference for exact attention.  TEST INFRASTRUCTURE ONLY.
 * Loaded by the test suite, the smoke check and the benchmark's CPU-baseline
 * leg; never by the CUDA library.
 */
#ifndef FA_ORACLE_H
#define FA_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Exact attention for one (batch, head) slice, in double.
 *
 *   q, k, v, dout : [N, D] row-major.  dout may be NULL (forward only).
 *   rows          : nrows query-row indices in [0, N), or NULL for 0..nrows-1.
 *   o             : [nrows, D] output rows O_i.
 *   lse           : [nrows]    LSE_i = m_i + ln sum_j exp(S_ij - m_i).
 *   dq, di        : [nrows, D], [nrows]; may be NULL.  Need dout.
 *   dk, dv        : [kv_end - kv_begin, D]; may be NULL.  Column sums over the
 *                   requested rows only, i.e. the full gradient when rows is
 *                   every row, or, under the causal mask, for keys j whose
 *                   visible queries i >= j are all among the requested rows.
 *
 * Returns 0 on success, 1 on an invalid argument, 2 when out of host memory.
 */
int fa_oracle_rows(const double* q, const double* k, const double* v,
                   const double* dout, long N, long D, double scale,
                   int causal, const long* rows, long nrows, double* o,
                   double* lse, double* dq, double* di, long kv_begin,
                   long kv_end, double* dk, double* dv);

/*
 * fa_oracle_rows with a sliding window and an ALiBi bias: query i sees key j
 * only when i - left <= j <= i + right (a bound of -1 is absent; with causal
 * also j <= i), and the scaled score gets -slope * |i - j| added.
 * fa_oracle_rows is this with left = right = -1 and slope = 0.
 */
int fa_oracle_rows_ex(const double* q, const double* k, const double* v,
                      const double* dout, long N, long D, double scale,
                      int causal, long left, long right, double slope,
                      const long* rows, long nrows, double* o, double* lse,
                      double* dq, double* di, long kv_begin, long kv_end,
                      double* dk, double* dv);

/*
 * fa_oracle_rows_ex with a block mask: key j is visible to query i only when
 * mask[(i / tile) * ceil(N / tile) + j / tile] != 0 (mask == NULL: every
 * block).  A row that sees no key gets O = 0 and LSE = -inf, and no gradient.
 */
int fa_oracle_rows_bs(const double* q, const double* k, const double* v,
                      const double* dout, long N, long D, double scale,
                      int causal, long left, long right, double slope,
                      const unsigned char* mask, long tile,
                      const long* rows, long nrows, double* o, double* lse,
                      double* dq, double* di, long kv_begin, long kv_end,
                      double* dk, double* dv);

/*
 * fa_oracle_rows_bs that also returns the probability rows: p (may be NULL)
 * is [nrows, N], p[r][j] = P_ij for query i = rows[r] (0 where masked).
 */
int fa_oracle_rows_p(const double* q, const double* k, const double* v,
                     const double* dout, long N, long D, double scale,
                     int causal, long left, long right, double slope,
                     const unsigned char* mask, long tile,
                     const long* rows, long nrows, double* o, double* lse,
                     double* dq, double* di, long kv_begin, long kv_end,
                     double* dk, double* dv, double* p);

/* OpenMP threads the next call will use, and a way to set them. */
int fa_oracle_threads(void);
void fa_oracle_set_threads(int n);

#ifdef __cplusplus
}
#endif

#endif

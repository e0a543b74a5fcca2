/*
 * All-cores copy of the oracle's three product loops, for the CPU baseline.
 *
 * TEST INFRASTRUCTURE ONLY, like snack_oracle.c: only the benchmark's
 * CPU-baseline leg and the test suite load it.  The arithmetic is exactly
 * that of snack_oracle.c (fp64 terms, fp64 sums, one rounding to float), and
 * every output element is summed over the same terms in the same order, so
 * the results are bit-identical to the single-threaded oracle
 * (tests/test_oracle_pins.py checks this).  Only the work is split:
 *
 *   forward (§3.1 Algorithm 1): Y[l][i] sums the entries of row i in
 *     canonical order; threads take disjoint ranges of whole rows.
 *   backward_input (§3.4, Appendix F): dX[l][j] sums the entries of column
 *     j in canonical order, i.e. in the column-ordered (CSC) order of
 *     Appendix B Table 7; threads take disjoint ranges of whole columns.
 *   backward_weight (§3.4, Appendix F): every stored entry is independent;
 *     threads take disjoint ranges of entries.
 *
 * Inputs are in canonical order (rows ascending, columns ascending within a
 * row), with row_ptr [out+1] for the forward and col_ptr [in+1], csc_perm
 * [nnz] for the backward-input, as produced by oracle_canonicalize.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>

int oracle_omp_threads(void) { return omp_get_max_threads(); }

int oracle_omp_forward(int64_t out, int64_t in, const int32_t *row_ptr, const int32_t *col,
                       const float *val, int64_t B, const float *X, float *Y, double *S,
                       int threads) {
  int64_t i;
#pragma omp parallel for schedule(dynamic, 64) num_threads(threads)
  for (i = 0; i < out; ++i) {
    int64_t l, k;
    for (l = 0; l < B; ++l) {
      double acc = 0.0, sabs = 0.0;
      for (k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
        const double t = (double)val[k] * (double)X[l * in + col[k]];
        acc += t;
        sabs += fabs(t);
      }
      Y[l * out + i] = (float)acc;
      if (S) S[l * out + i] = sabs;
    }
  }
  return 0;
}

int oracle_omp_backward_input(int64_t out, int64_t in, const int32_t *col_ptr,
                              const int32_t *csc_perm, const int32_t *row, const float *val,
                              int64_t B, const float *dY, float *dX, double *S, int threads) {
  int64_t j;
#pragma omp parallel for schedule(dynamic, 64) num_threads(threads)
  for (j = 0; j < in; ++j) {
    int64_t l, s;
    for (l = 0; l < B; ++l) {
      double acc = 0.0, sabs = 0.0;
      for (s = col_ptr[j]; s < col_ptr[j + 1]; ++s) {
        const int64_t k = csc_perm[s];
        const double t = (double)val[k] * (double)dY[l * out + row[k]];
        acc += t;
        sabs += fabs(t);
      }
      dX[l * in + j] = (float)acc;
      if (S) S[l * in + j] = sabs;
    }
  }
  return 0;
}

int oracle_omp_backward_weight(int64_t out, int64_t in, int64_t nnz, const int32_t *row,
                               const int32_t *col, int64_t B, const float *X, const float *dY,
                               float *dW, double *S, int threads) {
  int64_t k;
#pragma omp parallel for schedule(static, 4096) num_threads(threads)
  for (k = 0; k < nnz; ++k) {
    const int64_t i = row[k], j = col[k];
    double acc = 0.0, sabs = 0.0;
    int64_t t;
    for (t = 0; t < B; ++t) {
      const double p = (double)dY[t * out + i] * (double)X[t * in + j];
      acc += p;
      sabs += fabs(p);
    }
    dW[k] = (float)acc;
    if (S) S[k] = sabs;
  }
  return 0;
}

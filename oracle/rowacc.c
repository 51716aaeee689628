/* GPTQ on vec(W) with a Kronecker Hessian A (x) B in the row-accumulator form.
 *
 * TEST INFRASTRUCTURE ONLY: part of the fp64 CPU oracle (see oracle/__init__.py).
 * It shares no code with the CUDA library.
 *
 * What it computes (summary page "FastKron: Efficient Quantization with
 * Kronecker-Factored Hessians", problem set-up and section 3): with the update
 * factors U_A, U_B (upper triangular, U^T U = A^{-1}), entry (i, j) is rounded
 * after every entry to its top-left and receives from each of them the update
 *     w~_ij -= U_B[i', i] E_i'j' U_A[j', j]      (i' <= i, j' <= j),
 * where E_ij = (w~_ij - q_ij) l^B_i l^A_j and l = 1 / diag(U).  Grouping the
 * sum by the source row gives, for the pre-rounding value,
 *     w~_ij = W_ij - sum_{i' < i} U_B[i', i] R_i'(j) - U_B[i, i] R_i(j),
 * with the row accumulator R_i(j) = sum_{j'} E_ij' U_A[j', j] over the entries
 * of row i rounded so far (U_A is upper triangular, so only j' <= j count).
 * R_i'(j) is final once entry (i', j) is rounded; it is then pushed down its
 * column into S(j, i) = sum_{i' < i} U_B[i', i] R_i'(j).  Every entry costs one
 * row update (n - j multiply-adds) and one column push (m - i), so a solve is
 * m n (m + n) flops, the count the pages quote for BaKron.
 *
 * Anti-diagonals d = i + j are taken in order; the entries of one diagonal are
 * independent of each other (none is to the top-left of another) and touch
 * disjoint rows of R and S, so they may run in parallel.  By Theorem 3.2 (any
 * order that rounds an entry after all entries to its top-left) the result is
 * the GPTQ output; it equals the other oracle variants up to fp64 rounding.
 *
 * Base quantizer: the per-row symmetric grid.  The rounding decision is taken
 * in fp32, as in oracle/quantizer.py: c = clamp(rint(fl32(w~) / s_i)) with one
 * fp32 division, round half to even; no clamp when `clamp` is 0.  Near ties
 * (|w~ / s - (k + 1/2)| < tol in fp64, boundary inside the clamp range) take
 * the guide's code when a guide is given.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

static int near_tie(double x, double s, int clamp, double qmin, double qmax, double tol) {
  const double t = x / s;
  const double k = floor(t);
  if (!(fabs(t - (k + 0.5)) < tol)) return 0;
  if (clamp && (k < qmin || k + 1.0 > qmax)) return 0;
  return 1;
}

/* W (m x n), UA (n x n), UB (m x m): row-major fp64; s: m fp32 row scales.
 * Outputs (m x n, fp64): codes, preround (w~ when rounded), E.  guide: m x n
 * codes or NULL.  Returns the number of guided decisions that changed a code,
 * or -1 if the scratch could not be allocated. */
long long rowacc_solve(const double* W, const double* UA, const double* UB, const float* s,
                       int64_t m, int64_t n, int clamp, double qmin, double qmax,
                       const double* guide, double guide_tol, double* codes, double* preround,
                       double* E) {
  double* R = (double*)calloc((size_t)(m * n), sizeof(double));   /* R[i][j]   */
  double* S = (double*)calloc((size_t)(n * m), sizeof(double));   /* S[j][i]   */
  if (!R || !S) {
    free(R);
    free(S);
    return -1;
  }
  long long overrides = 0;
  for (int64_t d = 0; d < m + n - 1; ++d) {
    const int64_t ilo = d - n + 1 > 0 ? d - n + 1 : 0;
    const int64_t ihi = d < m - 1 ? d : m - 1;
#pragma omp parallel for schedule(dynamic, 4) reduction(+ : overrides)
    for (int64_t i = ilo; i <= ihi; ++i) {
      const int64_t j = d - i;
      double* Ri = R + i * n;
      double* Sj = S + j * m;
      const double x = W[i * n + j] - Sj[i] - UB[i * m + i] * Ri[j];
      const float t = (float)x / s[i];
      double c = (double)rintf(t);
      if (clamp) {
        if (c < qmin) c = qmin;
        if (c > qmax) c = qmax;
      }
      if (guide && near_tie(x, (double)s[i], clamp, qmin, qmax, guide_tol)) {
        const double g = guide[i * n + j];
        if (g != c) ++overrides;
        c = g;
      }
      const double lB = 1.0 / UB[i * m + i], lA = 1.0 / UA[j * n + j];
      const double e = (x - (double)s[i] * c) * lB * lA;
      codes[i * n + j] = c;
      preround[i * n + j] = x;
      E[i * n + j] = e;
      const double* ua = UA + j * n;
      for (int64_t jj = j; jj < n; ++jj) Ri[jj] += e * ua[jj];
      const double r = Ri[j];
      const double* ub = UB + i * m;
      for (int64_t ii = i + 1; ii < m; ++ii) Sj[ii] += r * ub[ii];
    }
  }
  free(R);
  free(S);
  return overrides;
}

/* The same solve, traversed by blocks of `rb` consecutive rows instead of by
 * anti-diagonals, for speed at the full workload sizes (the arithmetic per
 * entry is the one above).  A block takes its columns left to right; column
 * j of block b starts once block b - 1 has finished column j (a progress
 * counter per block), which, by induction over the blocks above, puts every
 * entry to the top-left of (i, j) before it: the order Theorem 3.2 allows.
 * Inside a block, the entries of column j go top to bottom; each pushes its
 * finished row accumulator R_i(j) into the block's later rows at once, and
 * into the rows below the block together with the block's other rows (one
 * pass over S(j, .)); the row updates R_i(j'') += E_ij U_A[j, j''] of the
 * block's rows share one pass over row j of U_A.  The rows of R and U_B a
 * block works on stay in its thread's cache, so memory traffic drops by
 * about `rb` against the anti-diagonal traversal.  Only the grouping of the
 * column sums S(j, i) changes (sums of each block's contributions are added
 * to S in one step), so the result agrees with rowacc_solve up to fp64
 * rounding.  Blocks are dealt to threads in turn; each thread takes its
 * blocks in increasing order and every wait is on a lower block, so the
 * waits always end. */
long long rowacc_solve_blocked(const double* W, const double* UA, const double* UB, const float* s,
                               int64_t m, int64_t n, int clamp, double qmin, double qmax,
                               const double* guide, double guide_tol, double* codes,
                               double* preround, double* E, int rb) {
  if (rb < 1) rb = 1;
  if (rb > 64) rb = 64;
  const int64_t nb = (m + rb - 1) / rb;
  double* R = (double*)calloc((size_t)(m * n), sizeof(double));   /* R[i][j] */
  double* S = (double*)calloc((size_t)(n * m), sizeof(double));   /* S[j][i] */
  int64_t* done = (int64_t*)calloc((size_t)nb, sizeof(int64_t));  /* columns finished per block */
  if (!R || !S || !done) {
    free(R);
    free(S);
    free(done);
    return -1;
  }
  long long overrides = 0;
#pragma omp parallel reduction(+ : overrides)
  {
    int nt = 1, t = 0;
#ifdef _OPENMP
    nt = omp_get_num_threads();
    t = omp_get_thread_num();
#endif
    double sl[64], ev[64], rf[64];
    for (int64_t b = t; b < nb; b += nt) {
      const int64_t i0 = b * rb, i1 = i0 + rb < m ? i0 + rb : m;
      const int rows = (int)(i1 - i0);
      for (int64_t j = 0; j < n; ++j) {
        if (b > 0)
          while (__atomic_load_n(&done[b - 1], __ATOMIC_ACQUIRE) < j + 1) {
          }
        double* Sj = S + j * m;
        for (int r = 0; r < rows; ++r) sl[r] = Sj[i0 + r];
        const double ua = UA[j * n + j];
        for (int r = 0; r < rows; ++r) {
          const int64_t i = i0 + r;
          const double x = W[i * n + j] - sl[r] - UB[i * m + i] * R[i * n + j];
          const float tq = (float)x / s[i];
          double c = (double)rintf(tq);
          if (clamp) {
            if (c < qmin) c = qmin;
            if (c > qmax) c = qmax;
          }
          if (guide && near_tie(x, (double)s[i], clamp, qmin, qmax, guide_tol)) {
            const double g = guide[i * n + j];
            if (g != c) ++overrides;
            c = g;
          }
          const double lB = 1.0 / UB[i * m + i], lA = 1.0 / ua;
          const double e = (x - (double)s[i] * c) * lB * lA;
          codes[i * n + j] = c;
          preround[i * n + j] = x;
          E[i * n + j] = e;
          ev[r] = e;
          rf[r] = R[i * n + j] + e * ua;   /* R_i(j), final */
          R[i * n + j] = rf[r];
          for (int r2 = r + 1; r2 < rows; ++r2) sl[r2] += rf[r] * UB[i * m + i0 + r2];
        }
        /* row updates of the block's rows for the later columns */
        const double* uaj = UA + j * n;
        for (int r = 0; r < rows; ++r) {
          double* Ri = R + (i0 + r) * n;
          const double e = ev[r];
          for (int64_t jj = j + 1; jj < n; ++jj) Ri[jj] += e * uaj[jj];
        }
        /* the block's finished accumulators into the rows below it */
        for (int64_t c0 = i1; c0 < m; c0 += 64) {
          const int len = m - c0 < 64 ? (int)(m - c0) : 64;
          double acc[64];
          for (int k = 0; k < len; ++k) acc[k] = 0.0;
          for (int r = 0; r < rows; ++r) {
            const double f = rf[r];
            const double* ub = UB + (i0 + r) * m + c0;
            for (int k = 0; k < len; ++k) acc[k] += f * ub[k];
          }
          for (int k = 0; k < len; ++k) Sj[c0 + k] += acc[k];
        }
        __atomic_store_n(&done[b], j + 1, __ATOMIC_RELEASE);
      }
    }
  }
  free(R);
  free(S);
  free(done);
  return overrides;
}

/* Threads the parallel loop may use (0: the OpenMP default). */
#ifdef _OPENMP
int rowacc_threads(int want) {
  if (want > 0) omp_set_num_threads(want);
  return omp_get_max_threads();
}
#else
int rowacc_threads(int want) {
  (void)want;
  return 1;
}
#endif

/*
 * attention_oracle.c -- CPU fp64 oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) links, imports or calls this file.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark use it.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * What it computes is the plain definition of the operation described on
 *   "RTX Flash Attention Implementation COMPLETE", section "Usage Examples"
 *   (forward(q, k, v, causal, scale) -> output, lse over tensors laid out as
 *   [batch, heads, seq_len, head_dim]; backward(dout, q, k, v, output, lse,
 *   causal, scale) -> dq, dk, dv),
 * i.e. O = softmax(scale * Q K^T [+ causal mask]) V, its per-row log-sum-exp,
 * and the gradients of a loss L with dL/dO = dout.
 *
 * All arithmetic is in double precision, no blocking or fusion beyond the
 * definition: one row of scores at a time (so an N x N matrix is never held),
 * two passes over that row (max, then sum of exponentials).  Every (b,h) head
 * is independent; heads are spread over OpenMP threads.
 *
 * Readings of points the pages leave open (each listed in the design notes):
 *   - LSE is the natural logarithm of sum_j exp(scale * q_i . k_j).
 *   - Causal means key j is visible to query i iff j <= i (equal lengths).
 *   - scale multiplies Q K^T before the mask and the softmax.
 *
 * The gradient formulas are not printed on the pages; they follow from the
 * definition by the chain rule through softmax:
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij = dO_i . O_i,
 *   dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
 * The pages' backward recomputes P from the saved LSE ("GPU Performance
 * Optimization Batch 1 -- Design Spec", Item 3, the FlashAttention-3 backward
 * paragraph; "RTX Flash Attention Implementation COMPLETE", "Flash Attention
 * Backward Kernel: Gradient Recomputation").  Here P is recomputed from the
 * oracle's own fp64 LSE in the same way.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads of the later calls made from this thread (n >= 1). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

static double dot(const double* a, const double* b, int64_t d) {
  double s = 0.0;
  for (int64_t t = 0; t < d; ++t) s += a[t] * b[t];
  return s;
}

/* Number of keys visible to query row i (no window). */
static int64_t visible_keys(int64_t i, int64_t n, int causal) {
  return causal ? (i + 1) : n;
}

/*
 * Keys visible to query row i: lo <= j < hi.  Causal: j <= i.  A window
 * w >= 0 (local attention) further keeps only |i - j| <= w; w < 0 means no
 * window.
 */
static void visible_range(int64_t i, int64_t n, int causal, int64_t window,
                          int64_t* lo, int64_t* hi) {
  int64_t a = 0, b = causal ? i + 1 : n;
  if (window >= 0) {
    if (i - window > a) a = i - window;
    if (!causal && i + window + 1 < b) b = i + window + 1;
  }
  *lo = a;
  *hi = b;
}

/*
 * Scores s_j = scale * q_i . k_j for the visible keys, then the two-pass
 * log-sum-exp: m = max_j s_j, Z = sum_j exp(s_j - m), lse = m + ln Z.
 * Returns lse; s[] holds the scores (s[0] is key `lo`).
 */
static double row_scores_lse_range(const double* qi, const double* k,
                                   int64_t lo, int64_t hi, int64_t d,
                                   double scale, double* s) {
  double m = -INFINITY;
  for (int64_t j = lo; j < hi; ++j) {
    s[j - lo] = scale * dot(qi, k + j * d, d);
    if (s[j - lo] > m) m = s[j - lo];
  }
  double z = 0.0;
  for (int64_t j = lo; j < hi; ++j) z += exp(s[j - lo] - m);
  return m + log(z);
}

static double row_scores_lse(const double* qi, const double* k, int64_t nvis,
                             int64_t d, double scale, double* s) {
  return row_scores_lse_range(qi, k, 0, nvis, d, scale, s);
}

/*
 * Forward.  q, k, v, o: [BH, N, d] row-major doubles; lse: [BH, N].
 * P_ij = exp(s_ij - lse_i); O_i = sum_j P_ij v_j.
 * The _rows variant computes only query rows r0 <= i < r1 (each row is
 * independent) and leaves the other rows of o and lse untouched.  Every
 * (head, row) is independent of every other, so they are spread over the
 * OpenMP threads one by one; each row's arithmetic is the same whichever
 * thread runs it.
 */
void oracle_fwd_rows(const double* q, const double* k, const double* v,
                     int64_t BH, int64_t N, int64_t d, int causal,
                     double scale, int64_t r0, int64_t r1, double* o,
                     double* lse) {
  const int64_t rows = r1 > r0 ? r1 - r0 : 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 8)
    for (int64_t u = 0; u < BH * rows; ++u) {
      const int64_t bh = u / rows, i = r0 + u % rows;
      const double* qh = q + bh * N * d;
      const double* kh = k + bh * N * d;
      const double* vh = v + bh * N * d;
      int64_t nvis = visible_keys(i, N, causal);
      double l = row_scores_lse(qh + i * d, kh, nvis, d, scale, s);
      lse[bh * N + i] = l;
      double* oi = o + (bh * N + i) * d;
      for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
      for (int64_t j = 0; j < nvis; ++j) {
        double p = exp(s[j] - l);
        const double* vj = vh + j * d;
        for (int64_t t = 0; t < d; ++t) oi[t] += p * vj[t];
      }
    }
    free(s);
  }
}

void oracle_fwd(const double* q, const double* k, const double* v,
                int64_t BH, int64_t N, int64_t d, int causal, double scale,
                double* o, double* lse) {
  oracle_fwd_rows(q, k, v, BH, N, d, causal, scale, 0, N, o, lse);
}

/*
 * Forward by the online softmax of "RTX Flash Attention Implementation
 * COMPLETE", section "Online Softmax Algorithm": a running max m and a running
 * sum l are updated as new scores arrive, m' = max(m, x),
 * l' = l * exp(m - m') + exp(x - m').  The output accumulator is rescaled by the
 * same factor exp(m - m').  Scores arrive in tiles of `tile` keys; with
 * tile = 1 this is the page's element-by-element rule.
 *
 * `tau` >= 0 enables the lazy variant: the reference maximum is only replaced
 * when the tile maximum exceeds it by more than tau (natural-log units);
 * otherwise exp(x - m) may exceed 1 but the result is unchanged.
 * tau = 0 is the eager rule.
 */
void oracle_fwd_online(const double* q, const double* k, const double* v,
                       int64_t BH, int64_t N, int64_t d, int causal,
                       double scale, int64_t tile, double tau, double* o,
                       double* lse) {
  if (tile < 1) tile = 1;
#pragma omp parallel
  {
    double* acc = (double*)malloc(sizeof(double) * (size_t)(d > 0 ? d : 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(tile));
#pragma omp for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
      const double* qh = q + bh * N * d;
      const double* kh = k + bh * N * d;
      const double* vh = v + bh * N * d;
      for (int64_t i = 0; i < N; ++i) {
        int64_t nvis = visible_keys(i, N, causal);
        double m = -INFINITY, l = 0.0;
        for (int64_t t = 0; t < d; ++t) acc[t] = 0.0;
        for (int64_t j0 = 0; j0 < nvis; j0 += tile) {
          int64_t j1 = j0 + tile < nvis ? j0 + tile : nvis;
          double mt = -INFINITY;
          for (int64_t j = j0; j < j1; ++j) {
            s[j - j0] = scale * dot(qh + i * d, kh + j * d, d);
            if (s[j - j0] > mt) mt = s[j - j0];
          }
          double mnew = m;
          if (m == -INFINITY || mt > m + tau) mnew = (mt > m ? mt : m);
          double alpha = (m == -INFINITY) ? 0.0 : exp(m - mnew);
          l *= alpha;
          for (int64_t t = 0; t < d; ++t) acc[t] *= alpha;
          for (int64_t j = j0; j < j1; ++j) {
            double p = exp(s[j - j0] - mnew);
            l += p;
            const double* vj = vh + j * d;
            for (int64_t t = 0; t < d; ++t) acc[t] += p * vj[t];
          }
          m = mnew;
        }
        double* oi = o + (bh * N + i) * d;
        for (int64_t t = 0; t < d; ++t) oi[t] = acc[t] / l;
        lse[bh * N + i] = m + log(l);
      }
    }
    free(s);
    free(acc);
  }
}

/*
 * Backward.  q, k, v, dout: [BH, N, d]; outputs dq, dk, dv: [BH, N, d].
 * Per query row i: the scores and lse_i, P_ij = exp(s_ij - lse_i),
 * O_i = sum_j P_ij v_j and D_i = dO_i . O_i; then, for each visible pair
 * (i, j):
 *   dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i),
 *   dQ_i += scale dS_ij k_j,  dK_j += scale dS_ij q_i,  dV_j += P_ij dO_i.
 * The sums are taken in two passes so that rows and keys can be spread over
 * threads with no two threads adding into the same output row:
 *   pass 1, one query row at a time: lse_i, O_i, D_i and dQ_i (sum over j
 *           in increasing order);
 *   pass 2, one key at a time: dK_j and dV_j, summing over the rows i that
 *           see key j in increasing order, with P_ij and dS_ij recomputed
 *           from the same expressions and the saved lse_i, D_i.
 * Each output element is the same sum, in the same order, as one loop over
 * i (outer) and j (inner) would take.
 * The _rows variant sums the contributions of query rows r0 <= i < r1 only:
 * dq is exact on those rows (zero elsewhere); dk and dv hold the partial sums
 * over those rows, which are the full gradients for keys j >= r0 when causal
 * and r1 = N (no other row sees such a key).
 */
void oracle_bwd_rows(const double* q, const double* k, const double* v,
                     const double* dout, int64_t BH, int64_t N, int64_t d,
                     int causal, double scale, int64_t r0, int64_t r1,
                     double* dq, double* dk, double* dv) {
  const int64_t rows = r1 > r0 ? r1 - r0 : 0;
  double* lse_s = (double*)malloc(sizeof(double) * (size_t)(BH * N > 0 ? BH * N : 1));
  double* dd_s = (double*)malloc(sizeof(double) * (size_t)(BH * N > 0 ? BH * N : 1));
  memset(dq, 0, sizeof(double) * (size_t)(BH * N * d));
  memset(dk, 0, sizeof(double) * (size_t)(BH * N * d));
  memset(dv, 0, sizeof(double) * (size_t)(BH * N * d));
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double* oi = (double*)malloc(sizeof(double) * (size_t)(d > 0 ? d : 1));
    /* pass 1: query rows */
#pragma omp for schedule(dynamic, 8)
    for (int64_t u = 0; u < BH * rows; ++u) {
      const int64_t bh = u / rows, i = r0 + u % rows;
      const double* kh = k + bh * N * d;
      const double* vh = v + bh * N * d;
      int64_t nvis = visible_keys(i, N, causal);
      const double* qi = q + (bh * N + i) * d;
      const double* doi = dout + (bh * N + i) * d;
      double l = row_scores_lse(qi, kh, nvis, d, scale, s);
      for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
      for (int64_t j = 0; j < nvis; ++j) {
        s[j] = exp(s[j] - l); /* s now holds P_ij */
        const double* vj = vh + j * d;
        for (int64_t t = 0; t < d; ++t) oi[t] += s[j] * vj[t];
      }
      double D = dot(doi, oi, d);
      lse_s[bh * N + i] = l;
      dd_s[bh * N + i] = D;
      double* dqi = dq + (bh * N + i) * d;
      for (int64_t j = 0; j < nvis; ++j) {
        double ds = s[j] * (dot(doi, vh + j * d, d) - D);
        const double* kj = kh + j * d;
        for (int64_t t = 0; t < d; ++t) dqi[t] += scale * ds * kj[t];
      }
    }
    /* pass 2: keys (the implicit barrier above orders it after pass 1) */
#pragma omp for schedule(dynamic, 8)
    for (int64_t u = 0; u < BH * N; ++u) {
      const int64_t bh = u / N, j = u % N;
      const double* kj = k + (bh * N + j) * d;
      const double* vj = v + (bh * N + j) * d;
      double* dkj = dk + (bh * N + j) * d;
      double* dvj = dv + (bh * N + j) * d;
      for (int64_t i = r0; i < r1; ++i) {
        if (j >= visible_keys(i, N, causal)) continue;
        const double* qi = q + (bh * N + i) * d;
        const double* doi = dout + (bh * N + i) * d;
        double p = exp(scale * dot(qi, kj, d) - lse_s[bh * N + i]);
        double ds = p * (dot(doi, vj, d) - dd_s[bh * N + i]);
        for (int64_t t = 0; t < d; ++t) {
          dkj[t] += scale * ds * qi[t];
          dvj[t] += p * doi[t];
        }
      }
    }
    free(oi);
    free(s);
  }
  free(dd_s);
  free(lse_s);
}

void oracle_bwd(const double* q, const double* k, const double* v,
                const double* dout, int64_t BH, int64_t N, int64_t d,
                int causal, double scale, double* dq, double* dk, double* dv) {
  oracle_bwd_rows(q, k, v, dout, BH, N, d, causal, scale, 0, N, dq, dk, dv);
}

/*
 * Grouped / multi-query attention with an optional sliding window.
 * q, o: [B, H, N, d]; k, v: [B, Hkv, N, d] with H % Hkv == 0; query head h
 * reads key/value head h / (H / Hkv).  Visible keys as in visible_range.
 * Rows r0 <= i < r1 only (the other rows of o and lse are untouched); every
 * (query head, row) is independent and they are spread over the threads.
 */
void oracle_fwd_ext_rows(const double* q, const double* k, const double* v,
                         int64_t B, int64_t H, int64_t Hkv, int64_t N,
                         int64_t d, int causal, int64_t window, double scale,
                         int64_t r0, int64_t r1, double* o, double* lse) {
  const int64_t group = H / Hkv;
  const int64_t rows = r1 > r0 ? r1 - r0 : 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 8)
    for (int64_t u = 0; u < B * H * rows; ++u) {
      const int64_t bh = u / rows, i = r0 + u % rows;
      const int64_t b = bh / H, h = bh % H;
      const int64_t bkv = b * Hkv + h / group;
      const double* kh = k + bkv * N * d;
      const double* vh = v + bkv * N * d;
      int64_t lo, hi;
      visible_range(i, N, causal, window, &lo, &hi);
      const double l = row_scores_lse_range(q + (bh * N + i) * d, kh, lo, hi,
                                            d, scale, s);
      lse[bh * N + i] = l;
      double* oi = o + (bh * N + i) * d;
      for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
      for (int64_t j = lo; j < hi; ++j) {
        const double p = exp(s[j - lo] - l);
        const double* vj = vh + j * d;
        for (int64_t t = 0; t < d; ++t) oi[t] += p * vj[t];
      }
    }
    free(s);
  }
}

/*
 * Backward of the grouped / windowed forward: dq [B, H, N, d] per query
 * head; dk, dv [B, Hkv, N, d] summed over the query heads of each group
 * (each head's contribution is the chain rule of its own softmax, as in
 * oracle_bwd_rows).  Query rows r0 <= i < r1 only contribute.  The same two
 * passes as oracle_bwd_rows: query rows (lse_i, O_i, D_i, dQ_i), then keys
 * (dK_j, dV_j summed over the group's query heads in order, and within a
 * head over the rows that see key j in increasing order).
 */
void oracle_bwd_ext_rows(const double* q, const double* k, const double* v,
                         const double* dout, int64_t B, int64_t H, int64_t Hkv,
                         int64_t N, int64_t d, int causal, int64_t window,
                         double scale, int64_t r0, int64_t r1, double* dq,
                         double* dk, double* dv) {
  const int64_t group = H / Hkv;
  const int64_t rows = r1 > r0 ? r1 - r0 : 0;
  const int64_t nrow = B * H * N;
  double* lse_s = (double*)malloc(sizeof(double) * (size_t)(nrow > 0 ? nrow : 1));
  double* dd_s = (double*)malloc(sizeof(double) * (size_t)(nrow > 0 ? nrow : 1));
  memset(dq, 0, sizeof(double) * (size_t)(B * H * N * d));
  memset(dk, 0, sizeof(double) * (size_t)(B * Hkv * N * d));
  memset(dv, 0, sizeof(double) * (size_t)(B * Hkv * N * d));
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double* oi = (double*)malloc(sizeof(double) * (size_t)(d > 0 ? d : 1));
    /* pass 1: query rows */
#pragma omp for schedule(dynamic, 8)
    for (int64_t u = 0; u < B * H * rows; ++u) {
      const int64_t bh = u / rows, i = r0 + u % rows;
      const int64_t b = bh / H, h = bh % H;
      const int64_t bkv = b * Hkv + h / group;
      const double* kh = k + bkv * N * d;
      const double* vh = v + bkv * N * d;
      const double* qi = q + (bh * N + i) * d;
      const double* doi = dout + (bh * N + i) * d;
      int64_t lo, hi;
      visible_range(i, N, causal, window, &lo, &hi);
      const double l = row_scores_lse_range(qi, kh, lo, hi, d, scale, s);
      for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
      for (int64_t j = lo; j < hi; ++j) {
        s[j - lo] = exp(s[j - lo] - l); /* now P_ij */
        const double* vj = vh + j * d;
        for (int64_t t = 0; t < d; ++t) oi[t] += s[j - lo] * vj[t];
      }
      const double D = dot(doi, oi, d);
      lse_s[bh * N + i] = l;
      dd_s[bh * N + i] = D;
      double* dqi = dq + (bh * N + i) * d;
      for (int64_t j = lo; j < hi; ++j) {
        const double ds = s[j - lo] * (dot(doi, vh + j * d, d) - D);
        const double* kj = kh + j * d;
        for (int64_t t = 0; t < d; ++t) dqi[t] += scale * ds * kj[t];
      }
    }
    /* pass 2: keys of each key/value head */
#pragma omp for schedule(dynamic, 8)
    for (int64_t u = 0; u < B * Hkv * N; ++u) {
      const int64_t bkv = u / N, j = u % N;
      const int64_t b = bkv / Hkv, g = bkv % Hkv;
      const double* kj = k + (bkv * N + j) * d;
      const double* vj = v + (bkv * N + j) * d;
      double* dkj = dk + (bkv * N + j) * d;
      double* dvj = dv + (bkv * N + j) * d;
      for (int64_t h = g * group; h < (g + 1) * group; ++h) {
        const int64_t bh = b * H + h;
        for (int64_t i = r0; i < r1; ++i) {
          int64_t lo, hi;
          visible_range(i, N, causal, window, &lo, &hi);
          if (j < lo || j >= hi) continue;
          const double* qi = q + (bh * N + i) * d;
          const double* doi = dout + (bh * N + i) * d;
          const double p = exp(scale * dot(qi, kj, d) - lse_s[bh * N + i]);
          const double ds = p * (dot(doi, vj, d) - dd_s[bh * N + i]);
          for (int64_t t = 0; t < d; ++t) {
            dkj[t] += scale * ds * qi[t];
            dvj[t] += p * doi[t];
          }
        }
      }
    }
    free(oi);
    free(s);
  }
  free(dd_s);
  free(lse_s);
}

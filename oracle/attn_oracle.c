/*
 * attn_oracle.c -- plain fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes is the plain definition, with no tiling, fusion or online
 * rescaling:
 *
 *   s_ij  = scale * sum_d q_id k_jd                 (for j in the allowed set A_i)
 *   LSE_i = m_i + ln sum_{j in A_i} exp(s_ij - m_i),   m_i = max_j s_ij
 *   P_ij  = exp(s_ij - LSE_i)
 *   O_i   = sum_j P_ij v_j
 *
 * with A_i = {0..N-1}, or {0..i} when causal.  Sources:
 *   - exact attention O = softmax(scale QK^T) V, never materialising N x N:
 *     FlashNystrom page, "Scope"; FlashStieltjes page, "The kernel";
 *     "From-scratch CUDA attention kernel reaches 94.4% of FlashAttention-4",
 *     "How the kernel partitions its work".
 *   - the running-max / running-sum softmax reaches exactly this result:
 *     FlashStieltjes page, "The challenge".
 *   - causal keys j <= i, grouped-query heads (Hq a multiple of Hkv), ragged N:
 *     FlashAttention for Tesla P100 page, "What it supports" and "Quick start"
 *     (q is (B,Hq,N,D), k and v are (B,Hkv,N,D)).
 *   - backward dS = P o (dP - Delta), Delta_i = dO_i . O_i, dV = P^T dO:
 *     FlashAttention for Tesla P100 page, "Documentation".
 *
 * Readings where the pages are silent (stated once here, tested in tests/):
 *   - query head h uses key/value head h / (Hq/Hkv) (consecutive groups);
 *   - causal means key j <= query i (Nq == Nk, so both alignments agree);
 *   - LSE is the natural log of the scaled scores;
 *   - the backward's Delta uses the oracle's own fp64 O.
 *
 * All inputs are fp64 arrays (the caller widens bf16 exactly).  Layouts are
 * contiguous [B, H, N, D] row-major; lse is [B, Hq, N].  OpenMP parallelises
 * over independent rows (forward) and over the query rows of one (batch, kv-head)
 * group at a time (backward).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Index of element (b, h, n, d) in a contiguous [B, H, N, D] tensor. */
static inline int64_t at4(int64_t b, int64_t h, int64_t n, int64_t d,
                          int64_t H, int64_t N, int64_t D) {
  return ((b * H + h) * N + n) * D + d;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Scores of one query row against its allowed keys; returns |A_i|. */
static int64_t row_scores(const double* qi, const double* kh, int64_t N, int64_t D,
                          int64_t i, int causal, double scale, double* s) {
  int64_t nallowed = causal ? (i + 1 < N ? i + 1 : N) : N;
  for (int64_t j = 0; j < nallowed; ++j) {
    const double* kj = kh + j * D;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += qi[d] * kj[d];
    s[j] = scale * dot;
  }
  return nallowed;
}

/* Softmax of a score row into probabilities; returns LSE (natural log). */
static double row_softmax(double* s, int64_t n) {
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) if (s[j] > m) m = s[j];
  double sum = 0.0;
  for (int64_t j = 0; j < n; ++j) sum += exp(s[j] - m);
  double lse = m + log(sum);
  for (int64_t j = 0; j < n; ++j) s[j] = exp(s[j] - lse);
  return lse;
}

/*
 * Forward on a list of rows.  rows[r] is the flat row id (b*Hq + h)*N + i;
 * rows == NULL means every row in order.  o is [nrows, D], lse is [nrows].
 * Returns 0, or -1 on bad sizes / allocation failure.
 */
int oracle_fwd_rows(const double* q, const double* k, const double* v,
                    int B, int Hq, int Hkv, int N, int D, int causal, double scale,
                    const int64_t* rows, int64_t nrows, double* o, double* lse) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || D <= 0 || Hq % Hkv) return -1;
  const int64_t G = Hq / Hkv;
  const int64_t total = (int64_t)B * Hq * N;
  if (!rows) nrows = total;
  int err = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
    if (!s) {
#pragma omp atomic write
      err = -1;
    }
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < nrows; ++r) {
      if (!s) continue;
      int64_t id = rows ? rows[r] : r;
      if (id < 0 || id >= total) {
#pragma omp atomic write
        err = -1;
        continue;
      }
      int64_t i = id % N, bh = id / N, h = bh % Hq, b = bh / Hq, hk = h / G;
      const double* qi = q + at4(b, h, i, 0, Hq, N, D);
      const double* kh = k + at4(b, hk, 0, 0, Hkv, N, D);
      const double* vh = v + at4(b, hk, 0, 0, Hkv, N, D);
      int64_t n = row_scores(qi, kh, N, D, i, causal, scale, s);
      lse[r] = row_softmax(s, n);
      double* oi = o + r * (int64_t)D;
      for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
      for (int64_t j = 0; j < n; ++j) {
        const double* vj = vh + j * D;
        for (int64_t d = 0; d < D; ++d) oi[d] += s[j] * vj[d];
      }
    }
    free(s);
  }
  return err;
}

/*
 * Backward: given dO, returns dQ [B,Hq,N,D], dK and dV [B,Hkv,N,D].
 *   Delta_i = sum_d dO_id O_id,  dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - Delta_i)
 *   dQ_i = scale sum_j dS_ij k_j
 *   dK_j = scale sum_{h in group} sum_i dS_ij q_i
 *   dV_j = sum_{h in group} sum_i P_ij dO_i
 * The (batch, kv-head) groups run one after another; inside a group OpenMP
 * splits the query rows of all its heads, each thread summing its rows' dK/dV
 * terms privately before one reduction per group.
 */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
               int B, int Hq, int Hkv, int N, int D, int causal, double scale,
               double* dq, double* dk, double* dv) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || D <= 0 || Hq % Hkv) return -1;
  const int64_t G = Hq / Hkv;
  const int64_t ND = (int64_t)N * D;
  memset(dq, 0, sizeof(double) * (size_t)B * Hq * N * D);
  memset(dk, 0, sizeof(double) * (size_t)B * Hkv * N * D);
  memset(dv, 0, sizeof(double) * (size_t)B * Hkv * N * D);
  int err = 0;
  for (int64_t g = 0; g < (int64_t)B * Hkv && !err; ++g) {
    const int64_t b = g / Hkv, hk = g % Hkv;
    const double* kh = k + at4(b, hk, 0, 0, Hkv, N, D);
    const double* vh = v + at4(b, hk, 0, 0, Hkv, N, D);
    double* dkh = dk + at4(b, hk, 0, 0, Hkv, N, D);
    double* dvh = dv + at4(b, hk, 0, 0, Hkv, N, D);
#pragma omp parallel
    {
      double* s = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
      double* oi = (double*)malloc(sizeof(double) * D);
      double* dkp = (double*)calloc((size_t)(ND > 0 ? ND : 1), sizeof(double));
      double* dvp = (double*)calloc((size_t)(ND > 0 ? ND : 1), sizeof(double));
      const int have = s && oi && dkp && dvp;
      if (!have) {
#pragma omp atomic write
        err = -1;
      }
#pragma omp for schedule(dynamic, 4)
      for (int64_t r = 0; r < G * N; ++r) {
        if (!have) continue;
        const int64_t h = hk * G + r / N, i = r % N;
        const double* qi = q + at4(b, h, i, 0, Hq, N, D);
        const double* doi = dout + at4(b, h, i, 0, Hq, N, D);
        double* dqi = dq + at4(b, h, i, 0, Hq, N, D);
        int64_t n = row_scores(qi, kh, N, D, i, causal, scale, s);
        row_softmax(s, n);
        for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
        for (int64_t j = 0; j < n; ++j)
          for (int64_t d = 0; d < D; ++d) oi[d] += s[j] * vh[j * D + d];
        double delta = 0.0;
        for (int64_t d = 0; d < D; ++d) delta += doi[d] * oi[d];
        for (int64_t j = 0; j < n; ++j) {
          const double* vj = vh + j * D;
          double dp = 0.0;
          for (int64_t d = 0; d < D; ++d) dp += doi[d] * vj[d];
          double p = s[j];
          double ds = p * (dp - delta);
          for (int64_t d = 0; d < D; ++d) {
            dqi[d] += scale * ds * kh[j * D + d];
            dkp[j * D + d] += scale * ds * qi[d];
            dvp[j * D + d] += p * doi[d];
          }
        }
      }
      if (have) {
#pragma omp critical
        {
          for (int64_t e = 0; e < ND; ++e) {
            dkh[e] += dkp[e];
            dvh[e] += dvp[e];
          }
        }
      }
      free(s);
      free(oi);
      free(dkp);
      free(dvp);
    }
  }
  return err;
}

/*
 * dQ of selected query rows (the dQ_i line of the backward above), for
 * problems too large for the whole backward: per row i of head h, the allowed
 * scores, P_i = softmax, O_i = sum_j P_ij v_j, Delta_i = dO_i . O_i,
 * dS_ij = P_ij (dO_i . v_j - Delta_i) and dQ_i = scale sum_j dS_ij k_j.
 * rows: flat ids (b*Hq + h)*N + i.  dq: [nrows, D].
 */
int oracle_bwd_dq_rows(const double* q, const double* k, const double* v, const double* dout,
                       int B, int Hq, int Hkv, int N, int D, int causal, double scale,
                       const int64_t* rows, int64_t nrows, double* dq) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || D <= 0 || Hq % Hkv || !rows) return -1;
  const int64_t G = Hq / Hkv;
  const int64_t total = (int64_t)B * Hq * N;
  int err = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
    double* oi = (double*)malloc(sizeof(double) * D);
    const int have = s && oi;
    if (!have) {
#pragma omp atomic write
      err = -1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
      if (!have) continue;
      const int64_t id = rows[r];
      if (id < 0 || id >= total) {
#pragma omp atomic write
        err = -1;
        continue;
      }
      const int64_t i = id % N, bh = id / N, h = bh % Hq, b = bh / Hq, hk = h / G;
      const double* qi = q + at4(b, h, i, 0, Hq, N, D);
      const double* doi = dout + at4(b, h, i, 0, Hq, N, D);
      const double* kh = k + at4(b, hk, 0, 0, Hkv, N, D);
      const double* vh = v + at4(b, hk, 0, 0, Hkv, N, D);
      double* dqi = dq + r * (int64_t)D;
      const int64_t n = row_scores(qi, kh, N, D, i, causal, scale, s);
      row_softmax(s, n);
      for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
      for (int64_t j = 0; j < n; ++j)
        for (int64_t d = 0; d < D; ++d) oi[d] += s[j] * vh[j * D + d];
      double delta = 0.0;
      for (int64_t d = 0; d < D; ++d) delta += doi[d] * oi[d];
      for (int64_t d = 0; d < D; ++d) dqi[d] = 0.0;
      for (int64_t j = 0; j < n; ++j) {
        const double* vj = vh + j * D;
        double dp = 0.0;
        for (int64_t d = 0; d < D; ++d) dp += doi[d] * vj[d];
        const double ds = s[j] * (dp - delta);
        for (int64_t d = 0; d < D; ++d) dqi[d] += scale * ds * kh[j * D + d];
      }
    }
    free(s);
    free(oi);
  }
  return err;
}

/*
 * Stieltjes attention forward, a second method on the same tiling.
 * FlashStieltjes page, "Why touch softmax": weights
 * p_j = (lambda - s_j)^-q with the pole lambda above the best score, placed so
 * that the weights add up to 1; "The challenge": subtract the row's largest
 * score, then Newton-Raphson from lambda = 1.1 (three steps by default);
 * "The kernel": sweep 1 the row max, sweeps 2-4 the Newton steps, sweep 5
 * weights and values.  For each row, over its allowed keys:
 *
 *   m   = max_j s_j,   t_j = s_j - m  (<= 0)
 *   f(l) = sum_j (l - t_j)^-q - 1,   f'(l) = -q sum_j (l - t_j)^-(q+1)
 *   l_0 = 1.1,  l_{n+1} = l_n - f(l_n) / f'(l_n)   (`steps` times)
 *   p_j = (l - t_j)^-q,   O = sum_j p_j v_j,   pole = m + l
 *
 * steps <= 0 iterates to convergence instead (step below 1e-15 l, at most 200
 * steps): the exact pole, for the tests' closed forms.  The weights are used
 * as they come out of the last step (no renormalisation), as the page's fifth
 * sweep does.
 */
static double row_stj_pole(const double* s, int64_t n, int order, int steps) {
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) if (s[j] > m) m = s[j];
  double l = 1.1;
  const int limit = steps > 0 ? steps : 200;
  for (int it = 0; it < limit; ++it) {
    double f = -1.0, fp = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      const double a = l - (s[j] - m);
      f += pow(a, -(double)order);
      fp += -(double)order * pow(a, -(double)(order + 1));
    }
    const double step = f / fp;
    l -= step;
    if (steps <= 0 && fabs(step) <= 1e-15 * l) break;
  }
  return m + l;
}

int oracle_stj_fwd_rows(const double* q, const double* k, const double* v,
                        int B, int Hq, int Hkv, int N, int D, int causal, double scale,
                        int order, int steps, const int64_t* rows, int64_t nrows,
                        double* o, double* pole) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || D <= 0 || Hq % Hkv || order < 1) return -1;
  const int64_t G = Hq / Hkv;
  const int64_t total = (int64_t)B * Hq * N;
  if (!rows) nrows = total;
  int err = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
    if (!s) {
#pragma omp atomic write
      err = -1;
    }
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < nrows; ++r) {
      if (!s) continue;
      int64_t id = rows ? rows[r] : r;
      if (id < 0 || id >= total) {
#pragma omp atomic write
        err = -1;
        continue;
      }
      int64_t i = id % N, bh = id / N, h = bh % Hq, b = bh / Hq, hk = h / G;
      const double* qi = q + at4(b, h, i, 0, Hq, N, D);
      const double* kh = k + at4(b, hk, 0, 0, Hkv, N, D);
      const double* vh = v + at4(b, hk, 0, 0, Hkv, N, D);
      int64_t n = row_scores(qi, kh, N, D, i, causal, scale, s);
      const double pl = row_stj_pole(s, n, order, steps);
      pole[r] = pl;
      double* oi = o + r * (int64_t)D;
      for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
      for (int64_t j = 0; j < n; ++j) {
        const double pj = pow(pl - s[j], -(double)order);
        const double* vj = vh + j * D;
        for (int64_t d = 0; d < D; ++d) oi[d] += pj * vj[d];
      }
    }
    free(s);
  }
  return err;
}

/*
 * Nystrom attention forward, a third method.  FlashNystrom page, "Scope":
 * the factorisation
 *
 *   O = softmax(Q Kt^T) . pinv(softmax(Qt Kt^T)) . softmax(Qt K^T) . V
 *
 * with landmarks Qt, Kt the segment means of Q and K, and the pseudo-inverse
 * taken by a fixed number of unrolled Newton-Schulz steps; "Configuration":
 * with the Tikhonov ridge on (kappa* > 0) the iteration inverts
 * M = A^T A + lambda I, lambda = ||A||_1 ||A||_inf / kappa*, for A the m x m
 * landmark softmax.  Readings taken where the page is silent:
 *   - landmark i averages rows floor(i N / m) .. floor((i+1) N / m) - 1
 *     (every segment non-empty since N >= m);
 *   - the caller's scale multiplies all three score matrices;
 *   - Newton-Schulz is the textbook pseudo-inverse iteration
 *     X_0 = A^T / (||A||_1 ||A||_inf),  X_{t+1} = 2 X_t - X_t A X_t;
 *   - with the ridge, pinv(A) is taken as X(M) A^T, X(M) the iteration on M;
 *   - a query head h uses key/value head h / (Hq / Hkv), whose landmarks Kt
 *     come from that key head's rows.
 */

/* max column sum (1-norm) and max row sum (inf-norm) of an m x m matrix */
static double mat_norm1(const double* a, int m) {
  double best = 0.0;
  for (int c = 0; c < m; ++c) {
    double s = 0.0;
    for (int r = 0; r < m; ++r) s += fabs(a[r * m + c]);
    if (s > best) best = s;
  }
  return best;
}
static double mat_norm_inf(const double* a, int m) {
  double best = 0.0;
  for (int r = 0; r < m; ++r) {
    double s = 0.0;
    for (int c = 0; c < m; ++c) s += fabs(a[r * m + c]);
    if (s > best) best = s;
  }
  return best;
}
/* c = a b for m x m matrices (c must not alias a or b) */
static void mat_mul(const double* a, const double* b, double* c, int m) {
  for (int r = 0; r < m; ++r)
    for (int col = 0; col < m; ++col) {
      double s = 0.0;
      for (int t = 0; t < m; ++t) s += a[r * m + t] * b[t * m + col];
      c[r * m + col] = s;
    }
}

/*
 * Newton-Schulz pseudo-inverse of the m x m matrix a after `iters` steps, with
 * the ridge when kappa > 0 (see above).  out is m x m.  Returns 0, or -1 on
 * bad arguments or allocation failure.
 */
int oracle_ns_pinv(const double* a, int m, int iters, double kappa, double* out) {
  if (m <= 0 || iters < 0) return -1;
  const size_t mm = (size_t)m * m;
  double* mat = (double*)malloc(sizeof(double) * mm);
  double* x = (double*)malloc(sizeof(double) * mm);
  double* t1 = (double*)malloc(sizeof(double) * mm);
  double* t2 = (double*)malloc(sizeof(double) * mm);
  if (!mat || !x || !t1 || !t2) {
    free(mat); free(x); free(t1); free(t2);
    return -1;
  }
  if (kappa > 0.0) {
    const double lambda = mat_norm1(a, m) * mat_norm_inf(a, m) / kappa;
    for (int r = 0; r < m; ++r)
      for (int c = 0; c < m; ++c) {
        double s = 0.0;
        for (int t = 0; t < m; ++t) s += a[t * m + r] * a[t * m + c];
        mat[r * m + c] = s + (r == c ? lambda : 0.0);
      }
  } else {
    memcpy(mat, a, sizeof(double) * mm);
  }
  const double c0 = mat_norm1(mat, m) * mat_norm_inf(mat, m);
  for (int r = 0; r < m; ++r)
    for (int c = 0; c < m; ++c) x[r * m + c] = c0 > 0.0 ? mat[c * m + r] / c0 : 0.0;
  for (int it = 0; it < iters; ++it) {
    mat_mul(mat, x, t1, m);   /* A X */
    mat_mul(x, t1, t2, m);    /* X A X */
    for (size_t e = 0; e < mm; ++e) x[e] = 2.0 * x[e] - t2[e];
  }
  if (kappa > 0.0) {
    /* pinv(A) = X(M) A^T */
    for (int r = 0; r < m; ++r)
      for (int c = 0; c < m; ++c) {
        double s = 0.0;
        for (int t = 0; t < m; ++t) s += x[r * m + t] * a[c * m + t];
        out[r * m + c] = s;
      }
  } else {
    memcpy(out, x, sizeof(double) * mm);
  }
  free(mat); free(x); free(t1); free(t2);
  return 0;
}

/* landmark i of one head: mean of rows floor(i N / m) .. floor((i+1) N / m) - 1 */
static void landmarks(const double* xh, int64_t N, int64_t D, int m, double* out) {
  for (int i = 0; i < m; ++i) {
    const int64_t lo = (int64_t)i * N / m, hi = (int64_t)(i + 1) * N / m;
    double* oi = out + (int64_t)i * D;
    for (int64_t d = 0; d < D; ++d) oi[d] = 0.0;
    for (int64_t r = lo; r < hi; ++r)
      for (int64_t d = 0; d < D; ++d) oi[d] += xh[r * D + d];
    for (int64_t d = 0; d < D; ++d) oi[d] /= (double)(hi - lo);
  }
}

/*
 * Full Nystrom forward.  q [B,Hq,N,D], k and v [B,Hkv,N,D], o [B,Hq,N,D].
 * Optional intermediates (NULL to skip): qt [B,Hq,m,D], kt [B,Hkv,m,D],
 * pinv [B,Hq,m,m] (the pseudo-inverse of the landmark softmax), w [B,Hq,m,D]
 * (softmax(Qt K^T) V).  Returns 0, or -1 on bad sizes / allocation failure.
 */
int oracle_nys_fwd(const double* q, const double* k, const double* v,
                   int B, int Hq, int Hkv, int N, int D, int m, int iters, double kappa,
                   double scale, double* o, double* qt_out, double* kt_out,
                   double* pinv_out, double* w_out) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv || m <= 0 || N < m || iters < 0)
    return -1;
  const int64_t G = Hq / Hkv, BH = (int64_t)B * Hq, BHk = (int64_t)B * Hkv;
  const int64_t mD = (int64_t)m * D, mm = (int64_t)m * m;
  double* qt = (double*)malloc(sizeof(double) * (BH * mD + 1));
  double* kt = (double*)malloc(sizeof(double) * (BHk * mD + 1));
  double* pinv = (double*)malloc(sizeof(double) * (BH * mm + 1));
  double* w = (double*)malloc(sizeof(double) * (BH * mD + 1));
  double* y = (double*)malloc(sizeof(double) * (BH * mD + 1));
  int err = (!qt || !kt || !pinv || !w || !y) ? -1 : 0;
  if (!err) {
    /* landmarks */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH + BHk; ++bh) {
      if (bh < BH) landmarks(q + bh * (int64_t)N * D, N, D, m, qt + bh * mD);
      else landmarks(k + (bh - BH) * (int64_t)N * D, N, D, m, kt + (bh - BH) * mD);
    }
    /* landmark softmax A2 = softmax(Qt Kt^T) and its pseudo-inverse */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
      const int64_t b = bh / Hq, h = bh % Hq, hk = b * Hkv + h / G;
      double* a2 = (double*)malloc(sizeof(double) * mm);
      if (!a2) {
#pragma omp atomic write
        err = -1;
        continue;
      }
      for (int i = 0; i < m; ++i) {
        row_scores(qt + bh * mD + (int64_t)i * D, kt + hk * mD, m, D, 0, 0, scale, a2 + (int64_t)i * m);
        row_softmax(a2 + (int64_t)i * m, m);
      }
      if (oracle_ns_pinv(a2, m, iters, kappa, pinv + bh * mm)) {
#pragma omp atomic write
        err = -1;
      }
      free(a2);
    }
  }
  if (!err) {
    /* W = softmax(Qt K^T) V, one landmark row at a time */
#pragma omp parallel
    {
      double* s = (double*)malloc(sizeof(double) * N);
      if (!s) {
#pragma omp atomic write
        err = -1;
      }
#pragma omp for schedule(dynamic, 1)
      for (int64_t r = 0; r < BH * m; ++r) {
        if (!s) continue;
        const int64_t bh = r / m, i = r % m, b = bh / Hq, h = bh % Hq;
        const int64_t hk = b * Hkv + h / G;
        const double* vh = v + hk * (int64_t)N * D;
        row_scores(qt + bh * mD + i * D, k + hk * (int64_t)N * D, N, D, 0, 0, scale, s);
        row_softmax(s, N);
        double* wi = w + bh * mD + i * D;
        for (int64_t d = 0; d < D; ++d) wi[d] = 0.0;
        for (int64_t j = 0; j < N; ++j)
          for (int64_t d = 0; d < D; ++d) wi[d] += s[j] * vh[j * D + d];
      }
      free(s);
    }
  }
  if (!err) {
    /* Y = pinv W */
#pragma omp parallel for schedule(static)
    for (int64_t bh = 0; bh < BH; ++bh)
      for (int i = 0; i < m; ++i)
        for (int64_t d = 0; d < D; ++d) {
          double s = 0.0;
          for (int t = 0; t < m; ++t) s += pinv[bh * mm + (int64_t)i * m + t] * w[bh * mD + (int64_t)t * D + d];
          y[bh * mD + (int64_t)i * D + d] = s;
        }
    /* O_r = softmax(q_r Kt^T) Y */
#pragma omp parallel
    {
      double* s = (double*)malloc(sizeof(double) * m);
      if (!s) {
#pragma omp atomic write
        err = -1;
      }
#pragma omp for schedule(dynamic, 64)
      for (int64_t r = 0; r < BH * (int64_t)N; ++r) {
        if (!s) continue;
        const int64_t bh = r / N, b = bh / Hq, h = bh % Hq, hk = b * Hkv + h / G;
        row_scores(q + r * D, kt + hk * mD, m, D, 0, 0, scale, s);
        row_softmax(s, m);
        double* orow = o + r * D;
        for (int64_t d = 0; d < D; ++d) orow[d] = 0.0;
        for (int t = 0; t < m; ++t)
          for (int64_t d = 0; d < D; ++d) orow[d] += s[t] * y[bh * mD + (int64_t)t * D + d];
      }
      free(s);
    }
  }
  if (!err) {
    if (qt_out) memcpy(qt_out, qt, sizeof(double) * BH * mD);
    if (kt_out) memcpy(kt_out, kt, sizeof(double) * BHk * mD);
    if (pinv_out) memcpy(pinv_out, pinv, sizeof(double) * BH * mm);
    if (w_out) memcpy(w_out, w, sizeof(double) * BH * mD);
  }
  free(qt); free(kt); free(pinv); free(w); free(y);
  return err;
}

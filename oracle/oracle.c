/*
 * Exact-attention oracle: plain, slow, fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do. It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes is the plain definition of scaled dot-product attention,
 * one query row at a time, with no tiling:
 *   S = scale * Q K^T                      (tutorial page "research-attention",
 *                                           section 01, first equation)
 *   P = row-softmax(S)                     (same section, second equation)
 *   O = P V                                (same section, third equation)
 *   L_i = log sum_j exp(S_ij) = m_i + log l_i
 *                                          (same page, section 04: the saved
 *                                           statistic L = m + log(l))
 * With a causal mask, S_ij = -inf for key j > query i (standard lower
 * triangle; the pages only name the mask as an experiment parameter, section
 * 06 of the same page). With Nq queries and Nk >= Nq keys the triangle is
 * aligned at the bottom right: query i sees key j iff j <= i + (Nk - Nq), so
 * the last query sees every key (the decode / prefill reading).
 *
 * Backward, for an upstream gradient dO and no gradient through L (blog page
 * "Flash Attention 原理与实现", section "Backward 的 Tiling 策略", written out):
 *   dV = P^T dO
 *   dP = dO V^T
 *   D_i = sum_c dO_ic O_ic
 *   dS = P o (dP - D)            (softmax gradient, row-wise)
 *   dQ = scale * dS K
 *   dK = scale * dS^T Q
 * The factor `scale` in dQ/dK makes these the true derivatives of O(Q,K,V);
 * the finite-difference tests pin it.
 *
 * Layout: every matrix is contiguous [B][H][rows][d] (row-major) with Nq rows
 * for Q, O, dO, dQ and Nk rows for K, V, dK, dV; L is [B][H][Nq].
 * All arithmetic is double precision; the max is subtracted before exp, as
 * the tutorial's section 02 prescribes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double dot(const double *a, const double *b, int d) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += a[c] * b[c];
  return s;
}

/* Number of keys query row i may see (a prefix of the keys). */
static int visible_keys(int i, int Nq, int Nk, int causal) {
  if (!causal) return Nk;
  const int n = i + 1 + (Nk - Nq);
  return n < Nk ? n : Nk;
}

/* One query row of one head: scores s[0..nk), probabilities p, output o, and
 * the log-sum-exp. q is the query row, k/v point at the head's [N][d] keys and
 * values. Returns L_i. */
static double row_forward(const double *q, const double *k, const double *v,
                          int nk, int d, double scale, double *s, double *p,
                          double *o) {
  double m = -INFINITY;
  for (int j = 0; j < nk; ++j) {
    s[j] = scale * dot(q, k + (size_t)j * d, d);
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int j = 0; j < nk; ++j) {
    p[j] = exp(s[j] - m);
    l += p[j];
  }
  for (int j = 0; j < nk; ++j) p[j] /= l;
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  for (int j = 0; j < nk; ++j) {
    const double *vj = v + (size_t)j * d;
    for (int c = 0; c < d; ++c) o[c] += p[j] * vj[c];
  }
  return m + log(l);
}

/* Forward over all heads and rows, Nq queries and Nk keys per head. */
void oracle_fwd_kv(const double *q, const double *k, const double *v, double *o,
                   double *lse, int B, int H, int Nq, int Nk, int d, double scale,
                   int causal) {
  const int64_t rows = (int64_t)B * H * Nq;
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
    double *p = (double *)malloc(sizeof(double) * (size_t)Nk);
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < rows; ++r) {
      const int64_t bh = r / Nq;
      const int i = (int)(r % Nq);
      const size_t khead = (size_t)bh * Nk * d;
      lse[r] = row_forward(q + (size_t)r * d, k + khead, v + khead,
                           visible_keys(i, Nq, Nk, causal), d, scale, s, p,
                           o + (size_t)r * d);
    }
    free(s);
    free(p);
  }
}

/* Forward with Nq = Nk = N. */
void oracle_fwd(const double *q, const double *k, const double *v, double *o,
                double *lse, int B, int H, int N, int d, double scale,
                int causal) {
  oracle_fwd_kv(q, k, v, o, lse, B, H, N, N, d, scale, causal);
}

/* Full softmax matrix P of one head (small N only; for invariant tests). */
void oracle_probs(const double *q, const double *k, int N, int d, double scale,
                  int causal, double *P) {
  double *s = (double *)malloc(sizeof(double) * (size_t)N);
  double *o = (double *)malloc(sizeof(double) * (size_t)d);
  double *vz = (double *)calloc((size_t)N * d, sizeof(double));
  for (int i = 0; i < N; ++i) {
    double *prow = P + (size_t)i * N;
    int nk = visible_keys(i, N, N, causal);
    row_forward(q + (size_t)i * d, k, vz, nk, d, scale, s, prow, o);
    for (int j = nk; j < N; ++j) prow[j] = 0.0;
  }
  free(s);
  free(o);
  free(vz);
}

/* Backward over all heads, Nq queries and Nk keys per head. Outputs dq, dk,
 * dv are overwritten.
 * Heads are processed one after another; inside a head the query rows are
 * dealt to threads in fixed chunks of 16 rows, round robin (so the long rows
 * of a causal head are spread evenly). Each thread runs its rows forward in full
 * (S row, P row, O row, D_i), writes dQ_i, and adds its rows' terms of dK and
 * dV into private [N][d] sums, which are then added together in thread order
 * (so the result does not depend on scheduling). */
void oracle_bwd_kv(const double *q, const double *k, const double *v,
                   const double *dO, double *dq, double *dk, double *dv, int B,
                   int H, int Nq, int Nk, int d, double scale, int causal) {
  const int64_t heads = (int64_t)B * H;
  const size_t qs = (size_t)Nq * d, hs = (size_t)Nk * d;
  int nthr = 1;
#ifdef _OPENMP
  nthr = omp_get_max_threads();
#endif
  double *part = (double *)malloc(sizeof(double) * 2 * hs * (size_t)nthr);
  for (int64_t bh = 0; bh < heads; ++bh) {
    const size_t qoff = (size_t)bh * qs, off = (size_t)bh * hs;
    const double *qh = q + qoff, *kh = k + off, *vh = v + off, *doh = dO + qoff;
    double *dqh = dq + qoff;
    int used = 1;
#pragma omp parallel num_threads(nthr)
    {
      int t = 0;
#ifdef _OPENMP
      t = omp_get_thread_num();
#pragma omp single
      used = omp_get_num_threads();
#endif
      double *pk = part + (size_t)t * 2 * hs;
      double *pv = pk + hs;
      memset(pk, 0, sizeof(double) * 2 * hs);
      double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
      double *p = (double *)malloc(sizeof(double) * (size_t)Nk);
      double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static, 16)
      for (int i = 0; i < Nq; ++i) {
        const double *qi = qh + (size_t)i * d;
        const double *doi = doh + (size_t)i * d;
        const int nk = visible_keys(i, Nq, Nk, causal);
        row_forward(qi, kh, vh, nk, d, scale, s, p, o);
        const double Di = dot(doi, o, d);
        double *dqi = dqh + (size_t)i * d;
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        for (int j = 0; j < nk; ++j) {
          const double *kj = kh + (size_t)j * d;
          const double dPij = dot(doi, vh + (size_t)j * d, d);
          const double dSij = p[j] * (dPij - Di);
          double *dkj = pk + (size_t)j * d;
          double *dvj = pv + (size_t)j * d;
          for (int c = 0; c < d; ++c) {
            dqi[c] += scale * dSij * kj[c];
            dkj[c] += scale * dSij * qi[c];
            dvj[c] += p[j] * doi[c];
          }
        }
      }
      free(s);
      free(p);
      free(o);
    }
    double *dkh = dk + off, *dvh = dv + off;
    memset(dkh, 0, sizeof(double) * hs);
    memset(dvh, 0, sizeof(double) * hs);
    for (int t = 0; t < used; ++t) {
      const double *pk = part + (size_t)t * 2 * hs;
      const double *pv = pk + hs;
      for (size_t x = 0; x < hs; ++x) {
        dkh[x] += pk[x];
        dvh[x] += pv[x];
      }
    }
  }
  free(part);
}

/* Backward with Nq = Nk = N. */
void oracle_bwd(const double *q, const double *k, const double *v,
                const double *dO, double *dq, double *dk, double *dv, int B,
                int H, int N, int d, double scale, int causal) {
  oracle_bwd_kv(q, k, v, dO, dq, dk, dv, B, H, N, N, d, scale, causal);
}

/* Sampled query rows of one head: O_i, L_i and dQ_i for rows[0..nrows).
 * q,k,v,dO are the head's [N][d] blocks. Each row costs O(N d). */
void oracle_query_rows(const double *q, const double *k, const double *v,
                       const double *dO, int N, int d, double scale, int causal,
                       const int64_t *rows, int nrows, double *o_out,
                       double *lse_out, double *dq_out) {
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < nrows; ++r) {
      const int i = (int)rows[r];
      const double *qi = q + (size_t)i * d;
      const double *doi = dO + (size_t)i * d;
      double *oi = o_out + (size_t)r * d;
      const int nk = visible_keys(i, N, N, causal);
      lse_out[r] = row_forward(qi, k, v, nk, d, scale, s, p, oi);
      const double Di = dot(doi, oi, d);
      double *dqi = dq_out + (size_t)r * d;
      for (int c = 0; c < d; ++c) dqi[c] = 0.0;
      for (int j = 0; j < nk; ++j) {
        const double dSij = p[j] * (dot(doi, v + (size_t)j * d, d) - Di);
        const double *kj = k + (size_t)j * d;
        for (int c = 0; c < d; ++c) dqi[c] += scale * dSij * kj[c];
      }
    }
    free(s);
    free(p);
  }
}

/* Sampled key rows of one head: dK_j and dV_j for keys[0..nkeys).
 * Every query row that sees one of the keys contributes, so each such row is
 * run forward in full (its P row and D_i), then its terms for the sampled keys
 * are added. Rows are split over threads with private partial sums that are
 * added at the end. */
void oracle_key_rows(const double *q, const double *k, const double *v,
                     const double *dO, int N, int d, double scale, int causal,
                     const int64_t *keys, int nkeys, double *dk_out,
                     double *dv_out) {
  int64_t jmin = N;
  for (int t = 0; t < nkeys; ++t)
    if (keys[t] < jmin) jmin = keys[t];
  const int first_row = causal ? (int)jmin : 0;
  const size_t acc = (size_t)nkeys * d;
  memset(dk_out, 0, sizeof(double) * acc);
  memset(dv_out, 0, sizeof(double) * acc);
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    double *pk = (double *)calloc(acc, sizeof(double));
    double *pv = (double *)calloc(acc, sizeof(double));
#pragma omp for schedule(dynamic, 8)
    for (int i = first_row; i < N; ++i) {
      const double *qi = q + (size_t)i * d;
      const double *doi = dO + (size_t)i * d;
      const int nk = visible_keys(i, N, N, causal);
      row_forward(qi, k, v, nk, d, scale, s, p, o);
      const double Di = dot(doi, o, d);
      for (int t = 0; t < nkeys; ++t) {
        const int j = (int)keys[t];
        if (j >= nk) continue;
        const double dSij = p[j] * (dot(doi, v + (size_t)j * d, d) - Di);
        double *a = pk + (size_t)t * d;
        double *b = pv + (size_t)t * d;
        for (int c = 0; c < d; ++c) {
          a[c] += scale * dSij * qi[c];
          b[c] += p[j] * doi[c];
        }
      }
    }
#pragma omp critical
    {
      for (size_t x = 0; x < acc; ++x) {
        dk_out[x] += pk[x];
        dv_out[x] += pv[x];
      }
    }
    free(s);
    free(p);
    free(o);
    free(pk);
    free(pv);
  }
}

/* ------------------------------------------------------------------ dropout
 *
 * Dropout on the attention probabilities. The tutorial page
 * "research-attention" leaves it out of the plain definition (section 01) and
 * asks that its probability and its forward/backward scope be held fixed in a
 * comparison (section 06); the pages give neither its placement nor a random
 * number generator. The reading taken here is the usual one:
 *   Z_ij in {0, 1} i.i.d. with P(Z_ij = 1) = 1 - p,
 *   Pd = P o Z / (1 - p),  O = Pd V,
 *   L stays the log-sum-exp of the undropped scores;
 * and the backward with the same Z:
 *   dV = Pd^T dO,  dP = (dO V^T) o Z / (1 - p),  D_i = sum_c dO_ic O_ic,
 *   dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q
 * (dropped entries still enter dS through -P_ij D_i).
 *
 * Z comes from the counter-based generator Philox4x32-10 (Salmon, Moraes,
 * Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
 * ten rounds of two 32x32 -> 64-bit products with the multipliers and
 * Weyl key increments that paper gives. The key is the 64-bit seed (low word
 * first); the call for element (i, j) of head h has counter
 * (j / 4, i / 4, h, offset) and returns four 32-bit words; byte j mod 4 of
 * word i mod 4 (least significant byte first) is u_ij in 0..255, and the
 * element is kept iff u_ij >= t. The caller passes t = round(256 p) in
 * [0, 255]: the probability is applied as t / 256 and kept entries are scaled
 * by 256 / (256 - t).
 */
static void philox_round(uint32_t c[4], const uint32_t k[2]) {
  const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
  const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
  const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
  const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
  const uint32_t n0 = hi1 ^ c[1] ^ k[0], n2 = hi0 ^ c[3] ^ k[1];
  c[0] = n0;
  c[1] = lo1;
  c[2] = n2;
  c[3] = lo0;
}

/* Philox4x32 with ten rounds: out = f(ctr, key). */
void oracle_philox4x32_10(const uint32_t *ctr, const uint32_t *key, uint32_t *out) {
  uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
  uint32_t k[2] = {key[0], key[1]};
  for (int r = 0; r < 10; ++r) {
    philox_round(c, k);
    k[0] += 0x9E3779B9u;
    k[1] += 0xBB67AE85u;
  }
  for (int w = 0; w < 4; ++w) out[w] = c[w];
}

/* 1 if element (i, j) of head h is kept, 0 if dropped. */
static int dropout_keep(uint64_t seed, uint32_t offset, int t, int64_t h, int i, int j) {
  const uint32_t ctr[4] = {(uint32_t)(j / 4), (uint32_t)(i / 4), (uint32_t)h, offset};
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t w[4];
  oracle_philox4x32_10(ctr, key, w);
  const uint32_t u = (w[i % 4] >> (8 * (j % 4))) & 0xFFu;
  return u >= (uint32_t)t;
}

/* Keep mask [Nq][Nk] of head h (1 = kept). */
void oracle_dropout_mask(uint64_t seed, uint32_t offset, int t, int64_t h, int Nq, int Nk,
                         unsigned char *mask) {
  for (int i = 0; i < Nq; ++i)
    for (int j = 0; j < Nk; ++j) mask[(size_t)i * Nk + j] = (unsigned char)dropout_keep(seed, offset, t, h, i, j);
}

/* One query row with dropout: L_i (undropped), the dropped output o, and the
 * undropped probabilities p[0..nk) of the row. */
static double row_forward_dropout(const double *q, const double *k, const double *v, int nk, int d,
                                  double scale, uint64_t seed, uint32_t offset, int t, int64_t h, int i,
                                  double *s, double *p, double *o) {
  const double L = row_forward(q, k, v, nk, d, scale, s, p, o);
  const double inv_keep = 256.0 / (256.0 - t);
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  for (int j = 0; j < nk; ++j) {
    if (!dropout_keep(seed, offset, t, h, i, j)) continue;
    const double *vj = v + (size_t)j * d;
    for (int c = 0; c < d; ++c) o[c] += p[j] * inv_keep * vj[c];
  }
  return L;
}

/* Forward with dropout, Nq queries and Nk keys per head. */
void oracle_fwd_dropout_kv(const double *q, const double *k, const double *v, double *o, double *lse,
                           int B, int H, int Nq, int Nk, int d, double scale, int causal, uint64_t seed,
                           uint32_t offset, int t) {
  const int64_t rows = (int64_t)B * H * Nq;
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
    double *p = (double *)malloc(sizeof(double) * (size_t)Nk);
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < rows; ++r) {
      const int64_t bh = r / Nq;
      const int i = (int)(r % Nq);
      const size_t khead = (size_t)bh * Nk * d;
      lse[r] = row_forward_dropout(q + (size_t)r * d, k + khead, v + khead, visible_keys(i, Nq, Nk, causal), d,
                                   scale, seed, offset, t, bh, i, s, p, o + (size_t)r * d);
    }
    free(s);
    free(p);
  }
}

/* Backward with dropout (same Z as the forward with the same seed, offset
 * and t). Rows of a head are split statically over threads as in
 * oracle_bwd_kv, with the dK / dV partial sums added in thread order. */
void oracle_bwd_dropout_kv(const double *q, const double *k, const double *v, const double *dO, double *dq,
                           double *dk, double *dv, int B, int H, int Nq, int Nk, int d, double scale, int causal,
                           uint64_t seed, uint32_t offset, int t) {
  const int64_t heads = (int64_t)B * H;
  const size_t qs = (size_t)Nq * d, hs = (size_t)Nk * d;
  const double inv_keep = 256.0 / (256.0 - t);
  int nthr = 1;
#ifdef _OPENMP
  nthr = omp_get_max_threads();
#endif
  double *part = (double *)malloc(sizeof(double) * 2 * hs * (size_t)nthr);
  for (int64_t bh = 0; bh < heads; ++bh) {
    const size_t qoff = (size_t)bh * qs, off = (size_t)bh * hs;
    const double *qh = q + qoff, *kh = k + off, *vh = v + off, *doh = dO + qoff;
    double *dqh = dq + qoff;
    int used = 1;
#pragma omp parallel num_threads(nthr)
    {
      int tid = 0;
#ifdef _OPENMP
      tid = omp_get_thread_num();
#pragma omp single
      used = omp_get_num_threads();
#endif
      double *pk = part + (size_t)tid * 2 * hs;
      double *pv = pk + hs;
      memset(pk, 0, sizeof(double) * 2 * hs);
      double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
      double *p = (double *)malloc(sizeof(double) * (size_t)Nk);
      double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static, 16)
      for (int i = 0; i < Nq; ++i) {
        const double *qi = qh + (size_t)i * d;
        const double *doi = doh + (size_t)i * d;
        const int nk = visible_keys(i, Nq, Nk, causal);
        row_forward_dropout(qi, kh, vh, nk, d, scale, seed, offset, t, bh, i, s, p, o);
        const double Di = dot(doi, o, d);
        double *dqi = dqh + (size_t)i * d;
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        for (int j = 0; j < nk; ++j) {
          const double *kj = kh + (size_t)j * d;
          const int z = dropout_keep(seed, offset, t, bh, i, j);
          const double dPij = z ? dot(doi, vh + (size_t)j * d, d) * inv_keep : 0.0;
          const double dSij = p[j] * (dPij - Di);
          const double pdij = z ? p[j] * inv_keep : 0.0;
          double *dkj = pk + (size_t)j * d;
          double *dvj = pv + (size_t)j * d;
          for (int c = 0; c < d; ++c) {
            dqi[c] += scale * dSij * kj[c];
            dkj[c] += scale * dSij * qi[c];
            dvj[c] += pdij * doi[c];
          }
        }
      }
      free(s);
      free(p);
      free(o);
    }
    double *dkh = dk + off, *dvh = dv + off;
    memset(dkh, 0, sizeof(double) * hs);
    memset(dvh, 0, sizeof(double) * hs);
    for (int u = 0; u < used; ++u) {
      const double *pk = part + (size_t)u * 2 * hs;
      const double *pv = pk + hs;
      for (size_t x = 0; x < hs; ++x) {
        dkh[x] += pk[x];
        dvh[x] += pv[x];
      }
    }
  }
  free(part);
}

/* Threads the OpenMP runtime will use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

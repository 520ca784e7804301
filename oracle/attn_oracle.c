/* Plain fp64 CPU oracle for causal grouped-query attention, forward and
 * closed-form backward.  TEST INFRASTRUCTURE ONLY: see attn_oracle.h for what
 * it computes, the passages it follows and who may use it.
 *
 * Written for readability, not speed: one explicit softmax row per query, no
 * tiling, no online softmax, no fusion.  Every sum runs in ascending index
 * order inside one thread.
 */
#include "attn_oracle.h"

#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Offset of element [b, t, h, 0] in a [B, T, H, D] tensor. */
static size_t row_off(int b, int t, int h, int T, int H, int D) {
  return (((size_t)b * T + t) * H + h) * (size_t)D;
}

/* Number of keys query i may attend to. */
static int visible_keys(int i, int T, int causal) { return causal ? i + 1 : T; }

static double dot(const double* x, const double* y, int D) {
  double s = 0.0;
  for (int d = 0; d < D; ++d) s += x[d] * y[d];
  return s;
}

/* Softmax row of query (b, h, i): p[j] = P_ij for every j < T (exactly 0 for
 * masked keys) and *lse = LSE_i. */
static void softmax_row(const double* q, const double* k, int b, int h, int i, int T, int Hq,
                        int Hkv, int D, double scale, int causal, double* p, double* lse) {
  const int g = h / (Hq / Hkv);
  const int n = visible_keys(i, T, causal);
  const double* qi = q + row_off(b, i, h, T, Hq, D);
  double m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    const double s = scale * dot(qi, k + row_off(b, j, g, T, Hkv, D), D);
    p[j] = s;
    if (s > m) m = s;
  }
  double sum = 0.0;
  for (int j = 0; j < n; ++j) sum += exp(p[j] - m);
  const double l = m + log(sum);
  for (int j = 0; j < n; ++j) p[j] = exp(p[j] - l);
  for (int j = n; j < T; ++j) p[j] = 0.0;
  *lse = l;
}

/* O_i = sum_j P_ij V_j for the KV head g. */
static void weighted_values(const double* p, const double* v, int b, int g, int n, int T, int Hkv,
                            int D, double* out) {
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  for (int j = 0; j < n; ++j) {
    const double* vj = v + row_off(b, j, g, T, Hkv, D);
    for (int d = 0; d < D; ++d) out[d] += p[j] * vj[d];
  }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_attn_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                     int B, int T, int Hq, int Hkv, int D, double scale, int causal) {
  const int G = Hq / Hkv;
#pragma omp parallel
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#pragma omp for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < Hq; ++h)
        for (int i = 0; i < T; ++i) {
          double l;
          softmax_row(q, k, b, h, i, T, Hq, Hkv, D, scale, causal, p, &l);
          lse[((size_t)b * Hq + h) * T + i] = l;
          weighted_values(p, v, b, h / G, visible_keys(i, T, causal), T, Hkv, D,
                          o + row_off(b, i, h, T, Hq, D));
        }
    free(p);
  }
}

double oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                       double* dq, double* dk, double* dv, double* delta, int B, int T, int Hq,
                       int Hkv, int D, double scale, int causal) {
  const int G = Hq / Hkv;
  double worst = 0.0;
#pragma omp parallel reduction(max : worst)
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double* dp = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double* oi = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
      for (int g = 0; g < Hkv; ++g) {
        /* This thread owns dK and dV of (b, g). */
        for (int j = 0; j < T; ++j) {
          memset(dk + row_off(b, j, g, T, Hkv, D), 0, sizeof(double) * (size_t)D);
          memset(dv + row_off(b, j, g, T, Hkv, D), 0, sizeof(double) * (size_t)D);
        }
        for (int h = g * G; h < (g + 1) * G; ++h)
          for (int i = 0; i < T; ++i) {
            const int n = visible_keys(i, T, causal);
            const double* qi = q + row_off(b, i, h, T, Hq, D);
            const double* doi = dout + row_off(b, i, h, T, Hq, D);
            double l;
            softmax_row(q, k, b, h, i, T, Hq, Hkv, D, scale, causal, p, &l);
            weighted_values(p, v, b, g, n, T, Hkv, D, oi);
            const double d1 = dot(doi, oi, D);
            double d2 = 0.0;
            for (int j = 0; j < n; ++j) {
              dp[j] = dot(doi, v + row_off(b, j, g, T, Hkv, D), D);
              d2 += p[j] * dp[j];
            }
            const double dis = fabs(d1 - d2) / fmax(1.0, fabs(d1));
            if (dis > worst) worst = dis;
            delta[((size_t)b * Hq + h) * T + i] = d1;
            double* dqi = dq + row_off(b, i, h, T, Hq, D);
            for (int d = 0; d < D; ++d) dqi[d] = 0.0;
            for (int j = 0; j < n; ++j) {
              const double ds = p[j] * (dp[j] - d1);
              const double* kj = k + row_off(b, j, g, T, Hkv, D);
              double* dkj = dk + row_off(b, j, g, T, Hkv, D);
              double* dvj = dv + row_off(b, j, g, T, Hkv, D);
              for (int d = 0; d < D; ++d) {
                dqi[d] += ds * kj[d];
                dkj[d] += ds * qi[d];
                dvj[d] += p[j] * doi[d];
              }
            }
            for (int d = 0; d < D; ++d) dqi[d] *= scale;
          }
        for (int j = 0; j < T; ++j) {
          double* dkj = dk + row_off(b, j, g, T, Hkv, D);
          for (int d = 0; d < D; ++d) dkj[d] *= scale;
        }
      }
    free(p);
    free(dp);
    free(oi);
  }
  return worst;
}

void oracle_rowdot(const double* o, const double* dout, double* delta, int B, int T, int H, int D) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h)
      for (int i = 0; i < T; ++i)
        delta[((size_t)b * H + h) * T + i] =
            dot(dout + row_off(b, i, h, T, H, D), o + row_off(b, i, h, T, H, D), D);
}

void oracle_attn_probs(const double* q, const double* k, double* p, int b, int h, int B, int T,
                       int Hq, int Hkv, int D, double scale, int causal) {
  (void)B;
  for (int i = 0; i < T; ++i) {
    double l;
    softmax_row(q, k, b, h, i, T, Hq, Hkv, D, scale, causal, p + (size_t)i * T, &l);
  }
}

void oracle_attn_rows(const double* q, const double* k, const double* v, const double* dout, int n,
                      const int* rb, const int* rh, const int* ri, double* o_rows,
                      double* lse_rows, double* dq_rows, int B, int T, int Hq, int Hkv, int D,
                      double scale, int causal) {
  (void)B;
  const int G = Hq / Hkv;
#pragma omp parallel
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#pragma omp for schedule(dynamic)
    for (int s = 0; s < n; ++s) {
      const int b = rb[s], h = rh[s], i = ri[s], g = h / G;
      const int nv = visible_keys(i, T, causal);
      double* oi = o_rows + (size_t)s * D;
      softmax_row(q, k, b, h, i, T, Hq, Hkv, D, scale, causal, p, &lse_rows[s]);
      weighted_values(p, v, b, g, nv, T, Hkv, D, oi);
      if (dq_rows) {
        const double* doi = dout + row_off(b, i, h, T, Hq, D);
        const double d1 = dot(doi, oi, D);
        double* dqi = dq_rows + (size_t)s * D;
        for (int d = 0; d < D; ++d) dqi[d] = 0.0;
        for (int j = 0; j < nv; ++j) {
          const double* kj = k + row_off(b, j, g, T, Hkv, D);
          const double ds = p[j] * (dot(doi, v + row_off(b, j, g, T, Hkv, D), D) - d1);
          for (int d = 0; d < D; ++d) dqi[d] += ds * kj[d];
        }
        for (int d = 0; d < D; ++d) dqi[d] *= scale;
      }
    }
    free(p);
  }
}

void oracle_kv_rows(const double* q, const double* k, const double* v, const double* dout, int b,
                    int g, int nj, const int* js, double* dk_rows, double* dv_rows, int B, int T,
                    int Hq, int Hkv, int D, double scale, int causal) {
  (void)B;
  const int G = Hq / Hkv;
  double* lse = (double*)malloc(sizeof(double) * (size_t)G * (size_t)(T > 0 ? T : 1));
  double* del = (double*)malloc(sizeof(double) * (size_t)G * (size_t)(T > 0 ? T : 1));
  /* Row statistics (LSE_i and D_i) of every query row of the group's heads. */
#pragma omp parallel
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double* oi = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for collapse(2) schedule(dynamic)
    for (int hh = 0; hh < G; ++hh)
      for (int i = 0; i < T; ++i) {
        const int h = g * G + hh;
        double l;
        softmax_row(q, k, b, h, i, T, Hq, Hkv, D, scale, causal, p, &l);
        weighted_values(p, v, b, g, visible_keys(i, T, causal), T, Hkv, D, oi);
        lse[(size_t)hh * T + i] = l;
        del[(size_t)hh * T + i] = dot(dout + row_off(b, i, h, T, Hq, D), oi, D);
      }
    free(p);
    free(oi);
  }
#pragma omp parallel for schedule(dynamic)
  for (int s = 0; s < nj; ++s) {
    const int j = js[s];
    const double* kj = k + row_off(b, j, g, T, Hkv, D);
    const double* vj = v + row_off(b, j, g, T, Hkv, D);
    double* dkj = dk_rows + (size_t)s * D;
    double* dvj = dv_rows + (size_t)s * D;
    for (int d = 0; d < D; ++d) dkj[d] = dvj[d] = 0.0;
    for (int hh = 0; hh < G; ++hh) {
      const int h = g * G + hh;
      for (int i = causal ? j : 0; i < T; ++i) {
        const double* qi = q + row_off(b, i, h, T, Hq, D);
        const double* doi = dout + row_off(b, i, h, T, Hq, D);
        const double pij = exp(scale * dot(qi, kj, D) - lse[(size_t)hh * T + i]);
        const double ds = pij * (dot(doi, vj, D) - del[(size_t)hh * T + i]);
        for (int d = 0; d < D; ++d) {
          dvj[d] += pij * doi[d];
          dkj[d] += ds * qi[d];
        }
      }
    }
    for (int d = 0; d < D; ++d) dkj[d] *= scale;
  }
  free(lse);
  free(del);
}

/* ------------------------------------------------------------------------
 * Packed variable-length batches, Tq != Tk allowed (see attn_oracle.h).
 * Sequence s owns query rows cu_q[s] .. cu_q[s+1]-1 and key rows
 * cu_k[s] .. cu_k[s+1]-1; nothing crosses a sequence boundary.  The loops
 * follow the fixed-length functions above in the same order, so a batch of
 * equal-length sequences gives the same bytes as those functions.
 * ------------------------------------------------------------------------ */

/* Keys 0 .. n-1 of its sequence that query i sees: all tk, or under the
 * causal mask those with j <= i + (tk - tq) (the mask's diagonal ends in the
 * bottom-right corner of the tq x tk score matrix), clamped to [0, tk]. */
static int seq_visible(int i, int tq, int tk, int causal) {
  if (!causal) return tk;
  const int n = i + 1 + (tk - tq);
  return n < 0 ? 0 : (n > tk ? tk : n);
}

static size_t packed_off(int row, int h, int H, int D) { return ((size_t)row * H + h) * (size_t)D; }

/* Softmax row of packed query row `qrow` (head h) against the n keys from
 * packed key row `k0` (KV head g): prob[j] for j < n, *lse_out.  n == 0 gives
 * *lse_out = -inf and no probabilities. */
static void seq_softmax_row(const double* q, const double* k, int qrow, int k0, int n, int h,
                            int g, int Hq, int Hkv, int D, double scale, double* prob,
                            double* lse_out) {
  if (n == 0) {
    *lse_out = -INFINITY;
    return;
  }
  const double* qr = q + packed_off(qrow, h, Hq, D);
  double mx = -INFINITY;
  for (int j = 0; j < n; ++j) {
    prob[j] = scale * dot(qr, k + packed_off(k0 + j, g, Hkv, D), D);
    if (prob[j] > mx) mx = prob[j];
  }
  double tot = 0.0;
  for (int j = 0; j < n; ++j) tot += exp(prob[j] - mx);
  const double lrow = mx + log(tot);
  for (int j = 0; j < n; ++j) prob[j] = exp(prob[j] - lrow);
  *lse_out = lrow;
}

/* orow = sum_{j < n} prob[j] V[k0 + j, g, :]; zero when n == 0. */
static void seq_weighted_values(const double* prob, const double* v, int k0, int n, int g, int Hkv,
                                int D, double* orow) {
  for (int d = 0; d < D; ++d) orow[d] = 0.0;
  for (int j = 0; j < n; ++j) {
    const double* vr = v + packed_off(k0 + j, g, Hkv, D);
    for (int d = 0; d < D; ++d) orow[d] += prob[j] * vr[d];
  }
}

static int max_len(int n_seq, const int* cu) {
  int m = 1;
  for (int s = 0; s < n_seq; ++s)
    if (cu[s + 1] - cu[s] > m) m = cu[s + 1] - cu[s];
  return m;
}

void oracle_attn_fwd_varlen(const double* q, const double* k, const double* v, double* o,
                            double* lse, int n_seq, const int* cu_q, const int* cu_k, int Hq,
                            int Hkv, int D, double scale, int causal) {
  const int G = Hq / Hkv;
  const int total_q = cu_q[n_seq];
  const int tk_max = max_len(n_seq, cu_k);
#pragma omp parallel
  {
    double* prob = (double*)malloc(sizeof(double) * (size_t)tk_max);
#pragma omp for collapse(2) schedule(dynamic)
    for (int s = 0; s < n_seq; ++s)
      for (int h = 0; h < Hq; ++h) {
        const int tq = cu_q[s + 1] - cu_q[s], tk = cu_k[s + 1] - cu_k[s];
        for (int i = 0; i < tq; ++i) {
          const int row = cu_q[s] + i, n = seq_visible(i, tq, tk, causal);
          seq_softmax_row(q, k, row, cu_k[s], n, h, h / G, Hq, Hkv, D, scale, prob,
                          &lse[(size_t)h * total_q + row]);
          seq_weighted_values(prob, v, cu_k[s], n, h / G, Hkv, D, o + packed_off(row, h, Hq, D));
        }
      }
    free(prob);
  }
}

double oracle_attn_bwd_varlen(const double* q, const double* k, const double* v,
                              const double* dout, double* dq, double* dk, double* dv,
                              double* delta, int n_seq, const int* cu_q, const int* cu_k, int Hq,
                              int Hkv, int D, double scale, int causal) {
  const int G = Hq / Hkv;
  const int total_q = cu_q[n_seq];
  const int tk_max = max_len(n_seq, cu_k);
  double worst = 0.0;
#pragma omp parallel reduction(max : worst)
  {
    double* prob = (double*)malloc(sizeof(double) * (size_t)tk_max);
    double* dprob = (double*)malloc(sizeof(double) * (size_t)tk_max);
    double* orow = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for collapse(2) schedule(dynamic)
    for (int s = 0; s < n_seq; ++s)
      for (int g = 0; g < Hkv; ++g) {
        /* This thread owns dK, dV of (s, g) and dQ of the group's query rows. */
        const int tq = cu_q[s + 1] - cu_q[s], tk = cu_k[s + 1] - cu_k[s], k0 = cu_k[s];
        for (int j = 0; j < tk; ++j) {
          memset(dk + packed_off(k0 + j, g, Hkv, D), 0, sizeof(double) * (size_t)D);
          memset(dv + packed_off(k0 + j, g, Hkv, D), 0, sizeof(double) * (size_t)D);
        }
        for (int h = g * G; h < g * G + G; ++h)
          for (int i = 0; i < tq; ++i) {
            const int row = cu_q[s] + i, n = seq_visible(i, tq, tk, causal);
            const double* qr = q + packed_off(row, h, Hq, D);
            const double* dor = dout + packed_off(row, h, Hq, D);
            double* dqr = dq + packed_off(row, h, Hq, D);
            double lrow;
            seq_softmax_row(q, k, row, k0, n, h, g, Hq, Hkv, D, scale, prob, &lrow);
            seq_weighted_values(prob, v, k0, n, g, Hkv, D, orow);
            const double dl = dot(dor, orow, D);
            double dl2 = 0.0;
            for (int j = 0; j < n; ++j) {
              dprob[j] = dot(dor, v + packed_off(k0 + j, g, Hkv, D), D);
              dl2 += prob[j] * dprob[j];
            }
            const double gap = fabs(dl - dl2) / fmax(1.0, fabs(dl));
            if (gap > worst) worst = gap;
            delta[(size_t)h * total_q + row] = dl;
            for (int d = 0; d < D; ++d) dqr[d] = 0.0;
            for (int j = 0; j < n; ++j) {
              const double dsc = prob[j] * (dprob[j] - dl);
              const double* kr = k + packed_off(k0 + j, g, Hkv, D);
              double* dkr = dk + packed_off(k0 + j, g, Hkv, D);
              double* dvr = dv + packed_off(k0 + j, g, Hkv, D);
              for (int d = 0; d < D; ++d) {
                dqr[d] += dsc * kr[d];
                dkr[d] += dsc * qr[d];
                dvr[d] += prob[j] * dor[d];
              }
            }
            for (int d = 0; d < D; ++d) dqr[d] = dqr[d] * scale;
          }
        for (int j = 0; j < tk; ++j) {
          double* dkr = dk + packed_off(k0 + j, g, Hkv, D);
          for (int d = 0; d < D; ++d) dkr[d] = dkr[d] * scale;
        }
      }
    free(prob);
    free(dprob);
    free(orow);
  }
  return worst;
}

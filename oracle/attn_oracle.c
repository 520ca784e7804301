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

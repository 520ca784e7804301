/* Plain fp64 CPU oracle for the embedding-lookup gradient.  TEST
 * INFRASTRUCTURE ONLY: see embed_oracle.h for what it computes, the passages
 * it follows and who may use it. */
#include "embed_oracle.h"

#include <stddef.h>
#include <string.h>

int oracle_embed_grad(const int* ids, const double* dy, double* dw, int N, int V, int E) {
  if (N < 0 || V < 0 || E < 0) return -1;
  for (int t = 0; t < N; ++t)
    if (ids[t] < 0 || ids[t] >= V) return -1;
  memset(dw, 0, sizeof(double) * (size_t)V * (size_t)E);
  /* Each thread owns whole columns of dw and walks the tokens in ascending
   * order, so every element is one sum in one fixed order. */
#pragma omp parallel for schedule(static)
  for (int col = 0; col < E; ++col)
    for (int t = 0; t < N; ++t) dw[(size_t)ids[t] * E + col] += dy[(size_t)t * E + col];
  return 0;
}

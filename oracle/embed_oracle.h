/* Plain fp64 CPU oracle for the gradient of an embedding lookup.
 *
 * TEST INFRASTRUCTURE ONLY, like attn_oracle.h: only the test suite and the
 * benchmark's CPU legs use it, and it shares no code with the CUDA path.
 *
 * What it computes (oxide-train README, "The trainer is not bit-identical to
 * itself after step 1": the embedding gradient there is accumulated with
 * atomics, whose order changes from launch to launch, so two runs of one
 * binary disagree from step 2 on; "Full-step profiling": B = 32, T = 1024,
 * a vocabulary of 50,257 padded to 50,432, model width 1536).  The forward
 * lookup X[t, :] = W[ids[t], :] has the gradient
 *
 *   dW[v, :] = sum over t with ids[t] == v of dY[t, :]
 *
 * written out here with the sum over t in ascending order, one fixed order,
 * so repeated runs give identical bytes.  Rows of W that no token selects get
 * exactly zero.
 *
 * Layouts (row-major, contiguous): ids int32 [N]; dy fp64 [N, E];
 * dw fp64 [V, E].
 */
#ifndef DETATTN_EMBED_ORACLE_H
#define DETATTN_EMBED_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

/* Writes dw.  Returns 0, or -1 (dw untouched) when an id lies outside
 * [0, V) or a size is negative. */
int oracle_embed_grad(const int* ids, const double* dy, double* dw, int N, int V, int E);

#ifdef __cplusplus
}
#endif
#endif

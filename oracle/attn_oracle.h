/* Plain fp64 CPU oracle for causal grouped-query scaled-dot-product attention
 * and its closed-form backward.
 *
 * TEST INFRASTRUCTURE ONLY.  The library under test never links, loads or
 * calls this code; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or table with the CUDA
 * path.
 *
 * What it computes (RustingBrain vs PyTorch/TensorFlow page, "Step 1: measure
 * before changing anything" and "Step 2: fused flash attention": a causal
 * softmax over the [seq_len, seq_len] score matrix with a per-row logsumexp,
 * probabilities recomputed from that logsumexp, and a backward producing the
 * query, key and value gradients; "The setup": grouped-query attention with
 * 12 query heads sharing 4 KV heads, head_dim 64).  The pages give no
 * formulas, so the oracle is the textbook definition of attention written out
 * with an explicit softmax row per query:
 *
 *   S_ij  = scale * sum_d Q[b,i,h,d] K[b,j,g,d],  g = h / (Hq/Hkv)
 *   S_ij  = -inf for j > i when causal
 *   LSE_i = log sum_j exp(S_ij)                     (natural log)
 *   P_ij  = exp(S_ij - LSE_i)
 *   O_i   = sum_j P_ij V[b,j,g,:]
 *   dV_j  = sum_{h in group g} sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   D_i   = dO_i . O_i      (also equal to sum_j P_ij dP_ij; both are formed)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij K_j
 *   dK_j  = scale sum_{h in group g} sum_i dS_ij Q_i
 *
 * Layouts (row-major, contiguous, all fp64):
 *   q, o, dout, dq : [B, T, Hq,  D]
 *   k, v, dk, dv   : [B, T, Hkv, D]
 *   lse, delta     : [B, Hq, T]
 *
 * Each output element is owned by one OpenMP thread and accumulated in a fixed
 * order, so repeated runs give identical bytes.
 */
#ifndef DETATTN_ORACLE_H
#define DETATTN_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

/* Forward: o and lse. */
void oracle_attn_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                     int B, int T, int Hq, int Hkv, int D, double scale, int causal);

/* Backward given dout.  The forward is recomputed inside from q, k, v.
 * Writes dq, dk, dv and delta (= rowsum(dout * o)).  Returns the largest
 * relative disagreement between the two forms of delta (dout.o versus
 * sum_j P_ij dP_ij), measured against max(1, |delta|). */
double oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                       double* dq, double* dk, double* dv, double* delta, int B, int T, int Hq,
                       int Hkv, int D, double scale, int causal);

/* The explicit probability matrix P [T, T] of one (b, h). */
void oracle_attn_probs(const double* q, const double* k, double* p, int b, int h, int B, int T,
                       int Hq, int Hkv, int D, double scale, int causal);

/* Sampled query rows: for n samples (rb[s], rh[s], ri[s]) writes
 * o_rows[s, D], lse_rows[s], dq_rows[s, D] (dq_rows may be NULL). */
void oracle_attn_rows(const double* q, const double* k, const double* v, const double* dout, int n,
                      const int* rb, const int* rh, const int* ri, double* o_rows,
                      double* lse_rows, double* dq_rows, int B, int T, int Hq, int Hkv, int D,
                      double scale, int causal);

/* Sampled key/value rows of one (b, KV head g): for the nj key positions js[s]
 * writes dk_rows[s, D] and dv_rows[s, D]. */
void oracle_kv_rows(const double* q, const double* k, const double* v, const double* dout, int b,
                    int g, int nj, const int* js, double* dk_rows, double* dv_rows, int B, int T,
                    int Hq, int Hkv, int D, double scale, int causal);

/* delta[b, h, i] = sum_d dout[b, i, h, d] * o[b, i, h, d] for a given o
 * (the rowsum that the backward's first step forms from the stored output). */
void oracle_rowdot(const double* o, const double* dout, double* delta, int B, int T, int H, int D);

/* Packed variable-length batches (no page describes them; the plainest
 * extension of the definition above).  n_seq sequences; sequence s has the
 * tq = cu_q[s+1] - cu_q[s] query rows from cu_q[s] and the tk = cu_k[s+1] -
 * cu_k[s] key rows from cu_k[s] (cu_q[0] = cu_k[0] = 0, non-decreasing).
 * Layouts: q, o, dout, dq [cu_q[n_seq], Hq, D]; k, v, dk, dv
 * [cu_k[n_seq], Hkv, D]; lse, delta [Hq, cu_q[n_seq]].  Readings:
 *   - the causal mask ends in the bottom-right corner of each sequence's
 *     tq x tk score matrix: query i sees key j iff j <= i + (tk - tq), which
 *     is j <= i when tq == tk;
 *   - a query row that sees no key (tq > tk under the mask, or tk == 0) has
 *     O = 0, LSE = -inf, dQ = 0 and delta = 0, and adds nothing to dK, dV.
 * With every tq == tk == T these equal the fixed-length functions bit for bit
 * (same operations in the same order). */
void oracle_attn_fwd_varlen(const double* q, const double* k, const double* v, double* o,
                            double* lse, int n_seq, const int* cu_q, const int* cu_k, int Hq,
                            int Hkv, int D, double scale, int causal);
double oracle_attn_bwd_varlen(const double* q, const double* k, const double* v,
                              const double* dout, double* dq, double* dk, double* dv,
                              double* delta, int n_seq, const int* cu_q, const int* cu_k, int Hq,
                              int Hkv, int D, double scale, int causal);

/* Number of OpenMP threads the oracle uses. */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif

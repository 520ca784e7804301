/* detattn: deterministic causal grouped-query flash attention for sm_103a.
 *
 * The operation (RustingBrain vs PyTorch/TensorFlow page, "Step 2: fused flash
 * attention": a fused causal attention forward and backward that never forms
 * the [seq_len, seq_len] score matrix; "Step 1": the per-row logsumexp and
 * probabilities recomputed from it; "The setup": 12 query heads sharing 4 KV
 * heads, head_dim 64; oxide-train README, "The trainer is not bit-identical to
 * itself after step 1": atomically accumulated gradients differ from run to
 * run, which this library avoids).  With g = h / (Hq / Hkv):
 *
 *   S_ij  = scale * Q[b,i,h,:] . K[b,j,g,:]      (j <= i when causal)
 *   LSE_i = ln sum_j exp(S_ij),  P_ij = exp(S_ij - LSE_i)
 *   O_i   = sum_j P_ij V[b,j,g,:]
 *   Delta_i = dO_i . O_i,  dS_ij = P_ij (dO_i . V_j - Delta_i)
 *   dQ_i  = scale sum_j dS_ij K_j
 *   dK_j  = scale sum_{h in g} sum_i dS_ij Q_i,  dV_j = sum_{h in g} sum_i P_ij dO_i
 *
 * Data layout (row-major, contiguous, device memory):
 *   q, o, dout, dq : bf16 [B, T, Hq,  D]
 *   k, v, dk, dv   : bf16 [B, T, Hkv, D]
 *   lse            : fp32 [B, Hq, T]   natural-log logsumexp of the scaled scores
 *   workspace      : caller-owned device scratch of attn_bwd_workspace_bytes()
 *
 * Conventions shared by every entry point:
 *   - Pointers are device pointers, 16-byte aligned.  The caller owns every
 *     buffer; the library allocates no device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream and never synchronise.
 *   - Arguments are validated on the host before any CUDA call; a call that
 *     returns an error launched nothing.  detattn_last_error() then gives a
 *     one-line reason (thread-local).
 *   - Inputs are never written.  Outputs are fully overwritten (no zero-fill
 *     needed); rows t >= T are never touched.
 *   - Results are bitwise identical from call to call for identical inputs
 *     and shapes on the same GPU model: every output element is produced by
 *     one thread block in a fixed order, with no atomics.
 *   - B == 0 or T == 0 is a valid empty problem: nothing is launched.
 *   - D must be 64 or 128; Hq must be a multiple of Hkv; scale must be finite
 *     and > 0; causal is 0 (full attention) or 1 (key j visible to query i iff
 *     j <= i).
 */
#ifndef DETATTN_H
#define DETATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DETATTN_OK = 0,
  DETATTN_ERR_NULL = -1,           /* a required pointer is NULL */
  DETATTN_ERR_ALIGN = -2,          /* a pointer is not 16-byte aligned */
  DETATTN_ERR_SHAPE = -3,          /* B or T < 0, Hq/Hkv < 1, Hq % Hkv != 0, or too large */
  DETATTN_ERR_HEADDIM = -4,        /* D is not 64 or 128 */
  DETATTN_ERR_SCALE = -5,          /* scale not finite or <= 0, or causal not 0/1 */
  DETATTN_ERR_CUDA = -6,           /* a CUDA runtime / driver call failed */
  DETATTN_ERR_DEVICE_TIMEOUT = -7, /* a kernel gave up waiting on a pipeline barrier */
  DETATTN_ERR_ARCH = -8,           /* current device is not compute capability 10.3 */
  DETATTN_ERR_WORKSPACE = -9       /* workspace NULL or too small */
} detattn_status;

/* Forward.  Writes o [B,T,Hq,D] (bf16) and lse [B,Hq,T] (fp32).
 * Passage: "Step 2: fused flash attention" (RustingBrain page): tiled Q K^T,
 * online softmax in base 2 with a per-row logsumexp, P V, causal tiles past the
 * diagonal skipped. */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T,
             int Hq, int Hkv, int D, float scale, int causal, void* stream);

/* Bytes of device workspace attn_bwd needs (Delta, fp32 [B,Hq,T], rounded up
 * to 256 bytes).  Returns 0 for an empty or invalid shape. */
size_t attn_bwd_workspace_bytes(int B, int T, int Hq, int Hkv, int D);

/* Backward.  Given q, k, v, the forward's o and lse, and dout, writes dq, dk,
 * dv (bf16).  Runs attn_bwd_delta, attn_bwd_dkdv and attn_bwd_dq in that
 * order on `stream`.  `workspace` (>= attn_bwd_workspace_bytes) holds Delta.
 * Passage: "Step 2: fused flash attention" and "Where the time goes now"
 * (the flash_attention_dkv kernel) on the RustingBrain page. */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, void* workspace,
             size_t workspace_bytes, int B, int T, int Hq, int Hkv, int D, float scale,
             int causal, void* stream);

/* Backward step 1 alone: delta [B,Hq,T] fp32 = rowsum(dout * o), summed in a
 * fixed order.  (Implied by recomputing P from the logsumexp in "Step 1" of
 * the RustingBrain page.) */
int attn_bwd_delta(const void* o, const void* dout, float* delta, int B, int T, int Hq, int D,
                   void* stream);

/* Backward step 2 alone: dk, dv for every KV tile, summing the query heads of
 * the GQA group inside the tile in ascending head order ("Where the time goes
 * now": flash_attention_dkv).  `delta` is the output of attn_bwd_delta. */
int attn_bwd_dkdv(const void* q, const void* k, const void* v, const float* lse,
                  const float* delta, const void* dout, void* dk, void* dv, int B, int T, int Hq,
                  int Hkv, int D, float scale, int causal, void* stream);

/* Backward step 3 alone: dq, reduced over KV tiles in ascending order by the
 * single block that owns the query tile (no atomics). */
int attn_bwd_dq(const void* q, const void* k, const void* v, const float* lse,
                const float* delta, const void* dout, void* dq, int B, int T, int Hq, int Hkv,
                int D, float scale, int causal, void* stream);

/* Synchronises `stream`, then reads and clears the device-side status word
 * that kernels set when a pipeline wait runs out (a bounded wait, default
 * limit 1 s).  Returns DETATTN_OK, DETATTN_ERR_DEVICE_TIMEOUT or
 * DETATTN_ERR_CUDA. */
int detattn_check_status(void* stream);

/* Sets the per-wait time limit used by kernels launched afterwards, in
 * nanoseconds (clamped to [1 ms, 60 s]).  Host-side setting, per process. */
void detattn_set_wait_limit_ns(unsigned long long ns);

/* Text for the last non-OK return on this thread ("" if none). */
const char* detattn_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int detattn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DETATTN_H */

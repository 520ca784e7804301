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
 *                    (row statistics of the backward; layout below)
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
 *     and shapes on the same GPU model: every output element is produced in a
 *     fixed order by one thread block (dk, dv: by the block that owns the
 *     row, adding its cluster's partial sums in rank order), with no atomics
 *     on the data.  The one atomic, the dQ step's tile counter, only deals out
 *     work.
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
  DETATTN_ERR_WORKSPACE = -9       /* workspace NULL or too small; from detattn_check_status:
                                      a dQ step ran on a workspace attn_bwd_delta had not
                                      prepared */
} detattn_status;

/* Forward.  Writes o [B,T,Hq,D] (bf16) and lse [B,Hq,T] (fp32).
 * Passage: "Step 2: fused flash attention" (RustingBrain page): tiled Q K^T,
 * online softmax in base 2 with a per-row logsumexp, P V, causal tiles past the
 * diagonal skipped. */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T,
             int Hq, int Hkv, int D, float scale, int causal, void* stream);

/* Bytes of device workspace the backward uses: R + 256, where
 * R = B * Hq * Tp * 8 rounded up to a multiple of 256 and Tp = T rounded up to
 * a multiple of 128.  Returns 0 for an empty or invalid shape.  Only the first
 * B * Hq * Tp * 8 bytes are required; see the layout below for the rest.
 *
 * Workspace layout (written by attn_bwd_delta, read by attn_bwd_dkdv and
 * attn_bwd_dq): row statistics, one (float, float) pair per (b, h, t),
 * pairs ordered [b][h][t] with t < Tp:
 *   pair.x = -LSE[b,h,t] * log2(e),   pair.y = -Delta[b,h,t]
 *   Delta[b,h,t] = sum_d dout[b,t,h,d] * o[b,t,h,d]   (fp32, fixed order)
 * and (-inf, -0) for t >= T.  Stored negated and in base 2 because the
 * kernels add them: P = exp2(S*scale*log2(e) + pair.x), dS = P (dP + pair.y).
 * At byte R: two unsigned words, a counter the dQ step takes its 128-query
 * tiles from, heaviest first (so its blocks that start early, on SMs the
 * concurrent dK/dV step frees first, take more of them), and a count of its
 * pipelines done; the last pipeline puts both back to zero, and
 * attn_bwd_delta clears them too.  Which block computes a tile changes none
 * of its bits.  Without room for them (workspace_bytes < R + 8) the dQ step
 * follows a static deal fixed by the shape and the SM count. */
size_t attn_bwd_workspace_bytes(int B, int T, int Hq, int Hkv, int D);

/* Backward.  Given q, k, v, the forward's o and lse, and dout, writes dq, dk,
 * dv (bf16).  Runs attn_bwd_delta on `stream`, then attn_bwd_dkdv on `stream`
 * and attn_bwd_dq concurrently on a library-owned side stream (forked from
 * `stream` after the Delta step with an event and joined back before the call
 * returns; created on the first call per device), so all work is ordered
 * after earlier work on `stream` and later work on `stream` sees the results.
 * `workspace` (attn_bwd_workspace_bytes, at least the row statistics' share;
 * 16-byte aligned, caller-owned, contents on entry irrelevant) holds the row
 * statistics and the dQ step's tile counter (layout above).  Passage: "Step 2: fused flash attention" and "Where the time
 * goes now" (the flash_attention_dkv kernel) on the RustingBrain page. */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, void* workspace,
             size_t workspace_bytes, int B, int T, int Hq, int Hkv, int D, float scale,
             int causal, void* stream);

/* Backward without a caller workspace, for callers that cannot allocate
 * device memory: for example a plug-in whose host application gives it no
 * allocator, or code inside a framework whose device memory is all owned by
 * its own pooled allocator, where a stray cudaMalloc can fail or fragment the
 * pool.  Same arguments, results and errors as attn_bwd minus the workspace.
 * The method has no counterpart of this on the pages; it is an interface
 * convenience.
 *
 * The row statistics live in an 8 MiB array built into the library (every
 * GPU that loads the library holds it until the process exits), so
 * B * Hq * Tp must not exceed 1,048,576 (Tp = T rounded up to 128); larger
 * problems return DETATTN_ERR_WORKSPACE without launching anything.  This
 * call never allocates memory.  Its first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current,
 * and so does the first call after that device's context was re-created
 * (cudaDeviceReset loads the library's module anew, and the array may then
 * sit elsewhere); make such a first call before any stream capture.  Every call shares the one
 * array: each call overwrites all the statistics it reads before reading
 * them, so nothing needs to start at zero, but calls that overlap on the GPU
 * (on different streams, or different host threads without ordering) race
 * on it and must not be issued. */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, int B, int T, int Hq,
                     int Hkv, int D, float scale, int causal, void* stream);

/* Backward step 1 alone: writes the workspace row statistics (layout above)
 * from o, dout and lse; Delta is the rowsum of dout * o summed in a fixed
 * order.  (Implied by recomputing P from the logsumexp, "Step 1" of the
 * RustingBrain page.) */
int attn_bwd_delta(const void* o, const void* dout, const float* lse, void* workspace,
                   size_t workspace_bytes, int B, int T, int Hq, int D, void* stream);

/* Backward step 2 alone: dk, dv for every 128-key tile, summing the query
 * heads of the GQA group inside the tile in ascending head order ("Where the
 * time goes now": flash_attention_dkv).  `workspace` holds the row statistics
 * of attn_bwd_delta. */
int attn_bwd_dkdv(const void* q, const void* k, const void* v, const void* dout,
                  const void* workspace, size_t workspace_bytes, void* dk, void* dv, int B, int T,
                  int Hq, int Hkv, int D, float scale, int causal, void* stream);

/* Backward step 3 alone: dq, reduced over key tiles in ascending order by the
 * single block that owns the 128-query tile (no atomics on the data).  Pass
 * the workspace_bytes that attn_bwd_delta got on this workspace (that call
 * cleared the tile counter; every dQ call leaves it cleared). */
int attn_bwd_dq(const void* q, const void* k, const void* v, const void* dout,
                const void* workspace, size_t workspace_bytes, void* dq, int B, int T, int Hq,
                int Hkv, int D, float scale, int causal, void* stream);

/* Synchronises `stream`, then reads and clears the device-side status word
 * that kernels set when a pipeline wait runs out (a bounded wait, default
 * limit 1 s).  Returns DETATTN_OK, DETATTN_ERR_DEVICE_TIMEOUT,
 * DETATTN_ERR_WORKSPACE (a dQ step found the workspace's tile counter not
 * cleared, i.e. attn_bwd_delta had not run on that workspace: that dQ
 * step's dq is not valid) or DETATTN_ERR_CUDA. */
int detattn_check_status(void* stream);

/* Diagnostic for accuracy tests: evaluates on n device floats x the three
 * ways the kernels form 2^x -- the FMA-pipe polynomial (Cody-Waite range
 * reduction plus a fitted cubic, max relative error 7.5e-5, inputs clamped at
 * -126), the same polynomial in its paired f32x2 form, and the special-function
 * unit's ex2.approx -- into y_poly, y_pair and y_sfu.  Not tied to a passage
 * of the method. */
int detattn_diag_exp2(const float* x, float* y_poly, float* y_pair, float* y_sfu, int n,
                      void* stream);

/* Diagnostic for host-side tests (no GPU needed): the static deal of
 * 128-query tiles to persistent pipelines that the forward uses, and the dQ
 * step without its tile counter, for a shape and an SM count.  Units are
 * numbered heaviest first: unit u is query tile ceil(T/128) - 1 - u / (B*Hq)
 * of (b, h) with b*Hq + h = u % (B*Hq).  Writes pipe_of_unit[u] for all
 * n_units = B * Hq * ceil(T / 128) units (n_units must equal that) and returns
 * the number of pipelines, 0 for an empty shape, or a negative status.  Not
 * tied to a passage of the method. */
int detattn_diag_qtile_deal(int D, int B, int T, int Hq, int causal, int sms, int* pipe_of_unit,
                            int n_units);

/* Diagnostic for host-side tests (no GPU needed): the dK/dV step's choice of
 * C, the blocks that share one 128-key tile, and NG, the resident clusters of
 * C blocks that walk the key tiles, for a shape and a device described by
 * resident[0..3]: how many clusters of 1, 2, 4 and 8 blocks it holds at once
 * (0 where that size cannot be resident; sizes above the kernel's limit for
 * D are not considered).  blocks_per_key_tile: 0 for the automatic choice,
 * else the C to take (as detattn_set_dkdv_split).  Writes *c_out and *ng_out
 * (both 0 for an empty shape).  Returns DETATTN_OK, DETATTN_ERR_SHAPE /
 * DETATTN_ERR_HEADDIM for a bad shape, split or a device with no usable size,
 * DETATTN_ERR_NULL for a NULL pointer.  The attention calls make the same
 * choice from the current device's occupancy.  Not tied to a passage of the
 * method. */
int detattn_diag_dkdv_split(int B, int T, int Hq, int Hkv, int D, int causal,
                            const int* resident, int blocks_per_key_tile, int* c_out,
                            int* ng_out);

/* Failure-detection self-test.  Launches a one-thread kernel on `stream`
 * that waits, with the same bounded wait the attention kernels use, on a
 * barrier nothing ever completes; after `limit_ns` (clamped to [1 ms, 10 s])
 * it gives up, records a timeout in the device status word and returns, so
 * the context stays usable.  A following detattn_check_status() returns
 * DETATTN_ERR_DEVICE_TIMEOUT (and clears the word).  Not tied to a passage of
 * the method: it exists to test the timeout path without faulting a GPU. */
int detattn_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/* Tuning knob: number of thread blocks that share one 128-key tile in the
 * dK/dV step (1, 2, 4 or 8; 0 = automatic, the default; at D = 128 values
 * above 2 act as 2).  The blocks of such a cluster split the tile's (query
 * head, query tile) items into contiguous chunks and add their partial sums
 * in a fixed order, so results stay bitwise reproducible for a given
 * setting; different settings round differently.  Automatic picks from the
 * shape and the device's resident-cluster count only.  Host-side, per
 * process.
 * Returns DETATTN_OK or DETATTN_ERR_SHAPE for another value. */
int detattn_set_dkdv_split(int blocks_per_key_tile);

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

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
  DETATTN_ERR_WORKSPACE = -9,      /* workspace NULL or too small; from detattn_check_status:
                                      a dQ step ran on a workspace attn_bwd_delta had not
                                      prepared */
  DETATTN_ERR_INDEX = -10          /* from detattn_check_status: embed_grad met token ids
                                      outside [0, V) (it left those tokens out) */
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
 * dv (bf16).  Runs attn_bwd_delta, attn_bwd_dkdv and attn_bwd_dq on `stream`,
 * the last two as programmatic dependents of the step before: the dQ step
 * starts once every dK/dV block has seen the Delta step complete and runs on
 * the SMs the dK/dV step frees, and it completes only after the dK/dV step
 * has, so all work is ordered after earlier work on `stream` and later work
 * on `stream` sees the results.
 * `workspace` (attn_bwd_workspace_bytes, at least the row statistics' share;
 * 16-byte aligned, caller-owned, contents on entry irrelevant) holds the row
 * statistics and the dQ step's tile counter (layout above).  Passage: "Step 2: fused flash attention" and "Where the time
 * goes now" (the flash_attention_dkv kernel) on the RustingBrain page. */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, void* workspace,
             size_t workspace_bytes, int B, int T, int Hq, int Hkv, int D, float scale,
             int causal, void* stream);

/* Workspace bytes for the stored-dS form of attn_bwd: the bytes of
 * attn_bwd_workspace_bytes, then (from byte R + 256) every dS tile the dK/dV
 * step forms, bf16: per (b, h) the pairs (128-query tile mt, 128-key tile
 * kt) visible under the mask (kt <= mt when causal, in the order
 * mt (mt + 1) / 2 + kt; all pairs mt * n + kt otherwise), each pair two
 * halves of 64 queries stored [128 keys][64 queries] (32 KiB a pair).  With
 * detattn_set_bwd_dq_mode(1), an attn_bwd call whose workspace_bytes reaches
 * this size stores dS in the dK/dV step and forms dQ = scale * dS K with one
 * tensor-core product per tile instead of recomputing S, P and dP
 * (RustingBrain page, "Where the time goes now": the backward's time is in
 * the kernels that recompute the probabilities); both forms are
 * deterministic, and dk, dv are the same bits in both.  Measured on GB300 the
 * recompute form is the faster at every benchmarked shape (it runs dQ beside
 * dK/dV; the stored form must run after it), so it is the default.  Returns
 * 0 for an invalid shape or one whose dS rows would exceed 2^31. */
size_t attn_bwd_ds_workspace_bytes(int B, int T, int Hq, int Hkv, int D, int causal);

/* 0 (default): attn_bwd recomputes S and dP in its dQ step; 1: it takes the
 * stored-dS form whenever its workspace is long enough for it
 * (attn_bwd_ds_workspace_bytes).  Host-side, per process.  Returns
 * DETATTN_OK or DETATTN_ERR_SHAPE.  Not tied to a passage of the method. */
int detattn_set_bwd_dq_mode(int mode);

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

/* ------------------------------------------------------------------------
 * Packed variable-length batches (several sequences of their own lengths in
 * one call, and cross-attention with Tq != Tk).  No page describes them; they
 * are the same computation per sequence (the operation above, with the
 * RustingBrain page's fused kernels) over packed rows:
 *
 *   q, o, dout, dq : bf16 [total_q, Hq, D]    k, v, dk, dv : bf16 [total_k, Hkv, D]
 *   lse            : fp32 [Hq, total_q]
 *   cu_q, cu_k     : HOST int32 arrays of n_seq + 1 nondecreasing offsets,
 *                    cu[0] = 0, total = cu[n_seq]; sequence s owns query rows
 *                    cu_q[s] .. cu_q[s+1]-1 and key rows cu_k[s] .. cu_k[s+1]-1
 *
 * With tq = cu_q[s+1] - cu_q[s] and tk likewise, query i of s sees key j of
 * s iff j <= i + tk - tq when causal (the mask ends in the bottom-right
 * corner, which is j <= i when tq == tk), every key of s otherwise.  A query
 * row that sees no key (causal, tq > tk) gets o = 0, lse = -inf and dq = 0;
 * a key no query sees gets dk = dv = 0.  Empty sequences are allowed.
 * Limits: n_seq <= 256; each sequence <= 2^22 rows; at most 2048 tiles of
 * 128 query rows and 2048 of 128 key rows over the batch (DETATTN_ERR_SHAPE
 * beyond).  Results are deterministic like the fixed-length calls.  The
 * tile tables are built on the host from cu_q, cu_k at every call and passed
 * as kernel parameters, so nothing is allocated. */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_q, const int* cu_k, int n_seq, int Hq, int Hkv, int D,
                    float scale, int causal, void* stream);

/* Workspace bytes of attn_bwd_varlen: R + 256, with R = Hq * Tp * 8 rounded
 * up to 256 and Tp = the sum over sequences of tq rounded up to 128 (row
 * statistics per query head, each sequence's starting at a multiple of 128,
 * then the dQ step's two counter words).  0 for an invalid or query-less
 * batch. */
size_t attn_bwd_varlen_workspace_bytes(const int* cu_q, const int* cu_k, int n_seq, int Hq,
                                       int Hkv, int D);

/* Packed variable-length backward: writes dq, dk, dv.  Runs the Delta,
 * dK/dV and dQ steps on `stream` in that order. */
int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, void* workspace,
                    size_t workspace_bytes, const int* cu_q, const int* cu_k, int n_seq, int Hq,
                    int Hkv, int D, float scale, int causal, void* stream);

/* ------------------------------------------------------------------------
 * Deterministic embedding-lookup gradient (oxide-train README, "The trainer
 * is not bit-identical to itself after step 1": its embedding gradient is
 * summed with atomics, so two runs of one binary disagree from step 2 on;
 * "Full-step profiling": B = 32, T = 1024, vocabulary 50,257 padded to
 * 50,432, width 1536).  For the lookup X[t,:] = W[ids[t],:]:
 *
 *   dw[v,:] = sum over t with ids[t] == v of dy[t,:]
 *
 * Every element is one fp32 sum whose order depends on the ids only: the
 * tokens of an id are taken in ascending position, in runs of 32 entries of
 * the id-sorted token list; an id whose tokens span several runs has one
 * partial sum per run, added in run order.  Integer atomics only count
 * tokens and hand out slots, which changes no bit of dw, so repeated calls
 * give identical bytes.
 *
 * Layout: ids int32 [N]; dy bf16 [N, E] (row-major); dw fp32 [V, E]
 * (row-major, fully overwritten: rows no token selects are zero).  E must be
 * a multiple of 4 (up to 2^20), N in [0, 2^30], V in [1, 2^30].  Pointers are
 * device pointers, 16-byte aligned; ids and dy may be NULL when N == 0.
 * Tokens whose id lies outside [0, V) are left out of dw and reported by
 * detattn_check_status (DETATTN_ERR_INDEX); they are never used as an index.
 * The call queues one memset and up to six kernels on `stream`.
 */

/* Bytes of workspace embed_grad needs: int32 counts [V], offsets [V + 1],
 * cursor [V], two token lists [N], and two fp32 [ceil(N / 32), E] blocks of
 * partial rows, each part 256-byte aligned.  0 for an invalid shape. */
size_t embed_grad_workspace_bytes(int N, int V, int E);

/* Writes dw from ids and dy (see above).  `workspace` is caller-owned device
 * memory of embed_grad_workspace_bytes(N, V, E) bytes, contents on entry
 * irrelevant.  Returns DETATTN_OK or DETATTN_ERR_SHAPE / _NULL / _ALIGN /
 * _WORKSPACE / _ARCH / _CUDA (nothing launched on an error). */
int embed_grad(const int* ids, const void* dy, float* dw, void* workspace, size_t workspace_bytes,
               int N, int V, int E, void* stream);

/* ------------------------------------------------------------------------
 * One attention layer of a training step, and its AdamW update (RustingBrain
 * vs PyTorch/TensorFlow page, "The setup": d_model 768, 12 query heads over 4
 * KV heads of head_dim 64, rotary positions; "Where the time goes now":
 * GEMMs are most of the step; oxide-train README: the step ends in AdamW
 * with LR 3e-4 and weight decay 0.1, and "The trainer is not bit-identical
 * to itself after step 1").  Every kernel writes each output element once in
 * a fixed order, with no atomics on data, so repeated steps give identical
 * gradients and weights.
 */

/* C[M, N] = alpha * A[M, K] B[K, N] on the tensor cores: bf16 A and B, fp32
 * accumulation, C bf16 (c_fp32 = 0) or fp32 (c_fp32 = 1), row-major with row
 * stride ldc elements.  a_mn_major = 0: A is stored [M rows, K] (row stride
 * lda); 1: A is stored transposed, [K rows, M] (row stride lda).  Likewise
 * b_mn_major = 1: B stored [K rows, N]; 0: stored transposed, [N rows, K].
 * M must be a multiple of 128, N of 128 and K of 64; row strides hold whole
 * rows and make 16-byte rows.  Every element of C is one block's sum over K
 * in ascending order.  Device pointers, 16-byte aligned. */
int layer_gemm(const void* a, int a_mn_major, int lda, const void* b, int b_mn_major, int ldb,
               void* c, int c_fp32, int ldc, int M, int N, int K, float alpha, void* stream);

/* Workspace bytes of layer_train_step (its intermediates: the joined QKV
 * projection, the rotated Q, K and V, O, LSE, dO, dQ, dK, dV, the joined
 * gradient of the projection, the attention backward's workspace, and the
 * fp32 partial sums of the two split-K weight-gradient products).  0 for an
 * invalid shape. */
size_t layer_workspace_bytes(int B, int T, int d, int Hq, int Hkv, int D);

/* One training step of one attention layer at the current weights, then one
 * AdamW update of them:
 *
 *   QKV = X Wqkv  (Wqkv = [Wq | Wk | Wv], [d, (Hq + 2 Hkv) D])
 *   Q, K = rope(Q, K), V      (rotate-half: component i of a head's first
 *                              half turns with component i of its second half
 *                              by t * 10000^(-2i/D), t = position in the
 *                              sequence; the pages name rotary positions
 *                              without a convention)
 *   O = causal GQA attention (attn_fwd), Y = O Wo
 *   dO = dY Wo^T, (dQ, dK, dV) = attn_bwd, dQ, dK = rope^T(dQ, dK)
 *   g_o = O^T dY, g_qkv = X^T [dQ | dK | dV], dX = [dQ | dK | dV] Wqkv^T
 *   AdamW (decoupled decay):  w *= 1 - lr wd; m = b1 m + (1 - b1) g;
 *     v = b2 v + (1 - b2) g^2; w -= lr (m / (1 - b1^step)) / (sqrt(v / (1 - b2^step)) + eps)
 *
 * x, dy, y, dx: bf16 [B, T, d]; w_qkv, m_qkv, v_qkv, g_qkv: fp32 [d, (Hq +
 * 2 Hkv) D]; w_o, m_o, v_o, g_o: fp32 [Hq D, d]; w_qkv_bf16, w_o_bf16: the
 * bf16 copies the GEMMs read (the caller sets them from the fp32 weights
 * before the first step; each step rewrites them after the update).  g_qkv
 * and g_o receive this step's gradients (at the weights before the update);
 * dx may be NULL.  The scale is 1/sqrt(D) and the attention is causal.
 * B*T, d, Hq*D and (Hq + 2 Hkv)*D must be multiples of 128, D 64 or 128.
 * step counts from 1.  Stream-ordered on `stream`: the call forks a
 * library-owned second stream from it (dO = dY Wo^T during the forward; g_o
 * and the Wo update during the attention backward) and joins it back before
 * returning, so work queued on `stream` afterwards sees every result, and a
 * stream capture of the call closes over both streams.  Calls from several
 * host threads are serialised while they enqueue. */
int layer_train_step(const void* x, const void* dy, float* w_qkv, float* w_o, float* m_qkv,
                     float* v_qkv, float* m_o, float* v_o, void* w_qkv_bf16, void* w_o_bf16,
                     float* g_qkv, float* g_o, void* y, void* dx, void* workspace,
                     size_t workspace_bytes, int B, int T, int d, int Hq, int Hkv, int D, int step,
                     float lr, float weight_decay, float beta1, float beta2, float eps,
                     void* stream);

/* Synchronises `stream`, then reads and clears the device-side status word
 * that kernels set when a pipeline wait runs out (a bounded wait, default
 * limit 1 s).  Returns DETATTN_OK, DETATTN_ERR_DEVICE_TIMEOUT,
 * DETATTN_ERR_WORKSPACE (a dQ step found the workspace's tile counter not
 * cleared, i.e. attn_bwd_delta had not run on that workspace: that dQ
 * step's dq is not valid), DETATTN_ERR_INDEX (embed_grad met ids outside
 * [0, V)) or DETATTN_ERR_CUDA. */
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

/* Diagnostic for host-side tests (no GPU needed): the listed deal of the
 * dK/dV step's 128-key tiles at D = 64 (fixed length) over ng clusters of c
 * blocks (c >= 2).  Tiles are numbered in walk order, t = nt * B*Hkv + b*Hkv
 * + g (nt the tile's position along T).  A tile is either shared by all c
 * blocks of one cluster (each takes a contiguous chunk of its items and the
 * partial sums are added in rank order) or taken whole by one block.  Block
 * i's tiles are entry[start[i] .. start[i + 1] - 1], each t * 2 + 1 when
 * shared and t * 2 when whole; shared ones come first.  force = 0 builds the
 * list only where its load model beats the plain walk, as attn_bwd does;
 * force = 1 whenever it fits.  start must hold ng * c + 1 ints and entry
 * max_entries.  Returns the number of entries, 0 when no list is used
 * (the plain walk), or a negative status (DETATTN_ERR_SHAPE for a bad
 * shape or c, ng; DETATTN_ERR_NULL for a NULL pointer).  Not tied to a
 * passage of the method. */
int detattn_diag_dkdv_list(int B, int T, int Hq, int Hkv, int causal, int c, int ng, int force,
                           int* start, int* entry, int max_entries);

/* Tuning knob: how the dK/dV step at D = 64 deals its key tiles when C > 1
 * blocks share one (fixed-length inputs with either backward form, and
 * packed batches, whose list is built the same way over their key tiles).
 * 0 (default): the listed deal of detattn_diag_dkdv_list where its load
 * model beats the plain walk; 1: always the plain walk (every tile shared,
 * tiles dealt to the clusters in alternating order); 2: the listed deal
 * whenever it fits.  Results are bitwise reproducible for a given setting;
 * different settings round dK, dV differently.  Host-side, per process.
 * Returns DETATTN_OK or DETATTN_ERR_SHAPE for another value. */
int detattn_set_dkdv_deal(int mode);

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

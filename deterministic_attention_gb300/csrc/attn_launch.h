// Internal interface between the C-ABI host layer and the kernel translation
// units: argument blocks and launch functions.  Not part of the public API.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace detattn {

constexpr int kTileM = 128;     // query rows per forward / dQ tile
constexpr int kTileN = 128;     // key rows per dK/dV tile
constexpr int kFwdTileN = 128;  // key rows per forward KV tile
constexpr int kDqTileN = 128;   // key rows per dQ-kernel KV tile
// Query rows per dK/dV-kernel item: 128 at D = 64 (S^T, dP^T, P^T, dS^T and
// both accumulators fill TMEM), 64 at D = 128 (the accumulators take twice
// the columns).
constexpr int dkdv_tile_m(int D) { return D == 64 ? 128 : 64; }
// Query rows the dK/dV kernel that runs with C blocks per key tile loads per
// item (the rows of its Q, dO tensor-map boxes): 128, except at D = 128 with
// a tile split over a cluster, which runs the 64-query kernel.
constexpr int dkdv_item_rows(int D, int C) { return D == 64 || C == 1 ? 128 : 64; }

// Static deal of query-tile work units (forward and dQ) to persistent
// pipelines.  Unit u (in heaviest-first order) is query tile n_m - 1 - u / BHq
// of (b, h) = u % BHq.
// Pipeline i takes units unit[start[i]] .. unit[start[i + 1] - 1]; with
// n_listed == 0 it takes one unit per round of n_pipes units instead, rounds
// dealt to the pipelines forward and backward in turn (qtile_snake_*).
constexpr int kQTileMaxPipes = 320;
constexpr int kQTileMaxListed = 1024;
struct QTileSched {
  int n_pipes;
  int n_listed;
  uint16_t start[kQTileMaxPipes + 1];
  uint16_t unit[kQTileMaxListed];
};
// The unlisted deal: pipeline i's k-th unit, and how many it takes of `total`.
// Alternating the direction of the rounds pairs heavy units with light ones.
__host__ __device__ inline int qtile_snake_unit(int i, int k, int n_pipes) {
  return k * n_pipes + ((k & 1) ? n_pipes - 1 - i : i);
}
__host__ __device__ inline int qtile_snake_count(int i, int total, int n_pipes) {
  const int full = total / n_pipes, rem = total % n_pipes;
  return full + (((full & 1) ? n_pipes - 1 - i : i) < rem ? 1 : 0);
}
// Pipelines per dQ block (one: S, dP, dS and dQ take most of TMEM).
constexpr int dq_pipes_per_block(int) { return 1; }
// Pipelines per forward block: two at D = 64 (256 TMEM columns each), one
// at D = 128.
constexpr int fwd_pipes_per_block(int D) { return D == 64 ? 2 : 1; }

// Packed variable-length batches: sequence s holds query rows cu_q[s] ..
// cu_q[s + 1] - 1 of the packed [total_q, Hq, D] tensors and key rows
// cu_k[s] .. cu_k[s + 1] - 1 of the [total_k, Hkv, D] ones.  Under the
// causal mask query i of s sees key j of s iff j <= i + tk - tq (the mask
// ends in the bottom-right corner of the tq x tk score matrix).  The table
// travels as a __grid_constant__ kernel parameter; `tile` lists the work
// tiles heaviest first as (s << 16) | tile index within s: 128-query tiles
// for the forward and dQ steps, 128-key tiles for the dK/dV step.  The
// backward's row statistics of sequence s start at position ps[s] (a
// multiple of 128) of each query head's row, so every tile of them is
// aligned and positions past tq hold (-inf, -0).
constexpr int kVarlenMaxSeqs = 256;
constexpr int kVarlenMaxTiles = 2048;
struct VarlenTable {
  int n_seq;
  int n_tiles;
  int cu_q[kVarlenMaxSeqs + 1];
  int cu_k[kVarlenMaxSeqs + 1];
  int ps[kVarlenMaxSeqs + 1];
  uint32_t tile[kVarlenMaxTiles];
};
// The fixed-length kernels take this empty parameter in its place.
struct NoVarlen {};
// Table accessors that also compile (and are never called) for NoVarlen.
__host__ __device__ inline int vt_tiles(const VarlenTable& v) { return v.n_tiles; }
__host__ __device__ inline int vt_tiles(const NoVarlen&) { return 0; }
__host__ __device__ inline uint32_t vt_tile(const VarlenTable& v, int i) { return v.tile[i]; }
__host__ __device__ inline uint32_t vt_tile(const NoVarlen&, int) { return 0u; }
__host__ __device__ inline int vt_cu_q(const VarlenTable& v, int s) { return v.cu_q[s]; }
__host__ __device__ inline int vt_cu_q(const NoVarlen&, int) { return 0; }
__host__ __device__ inline int vt_cu_k(const VarlenTable& v, int s) { return v.cu_k[s]; }
__host__ __device__ inline int vt_cu_k(const NoVarlen&, int) { return 0; }
__host__ __device__ inline int vt_ps(const VarlenTable& v, int s) { return v.ps[s]; }
__host__ __device__ inline int vt_ps(const NoVarlen&, int) { return 0; }

struct FwdArgs {
  void* o;               // bf16 [B, T, Hq, D]
  float* lse;            // fp32 [B, Hq, T]
  int T, Hq, Hkv;
  int n_m;               // query tiles per (b, h)
  int BHq;               // B * Hq
  int causal;
  float scale_log2;      // scale * log2(e)
  unsigned long long wait_ns;
};

// Row statistics of the backward, in the caller's workspace: for every (b, h)
// and every position t < Tp = T rounded up to 128, the pair
// (-LSE * log2(e), -Delta); positions t >= T hold (-inf, -0) so padded query
// rows contribute exactly nothing.  Both are stored negated because the
// kernels add them: x = S * scale * log2(e) + (-LSE * log2 e), dP + (-Delta).
inline int padded_T(int T) { return (T + 127) / 128 * 128; }

struct DeltaArgs {
  const void* o;         // bf16 [B, T, Hq, D]
  const void* dout;      // bf16 [B, T, Hq, D]
  const float* lse;      // fp32 [B, Hq, T]
  float2* rowstats;      // [B * Hq, Tp] pairs
  int B, T, Tp, Hq, D;
  unsigned* unit_counter;  // the dQ step's unit counter, cleared here (may be null)
};

struct BwdArgs {
  const float2* rowstats;  // [B * Hq, Tp] pairs written by the Delta step
  void* dq;              // bf16 [B, T, Hq, D]   (dQ kernel)
  void* dk;              // bf16 [B, Tk, Hkv, D]  (dK/dV kernel)
  void* dv;
  int T, Tp, Hq, Hkv;
  int Tk;                // key rows per batch: T, or total_k when packed
  int n_tiles;           // tiles per (b, head) along T
  int BH;                // B * Hq (dQ) or B * Hkv (dK/dV)
  int cluster;           // dK/dV: blocks sharing one key tile (1, 2, 4 or 8)
  int n_groups;          // dK/dV: resident clusters (persistent), each walking its key tiles
  // dK/dV tile order: 0 walks every (b, KV head)'s tile nt before any tile
  // nt + 1 (heaviest first); g > 0 does so within chunks of g (b, KV head)
  // pairs, one chunk after the other, so the queries the clusters read at
  // once (those of g KV groups) stay in L2 on long sequences.
  int bg_chunk;
  int causal;
  float scale;
  float scale_log2;
  unsigned long long wait_ns;
  // dQ: units are taken from this counter (zero at launch) instead of the
  // static deal, when not null.
  unsigned* unit_counter;
  // Stored-dS backward (fixed-length only): when not null the dK/dV step
  // also writes every item's dS^T (bf16) here, pairs (128-query tile mt,
  // 128-key tile kt) of each (b, h) in the order kt <= mt, mt(mt+1)/2 + kt
  // (causal) or mt * n_tiles + kt (full); per pair two halves of 64 queries,
  // each [128 keys][64 queries].  attn_dq_from_ds reads them back.
  void* ds;
  long ds_pairs;         // pairs per (b, h)
};

// dQ from the stored dS: for each 128-query tile, dQ = scale * sum over its
// key tiles (ascending) of dS K, on the tensor cores.  `mds` is a 2-D map
// over the dS rows ({64, rows}, box {64, 64}); `mk` maps K with 64-row
// boxes.  Units (b, h, query tile) heaviest first, one block each.
cudaError_t launch_dq_from_ds(int D, const CUtensorMap& mds, const CUtensorMap& mk,
                              const BwdArgs& a, int n_units, cudaStream_t st);
cudaError_t take_ds_status(cudaStream_t st, unsigned* out);

// Listed deal of the dK/dV key tiles (the 128-query kernel at D = 64):
// block i walks entries start[i] .. start[i + 1] - 1, each (tile << 1) |
// shared.  A shared tile is taken by every block of the cluster (its items
// split by rank, the partial sums exchanged); any other goes whole to one
// block, which stores all its rows.  Every block lists its shared tiles
// first, and the blocks of a cluster list the same ones in the same order.
// n_blocks == 0: the snake walk of the tiles over the clusters instead.
constexpr int kDkvListMaxBlocks = 256;
constexpr int kDkvListMaxEntries = 1024;
struct DkvList {
  int n_blocks;
  uint16_t start[kDkvListMaxBlocks + 1];
  uint16_t entry[kDkvListMaxEntries];
};

// Key tile t of the dK/dV walk as (nt, bg): position nt along T, bg = b Hkv + g.
__host__ __device__ inline void dkdv_tile_coords(int t, int n_tiles, int BH, int bg_chunk, int* nt,
                                                 int* bg) {
  if (bg_chunk <= 0 || bg_chunk >= BH) {
    *nt = t / BH;
    *bg = t % BH;
    return;
  }
  const int per = n_tiles * bg_chunk;
  const int chunk = t / per, r = t % per;
  *nt = r / bg_chunk;
  *bg = chunk * bg_chunk + r % bg_chunk;
}

// Each returns the launch error (cudaSuccess when the kernel was queued).
// `vt` (not null) selects the packed variable-length form: the tensor maps
// then cover the packed rows with B = 1, FwdArgs::T / BwdArgs::T is the
// number of packed query rows, and units / tiles come from the table.
// The forward's `mo` map covers O ([B, T, Hq, D], or the packed rows) with
// boxes of 32 rows x 64 columns: each softmax warp stores its rows of a tile.
constexpr int kFwdStoreRows = 32;
cudaError_t launch_fwd(int D, int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mo, const FwdArgs& a,
                       const QTileSched& sched, const VarlenTable* vt, cudaStream_t st);
// `sms`: the current device's SM count (the grid is persistent).
cudaError_t launch_delta(const DeltaArgs& a, int sms, const VarlenTable* vt, cudaStream_t st);
// Clusters of c blocks of the dK/dV kernel that can be resident at once on the
// current device (c = 1: blocks), and the largest c the kernel supports.
cudaError_t dkdv_max_clusters(int D, int c, int* out);
int dkdv_max_cluster_size(int D);
// `dependent`: launched as a programmatic dependent of the Delta step just
// before it in `st` (the kernel waits for it only before reading the row
// statistics; Q, K, V, dO must not be written by that step).  `list` (not
// null, n_blocks == grid) deals the tiles by that list: D = 64, without the
// chunked walk (tile t of a packed batch: table entry t / Hkv, KV head t % Hkv).
cudaError_t launch_dkdv(int D, int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                        const CUtensorMap& mv, const CUtensorMap& mdo, const BwdArgs& a,
                        bool dependent, const VarlenTable* vt, const DkvList* list,
                        cudaStream_t st);
// `mdq` covers dQ with boxes of 32 rows x D/2 columns, unswizzled: each
// element-wise warp of the dQ step stores its rows of a tile (D = 64).
// `after_dkdv`: launched as a programmatic dependent of the dK/dV step just
// before it in `st`, which lets it start once every dK/dV block has seen the
// Delta step complete; it then runs beside that step, and completes only
// after it.
constexpr int kDqStoreRows = 32;
cudaError_t launch_dq(int D, int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                      const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap& mdq,
                      const BwdArgs& a, const QTileSched& sched, const VarlenTable* vt,
                      bool after_dkdv, cudaStream_t st);

// Launches a one-thread kernel whose bounded wait on a never-completed
// mbarrier runs out after limit_ns (sets the timeout bit, then returns).
cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t st);

cudaError_t launch_exp2_diag(const float* x, float* y_poly, float* y_pair, float* y_sfu, int n,
                             cudaStream_t st);

// Unique id (cuCtxGetId) of the CUDA context current on the calling thread,
// or 0 when none is current or the driver cannot say.  Per-device caches of
// context-bound state (function attributes, streams, symbol addresses) are
// keyed on it, so that they are rebuilt after the context is destroyed and
// re-created (cudaDeviceReset, or a primary-context reset by another module).
unsigned long long current_context_id();

// Read-and-clear of the device status words the kernels set when a bounded
// wait runs out (synchronous on `st`).  Returns the OR of the words.
cudaError_t take_fwd_status(cudaStream_t st, unsigned* out);
cudaError_t take_bwd_status(cudaStream_t st, unsigned* out);

}  // namespace detattn

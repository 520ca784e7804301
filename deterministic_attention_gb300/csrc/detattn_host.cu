// C-ABI host layer of libdetattn: argument validation, TMA descriptor
// encoding and kernel launches.  Declarations and contracts: include/detattn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <functional>
#include <memory>
#include <mutex>
#include <queue>
#include <vector>

#include "../../include/detattn.h"
#include "attn_launch.h"
#include "embed_launch.h"
#include "layer_launch.h"

using namespace detattn;

namespace {

constexpr int kVersion = 10000;  // 1.0.0
thread_local char g_err[512] = "";
unsigned long long g_wait_ns = 1000000000ull;  // 1 s per bounded wait
int g_dkdv_split = 0;                           // 0: automatic
int g_dkdv_deal = 0;  // 0: listed deal when its model beats the snake walk; 1: never; 2: always

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}
int ok_status() {
  g_err[0] = '\0';
  return DETATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by all entry points.  Sets *empty for B*T == 0.
int check_shape(int B, int T, int Hq, int Hkv, int D, bool* empty) {
  if (B < 0 || T < 0) return fail(DETATTN_ERR_SHAPE, "B=%d T=%d must be >= 0", B, T);
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return fail(DETATTN_ERR_SHAPE, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  if (D != 64 && D != 128) return fail(DETATTN_ERR_HEADDIM, "D=%d: only 64 and 128", D);
  // Grid and index limits: tiles per launch and elements per tensor.
  const double tiles = static_cast<double>(B) * Hq * ((T + 63) / 64);
  const double elems = static_cast<double>(B) * T * Hq * D;
  if (tiles > 2.0e9 || elems > 1.0e12 || T > (1 << 30))
    return fail(DETATTN_ERR_SHAPE, "problem too large (B=%d T=%d Hq=%d)", B, T, Hq);
  *empty = (B == 0 || T == 0);
  return DETATTN_OK;
}

// Blocks per dK/dV key tile: 0 (automatic) or a power of two up to 8.
int check_split(int c) {
  if (c != 0 && c != 1 && c != 2 && c != 4 && c != 8)
    return fail(DETATTN_ERR_SHAPE, "dK/dV split %d: must be 0 (automatic), 1, 2, 4 or 8", c);
  return DETATTN_OK;
}

int check_scale(float scale, int causal) {
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(DETATTN_ERR_SCALE, "scale=%g must be finite and > 0", static_cast<double>(scale));
  if (causal != 0 && causal != 1) return fail(DETATTN_ERR_SCALE, "causal=%d must be 0 or 1", causal);
  return DETATTN_OK;
}

int check_ptrs(std::initializer_list<std::pair<const void*, const char*>> ps) {
  for (const auto& p : ps)
    if (p.first == nullptr) return fail(DETATTN_ERR_NULL, "%s is NULL", p.second);
  for (const auto& p : ps)
    if (!aligned16(p.first)) return fail(DETATTN_ERR_ALIGN, "%s is not 16-byte aligned", p.second);
  return DETATTN_OK;
}

// ------------------------------------------------------------ device checks
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

int check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DETATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  static int arch_ok[64] = {};  // 0 unknown, 1 ok, 2 wrong arch
  if (dev >= 64 || arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess)
      return fail(DETATTN_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    const int v = (major == 10 && minor == 3) ? 1 : 2;
    if (dev < 64) arch_ok[dev] = v;
    if (v == 2)
      return fail(DETATTN_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                  major, minor);
  } else if (arch_ok[dev] == 2) {
    return fail(DETATTN_ERR_ARCH, "device %d is not sm_103", dev);
  }
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    g_encode_err = cudaGetDriverEntryPointByVersion(
        "cuTensorMapEncodeTiled", reinterpret_cast<void**>(&g_encode), 12000, cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
      g_encode_err = cudaErrorNotSupported;
  });
  if (g_encode_err != cudaSuccess || g_encode == nullptr)
    return fail(DETATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable: %s",
                cudaGetErrorString(g_encode_err));
  return DETATTN_OK;
}

// Tensor map over a bf16 [B, T, H, D] tensor whose box is `rows` consecutive
// positions t of one (b, h) and 64 columns of d (one 128-byte swizzle atom).
// Rows past T read as zero.
int encode_rows(CUtensorMap* m, const void* ptr, int B, int T, int H, int D, int rows,
                const char* what) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                           static_cast<cuuint64_t>(T) * H * D * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DETATTN_ERR_CUDA, "tensor map for %s: CUresult %d", what, (int)r);
  return DETATTN_OK;
}

// Tensor map over a [B, T, H, D] bf16 tensor for unswizzled stores of boxes
// `inner` columns x `rows` rows (inner * 2 a multiple of 16 bytes).
int encode_rows_store(CUtensorMap* m, const void* ptr, int B, int T, int H, int D, int inner,
                      int rows, const char* what) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                           static_cast<cuuint64_t>(T) * H * D * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(inner), 1, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DETATTN_ERR_CUDA, "tensor map for %s: CUresult %d", what, (int)r);
  return DETATTN_OK;
}

// Tensor map over the stored dS tiles: bf16 rows of 64 (one 128-byte
// swizzle atom), boxes of 64 rows.
int encode_2d_rows64(CUtensorMap* m, const void* ptr, long rows) {
  cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DETATTN_ERR_CUDA, "tensor map for dS: CUresult %d", (int)r);
  return DETATTN_OK;
}

int launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(DETATTN_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
  return ok_status();
}

float log2e_times(float scale) { return scale * 1.4426950408889634f; }

int sm_count(int* out);

// Deal of the forward's work units to persistent pipelines (see QTileSched).
// Heaviest first, each unit goes to the block with the least work so far and
// within it to the pipeline with the least: the pipelines of one block share
// an SM, so it is the block totals that must balance.  A unit's work counts
// its key tiles plus two for its Q load and epilogue.  Beyond the size of the
// listed form, units are dealt round-robin (many units balance by number).
// Built on the host from the shape and the SM count only; cached.
//
// Units are numbered heaviest first in groups of `per_group` equal units
// (the heads, or batches and heads, of one query tile): unit u weighs
// group_w[u / per_group].
void qtile_schedule_w(int NP, const std::vector<double>& group_w, int per_group, int sms,
                      QTileSched* out, int* grid) {
  const long units = static_cast<long>(group_w.size()) * per_group;
  // One block per SM while there are units for it: a second pipeline on an
  // SM adds far less than a second SM does.
  long blocks = units < sms ? units : sms;
  if (blocks < 1) blocks = 1;
  const int pipes = static_cast<int>(blocks) * NP;
  out->n_pipes = pipes;
  *grid = static_cast<int>(blocks);
  if (units > kQTileMaxListed || pipes > kQTileMaxPipes) {
    out->n_listed = 0;
    return;
  }
  std::vector<double> block_load(blocks, 0.0), pipe_load(pipes, 0.0);
  std::vector<std::vector<uint16_t>> lists(pipes);
  for (long u = 0; u < units; ++u) {
    const double w = group_w[u / per_group];
    long bi = 0;
    for (long i = 1; i < blocks; ++i)
      if (block_load[i] < block_load[bi]) bi = i;
    int pi = static_cast<int>(bi) * NP;
    for (int k = 1; k < NP; ++k)
      if (pipe_load[bi * NP + k] < pipe_load[pi]) pi = static_cast<int>(bi) * NP + k;
    block_load[bi] += w;
    pipe_load[pi] += w;
    lists[pi].push_back(static_cast<uint16_t>(u));
  }
  int n = 0;
  for (int i = 0; i < pipes; ++i) {
    out->start[i] = static_cast<uint16_t>(n);
    for (uint16_t u : lists[i]) out->unit[n++] = u;
  }
  out->start[pipes] = static_cast<uint16_t>(n);
  out->n_listed = n;
}

void qtile_schedule(int NP, int B, int T, int Hq, int causal, int sms, QTileSched* out, int* grid) {
  const int n_m = (T + kTileM - 1) / kTileM;
  const int kv_tiles = (T + kDqTileN - 1) / kDqTileN;
  std::vector<double> w(n_m);
  for (int g = 0; g < n_m; ++g) {
    const int mt = n_m - 1 - g;
    const int n_kv = causal ? std::min(kv_tiles, (mt * kTileM + kTileM) / kDqTileN) : kv_tiles;
    w[g] = n_kv + 2.0;
  }
  qtile_schedule_w(NP, w, B * Hq, sms, out, grid);
}

// The schedule depends only on (pipelines per block, B, T, Hq, causal, SMs):
// the last one for each pipeline count is kept (the forward and dQ of one
// layer each reuse theirs).
void cached_qtile_schedule(int NP, int B, int T, int Hq, int causal, int sms, QTileSched* out,
                           int* grid) {
  static std::mutex mu;
  static int key[2][6] = {{-1, -1, -1, -1, -1, -1}, {-1, -1, -1, -1, -1, -1}};
  static QTileSched sched[2];
  static int g[2] = {0, 0};
  std::lock_guard<std::mutex> lock(mu);
  const int slot = NP > 1 ? 1 : 0;
  const int want[6] = {NP, B, T, Hq, causal, sms};
  if (!std::equal(want, want + 6, key[slot])) {
    qtile_schedule(NP, B, T, Hq, causal, sms, &sched[slot], &g[slot]);
    std::copy(want, want + 6, key[slot]);
  }
  *out = sched[slot];
  *grid = g[slot];
}

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T,
             int Hq, int Hkv, int D, float scale, int causal, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mo;
  int rc;
  if ((rc = encode_rows(&mq, q, B, T, Hq, D, kTileM, "q")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mk, k, B, T, Hkv, D, kFwdTileN, "k")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mv, v, B, T, Hkv, D, kFwdTileN, "v")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mo, o, B, T, Hq, D, kFwdStoreRows, "o")) != DETATTN_OK) return rc;
  FwdArgs a{};
  a.o = o;
  a.lse = lse;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.n_m = (T + kTileM - 1) / kTileM;
  a.BHq = B * Hq;
  a.causal = causal;
  a.scale_log2 = log2e_times(scale);
  a.wait_ns = g_wait_ns;
  int sms = 0;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  QTileSched sc;
  int g;
  cached_qtile_schedule(fwd_pipes_per_block(D), B, T, Hq, causal, sms, &sc, &g);
  return launched(launch_fwd(D, g, mq, mk, mv, mo, a, sc, nullptr, st), "attn_fwd");
}

// Workspace: the row statistics, then (from a 256-byte boundary) the dQ
// step's unit counter (two words: units taken, pipelines done).  A workspace too short for the counter runs the dQ
// step on the host's static deal instead.
size_t rowstat_bytes(int B, int T, int Hq) {
  return static_cast<size_t>(B) * Hq * padded_T(T) * sizeof(float2);
}
size_t counter_offset(int B, int T, int Hq) { return (rowstat_bytes(B, T, Hq) + 255) / 256 * 256; }
unsigned* unit_counter_ptr(const void* ws, size_t bytes, int B, int T, int Hq) {
  if (bytes < counter_offset(B, T, Hq) + 2 * sizeof(unsigned)) return nullptr;
  return reinterpret_cast<unsigned*>(static_cast<char*>(const_cast<void*>(ws)) +
                                     counter_offset(B, T, Hq));
}

int delta_impl(const void* o, const void* dout, const float* lse, void* workspace, int B, int T,
               int Hq, int D, unsigned* counter, cudaStream_t st) {
  DeltaArgs a{o, dout, lse, static_cast<float2*>(workspace), B, T, padded_T(T), Hq, D, counter};
  int sms = 0;
  int rc;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  return launched(launch_delta(a, sms, nullptr, st), "attn_bwd_delta");
}

BwdArgs bwd_args(const void* workspace, int T, int Hq, int Hkv, float scale, int causal) {
  BwdArgs a{};
  a.rowstats = static_cast<const float2*>(workspace);
  a.T = T;
  a.Tk = T;
  a.Tp = padded_T(T);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.causal = causal;
  a.scale = scale;
  a.scale_log2 = log2e_times(scale);
  a.wait_ns = g_wait_ns;
  return a;
}

int sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  static int cached[64] = {};
  if (e == cudaSuccess && dev < 64 && cached[dev] > 0) {
    *out = cached[dev];
    return DETATTN_OK;
  }
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(DETATTN_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
  if (dev < 64) cached[dev] = *out;
  return DETATTN_OK;
}

// Shape of the persistent dK/dV launch: C blocks per key tile (a cluster) and
// NG resident clusters, dealt the key tiles (heaviest first) in snake order.
// C is the power of two (up to the kernel's limit for D) that minimises the
// largest per-block load of that deal, counting a tile's K/V reload and
// epilogue as two items; NG is every cluster of C blocks that can be resident
// at once (at most one per tile).  Both depend only on the shape and the
// device, so the summation order, and with it every output bit, is fixed for
// a given problem and GPU.  `forced_c` > 0 takes that C (capped at the limit).
// `resident[i]`: clusters of 2^i blocks the device holds at once (0: none).
// Returns false when no allowed C can be resident.
// The choice over key tiles in walk order: tile t carries items[t / per_group]
// items (per_group = 1: one entry per tile).
// At D = 128 with one block per tile the 128-query kernel runs: `items_one`
// (tiles in that walk's order) then holds its 64-query halves, each weighted
// kQ128Weight of a 64-query item of the clustered kernel (measured at B = 1,
// T = 8192, Hq = 32, Hkv = 8: 2.13 us per 128 queries against 1.22 us per
// 64); `items_split` is the walk of C > 1.
constexpr double kQ128Weight = 0.875;
bool dkdv_choose_items(const std::vector<int>& items_one, const std::vector<int>& items_split,
                       int per_group, int D, const int resident[4], int forced_c, int* c_out,
                       int* ng_out) {
  const long total = static_cast<long>(items_split.size()) * per_group;
  const int cmax = dkdv_max_cluster_size(D);
  const double per_item64 = 64.0 / dkdv_tile_m(D);  // fixed costs in this kernel's items
  double best = 0.0;
  *c_out = 0;
  *ng_out = 0;
  for (int c = 1, i = 0; c <= cmax && i < 4; c *= 2, ++i) {
    if (forced_c > 0 && c != (forced_c < cmax ? forced_c : cmax)) continue;
    if (resident[i] < 1) continue;
    const long ng = total < resident[i] ? total : resident[i];
    const std::vector<int>& items_per_group = c == 1 ? items_one : items_split;
    const double w = (c == 1 && D == 128) ? kQ128Weight : 1.0;
    double worst = 0.0;
    for (long k = 0; k < ng; ++k) {
      double load = 0.0;
      for (long kt = 0;; ++kt) {
        const long t = kt * ng + ((kt & 1) ? ng - 1 - k : k);
        if (t >= total) break;
        const int items = items_per_group[t / per_group];
        // Per tile: its share of the items, one 64-query item's worth for
        // writing the sums out, and two per peer for the partial-sum exchange
        // (measured: distributed shared memory moves ~9 bytes per clock per
        // SM, and a 64-query item takes ~1,500 clocks); items of TM queries
        // count TM / 64 such items.
        load += w * ((items + c - 1) / c) + (1.0 + 2.0 * (c - 1)) * per_item64;
      }
      if (load > worst) worst = load;
    }
    if (*c_out == 0 || worst < best - 1e-9) {
      best = worst;
      *c_out = c;
      *ng_out = static_cast<int>(ng);
    }
  }
  return *c_out != 0;
}

// (b, KV head) pairs per chunk of the dK/dV walk (0: no chunks): chunks keep
// the queries and output gradients the clusters read at once to about 32 MB
// (they stay in L2) when all of them together would not fit.
int dkdv_bg_chunk(int B, int T, int Hq, int Hkv, int D) {
  const double group_bytes = static_cast<double>(T) * (Hq / Hkv) * D * 2 * 2;  // Q and dO
  const int BH = B * Hkv;
  if (group_bytes * BH <= 48.0 * (1 << 20)) return 0;
  int g = static_cast<int>(32.0 * (1 << 20) / group_bytes);
  if (g < 1) g = 1;
  while (g > 1 && BH % g != 0) --g;  // whole chunks
  return g >= BH ? 0 : g;
}

// The chunk of the walk with one block per tile: none at D = 128.
int dkdv_bg_chunk_one(int D, int chunk) { return D == 128 ? 0 : chunk; }

bool dkdv_choose(int B, int T, int Hq, int Hkv, int D, int causal, const int resident[4],
                 int forced_c, int* c_out, int* ng_out) {
  const int G = Hq / Hkv;
  const int n_tiles = (T + kTileN - 1) / kTileN;
  const int tm = dkdv_tile_m(D);
  const int m_end = (T + tm - 1) / tm;
  const int BH = B * Hkv;
  const int chunk = dkdv_bg_chunk(B, T, Hq, Hkv, D);
  // The walk with clusters (chunked when Q and dO do not fit in L2 at once)
  // and the walk of one block per tile, which at D = 128 takes the tiles
  // heaviest first without chunks (measured: the chunked walk of that kernel
  // left blocks idle for up to 40 % of the step).
  std::vector<int> items(static_cast<size_t>(n_tiles) * BH), items_one(items.size());
  for (long t = 0; t < static_cast<long>(items.size()); ++t) {
    int nt, bg;
    dkdv_tile_coords(static_cast<int>(t), n_tiles, BH, chunk, &nt, &bg);
    items[t] = G * (m_end - (causal ? nt * kTileN / tm : 0));
    dkdv_tile_coords(static_cast<int>(t), n_tiles, BH, dkdv_bg_chunk_one(D, chunk), &nt, &bg);
    items_one[t] = G * (m_end - (causal ? nt * kTileN / tm : 0));
  }
  return dkdv_choose_items(items_one, items, 1, D, resident, forced_c, c_out, ng_out);
}

// dkdv_choose with the current device's residency: `sms` blocks alone, and
// the cluster sizes it supports from the occupancy query.
int dkdv_schedule(int B, int T, int Hq, int Hkv, int D, int causal, int sms, int forced_c,
                  int* c_out, int* ng_out) {
  const int cmax = dkdv_max_cluster_size(D);
  int resident[4] = {sms, 0, 0, 0};
  for (int c = 2, i = 1; c <= cmax && i < 4; c *= 2, ++i) {
    if (forced_c > 0 && c != (forced_c < cmax ? forced_c : cmax)) continue;
    cudaError_t e = dkdv_max_clusters(D, c, &resident[i]);
    if (e != cudaSuccess) {
      return fail(DETATTN_ERR_CUDA, "attn_bwd_dkdv: cluster occupancy query: %s",
                  cudaGetErrorString(e));
    }
  }
  if (!dkdv_choose(B, T, Hq, Hkv, D, causal, resident, forced_c, c_out, ng_out)) {
    return fail(DETATTN_ERR_CUDA, "attn_bwd_dkdv: no resident cluster shape for D = %d", D);
  }
  return DETATTN_OK;
}

// Listed deal of the 64-dim dK/dV kernel's key tiles over NG clusters of C
// blocks (the walk without chunks; see DkvList).  `items[t]`: the items of
// tile t in walk order.  Tiles with at least x items are shared by a
// cluster, lighter ones go whole to single blocks.  Heaviest first, a shared
// tile goes to the cluster whose blocks carry the least and adds its share
// of the items to each of them, a whole tile to the block with the least.
// Besides its items a tile costs its end: reading the sums, and when shared
// sending the peers' rows and waiting for theirs (measured at B = 4, T =
// 1024, 12 query and 4 KV heads of 64: a shared tile's end and the next
// tile's start take 4.3-5 us, about four 1.1 us items; a whole tile's end,
// without the exchange, is taken as one and a half).
// x is the item count that minimises the largest block load; the list is
// kept when that load is below the snake walk's under the same costs (always
// with `force`).  Returns false without a list, or when it does not fit.
// Depends only on the tile loads, C and NG, so the sums' order is fixed for a
// problem and a device.
constexpr double kDkvSharedEnd = 4.0, kDkvOwnEnd = 1.5;
bool dkdv_mixed_list(const std::vector<int>& items, int C, int NG, bool force, DkvList* out) {
  const int n = static_cast<int>(items.size());
  const int nb = NG * C;
  if (C < 2 || NG < 1 || nb > kDkvListMaxBlocks || n < 1 || n >= 32768) return false;
  double snake = 0.0;
  for (int k = 0; k < NG; ++k) {
    double load = 0.0;
    for (int kt = 0;; ++kt) {
      const int t = kt * NG + ((kt & 1) ? NG - 1 - k : k);
      if (t >= n) break;
      load += (items[t] + C - 1) / C + kDkvSharedEnd;
    }
    snake = std::max(snake, load);
  }
  std::vector<int> order(n);
  for (int t = 0; t < n; ++t) order[t] = t;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return items[x] > items[y]; });
  std::vector<int> xs;
  for (int t : order)
    if (xs.empty() || items[t] != xs.back()) xs.push_back(items[t]);
  xs.push_back(INT32_MAX);  // nothing shared
  double best = 0.0;
  std::vector<std::vector<uint16_t>> best_lists;
  // Loads are sums of whole items and the two end costs (exact in double);
  // each pick takes the least load, the lowest index among equals.
  using Slot = std::pair<double, int>;
  using MinHeap = std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>>;
  for (int x : xs) {
    std::vector<double> load(nb, 0.0);
    std::vector<std::vector<uint16_t>> lists(nb);
    long entries = 0;
    // Shared tiles first: a cluster's blocks carry equal loads until then.
    MinHeap clusters;
    for (int c = 0; c < NG; ++c) clusters.push({0.0, c});
    for (int t : order) {
      if (items[t] < x) continue;
      const Slot top = clusters.top();
      clusters.pop();
      const double add = (items[t] + C - 1) / C + kDkvSharedEnd;
      for (int j = 0; j < C; ++j) {
        load[top.second * C + j] += add;
        lists[top.second * C + j].push_back(static_cast<uint16_t>((t << 1) | 1));
      }
      clusters.push({top.first + add, top.second});
      entries += C;
    }
    MinHeap blocks;
    for (int j = 0; j < nb; ++j) blocks.push({load[j], j});
    for (int t : order) {
      if (items[t] >= x) continue;
      const Slot top = blocks.top();
      blocks.pop();
      load[top.second] += items[t] + kDkvOwnEnd;
      lists[top.second].push_back(static_cast<uint16_t>(t << 1));
      blocks.push({load[top.second], top.second});
      ++entries;
    }
    if (entries > kDkvListMaxEntries) continue;
    const double m = *std::max_element(load.begin(), load.end());
    if (best_lists.empty() || m < best - 1e-9) {
      best = m;
      best_lists = std::move(lists);
    }
  }
  if (best_lists.empty() || (!force && !(best < snake - 1e-9))) return false;
  out->n_blocks = nb;
  int e = 0;
  for (int i = 0; i < nb; ++i) {
    out->start[i] = static_cast<uint16_t>(e);
    for (uint16_t v : best_lists[i]) out->entry[e++] = v;
  }
  out->start[nb] = static_cast<uint16_t>(e);
  return true;
}

// dkdv_mixed_list for a fixed-length shape (tiles in the unchunked walk's
// order), the last result kept: one layer's backward asks again every step.
// Copied into *out under the lock (another thread may replace the kept one).
bool cached_dkdv_list(int B, int T, int Hq, int Hkv, int causal, int C, int NG, int deal,
                      DkvList* out) {
  static std::mutex mu;
  static int key[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
  static DkvList list;
  static bool have = false;
  std::lock_guard<std::mutex> lock(mu);
  const int want[8] = {B, T, Hq, Hkv, causal, C, NG, deal};
  if (!std::equal(want, want + 8, key)) {
    const int G = Hq / Hkv, BH = B * Hkv;
    const int tm = dkdv_tile_m(64);
    const int n_tiles = (T + kTileN - 1) / kTileN, m_end = (T + tm - 1) / tm;
    std::vector<int> items(static_cast<size_t>(n_tiles) * BH);
    for (size_t t = 0; t < items.size(); ++t) {
      const int nt = static_cast<int>(t) / BH;
      items[t] = G * (m_end - (causal ? nt * kTileN / tm : 0));
    }
    have = dkdv_mixed_list(items, C, NG, deal == 2, &list);
    std::copy(want, want + 8, key);
  }
  if (have) std::memcpy(out, &list, sizeof(DkvList));
  return have;
}

int dkdv_impl(const void* q, const void* k, const void* v, const void* dout,
              const void* workspace, void* dk, void* dv, int B, int T, int Hq, int Hkv, int D,
              float scale, int causal, cudaStream_t st, bool after_delta = false,
              void* ds = nullptr, long ds_pairs = 0) {
  CUtensorMap mq, mk, mv, mdo;
  int rc;
  BwdArgs a = bwd_args(workspace, T, Hq, Hkv, scale, causal);
  a.dk = dk;
  a.dv = dv;
  a.n_tiles = (T + kTileN - 1) / kTileN;
  a.BH = B * Hkv;
  a.ds = ds;
  a.ds_pairs = ds_pairs;
  a.bg_chunk = dkdv_bg_chunk(B, T, Hq, Hkv, D);
  int sms = 0;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  if ((rc = dkdv_schedule(B, T, Hq, Hkv, D, causal, sms, g_dkdv_split, &a.cluster, &a.n_groups)) !=
      DETATTN_OK)
    return rc;
  if (a.cluster == 1 && ds == nullptr) a.bg_chunk = dkdv_bg_chunk_one(D, a.bg_chunk);
  DkvList own;
  const DkvList* list = nullptr;
  // (The stored-dS form takes the same deal, so both forms give the same dK, dV.)
  if (D == 64 && a.bg_chunk == 0 && a.cluster > 1 && g_dkdv_deal != 1)
    list = cached_dkdv_list(B, T, Hq, Hkv, causal, a.cluster, a.n_groups, g_dkdv_deal, &own)
               ? &own
               : nullptr;
  // The stored-dS form keeps 64-query items at D = 128.
  const int rows = ds != nullptr && D == 128 ? 64 : dkdv_item_rows(D, a.cluster);
  if ((rc = encode_rows(&mq, q, B, T, Hq, D, rows, "q")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mdo, dout, B, T, Hq, D, rows, "dout")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mk, k, B, T, Hkv, D, kTileN, "k")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mv, v, B, T, Hkv, D, kTileN, "v")) != DETATTN_OK) return rc;
  return launched(
      launch_dkdv(D, a.n_groups * a.cluster, mq, mk, mv, mdo, a, after_delta, nullptr, list, st),
      "attn_bwd_dkdv");
}

int dq_impl(const void* q, const void* k, const void* v, const void* dout, const void* workspace,
            void* dq, int B, int T, int Hq, int Hkv, int D, float scale, int causal,
            unsigned* counter, cudaStream_t st, bool after_dkdv = false) {
  CUtensorMap mq, mk, mv, mdo, mdq;
  int rc;
  if ((rc = encode_rows(&mq, q, B, T, Hq, D, kTileM, "q")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mdo, dout, B, T, Hq, D, kTileM, "dout")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mk, k, B, T, Hkv, D, kDqTileN, "k")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mv, v, B, T, Hkv, D, kDqTileN, "v")) != DETATTN_OK) return rc;
  if ((rc = encode_rows_store(&mdq, dq, B, T, Hq, D, D / 2, kDqStoreRows, "dq")) != DETATTN_OK)
    return rc;
  BwdArgs a = bwd_args(workspace, T, Hq, Hkv, scale, causal);
  a.dq = dq;
  a.n_tiles = (T + kTileM - 1) / kTileM;
  a.BH = B * Hq;
  a.unit_counter = counter;
  int sms = 0;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  QTileSched sc;
  int g;
  cached_qtile_schedule(dq_pipes_per_block(D), B, T, Hq, causal, sms, &sc, &g);
  return launched(launch_dq(D, g, mq, mk, mv, mdo, mdq, a, sc, nullptr, after_dkdv, st),
                  "attn_bwd_dq");
}

int check_workspace(const void* ws, size_t bytes, int B, int T, int Hq) {
  if (ws == nullptr || bytes < rowstat_bytes(B, T, Hq))
    return fail(DETATTN_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu%s",
                rowstat_bytes(B, T, Hq), bytes, ws ? "" : " (NULL)");
  if (!aligned16(ws)) return fail(DETATTN_ERR_ALIGN, "workspace is not 16-byte aligned");
  return DETATTN_OK;
}

// ------------------------------------------------------------ stored-dS backward
// With a workspace long enough, the dK/dV step also stores each dS tile it
// forms and the dQ step becomes a plain product dQ = scale dS K (no
// recomputed S, P, dP): pairs (query tile, key tile) of 128 x 128, two bf16
// halves of 128 x 64 each, after the row statistics and the counter.
int g_bwd_dq_mode = 0;  // 0: recompute in the dQ step; 1: stored dS when the workspace holds it

long ds_pairs(int T, int causal) {
  const long n = (T + kTileM - 1) / kTileM;
  return causal ? n * (n + 1) / 2 : n * n;
}
size_t ds_offset(int B, int T, int Hq) { return counter_offset(B, T, Hq) + 256; }
size_t ds_region_bytes(int B, int T, int Hq, int causal) {
  return static_cast<size_t>(B) * Hq * ds_pairs(T, causal) * 2 * kTileN * 64 * 2;
}

int dq_from_ds_impl(const void* k, const void* ds, void* dq, long pairs, int B, int T, int Hq,
                    int Hkv, int D, float scale, int causal, cudaStream_t st) {
  CUtensorMap mds, mk;
  int rc;
  const long rows = static_cast<long>(B) * Hq * pairs * 2 * kTileN;
  if ((rc = encode_2d_rows64(&mds, ds, rows)) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mk, k, B, T, Hkv, D, 64, "k")) != DETATTN_OK) return rc;
  BwdArgs a = bwd_args(nullptr, T, Hq, Hkv, scale, causal);
  a.dq = dq;
  a.n_tiles = (T + kTileM - 1) / kTileM;
  a.BH = B * Hq;
  a.ds_pairs = pairs;
  return launched(launch_dq_from_ds(D, mds, mk, a, a.n_tiles * a.BH, st), "attn_bwd dQ from dS");
}

// Delta, dK/dV and dQ on `st`, each a programmatic dependent of the one
// before: dK/dV loads its operands while Delta runs, and dQ, which needs only
// Delta's results, starts once every dK/dV block is past Delta and takes the
// SMs the dK/dV grid frees (or, with a workspace that holds the dS tiles,
// dK/dV then dQ from dS).
int bwd_steps(const void* q, const void* k, const void* v, const void* o, const float* lse,
              const void* dout, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, int B,
              int T, int Hq, int Hkv, int D, float scale, int causal, cudaStream_t st) {
  int rc;
  unsigned* counter = unit_counter_ptr(ws, ws_bytes, B, T, Hq);
  if (g_bwd_dq_mode == 1 && ws_bytes >= ds_offset(B, T, Hq) + ds_region_bytes(B, T, Hq, causal) &&
      static_cast<double>(B) * Hq * ds_pairs(T, causal) * 2 * kTileN < 2.0e9) {
    void* ds = static_cast<char*>(ws) + ds_offset(B, T, Hq);
    const long pairs = ds_pairs(T, causal);
    if ((rc = delta_impl(o, dout, lse, ws, B, T, Hq, D, counter, st)) != DETATTN_OK) return rc;
    if ((rc = dkdv_impl(q, k, v, dout, ws, dk, dv, B, T, Hq, Hkv, D, scale, causal, st,
                        /*after_delta=*/true, ds, pairs)) != DETATTN_OK)
      return rc;
    if ((rc = dq_from_ds_impl(k, ds, dq, pairs, B, T, Hq, Hkv, D, scale, causal, st)) != DETATTN_OK)
      return rc;
    return ok_status();
  }
  if ((rc = delta_impl(o, dout, lse, ws, B, T, Hq, D, counter, st)) != DETATTN_OK) return rc;
  if ((rc = dkdv_impl(q, k, v, dout, ws, dk, dv, B, T, Hq, Hkv, D, scale, causal, st,
                      /*after_delta=*/true)) != DETATTN_OK)
    return rc;
  if ((rc = dq_impl(q, k, v, dout, ws, dq, B, T, Hq, Hkv, D, scale, causal, counter, st,
                    /*after_dkdv=*/true)) != DETATTN_OK)
    return rc;
  return ok_status();
}

// ------------------------------------------------------------ packed variable-length batches
// Host form of a packed batch: the kernel tables (query tiles for the
// forward and dQ steps, key tiles for the dK/dV step) and the per-group work
// the deals weigh.  Built from the host arrays cu_q, cu_k on every call.
struct Packed {
  int n_seq = 0, total_q = 0, total_k = 0, Tp = 0;
  VarlenTable qt{}, kt{};
  std::vector<double> q_weight;  // per q-table entry: visible 64-key tiles + 2
  std::vector<int> k_items;      // per k-table entry: items of one KV head
};

int check_packed(const int* cu_q, const int* cu_k, int n_seq, int Hq, int Hkv, int D, int causal,
                 Packed* pk) {
  if (n_seq < 0 || n_seq > kVarlenMaxSeqs)
    return fail(DETATTN_ERR_SHAPE, "n_seq=%d: must be in [0, %d]", n_seq, kVarlenMaxSeqs);
  if (n_seq > 0 && (cu_q == nullptr || cu_k == nullptr))
    return fail(DETATTN_ERR_NULL, "cu_q and cu_k must not be NULL");
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return fail(DETATTN_ERR_SHAPE, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  if (D != 64 && D != 128) return fail(DETATTN_ERR_HEADDIM, "D=%d: only 64 and 128", D);
  pk->n_seq = n_seq;
  if (n_seq == 0) return DETATTN_OK;
  if (cu_q[0] != 0 || cu_k[0] != 0) return fail(DETATTN_ERR_SHAPE, "cu_q[0] and cu_k[0] must be 0");
  long ps = 0;
  for (int s = 0; s < n_seq; ++s) {
    const long tq = static_cast<long>(cu_q[s + 1]) - cu_q[s];
    const long tk = static_cast<long>(cu_k[s + 1]) - cu_k[s];
    if (tq < 0 || tk < 0)
      return fail(DETATTN_ERR_SHAPE, "sequence %d: cu_q / cu_k must not decrease", s);
    if (tq > (1L << 22) || tk > (1L << 22))
      return fail(DETATTN_ERR_SHAPE, "sequence %d longer than 2^22 rows", s);
    ps += (tq + 127) / 128 * 128;
  }
  const double elems = static_cast<double>(cu_q[n_seq]) * Hq * D + static_cast<double>(cu_k[n_seq]) * Hkv * D;
  if (ps > (1L << 30) || static_cast<double>(ps) * Hq > 1.0e11 || elems > 1.0e12)
    return fail(DETATTN_ERR_SHAPE, "packed problem too large");
  pk->total_q = cu_q[n_seq];
  pk->total_k = cu_k[n_seq];
  pk->Tp = static_cast<int>(ps);
  for (VarlenTable* t : {&pk->qt, &pk->kt}) {
    t->n_seq = n_seq;
    int p = 0;
    for (int s = 0; s <= n_seq; ++s) {
      t->cu_q[s] = cu_q[s];
      t->cu_k[s] = cu_k[s];
      t->ps[s] = p;
      if (s < n_seq) p += (cu_q[s + 1] - cu_q[s] + 127) / 128 * 128;
    }
  }
  // Query tiles, heaviest first (visible 64-key tiles of the tile's last row).
  struct QE { double w; int s, mt; };
  std::vector<QE> qe;
  for (int s = 0; s < n_seq; ++s) {
    const int tq = cu_q[s + 1] - cu_q[s], tk = cu_k[s + 1] - cu_k[s], off = tk - tq;
    const int tiles = (tk + kDqTileN - 1) / kDqTileN;
    for (int mt = 0; mt * kTileM < tq; ++mt) {
      const int last = std::min(mt * kTileM + kTileM - 1, tq - 1) + off;
      const int n_kv = causal ? (last < 0 ? 0 : std::min(tiles, last / kDqTileN + 1)) : tiles;
      qe.push_back({n_kv + 2.0, s, mt});
    }
  }
  // Key tiles, heaviest first (items: query tiles of TM rows that see them).
  const int tm = dkdv_tile_m(D), G = Hq / Hkv;
  struct KE { int items, s, nt; };
  std::vector<KE> ke;
  for (int s = 0; s < n_seq; ++s) {
    const int tq = cu_q[s + 1] - cu_q[s], tk = cu_k[s + 1] - cu_k[s], off = tk - tq;
    const int mq_end = (tq + tm - 1) / tm;
    for (int nt = 0; nt * kTileN < tk; ++nt) {
      const int first_q = nt * kTileN - off;
      const int m_begin = causal ? std::min(mq_end, std::max(0, first_q) / tm) : 0;
      ke.push_back({G * (mq_end - m_begin), s, nt});
    }
  }
  if (qe.size() > static_cast<size_t>(kVarlenMaxTiles) ||
      ke.size() > static_cast<size_t>(kVarlenMaxTiles))
    return fail(DETATTN_ERR_SHAPE, "packed batch has %zu query / %zu key tiles of 128; at most %d",
                qe.size(), ke.size(), kVarlenMaxTiles);
  std::stable_sort(qe.begin(), qe.end(), [](const QE& x, const QE& y) { return x.w > y.w; });
  std::stable_sort(ke.begin(), ke.end(), [](const KE& x, const KE& y) { return x.items > y.items; });
  pk->qt.n_tiles = static_cast<int>(qe.size());
  pk->kt.n_tiles = static_cast<int>(ke.size());
  for (size_t i = 0; i < qe.size(); ++i) {
    pk->qt.tile[i] = (static_cast<uint32_t>(qe[i].s) << 16) | static_cast<uint32_t>(qe[i].mt);
    pk->q_weight.push_back(qe[i].w);
  }
  for (size_t i = 0; i < ke.size(); ++i) {
    pk->kt.tile[i] = (static_cast<uint32_t>(ke[i].s) << 16) | static_cast<uint32_t>(ke[i].nt);
    pk->k_items.push_back(ke[i].items);
  }
  return DETATTN_OK;
}

size_t packed_rowstat_bytes(const Packed& pk, int Hq) {
  return static_cast<size_t>(Hq) * pk.Tp * sizeof(float2);
}
size_t packed_counter_offset(const Packed& pk, int Hq) {
  return (packed_rowstat_bytes(pk, Hq) + 255) / 256 * 256;
}

int fwd_varlen_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                    const Packed& pk, int Hq, int Hkv, int D, float scale, int causal,
                    cudaStream_t st) {
  if (pk.qt.n_tiles == 0) return ok_status();
  CUtensorMap mq, mk, mv, mo;
  int rc;
  // Without any key rows the kernels never load K, V, but the tensor maps
  // still need an address: q stands in.
  const int tk_rows = pk.total_k > 0 ? pk.total_k : 1;
  const void* kk = pk.total_k > 0 ? k : q;
  const void* vv = pk.total_k > 0 ? v : q;
  if ((rc = encode_rows(&mq, q, 1, pk.total_q, Hq, D, kTileM, "q")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mk, kk, 1, tk_rows, Hkv, D, kFwdTileN, "k")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mv, vv, 1, tk_rows, Hkv, D, kFwdTileN, "v")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mo, o, 1, pk.total_q, Hq, D, kFwdStoreRows, "o")) != DETATTN_OK) return rc;
  FwdArgs a{};
  a.o = o;
  a.lse = lse;
  a.T = pk.total_q;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.n_m = 0;
  a.BHq = Hq;
  a.causal = causal;
  a.scale_log2 = log2e_times(scale);
  a.wait_ns = g_wait_ns;
  int sms = 0;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  QTileSched sc;
  int g;
  qtile_schedule_w(fwd_pipes_per_block(D), pk.q_weight, Hq, sms, &sc, &g);
  return launched(launch_fwd(D, g, mq, mk, mv, mo, a, sc, &pk.qt, st), "attn_fwd_varlen");
}

int bwd_varlen_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                    const Packed& pk, int Hq, int Hkv, int D, float scale, int causal,
                    cudaStream_t st) {
  int rc;
  int sms = 0;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  unsigned* counter = nullptr;
  if (ws_bytes >= packed_counter_offset(pk, Hq) + 2 * sizeof(unsigned))
    counter = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + packed_counter_offset(pk, Hq));
  if (pk.total_q > 0) {
    DeltaArgs da{o, dout, lse, static_cast<float2*>(ws), 1, pk.total_q, pk.Tp, Hq, D, counter};
    if ((rc = launched(launch_delta(da, sms, &pk.qt, st), "attn_bwd_varlen (Delta)")) != DETATTN_OK)
      return rc;
  }
  BwdArgs a{};
  a.rowstats = static_cast<const float2*>(ws);
  a.T = pk.total_q;
  a.Tk = pk.total_k;
  a.Tp = pk.Tp;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.causal = causal;
  a.scale = scale;
  a.scale_log2 = log2e_times(scale);
  a.wait_ns = g_wait_ns;
  // Maps over rows that no kernel will load (no query rows, or no key rows)
  // still need an address: the other side's tensor stands in.
  const int tq_rows = pk.total_q > 0 ? pk.total_q : 1, tk_rows = pk.total_k > 0 ? pk.total_k : 1;
  const void* qq = pk.total_q > 0 ? q : k;
  const void* dd = pk.total_q > 0 ? dout : k;
  const void* kk = pk.total_k > 0 ? k : q;
  const void* vv = pk.total_k > 0 ? v : q;
  if (pk.kt.n_tiles > 0) {
    // dK/dV (every key row belongs to some key tile, so all of dk, dv is written).
    CUtensorMap mq, mk, mv, mdo;
    BwdArgs b = a;
    b.dk = dk;
    b.dv = dv;
    b.BH = Hkv;
    const int cmax = dkdv_max_cluster_size(D);
    int resident[4] = {sms, 0, 0, 0};
    for (int c = 2, i = 1; c <= cmax && i < 4; c *= 2, ++i) {
      if (g_dkdv_split > 0 && c != (g_dkdv_split < cmax ? g_dkdv_split : cmax)) continue;
      cudaError_t e = dkdv_max_clusters(D, c, &resident[i]);
      if (e != cudaSuccess)
        return fail(DETATTN_ERR_CUDA, "attn_bwd_varlen: cluster occupancy query: %s",
                    cudaGetErrorString(e));
    }
    if (!dkdv_choose_items(pk.k_items, pk.k_items, Hkv, D, resident, g_dkdv_split, &b.cluster,
                           &b.n_groups))
      return fail(DETATTN_ERR_CUDA, "attn_bwd_varlen: no resident cluster shape for D = %d", D);
    // The listed deal as for fixed lengths, over the table's tiles (the
    // items of tile t are those of its entry t / Hkv).
    DkvList list;
    bool listed = false;
    if (D == 64 && b.cluster > 1 && g_dkdv_deal != 1) {
      std::vector<int> items(pk.k_items.size() * static_cast<size_t>(Hkv));
      for (size_t t = 0; t < items.size(); ++t) items[t] = pk.k_items[t / Hkv];
      listed = dkdv_mixed_list(items, b.cluster, b.n_groups, g_dkdv_deal == 2, &list);
    }
    const int rows = dkdv_item_rows(D, b.cluster);
    if ((rc = encode_rows(&mq, qq, 1, tq_rows, Hq, D, rows, "q")) != DETATTN_OK) return rc;
    if ((rc = encode_rows(&mdo, dd, 1, tq_rows, Hq, D, rows, "dout")) != DETATTN_OK) return rc;
    if ((rc = encode_rows(&mk, kk, 1, tk_rows, Hkv, D, kTileN, "k")) != DETATTN_OK) return rc;
    if ((rc = encode_rows(&mv, vv, 1, tk_rows, Hkv, D, kTileN, "v")) != DETATTN_OK) return rc;
    if ((rc = launched(launch_dkdv(D, b.n_groups * b.cluster, mq, mk, mv, mdo, b, pk.total_q > 0,
                                   &pk.kt, listed ? &list : nullptr, st),
                       "attn_bwd_varlen (dK/dV)")) != DETATTN_OK)
      return rc;
  }
  if (pk.qt.n_tiles > 0) {
    CUtensorMap mq, mk, mv, mdo, mdq;
    if ((rc = encode_rows(&mq, qq, 1, tq_rows, Hq, D, kTileM, "q")) != DETATTN_OK) return rc;
    if ((rc = encode_rows(&mdo, dd, 1, tq_rows, Hq, D, kTileM, "dout")) != DETATTN_OK) return rc;
    if ((rc = encode_rows(&mk, kk, 1, tk_rows, Hkv, D, kDqTileN, "k")) != DETATTN_OK) return rc;
    if ((rc = encode_rows(&mv, vv, 1, tk_rows, Hkv, D, kDqTileN, "v")) != DETATTN_OK) return rc;
    if ((rc = encode_rows_store(&mdq, dq, 1, pk.total_q, Hq, D, D / 2, kDqStoreRows, "dq")) !=
        DETATTN_OK)
      return rc;
    BwdArgs b = a;
    b.dq = dq;
    b.BH = Hq;
    b.unit_counter = counter;
    QTileSched sc;
    int g;
    qtile_schedule_w(dq_pipes_per_block(D), pk.q_weight, Hq, sms, &sc, &g);
    // A programmatic dependent of the dK/dV step when it was launched just
    // before (not of the Delta step, which lets its dependents start early).
    if ((rc = launched(
             launch_dq(D, g, mq, mk, mv, mdo, mdq, b, sc, &pk.qt, pk.kt.n_tiles > 0, st),
             "attn_bwd_varlen (dQ)")) != DETATTN_OK)
      return rc;
  }
  return ok_status();
}

// ------------------------------------------------------------ layer GEMM and training step
// 2-D bf16 tensor map of a row-major matrix with `outer` rows of `inner`
// contiguous elements (row stride ld elements), box {box_inner, box_outer},
// 128-byte swizzle.
int encode_2d(CUtensorMap* m, const void* ptr, long inner, long outer, long ld, int box_inner,
              int box_outer, const char* what) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DETATTN_ERR_CUDA, "tensor map for %s: CUresult %d", what, (int)r);
  return DETATTN_OK;
}

int check_gemm(const void* a, int a_mn, long lda, const void* b, int b_mn, long ldb, const void* c,
               int c_f32, long ldc, int M, int N, int K) {
  int rc;
  if ((rc = check_ptrs({{a, "a"}, {b, "b"}, {c, "c"}})) != DETATTN_OK) return rc;
  if (M < kTileM || N < kGemmBN || K < 64 || M % kTileM || N % kGemmBN || K % 64)
    return fail(DETATTN_ERR_SHAPE, "GEMM M=%d N=%d K=%d: need multiples of 128, %d and 64", M, N,
                K, kGemmBN);
  if (static_cast<double>(M) * N > 4.0e9 || static_cast<double>(M) * K > 4.0e9 ||
      static_cast<double>(K) * N > 4.0e9 || M > (1 << 24) || N > (1 << 24) || K > (1 << 24))
    return fail(DETATTN_ERR_SHAPE, "GEMM too large (M=%d N=%d K=%d)", M, N, K);
  if (a_mn < 0 || a_mn > 1 || b_mn < 0 || b_mn > 1 || c_f32 < 0 || c_f32 > 1)
    return fail(DETATTN_ERR_SHAPE, "GEMM layout flags must be 0 or 1");
  if (lda < (a_mn ? M : K) || ldb < (b_mn ? N : K) || ldc < N || lda % 8 || ldb % 8 ||
      ldc % (c_f32 ? 4 : 8))
    return fail(DETATTN_ERR_SHAPE,
                "GEMM leading dimensions lda=%ld ldb=%ld ldc=%ld: too short or not 16-byte rows",
                lda, ldb, ldc);
  return DETATTN_OK;
}

int gemm_impl(const void* a, int a_mn, long lda, const void* b, int b_mn, long ldb, void* c,
              int c_f32, long ldc, int M, int N, int K, float alpha, cudaStream_t st,
              int k_splits = 1, float* partial = nullptr) {
  CUtensorMap ma, mb;
  int rc;
  if (a_mn)
    rc = encode_2d(&ma, a, M, K, lda, 64, 64, "a");
  else
    rc = encode_2d(&ma, a, K, M, lda, 64, kTileM, "a");
  if (rc != DETATTN_OK) return rc;
  if (b_mn)
    rc = encode_2d(&mb, b, N, K, ldb, 64, 64, "b");
  else
    rc = encode_2d(&mb, b, K, N, ldb, 64, kGemmBN, "b");
  if (rc != DETATTN_OK) return rc;
  GemmArgs g{};
  g.c = c;
  g.M = M;
  g.N = N;
  g.K = K;
  g.ldc = ldc;
  g.alpha = alpha;
  g.wait_ns = g_wait_ns;
  g.k_splits = (k_splits > 1 && partial != nullptr && (K / 64) % k_splits == 0) ? k_splits : 1;
  g.partial = partial;
  if ((rc = launched(launch_gemm(a_mn != 0, b_mn != 0, c_f32 != 0, ma, mb, g, st),
                     "layer_gemm")) != DETATTN_OK)
    return rc;
  if (g.k_splits == 1) return DETATTN_OK;
  int sms = 0;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  return launched(launch_gemm_reduce(g, c_f32 != 0, sms, st), "layer_gemm (split-K sum)");
}

// Workspace of layer_train_step: the step's intermediates, each 256-byte
// aligned.  N3 = (Hq + 2 Hkv) D columns of the joined projection.
struct LayerLayout {
  size_t qkv, q, k, v, o, lse, dout, dq, dk, dv, dqkv, attn, attn_bytes, partial, partial_o, total;
};
// The weight-gradient products (M = d or Hq D, K = B T) have few output
// tiles and a long K: they split K in kWgradSplits blocks, whose fp32
// partials a second kernel adds in a fixed order.
constexpr int kWgradSplits = 4;
LayerLayout layer_layout(int B, int T, int d, int Hq, int Hkv, int D) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t BT = static_cast<size_t>(B) * T;
  const size_t N3 = static_cast<size_t>(Hq + 2 * Hkv) * D;
  LayerLayout l{};
  size_t at = 0;
  l.qkv = at;  at += up(BT * N3 * 2);
  l.q = at;    at += up(BT * Hq * D * 2);
  l.k = at;    at += up(BT * Hkv * D * 2);
  l.v = at;    at += up(BT * Hkv * D * 2);
  l.o = at;    at += up(BT * Hq * D * 2);
  l.lse = at;  at += up(static_cast<size_t>(B) * Hq * T * 4);
  l.dout = at; at += up(BT * Hq * D * 2);
  l.dq = at;   at += up(BT * Hq * D * 2);
  l.dk = at;   at += up(BT * Hkv * D * 2);
  l.dv = at;   at += up(BT * Hkv * D * 2);
  l.dqkv = at; at += up(BT * N3 * 2);
  l.attn_bytes = counter_offset(B, T, Hq) + 256;
  l.attn = at; at += up(l.attn_bytes);
  l.partial = at; at += up(static_cast<size_t>(kWgradSplits) * d * N3 * 4);
  l.partial_o = at; at += up(static_cast<size_t>(kWgradSplits) * Hq * D * d * 4);
  l.total = at;
  return l;
}

// The layer step's second stream: the products that do not wait on the
// attention (dO = dY Wo^T during the forward, the Wo gradient and its AdamW
// update during the attention backward) run there.  Per device and context,
// created on first use; fork and join are events.
struct LayerStreams {
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, dout = nullptr, o = nullptr, y = nullptr, done = nullptr;
  unsigned long long ctx = 0;
};
int layer_streams(LayerStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DETATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 64) return fail(DETATTN_ERR_CUDA, "device index %d too large", dev);
  static LayerStreams per_dev[64];
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  LayerStreams& ls = per_dev[dev];
  const unsigned long long ctx = current_context_id();
  if (ls.side != nullptr && ctx != 0 && ls.ctx != ctx) ls = LayerStreams{};
  if (ls.side == nullptr) {
    e = cudaStreamCreateWithFlags(&ls.side, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&ls.fork, &ls.dout, &ls.o, &ls.y, &ls.done})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      ls = LayerStreams{};
      return fail(DETATTN_ERR_CUDA, "layer side stream: %s", cudaGetErrorString(e));
    }
    ls.ctx = current_context_id();
  }
  *out = &ls;
  return DETATTN_OK;
}

int check_layer(int B, int T, int d, int Hq, int Hkv, int D) {
  bool empty = false;
  int rc;
  if ((rc = check_shape(B, T, Hq, Hkv, D, &empty)) != DETATTN_OK) return rc;
  if (empty) return fail(DETATTN_ERR_SHAPE, "layer step needs B, T >= 1");
  const long BT = static_cast<long>(B) * T;
  if (BT % kTileM || d % kTileM || d % kGemmBN || (Hq * D) % kGemmBN ||
      ((Hq + 2 * Hkv) * D) % kGemmBN)
    return fail(DETATTN_ERR_SHAPE,
                "layer step: B*T=%ld, d=%d, Hq*D=%d and (Hq+2Hkv)*D=%d must be multiples of 128", BT,
                d, Hq * D, (Hq + 2 * Hkv) * D);
  if (BT > (1 << 24) || d > (1 << 16)) return fail(DETATTN_ERR_SHAPE, "layer step too large");
  return DETATTN_OK;
}

// ------------------------------------------------------------ built-in scratch
// Row statistics for attn_bwd_noalloc: a file-scope device array, so callers
// that cannot allocate device memory still get the backward.  Every GPU that
// loads this library holds it (8 MiB) until the process exits.  In host code
// the name is only a host-side stand-in; its device address comes from
// cudaGetSymbolAddress, looked up once per device and context with that
// device current.  The context is part of the key: after a device reset the
// library's module is loaded again and the array may sit elsewhere, and an
// address kept from the old context would send the kernels' stores there.
constexpr size_t kNoallocMaxPairs = size_t(1) << 20;
static __device__ __align__(256) float2 g_noalloc_rowstats[kNoallocMaxPairs];

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DETATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  struct Entry {
    unsigned long long ctx;
    void* ptr;
  };
  static Entry cached[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (dev < 64 && ctx != 0 && cached[dev].ctx == ctx && cached[dev].ptr != nullptr) {
    *out = cached[dev].ptr;
    return DETATTN_OK;
  }
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_noalloc_rowstats);
  if (e != cudaSuccess || ptr == nullptr)
    return fail(DETATTN_ERR_CUDA, "cudaGetSymbolAddress of the built-in scratch: %s",
                cudaGetErrorString(e));
  // The lookup made the device's context current if it was not yet.
  if (dev < 64) cached[dev] = Entry{current_context_id(), ptr};
  *out = ptr;
  return DETATTN_OK;
}

// ------------------------------------------------------------ embedding gradient
// Workspace of embed_grad: counts [V], offsets [V + 1], cursor [V], unsorted
// [N], sorted [N] (int32), then the head and tail partial rows, fp32
// [ceil(N / 32), E] each; every part starts on a 256-byte boundary.
struct EmbedLayout {
  size_t counts, offsets, cursor, unsorted, sorted, head, tail, total;
};
EmbedLayout embed_layout(int N, int V, int E) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  EmbedLayout l{};
  size_t at = 0;
  l.counts = at;   at += up(sizeof(int) * static_cast<size_t>(V));
  l.offsets = at;  at += up(sizeof(int) * (static_cast<size_t>(V) + 1));
  l.cursor = at;   at += up(sizeof(int) * static_cast<size_t>(V));
  l.unsorted = at; at += up(sizeof(int) * static_cast<size_t>(N));
  l.sorted = at;   at += up(sizeof(int) * static_cast<size_t>(N));
  const size_t runs = (static_cast<size_t>(N) + 31) / 32;
  l.head = at;     at += up(sizeof(float) * runs * static_cast<size_t>(E));
  l.tail = at;     at += up(sizeof(float) * runs * static_cast<size_t>(E));
  l.total = at;
  return l;
}

int check_embed_shape(int N, int V, int E) {
  if (N < 0 || N > (1 << 30))
    return fail(DETATTN_ERR_SHAPE, "N=%d tokens: must be in [0, 2^30]", N);
  if (V < 1 || V > (1 << 30)) return fail(DETATTN_ERR_SHAPE, "V=%d rows: must be in [1, 2^30]", V);
  if (E < 4 || E % 4 != 0 || E > (1 << 20))
    return fail(DETATTN_ERR_SHAPE, "E=%d columns: must be a positive multiple of 4 up to 2^20", E);
  if (static_cast<double>(V) * E > 4.0e11 || static_cast<double>(N) * E > 4.0e11)
    return fail(DETATTN_ERR_SHAPE, "embedding problem too large (N=%d V=%d E=%d)", N, V, E);
  return DETATTN_OK;
}

}  // namespace

namespace detattn {

unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", reinterpret_cast<void**>(&get_current),
                                         4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      get_current = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", reinterpret_cast<void**>(&get_id), 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      get_id = nullptr;
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

}  // namespace detattn

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T,
             int Hq, int Hkv, int D, float scale, int causal, void* stream) {
  bool empty = false;
  int rc;
  if ((rc = check_shape(B, T, Hq, Hkv, D, &empty)) != DETATTN_OK) return rc;
  if ((rc = check_scale(scale, causal)) != DETATTN_OK) return rc;
  if (empty) return ok_status();
  if ((rc = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {o, "o"}, {lse, "lse"}})) != DETATTN_OK)
    return rc;
  if ((rc = check_device()) != DETATTN_OK) return rc;
  return fwd_impl(q, k, v, o, lse, B, T, Hq, Hkv, D, scale, causal,
                  static_cast<cudaStream_t>(stream));
}

size_t attn_bwd_workspace_bytes(int B, int T, int Hq, int Hkv, int D) {
  bool empty = false;
  if (check_shape(B, T, Hq, Hkv, D, &empty) != DETATTN_OK || empty) return 0;
  return counter_offset(B, T, Hq) + 256;
}

size_t attn_bwd_ds_workspace_bytes(int B, int T, int Hq, int Hkv, int D, int causal) {
  bool empty = false;
  if (check_shape(B, T, Hq, Hkv, D, &empty) != DETATTN_OK || empty) return 0;
  if (causal != 0 && causal != 1) return 0;
  if (static_cast<double>(B) * Hq * ds_pairs(T, causal) * 2 * kTileN >= 2.0e9) return 0;
  return ds_offset(B, T, Hq) + ds_region_bytes(B, T, Hq, causal);
}

int detattn_set_bwd_dq_mode(int mode) {
  if (mode != 0 && mode != 1) return fail(DETATTN_ERR_SHAPE, "dQ mode %d: must be 0 or 1", mode);
  g_bwd_dq_mode = mode;
  return ok_status();
}

int attn_bwd_delta(const void* o, const void* dout, const float* lse, void* workspace,
                   size_t workspace_bytes, int B, int T, int Hq, int D, void* stream) {
  bool empty = false;
  int rc;
  if ((rc = check_shape(B, T, Hq, 1, D, &empty)) != DETATTN_OK) return rc;
  if (empty) return ok_status();
  if ((rc = check_ptrs({{o, "o"}, {dout, "dout"}, {lse, "lse"}})) != DETATTN_OK) return rc;
  if ((rc = check_workspace(workspace, workspace_bytes, B, T, Hq)) != DETATTN_OK) return rc;
  if ((rc = check_device()) != DETATTN_OK) return rc;
  return delta_impl(o, dout, lse, workspace, B, T, Hq, D,
                    unit_counter_ptr(workspace, workspace_bytes, B, T, Hq),
                    static_cast<cudaStream_t>(stream));
}

int attn_bwd_dkdv(const void* q, const void* k, const void* v, const void* dout,
                  const void* workspace, size_t workspace_bytes, void* dk, void* dv, int B, int T,
                  int Hq, int Hkv, int D, float scale, int causal, void* stream) {
  bool empty = false;
  int rc;
  if ((rc = check_shape(B, T, Hq, Hkv, D, &empty)) != DETATTN_OK) return rc;
  if ((rc = check_scale(scale, causal)) != DETATTN_OK) return rc;
  if (empty) return ok_status();
  if ((rc = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {dout, "dout"}, {dk, "dk"}, {dv, "dv"}})) !=
      DETATTN_OK)
    return rc;
  if ((rc = check_workspace(workspace, workspace_bytes, B, T, Hq)) != DETATTN_OK) return rc;
  if ((rc = check_device()) != DETATTN_OK) return rc;
  return dkdv_impl(q, k, v, dout, workspace, dk, dv, B, T, Hq, Hkv, D, scale, causal,
                   static_cast<cudaStream_t>(stream));
}

int attn_bwd_dq(const void* q, const void* k, const void* v, const void* dout,
                const void* workspace, size_t workspace_bytes, void* dq, int B, int T, int Hq,
                int Hkv, int D, float scale, int causal, void* stream) {
  bool empty = false;
  int rc;
  if ((rc = check_shape(B, T, Hq, Hkv, D, &empty)) != DETATTN_OK) return rc;
  if ((rc = check_scale(scale, causal)) != DETATTN_OK) return rc;
  if (empty) return ok_status();
  if ((rc = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {dout, "dout"}, {dq, "dq"}})) != DETATTN_OK)
    return rc;
  if ((rc = check_workspace(workspace, workspace_bytes, B, T, Hq)) != DETATTN_OK) return rc;
  if ((rc = check_device()) != DETATTN_OK) return rc;
  return dq_impl(q, k, v, dout, workspace, dq, B, T, Hq, Hkv, D, scale, causal,
                 unit_counter_ptr(workspace, workspace_bytes, B, T, Hq),
                 static_cast<cudaStream_t>(stream));
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, void* workspace,
             size_t workspace_bytes, int B, int T, int Hq, int Hkv, int D, float scale,
             int causal, void* stream) {
  bool empty = false;
  int rc;
  if ((rc = check_shape(B, T, Hq, Hkv, D, &empty)) != DETATTN_OK) return rc;
  if ((rc = check_scale(scale, causal)) != DETATTN_OK) return rc;
  if (empty) return ok_status();
  if ((rc = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {o, "o"}, {lse, "lse"}, {dout, "dout"},
                        {dq, "dq"}, {dk, "dk"}, {dv, "dv"}})) != DETATTN_OK)
    return rc;
  if ((rc = check_workspace(workspace, workspace_bytes, B, T, Hq)) != DETATTN_OK) return rc;
  if ((rc = check_device()) != DETATTN_OK) return rc;
  return bwd_steps(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, T, Hq, Hkv, D,
                   scale, causal,
                   static_cast<cudaStream_t>(stream));
}

int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, int B, int T, int Hq,
                     int Hkv, int D, float scale, int causal, void* stream) {
  bool empty = false;
  int rc;
  if ((rc = check_shape(B, T, Hq, Hkv, D, &empty)) != DETATTN_OK) return rc;
  if ((rc = check_scale(scale, causal)) != DETATTN_OK) return rc;
  if (empty) return ok_status();
  const size_t pairs = static_cast<size_t>(B) * Hq * padded_T(T);
  if (pairs > kNoallocMaxPairs)
    return fail(DETATTN_ERR_WORKSPACE,
                "attn_bwd_noalloc: B*Hq*Tp = %zu row-statistic pairs (Tp = T rounded up to 128) "
                "exceeds the built-in scratch of %zu pairs; use attn_bwd with a workspace",
                pairs, kNoallocMaxPairs);
  if ((rc = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {o, "o"}, {lse, "lse"}, {dout, "dout"},
                        {dq, "dq"}, {dk, "dk"}, {dv, "dv"}})) != DETATTN_OK)
    return rc;
  if ((rc = check_device()) != DETATTN_OK) return rc;
  void* ws = nullptr;
  if ((rc = noalloc_scratch(&ws)) != DETATTN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The built-in scratch holds the row statistics only: the dQ step follows
  // the static deal.
  if ((rc = delta_impl(o, dout, lse, ws, B, T, Hq, D, nullptr, st)) != DETATTN_OK) return rc;
  if ((rc = dkdv_impl(q, k, v, dout, ws, dk, dv, B, T, Hq, Hkv, D, scale, causal, st,
                      /*after_delta=*/true)) != DETATTN_OK)
    return rc;
  return dq_impl(q, k, v, dout, ws, dq, B, T, Hq, Hkv, D, scale, causal, nullptr, st);
}

size_t embed_grad_workspace_bytes(int N, int V, int E) {
  if (check_embed_shape(N, V, E) != DETATTN_OK) return 0;
  return embed_layout(N, V, E).total;
}

int embed_grad(const int* ids, const void* dy, float* dw, void* workspace, size_t workspace_bytes,
               int N, int V, int E, void* stream) {
  int rc;
  if ((rc = check_embed_shape(N, V, E)) != DETATTN_OK) return rc;
  if (N > 0 && (rc = check_ptrs({{ids, "ids"}, {dy, "dy"}})) != DETATTN_OK) return rc;
  if ((rc = check_ptrs({{dw, "dw"}, {workspace, "workspace"}})) != DETATTN_OK) return rc;
  const EmbedLayout l = embed_layout(N, V, E);
  if (workspace_bytes < l.total)
    return fail(DETATTN_ERR_WORKSPACE, "embed_grad workspace needs %zu bytes, got %zu", l.total,
                workspace_bytes);
  if ((rc = check_device()) != DETATTN_OK) return rc;
  int sms = 0;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  char* w = static_cast<char*>(workspace);
  EmbedArgs a{};
  a.ids = ids;
  a.dy = dy;
  a.dw = dw;
  a.N = N;
  a.V = V;
  a.E = E;
  a.counts = reinterpret_cast<int*>(w + l.counts);
  a.offsets = reinterpret_cast<int*>(w + l.offsets);
  a.cursor = reinterpret_cast<int*>(w + l.cursor);
  a.unsorted = reinterpret_cast<int*>(w + l.unsorted);
  a.sorted = reinterpret_cast<int*>(w + l.sorted);
  a.head = reinterpret_cast<float*>(w + l.head);
  a.tail = reinterpret_cast<float*>(w + l.tail);
  return launched(launch_embed_grad(a, sms, static_cast<cudaStream_t>(stream)), "embed_grad");
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_q, const int* cu_k, int n_seq, int Hq, int Hkv, int D,
                    float scale, int causal, void* stream) {
  int rc;
  static thread_local Packed pk;
  pk = Packed{};
  if ((rc = check_packed(cu_q, cu_k, n_seq, Hq, Hkv, D, causal, &pk)) != DETATTN_OK) return rc;
  if ((rc = check_scale(scale, causal)) != DETATTN_OK) return rc;
  if (pk.total_q == 0) return ok_status();
  if ((rc = check_ptrs({{q, "q"}, {o, "o"}, {lse, "lse"}})) != DETATTN_OK) return rc;
  if (pk.total_k > 0 && (rc = check_ptrs({{k, "k"}, {v, "v"}})) != DETATTN_OK) return rc;
  if ((rc = check_device()) != DETATTN_OK) return rc;
  return fwd_varlen_impl(q, k, v, o, lse, pk, Hq, Hkv, D, scale, causal,
                         static_cast<cudaStream_t>(stream));
}

size_t attn_bwd_varlen_workspace_bytes(const int* cu_q, const int* cu_k, int n_seq, int Hq,
                                       int Hkv, int D) {
  static thread_local Packed pk;
  pk = Packed{};
  if (check_packed(cu_q, cu_k, n_seq, Hq, Hkv, D, 1, &pk) != DETATTN_OK || pk.total_q == 0)
    return 0;
  return packed_counter_offset(pk, Hq) + 256;
}

int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, void* workspace,
                    size_t workspace_bytes, const int* cu_q, const int* cu_k, int n_seq, int Hq,
                    int Hkv, int D, float scale, int causal, void* stream) {
  int rc;
  static thread_local Packed pk;
  pk = Packed{};
  if ((rc = check_packed(cu_q, cu_k, n_seq, Hq, Hkv, D, causal, &pk)) != DETATTN_OK) return rc;
  if ((rc = check_scale(scale, causal)) != DETATTN_OK) return rc;
  if (pk.total_q == 0 && pk.total_k == 0) return ok_status();
  if (pk.total_q > 0 &&
      (rc = check_ptrs({{q, "q"}, {o, "o"}, {lse, "lse"}, {dout, "dout"}, {dq, "dq"}})) != DETATTN_OK)
    return rc;
  if (pk.total_k > 0 && (rc = check_ptrs({{k, "k"}, {v, "v"}, {dk, "dk"}, {dv, "dv"}})) != DETATTN_OK)
    return rc;
  if (pk.total_q > 0) {
    if (workspace == nullptr || workspace_bytes < packed_rowstat_bytes(pk, Hq))
      return fail(DETATTN_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu%s",
                  packed_rowstat_bytes(pk, Hq), workspace_bytes, workspace ? "" : " (NULL)");
    if (!aligned16(workspace)) return fail(DETATTN_ERR_ALIGN, "workspace is not 16-byte aligned");
  }
  if ((rc = check_device()) != DETATTN_OK) return rc;
  return bwd_varlen_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, pk, Hq, Hkv,
                         D, scale, causal, static_cast<cudaStream_t>(stream));
}

int layer_gemm(const void* a, int a_mn_major, int lda, const void* b, int b_mn_major, int ldb,
               void* c, int c_fp32, int ldc, int M, int N, int K, float alpha, void* stream) {
  int rc;
  if ((rc = check_gemm(a, a_mn_major, lda, b, b_mn_major, ldb, c, c_fp32, ldc, M, N, K)) !=
      DETATTN_OK)
    return rc;
  if (!std::isfinite(alpha)) return fail(DETATTN_ERR_SCALE, "alpha must be finite");
  if ((rc = check_device()) != DETATTN_OK) return rc;
  return gemm_impl(a, a_mn_major, lda, b, b_mn_major, ldb, c, c_fp32, ldc, M, N, K, alpha,
                   static_cast<cudaStream_t>(stream));
}

size_t layer_workspace_bytes(int B, int T, int d, int Hq, int Hkv, int D) {
  if (check_layer(B, T, d, Hq, Hkv, D) != DETATTN_OK) return 0;
  return layer_layout(B, T, d, Hq, Hkv, D).total;
}

int layer_train_step(const void* x, const void* dy, float* w_qkv, float* w_o, float* m_qkv,
                     float* v_qkv, float* m_o, float* v_o, void* w_qkv_bf16, void* w_o_bf16,
                     float* g_qkv, float* g_o, void* y, void* dx, void* workspace,
                     size_t workspace_bytes, int B, int T, int d, int Hq, int Hkv, int D, int step,
                     float lr, float weight_decay, float beta1, float beta2, float eps,
                     void* stream) {
  int rc;
  if ((rc = check_layer(B, T, d, Hq, Hkv, D)) != DETATTN_OK) return rc;
  if ((rc = check_ptrs({{x, "x"}, {dy, "dy"}, {w_qkv, "w_qkv"}, {w_o, "w_o"}, {m_qkv, "m_qkv"},
                        {v_qkv, "v_qkv"}, {m_o, "m_o"}, {v_o, "v_o"}, {w_qkv_bf16, "w_qkv_bf16"},
                        {w_o_bf16, "w_o_bf16"}, {g_qkv, "g_qkv"}, {g_o, "g_o"}, {y, "y"},
                        {workspace, "workspace"}})) != DETATTN_OK)
    return rc;
  if (dx != nullptr && !aligned16(dx)) return fail(DETATTN_ERR_ALIGN, "dx is not 16-byte aligned");
  if (step < 1) return fail(DETATTN_ERR_SHAPE, "step=%d: AdamW steps count from 1", step);
  for (float f : {lr, weight_decay, beta1, beta2, eps})
    if (!std::isfinite(f) || f < 0.f) return fail(DETATTN_ERR_SCALE, "AdamW settings must be finite and >= 0");
  if (!(beta1 < 1.f) || !(beta2 < 1.f)) return fail(DETATTN_ERR_SCALE, "AdamW betas must be < 1");
  const LayerLayout l = layer_layout(B, T, d, Hq, Hkv, D);
  if (workspace_bytes < l.total)
    return fail(DETATTN_ERR_WORKSPACE, "layer workspace needs %zu bytes, got %zu", l.total,
                workspace_bytes);
  if ((rc = check_device()) != DETATTN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  char* w = static_cast<char*>(workspace);
  void *qkv = w + l.qkv, *q = w + l.q, *k = w + l.k, *v = w + l.v, *o = w + l.o, *dout = w + l.dout;
  void *dq = w + l.dq, *dk = w + l.dk, *dv = w + l.dv, *dqkv = w + l.dqkv, *aws = w + l.attn;
  float* lse = reinterpret_cast<float*>(w + l.lse);
  const int BT = B * T, HqD = Hq * D, N3 = (Hq + 2 * Hkv) * D;
  const float scale = 1.0f / std::sqrt(static_cast<float>(D));
  RopeArgs ra{B, T, Hq, Hkv, D, 13.287712379549449f /* log2(10000) */};
  // One enqueue at a time: the side stream and its events are shared by all
  // callers on a device.
  static std::mutex enqueue_mu;
  std::lock_guard<std::mutex> enqueue_lock(enqueue_mu);
  LayerStreams* ls = nullptr;
  if ((rc = layer_streams(&ls)) != DETATTN_OK) return rc;
  cudaStream_t s2 = ls->side;
  auto ev = [&](cudaError_t e, const char* what) {
    return e == cudaSuccess ? DETATTN_OK : fail(DETATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  };
  float* part = reinterpret_cast<float*>(w + l.partial);
  float* part_o = reinterpret_cast<float*>(w + l.partial_o);
  AdamArgs aa{lr, weight_decay, beta1, beta2, eps, step};
  // Fork: the side stream follows everything queued on `stream` so far.
  if ((rc = ev(cudaEventRecord(ls->fork, st), "fork")) != DETATTN_OK) return rc;
  if ((rc = ev(cudaStreamWaitEvent(s2, ls->fork, 0), "fork")) != DETATTN_OK) return rc;
  rc = [&]() -> int {
    int r;
    // Side: dO = dY Wo^T (needs only dY and Wo), during the forward.
    if ((r = gemm_impl(dy, 0, d, w_o_bf16, 0, d, dout, 0, HqD, BT, HqD, d, 1.f, s2)) != DETATTN_OK)
      return r;
    if ((r = ev(cudaEventRecord(ls->dout, s2), "dO event")) != DETATTN_OK) return r;
    // Forward: projection, rotary positions, attention, output projection.
    if ((r = gemm_impl(x, 0, d, w_qkv_bf16, 1, N3, qkv, 0, N3, BT, N3, d, 1.f, st)) != DETATTN_OK)
      return r;
    if ((r = launched(launch_rope_split(qkv, q, k, v, ra, sms, st), "rope")) != DETATTN_OK) return r;
    if ((r = fwd_impl(q, k, v, o, lse, B, T, Hq, Hkv, D, scale, 1, st)) != DETATTN_OK) return r;
    if ((r = ev(cudaEventRecord(ls->o, st), "O event")) != DETATTN_OK) return r;
    if ((r = gemm_impl(o, 0, HqD, w_o_bf16, 1, d, y, 0, d, BT, d, HqD, 1.f, st)) != DETATTN_OK)
      return r;
    if ((r = ev(cudaEventRecord(ls->y, st), "Y event")) != DETATTN_OK) return r;
    // Side: the Wo gradient (needs O and dY), then, once the Y product has
    // read the old bf16 Wo, its AdamW update -- during the attention backward.
    if ((r = ev(cudaStreamWaitEvent(s2, ls->o, 0), "O wait")) != DETATTN_OK) return r;
    if ((r = gemm_impl(o, 1, HqD, dy, 1, d, g_o, 1, d, HqD, d, BT, 1.f, s2, kWgradSplits,
                       part_o)) != DETATTN_OK)
      return r;
    if ((r = ev(cudaStreamWaitEvent(s2, ls->y, 0), "Y wait")) != DETATTN_OK) return r;
    if ((r = launched(launch_adamw(w_o, m_o, v_o, g_o, w_o_bf16, static_cast<long>(HqD) * d, aa,
                                   sms, s2),
                      "adamw")) != DETATTN_OK)
      return r;
    // Backward: attention backward (after dO), rotary transpose, the Wqkv
    // gradient, the input gradient, AdamW on Wqkv.
    if ((r = ev(cudaStreamWaitEvent(st, ls->dout, 0), "dO wait")) != DETATTN_OK) return r;
    if ((r = bwd_steps(q, k, v, o, lse, dout, dq, dk, dv, aws, l.attn_bytes, B, T, Hq, Hkv, D,
                       scale, 1, st)) != DETATTN_OK)
      return r;
    if ((r = launched(launch_rope_merge(dq, dk, dv, dqkv, ra, sms, st), "rope")) != DETATTN_OK)
      return r;
    if ((r = gemm_impl(x, 1, d, dqkv, 1, N3, g_qkv, 1, N3, d, N3, BT, 1.f, st, kWgradSplits,
                       part)) != DETATTN_OK)
      return r;
    if (dx != nullptr &&
        (r = gemm_impl(dqkv, 0, N3, w_qkv_bf16, 0, N3, dx, 0, d, BT, d, N3, 1.f, st)) != DETATTN_OK)
      return r;
    return launched(launch_adamw(w_qkv, m_qkv, v_qkv, g_qkv, w_qkv_bf16,
                                 static_cast<long>(d) * N3, aa, sms, st),
                    "adamw");
  }();
  // Join, on success and on failure alike: later work on `stream` follows the
  // side stream, and a stream capture in progress stays closed over both.
  const int jr = ev(cudaEventRecord(ls->done, s2), "join");
  const int jw = jr == DETATTN_OK ? ev(cudaStreamWaitEvent(st, ls->done, 0), "join") : jr;
  return rc != DETATTN_OK ? rc : jw;
}

int detattn_check_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned f = 0, b = 0, em = 0, ly = 0;
  cudaError_t e = take_fwd_status(st, &f);
  if (e == cudaSuccess) e = take_bwd_status(st, &b);
  if (e == cudaSuccess) e = take_embed_status(st, &em);
  if (e == cudaSuccess) e = take_layer_status(st, &ly);
  unsigned dsf = 0;
  if (e == cudaSuccess) e = take_ds_status(st, &dsf);
  if (dsf) b |= 32u;
  if (e != cudaSuccess) return fail(DETATTN_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (em & 1u)
    return fail(DETATTN_ERR_INDEX,
                "embed_grad found token ids outside [0, V); those tokens were left out of dw");
  if (b & 16u)
    return fail(DETATTN_ERR_WORKSPACE,
                "the dQ step found its tile counter not cleared: run attn_bwd_delta on this "
                "workspace (with the same workspace_bytes) first");
  if (f | b | ly)
    return fail(DETATTN_ERR_DEVICE_TIMEOUT,
                "a kernel gave up on a pipeline wait (fwd flags %u, bwd flags %u, layer flags %u)",
                f, b, ly);
  return ok_status();
}

int detattn_diag_qtile_deal(int D, int B, int T, int Hq, int causal, int sms, int* pipe_of_unit,
                            int n_units) {
  bool empty = false;
  int rc;
  if ((rc = check_shape(B, T, Hq, 1, D, &empty)) != DETATTN_OK) return rc;
  if (causal != 0 && causal != 1) return fail(DETATTN_ERR_SCALE, "causal must be 0 or 1");
  if (sms < 1) return fail(DETATTN_ERR_SHAPE, "sms=%d", sms);
  if (pipe_of_unit == nullptr) return fail(DETATTN_ERR_NULL, "pipe_of_unit is NULL");
  const long units = empty ? 0 : static_cast<long>((T + kTileM - 1) / kTileM) * B * Hq;
  if (n_units != units)
    return fail(DETATTN_ERR_SHAPE, "n_units=%d, the shape has %ld units", n_units, units);
  if (empty) return 0;
  QTileSched sc;
  int grid = 0;
  qtile_schedule(dq_pipes_per_block(D), B, T, Hq, causal, sms, &sc, &grid);
  for (long u = 0; u < units; ++u) pipe_of_unit[u] = -1;
  for (int i = 0; i < sc.n_pipes; ++i) {
    if (sc.n_listed > 0) {
      for (int k = sc.start[i]; k < sc.start[i + 1]; ++k) pipe_of_unit[sc.unit[k]] = i;
    } else {
      const int n = qtile_snake_count(i, static_cast<int>(units), sc.n_pipes);
      for (int k = 0; k < n; ++k) pipe_of_unit[qtile_snake_unit(i, k, sc.n_pipes)] = i;
    }
  }
  return sc.n_pipes;
}

int detattn_diag_dkdv_split(int B, int T, int Hq, int Hkv, int D, int causal,
                            const int* resident, int blocks_per_key_tile, int* c_out,
                            int* ng_out) {
  bool empty = false;
  int rc;
  if ((rc = check_shape(B, T, Hq, Hkv, D, &empty)) != DETATTN_OK) return rc;
  if (causal != 0 && causal != 1) return fail(DETATTN_ERR_SHAPE, "causal=%d must be 0 or 1", causal);
  if (resident == nullptr || c_out == nullptr || ng_out == nullptr)
    return fail(DETATTN_ERR_NULL, "resident, c_out and ng_out must not be NULL");
  if ((rc = check_split(blocks_per_key_tile)) != DETATTN_OK) return rc;
  *c_out = 0;
  *ng_out = 0;
  if (empty) return ok_status();
  if (!dkdv_choose(B, T, Hq, Hkv, D, causal, resident, blocks_per_key_tile, c_out, ng_out))
    return fail(DETATTN_ERR_SHAPE, "no cluster size with resident clusters for D = %d", D);
  return ok_status();
}

int detattn_diag_exp2(const float* x, float* y_poly, float* y_pair, float* y_sfu, int n,
                      void* stream) {
  int rc;
  if (n < 0) return fail(DETATTN_ERR_SHAPE, "n=%d", n);
  if (n == 0) return ok_status();
  if ((rc = check_ptrs({{x, "x"}, {y_poly, "y_poly"}, {y_pair, "y_pair"}, {y_sfu, "y_sfu"}})) !=
      DETATTN_OK)
    return rc;
  if ((rc = check_device()) != DETATTN_OK) return rc;
  return launched(launch_exp2_diag(x, y_poly, y_pair, y_sfu, n, static_cast<cudaStream_t>(stream)),
                  "detattn_diag_exp2");
}

int detattn_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
  int rc;
  if ((rc = check_device()) != DETATTN_OK) return rc;
  if (limit_ns < 1000000ull) limit_ns = 1000000ull;
  if (limit_ns > 10000000000ull) limit_ns = 10000000000ull;
  return launched(launch_wait_timeout_selftest(limit_ns, static_cast<cudaStream_t>(stream)),
                  "detattn_selftest_wait_timeout");
}

int detattn_diag_dkdv_list(int B, int T, int Hq, int Hkv, int causal, int c, int ng, int force,
                           int* start, int* entry, int max_entries) {
  bool empty = false;
  int rc;
  if ((rc = check_shape(B, T, Hq, Hkv, 64, &empty)) != DETATTN_OK) return rc;
  if (causal != 0 && causal != 1) return fail(DETATTN_ERR_SHAPE, "causal=%d must be 0 or 1", causal);
  if (force != 0 && force != 1) return fail(DETATTN_ERR_SHAPE, "force=%d must be 0 or 1", force);
  if (c < 2 || c > dkdv_max_cluster_size(64) || (c & (c - 1)) != 0 || ng < 1)
    return fail(DETATTN_ERR_SHAPE, "c=%d, ng=%d", c, ng);
  if (start == nullptr || entry == nullptr) return fail(DETATTN_ERR_NULL, "start and entry must not be NULL");
  if (empty) return ok_status();
  std::unique_ptr<DkvList> list(new DkvList());
  const int G = Hq / Hkv, BH = B * Hkv, tm = dkdv_tile_m(64);
  const int n_tiles = (T + kTileN - 1) / kTileN, m_end = (T + tm - 1) / tm;
  std::vector<int> items(static_cast<size_t>(n_tiles) * BH);
  for (size_t t = 0; t < items.size(); ++t)
    items[t] = G * (m_end - (causal ? static_cast<int>(t) / BH * kTileN / tm : 0));
  if (!dkdv_mixed_list(items, c, ng, force == 1, list.get())) {
    ok_status();
    return 0;
  }
  const int n = list->start[list->n_blocks];
  if (n > max_entries) return fail(DETATTN_ERR_SHAPE, "the list holds %d entries, max_entries=%d", n, max_entries);
  for (int i = 0; i <= list->n_blocks; ++i) start[i] = list->start[i];
  for (int i = 0; i < n; ++i) entry[i] = list->entry[i];
  ok_status();
  return n;
}

int detattn_set_dkdv_deal(int mode) {
  if (mode < 0 || mode > 2) return fail(DETATTN_ERR_SHAPE, "dkdv deal mode %d (0, 1 or 2)", mode);
  g_dkdv_deal = mode;
  return ok_status();
}

int detattn_set_dkdv_split(int blocks_per_key_tile) {
  int rc;
  if ((rc = check_split(blocks_per_key_tile)) != DETATTN_OK) return rc;
  g_dkdv_split = blocks_per_key_tile;
  return ok_status();
}

void detattn_set_wait_limit_ns(unsigned long long ns) {
  if (ns < 1000000ull) ns = 1000000ull;
  if (ns > 60000000000ull) ns = 60000000000ull;
  g_wait_ns = ns;
}

const char* detattn_last_error(void) { return g_err; }

int detattn_version(void) { return kVersion; }

}  // extern "C"

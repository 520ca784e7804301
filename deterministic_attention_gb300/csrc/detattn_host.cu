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
#include <mutex>
#include <vector>

#include "../../include/detattn.h"
#include "attn_launch.h"

using namespace detattn;

namespace {

constexpr int kVersion = 10000;  // 1.0.0
thread_local char g_err[512] = "";
unsigned long long g_wait_ns = 1000000000ull;  // 1 s per bounded wait
int g_dkdv_split = 0;                           // 0: automatic

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
void qtile_schedule(int D, int B, int T, int Hq, int causal, int sms, QTileSched* out, int* grid) {
  const int NP = qtile_pipes_per_block(D);
  const int n_m = (T + kTileM - 1) / kTileM;
  const int BHq = B * Hq;
  const long units = static_cast<long>(n_m) * BHq;
  const int kv_tiles = (T + kFwdTileN - 1) / kFwdTileN;
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
    const int mt = n_m - 1 - static_cast<int>(u / BHq);
    const int n_kv = causal ? std::min(kv_tiles, (mt * kTileM + kTileM) / kFwdTileN) : kv_tiles;
    const double w = n_kv + 2.0;
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

// The schedule depends only on (D, B, T, Hq, causal, SMs): the last one is
// kept (the forward and dQ of one layer share it).
void cached_qtile_schedule(int D, int B, int T, int Hq, int causal, int sms, QTileSched* out,
                           int* grid) {
  static std::mutex mu;
  static int key[6] = {-1, -1, -1, -1, -1, -1};
  static QTileSched sched;
  static int g = 0;
  std::lock_guard<std::mutex> lock(mu);
  const int want[6] = {D, B, T, Hq, causal, sms};
  if (!std::equal(want, want + 6, key)) {
    qtile_schedule(D, B, T, Hq, causal, sms, &sched, &g);
    std::copy(want, want + 6, key);
  }
  *out = sched;
  *grid = g;
}

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T,
             int Hq, int Hkv, int D, float scale, int causal, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  int rc;
  if ((rc = encode_rows(&mq, q, B, T, Hq, D, kTileM, "q")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mk, k, B, T, Hkv, D, kFwdTileN, "k")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mv, v, B, T, Hkv, D, kFwdTileN, "v")) != DETATTN_OK) return rc;
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
  cached_qtile_schedule(D, B, T, Hq, causal, sms, &sc, &g);
  return launched(launch_fwd(D, g, mq, mk, mv, a, sc, st), "attn_fwd");
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
  return launched(launch_delta(a, sms, st), "attn_bwd_delta");
}

BwdArgs bwd_args(const void* workspace, int T, int Hq, int Hkv, float scale, int causal) {
  BwdArgs a{};
  a.rowstats = static_cast<const float2*>(workspace);
  a.T = T;
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
bool dkdv_choose(int B, int T, int Hq, int Hkv, int D, int causal, const int resident[4],
                 int forced_c, int* c_out, int* ng_out) {
  const int G = Hq / Hkv;
  const int n_tiles = (T + kTileN - 1) / kTileN;
  const int BH = B * Hkv;
  const int tm = dkdv_tile_m(D);
  const int m_end = (T + tm - 1) / tm;
  const long total = static_cast<long>(n_tiles) * BH;
  const int cmax = dkdv_max_cluster_size(D);
  double best = 0.0;
  *c_out = 0;
  *ng_out = 0;
  for (int c = 1, i = 0; c <= cmax && i < 4; c *= 2, ++i) {
    if (forced_c > 0 && c != (forced_c < cmax ? forced_c : cmax)) continue;
    if (resident[i] < 1) continue;
    const long ng = total < resident[i] ? total : resident[i];
    double worst = 0.0;
    for (long k = 0; k < ng; ++k) {
      double load = 0.0;
      for (long kt = 0;; ++kt) {
        const long t = kt * ng + ((kt & 1) ? ng - 1 - k : k);
        if (t >= total) break;
        const int nt = static_cast<int>(t / BH);
        const int items = G * (m_end - (causal ? nt * kTileN / tm : 0));
        // Per tile: its share of the items, one item's worth for writing the
        // sums out, and two per peer for the partial-sum exchange (measured:
        // distributed shared memory moves ~9 bytes per clock per SM, and an
        // item takes ~1,500 clocks).
        load += (items + c - 1) / c + 1.0 + 2.0 * (c - 1);
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

int dkdv_impl(const void* q, const void* k, const void* v, const void* dout,
              const void* workspace, void* dk, void* dv, int B, int T, int Hq, int Hkv, int D,
              float scale, int causal, cudaStream_t st, bool after_delta = false) {
  CUtensorMap mq, mk, mv, mdo;
  int rc;
  if ((rc = encode_rows(&mq, q, B, T, Hq, D, dkdv_tile_m(D), "q")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mdo, dout, B, T, Hq, D, dkdv_tile_m(D), "dout")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mk, k, B, T, Hkv, D, kTileN, "k")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mv, v, B, T, Hkv, D, kTileN, "v")) != DETATTN_OK) return rc;
  BwdArgs a = bwd_args(workspace, T, Hq, Hkv, scale, causal);
  a.dk = dk;
  a.dv = dv;
  a.n_tiles = (T + kTileN - 1) / kTileN;
  a.BH = B * Hkv;
  int sms = 0;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  if ((rc = dkdv_schedule(B, T, Hq, Hkv, D, causal, sms, g_dkdv_split, &a.cluster, &a.n_groups)) !=
      DETATTN_OK)
    return rc;
  return launched(launch_dkdv(D, a.n_groups * a.cluster, mq, mk, mv, mdo, a, after_delta, st),
                  "attn_bwd_dkdv");
}

int dq_impl(const void* q, const void* k, const void* v, const void* dout, const void* workspace,
            void* dq, int B, int T, int Hq, int Hkv, int D, float scale, int causal,
            unsigned* counter, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mdo;
  int rc;
  if ((rc = encode_rows(&mq, q, B, T, Hq, D, kTileM, "q")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mdo, dout, B, T, Hq, D, kTileM, "dout")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mk, k, B, T, Hkv, D, kDqTileN, "k")) != DETATTN_OK) return rc;
  if ((rc = encode_rows(&mv, v, B, T, Hkv, D, kDqTileN, "v")) != DETATTN_OK) return rc;
  BwdArgs a = bwd_args(workspace, T, Hq, Hkv, scale, causal);
  a.dq = dq;
  a.n_tiles = (T + kTileM - 1) / kTileM;
  a.BH = B * Hq;
  a.unit_counter = counter;
  int sms = 0;
  if ((rc = sm_count(&sms)) != DETATTN_OK) return rc;
  static_assert(kDqTileN == kFwdTileN, "the forward's schedule weights fit dQ");
  QTileSched sc;
  int g;
  cached_qtile_schedule(D, B, T, Hq, causal, sms, &sc, &g);
  return launched(launch_dq(D, g, mq, mk, mv, mdo, a, sc, st), "attn_bwd_dq");
}

int check_workspace(const void* ws, size_t bytes, int B, int T, int Hq) {
  if (ws == nullptr || bytes < rowstat_bytes(B, T, Hq))
    return fail(DETATTN_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu%s",
                rowstat_bytes(B, T, Hq), bytes, ws ? "" : " (NULL)");
  if (!aligned16(ws)) return fail(DETATTN_ERR_ALIGN, "workspace is not 16-byte aligned");
  return DETATTN_OK;
}

// ------------------------------------------------------------ side stream
// attn_bwd runs dK/dV and dQ, which both need only the Delta step's output,
// on two streams: dQ on a per-device side stream forked from the caller's
// stream after Delta and joined back before attn_bwd returns.  The two grids
// then fill each other's idle SMs.  Stream capture records the fork and join
// as graph edges.  The side stream and events are created on first use.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  unsigned long long ctx = 0;  // id of the context the handles belong to
};

int side_stream(SideStream** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DETATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  static SideStream per_dev[64];
  static std::mutex mu;
  if (dev >= 64) return fail(DETATTN_ERR_CUDA, "device index %d too large", dev);
  std::lock_guard<std::mutex> lock(mu);
  SideStream& ss = per_dev[dev];
  // Handles of a context that has since been destroyed (device reset) are
  // dropped, not destroyed: they went with it.
  const unsigned long long ctx = current_context_id();
  if (ss.stream != nullptr && ctx != 0 && ss.ctx != ctx) ss = SideStream{};
  if (ss.stream == nullptr) {
    e = cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      ss = SideStream{};
      return fail(DETATTN_ERR_CUDA, "side stream: %s", cudaGetErrorString(e));
    }
    ss.ctx = current_context_id();
  }
  *out = &ss;
  return DETATTN_OK;
}

// Delta, then dK/dV on `st` and dQ on the side stream.
int bwd_steps(const void* q, const void* k, const void* v, const void* o, const float* lse,
              const void* dout, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, int B,
              int T, int Hq, int Hkv, int D, float scale, int causal, cudaStream_t st) {
  int rc;
  unsigned* counter = unit_counter_ptr(ws, ws_bytes, B, T, Hq);
  if ((rc = delta_impl(o, dout, lse, ws, B, T, Hq, D, counter, st)) != DETATTN_OK) return rc;
  SideStream* ss = nullptr;
  if ((rc = side_stream(&ss)) != DETATTN_OK) return rc;
  cudaError_t e = cudaEventRecord(ss->fork, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->stream, ss->fork, 0);
  if (e != cudaSuccess) return fail(DETATTN_ERR_CUDA, "fork: %s", cudaGetErrorString(e));
  if ((rc = dq_impl(q, k, v, dout, ws, dq, B, T, Hq, Hkv, D, scale, causal, counter,
                    ss->stream)) !=
      DETATTN_OK)
    return rc;
  // dK/dV follows the Delta step directly in `st`: its prologue and
  // operand loads overlap that step (it waits only for the row statistics).
  if ((rc = dkdv_impl(q, k, v, dout, ws, dk, dv, B, T, Hq, Hkv, D, scale, causal, st,
                      /*after_delta=*/true)) != DETATTN_OK)
    return rc;
  e = cudaEventRecord(ss->join, ss->stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ss->join, 0);
  if (e != cudaSuccess) return fail(DETATTN_ERR_CUDA, "join: %s", cudaGetErrorString(e));
  return ok_status();
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

int detattn_check_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned f = 0, b = 0;
  cudaError_t e = take_fwd_status(st, &f);
  if (e == cudaSuccess) e = take_bwd_status(st, &b);
  if (e != cudaSuccess) return fail(DETATTN_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (b & 16u)
    return fail(DETATTN_ERR_WORKSPACE,
                "the dQ step found its tile counter not cleared: run attn_bwd_delta on this "
                "workspace (with the same workspace_bytes) first");
  if (f | b)
    return fail(DETATTN_ERR_DEVICE_TIMEOUT,
                "a kernel gave up on a pipeline wait (fwd flags %u, bwd flags %u)", f, b);
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
  qtile_schedule(D, B, T, Hq, causal, sms, &sc, &grid);
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

// Deterministic flash-attention backward for sm_103a: Delta preprocess,
// dK/dV kernel and dQ kernel.
//
// RustingBrain vs PyTorch/TensorFlow page, "Step 2: fused flash attention"
// (the backward is fused too) and "Where the time goes now" (the dK/dV kernel
// flash_attention_dkv recomputes the probabilities and dominates the
// backward).  oxide-train README, "The trainer is not bit-identical to itself
// after step 1": gradients summed with atomics change from run to run.  Here
// every output element is written once, by the one block that owns its tile,
// after a reduction whose order is fixed:
//   * Delta_i = sum_d dO_id O_id       one warp per 32 rows, fixed shuffle tree
//   * dK_j, dV_j                       one block per (b, KV head, 128-key tile);
//                                      query heads of the group in ascending
//                                      order, query tiles ascending, all summed
//                                      in the block's TMEM accumulators
//   * dQ_i                             one block per (b, query head, 128-query
//                                      tile); key tiles ascending
// The probabilities are recomputed from LSE: P = exp2(S * scale * log2e -
// LSE * log2e), dS = P * (dP - Delta).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <type_traits>
#include <utility>

#include "attn_launch.h"
#include "exp2_poly.cuh"
#include "sm103_ptx.cuh"

namespace detattn {

__device__ unsigned int g_bwd_status;

namespace {

constexpr float kLog2e = 1.4426950408889634f;
// Of every 8 consecutive pairs of probabilities, this many take 2^x from the
// FMA-pipe polynomial instead of the special-function unit.
#ifndef DETATTN_BWD_POLY_OF8
#define DETATTN_BWD_POLY_OF8 0
#endif
constexpr int kPolyOf8 = DETATTN_BWD_POLY_OF8;

__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

// f(std::integral_constant<int, i>{}) for i = 0 .. N-1, unrolled at compile
// time (so i can be a template argument inside f).
template <typename F, int... I>
__device__ __forceinline__ void static_for_impl(F&& f, std::integer_sequence<int, I...>) {
  (f(std::integral_constant<int, I>{}), ...);
}
template <int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  static_for_impl(f, std::make_integer_sequence<int, N>{});
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// ============================================================== Delta
// Rows (b, t, h) in memory order, so a run of rows is one contiguous stretch
// of O and of dO (whole DRAM pages, where one head's rows alone lie
// Hq * D * 2 bytes apart).  Each row of D bf16 is split in 16-byte chunks over
// D/8 lanes, so one warp-wide load covers kRpi = 256 / D rows; a warp takes
// batches of kBatch such loads (kBatch * kRpi contiguous rows, 2 KB of O and
// 2 KB of dO per load step), batch index striding by the number of warps in
// the grid, and issues all of a batch's loads before it uses any.  The grid
// holds four blocks per SM, so every SM keeps about 128 KB of loads in flight
// through the whole pass.  A lane forms its 8 products per chunk in order and
// the lanes of a row are combined by a fixed xor-shuffle tree; the first lane
// of a row reads that row's LSE and stores its (-LSE*log2e, -Delta) pair.
// The padding positions T..Tp-1 of every (b, h) get (-inf, -0).
constexpr int kDeltaBlocksPerSm = 4;
// Packed batches (VL): B = 1 and T = total_q; the row statistics of query
// row t of sequence s go to position ps[s] + t - cu_q[s] (sequence found by a
// binary search of cu_q), and each sequence's padding positions up to the
// next multiple of 128 get (-inf, -0).  Rows whose LSE is -inf (packed rows
// that see no key) store -inf, so every P formed from them is 0.
__device__ __forceinline__ int seq_of_row(const VarlenTable& vt, int t) {
  int lo = 0, hi = vt.n_seq - 1;
  while (lo < hi) {  // last s with cu_q[s] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (vt.cu_q[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int D, class VT>
__global__ void __launch_bounds__(256, kDeltaBlocksPerSm) attn_delta_kernel(const DeltaArgs a,
                                                                             const __grid_constant__ VT vt) {
  constexpr bool VL = std::is_same<VT, VarlenTable>::value;
  constexpr int kCpr = D / 8;          // 16-byte chunks per row
  constexpr int kRpi = 32 / kCpr;      // rows per warp-wide load
  constexpr int kBatch = 4;            // loads per operand per batch
  constexpr int kRows = kBatch * kRpi; // rows per batch
  const int lane = threadIdx.x & 31;
  const long n_warps = static_cast<long>(gridDim.x) * (blockDim.x / 32);
  const long gw = static_cast<long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const long rows = static_cast<long>(a.B) * a.T * a.Hq;
  const long n_batches = (rows + kRows - 1) / kRows;
  const uint4* O = static_cast<const uint4*>(a.o);
  const uint4* dO = static_cast<const uint4*>(a.dout);
  // This warp's first batch of dO into L2 while the kernel before this one
  // (the forward, in a training step) may still run; the loads below come
  // after the wait, so they see the final values either way.
  if (lane == 0 && gw < n_batches) {
    const long r0 = gw * kRows;
    const long nr = rows - r0 < kRows ? rows - r0 : kRows;
    bulk_prefetch_l2(dO + r0 * kCpr, static_cast<uint32_t>(nr * kCpr * 16));
  }
  // Launched as a dependent of whatever precedes it (the forward, in a
  // training step): everything below reads that kernel's output.  Only after
  // this wait may the next kernel (the dK/dV step) start its own prologue.
  griddep_wait();
  griddep_launch_dependents();
  // The dQ step's unit counter (two words) starts each backward at zero.
  if (a.unit_counter != nullptr && blockIdx.x == 0 && threadIdx.x < 2) a.unit_counter[threadIdx.x] = 0u;
  for (long bi = gw; bi < n_batches; bi += n_warps) {
    // (b, t, h) of this lane's row in load step 0, advanced by kRpi rows per
    // step.
    const long r_lane = bi * kRows + lane / kCpr;
    int h = static_cast<int>(r_lane % a.Hq);
    const long bt0 = r_lane / a.Hq;
    int b = static_cast<int>(bt0 / a.T), t = static_cast<int>(bt0 % a.T);
    uint4 xo[kBatch], xd[kBatch];
    float lse[kBatch];
    size_t dst[kBatch];
#pragma unroll
    for (int it = 0; it < kBatch; ++it) {
      const long r = r_lane + it * kRpi;
      xo[it] = make_uint4(0u, 0u, 0u, 0u);
      xd[it] = xo[it];
      lse[it] = 0.f;
      dst[it] = 0;
      if (r < rows) {
        const size_t off = static_cast<size_t>(r) * kCpr + lane % kCpr;
        xo[it] = O[off];
        xd[it] = dO[off];
        const size_t bh = static_cast<size_t>(b) * a.Hq + h;
        if (lane % kCpr == 0) lse[it] = a.lse[bh * a.T + t];
        if constexpr (VL) {
          if (lane % kCpr == 0) {
            const int sq = seq_of_row(vt, t);
            dst[it] = bh * a.Tp + vt.ps[sq] + (t - vt.cu_q[sq]);
          }
        } else {
          dst[it] = bh * a.Tp + t;
        }
      }
      h += kRpi;
      while (h >= a.Hq) {
        h -= a.Hq;
        if (++t == a.T) {
          t = 0;
          ++b;
        }
      }
    }
#pragma unroll
    for (int it = 0; it < kBatch; ++it) {
      const uint32_t xs[4] = {xo[it].x, xo[it].y, xo[it].z, xo[it].w};
      const uint32_t ys[4] = {xd[it].x, xd[it].y, xd[it].z, xd[it].w};
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 xf = bf16x2_to_float2(xs[k]), yf = bf16x2_to_float2(ys[k]);
        acc = fmaf(xf.x, yf.x, acc);
        acc = fmaf(xf.y, yf.y, acc);
      }
#pragma unroll
      for (int s2 = kCpr / 2; s2 >= 1; s2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s2);
      const long r = r_lane + it * kRpi;
      if (lane % kCpr == 0 && r < rows)
        a.rowstats[dst[it]] = make_float2(lse[it] > -INFINITY ? -lse[it] * kLog2e : -INFINITY, -acc);
    }
  }
  if constexpr (VL) {
    // Padding positions: for every (h, s), [ps[s] + tq_s, ps[s + 1]).  Each
    // thread walks position slots of the whole padded row and writes those
    // that no query row of their sequence fills.
    const long n_all = static_cast<long>(a.Hq) * a.Tp;
    for (long p = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; p < n_all;
         p += static_cast<long>(gridDim.x) * blockDim.x) {
      const int pos = static_cast<int>(p % a.Tp);
      int lo = 0, hi = vt.n_seq - 1;  // last s with ps[s] <= pos
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (vt.ps[mid] <= pos) lo = mid; else hi = mid - 1;
      }
      if (pos - vt.ps[lo] >= vt.cu_q[lo + 1] - vt.cu_q[lo]) a.rowstats[p] = make_float2(-INFINITY, -0.f);
    }
  } else {
    // Padding positions: (b, h, t) for t in [T, Tp).
    const int pad = a.Tp - a.T;
    const long n_pad = static_cast<long>(a.B) * a.Hq * pad;
    for (long p = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; p < n_pad;
         p += static_cast<long>(gridDim.x) * blockDim.x) {
      const long bh = p / pad;
      const int t = a.T + static_cast<int>(p % pad);
      a.rowstats[bh * a.Tp + t] = make_float2(-INFINITY, -0.f);
    }
  }
}

// ============================================================== dK / dV
// This kernel (64-query items) runs at D = 128 when a key tile is split over
// a cluster of two blocks, and for the stored-dS form at D = 128; every other
// dK/dV launch runs attn_dkdvq_kernel below.  (Its D = 64 configuration, with
// K and V copied into TMEM, is no longer instantiated.)
// Persistent: the grid is n_groups clusters of C blocks, all resident.  Key
// tiles (b, KV head, 128 keys), heaviest first under the causal mask, are
// dealt to the clusters in snake order (round r: tiles r*NG .. r*NG + NG - 1,
// reversed in odd rounds), and a cluster's C blocks split each of its tiles:
// the tile's items -- one per (query head of the group, query tile of TM rows
// at or after the key tile) -- are cut into C contiguous chunks, and block r
// sums chunk r.  The split and the deal
// depend only on the shape and the SM count, so every output bit is fixed for
// a given problem and GPU.
//   warp 0     loads each tile's K, V (once the previous tile's S^T MMAs are
//              done with them), then each item's Q, dO tiles and row
//              statistics into a ring of shared-memory stages;
//   warp 1     issues S^T = K Q^T and dP^T = V dO^T into one TMEM buffer, as
//              soon as the element-wise warps hold the previous item's in
//              registers;
//   warps 2-17 turn S^T, dP^T into P^T, dS^T (four threads per key row, TM/4
//              queries each) and store them, as packed bf16, into a separate
//              TMEM buffer; after a tile's last item they read its dV, dK
//              accumulators and write them out;
//   warp 18    issues dV += P^T dO and dK += dS^T Q from that buffer.
// With the two MMA streams in separate warps and S^T, dP^T released early, the
// next item's scores are computed while the element-wise warps still work on
// this one: each issuing warp shares its scheduler with four busy
// element-wise warps, and any step that waits behind another lands on the
// critical path.  Tiles follow one another without a break in the pipeline:
// the next tile's loads and S^T MMAs start while this one's accumulators are
// being written out.
//
// Cluster partial sums (C > 1): block p owns key rows [p R, (p + 1) R) of
// the tile, R = 128 / C.  Each block sends the partial sums of rows other
// blocks own with asynchronous 16-byte stores into the owner's receive
// region (slot j = sender rank, minus one above the owner), completing on the
// owner's receive mbarrier; the owner adds the C partial sums in rank order
// (its own from registers) and stores bf16 dV, dK (dK * scale).  Before a
// sender reuses a receive region for the next tile it waits until the owner
// has read it (each owner warp arrives, remotely, on the senders' "region
// free" mbarrier).
constexpr int kBwdThreads = 608;  // producer, S issuer, 16 compute warps, dV/dK issuer
constexpr int kComputeWarps = 16;
constexpr int kDkvAccWarp = 2 + kComputeWarps;

template <int D>
struct DkvCfg {
  static constexpr int kTM = dkdv_tile_m(D);   // query rows per item
  static constexpr int kQG = kTM / 4;          // queries per element-wise thread
  static constexpr int kAtoms = D / 64;
  static constexpr int kKvBytes = kTileN * 128 * kAtoms;  // 128 keys x D
  static constexpr int kQBytes = kTM * 128 * kAtoms;      // TM queries x D
  static constexpr int kStages = (D == 64) ? 6 : 2;
  static constexpr int kStageBytes = 2 * kQBytes + 1024;  // Q, dO, then TM row statistics
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kKvBytes;
  static constexpr int kOffStage = 2 * kKvBytes;
  // Receive region for cluster partial sums: (C - 1) R rows of [dV | dK] fp32.
  static constexpr int kMaxCluster = (D == 64) ? 8 : 2;
  static constexpr int kRowBytes = 2 * D * 4;
  static constexpr int kOffRecv = kOffStage + kStages * kStageBytes;
  static constexpr int kRecvBytes = (kTileN - kTileN / kMaxCluster) * kRowBytes;
  static constexpr int kSmemBytes = kOffRecv + kRecvBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;
  // S^T and dP^T of item gi (TM fp32 columns each, one per query) go to score
  // buffer gi % kNumSB: S^T at 2 TM b, dP^T at 2 TM b + TM.  With two buffers
  // the issuer computes the next item's scores while the element-wise warps
  // work on this one.  P^T and dS^T of item gi go to buffer gi % kNumPB at
  // kColPB + TM * buffer: P^T as packed bf16 pairs over TM/2 columns (two
  // queries per column), dS^T over the next TM/2; group g writes columns
  // g*TM/8 .. of each.  At D = 64 the tile's K and V also live in TMEM as
  // packed bf16 pairs (the A operands of S^T and dP^T, which then run with
  // only Q / dO read from shared memory).
  static constexpr int kNumSB = (D == 64) ? 2 : 1;
  static constexpr int kNumPB = (D == 64) ? 1 : 2;
  static constexpr bool kKvInTmem = (D == 64);
  static constexpr uint32_t kColPB = kNumSB * 2 * kTM;
  static constexpr uint32_t kColDV = kColPB + kNumPB * kTM;  // dV accumulator, D cols
  static constexpr uint32_t kColDK = kColDV + D;             // dK accumulator, D cols
  static constexpr uint32_t kColK = kColDK + D;              // K (D = 64), D/2 columns
  static constexpr uint32_t kColV = kColK + D / 2;           // V (D = 64), D/2 columns
  static_assert(kColDK + D + (kKvInTmem ? D : 0) <= kTmemCols, "TMEM layout");
  static_assert(kTM * 8 <= 1024, "row statistics fit their stage slot");
  static_assert(kSmemBytes + 512 <= 227 * 1024, "shared memory per block (with the static part)");
};

constexpr int kDkvMaxStages = 6;
enum : int {
  kDkvBarKV = 0,                             // this tile's K, V landed
  kDkvBarKVFree = 1,                         // the previous tile's S^T MMAs are done with K, V
  kDkvBarKvTmem = 2,                         // this tile's K, V copied into TMEM (D = 64)
  kDkvBarQFull = 3,
  kDkvBarQEmpty = kDkvBarQFull + kDkvMaxStages,
  kDkvBarS = kDkvBarQEmpty + kDkvMaxStages,  // [2] S^T, dP^T of the buffer's item landed
  kDkvBarSFree = kDkvBarS + 2,               // [2] element-wise warps hold them in registers
  kDkvBarP = kDkvBarSFree + 2,               // [2] P^T, dS^T of the buffer's item written
  kDkvBarFree = kDkvBarP + 2,                // [2] dV, dK of the buffer's item done
  kDkvBarAcc = kDkvBarFree + 2,              // this tile's dV, dK complete
  kDkvBarAccFree = kDkvBarAcc + 1,           // element-wise warps hold them in registers
  kDkvBarDrain = kDkvBarAccFree + 1,
  kDkvBarDrainAcc = kDkvBarDrain + 1,
  kDkvBarRecv = kDkvBarDrainAcc + 1,         // the peers' partial sums of this tile landed
  kDkvBarRegionFree = kDkvBarRecv + 1,       // every peer has read this block's previous sums
  kDkvBarRecvRead = kDkvBarRegionFree + 1,   // (D = 64) this block has read the peers' sums
  kDkvBarKV2 = kDkvBarRecvRead + 1,          // (D = 64) K, V landed in the second buffer
  kDkvBarKVFree2 = kDkvBarKV2 + 1,           // (D = 64) the second buffer's S^T MMAs are done
  kDkvNumBars = kDkvBarKVFree2 + 1
};

// TMEM columns [taddr, taddr + N) of this warp's 32 lanes into v (N = 16, 32).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 16) tmem_ld16_nowait(taddr, v);
  else tmem_ld32_nowait(taddr, v);
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[N]) {
  static_assert(N == 8 || N == 16, "8 or 16 columns");
  if constexpr (N == 8) tmem_st8_nowait(taddr, v);
  else tmem_st16_nowait(taddr, v);
}
template <int N>
__device__ __forceinline__ void reg_fence_cols(uint32_t (&v)[N]) {
  if constexpr (N == 16) reg_fence16(v);
  else reg_fence32(v);
}

// One key tile of the dK/dV work, as one block of its cluster sees it.
// Rows are relative to the tile's sequence: its keys start at row kbase of
// the K, V maps, its queries at qbase of the Q, dO maps, and their row
// statistics at rbase of each head's row; query i sees key j iff
// j <= i + off under the causal mask (off = 0, bases 0 unless packed).
struct DkvTile {
  int b, g, n0;
  int m_begin, per_head;  // first query tile, query tiles per head
  int it_lo, n_it;        // this block's chunk of the tile's G * per_head items
  int qbase, kbase, rbase, tk, off;
};

// MODE bit 0: the chunked tile walk (BwdArgs::bg_chunk); bit 1: store every
// item's dS^T (BwdArgs::ds).  Separate instantiations keep the plain walk
// free of both (each measured to cost about a microsecond at page3 as a
// run-time branch).
constexpr int kDkvChunked = 1, kDkvStoreDs = 2;
template <int D, class VT, int MODE>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_dkdv_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                     const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mdO,
                     const BwdArgs a, const __grid_constant__ VT vt) {
  using Cf = DkvCfg<D>;
  constexpr bool VL = std::is_same<VT, VarlenTable>::value;
  static_assert(!VL || MODE == 0, "the packed form walks its own table");
  constexpr int NS = Cf::kStages;
  constexpr int TM = Cf::kTM;
  constexpr int QG = Cf::kQG;
  constexpr int NPB = Cf::kNumPB;
  constexpr int NSB = Cf::kNumSB;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kDkvNumBars];
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.cluster;
  const int crank = C > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int group = static_cast<int>(blockIdx.x) / C;
  const int NG = a.n_groups;
  const int n_tiles_all = (VL ? vt_tiles(vt) : a.n_tiles) * a.BH;
  const int G = a.Hq / a.Hkv;
  const int m_end = (a.T + TM - 1) / TM;
  const int R = kTileN / C;
  // Tile of this cluster's kt-th turn, or -1 past its last.
  auto tile_of = [&](int kt) {
    const int t = kt * NG + ((kt & 1) ? NG - 1 - group : group);
    return t < n_tiles_all ? t : -1;
  };
  auto tile_info = [&](int t) {
    DkvTile ti;
    if constexpr (VL) {
      const uint32_t e = vt_tile(vt, t / a.BH);
      const int s = static_cast<int>(e >> 16);
      ti.b = 0;
      ti.g = t % a.BH;
      ti.n0 = static_cast<int>(e & 0xFFFFu) * kTileN;
      ti.qbase = vt_cu_q(vt, s);
      const int tq = vt_cu_q(vt, s + 1) - ti.qbase;
      ti.kbase = vt_cu_k(vt, s);
      ti.tk = vt_cu_k(vt, s + 1) - ti.kbase;
      ti.rbase = vt_ps(vt, s);
      ti.off = ti.tk - tq;
      // Query tiles whose last row sees the tile's first key.
      const int first_q = ti.n0 - ti.off;  // first query that sees key n0
      const int mq_end = (tq + TM - 1) / TM;
      ti.m_begin = a.causal ? min(mq_end, max(0, first_q) / TM) : 0;
      ti.per_head = mq_end - ti.m_begin;
    } else {
      int nt, bg;
      if constexpr ((MODE & kDkvChunked) != 0) {
        dkdv_tile_coords(t, a.n_tiles, a.BH, a.bg_chunk, &nt, &bg);
      } else {
        nt = t / a.BH;
        bg = t % a.BH;
      }
      ti.b = bg / a.Hkv;
      ti.g = bg % a.Hkv;
      ti.n0 = nt * kTileN;
      ti.m_begin = a.causal ? ti.n0 / TM : 0;
      ti.per_head = m_end - ti.m_begin;
      ti.qbase = ti.kbase = ti.rbase = 0;
      ti.tk = a.T;
      ti.off = 0;
    }
    const int n_all = G * ti.per_head;
    ti.it_lo = static_cast<int>(static_cast<long>(crank) * n_all / C);
    ti.n_it = static_cast<int>(static_cast<long>(crank + 1) * n_all / C) - ti.it_lo;
    return ti;
  };

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + Cf::kOffK, sV = s0 + Cf::kOffV;
  auto stage_base = [&](int s) { return s0 + Cf::kOffStage + s * Cf::kStageBytes; };
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  // Byte offset of 16-byte chunk `chunk` of row `row` of a receive slot
  // ([dV | dK] fp32 per row, chunks XOR-swizzled by row % 8).
  auto slot_off = [](int row, int chunk) {
    return static_cast<uint32_t>(row * Cf::kRowBytes + ((chunk ^ (row & 7)) * 16));
  };
  const uint32_t recv_bytes = static_cast<uint32_t>((C - 1) * R * Cf::kRowBytes);

  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), Cf::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(kDkvBarKV), 1);
    mbar_init(bar(kDkvBarKVFree), 1);
    for (int s = 0; s < kDkvMaxStages; ++s) {
      mbar_init(bar(kDkvBarQFull + s), 1);
      mbar_init(bar(kDkvBarQEmpty + s), 1);
    }
    mbar_init(bar(kDkvBarKvTmem), kComputeWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kDkvBarS + i), 1);
      mbar_init(bar(kDkvBarSFree + i), kComputeWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kDkvBarP + i), kComputeWarps);
      mbar_init(bar(kDkvBarFree + i), 1);
    }
    mbar_init(bar(kDkvBarAcc), 1);
    mbar_init(bar(kDkvBarAccFree), kComputeWarps);
    mbar_init(bar(kDkvBarDrain), 1);
    mbar_init(bar(kDkvBarDrainAcc), 1);
    mbar_init(bar(kDkvBarRecv), 1);
    mbar_init(bar(kDkvBarRegionFree), kComputeWarps * (C > 1 ? C - 1 : 1));
    // The first tile's partial sums may arrive any time from now on.
    if (C > 1) mbar_arrive_expect_tx(bar(kDkvBarRecv), recv_bytes);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&mQ);
    tma_prefetch_desc(&mK);
    tma_prefetch_desc(&mV);
    tma_prefetch_desc(&mdO);
  }
  __syncthreads();
  // Peers' remote stores and arrivals target this block's mbarriers: they must
  // be initialised first.
  if (C > 1) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint64_t wait_ns = a.wait_ns;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int last[kDkvMaxStages];
      for (int s = 0; s < kDkvMaxStages; ++s) last[s] = -1;
      int last_kv = -1;
      int gi = 0;  // items loaded so far, over all tiles
      bool waited = false;  // for the Delta step's row statistics (dependent launch)
      for (int kt = 0; ok; ++kt) {
        const int t = tile_of(kt);
        if (t < 0) break;
        const DkvTile ti = tile_info(t);
        // K, V of the previous tile must no longer be read from shared
        // memory: copied into TMEM (D = 64) or consumed by its S^T MMAs.
        if (kt > 0 && !(ok = mbar_wait(bar(Cf::kKvInTmem ? kDkvBarKvTmem : kDkvBarKVFree),
                                       (kt - 1) & 1, wait_ns)))
          break;
        mbar_arrive_expect_tx(bar(kDkvBarKV), 2 * Cf::kKvBytes);
        for (int at = 0; at < Cf::kAtoms; ++at) {
          tma_load_4d(sK + at * (kTileN * 128), &mK, bar(kDkvBarKV), at * 64, ti.g,
                      ti.kbase + ti.n0, ti.b);
          tma_load_4d(sV + at * (kTileN * 128), &mV, bar(kDkvBarKV), at * 64, ti.g,
                      ti.kbase + ti.n0, ti.b);
        }
        last_kv = kt;
        int h = ti.g * G + (ti.n_it > 0 ? ti.it_lo / ti.per_head : 0);
        int m_idx = ti.n_it > 0 ? ti.it_lo % ti.per_head : 0;
        for (int li = 0; li < ti.n_it; ++li, ++gi) {
          const int s = gi % NS;
          const uint32_t ph = (gi / NS) & 1;
          const int i0 = (ti.m_begin + m_idx) * TM;
          if (gi >= NS && !(ok = mbar_wait(bar(kDkvBarQEmpty + s), ph ^ 1, wait_ns))) break;
          const uint32_t st = stage_base(s);
          mbar_arrive_expect_tx(bar(kDkvBarQFull + s), 2 * Cf::kQBytes + TM * 8);
          for (int at = 0; at < Cf::kAtoms; ++at) {
            tma_load_4d(st + at * (TM * 128), &mQ, bar(kDkvBarQFull + s), at * 64, h,
                        ti.qbase + i0, ti.b);
            tma_load_4d(st + Cf::kQBytes + at * (TM * 128), &mdO, bar(kDkvBarQFull + s), at * 64,
                        h, ti.qbase + i0, ti.b);
          }
          if (!waited) {
            // Launched as a dependent of the Delta step: only the row
            // statistics are its output, so everything up to here (setup,
            // K, V, Q, dO loads) overlaps it.  Once it is complete, the dQ
            // step (a programmatic dependent of this grid, reading only the
            // Delta step's results) may start on the SMs this grid frees.
            griddep_wait();
            griddep_launch_dependents();
            waited = true;
          }
          bulk_load(st + 2 * Cf::kQBytes,
                    a.rowstats + (static_cast<size_t>(ti.b) * a.Hq + h) * a.Tp + ti.rbase + i0,
                    TM * 8, bar(kDkvBarQFull + s));
          last[s] = gi;
          if (++m_idx == ti.per_head) {
            m_idx = 0;
            ++h;
          }
        }
      }
      if (!ok) {
        // Copies still in flight must land before the block may exit.
        if (last_kv >= 0) mbar_wait(bar(kDkvBarKV), last_kv & 1, wait_ns);
        for (int s = 0; s < NS; ++s)
          if (last[s] >= 0) mbar_wait(bar(kDkvBarQFull + s), (last[s] / NS) & 1, wait_ns);
      }
      // A block without items still lets the dQ step start only after the
      // Delta step is complete.
      if (!waited) {
        griddep_wait();
        griddep_launch_dependents();
      }
    }
    // The warp meets again before the block-wide barriers below (lanes 1-31
    // skipped the producer loop).
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ S^T / dP^T issuer
    // The whole warp runs this loop (MMA issue is warp-collective); every
    // wait is made warp-uniform so the warp stays converged.
    constexpr uint32_t kIdS = idesc_bf16(kTileN, TM, false, false);
    // Operand descriptors built once; the loop only adds constant offsets.
    const uint64_t dK = sdesc_sw128(sK, 16, 1024), dV = sdesc_sw128(sV, 16, 1024);
    const uint64_t dQk0 = sdesc_sw128(stage_base(0), 16, 1024);  // K-major B
    int gi = 0;
    for (int kt = 0; ok; ++kt) {
      const int t = tile_of(kt);
      if (t < 0) break;
      const DkvTile ti = tile_info(t);
      // The tile's K, V: in TMEM (D = 64, copied by the element-wise warps)
      // or in shared memory.
      if (!(ok = warp_all(mbar_wait(bar(Cf::kKvInTmem ? kDkvBarKvTmem : kDkvBarKV), kt & 1,
                                    wait_ns))))
        break;
      tc_fence_after();
      for (int li = 0; li < ti.n_it; ++li, ++gi) {
        const int s = gi % NS;
        const int sb = gi % NSB;
        // The element-wise warps must hold S^T, dP^T of the buffer's previous
        // item in registers before those of this one overwrite them.
        if (gi >= NSB &&
            !(ok = warp_all(mbar_wait(bar(kDkvBarSFree + sb), ((gi - NSB) / NSB) & 1, wait_ns))))
          break;
        if (!(ok = warp_all(mbar_wait(bar(kDkvBarQFull + s), (gi / NS) & 1, wait_ns)))) break;
        tc_fence_after();
        const uint64_t dQk = desc_add(dQk0, s * Cf::kStageBytes);
        const uint64_t ddOk = desc_add(dQk, Cf::kQBytes);
        const uint32_t tS = tmem + sb * 2 * TM, tDP = tS + TM;
        if constexpr (Cf::kKvInTmem) {
          // K = D = 64: four steps over the packed K / V columns and the
          // 32-byte K-major slices of Q / dO.
          const uint32_t aK = tmem + Cf::kColK, aV = tmem + Cf::kColV;
          mma_ts_x4(tS, aK, aK + 8, aK + 16, aK + 24, dQk, desc_add(dQk, 32), desc_add(dQk, 64),
                    desc_add(dQk, 96), kIdS, 0u);
          mma_ts_x4(tDP, aV, aV + 8, aV + 16, aV + 24, ddOk, desc_add(ddOk, 32), desc_add(ddOk, 64),
                    desc_add(ddOk, 96), kIdS, 0u);
        } else {
          // K = D in groups of 64 (one 128-byte swizzle atom): four 32-byte steps.
#pragma unroll
          for (int at = 0; at < Cf::kAtoms; ++at) {
            const uint64_t k = desc_add(dK, at * (kTileN * 128)), q = desc_add(dQk, at * (TM * 128));
            mma_ss_x4(tS, k, desc_add(k, 32), desc_add(k, 64), desc_add(k, 96), q, desc_add(q, 32),
                      desc_add(q, 64), desc_add(q, 96), kIdS, at > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int at = 0; at < Cf::kAtoms; ++at) {
            const uint64_t v = desc_add(dV, at * (kTileN * 128)), o = desc_add(ddOk, at * (TM * 128));
            mma_ss_x4(tDP, v, desc_add(v, 32), desc_add(v, 64), desc_add(v, 96), o, desc_add(o, 32),
                      desc_add(o, 64), desc_add(o, 96), kIdS, at > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(kDkvBarS + sb));
      }
      if (!ok) break;
      // K, V of this tile are free once these MMAs complete.
      mma_commit(bar(kDkvBarKVFree));
    }
    // Every issued MMA must finish before TMEM is released.
    mma_commit(bar(kDkvBarDrain));
    warp_all(mbar_wait(bar(kDkvBarDrain), 0, wait_ns));
  } else if (warp == kDkvAccWarp) {
    // ------------------------------------------------------------ dV / dK issuer
    constexpr uint32_t kIdAcc = idesc_bf16(kTileN, D, false, true);
    const uint32_t tDV = tmem + Cf::kColDV, tDK = tmem + Cf::kColDK;
    // Q, dO as MN-major B operands: 16 queries per 2048-byte step, the
    // 64-column blocks of D = 128 TM * 128 bytes apart.
    const uint64_t dQm0 = sdesc_sw128(stage_base(0), TM * 128, 1024);
    int gi = 0;
    for (int kt = 0; ok; ++kt) {
      const int t = tile_of(kt);
      if (t < 0) break;
      const DkvTile ti = tile_info(t);
      // The element-wise warps must have read the previous tile's sums before
      // this tile's first MMA overwrites them -- and before this tile's
      // completion is signalled at all: a tile without items here signals at
      // once, and two completions ahead of the readers would alias the
      // parity they wait on.
      if (kt > 0 && !(ok = warp_all(mbar_wait(bar(kDkvBarAccFree), (kt - 1) & 1, wait_ns)))) break;
      for (int li = 0; li < ti.n_it; ++li, ++gi) {
        const int s = gi % NS;
        const int pb = gi % NPB;
        if (!(ok = warp_all(mbar_wait(bar(kDkvBarP + pb), (gi / NPB) & 1, wait_ns)))) break;
        tc_fence_after();
        const uint64_t dQm = desc_add(dQm0, s * Cf::kStageBytes);
        const uint64_t ddOm = desc_add(dQm, Cf::kQBytes);
        // P^T / dS^T of queries 16ks..16ks+15: 8 packed columns at 8ks.
        const uint32_t tP = tmem + Cf::kColPB + pb * TM, tDS = tP + TM / 2;
#pragma unroll
        for (int q4 = 0; q4 < TM / 64; ++q4) {
          const uint32_t acc = (li > 0 || q4 > 0) ? 1u : 0u;
          const uint32_t p = tP + q4 * 32;
          const uint64_t o = desc_add(ddOm, q4 * 8192);
          mma_ts_x4(tDV, p, p + 8, p + 16, p + 24, o, desc_add(o, 2048), desc_add(o, 4096),
                    desc_add(o, 6144), kIdAcc, acc);
        }
#pragma unroll
        for (int q4 = 0; q4 < TM / 64; ++q4) {
          const uint32_t acc = (li > 0 || q4 > 0) ? 1u : 0u;
          const uint32_t p = tDS + q4 * 32;
          const uint64_t q = desc_add(dQm, q4 * 8192);
          mma_ts_x4(tDK, p, p + 8, p + 16, p + 24, q, desc_add(q, 2048), desc_add(q, 4096),
                    desc_add(q, 6144), kIdAcc, acc);
        }
        // Both MMA streams of item gi have read stage s (the S^T stream
        // finished before the element-wise warps released P): free it, and the
        // P^T / dS^T buffer.
        mma_commit(bar(kDkvBarQEmpty + s));
        mma_commit(bar(kDkvBarFree + pb));
      }
      if (!ok) break;
      mma_commit(bar(kDkvBarAcc));  // this tile's sums (at once when it has no items)
    }
    mma_commit(bar(kDkvBarDrainAcc));
    warp_all(mbar_wait(bar(kDkvBarDrainAcc), 0, wait_ns));
  } else {
    // ------------------------------------------------------------ P^T / dS^T warps
    // Warps w, w+4, w+8, w+12 share TMEM lane quarter (w & 3), i.e. the same
    // 32 key rows; group grp = (w - 2) / 4 takes queries QG grp..QG grp+QG-1
    // of each item, and columns grp D/4 .. of dV, dK in the tile epilogue.
    const int quarter = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    const int owner = r / R;  // block of the cluster that stores key row r
    // D = 64: K and V row r of tile kt into TMEM as the A operands of S^T and
    // dP^T, once they have landed and the previous tile's S^T MMAs no longer
    // read TMEM's copy; this thread copies elements 16 grp..16 grp+15 (two
    // 16-byte chunks of the 128-byte-swizzled tile row) as 8 packed pairs.
    // Done for the next tile before this tile's epilogue, so the next tile's
    // first scores overlap the epilogue.
    auto copy_kv = [&](int kt) -> bool {
      bool good = warp_all(mbar_wait(bar(kDkvBarKV), kt & 1, wait_ns));
      if (good && kt > 0) good = warp_all(mbar_wait(bar(kDkvBarKVFree), (kt - 1) & 1, wait_ns));
      if (good) {
        tc_fence_after();
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t base = (which == 0 ? sK : sV) + r * 128;
          uint32_t v8[8];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint4 x = ld_shared_u4(base + (((2 * grp + c) ^ (r & 7)) * 16));
            v8[4 * c] = x.x;
            v8[4 * c + 1] = x.y;
            v8[4 * c + 2] = x.z;
            v8[4 * c + 3] = x.w;
          }
          tmem_st8_nowait(tl + (which == 0 ? Cf::kColK : Cf::kColV) + grp * 8, v8);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kDkvBarKvTmem));
      return good;
    };
    if (Cf::kKvInTmem && tile_of(0) >= 0) ok = copy_kv(0);
    int gi = 0;
    for (int kt = 0; ok; ++kt) {
      const int t = tile_of(kt);
      if (t < 0) break;
      const DkvTile ti = tile_info(t);
      const int krow = ti.n0 + r;
      int m_idx = ti.n_it > 0 ? ti.it_lo % ti.per_head : 0;  // query tile of the item in its head
      for (int li = 0; li < ti.n_it && ok; ++li, ++gi) {
        const int s = gi % NS;
        const int pb = gi % NPB;
        const int i0 = (ti.m_begin + m_idx) * TM + grp * QG;  // this group's first query
        if (++m_idx == ti.per_head) m_idx = 0;
        const int sb = gi % NSB;
        ok = warp_all(mbar_wait(bar(kDkvBarS + sb), (gi / NSB) & 1, wait_ns));
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[QG], dp[QG];
        const uint32_t tSb = tl + sb * 2 * TM;
        tmem_ld_cols<QG>(tSb + grp * QG, sv);
        tmem_ld_cols<QG>(tSb + TM + grp * QG, dp);
        tmem_wait_ld();
        reg_fence_cols<QG>(sv);
        reg_fence_cols<QG>(dp);
        // S^T, dP^T are in registers: a later item's may overwrite them.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kDkvBarSFree + sb));
        // Causal: query i0 + c sees key krow iff c >= krow - i0.  Only a
        // block on the diagonal needs the mask, and lane 0 holds the warp's
        // smallest krow, so the test is made once for the whole warp and the
        // unmasked items run a loop without it.
        const int cmin = a.causal ? (krow - ti.off - i0) : -1;
        const bool warp_masked = a.causal && (ti.n0 + quarter * 32 - ti.off - i0) + 31 > 0;
        uint32_t pk[QG / 2], dk[QG / 2];
        // (-lse2, -delta) of this group's queries, two per float4.
        const uint32_t st4 = stage_base(s) + 2 * Cf::kQBytes + grp * QG * 8;
        auto element_loop = [&](auto masked) {
          constexpr bool kMasked = decltype(masked)::value;
          static_for<QG / 2>([&](auto ic) {
              constexpr int c2 = decltype(ic)::value;
              constexpr int c = 2 * c2;
              // (-lse2_c, -delta_c, -lse2_c+1, -delta_c+1)
              const float4 rs = ld_shared_f4_at<c2 * 16>(st4);
              const float x0 = fmaf(__uint_as_float(sv[c]), sl2, rs.x);
              const float x1 = fmaf(__uint_as_float(sv[c + 1]), sl2, rs.z);
              float p0, p1;
              if constexpr ((c2 & 7) < kPolyOf8) {
                p0 = exp2_poly(x0);
                p1 = exp2_poly(x1);
              } else {
                p0 = ex2_approx(x0);
                p1 = ex2_approx(x1);
              }
              if constexpr (kMasked) {
                if (c < cmin) p0 = 0.f;
                if (c + 1 < cmin) p1 = 0.f;
              }
              const float d0 = p0 * (__uint_as_float(dp[c]) + rs.y);
              const float d1 = p1 * (__uint_as_float(dp[c + 1]) + rs.w);
              pk[c2] = pack_bf16x2(p0, p1);
              dk[c2] = pack_bf16x2(d0, d1);
          });
        };
        if (warp_masked)
          element_loop(std::true_type{});
        else
          element_loop(std::false_type{});
        // P^T / dS^T buffer pb last held item gi - NPB: its dV, dK must have
        // read it.
        if (gi >= NPB) {
          ok = warp_all(mbar_wait(bar(kDkvBarFree + pb), ((gi - NPB) / NPB) & 1, wait_ns));
          if (!ok) break;
          tc_fence_after();
        }
        if constexpr ((MODE & kDkvStoreDs) != 0) {
          {
            // Stored-dS backward: this item's dS^T rows also go to the
            // workspace, for the dQ step to read instead of recomputing them.
            const int it = ti.it_lo + li;
            const int h = ti.g * G + it / ti.per_head;
            const int m = ti.m_begin + it % ti.per_head;
            const int mt = m >> 1, kt = ti.n0 / kTileN;
            const long pr = a.causal ? static_cast<long>(mt) * (mt + 1) / 2 + kt
                                     : static_cast<long>(mt) * a.n_tiles + kt;
            const size_t row =
                (((static_cast<size_t>(ti.b) * a.Hq + h) * a.ds_pairs + pr) * 2 + (m & 1)) * kTileN + r;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.ds) + row * TM +
                                                  grp * QG);
            static_assert(QG == 16, "two 16-byte stores per thread");
            dst[0] = make_uint4(dk[0], dk[1], dk[2], dk[3]);
            dst[1] = make_uint4(dk[4], dk[5], dk[6], dk[7]);
          }
        }
        const uint32_t tP = tl + Cf::kColPB + pb * TM + grp * (QG / 2);
        tmem_st_cols<QG / 2>(tP, pk);
        tmem_st_cols<QG / 2>(tP + TM / 2, dk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kDkvBarP + pb));
      }
      if (!ok) break;
      if (Cf::kKvInTmem && tile_of(kt + 1) >= 0 && !(ok = copy_kv(kt + 1))) break;

      // ---------------------------------------------------------- tile epilogue
      // This thread's share of key row r: D/4 columns of dV and of dK (zero
      // for a block without items in the tile).
      ok = warp_all(mbar_wait(bar(kDkvBarAcc), kt & 1, wait_ns));
      if (!ok) break;
      uint32_t part_v[D / 4], part_k[D / 4];
      if (ti.n_it > 0) {
        tc_fence_after();
        tmem_ld_cols<D / 4>(tl + Cf::kColDV + grp * (D / 4), part_v);
        tmem_ld_cols<D / 4>(tl + Cf::kColDK + grp * (D / 4), part_k);
        tmem_wait_ld();
        reg_fence_cols<D / 4>(part_v);
        reg_fence_cols<D / 4>(part_k);
      } else {
#pragma unroll
        for (int i = 0; i < D / 4; ++i) part_v[i] = part_k[i] = 0u;
      }
      // The next tile's first dV, dK MMA may overwrite the accumulators.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kDkvBarAccFree));

      if (C > 1) {
        // Rows another block owns: to its receive region, once it has read
        // the previous tile's.
        if (kt > 0) {
          ok = warp_all(mbar_wait(bar(kDkvBarRegionFree), (kt - 1) & 1, wait_ns));
          if (!ok) break;
        }
        if (owner != crank) {
          const int j = crank < owner ? crank : crank - 1;
          const int row = j * R + (r - owner * R);
          const uint32_t dst = map_shared_rank(s0 + Cf::kOffRecv, static_cast<uint32_t>(owner));
          const uint32_t rbar = map_shared_rank(bar(kDkvBarRecv), static_cast<uint32_t>(owner));
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const uint32_t* v = which == 0 ? part_v : part_k;
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
              const int chunk = (which * D + grp * (D / 4)) / 4 + i;
              st_async_f4(dst + slot_off(row, chunk),
                          make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                      __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])),
                          rbar);
            }
          }
        }
        // Own rows: this block's sums, then the peers' in rank order.
        ok = warp_all(mbar_wait(bar(kDkvBarRecv), kt & 1, wait_ns));
        if (!ok) break;
        // Arm the receive mbarrier for the next tile's sums.  Peers send them
        // only after every warp here has signalled (below, after this arm in
        // program order), and until then the barrier cannot move past the
        // phase the other warps are still checking.
        if (warp == 2 && lane == 0 && tile_of(kt + 1) >= 0)
          mbar_arrive_expect_tx(bar(kDkvBarRecv), recv_bytes);
        if (owner == crank) {
          const int rl = r - crank * R;
          for (int src = 0; src < C; ++src) {
            if (src == crank) continue;
            const int j = src < crank ? src : src - 1;
            const uint32_t slot = s0 + Cf::kOffRecv;
            const int row = j * R + rl;
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
              const float4 x = ld_shared_f4(slot + slot_off(row, (grp * (D / 4)) / 4 + i));
              const float4 y = ld_shared_f4(slot + slot_off(row, (D + grp * (D / 4)) / 4 + i));
              part_v[4 * i] = __float_as_uint(__uint_as_float(part_v[4 * i]) + x.x);
              part_v[4 * i + 1] = __float_as_uint(__uint_as_float(part_v[4 * i + 1]) + x.y);
              part_v[4 * i + 2] = __float_as_uint(__uint_as_float(part_v[4 * i + 2]) + x.z);
              part_v[4 * i + 3] = __float_as_uint(__uint_as_float(part_v[4 * i + 3]) + x.w);
              part_k[4 * i] = __float_as_uint(__uint_as_float(part_k[4 * i]) + y.x);
              part_k[4 * i + 1] = __float_as_uint(__uint_as_float(part_k[4 * i + 1]) + y.y);
              part_k[4 * i + 2] = __float_as_uint(__uint_as_float(part_k[4 * i + 2]) + y.z);
              part_k[4 * i + 3] = __float_as_uint(__uint_as_float(part_k[4 * i + 3]) + y.w);
            }
          }
        }
        // This block's receive region is read: the peers may send the next
        // tile's sums (after the last tile nothing more is sent).
        __syncwarp();
        if (lane == 0 && tile_of(kt + 1) >= 0) {
          for (int p = 0; p < C; ++p)
            if (p != crank)
              mbar_arrive_remote(map_shared_rank(bar(kDkvBarRegionFree), static_cast<uint32_t>(p)));
        }
      }
      if (owner == crank && krow < ti.tk) {
        const size_t rbase =
            ((static_cast<size_t>(ti.b) * a.Tk + ti.kbase + krow) * a.Hkv + ti.g) * D +
            grp * (D / 4);
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t* v = which == 0 ? part_v : part_k;
          const float mul = which == 0 ? 1.f : a.scale;
          uint4* dst = reinterpret_cast<uint4*>(
              static_cast<__nv_bfloat16*>(which == 0 ? a.dv : a.dk) + rbase);
          auto f = [&](int i) { return __uint_as_float(v[i]) * mul; };
#pragma unroll
          for (int i = 0; i < D / 32; ++i)
            dst[i] = make_uint4(pack_bf16x2(f(8 * i), f(8 * i + 1)), pack_bf16x2(f(8 * i + 2), f(8 * i + 3)),
                                pack_bf16x2(f(8 * i + 4), f(8 * i + 5)),
                                pack_bf16x2(f(8 * i + 6), f(8 * i + 7)));
        }
      }
    }
  }

  // No block may exit while a peer can still store into its shared memory or
  // arrive on its mbarriers: every block reaches this barrier (no early exit;
  // all waits above are bounded).
  if (C > 1) {
    __syncwarp();
    cluster_sync();
  }

  if (!ok) atomicOr(&g_bwd_status, 2u);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Cf::kTmemCols);
  }
}

// ============================================================== dK / dV, D = 64
// The same tile walk, cluster split and partial-sum exchange as above, with
// items of 128 queries and fewer, fuller element-wise threads:
//   warp 0      producer: each tile's K, V; each item's Q, dO and row
//               statistics into a ring of stages
//   warp 1      S^T = K Q^T and dP^T = V dO^T (both operands in shared
//               memory, M = 128 keys, N = 128 queries) as soon as the
//               element-wise warps hold the previous item's in registers
//   warp 2      dV += P^T dO and dK += dS^T Q, P^T and dS^T read from TMEM
//   warps 4..11 element-wise, two threads per key row (TMEM lane), one per
//               64-query half of the item: P^T, dS^T as packed bf16 into TMEM
//               columns of their own; at the tile's end D/2 columns each of
//               dV and dK for the exchange and the store
// TMEM: S^T [128 fp32 columns], dP^T [128], P^T [64 columns of bf16 pairs],
// dS^T [64], dV [64], dK [64].
// With a listed deal (DkvList) a block walks its own tiles: first those its
// cluster shares (items split, partial sums exchanged, as in the snake
// walk), then tiles of its own, whose rows it stores alone.
//
// At D = 128 the same kernel runs with one block per key tile (no cluster)
// and two stages; dV and dK take 256 TMEM columns, so P^T and dS^T go into
// the S^T and dP^T columns their own threads have just read, and the next
// item's S^T, dP^T wait for this item's dV, dK products.
constexpr int kDkwTM = 128;                // queries per item
constexpr int kDkwWarps = 12;
constexpr int kDkwThreads = kDkwWarps * 32;
constexpr uint32_t kDkwCtrlRegs = 104, kDkwElemRegs = 192;
constexpr int kDkwRegBudget = 128 * kDkwCtrlRegs + 256 * kDkwElemRegs;
template <int D>
struct DkwCfg {
  static constexpr int kAtoms = D / 64;                    // 128-byte swizzle atoms per row
  static constexpr int kKvBytes = kTileN * 128 * kAtoms;   // 128 keys x D
  static constexpr int kQBytes = kDkwTM * 128 * kAtoms;    // 128 queries x D
  static constexpr int kStages = D == 64 ? 3 : 2;
  static constexpr int kStageBytes = 2 * kQBytes + 1024;   // Q, dO, then 128 row statistics
  // K, V buffers: at D = 64 two, so the next tile's K, V load while this
  // tile's items run (tile kt in buffer kt % 2).
  static constexpr int kKvBufs = D == 64 ? 2 : 1;
  static constexpr int kOffK = 0;                          // buffer b: K at 2 b kKvBytes
  static constexpr int kOffV = kKvBytes;                   // V right after it
  static constexpr int kOffStage = 2 * kKvBufs * kKvBytes;
  static constexpr int kMaxCluster = D == 64 ? 8 : 1;
  static constexpr int kRowBytes = 2 * D * 4;              // [dV | dK] fp32
  static constexpr int kOffRecv = kOffStage + kStages * kStageBytes;
  static constexpr int kRecvBytes = (kTileN - kTileN / kMaxCluster) * kRowBytes;
  static constexpr int kSmemBytes = kOffRecv + kRecvBytes + 1024;
  // P^T and dS^T of query group g (64 queries, 32 packed columns) start at
  // kColP + g kGrp and kColDS + g kGrp.
  static constexpr uint32_t kColS = 0, kColDP = 128;
  static constexpr uint32_t kColP = D == 64 ? 256 : kColS, kColDS = D == 64 ? 320 : kColDP;
  static constexpr uint32_t kGrp = D == 64 ? 32 : 64;
  static constexpr uint32_t kColDV = D == 64 ? 384 : 256, kColDK = kColDV + D;
  static_assert(kColDK + D <= 512, "TMEM layout");
  static_assert(kSmemBytes + 512 <= 227 * 1024, "shared memory per block (with the static part)");
  static_assert(kStageBytes % 1024 == 0, "stages keep the swizzle alignment");
};

template <int D, class VT, int MODE>
__global__ void __launch_bounds__(kDkwThreads, 1)
    attn_dkdvq_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                      const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mdO,
                      const BwdArgs a, const __grid_constant__ VT vt,
                      const __grid_constant__ DkvList lst) {
  using Cf = DkwCfg<D>;
  constexpr bool VL = std::is_same<VT, VarlenTable>::value;
  static_assert(!VL || MODE == 0, "the packed form walks its own table");
  static_assert(D == 64 || (MODE & kDkvStoreDs) == 0, "dS^T stored at D = 64 only");
  constexpr int NS = Cf::kStages;
  constexpr int TM = kDkwTM;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kDkvNumBars];
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.cluster;
  const int crank = C > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int group = static_cast<int>(blockIdx.x) / C;
  const int NG = a.n_groups;
  const int n_tiles_all = (VL ? vt_tiles(vt) : a.n_tiles) * a.BH;
  const int G = a.Hq / a.Hkv;
  const int m_end = (a.T + TM - 1) / TM;
  const int R = kTileN / C;
  // This block's turns: kt < n_sh are tiles the cluster shares (the exchange
  // counts its phases by kt), the others tiles of this block alone.
  // Only the 64-dim walk without chunks is ever listed.
  constexpr bool kListable = D == 64 && (MODE & kDkvChunked) == 0;
  const bool listed = kListable && lst.n_blocks > 0;
  const int l0 = listed ? lst.start[blockIdx.x] : 0;
  const int l_n = listed ? lst.start[blockIdx.x + 1] - l0 : 0;
  int n_sh = C > 1 ? INT_MAX : 0;
  if (listed) {
    n_sh = 0;
    while (n_sh < l_n && (lst.entry[l0 + n_sh] & 1u) != 0) ++n_sh;
  }
  // Tile of this block's kt-th turn, or -1 past its last.
  auto tile_of = [&](int kt) {
    if (listed) return kt < l_n ? static_cast<int>(lst.entry[l0 + kt] >> 1) : -1;
    const int t = kt * NG + ((kt & 1) ? NG - 1 - group : group);
    return t < n_tiles_all ? t : -1;
  };
  // Whether turn kt + 1 is shared as well (the exchange goes on).
  auto shared_next = [&](int kt) { return kt + 1 < n_sh && tile_of(kt + 1) >= 0; };
  auto tile_info = [&](int t, bool shared) {
    DkvTile ti;
    if constexpr (VL) {
      const uint32_t e = vt_tile(vt, t / a.BH);
      const int s = static_cast<int>(e >> 16);
      ti.b = 0;
      ti.g = t % a.BH;
      ti.n0 = static_cast<int>(e & 0xFFFFu) * kTileN;
      ti.qbase = vt_cu_q(vt, s);
      const int tq = vt_cu_q(vt, s + 1) - ti.qbase;
      ti.kbase = vt_cu_k(vt, s);
      ti.tk = vt_cu_k(vt, s + 1) - ti.kbase;
      ti.rbase = vt_ps(vt, s);
      ti.off = ti.tk - tq;
      // Query tiles whose last row sees the tile's first key.
      const int first_q = ti.n0 - ti.off;  // first query that sees key n0
      const int mq_end = (tq + TM - 1) / TM;
      ti.m_begin = a.causal ? min(mq_end, max(0, first_q) / TM) : 0;
      ti.per_head = mq_end - ti.m_begin;
    } else {
      int nt, bg;
      if constexpr ((MODE & kDkvChunked) != 0) {
        dkdv_tile_coords(t, a.n_tiles, a.BH, a.bg_chunk, &nt, &bg);
      } else {
        nt = t / a.BH;
        bg = t % a.BH;
      }
      ti.b = bg / a.Hkv;
      ti.g = bg % a.Hkv;
      ti.n0 = nt * kTileN;
      ti.m_begin = a.causal ? ti.n0 / TM : 0;
      ti.per_head = m_end - ti.m_begin;
      ti.qbase = ti.kbase = ti.rbase = 0;
      ti.tk = a.T;
      ti.off = 0;
    }
    const int n_all = G * ti.per_head;
    const int cs = shared ? C : 1, cr = shared ? crank : 0;
    ti.it_lo = static_cast<int>(static_cast<long>(cr) * n_all / cs);
    ti.n_it = static_cast<int>(static_cast<long>(cr + 1) * n_all / cs) - ti.it_lo;
    return ti;
  };

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + Cf::kOffK, sV = s0 + Cf::kOffV;
  auto stage_base = [&](int s) { return s0 + Cf::kOffStage + s * Cf::kStageBytes; };
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  // Byte offset of 16-byte chunk `chunk` of row `row` of a receive slot
  // ([dV | dK] fp32 per row, chunks XOR-swizzled by row % 8).
  auto slot_off = [](int row, int chunk) {
    return static_cast<uint32_t>(row * Cf::kRowBytes + ((chunk ^ (row & 7)) * 16));
  };
  const uint32_t recv_bytes = static_cast<uint32_t>((C - 1) * R * Cf::kRowBytes);

  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(kDkvBarKV), 1);
    mbar_init(bar(kDkvBarKVFree), 1);
    mbar_init(bar(kDkvBarKV2), 1);
    mbar_init(bar(kDkvBarKVFree2), 1);
    for (int s = 0; s < kDkvMaxStages; ++s) {
      mbar_init(bar(kDkvBarQFull + s), 1);
      mbar_init(bar(kDkvBarQEmpty + s), 1);
    }
    // D = 128 uses the second entries as well: S^T and dP^T land (S, S + 1),
    // P^T and dS^T are written (P, P + 1), dV and dK products done (Free,
    // Free + 1).
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kDkvBarS + i), 1);
      mbar_init(bar(kDkvBarP + i), 8);
      mbar_init(bar(kDkvBarFree + i), 1);
    }
    mbar_init(bar(kDkvBarSFree), 8);
    mbar_init(bar(kDkvBarAcc), 1);
    mbar_init(bar(kDkvBarAccFree), 8);
    mbar_init(bar(kDkvBarDrain), 1);
    mbar_init(bar(kDkvBarDrainAcc), 1);
    mbar_init(bar(kDkvBarRecv), 1);
    mbar_init(bar(kDkvBarRegionFree), C > 1 ? C - 1 : 1);
    mbar_init(bar(kDkvBarRecvRead), 8);
    // The first tile's partial sums may arrive any time from now on.
    if (C > 1 && n_sh > 0) mbar_arrive_expect_tx(bar(kDkvBarRecv), recv_bytes);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&mQ);
    tma_prefetch_desc(&mK);
    tma_prefetch_desc(&mV);
    tma_prefetch_desc(&mdO);
  }
  __syncthreads();
  // Peers' remote stores and arrivals target this block's mbarriers: they must
  // be initialised first.
  if (C > 1) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint64_t wait_ns = a.wait_ns;
  bool ok = true;

  if (warp < 4) {
  // Each warpgroup changes its register count at the top of its own branch,
  // so the code after it is compiled for the new count.
  setmaxnreg_dec<kDkwCtrlRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int last[kDkvMaxStages];
      for (int s = 0; s < kDkvMaxStages; ++s) last[s] = -1;
      int last_kv = -1;
      int gi = 0;  // items loaded so far, over all tiles
      bool waited = false;  // for the Delta step's row statistics (dependent launch)
      for (int kt = 0; ok; ++kt) {
        const int t = tile_of(kt);
        if (t < 0) break;
        const DkvTile ti = tile_info(t, kt < n_sh);
        // The S^T, dP^T MMAs of the tile that last used this K, V buffer
        // must be done with it.
        const int kb = kt % Cf::kKvBufs, kuse = kt / Cf::kKvBufs;
        if (kuse > 0 && !(ok = mbar_wait(bar(kb == 0 ? kDkvBarKVFree : kDkvBarKVFree2),
                                         (kuse - 1) & 1, wait_ns)))
          break;
        const int kvbar = kb == 0 ? kDkvBarKV : kDkvBarKV2;
        mbar_arrive_expect_tx(bar(kvbar), 2 * Cf::kKvBytes);
        for (int at = 0; at < Cf::kAtoms; ++at) {
          tma_load_4d(sK + kb * 2 * Cf::kKvBytes + at * (kTileN * 128), &mK, bar(kvbar), at * 64,
                      ti.g, ti.kbase + ti.n0, ti.b);
          tma_load_4d(sV + kb * 2 * Cf::kKvBytes + at * (kTileN * 128), &mV, bar(kvbar), at * 64,
                      ti.g, ti.kbase + ti.n0, ti.b);
        }
        last_kv = kt;
        int h = ti.g * G + (ti.n_it > 0 ? ti.it_lo / ti.per_head : 0);
        int m_idx = ti.n_it > 0 ? ti.it_lo % ti.per_head : 0;
        for (int li = 0; li < ti.n_it; ++li, ++gi) {
          const int s = gi % NS;
          const uint32_t ph = (gi / NS) & 1;
          const int i0 = (ti.m_begin + m_idx) * TM;
          if (gi >= NS && !(ok = mbar_wait(bar(kDkvBarQEmpty + s), ph ^ 1, wait_ns))) break;
          const uint32_t st = stage_base(s);
          mbar_arrive_expect_tx(bar(kDkvBarQFull + s), 2 * Cf::kQBytes + TM * 8);
          for (int at = 0; at < Cf::kAtoms; ++at) {
            tma_load_4d(st + at * (TM * 128), &mQ, bar(kDkvBarQFull + s), at * 64, h,
                        ti.qbase + i0, ti.b);
            tma_load_4d(st + Cf::kQBytes + at * (TM * 128), &mdO, bar(kDkvBarQFull + s), at * 64,
                        h, ti.qbase + i0, ti.b);
          }
          if (!waited) {
            // Launched as a dependent of the Delta step: only the row
            // statistics are its output, so everything up to here (setup,
            // K, V, Q, dO loads) overlaps it.  Once it is complete, the dQ
            // step (a programmatic dependent of this grid, reading only the
            // Delta step's results) may start on the SMs this grid frees.
            griddep_wait();
            griddep_launch_dependents();
            waited = true;
          }
          bulk_load(st + 2 * Cf::kQBytes,
                    a.rowstats + (static_cast<size_t>(ti.b) * a.Hq + h) * a.Tp + ti.rbase + i0,
                    TM * 8, bar(kDkvBarQFull + s));
          last[s] = gi;
          if (++m_idx == ti.per_head) {
            m_idx = 0;
            ++h;
          }
        }
      }
      if (!ok) {
        // Copies still in flight must land before the block may exit.
        if (last_kv >= 0)
          mbar_wait(bar(last_kv % Cf::kKvBufs == 0 ? kDkvBarKV : kDkvBarKV2),
                    (last_kv / Cf::kKvBufs) & 1, wait_ns);
        for (int s = 0; s < NS; ++s)
          if (last[s] >= 0) mbar_wait(bar(kDkvBarQFull + s), (last[s] / NS) & 1, wait_ns);
      }
      // A block without items still lets the dQ step start only after the
      // Delta step is complete.
      if (!waited) {
        griddep_wait();
        griddep_launch_dependents();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ S^T / dP^T issuer
    // The whole warp runs this loop (MMA issue is warp-collective); every
    // wait is made warp-uniform so the warp stays converged.
    constexpr uint32_t kIdS = idesc_bf16(kTileN, TM, false, false);
    const uint64_t dK0 = sdesc_sw128(sK, 16, 1024), dV0 = sdesc_sw128(sV, 16, 1024);
    const uint64_t dQk0 = sdesc_sw128(stage_base(0), 16, 1024);  // K-major B
    const uint32_t tS = tmem + Cf::kColS, tDP = tmem + Cf::kColDP;
    int gi = 0;
    for (int kt = 0; ok; ++kt) {
      const int t = tile_of(kt);
      if (t < 0) break;
      const DkvTile ti = tile_info(t, kt < n_sh);
      const int kb = kt % Cf::kKvBufs;
      if (!(ok = warp_all(mbar_wait(bar(kb == 0 ? kDkvBarKV : kDkvBarKV2), (kt / Cf::kKvBufs) & 1,
                                    wait_ns))))
        break;
      const uint64_t dK = desc_add(dK0, kb * 2 * Cf::kKvBytes), dV = desc_add(dV0, kb * 2 * Cf::kKvBytes);
      // The previous tile's last dV, dK products go first: its epilogue waits
      // for them, while this tile's first scores are not needed before that
      // epilogue ends.  (Only before items of this block: with none, this
      // tile's sums are signalled at once and could complete the barrier's
      // next phase before this wait, which would then look for the wrong one.)
      if (kt > 0 && ti.n_it > 0 &&
          !(ok = warp_all(mbar_wait(bar(kDkvBarAcc), (kt - 1) & 1, wait_ns))))
        break;
      tc_fence_after();
      for (int li = 0; li < ti.n_it; ++li, ++gi) {
        const int s = gi % NS;
        if constexpr (D == 128) {
          // S^T and dP^T separately: S^T once the previous item's dV product
          // has read the P^T written over its columns, dP^T once its dK
          // product has read dS^T; each lands on a barrier of its own, so the
          // element-wise warps start on P^T while dP^T is computed.
          if (!(ok = warp_all(mbar_wait(bar(kDkvBarQFull + s), (gi / NS) & 1, wait_ns)))) break;
          const uint64_t q0 = desc_add(dQk0, s * Cf::kStageBytes), o0 = desc_add(q0, Cf::kQBytes);
          if (gi > 0 && !(ok = warp_all(mbar_wait(bar(kDkvBarFree), (gi - 1) & 1, wait_ns)))) break;
          tc_fence_after();
#pragma unroll
          for (int at = 0; at < Cf::kAtoms; ++at) {
            const uint64_t k = desc_add(dK, at * (kTileN * 128)), q = desc_add(q0, at * (TM * 128));
            mma_ss_x4(tS, k, desc_add(k, 32), desc_add(k, 64), desc_add(k, 96), q, desc_add(q, 32),
                      desc_add(q, 64), desc_add(q, 96), kIdS, at > 0 ? 1u : 0u);
          }
          mma_commit(bar(kDkvBarS));
          if (gi > 0 && !(ok = warp_all(mbar_wait(bar(kDkvBarFree + 1), (gi - 1) & 1, wait_ns))))
            break;
          tc_fence_after();
#pragma unroll
          for (int at = 0; at < Cf::kAtoms; ++at) {
            const uint64_t v = desc_add(dV, at * (kTileN * 128)), o = desc_add(o0, at * (TM * 128));
            mma_ss_x4(tDP, v, desc_add(v, 32), desc_add(v, 64), desc_add(v, 96), o, desc_add(o, 32),
                      desc_add(o, 64), desc_add(o, 96), kIdS, at > 0 ? 1u : 0u);
          }
          mma_commit(bar(kDkvBarS + 1));
          continue;
        }
        // The element-wise warps must hold the previous item's S^T, dP^T in
        // registers before this item's overwrite them.
        if (gi > 0 && !(ok = warp_all(mbar_wait(bar(kDkvBarSFree), (gi - 1) & 1, wait_ns)))) break;
        if (!(ok = warp_all(mbar_wait(bar(kDkvBarQFull + s), (gi / NS) & 1, wait_ns)))) break;
        tc_fence_after();
        const uint64_t q0 = desc_add(dQk0, s * Cf::kStageBytes), o0 = desc_add(q0, Cf::kQBytes);
        // K = D in groups of 64 (one 128-byte swizzle atom): four 32-byte steps.
#pragma unroll
        for (int at = 0; at < Cf::kAtoms; ++at) {
          const uint64_t k = desc_add(dK, at * (kTileN * 128)), q = desc_add(q0, at * (TM * 128));
          mma_ss_x4(tS, k, desc_add(k, 32), desc_add(k, 64), desc_add(k, 96), q, desc_add(q, 32),
                    desc_add(q, 64), desc_add(q, 96), kIdS, at > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int at = 0; at < Cf::kAtoms; ++at) {
          const uint64_t v = desc_add(dV, at * (kTileN * 128)), o = desc_add(o0, at * (TM * 128));
          mma_ss_x4(tDP, v, desc_add(v, 32), desc_add(v, 64), desc_add(v, 96), o, desc_add(o, 32),
                    desc_add(o, 64), desc_add(o, 96), kIdS, at > 0 ? 1u : 0u);
        }
        mma_commit(bar(kDkvBarS));
      }
      if (!ok) break;
      // K, V of this tile are free once these MMAs complete.
      mma_commit(bar(kb == 0 ? kDkvBarKVFree : kDkvBarKVFree2));
    }
    // Every issued MMA must finish before TMEM is released.
    mma_commit(bar(kDkvBarDrain));
    warp_all(mbar_wait(bar(kDkvBarDrain), 0, wait_ns));
  } else if (warp == 2) {
    // ------------------------------------------------------------ dV / dK issuer
    constexpr uint32_t kIdAcc = idesc_bf16(kTileN, D, false, true);
    const uint32_t tDV = tmem + Cf::kColDV, tDK = tmem + Cf::kColDK;
    const uint32_t tP = tmem + Cf::kColP, tDS = tmem + Cf::kColDS;
    // Q, dO as MN-major B operands: 16 queries per 2048-byte step, the
    // 64-column blocks of D = 128 TM * 128 bytes apart.
    const uint64_t dQm0 = sdesc_sw128(stage_base(0), TM * 128, 1024);
    int gi = 0;
    for (int kt = 0; ok; ++kt) {
      const int t = tile_of(kt);
      if (t < 0) break;
      const DkvTile ti = tile_info(t, kt < n_sh);
      // The element-wise warps must have read the previous tile's sums before
      // this tile's first MMA overwrites them -- and before this tile's
      // completion is signalled at all: a tile without items here signals at
      // once, and two completions ahead of the readers would alias the
      // parity they wait on.
      if (kt > 0 && !(ok = warp_all(mbar_wait(bar(kDkvBarAccFree), (kt - 1) & 1, wait_ns)))) break;
      for (int li = 0; li < ti.n_it; ++li, ++gi) {
        const int s = gi % NS;
        if (!(ok = warp_all(mbar_wait(bar(kDkvBarP), gi & 1, wait_ns)))) break;
        tc_fence_after();
        const uint64_t qm = desc_add(dQm0, s * Cf::kStageBytes), om = desc_add(qm, Cf::kQBytes);
        // P^T / dS^T of queries 16k..16k+15: 8 packed columns at 8k.
#pragma unroll
        for (int q4 = 0; q4 < TM / 64; ++q4) {
          const uint32_t acc = (li > 0 || q4 > 0) ? 1u : 0u;
          const uint32_t p = tP + q4 * Cf::kGrp;
          const uint64_t b = desc_add(om, q4 * 8192);
          mma_ts_x4(tDV, p, p + 8, p + 16, p + 24, b, desc_add(b, 2048), desc_add(b, 4096),
                    desc_add(b, 6144), kIdAcc, acc);
        }
        if constexpr (D == 128) {
          // dV has read P^T (the next S^T may go there); dS^T is written
          // separately, after P^T.
          mma_commit(bar(kDkvBarFree));
          if (!(ok = warp_all(mbar_wait(bar(kDkvBarP + 1), gi & 1, wait_ns)))) break;
          tc_fence_after();
        }
#pragma unroll
        for (int q4 = 0; q4 < TM / 64; ++q4) {
          const uint32_t acc = (li > 0 || q4 > 0) ? 1u : 0u;
          const uint32_t p = tDS + q4 * Cf::kGrp;
          const uint64_t b = desc_add(qm, q4 * 8192);
          mma_ts_x4(tDK, p, p + 8, p + 16, p + 24, b, desc_add(b, 2048), desc_add(b, 4096),
                    desc_add(b, 6144), kIdAcc, acc);
        }
        // Both MMA streams of item gi have read stage s (the S^T stream
        // finished before the element-wise warps released P): free it, and the
        // P^T / dS^T columns (D = 128: the dS^T ones, where dP^T goes next).
        mma_commit(bar(kDkvBarQEmpty + s));
        mma_commit(bar(D == 64 ? kDkvBarFree : kDkvBarFree + 1));
      }
      if (!ok) break;
      mma_commit(bar(kDkvBarAcc));  // this tile's sums (at once when it has no items)
    }
    mma_commit(bar(kDkvBarDrainAcc));
    warp_all(mbar_wait(bar(kDkvBarDrainAcc), 0, wait_ns));
  } else if (C > 1) {
    // ------------------------------------------------------------ receive-region release
    // After every tile but the last, once the element-wise warps have read
    // the peers' sums, each peer is told it may send the next tile's: a
    // remote arrival holds the issuing warp for about half a microsecond.
    for (int kt = 0; ok; ++kt) {
      if (tile_of(kt) < 0 || !shared_next(kt)) break;
      if (!(ok = warp_all(mbar_wait(bar(kDkvBarRecvRead), kt & 1, wait_ns)))) break;
      if (lane == 0) {
        for (int p = 0; p < C; ++p)
          if (p != crank)
            mbar_arrive_remote(map_shared_rank(bar(kDkvBarRegionFree), static_cast<uint32_t>(p)));
      }
      __syncwarp();
    }
  }
  } else {
    setmaxnreg_inc<kDkwElemRegs>();
    // ------------------------------------------------------------ P^T / dS^T warps
    // Warps w and w + 4 share TMEM lane quarter (w & 3), i.e. the same 32 key
    // rows; group grp = (w - 4) / 4 takes queries 64 grp .. 64 grp + 63 of
    // each item, and columns 32 grp .. of dV, dK in the tile epilogue.
    const int quarter = warp & 3;
    const int grp = (warp - 4) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    const int owner = r / R;  // block of the cluster that stores key row r
    int gi = 0;
    for (int kt = 0; ok; ++kt) {
      const int t = tile_of(kt);
      if (t < 0) break;
      const DkvTile ti = tile_info(t, kt < n_sh);
      const int krow = ti.n0 + r;
      int m_idx = ti.n_it > 0 ? ti.it_lo % ti.per_head : 0;  // query tile of the item in its head
      for (int li = 0; li < ti.n_it && ok; ++li, ++gi) {
        const int s = gi % NS;
        const int i0 = (ti.m_begin + m_idx) * TM + grp * 64;  // this group's first query
        if (++m_idx == ti.per_head) m_idx = 0;
        // Causal: query i0 + c sees key krow iff c >= krow - off - i0.  The
        // warp's rows span 32 keys: columns below the smallest row's bound
        // need no mask, chunks of 32 columns below the largest row's bound
        // are all zero.  (-lse2, -delta) of this group's queries: two per
        // float4 at st4.
        auto cmin_of = [&] { return a.causal ? (krow - ti.off - i0) : -1; };
        auto wmin_of = [&] { return ti.n0 + quarter * 32 - ti.off - i0; };  // smallest row's bound
        auto st4_of = [&] { return stage_base(s) + 2 * Cf::kQBytes + grp * 64 * 8; };
        if constexpr (D == 128) {
          // P^T first, from S^T alone, written over the S^T columns this
          // thread has read (the dV product starts on it); then dS^T, once
          // dP^T has landed, over the dP^T columns.  P stays in registers
          // (fp32) for dS.
          ok = warp_all(mbar_wait(bar(kDkvBarS), gi & 1, wait_ns));
          if (!ok) break;
          tc_fence_after();
          uint32_t pv[2][32];
#pragma unroll
          for (int c = 0; c < 2; ++c) tmem_ld32_nowait(tl + Cf::kColS + grp * 64 + 32 * c, pv[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 2; ++c) reg_fence32(pv[c]);
          const int cmin = cmin_of(), wmin = wmin_of();
          const bool warp_masked = a.causal && wmin + 31 > 0;
          const uint32_t st4 = st4_of();
          auto p_chunk = [&](auto ch_c, auto masked) {
            constexpr int ch = decltype(ch_c)::value;
            constexpr bool kMasked = decltype(masked)::value;
            uint32_t pk[16];
            if (kMasked && a.causal && 32 * ch + 31 < wmin) {
#pragma unroll
              for (int i = 0; i < 16; ++i) pk[i] = 0u;
#pragma unroll
              for (int i = 0; i < 32; ++i) pv[ch][i] = 0u;
            } else {
              static_for<16>([&](auto ic) {
                constexpr int c2 = decltype(ic)::value;
                constexpr int c = 2 * c2;
                const float4 rs = ld_shared_f4_at<(32 * ch + c) * 8>(st4);
                const float x0 = fmaf(__uint_as_float(pv[ch][c]), sl2, rs.x);
                const float x1 = fmaf(__uint_as_float(pv[ch][c + 1]), sl2, rs.z);
                float p0, p1;
                if constexpr ((c2 & 7) < kPolyOf8) {
                  p0 = exp2_poly(x0);
                  p1 = exp2_poly(x1);
                } else {
                  p0 = ex2_approx(x0);
                  p1 = ex2_approx(x1);
                }
                if constexpr (kMasked) {
                  if (32 * ch + c < cmin) p0 = 0.f;
                  if (32 * ch + c + 1 < cmin) p1 = 0.f;
                }
                pv[ch][c] = __float_as_uint(p0);
                pv[ch][c + 1] = __float_as_uint(p1);
                pk[c2] = pack_bf16x2(p0, p1);
              });
            }
            tmem_st16_nowait(tl + Cf::kColP + grp * Cf::kGrp + 16 * ch, pk);
          };
          if (warp_masked) {
            p_chunk(std::integral_constant<int, 0>{}, std::true_type{});
            p_chunk(std::integral_constant<int, 1>{}, std::true_type{});
          } else {
            p_chunk(std::integral_constant<int, 0>{}, std::false_type{});
            p_chunk(std::integral_constant<int, 1>{}, std::false_type{});
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kDkvBarP));
          ok = warp_all(mbar_wait(bar(kDkvBarS + 1), gi & 1, wait_ns));
          if (!ok) break;
          tc_fence_after();
          uint32_t dp[2][32];
#pragma unroll
          for (int c = 0; c < 2; ++c) tmem_ld32_nowait(tl + Cf::kColDP + grp * 64 + 32 * c, dp[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 2; ++c) reg_fence32(dp[c]);
          auto ds_chunk = [&](auto ch_c) {
            constexpr int ch = decltype(ch_c)::value;
            uint32_t dk[16];
            if (warp_masked && 32 * ch + 31 < wmin) {
#pragma unroll
              for (int i = 0; i < 16; ++i) dk[i] = 0u;
            } else {
              static_for<16>([&](auto ic) {
                constexpr int c2 = decltype(ic)::value;
                constexpr int c = 2 * c2;
                const float4 rs = ld_shared_f4_at<(32 * ch + c) * 8>(st4);
                const float d0 = __uint_as_float(pv[ch][c]) * (__uint_as_float(dp[ch][c]) + rs.y);
                const float d1 =
                    __uint_as_float(pv[ch][c + 1]) * (__uint_as_float(dp[ch][c + 1]) + rs.w);
                dk[c2] = pack_bf16x2(d0, d1);
              });
            }
            tmem_st16_nowait(tl + Cf::kColDS + grp * Cf::kGrp + 16 * ch, dk);
          };
          ds_chunk(std::integral_constant<int, 0>{});
          ds_chunk(std::integral_constant<int, 1>{});
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kDkvBarP + 1));
          continue;
        }
        ok = warp_all(mbar_wait(bar(kDkvBarS), gi & 1, wait_ns));
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[2][32], dp[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_ld32_nowait(tl + Cf::kColS + grp * 64 + 32 * c, sv[c]);
          tmem_ld32_nowait(tl + Cf::kColDP + grp * 64 + 32 * c, dp[c]);
        }
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          reg_fence32(sv[c]);
          reg_fence32(dp[c]);
        }
        // S^T, dP^T are in registers: the next item's may overwrite them (at
        // D = 128 only after this item's dV, dK products, which its issuer
        // waits for).
        tc_fence_before();
        __syncwarp();
        if (D == 64 && lane == 0) mbar_arrive(bar(kDkvBarSFree));
        const int cmin = cmin_of(), wmin = wmin_of();
        const bool warp_masked = a.causal && wmin + 31 > 0;
        const uint32_t st4 = st4_of();
        // The previous item's dV, dK MMAs must be done with the P^T, dS^T
        // columns before this item's go there.
        bool freed = gi == 0;
        auto chunk = [&](auto ch_c, auto masked) -> bool {
          constexpr int ch = decltype(ch_c)::value;
          constexpr bool kMasked = decltype(masked)::value;
          uint32_t pk[16], dk[16];
          if (kMasked && a.causal && 32 * ch + 31 < wmin) {
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = dk[i] = 0u;
          } else {
            static_for<16>([&](auto ic) {
              constexpr int c2 = decltype(ic)::value;
              constexpr int c = 2 * c2;
              // (-lse2_c, -delta_c, -lse2_c+1, -delta_c+1), the same for the whole warp
              const float4 rs = ld_shared_f4_at<(32 * ch + c) * 8>(st4);
              const float x0 = fmaf(__uint_as_float(sv[ch][c]), sl2, rs.x);
              const float x1 = fmaf(__uint_as_float(sv[ch][c + 1]), sl2, rs.z);
              float p0, p1;
              if constexpr ((c2 & 7) < kPolyOf8) {
                p0 = exp2_poly(x0);
                p1 = exp2_poly(x1);
              } else {
                p0 = ex2_approx(x0);
                p1 = ex2_approx(x1);
              }
              if constexpr (kMasked) {
                if (32 * ch + c < cmin) p0 = 0.f;
                if (32 * ch + c + 1 < cmin) p1 = 0.f;
              }
              const float d0 = p0 * (__uint_as_float(dp[ch][c]) + rs.y);
              const float d1 = p1 * (__uint_as_float(dp[ch][c + 1]) + rs.w);
              pk[c2] = pack_bf16x2(p0, p1);
              dk[c2] = pack_bf16x2(d0, d1);
            });
          }
          if constexpr ((MODE & kDkvStoreDs) != 0) {
            // Stored-dS backward: this item's dS^T rows also go to the
            // workspace, for the dQ step to read instead of recomputing them
            // (row = 64 queries of one half of the 128-query tile).
            const int it = ti.it_lo + li;
            const int h = ti.g * G + it / ti.per_head;
            const int mt = ti.m_begin + it % ti.per_head, kt2 = ti.n0 / kTileN;
            const long pr = a.causal ? static_cast<long>(mt) * (mt + 1) / 2 + kt2
                                     : static_cast<long>(mt) * a.n_tiles + kt2;
            const size_t row =
                (((static_cast<size_t>(ti.b) * a.Hq + h) * a.ds_pairs + pr) * 2 + grp) * kTileN + r;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.ds) + row * 64 + 32 * ch);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(dk[4 * i], dk[4 * i + 1], dk[4 * i + 2], dk[4 * i + 3]);
          }
          if (!freed) {
            if (!warp_all(mbar_wait(bar(kDkvBarFree), (gi - 1) & 1, wait_ns))) return false;
            tc_fence_after();
            freed = true;
          }
          tmem_st16_nowait(tl + Cf::kColP + grp * Cf::kGrp + 16 * ch, pk);
          tmem_st16_nowait(tl + Cf::kColDS + grp * Cf::kGrp + 16 * ch, dk);
          return true;
        };
        if (warp_masked)
          ok = chunk(std::integral_constant<int, 0>{}, std::true_type{}) &&
               chunk(std::integral_constant<int, 1>{}, std::true_type{});
        else
          ok = chunk(std::integral_constant<int, 0>{}, std::false_type{}) &&
               chunk(std::integral_constant<int, 1>{}, std::false_type{});
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kDkvBarP));
      }
      if (!ok) break;

      // ---------------------------------------------------------- tile epilogue
      // This thread's share of key row r: D/2 columns of dV and of dK (zero
      // for a block without items in the tile).
      ok = warp_all(mbar_wait(bar(kDkvBarAcc), kt & 1, wait_ns));
      if (!ok) break;
      if constexpr (D == 128) {
        // One block per tile: dV, then dK, from TMEM straight to memory.
        tc_fence_after();
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          uint32_t part[2][32];
          if (ti.n_it > 0) {
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tmem_ld32_nowait(tl + (which == 0 ? Cf::kColDV : Cf::kColDK) + grp * 64 + 32 * c, part[c]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 2; ++c) reg_fence32(part[c]);
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) part[i >> 5][i & 31] = 0u;
          }
          if (which == 1) {
            // The next tile's first dV, dK MMA may overwrite the accumulators.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kDkvBarAccFree));
          }
          if (krow < ti.tk) {
            const size_t rbase =
                ((static_cast<size_t>(ti.b) * a.Tk + ti.kbase + krow) * a.Hkv + ti.g) * D + grp * 64;
            const float mul = which == 0 ? 1.f : a.scale;
            uint4* dst =
                reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(which == 0 ? a.dv : a.dk) + rbase);
            auto f = [&](int i) { return __uint_as_float(part[i >> 5][i & 31]) * mul; };
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_uint4(pack_bf16x2(f(8 * i), f(8 * i + 1)), pack_bf16x2(f(8 * i + 2), f(8 * i + 3)),
                                  pack_bf16x2(f(8 * i + 4), f(8 * i + 5)),
                                  pack_bf16x2(f(8 * i + 6), f(8 * i + 7)));
          }
        }
        continue;
      }
      uint32_t part_v[D / 2], part_k[D / 2];
      if (ti.n_it > 0) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tmem_ld32_nowait(tl + Cf::kColDV + grp * (D / 2) + 32 * c,
                           *reinterpret_cast<uint32_t(*)[32]>(part_v + 32 * c));
          tmem_ld32_nowait(tl + Cf::kColDK + grp * (D / 2) + 32 * c,
                           *reinterpret_cast<uint32_t(*)[32]>(part_k + 32 * c));
        }
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(part_v + 32 * c));
          reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(part_k + 32 * c));
        }
      } else {
#pragma unroll
        for (int i = 0; i < D / 2; ++i) part_v[i] = part_k[i] = 0u;
      }
      // The next tile's first dV, dK MMA may overwrite the accumulators.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kDkvBarAccFree));

      const bool sh = kt < n_sh;
      if (Cf::kMaxCluster > 1 && C > 1 && sh) {
        // Rows another block owns: to its receive region, once it has read
        // the previous tile's.
        if (kt > 0) {
          ok = warp_all(mbar_wait(bar(kDkvBarRegionFree), (kt - 1) & 1, wait_ns));
          if (!ok) break;
        }
        if (owner != crank) {
          const int j = crank < owner ? crank : crank - 1;
          const int row = j * R + (r - owner * R);
          const uint32_t dst = map_shared_rank(s0 + Cf::kOffRecv, static_cast<uint32_t>(owner));
          const uint32_t rbar = map_shared_rank(bar(kDkvBarRecv), static_cast<uint32_t>(owner));
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const uint32_t* v = which == 0 ? part_v : part_k;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
              const int chunk16 = (which * D + grp * (D / 2)) / 4 + i;
              st_async_f4(dst + slot_off(row, chunk16),
                          make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                      __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])),
                          rbar);
            }
          }
        }
        // Own rows: this block's sums, then the peers' in rank order.
        ok = warp_all(mbar_wait(bar(kDkvBarRecv), kt & 1, wait_ns));
        if (!ok) break;
        // Arm the receive mbarrier for the next tile's sums.  Peers send them
        // only after every warp here has signalled (below, after this arm in
        // program order), and until then the barrier cannot move past the
        // phase the other warps are still checking.
        if (warp == 4 && lane == 0 && shared_next(kt))
          mbar_arrive_expect_tx(bar(kDkvBarRecv), recv_bytes);
        if (owner == crank) {
          const int rl = r - crank * R;
          for (int src = 0; src < C; ++src) {
            if (src == crank) continue;
            const int j = src < crank ? src : src - 1;
            const uint32_t slot = s0 + Cf::kOffRecv;
            const int row = j * R + rl;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
              const float4 x = ld_shared_f4(slot + slot_off(row, (grp * (D / 2)) / 4 + i));
              const float4 y = ld_shared_f4(slot + slot_off(row, (D + grp * (D / 2)) / 4 + i));
              part_v[4 * i] = __float_as_uint(__uint_as_float(part_v[4 * i]) + x.x);
              part_v[4 * i + 1] = __float_as_uint(__uint_as_float(part_v[4 * i + 1]) + x.y);
              part_v[4 * i + 2] = __float_as_uint(__uint_as_float(part_v[4 * i + 2]) + x.z);
              part_v[4 * i + 3] = __float_as_uint(__uint_as_float(part_v[4 * i + 3]) + x.w);
              part_k[4 * i] = __float_as_uint(__uint_as_float(part_k[4 * i]) + y.x);
              part_k[4 * i + 1] = __float_as_uint(__uint_as_float(part_k[4 * i + 1]) + y.y);
              part_k[4 * i + 2] = __float_as_uint(__uint_as_float(part_k[4 * i + 2]) + y.z);
              part_k[4 * i + 3] = __float_as_uint(__uint_as_float(part_k[4 * i + 3]) + y.w);
            }
          }
        }
        // This block's receive region is read: the peers may send the next
        // tile's sums (warp 3 tells them, off these warps' path; after the
        // last tile nothing more is sent).
        __syncwarp();
        if (lane == 0 && shared_next(kt)) mbar_arrive(bar(kDkvBarRecvRead));
      }
      if ((owner == crank || !sh) && krow < ti.tk) {
        const size_t rbase =
            ((static_cast<size_t>(ti.b) * a.Tk + ti.kbase + krow) * a.Hkv + ti.g) * D + grp * (D / 2);
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t* v = which == 0 ? part_v : part_k;
          const float mul = which == 0 ? 1.f : a.scale;
          uint4* dst = reinterpret_cast<uint4*>(
              static_cast<__nv_bfloat16*>(which == 0 ? a.dv : a.dk) + rbase);
          auto f = [&](int i) { return __uint_as_float(v[i]) * mul; };
#pragma unroll
          for (int i = 0; i < D / 16; ++i)
            dst[i] = make_uint4(pack_bf16x2(f(8 * i), f(8 * i + 1)), pack_bf16x2(f(8 * i + 2), f(8 * i + 3)),
                                pack_bf16x2(f(8 * i + 4), f(8 * i + 5)),
                                pack_bf16x2(f(8 * i + 6), f(8 * i + 7)));
        }
      }
    }
  }

  // No block may exit while a peer can still store into its shared memory or
  // arrive on its mbarriers: every block reaches this barrier (no early exit;
  // all waits above are bounded).  Every such store and arrival has landed
  // before its target block arrives here (its waits on them come first), so
  // the barrier orders nothing else: its arrival is relaxed and need not wait
  // for this block's dV, dK stores.
  if (C > 1) {
    __syncwarp();
    cluster_sync_relaxed();
  }

  if (!ok) atomicOr(&g_bwd_status, 2u);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================== dQ
// Work unit: one 128-query tile of one (b, query head), over 128-key tiles
// 0..diagonal in ascending order.  Persistent, one pipeline per SM, working
// through units it takes, heaviest first, from a counter in the workspace (or,
// without one, the units the host dealt it):
//   warp 0      TMA producer: each unit's Q and dO (two slots at D = 64, so
//               the next unit's load runs ahead), K_j and V_j into a ring
//   warp 1      tcgen05 issuer: S_j = Q K_j^T and dP_j = dO V_j^T (both
//               operands in shared memory, N = 128) as soon as the
//               element-wise warps hold S_{j-1}, dP_{j-1} in registers; then
//               dQ += dS_{j-1} K_{j-1} with dS read from TMEM
//   warps 4..11 element-wise, two threads per query row (TMEM lane), one per
//               64-key half: P = 2^(S scale log2e - LSE log2e), dS = P (dP -
//               Delta) as packed bf16 into TMEM columns of their own; at the
//               unit's end dQ = scale * (sum over key tiles) to bf16.
// TMEM: S [128 fp32 columns], dP [128], dS [64 columns of bf16 pairs], dQ [D].
// Every dQ row is summed by one block over its key tiles in ascending order.
// Warps 0..3 (one warpgroup): producer, MMA issuer, two idle; warps 4..11 (two
// warpgroups): element-wise.  The first warpgroup hands registers to the
// other two, whose threads each hold 64 scores and 64 dP values.
constexpr int kDqWarps = 12;
constexpr int kDqThreads = kDqWarps * 32;
constexpr uint32_t kDqCtrlRegs = 88, kDqElemRegs = 192;
constexpr int kDqRegBudget = 128 * kDqCtrlRegs + 256 * kDqElemRegs;
template <int D>
struct DqCfg {
  static constexpr int kAtoms = D / 64;
  static constexpr int kQBytes = kTileM * 128 * kAtoms;     // 128 queries x D
  static constexpr int kKvBytes = kDqTileN * 128 * kAtoms;  // 128 keys x D
  static constexpr int kQSlots = (D == 64) ? 2 : 1;         // Q, dO pairs
  // K stays until its tile's dQ MMA (late), V only until dP: K gets the
  // deeper ring.
  static constexpr int kKStages = 3;
  static constexpr int kVStages = (D == 64) ? 3 : 2;
  static constexpr int kOffQ = 0;  // slot i: Q at 2 i kQBytes, dO at (2 i + 1) kQBytes
  static constexpr int kOffK = 2 * kQSlots * kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKvBytes;
  // The unit's 128 row statistics (-LSE log2e, -Delta), one KB per slot,
  // loaded with its Q and dO.
  static constexpr int kOffRs = kOffV + kVStages * kKvBytes;
  // At D = 64, each element-wise warp's 32 rows x 32 columns of dQ are staged
  // here (2 KB per warp) for one TMA store.
  static constexpr bool kStageDq = (D == 64);
  static constexpr int kOffStage = kOffRs + kQSlots * 1024;
  static constexpr int kSmemBytes = kOffStage + (kStageDq ? 8 * 2048 : 0) + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDS = 256, kColDQ = 320;
  static_assert(kColDQ + D <= kTmemCols, "TMEM layout");
  static_assert(kSmemBytes + 512 <= 227 * 1024, "shared memory per block");
};
constexpr int kDqMaxStages = 3;

enum : int { kDqBarQFull = 0,                       // [2] Q, dO slot loaded
             kDqBarQFree = 2,                       // [2] the unit's S, dP MMAs are done with the slot
             kDqBarKFull = 4, kDqBarKEmpty = 7,     // [3]
             kDqBarVFull = 10, kDqBarVEmpty = 13,   // [3]
             kDqBarS = 16,        // S_j, dP_j are in TMEM
             kDqBarSFree = 17,    // element-wise warps hold S_j, dP_j in registers (8)
             kDqBarDS = 18,       // dS_j is in TMEM (8)
             kDqBarDSFree = 19,   // the dQ MMAs of tile j are done with dS
             kDqBarAcc = 20,      // the unit's last dQ MMA has finished
             kDqBarDrain = 21,
             kDqBarUnit = 22,     // [4] unit k published in ring slot k % 4
             kDqBarUnitFree = 26, // [4] ring slot k % 4 read by the MMA and element-wise warps (9)
             kDqBarRsRead = 30,   // [2] the element-wise warps hold the slot's row statistics (8)
             kDqNumBars = 32 };

template <int D, class VT>
__global__ void __launch_bounds__(kDqThreads, 1)
    attn_dq_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                   const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mdO,
                   const __grid_constant__ CUtensorMap mdQ, const BwdArgs a,
                   const __grid_constant__ QTileSched sched, const __grid_constant__ VT vt) {
  using C = DqCfg<D>;
  constexpr bool VL = std::is_same<VT, VarlenTable>::value;
  constexpr int NK = C::kKStages, NV = C::kVStages;
  constexpr int NQ = C::kQSlots;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kDqNumBars];
  __shared__ uint32_t tmem_slot;
  __shared__ int unit_ring[4];

  const int warp = static_cast<int>(threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int pipe_id = static_cast<int>(blockIdx.x);
  const int kv_tiles = (a.T + kDqTileN - 1) / kDqTileN;
  int first = pipe_id, n_units;
  if (sched.n_listed > 0) {
    first = sched.start[pipe_id];
    n_units = sched.start[pipe_id + 1] - first;
  } else {
    const int total = (VL ? vt_tiles(vt) : a.n_tiles) * a.BH;
    n_units = qtile_snake_count(pipe_id, total, sched.n_pipes);
  }
  auto u_of = [&](int k) {
    return sched.n_listed > 0 ? static_cast<int>(sched.unit[first + k])
                              : qtile_snake_unit(pipe_id, k, sched.n_pipes);
  };
  // Units are numbered heaviest first.  With a.unit_counter, the producer
  // takes the next unit from that counter whenever it is ready for one, so
  // blocks that start early (on SMs another kernel frees first) take the
  // heaviest units; otherwise it follows the host's deal.  Either way it
  // passes unit k (or -1 after the last) to the other warps in ring slot
  // k % 4.  Which block computes a unit does not change any bit of its result.
  const int n_all = (VL ? vt_tiles(vt) : a.n_tiles) * a.BH;
  // Rows relative to the unit's sequence, as in the forward: queries from row
  // qbase, keys from kbase, row statistics from rbase; key j visible to
  // query i iff j < tk and (causal) j <= i + off.
  struct Unit { int b, h, hkv, m0, n_kv, qbase, kbase, rbase, tq, tk, off; };
  auto unit_info = [&](int u) {
    Unit t;
    if constexpr (VL) {
      const uint32_t e = vt_tile(vt, u / a.BH);
      const int s = static_cast<int>(e >> 16);
      t.b = 0;
      t.h = u % a.BH;
      t.m0 = static_cast<int>(e & 0xFFFFu) * kTileM;
      t.qbase = vt_cu_q(vt, s);
      t.tq = vt_cu_q(vt, s + 1) - t.qbase;
      t.kbase = vt_cu_k(vt, s);
      t.tk = vt_cu_k(vt, s + 1) - t.kbase;
      t.rbase = vt_ps(vt, s);
      t.off = t.tk - t.tq;
      const int tiles = (t.tk + kDqTileN - 1) / kDqTileN;
      const int last = min(t.m0 + kTileM - 1, t.tq - 1) + t.off;
      t.n_kv = a.causal ? (last < 0 ? 0 : min(tiles, last / kDqTileN + 1)) : tiles;
    } else {
      const int mt = a.n_tiles - 1 - u / a.BH;
      const int bh = u % a.BH;
      t.b = bh / a.Hq;
      t.h = bh % a.Hq;
      t.m0 = mt * kTileM;
      t.n_kv = a.causal ? min(kv_tiles, (t.m0 + kTileM) / kDqTileN) : kv_tiles;
      t.qbase = t.kbase = t.rbase = 0;
      t.tq = t.tk = a.T;
      t.off = 0;
    }
    t.hkv = t.h / (a.Hq / a.Hkv);
    return t;
  };

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sQ0 = s0 + C::kOffQ, sK0 = s0 + C::kOffK, sV0 = s0 + C::kOffV;
  const uint32_t sRs = s0 + C::kOffRs, sStage = s0 + C::kOffStage;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (warp == 1 && lane == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kDqBarQFull + i), 1);
      mbar_init(bar(kDqBarQFree + i), 1);
      mbar_init(bar(kDqBarRsRead + i), 8);
    }
    for (int s = 0; s < kDqMaxStages; ++s) {
      mbar_init(bar(kDqBarKFull + s), 1);
      mbar_init(bar(kDqBarKEmpty + s), 1);
      mbar_init(bar(kDqBarVFull + s), 1);
      mbar_init(bar(kDqBarVEmpty + s), 1);
    }
    mbar_init(bar(kDqBarS), 1);
    mbar_init(bar(kDqBarSFree), 8);
    mbar_init(bar(kDqBarDS), 8);
    mbar_init(bar(kDqBarDSFree), 1);
    mbar_init(bar(kDqBarAcc), 1);
    mbar_init(bar(kDqBarDrain), 1);
    for (int k = 0; k < 4; ++k) {
      mbar_init(bar(kDqBarUnit + k), 1);
      mbar_init(bar(kDqBarUnitFree + k), 9);
    }
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&mQ);
    tma_prefetch_desc(&mK);
    tma_prefetch_desc(&mV);
    tma_prefetch_desc(&mdO);
    tma_prefetch_desc(&mdQ);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint64_t wait_ns = a.wait_ns;
  bool ok = true;
  // Unit k, for the MMA and element-wise warps (whole warp; -1 after the
  // last unit, or when the wait runs out with ok false).  The slot is handed
  // back once read.
  auto read_unit = [&](int k) -> int {
    if (!(ok = warp_all(mbar_wait(bar(kDqBarUnit + (k & 3)), (k >> 2) & 1, wait_ns)))) return -1;
    const int u = unit_ring[k & 3];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kDqBarUnitFree + (k & 3)));
    return u;
  };

  if (warp < 4) {
  // Each warpgroup changes its register count at the top of its own branch,
  // so the code after it is compiled for the new count.
  setmaxnreg_dec<kDqCtrlRegs>();
  if (warp == 0) {
    if (lane == 0) {
      int last_k[kDqMaxStages] = {-1, -1, -1}, last_v[kDqMaxStages] = {-1, -1, -1};
      int last_q[2] = {-1, -1};
      int ku = 0;  // units published so far
      // Takes the next unit (from the counter or the host's deal) and
      // publishes it in ring slot ku % 4 once that slot has been read for
      // unit ku - 4; -1 after the last.
      auto take = [&]() -> int {
        if (ku >= 4 && !(ok = mbar_wait(bar(kDqBarUnitFree + (ku & 3)), ((ku >> 2) - 1) & 1, wait_ns)))
          return -1;
        int u;
        if (a.unit_counter != nullptr) {
          const unsigned v = atomicAdd(a.unit_counter, 1u);
          u = v < static_cast<unsigned>(n_all) ? static_cast<int>(v) : -1;
          // A cleared counter never passes n_all plus one per block: a larger
          // value means it was not cleared before this launch.
          if (v >= static_cast<unsigned>(n_all) + gridDim.x) atomicOr(&g_bwd_status, 16u);
        } else {
          u = ku < n_units ? u_of(ku) : -1;
        }
        unit_ring[ku & 3] = u;
        mbar_arrive(bar(kDqBarUnit + (ku & 3)));
        ++ku;
        if (u < 0 && a.unit_counter != nullptr) {
          // Count this block out (second word); the last one to finish
          // taking units puts both words back to zero for the next launch.
          __threadfence();
          if (atomicAdd(a.unit_counter + 1, 1u) == gridDim.x - 1) {
            atomicExch(a.unit_counter, 0u);
            atomicExch(a.unit_counter + 1, 0u);
          }
        }
        return u;
      };
      // Q, dO and the row statistics of the ne-th unit with key tiles into
      // slot ne % NQ, once the unit that last used the slot is done with it:
      // its S, dP products have read Q and dO, and the element-wise warps
      // hold its row statistics (they wait on the slot's barrier later than
      // the MMA warp does; without this the barrier could complete twice
      // before their wait).
      auto issue_q = [&](const Unit& t, int ne) -> bool {
        const int slot = ne % NQ, use = ne / NQ;
        if (use > 0 && !(mbar_wait(bar(kDqBarQFree + slot), (use - 1) & 1, wait_ns) &&
                         mbar_wait(bar(kDqBarRsRead + slot), (use - 1) & 1, wait_ns)))
          return false;
        mbar_arrive_expect_tx(bar(kDqBarQFull + slot), 2 * C::kQBytes + 1024);
        const uint32_t sq = sQ0 + 2 * slot * C::kQBytes;
        for (int at = 0; at < C::kAtoms; ++at) {
          tma_load_4d(sq + at * (kTileM * 128), &mQ, bar(kDqBarQFull + slot), at * 64, t.h,
                      t.qbase + t.m0, t.b);
          tma_load_4d(sq + C::kQBytes + at * (kTileM * 128), &mdO, bar(kDqBarQFull + slot), at * 64,
                      t.h, t.qbase + t.m0, t.b);
        }
        bulk_load(sRs + slot * 1024,
                  a.rowstats + (static_cast<size_t>(t.b) * a.Hq + t.h) * a.Tp + t.rbase + t.m0, 1024,
                  bar(kDqBarQFull + slot));
        last_q[slot] = ne;
        return true;
      };
      int gj = 0;  // key tiles loaded so far, over all units
      int ne = 0;  // units with key tiles so far
      bool q_ahead = false;  // the current unit's Q was issued while the previous one loaded
      int u_next = take();
      while (ok && u_next >= 0) {
        const int u = u_next;
        const Unit t = unit_info(u);
        if (t.n_kv == 0) {  // a packed unit whose rows see no key: nothing to load
          u_next = take();
          continue;
        }
        if (!q_ahead && !(ok = issue_q(t, ne))) break;
        q_ahead = false;
        for (int j = 0; j < t.n_kv; ++j, ++gj) {
          const int sk = gj % NK, sv = gj % NV;
          if (gj >= NK && !(ok = mbar_wait(bar(kDqBarKEmpty + sk), ((gj / NK) & 1) ^ 1, wait_ns))) break;
          mbar_arrive_expect_tx(bar(kDqBarKFull + sk), C::kKvBytes);
          for (int at = 0; at < C::kAtoms; ++at)
            tma_load_4d(sK0 + sk * C::kKvBytes + at * (kDqTileN * 128), &mK, bar(kDqBarKFull + sk),
                        at * 64, t.hkv, t.kbase + j * kDqTileN, t.b);
          last_k[sk] = gj;
          if (gj >= NV && !(ok = mbar_wait(bar(kDqBarVEmpty + sv), ((gj / NV) & 1) ^ 1, wait_ns))) break;
          mbar_arrive_expect_tx(bar(kDqBarVFull + sv), C::kKvBytes);
          for (int at = 0; at < C::kAtoms; ++at)
            tma_load_4d(sV0 + sv * C::kKvBytes + at * (kDqTileN * 128), &mV, bar(kDqBarVFull + sv),
                        at * 64, t.hkv, t.kbase + j * kDqTileN, t.b);
          last_v[sv] = gj;
          if (j + 1 == t.n_kv) {
            // The next unit, taken once this unit's loads are all issued (a
            // block does not reserve work it cannot start soon: the counter
            // keeps dealing the heaviest units to whichever block is free
            // first); with two slots its Q, dO and row statistics load now.
            u_next = take();
            if (!ok) break;
            if (NQ == 2 && u_next >= 0) {
              const Unit tn = unit_info(u_next);
              if (tn.n_kv > 0) {
                if (!(ok = issue_q(tn, ne + 1))) break;
                q_ahead = true;
              }
            }
          }
        }
        ++ne;
      }
      if (!ok) {
        // Let every copy already issued land before the block's shared memory goes away.
        for (int i = 0; i < NQ; ++i)
          if (last_q[i] >= 0) mbar_wait(bar(kDqBarQFull + i), (last_q[i] / NQ) & 1, wait_ns);
        for (int s = 0; s < NK; ++s)
          if (last_k[s] >= 0) mbar_wait(bar(kDqBarKFull + s), (last_k[s] / NK) & 1, wait_ns);
        for (int s = 0; s < NV; ++s)
          if (last_v[s] >= 0) mbar_wait(bar(kDqBarVFull + s), (last_v[s] / NV) & 1, wait_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA issuer: the whole warp runs the loop (MMA issue is warp-collective);
    // every wait is made warp-uniform so the warp stays converged.
    const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP, tDS = tmem + C::kColDS,
                   tDQ = tmem + C::kColDQ;
    constexpr uint32_t kIdS = idesc_bf16(kTileM, kDqTileN, false, false);
    constexpr uint32_t kIdDQ = idesc_bf16(kTileM, D, false, true);
    // Operand descriptors built once; the loops only add constant offsets.
    const uint64_t dQ0 = sdesc_sw128(sQ0, 16, 1024);
    const uint64_t dK0 = sdesc_sw128(sK0, 16, 1024), dV0 = sdesc_sw128(sV0, 16, 1024);
    const uint64_t dKm0 = sdesc_sw128(sK0, kDqTileN * 128, 1024);  // K as MN-major B
    // S_g = Q K_g^T and dP_g = dO V_g^T, Q / dO from slot `slot`.
    auto issue_sdp = [&](int g, int slot) -> bool {
      const int sk = g % NK, sv = g % NV;
      if (!warp_all(mbar_wait(bar(kDqBarKFull + sk), (g / NK) & 1, wait_ns))) return false;
      tc_fence_after();
      const uint64_t dq = desc_add(dQ0, 2 * slot * C::kQBytes), ddo = desc_add(dq, C::kQBytes);
      const uint64_t dK = desc_add(dK0, sk * C::kKvBytes), dV = desc_add(dV0, sv * C::kKvBytes);
#pragma unroll
      for (int at = 0; at < C::kAtoms; ++at) {
        const uint64_t aq = desc_add(dq, at * (kTileM * 128)), b = desc_add(dK, at * (kDqTileN * 128));
        mma_ss_x4(tS, aq, desc_add(aq, 32), desc_add(aq, 64), desc_add(aq, 96), b, desc_add(b, 32),
                  desc_add(b, 64), desc_add(b, 96), kIdS, at > 0 ? 1u : 0u);
      }
      if (!warp_all(mbar_wait(bar(kDqBarVFull + sv), (g / NV) & 1, wait_ns))) return false;
      tc_fence_after();
#pragma unroll
      for (int at = 0; at < C::kAtoms; ++at) {
        const uint64_t ad = desc_add(ddo, at * (kTileM * 128)), b = desc_add(dV, at * (kDqTileN * 128));
        mma_ss_x4(tDP, ad, desc_add(ad, 32), desc_add(ad, 64), desc_add(ad, 96), b, desc_add(b, 32),
                  desc_add(b, 64), desc_add(b, 96), kIdS, at > 0 ? 1u : 0u);
      }
      mma_commit(bar(kDqBarS));
      mma_commit(bar(kDqBarVEmpty + sv));
      return true;
    };
    // dQ (+)= dS_g K_g: dS of key pair (2c, 2c + 1) in TMEM column c; K step
    // k (16 keys) reads columns 8k .. 8k + 7 and K rows 16k .. 16k + 15.
    auto issue_dq = [&](int g, bool first, bool last) -> bool {
      const int s = g % NK;
      if (!warp_all(mbar_wait(bar(kDqBarDS), g & 1, wait_ns))) return false;
      tc_fence_after();
      const uint64_t dKm = desc_add(dKm0, s * C::kKvBytes);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        mma_ts_x4(tDQ, tDS + 32 * h, tDS + 32 * h + 8, tDS + 32 * h + 16, tDS + 32 * h + 24,
                  desc_add(dKm, (4 * h) * 2048), desc_add(dKm, (4 * h + 1) * 2048),
                  desc_add(dKm, (4 * h + 2) * 2048), desc_add(dKm, (4 * h + 3) * 2048), kIdDQ,
                  (first && h == 0) ? 0u : 1u);
      mma_commit(bar(kDqBarKEmpty + s));
      mma_commit(bar(kDqBarDSFree));
      if (last) mma_commit(bar(kDqBarAcc));
      return true;
    };
    int gj = 0, ne = 0;
    int pend = -1;  // the key tile whose dQ MMA is still to be issued
    bool pend_first = false, pend_last = false;
    for (int ku = 0; ok; ++ku) {
      const int u = read_unit(ku);
      if (u < 0) break;
      const Unit t = unit_info(u);
      if (t.n_kv == 0) continue;
      const int slot = ne % NQ;
      // The previous unit's last dQ product goes first, so its epilogue never
      // waits behind this unit's Q load (with one Q slot that load cannot
      // even start before the previous unit's last S, dP).
      if (pend >= 0) {
        if (!(ok = issue_dq(pend, pend_first, pend_last))) break;
        pend = -1;
      }
      if (!(ok = warp_all(mbar_wait(bar(kDqBarQFull + slot), (ne / NQ) & 1, wait_ns)))) break;
      for (int j = 0; j < t.n_kv; ++j, ++gj) {
        // The score columns are free once the element-wise warps hold S, dP
        // of the previous tile.
        if (gj > 0 && !(ok = warp_all(mbar_wait(bar(kDqBarSFree), (gj - 1) & 1, wait_ns)))) break;
        if (!(ok = issue_sdp(gj, slot))) break;
        if (j + 1 == t.n_kv) mma_commit(bar(kDqBarQFree + slot));
        if (pend >= 0 && !(ok = issue_dq(pend, pend_first, pend_last))) break;
        pend = gj;
        pend_first = (j == 0);
        pend_last = (j + 1 == t.n_kv);
      }
      ++ne;
    }
    if (ok && pend >= 0) ok = issue_dq(pend, pend_first, pend_last);
    mma_commit(bar(kDqBarDrain));
    warp_all(mbar_wait(bar(kDqBarDrain), 0, wait_ns));
  }
  } else {
    setmaxnreg_inc<kDqElemRegs>();
    // Element-wise warps: warps w and w + 4 share a TMEM lane quarter, i.e.
    // the same 32 query rows; half 0 takes keys 0..63 of each tile, half 1
    // keys 64..127.
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t tS = tl + C::kColS + 64 * half, tDP = tl + C::kColDP + 64 * half;
    const uint32_t tDS = tl + C::kColDS + 32 * half;
    const float sl2 = a.scale_log2;
    int gj = 0, ne = 0;
    for (int ku = 0; ok; ++ku) {
      const int u = read_unit(ku);
      if (u < 0) break;
      const Unit t = unit_info(u);
      const int qrow = t.m0 + r;
      // (-LSE*log2e, -Delta) of this row, loaded with the unit's Q and dO;
      // rows past T hold (-inf, -0): P = 0.
      float2 rstat = make_float2(0.f, 0.f);
      if (t.n_kv > 0) {
        const int slot = ne % NQ;
        ok = warp_all(mbar_wait(bar(kDqBarQFull + slot), (ne / NQ) & 1, wait_ns));
        if (!ok) break;
        rstat = ld_shared_f2(sRs + slot * 1024 + r * 8);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kDqBarRsRead + slot));
      }
      const int wlast = t.m0 + quarter * 32 + 31 + t.off;  // last key any row of the warp sees
      for (int j = 0; j < t.n_kv; ++j, ++gj) {
        ok = warp_all(mbar_wait(bar(kDqBarS), gj & 1, wait_ns));
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[2][32], dp[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_ld32_nowait(tS + 32 * c, sv[c]);
          tmem_ld32_nowait(tDP + 32 * c, dp[c]);
        }
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          reg_fence32(sv[c]);
          reg_fence32(dp[c]);
        }
        // S, dP are in registers: the next tile's may overwrite them.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kDqBarSFree));
        const int kv0 = j * kDqTileN + 64 * half;  // key of this half's first column
        // key kv0 + c visible iff c <= lim
        const int lim = a.causal ? min(qrow + t.off - kv0, t.tk - 1 - kv0) : (t.tk - 1 - kv0);
        // Masking only where the warp's rows meet the diagonal (or tk),
        // decided for the whole warp; 32-key chunks past every row of the
        // warp (or past tk) are all zeros.
        const bool need_mask = (a.causal && kv0 + 63 > wlast - 31) || kv0 + 64 > t.tk;
        const int last_key = a.causal ? min(wlast, t.tk - 1) : t.tk - 1;
        const int live = last_key < kv0 ? 0 : min(2, (last_key - kv0) / 32 + 1);
        uint32_t dsk[32];
        auto element_loop = [&](auto masked) {
          constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            if (kMasked && ch >= live) {
#pragma unroll
              for (int i = 0; i < 16; ++i) dsk[16 * ch + i] = 0u;
              continue;
            }
            static_for<16>([&](auto ic) {
              constexpr int i = decltype(ic)::value;
              constexpr int c = 2 * i;  // column within the chunk
              const float x0 = fmaf(__uint_as_float(sv[ch][c]), sl2, rstat.x);
              const float x1 = fmaf(__uint_as_float(sv[ch][c + 1]), sl2, rstat.x);
              float p0, p1;
              if constexpr ((i & 7) < kPolyOf8) {
                p0 = exp2_poly(x0);
                p1 = exp2_poly(x1);
              } else {
                p0 = ex2_approx(x0);
                p1 = ex2_approx(x1);
              }
              if constexpr (kMasked) {
                if (32 * ch + c > lim) p0 = 0.f;
                if (32 * ch + c + 1 > lim) p1 = 0.f;
              }
              const float d0 = p0 * (__uint_as_float(dp[ch][c]) + rstat.y);
              const float d1 = p1 * (__uint_as_float(dp[ch][c + 1]) + rstat.y);
              dsk[16 * ch + i] = pack_bf16x2(d0, d1);
            });
          }
        };
        if (need_mask)
          element_loop(std::true_type{});
        else
          element_loop(std::false_type{});
        // The previous tile's dQ MMAs must be done reading the dS columns.
        if (gj > 0 && !(ok = warp_all(mbar_wait(bar(kDqBarDSFree), (gj - 1) & 1, wait_ns)))) break;
        tmem_st32_nowait(tDS, dsk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kDqBarDS));
      }
      if (!ok) break;
      const bool live_row = qrow < t.tq;
      uint32_t pkd[D / 4];
      if (t.n_kv > 0) {
        ok = warp_all(mbar_wait(bar(kDqBarAcc), ne & 1, wait_ns));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          const int c = half * (D / 64) + cc;  // this half's 32-column chunks of dQ
          uint32_t v[32];
          tmem_ld32(tl + C::kColDQ + c * 32, v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkd[16 * cc + i] = pack_bf16x2(__uint_as_float(v[2 * i]) * a.scale,
                                           __uint_as_float(v[2 * i + 1]) * a.scale);
        }
        // dQ is in registers: the next unit's first dQ MMA (issued after this
        // warp's next dS arrival) may overwrite it.
        tc_fence_before();
        ++ne;
      } else {
        // A packed unit whose rows see no key: dQ = 0.
#pragma unroll
        for (int i = 0; i < D / 4; ++i) pkd[i] = 0u;
      }
      // At D = 64 the warp's 32 rows x 32 columns go out through one TMA
      // store (rows past T are clipped by the map) unless they run past a
      // packed sequence's end, where the rows beyond belong to the next one.
      if (C::kStageDq && (!VL || t.m0 + quarter * 32 + 32 <= t.tq)) {
        const uint32_t stage = sStage + (warp - 4) * 2048;
        // The warp's previous store must have read the staging rows first.
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int i = 0; i < D / 16; ++i)
          st_shared_u4(stage + lane * (D / 2) * 2 + 16 * i,
                       make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_4d(&mdQ, stage, half * (D / 2), t.h, t.qbase + t.m0 + quarter * 32, t.b);
          bulk_commit_group();
        }
      } else if (live_row) {
        uint4* dst = reinterpret_cast<uint4*>(
            static_cast<__nv_bfloat16*>(a.dq) +
            ((static_cast<size_t>(t.b) * a.T + t.qbase + qrow) * a.Hq + t.h) * D + half * (D / 2));
#pragma unroll
        for (int i = 0; i < D / 16; ++i)
          dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
      }
    }
    // This block's units are done: whatever follows on the stream may start
    // its set-up (it waits for this grid to complete before reading).
    if (warp == 4 && lane == 0) griddep_launch_dependents();
    // Every store of dQ must be complete before the block (and its shared
    // memory) goes away.
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  // Launched as a programmatic dependent of the dK/dV step, this grid may run
  // beside it (it reads only the Delta step's results); it does not complete
  // before that grid has, so later work on the stream sees dk and dv too.
  if (threadIdx.x == 0) griddep_wait();
  if (!ok) atomicOr(&g_bwd_status, 4u);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_slot, C::kTmemCols);
  }
}

// Failure-detection self-test: one thread waits, with the same bounded wait
// the attention kernels use, on an mbarrier that nothing arrives on.  The wait
// runs out, the kernel records the timeout in the status word and returns; no
// asynchronous copy or MMA is in flight, so nothing else needs draining.
__global__ void wait_timeout_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  fence_barrier_init();
  if (!mbar_wait(smem_u32(&bar), 0, limit_ns)) atomicOr(&g_bwd_status, 8u);
}

// Sets the kernel's dynamic shared-memory limit once per device and context
// (the attribute belongs to the context's copy of the kernel, so a re-created
// context needs it again).  done[dev] holds the context id it was set for.
template <typename K>
cudaError_t set_smem_once(K kernel, int bytes, unsigned long long* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long ctx = current_context_id();
  if (dev >= 64 || ctx == 0 || done[dev] != ctx) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) done[dev] = current_context_id();
  }
  return cudaSuccess;
}

template <int D>
cudaError_t dkdv_max_clusters_t(int c, int* out) {
  static unsigned long long done[64] = {};
  cudaError_t e = set_smem_once(attn_dkdv_kernel<D, NoVarlen, 0>, DkvCfg<D>::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(c));
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = DkvCfg<D>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(c);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, attn_dkdv_kernel<D, NoVarlen, 0>, &cfg);
}

cudaError_t dkdv64_max_clusters(int c, int* out) {
  static unsigned long long done[64] = {};
  cudaError_t e = set_smem_once(attn_dkdvq_kernel<64, NoVarlen, 0>, DkwCfg<64>::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(c));
  cfg.blockDim = dim3(kDkwThreads);
  cfg.dynamicSmemBytes = DkwCfg<64>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(c);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, attn_dkdvq_kernel<64, NoVarlen, 0>, &cfg);
}

// The deal every launch without a list passes (n_blocks 0: the snake walk).
const DkvList& no_dkv_list() {
  static const DkvList none = [] {
    DkvList l;
    std::memset(&l, 0, sizeof(l));
    return l;
  }();
  return none;
}

template <int D, class VT, int MODE>
cudaError_t launch_dkdvq_t(int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const CUtensorMap& mdo, const BwdArgs& a,
                           bool dependent, const VT& vt, const DkvList& lst, cudaStream_t st) {
  static unsigned long long done[64] = {};
  cudaError_t e = set_smem_once(attn_dkdvq_kernel<D, VT, MODE>, DkwCfg<D>::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  // The block's registers at launch must cover the warpgroups' shares after
  // reallocation, or the element-wise warpgroups' increase never completes.
  static int regs_ok = 0;
  if (!regs_ok) {
    cudaFuncAttributes fa{};
    if ((e = cudaFuncGetAttributes(&fa, attn_dkdvq_kernel<D, VT, MODE>)) != cudaSuccess) return e;
    if (fa.numRegs * kDkwThreads < kDkwRegBudget) return cudaErrorInvalidConfiguration;
    regs_ok = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kDkwThreads);
  cfg.dynamicSmemBytes = DkwCfg<D>::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (a.cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(a.cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (dependent) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  e = cudaLaunchKernelEx(&cfg, attn_dkdvq_kernel<D, VT, MODE>, mq, mk, mv, mdo, a, vt, lst);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, class VT, int MODE>
cudaError_t launch_dkdv_t(int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                          const CUtensorMap& mv, const CUtensorMap& mdo, const BwdArgs& a,
                          bool dependent, const VT& vt, cudaStream_t st) {
  static unsigned long long done[64] = {};
  cudaError_t e = set_smem_once(attn_dkdv_kernel<D, VT, MODE>, DkvCfg<D>::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = DkvCfg<D>::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (a.cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(a.cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (dependent) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  e = cudaLaunchKernelEx(&cfg, attn_dkdv_kernel<D, VT, MODE>, mq, mk, mv, mdo, a, vt);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, class VT>
cudaError_t launch_dq_t(int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                        const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap& mdq,
                        const BwdArgs& a, const QTileSched& sched, const VT& vt, bool dependent,
                        cudaStream_t st) {
  static unsigned long long done[64] = {};
  cudaError_t e = set_smem_once(attn_dq_kernel<D, VT>, DqCfg<D>::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  // The block's registers at launch must cover the warpgroups' shares after
  // reallocation, or the element-wise warpgroups' increase never completes.
  static int regs_ok[2] = {0, 0};
  if (!regs_ok[D == 64 ? 0 : 1]) {
    cudaFuncAttributes fa{};
    if ((e = cudaFuncGetAttributes(&fa, attn_dq_kernel<D, VT>)) != cudaSuccess) return e;
    if (fa.numRegs * kDqThreads < kDqRegBudget) return cudaErrorInvalidConfiguration;
    regs_ok[D == 64 ? 0 : 1] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kDqThreads);
  cfg.dynamicSmemBytes = DqCfg<D>::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, attn_dq_kernel<D, VT>, mq, mk, mv, mdo, mdq, a, sched, vt);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_delta(const DeltaArgs& a, int sms, const VarlenTable* vt, cudaStream_t st) {
  // Persistent: kDeltaBlocksPerSm blocks per SM, fewer when there are fewer
  // batches of rows than warps.
  const int rows_per_batch = 4 * (256 / a.D);
  const long batches = (static_cast<long>(a.B) * a.T * a.Hq + rows_per_batch - 1) / rows_per_batch;
  const long want = std::max<long>(1, (batches + 7) / 8);
  const int grid = static_cast<int>(std::min<long>(want, static_cast<long>(sms) * kDeltaBlocksPerSm));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (vt != nullptr) {
    e = a.D == 64 ? cudaLaunchKernelEx(&cfg, attn_delta_kernel<64, VarlenTable>, a, *vt)
                  : cudaLaunchKernelEx(&cfg, attn_delta_kernel<128, VarlenTable>, a, *vt);
  } else {
    const NoVarlen none{};
    e = a.D == 64 ? cudaLaunchKernelEx(&cfg, attn_delta_kernel<64, NoVarlen>, a, none)
                  : cudaLaunchKernelEx(&cfg, attn_delta_kernel<128, NoVarlen>, a, none);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_dkdv(int D, int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                        const CUtensorMap& mv, const CUtensorMap& mdo, const BwdArgs& a,
                        bool dependent, const VarlenTable* vt, const DkvList* list,
                        cudaStream_t st) {
  // D = 128: items of 128 queries with one block per key tile, items of 64
  // queries when a tile is split over a cluster.
  const DkvList& nl = no_dkv_list();
  if (list != nullptr) {
    // Only the walk of the 64-dim kernel without chunks takes a list.
    if (D != 64 || a.bg_chunk > 0 || list->n_blocks != grid || grid > kDkvListMaxBlocks ||
        (vt != nullptr && a.ds != nullptr))
      return cudaErrorInvalidValue;
    if (vt != nullptr)
      return launch_dkdvq_t<64, VarlenTable, 0>(grid, mq, mk, mv, mdo, a, dependent, *vt, *list, st);
    if (a.ds != nullptr)
      return launch_dkdvq_t<64, NoVarlen, kDkvStoreDs>(grid, mq, mk, mv, mdo, a, dependent, NoVarlen{},
                                                       *list, st);
    return launch_dkdvq_t<64, NoVarlen, 0>(grid, mq, mk, mv, mdo, a, dependent, NoVarlen{}, *list, st);
  }
  if (vt != nullptr) {
    if (D == 64)
      return launch_dkdvq_t<64, VarlenTable, 0>(grid, mq, mk, mv, mdo, a, dependent, *vt, nl, st);
    if (a.cluster == 1)
      return launch_dkdvq_t<128, VarlenTable, 0>(grid, mq, mk, mv, mdo, a, dependent, *vt, nl, st);
    return launch_dkdv_t<128, VarlenTable, 0>(grid, mq, mk, mv, mdo, a, dependent, *vt, st);
  }
  const NoVarlen none{};
  const int mode = (a.bg_chunk > 0 ? kDkvChunked : 0) | (a.ds != nullptr ? kDkvStoreDs : 0);
  auto go = [&](auto m) {
    constexpr int M = decltype(m)::value;
    if (D == 64)
      return launch_dkdvq_t<64, NoVarlen, M>(grid, mq, mk, mv, mdo, a, dependent, none, nl, st);
    if constexpr ((M & kDkvStoreDs) == 0) {
      if (a.cluster == 1)
        return launch_dkdvq_t<128, NoVarlen, M>(grid, mq, mk, mv, mdo, a, dependent, none, nl, st);
    }
    return launch_dkdv_t<128, NoVarlen, M>(grid, mq, mk, mv, mdo, a, dependent, none, st);
  };
  switch (mode) {
    case 0: return go(std::integral_constant<int, 0>{});
    case 1: return go(std::integral_constant<int, 1>{});
    case 2: return go(std::integral_constant<int, 2>{});
    default: return go(std::integral_constant<int, 3>{});
  }
}

cudaError_t dkdv_max_clusters(int D, int c, int* out) {
  *out = 0;
  if (D == 64) return dkdv64_max_clusters(c, out);
  if (D == 128) return dkdv_max_clusters_t<128>(c, out);
  return cudaErrorInvalidValue;
}
int dkdv_max_cluster_size(int D) { return D == 64 ? DkwCfg<64>::kMaxCluster : DkvCfg<128>::kMaxCluster; }

cudaError_t launch_dq(int D, int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                      const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap& mdq,
                      const BwdArgs& a, const QTileSched& sched, const VarlenTable* vt,
                      bool after_dkdv, cudaStream_t st) {
  if (vt != nullptr)
    return D == 64 ? launch_dq_t<64>(grid, mq, mk, mv, mdo, mdq, a, sched, *vt, after_dkdv, st)
                   : launch_dq_t<128>(grid, mq, mk, mv, mdo, mdq, a, sched, *vt, after_dkdv, st);
  const NoVarlen none{};
  return D == 64 ? launch_dq_t<64>(grid, mq, mk, mv, mdo, mdq, a, sched, none, after_dkdv, st)
                 : launch_dq_t<128>(grid, mq, mk, mv, mdo, mdq, a, sched, none, after_dkdv, st);
}

// Diagnostic: the kernels' 2^x forms on n inputs (polynomial scalar form,
// polynomial pair form, special-function unit).
__global__ void exp2_diag_kernel(const float* x, float* y_poly, float* y_pair, float* y_sfu,
                                 int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float x0 = x[i], x1 = (i + 1 < n) ? x[i + 1] : 0.f;
  float p0, p1;
  exp2_poly2(x0, x1, p0, p1);
  y_poly[i] = exp2_poly(x0);
  y_pair[i] = p0;
  y_sfu[i] = ex2_approx(x0);
  if (i + 1 < n) {
    y_poly[i + 1] = exp2_poly(x1);
    y_pair[i + 1] = p1;
    y_sfu[i + 1] = ex2_approx(x1);
  }
}

cudaError_t launch_exp2_diag(const float* x, float* y_poly, float* y_pair, float* y_sfu, int n,
                             cudaStream_t st) {
  const int pairs = (n + 1) / 2;
  exp2_diag_kernel<<<(pairs + 255) / 256, 256, 0, st>>>(x, y_poly, y_pair, y_sfu, n);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t st) {
  wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t take_bwd_status(cudaStream_t st, unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_bwd_status, sizeof(v), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v)
    e = cudaMemcpyToSymbolAsync(g_bwd_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  *out = v;
  return e;
}

}  // namespace detattn

// Fused causal grouped-query flash-attention forward for sm_103a.
//
// RustingBrain vs PyTorch/TensorFlow page, "Step 2: fused flash attention":
// one fused kernel replaces the causal softmax kernels and never writes the
// [seq_len, seq_len] score matrix.  "Step 1" names the per-row logsumexp the
// forward hands to the backward.
//
// Work unit: one 128-row query tile of one (batch, query head), walking
// 128-key tiles 0..diagonal in ascending order.  The kernel is persistent: a
// block holds NP pipelines (two at D = 64, one at D = 128), each with its own
// warps, shared memory, mbarriers and TMEM columns, and each pipeline works
// through the list of units the host dealt it (heaviest first, balanced per
// SM).  Per pipeline:
//   warp 0      TMA producer: each unit's Q into one of two slots (the next
//               unit's Q is issued right after this unit's first K, V tile),
//               K_j and V_j into a ring of two stages
//   warp 1      tcgen05 issuer: S_{j+1} = Q K_{j+1}^T as soon as the softmax
//               warps hold S_j in registers, then O += P_j V_j once they have
//               written P_j, so the tensor core computes the next scores
//               while the softmax works on this tile
//   warps 2..5  softmax, one thread per query row (TMEM lane) over all 128
//               keys of a tile: online softmax in base 2 with a lazily moved
//               maximum, P_j as packed bf16 into TMEM columns of its own (not
//               over S), O rescaled in TMEM when the maximum moves; at the
//               unit's end O / l and LSE = ln2 * (m + log2 l); each warp
//               stages its 32 rows of O in shared memory and stores them with
//               one asynchronous TMA copy, so the next unit starts at once
// TMEM per pipeline: S in 128 fp32 columns, P in 64 (bf16 pairs), O in D.
// Every hand-off is an mbarrier; each moves a whole 128 x 128 tile, so a
// softmax thread does 128 exponentials per wait.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "attn_launch.h"
#include "exp2_poly.cuh"
#include "sm103_ptx.cuh"

namespace detattn {

__device__ unsigned int g_fwd_status;

namespace {

// Warps 0..3 (one warpgroup) are the producer and MMA issuer of each
// pipeline (warps 2p and 2p + 1; with one pipeline warps 2, 3 idle); pipeline
// p's four softmax warps are warpgroup 1 + p, so warp w's TMEM lane quarter
// is w % 4 = its row quarter.
constexpr int kSoftWarps = 4;                  // one thread per query row
constexpr int kCtrlWarps = 4;
constexpr int fwd_threads(int D) { return 32 * (kCtrlWarps + kSoftWarps * fwd_pipes_per_block(D)); }
// With two pipelines the block has 384 threads: the control warpgroup hands
// registers to the softmax warpgroups, whose threads each hold a row of 128
// scores.  The launch must provide kRegBudget registers in all.
constexpr uint32_t kCtrlRegs = 56, kSoftRegs = 208;
constexpr int kRegBudget = 128 * kCtrlRegs + 256 * kSoftRegs;
constexpr int kBN = kFwdTileN;                 // keys per tile (128)
static_assert(kBN == 128 && kTileM == 128, "one thread holds one row of a 128 x 128 tile");
// The row maximum used in the exponent is only moved when the true maximum
// exceeds it by more than 2^8; until then P <= 256, which bf16 and the fp32
// accumulators hold exactly as well.  The final O / l and LSE are exact for
// any value of the stale maximum.
constexpr float kRescaleLog2 = 8.0f;
// Of every 8 consecutive pairs of scores, this many take 2^x from the FMA-pipe
// polynomial instead of the special-function unit.
#ifndef DETATTN_FWD_POLY_OF8
#define DETATTN_FWD_POLY_OF8 0
#endif
constexpr int kPolyOf8 = DETATTN_FWD_POLY_OF8;

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;                  // 128-byte swizzle atoms per row
  static constexpr int kQBytes = kTileM * 128 * kAtoms;  // 128 rows x D bf16
  static constexpr int kKvBytes = kBN * 128 * kAtoms;    // 128 rows x D bf16
  static constexpr int kStages = 2;
  static constexpr int kOffQ = 0;                        // two slots
  static constexpr int kOffK = 2 * kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKvBytes;
  static constexpr int kOffO = kOffV + kStages * kKvBytes;      // O staging: 128 rows x D
  static constexpr int kPipeBytes = kOffO + kQBytes;             // one pipeline (multiple of 1024)
  static constexpr int NP = fwd_pipes_per_block(D);
  static constexpr int kSmemBytes = NP * kPipeBytes + 1024;      // + alignment slack
  static constexpr uint32_t kTmemCols = (D == 64) ? 256 : 512;   // per pipeline
  static constexpr uint32_t kColS = 0;                   // S: 128 fp32 columns
  static constexpr uint32_t kColP = kBN;                 // P: 64 columns of bf16 pairs
  static constexpr uint32_t kColO = kBN + kBN / 2;       // O: D fp32 columns
  static_assert(kPipeBytes % 1024 == 0, "pipelines keep the 1024-byte swizzle alignment");
  static_assert(kColO + D <= kTmemCols, "S, P and O fit the pipeline's TMEM columns");
  static_assert(NP * kTmemCols <= 512, "TMEM holds every pipeline of the block");
  static_assert(kSmemBytes + 512 <= 227 * 1024, "dynamic + static shared memory fit one block");
};

enum : int {
  kBarQFull = 0,   // [2] Q slot loaded
  kBarQFree = 2,   // [2] the unit's Q K^T MMAs are done with the slot
  kBarKFull = 4,   // [2]
  kBarKEmpty = 6,  // [2]
  kBarVFull = 8,   // [2]
  kBarVEmpty = 10, // [2]
  kBarS = 12,      // S_j is in TMEM
  kBarSFree = 13,  // the softmax warps hold S_j in registers (4 arrivals)
  kBarP = 14,      // P_j is in TMEM, and everything the softmax read of O before (4 arrivals)
  kBarO = 15,      // O += P_j V_j has finished
  kBarDrain = 16,
  kNumBars = 17
};

__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

template <int D, class VT>
__global__ void __launch_bounds__(fwd_threads(D), 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mO,
                    const FwdArgs a,
                    const __grid_constant__ QTileSched sched, const __grid_constant__ VT vt) {
  using C = Cfg<D>;
  constexpr bool VL = std::is_same<VT, VarlenTable>::value;
  constexpr int NS = C::kStages;
  constexpr int NP = C::NP;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars_all[NP][kNumBars];
  __shared__ uint32_t tmem_slot;

  const int gwarp = static_cast<int>(threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  // Role: 0 producer, 1 MMA issuer, 2 softmax, -1 idle.
  const int pipe = gwarp < kCtrlWarps ? (gwarp >> 1) : (gwarp - kCtrlWarps) / kSoftWarps;
  const int warp = gwarp < kCtrlWarps ? (pipe < NP ? (gwarp & 1) : -1) : 2;
  const int pipe_id = static_cast<int>(blockIdx.x) * NP + (pipe < NP ? pipe : 0);
  const int kv_tiles = (a.T + kBN - 1) / kBN;
  // This pipeline's units: u_of(k) for k = 0 .. n_units - 1.
  int first = pipe_id, n_units;
  if (sched.n_listed > 0) {
    first = sched.start[pipe_id];
    n_units = sched.start[pipe_id + 1] - first;
  } else {
    const int total = (VL ? vt_tiles(vt) : a.n_m) * a.BHq;
    n_units = qtile_snake_count(pipe_id, total, sched.n_pipes);
  }
  auto u_of = [&](int k) {
    return sched.n_listed > 0 ? static_cast<int>(sched.unit[first + k])
                              : qtile_snake_unit(pipe_id, k, sched.n_pipes);
  };
  // A unit's query tile starts at row qbase + m0 of the tensor maps and its
  // keys at row kbase; it has tq query and tk key rows, and with the causal
  // mask query i sees key j iff j <= i + off, off = tk - tq (0 unless packed).
  struct Unit { int b, h, hkv, m0, n_kv, qbase, kbase, tq, tk, off; };
  auto unit_info = [&](int u) {
    Unit t;
    if constexpr (VL) {
      const uint32_t e = vt_tile(vt, u / a.Hq);
      const int s = static_cast<int>(e >> 16);
      t.b = 0;
      t.h = u % a.Hq;
      t.m0 = static_cast<int>(e & 0xFFFFu) * kTileM;
      t.qbase = vt_cu_q(vt, s);
      t.tq = vt_cu_q(vt, s + 1) - t.qbase;
      t.kbase = vt_cu_k(vt, s);
      t.tk = vt_cu_k(vt, s + 1) - t.kbase;
      t.off = t.tk - t.tq;
      const int tiles = (t.tk + kBN - 1) / kBN;
      // Keys up to the last visible one of the tile's last row.
      const int last = min(t.m0 + kTileM - 1, t.tq - 1) + t.off;
      t.n_kv = a.causal ? (last < 0 ? 0 : min(tiles, last / kBN + 1)) : tiles;
    } else {
      const int mt = a.n_m - 1 - u / a.BHq;
      const int bh = u % a.BHq;
      t.b = bh / a.Hq;
      t.h = bh % a.Hq;
      t.m0 = mt * kTileM;
      t.n_kv = a.causal ? min(kv_tiles, (t.m0 + kTileM) / kBN) : kv_tiles;
      t.qbase = t.kbase = 0;
      t.tq = t.tk = a.T;
      t.off = 0;
    }
    t.hkv = t.h / (a.Hq / a.Hkv);
    return t;
  };

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sP = smem_u32(smem) + (pipe < NP ? pipe : 0) * C::kPipeBytes;
  const uint32_t sQ0 = sP + C::kOffQ;
  const uint32_t sK0 = sP + C::kOffK;
  const uint32_t sV0 = sP + C::kOffV;
  const uint32_t sO = sP + C::kOffO;
  uint64_t* bars = bars_all[pipe < NP ? pipe : 0];
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x < 32) {
    tmem_alloc(smem_u32(&tmem_slot), NP * C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (warp == 1 && lane == 0) {  // each pipeline's MMA warp sets up its own barriers
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarQFull + i), 1);
      mbar_init(bar(kBarQFree + i), 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    mbar_init(bar(kBarS), 1);
    mbar_init(bar(kBarSFree), kSoftWarps);
    mbar_init(bar(kBarP), kSoftWarps);
    mbar_init(bar(kBarO), 1);
    mbar_init(bar(kBarDrain), 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&mQ);
    tma_prefetch_desc(&mK);
    tma_prefetch_desc(&mV);
    tma_prefetch_desc(&mO);
  }
  __syncthreads();
  tc_fence_after();
  // A kernel launched after this one as a programmatic dependent (the
  // backward's Delta step) may be scheduled now: it takes SMs as this grid's
  // blocks leave them and waits (griddepcontrol.wait) for this grid to
  // finish before it reads anything, so its launch latency hides under this
  // grid's tail.
  if (threadIdx.x == 0) griddep_launch_dependents();
  const uint32_t tmem = tmem_slot + (pipe < NP ? pipe : 0) * C::kTmemCols;
  const uint64_t wait_ns = a.wait_ns;
  bool ok = true;

  if (gwarp < kCtrlWarps) {
  // Each warpgroup changes its register count at the top of its own branch,
  // so the code after it is compiled for the new count.
  if constexpr (NP == 2) setmaxnreg_dec<kCtrlRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // This kernel may start while the previous one in the stream is still
      // running (programmatic dependent launch): nothing is read before it
      // has finished.
      griddep_wait();
      int last_k[NS], last_v[NS], last_q[2] = {-1, -1};
      for (int s = 0; s < NS; ++s) last_k[s] = last_v[s] = -1;
      // Q of the units with key tiles, in order: the nq-th goes to slot nq & 1.
      auto next_with_tiles = [&](int k) {
        while (k < n_units && unit_info(u_of(k)).n_kv == 0) ++k;
        return k;
      };
      int qk = next_with_tiles(0), nq = 0;
      auto issue_q = [&]() -> bool {
        const Unit t = unit_info(u_of(qk));
        const int slot = nq & 1;
        // The unit two back, which used this slot, must be done with it.
        if (nq >= 2 && !mbar_wait(bar(kBarQFree + slot), ((nq >> 1) - 1) & 1, wait_ns)) return false;
        mbar_arrive_expect_tx(bar(kBarQFull + slot), C::kQBytes);
        for (int at = 0; at < C::kAtoms; ++at)
          tma_load_4d(sQ0 + slot * C::kQBytes + at * (kTileM * 128), &mQ, bar(kBarQFull + slot),
                      at * 64, t.h, t.qbase + t.m0, t.b);
        last_q[slot] = nq++;
        qk = next_with_tiles(qk + 1);
        return true;
      };
      if (qk < n_units) ok = issue_q();
      int gj = 0;  // key tiles loaded so far, over all units
      int ne = 0;  // units with key tiles so far
      for (int ku = 0; ku < n_units && ok; ++ku) {
        const Unit t = unit_info(u_of(ku));
        if (t.n_kv == 0) continue;
        for (int j = 0; j < t.n_kv; ++j, ++gj) {
          const int s = gj % NS;
          const uint32_t ph = (gj / NS) & 1;
          if (gj >= NS && !(ok = mbar_wait(bar(kBarKEmpty + s), ph ^ 1, wait_ns))) break;
          mbar_arrive_expect_tx(bar(kBarKFull + s), C::kKvBytes);
          for (int at = 0; at < C::kAtoms; ++at)
            tma_load_4d(sK0 + s * C::kKvBytes + at * (kBN * 128), &mK, bar(kBarKFull + s), at * 64,
                        t.hkv, t.kbase + j * kBN, t.b);
          last_k[s] = gj;
          if (gj >= NS && !(ok = mbar_wait(bar(kBarVEmpty + s), ph ^ 1, wait_ns))) break;
          mbar_arrive_expect_tx(bar(kBarVFull + s), C::kKvBytes);
          for (int at = 0; at < C::kAtoms; ++at)
            tma_load_4d(sV0 + s * C::kKvBytes + at * (kBN * 128), &mV, bar(kBarVFull + s), at * 64,
                        t.hkv, t.kbase + j * kBN, t.b);
          last_v[s] = gj;
          // The next unit's Q, once this unit's first tile is on its way.
          if (j == 0 && qk < n_units && nq == ne + 1 && !(ok = issue_q())) break;
        }
        ++ne;
      }
      if (!ok) {
        // Let every copy already issued land before the block's shared memory goes away.
        for (int i = 0; i < 2; ++i)
          if (last_q[i] >= 0) mbar_wait(bar(kBarQFull + i), (last_q[i] >> 1) & 1, wait_ns);
        for (int s = 0; s < NS; ++s) {
          if (last_k[s] >= 0) mbar_wait(bar(kBarKFull + s), (last_k[s] / NS) & 1, wait_ns);
          if (last_v[s] >= 0) mbar_wait(bar(kBarVFull + s), (last_v[s] / NS) & 1, wait_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (MMA issue is warp-collective); every
    // wait is made warp-uniform so the warp stays converged.
    constexpr uint32_t kIdQK = idesc_bf16(kTileM, kBN, false, false);
    constexpr uint32_t kIdPV = idesc_bf16(kTileM, D, false, true);
    // Operand descriptors built once; the loops only add constant offsets.
    const uint64_t dQ0 = sdesc_sw128(sQ0, 16, 1024);
    const uint64_t dK0 = sdesc_sw128(sK0, 16, 1024);
    const uint64_t dV0 = sdesc_sw128(sV0, kBN * 128, 1024);
    const uint32_t tS = tmem + C::kColS, tP = tmem + C::kColP, tO = tmem + C::kColO;
    // S of global key tile gj = Q K^T, Q from slot `slot`.
    auto issue_s = [&](int gj, int slot) -> bool {
      const int s = gj % NS;
      if (!warp_all(mbar_wait(bar(kBarKFull + s), (gj / NS) & 1, wait_ns))) return false;
      tc_fence_after();
      const uint64_t dK = desc_add(dK0, s * C::kKvBytes), dQ = desc_add(dQ0, slot * C::kQBytes);
#pragma unroll
      for (int g = 0; g < D / 64; ++g) {  // K = 64 per group of four steps
        const uint64_t q = desc_add(dQ, g * (kTileM * 128)), k = desc_add(dK, g * (kBN * 128));
        mma_ss_x4(tS, q, desc_add(q, 32), desc_add(q, 64), desc_add(q, 96), k, desc_add(k, 32),
                  desc_add(k, 64), desc_add(k, 96), kIdQK, g > 0 ? 1u : 0u);
      }
      mma_commit(bar(kBarS));
      mma_commit(bar(kBarKEmpty + s));
      return true;
    };
    // O (+)= P V of global key tile gj; the first tile of a unit overwrites
    // O.  P of key pair (2c, 2c + 1) sits in column c: K step k (16 keys)
    // reads columns 8k .. 8k + 7 and V rows 16k .. 16k + 15 (2 KB apart).
    // Waiting for P also covers the previous unit's epilogue: the softmax
    // threads read O before they write the next P.
    auto issue_pv = [&](int gj, bool first) -> bool {
      const int s = gj % NS;
      if (!warp_all(mbar_wait(bar(kBarP), gj & 1, wait_ns))) return false;
      if (!warp_all(mbar_wait(bar(kBarVFull + s), (gj / NS) & 1, wait_ns))) return false;
      tc_fence_after();
      const uint64_t dV = desc_add(dV0, s * C::kKvBytes);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        mma_ts_x4(tO, tP + 32 * h, tP + 32 * h + 8, tP + 32 * h + 16, tP + 32 * h + 24,
                  desc_add(dV, (4 * h) * 2048), desc_add(dV, (4 * h + 1) * 2048),
                  desc_add(dV, (4 * h + 2) * 2048), desc_add(dV, (4 * h + 3) * 2048), kIdPV,
                  (first && h == 0) ? 0u : 1u);
      mma_commit(bar(kBarVEmpty + s));
      mma_commit(bar(kBarO));
      return true;
    };
    int gj = 0, ne = 0;
    int pend = -1;          // the key tile whose P V is still to be issued
    bool pend_first = false;
    for (int ku = 0; ku < n_units && ok; ++ku) {
      const Unit t = unit_info(u_of(ku));
      if (t.n_kv == 0) continue;
      const int slot = ne & 1;
      if (!(ok = warp_all(mbar_wait(bar(kBarQFull + slot), (ne >> 1) & 1, wait_ns)))) break;
      tc_fence_after();
      for (int j = 0; j < t.n_kv; ++j, ++gj) {
        // The score columns are free once the softmax warps hold S_{gj-1}.
        if (gj > 0 && !(ok = warp_all(mbar_wait(bar(kBarSFree), (gj - 1) & 1, wait_ns)))) break;
        if (!(ok = issue_s(gj, slot))) break;
        if (j == t.n_kv - 1) mma_commit(bar(kBarQFree + slot));
        if (pend >= 0 && !(ok = issue_pv(pend, pend_first))) break;
        pend = gj;
        pend_first = (j == 0);
      }
      ++ne;
    }
    if (ok && pend >= 0) ok = issue_pv(pend, pend_first);
    // Every issued MMA must finish before TMEM is released.
    mma_commit(bar(kBarDrain));
    warp_all(mbar_wait(bar(kBarDrain), 0, wait_ns));
  }
  } else {
    // ------------------------------------------------------------ softmax warps
    if constexpr (NP == 2) setmaxnreg_inc<kSoftRegs>();
    const int quarter = gwarp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t tS = tl + C::kColS, tP = tl + C::kColP, tO = tl + C::kColO;
    const float sl2 = a.scale_log2;
    int gj = 0;
    for (int ku = 0; ku < n_units && ok; ++ku) {
      int qlast, wlast, tk, n_kv;
      {
        const Unit t0 = unit_info(u_of(ku));
        // Last key visible to this row and to the warp's last row (causal).
        qlast = t0.m0 + r + t0.off;
        wlast = t0.m0 + quarter * 32 + 31 + t0.off;
        tk = t0.tk;
        n_kv = t0.n_kv;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_kv; ++j, ++gj) {
        ok = warp_all(mbar_wait(bar(kBarS), gj & 1, wait_ns));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_nowait(tS + 32 * c, sr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence32(sr[c]);
        // S_j is in registers: the next scores may overwrite its columns.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSFree));

        const int kv0 = j * kBN;  // key of column 0
        // Masking only where this warp's rows meet the diagonal (or tk),
        // decided for the whole warp; other tiles run the code without it.
        const bool need_mask = (a.causal && kv0 + kBN - 1 > wlast - 31) || kv0 + kBN > tk;
        const int lim = a.causal ? min(qlast - kv0, tk - 1 - kv0) : (tk - 1 - kv0);
        // 32-key chunks past every row of the warp (or past tk) are all zeros:
        // only the first live_chunks take exponentials.
        const int last_key = a.causal ? min(wlast, tk - 1) : tk - 1;
        const int live_chunks = last_key < kv0 ? 0 : min(4, (last_key - kv0) / 32 + 1);
        float alpha = 1.f;
        bool moved = false;
        uint64_t sum2[4];
        uint32_t pk[2][32];
        auto softmax_tile = [&](auto masked) {
          constexpr bool kMasked = decltype(masked)::value;
          // Masked scores become -inf, so 2^(x - m) is exactly zero there;
          // chunks past live_chunks are all masked: they take no part in the
          // maximum and their P is zero without exponentials.
          const int lc = kMasked ? live_chunks : 4;
          if constexpr (kMasked) {
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (32 * ch + i > lim) sr[ch][i] = __float_as_uint(-INFINITY);
          }
          // Maximum over the row's live columns in four independent chains.
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
            if (ch < lc) {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                mx4[i & 3] = fmax3(mx4[i & 3], __uint_as_float(sr[ch][2 * i]),
                                   __uint_as_float(sr[ch][2 * i + 1]));
            }
          const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
          // A row may see no key in this tile (packed batches): mx = -inf
          // leaves the running maximum alone and every P zero.
          const float m_new = mx * sl2;
          if (m_new > m_run + kRescaleLog2) {
            alpha = ex2_approx(m_run - m_new);
            m_run = m_new;
            moved = true;
          }
          const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
          const uint64_t sl2x2 = f2_make(sl2, sl2), neg_m = f2_make(-m_use, -m_use);
#pragma unroll
          for (int q = 0; q < 4; ++q) sum2[q] = f2_make(0.f, 0.f);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            if (ch >= lc) {
#pragma unroll
              for (int i = 0; i < 16; ++i) pk[ch >> 1][16 * (ch & 1) + i] = 0u;
              continue;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint64_t x = f2_fma(f2_make(__uint_as_float(sr[ch][2 * i]),
                                                __uint_as_float(sr[ch][2 * i + 1])),
                                        sl2x2, neg_m);
              float x0, x1, p0, p1;
              f2_split(x, x0, x1);
              if ((i & 7) < kPolyOf8) {
                exp2_poly2(x0, x1, p0, p1);
              } else {
                p0 = ex2_approx(x0);
                p1 = ex2_approx(x1);
              }
              sum2[i & 3] = f2_add(sum2[i & 3], f2_make(p0, p1));
              pk[ch >> 1][16 * (ch & 1) + i] = pack_bf16x2(p0, p1);
            }
          }
        };
        if (need_mask)
          softmax_tile(std::true_type{});
        else
          softmax_tile(std::false_type{});
        // The previous tile's P V must be done: it read the P columns this
        // tile overwrites, and O must be final before a rescale.
        if (gj > 0) {
          ok = warp_all(mbar_wait(bar(kBarO), (gj - 1) & 1, wait_ns));
          if (!ok) break;
          tc_fence_after();
        }
        if (j > 0 && __any_sync(0xffffffffu, moved)) {
          // O holds the sum over earlier tiles scaled by the old maximum.
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + 32 * c, ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32_nowait(tO + 32 * c, ov);
          }
        }
        tmem_st32_nowait(tP, pk[0]);
        tmem_st32_nowait(tP + 32, pk[1]);
        tmem_wait_st();
        float s[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) f2_split(sum2[q], s[2 * q], s[2 * q + 1]);
        l_run = l_run * alpha + (((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7])));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarP));
      }
      if (!ok) break;
      // The unit again, for its epilogue (looked up anew rather than kept in
      // registers through the key loop).
      const Unit t = unit_info(u_of(ku));
      const int qrow = t.m0 + r;
      const bool live = qrow < t.tq;
      // Rows that see no key (packed sequences with more queries than keys,
      // or a unit without key tiles): O = 0 and LSE = -inf.
      const bool blind = VL && !(m_run > -INFINITY);
      uint32_t pkd[D / 2];
      if (n_kv > 0) {
        // The unit's last P V has finished once O's barrier passes its tile.
        ok = warp_all(mbar_wait(bar(kBarO), (gj - 1) & 1, wait_ns));
        if (!ok) break;
        tc_fence_after();
        const float inv_l = blind ? 0.f : 1.f / l_run;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tO + 32 * c, ov);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkd[16 * c + i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l,
                                          __uint_as_float(ov[2 * i + 1]) * inv_l);
        }
        // O is in registers; the next unit's first P V (issued after this
        // warp's next P arrival) may overwrite it.
        tc_fence_before();
      }
      if (blind || n_kv == 0) {
#pragma unroll
        for (int i = 0; i < D / 2; ++i) pkd[i] = 0u;
      }
      // This warp's 32 rows go out through one TMA store per 64 columns
      // (rows past T are clipped by the map), unless they run past a packed
      // sequence's end, where the rows beyond belong to the next sequence.
      if (!VL || t.m0 + quarter * 32 + 32 <= t.tq) {
        // The warp's previous store must have read the staging rows first.
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int at = 0; at < C::kAtoms; ++at) {
          const uint32_t row = sO + at * (kTileM * 128) + (quarter * 32 + lane) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int k = 32 * at + 4 * c;  // first of the chunk's four packed pairs
            st_shared_u4(row + ((c ^ (lane & 7)) << 4),
                         make_uint4(pkd[k], pkd[k + 1], pkd[k + 2], pkd[k + 3]));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int at = 0; at < C::kAtoms; ++at)
            tma_store_4d(&mO, sO + at * (kTileM * 128) + quarter * 32 * 128, at * 64, t.h,
                         t.qbase + t.m0 + quarter * 32, t.b);
          bulk_commit_group();
        }
      } else if (live) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) +
                                              ((static_cast<size_t>(t.b) * a.T + t.qbase + qrow) * a.Hq + t.h) * D);
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
          dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
      }
      if (live)
        a.lse[(static_cast<size_t>(t.b) * a.Hq + t.h) * a.T + t.qbase + qrow] =
            (blind || n_kv == 0) ? -INFINITY : (m_run + log2f(l_run)) * 0.69314718055994530942f;
    }
    // Every store of O must be complete before the block (and its shared
    // memory) goes away.
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  if (!ok) atomicOr(&g_fwd_status, 1u);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tmem_slot, NP * C::kTmemCols);
  }
}

template <int D, class VT>
cudaError_t launch_fwd_t(int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const CUtensorMap& mo, const FwdArgs& a,
                         const QTileSched& sched, const VT& vt, cudaStream_t st) {
  const int smem = Cfg<D>::kSmemBytes;
  // Once per device and context (holds the context id it was set for).
  static unsigned long long attr_ctx[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long ctx = current_context_id();
  if (dev >= 64 || ctx == 0 || attr_ctx[dev] != ctx) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D, VT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    if constexpr (Cfg<D>::NP == 2) {
      // The block's registers at launch must cover the warpgroups' shares
      // after reallocation, or the softmax warpgroups' increase never
      // completes: refuse to launch rather than start such a kernel.
      cudaFuncAttributes fa{};
      if ((e = cudaFuncGetAttributes(&fa, attn_fwd_kernel<D, VT>)) != cudaSuccess) return e;
      if (fa.numRegs * fwd_threads(D) < kRegBudget) return cudaErrorInvalidConfiguration;
    }
    if (dev < 64) attr_ctx[dev] = current_context_id();
  }
  // Launched as a programmatic dependent of whatever precedes it in the
  // stream: its set-up overlaps that kernel's tail, and its producer waits
  // for that kernel to finish before the first load.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(fwd_threads(D));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_fwd_kernel<D, VT>, mq, mk, mv, mo, a, sched, vt);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int D, int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mo, const FwdArgs& a,
                       const QTileSched& sched, const VarlenTable* vt, cudaStream_t st) {
  if (vt != nullptr)
    return D == 64 ? launch_fwd_t<64>(grid, mq, mk, mv, mo, a, sched, *vt, st)
                   : launch_fwd_t<128>(grid, mq, mk, mv, mo, a, sched, *vt, st);
  const NoVarlen none{};
  return D == 64 ? launch_fwd_t<64>(grid, mq, mk, mv, mo, a, sched, none, st)
                 : launch_fwd_t<128>(grid, mq, mk, mv, mo, a, sched, none, st);
}

cudaError_t take_fwd_status(cudaStream_t st, unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_fwd_status, sizeof(v), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v)
    e = cudaMemcpyToSymbolAsync(g_fwd_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  *out = v;
  return e;
}

}  // namespace detattn

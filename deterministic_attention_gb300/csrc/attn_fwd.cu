// Fused causal grouped-query flash-attention forward for sm_103a.
//
// RustingBrain vs PyTorch/TensorFlow page, "Step 2: fused flash attention":
// one fused kernel replaces the causal softmax kernels and never writes the
// [seq_len, seq_len] score matrix.  "Step 1" names the per-row logsumexp the
// forward hands to the backward.
//
// Work unit: one 128-row query tile of one (batch, query head), walking
// 64-key tiles 0..diagonal in ascending order.  The kernel is persistent: a
// block holds NP pipelines (two at D = 64, one at D = 128), each with its own
// warps, shared memory, mbarriers and TMEM columns, and each pipeline works
// through the list of units the host dealt it (heaviest first, balanced per
// SM, so the two pipelines of a block finish together).  Per pipeline:
//   warp 0      TMA producer: each unit's Q (once the previous unit's Q K^T
//               MMAs are done with Q), then K_j / V_j into a ring of stages
//   warp 1      tcgen05 issuer, one key tile ahead of the softmax: S_{j+1} =
//               Q K_{j+1}^T goes into the other of two TMEM score buffers while
//               the softmax works on S_j; then O += P_j V_j with P_j read from
//               TMEM (bf16, written over S_j by the softmax warps)
//   warps 2..9  softmax: two threads per query row (TMEM lane), each taking 32
//               of the tile's 64 keys, each with its own running maximum, row
//               sum and O accumulator (P of keys 0..31 of every tile goes to
//               O_0, of keys 32..63 to O_1); online softmax in base 2 with a
//               lazily moved maximum, P to TMEM, O_h rescaled in TMEM when its
//               maximum moves.  Each unit's epilogue merges the two halves:
//               O = (O_0 2^(m_0-M) + O_1 2^(m_1-M)) / (l_0 2^(m_0-M) + l_1 2^(m_1-M)),
//               M = max(m_0, m_1), LSE = ln2 * (M + log2 L).
// The next unit's first scores are computed while this unit's epilogue runs.
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

constexpr int kPipeWarps = 10;  // producer, MMA issuer, 8 softmax warps
constexpr int kPipeThreads = kPipeWarps * 32;
constexpr int kBN = kFwdTileN;  // keys per tile (64)
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
  static constexpr int kKvBytes = kBN * 128 * kAtoms;    // 64 rows x D bf16
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKvBytes;
  static constexpr int kPipeBytes = kOffV + kStages * kKvBytes;  // one pipeline (multiple of 1024)
  static constexpr int NP = qtile_pipes_per_block(D);
  static constexpr int kSmemBytes = NP * kPipeBytes + 1024;     // + alignment slack
  static constexpr uint32_t kTmemCols = (D == 64) ? 256 : 512;  // per pipeline
  static_assert(kPipeBytes % 1024 == 0, "pipelines keep the 1024-byte swizzle alignment");
  // Two score buffers of 64 fp32 columns (buffer b at 64 b).  The softmax
  // thread of half h owns columns 32h..32h+31 of a buffer and writes its 32
  // bf16 P values, packed in pairs, over the first 16 of them.
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO = 128;  // O_h accumulator at 128 + D h, D cols each
};

constexpr int kMaxStages = 4;
enum : int {
  kBarQ = 0,
  kBarKFull = 1,
  kBarVFull = kBarKFull + kMaxStages,
  kBarKEmpty = kBarVFull + kMaxStages,
  kBarVEmpty = kBarKEmpty + kMaxStages,
  kBarS = kBarVEmpty + kMaxStages,  // [2]: score buffer b holds S_j
  kBarP = kBarS + 2,                // [2]: softmax wrote P_j over buffer b
  kBarO = kBarP + 2,                // one arrival per finished O += P V
  kBarOFinal = kBarO + 1,           // the last O += P V has finished
  kBarDrain = kBarOFinal + 1,
  kBarPair = kBarDrain + 1,         // [4]: the two softmax halves of a lane quarter
  kBarQFree = kBarPair + 4,         // the unit's Q K^T MMAs are done with Q
  kBarOFree = kBarQFree + 1,        // the unit's epilogue has read O
  kNumBars = kBarOFree + 1
};

__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }


template <int D, class VT>
__global__ void __launch_bounds__(kPipeThreads * qtile_pipes_per_block(D), 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mV, const FwdArgs a,
                    const __grid_constant__ QTileSched sched, const __grid_constant__ VT vt) {
  using C = Cfg<D>;
  constexpr bool VL = std::is_same<VT, VarlenTable>::value;
  constexpr int NS = C::kStages;
  constexpr int NP = C::NP;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars_all[NP][kNumBars];
  __shared__ uint32_t tmem_slot;
  __shared__ float red_m_all[NP][2][kTileM];  // [pipe][half][row] final running maxima (log2 units)
  __shared__ float red_l_all[NP][2][kTileM];  // [pipe][half][row] final row sums

  const int pipe = static_cast<int>(threadIdx.x) / kPipeThreads;
  const int warp = (static_cast<int>(threadIdx.x) >> 5) % kPipeWarps;  // role within the pipeline
  const int lane = threadIdx.x & 31;
  const int gwarp = static_cast<int>(threadIdx.x) >> 5;               // TMEM lane quarter: gwarp & 3
  const int pipe_id = static_cast<int>(blockIdx.x) * NP + pipe;
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
  const uint32_t sP = smem_u32(smem) + pipe * C::kPipeBytes;
  const uint32_t sQ = sP + C::kOffQ;
  const uint32_t sK0 = sP + C::kOffK;
  const uint32_t sV0 = sP + C::kOffV;
  uint64_t* bars = bars_all[pipe];
  float (*red_m)[kTileM] = red_m_all[pipe];
  float (*red_l)[kTileM] = red_l_all[pipe];
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x < 32) {
    tmem_alloc(smem_u32(&tmem_slot), NP * C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (warp == 1 && lane == 0) {  // each pipeline's MMA warp sets up its own barriers
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarS + i), 1);
      mbar_init(bar(kBarP + i), 8);
    }
    mbar_init(bar(kBarO), 1);
    mbar_init(bar(kBarOFinal), 1);
    mbar_init(bar(kBarDrain), 1);
    for (int qq = 0; qq < 4; ++qq) mbar_init(bar(kBarPair + qq), 64);
    mbar_init(bar(kBarQFree), 1);
    mbar_init(bar(kBarOFree), 8);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&mQ);
    tma_prefetch_desc(&mK);
    tma_prefetch_desc(&mV);
  }
  __syncthreads();
  tc_fence_after();
  // A kernel launched after this one as a programmatic dependent (the
  // backward's Delta step) may be scheduled now: it takes SMs as this grid's
  // blocks leave them and waits (griddepcontrol.wait) for this grid to
  // finish before it reads anything, so its launch latency hides under this
  // grid's tail.
  if (threadIdx.x == 0) griddep_launch_dependents();
  const uint32_t tmem = tmem_slot + pipe * C::kTmemCols;
  const uint64_t wait_ns = a.wait_ns;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int last_k[kMaxStages], last_v[kMaxStages];
      for (int s = 0; s < kMaxStages; ++s) last_k[s] = last_v[s] = -1;
      int last_q = -1;
      int gj = 0;  // key tiles loaded so far, over all units
      for (int ku = 0; ku < n_units && ok; ++ku) {
        const Unit t = unit_info(u_of(ku));
        // The previous unit's Q K^T MMAs must be done with Q.
        if (ku > 0 && !(ok = mbar_wait(bar(kBarQFree), (ku - 1) & 1, wait_ns))) break;
        mbar_arrive_expect_tx(bar(kBarQ), C::kQBytes);
        for (int at = 0; at < C::kAtoms; ++at)
          tma_load_4d(sQ + at * (kTileM * 128), &mQ, bar(kBarQ), at * 64, t.h, t.qbase + t.m0, t.b);
        last_q = ku;
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
        }
      }
      if (!ok) {
        // Let every copy already issued land before the block's shared memory goes away.
        if (last_q >= 0) mbar_wait(bar(kBarQ), last_q & 1, wait_ns);
        for (int s = 0; s < NS; ++s) {
          if (last_k[s] >= 0) mbar_wait(bar(kBarKFull + s), (last_k[s] / NS) & 1, wait_ns);
          if (last_v[s] >= 0) mbar_wait(bar(kBarVFull + s), (last_v[s] / NS) & 1, wait_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (MMA issue is warp-collective); every
    // wait is made warp-uniform so the warp stays converged.
    constexpr uint32_t kIdQK = idesc_bf16(kTileM, kBN, false, false);
    constexpr uint32_t kIdPV = idesc_bf16(kTileM, D, false, true);
    // Operand descriptors built once; the loops only add constant offsets.
    const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dK0 = sdesc_sw128(sK0, 16, 1024);
    const uint64_t dV0 = sdesc_sw128(sV0, kBN * 128, 1024);
    // S of global key tile gj = Q K^T into score buffer gj & 1.
    auto issue_qk = [&](int gj) -> bool {
      const int s = gj % NS;
      if (!warp_all(mbar_wait(bar(kBarKFull + s), (gj / NS) & 1, wait_ns))) return false;
      tc_fence_after();
      const uint64_t dK = desc_add(dK0, s * C::kKvBytes);
      const uint32_t tS = tmem + C::kColS + (gj & 1) * kBN;
#pragma unroll
      for (int g = 0; g < D / 64; ++g) {  // K = 64 per group of four steps
        const uint64_t q = desc_add(dQ, g * (kTileM * 128)), k = desc_add(dK, g * (kBN * 128));
        mma_ss_x4(tS, q, desc_add(q, 32), desc_add(q, 64), desc_add(q, 96), k, desc_add(k, 32),
                  desc_add(k, 64), desc_add(k, 96), kIdQK, g > 0 ? 1u : 0u);
      }
      mma_commit(bar(kBarS + (gj & 1)));
      mma_commit(bar(kBarKEmpty + s));
      return true;
    };
    int gj = 0;
    for (int ku = 0; ku < n_units && ok; ++ku) {
      const Unit t = unit_info(u_of(ku));
      if (!(ok = warp_all(mbar_wait(bar(kBarQ), ku & 1, wait_ns)))) break;
      tc_fence_after();
      if (t.n_kv > 0 && !(ok = issue_qk(gj))) break;
      for (int j = 0; j < t.n_kv && ok; ++j, ++gj) {
        // One tile ahead: S_{j+1} lands in the other buffer while the softmax
        // works on S_j.  That buffer last held P_{j-1}, whose P V was issued
        // in the previous iteration (tcgen05 operations run in issue order).
        if (j + 1 < t.n_kv && !(ok = issue_qk(gj + 1))) break;
        const int s = gj % NS;
        if (!(ok = warp_all(mbar_wait(bar(kBarP + (gj & 1)), (gj >> 1) & 1, wait_ns)))) break;
        if (!(ok = warp_all(mbar_wait(bar(kBarVFull + s), (gj / NS) & 1, wait_ns)))) break;
        // The previous unit's epilogue must have read O before this unit's
        // first P V overwrites it.
        if (j == 0 && ku > 0 &&
            !(ok = warp_all(mbar_wait(bar(kBarOFree), (ku - 1) & 1, wait_ns))))
          break;
        tc_fence_after();
        const uint64_t dV = desc_add(dV0, s * C::kKvBytes);
        const uint32_t tP = tmem + C::kColS + (gj & 1) * kBN;
        // O_h += P_h V_h over the 32 keys of half h: half h wrote them as 16
        // packed columns at the start of its own 32 score columns.
        static_assert(kBN == 64, "the P V issue below takes 2 steps per half");
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          mma_ts_x2(tmem + C::kColO + hh * D, tP + hh * 32, tP + hh * 32 + 8,
                    desc_add(dV, (2 * hh) * 2048), desc_add(dV, (2 * hh + 1) * 2048), kIdPV,
                    j > 0 ? 1u : 0u);
        mma_commit(bar(kBarVEmpty + s));
        mma_commit(bar(kBarO));
      }
      if (!ok) break;
      // Q may be replaced once these MMAs finish; the epilogue waits on its
      // own barrier (with the issuer a tile ahead, the per-tile O barrier can
      // trail the softmax by two phases there, which a parity wait cannot
      // tell apart).
      mma_commit(bar(kBarQFree));
      mma_commit(bar(kBarOFinal));
    }
    // Every issued MMA must finish before TMEM is released.
    mma_commit(bar(kBarDrain));
    warp_all(mbar_wait(bar(kBarDrain), 0, wait_ns));
  } else {
    // ------------------------------------------------------------ softmax warps
    // Warps w and w+4 of a pipeline share a TMEM lane quarter, i.e. the same
    // 32 query rows; half 0 takes keys 0..31 of each tile, half 1 keys 32..63.
    // Each half runs its own online softmax into its own accumulator O_h; the
    // two meet once per unit, in the epilogue, at an mbarrier of the pair (64
    // arrivals, bounded wait).
    const int quarter = gwarp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    const uint32_t pair_bar = bar(kBarPair + quarter);  // the two halves of these rows
    int gj = 0;
    for (int ku = 0; ku < n_units && ok; ++ku) {
      int qlast, wlast, tk, n_kv;
      {
        const Unit t0 = unit_info(u_of(ku));
        // Last key visible to this row and to the warp's first row (causal).
        qlast = t0.m0 + r + t0.off;
        wlast = t0.m0 + quarter * 32 + t0.off;
        tk = t0.tk;
        n_kv = t0.n_kv;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_kv; ++j, ++gj) {
        ok = warp_all(mbar_wait(bar(kBarS + (gj & 1)), (gj >> 1) & 1, wait_ns));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tl + C::kColS + (gj & 1) * kBN + half * 32;  // this half's columns
        const int kv0 = j * kBN + half * 32;  // key of this thread's first column
        // This warp's 32 rows against this half's 32 keys, decided for the
        // whole warp: every key after every row (or past T) -- P is zero and
        // the running maximum and sum stay as they are; every key visible --
        // no mask.
        const bool all_masked = (a.causal && wlast + 31 < kv0) || kv0 >= tk;
        const bool need_mask = (a.causal && kv0 + 31 > wlast) || kv0 + 32 > tk;
        if (all_masked) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = 0u;
          tmem_st16_nowait(tS, pk);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarP + (gj & 1)));
          continue;
        }
        uint32_t sr[32];
        tmem_ld32_nowait(tS, sr);
        tmem_wait_ld();
        reg_fence32(sr);

        const int lim = a.causal ? min(qlast - kv0, tk - 1 - kv0) : (tk - 1 - kv0);
        float alpha = 1.f;
        bool moved = false;
        uint64_t sum2[2];  // four partial sums
        uint32_t pk[16];
        // Masking is needed only where this warp's rows meet the diagonal (or
        // T), decided for the whole warp; other tiles run the code without it.
        auto softmax_tile = [&](auto masked) {
          constexpr bool kMasked = decltype(masked)::value;
          if constexpr (kMasked) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c > lim) sr[c] = __float_as_uint(-INFINITY);
          }
          // Maximum over this half's 32 columns in four independent chains.
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 16; ++c)
            mx4[c & 3] = fmax3(mx4[c & 3], __uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1]));
          const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
          // A half-row may see no key in this tile (past its diagonal): mx =
          // -inf leaves the running maximum alone and every P zero.
          const float m_new = mx * sl2;
          if (m_new > m_run + kRescaleLog2) {
            alpha = ex2_approx(m_run - m_new);
            m_run = m_new;
            moved = true;
          }
          const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
          const uint64_t sl2x2 = f2_make(sl2, sl2), neg_m = f2_make(-m_use, -m_use);
          sum2[0] = sum2[1] = f2_make(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t x = f2_fma(f2_make(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])),
                                      sl2x2, neg_m);
            float x0, x1, p0, p1;
            f2_split(x, x0, x1);
            if ((i & 7) < kPolyOf8) {
              exp2_poly2(x0, x1, p0, p1);
            } else {
              p0 = ex2_approx(x0);
              p1 = ex2_approx(x1);
            }
            if constexpr (kMasked) {  // masked keys contribute exactly zero
              if (2 * i > lim) p0 = 0.f;
              if (2 * i + 1 > lim) p1 = 0.f;
            }
            sum2[i & 1] = f2_add(sum2[i & 1], f2_make(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
          }
        };
        if (need_mask)
          softmax_tile(std::true_type{});
        else
          softmax_tile(std::false_type{});
        tmem_st16_nowait(tS, pk);
        tmem_wait_st();
        if (j > 0 && __any_sync(0xffffffffu, moved)) {
          // O_h holds the sum over earlier tiles scaled by the old maximum:
          // wait for the last P V to land, then rescale O_h in TMEM.  (S of
          // tile gj was committed after P_{gj-2} V, so the O barrier is at
          // most one phase behind here and the parity wait is exact.)
          ok = warp_all(mbar_wait(bar(kBarO), (gj - 1) & 1, wait_ns));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            const uint32_t col = C::kColO + half * D + c * 32;
            tmem_ld32(tl + col, ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32_nowait(tl + col, ov);
          }
          tmem_wait_st();
        }
        float s0, s1, s2, s3;
        f2_split(sum2[0], s0, s1);
        f2_split(sum2[1], s2, s3);
        l_run = l_run * alpha + ((s0 + s1) + (s2 + s3));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarP + (gj & 1)));
      }
      if (!ok) break;
      ok = warp_all(mbar_wait(bar(kBarOFinal), ku & 1, wait_ns));
      if (!ok) break;
      // The unit again, for its epilogue (looked up anew rather than kept in
      // registers through the key loop).
      const Unit t = unit_info(u_of(ku));
      const int qrow = t.m0 + r;
      // Merge the two halves: M = max(m_0, m_1), f_h = 2^(m_h - M),
      // L = l_0 f_0 + l_1 f_1 (half 0 first), O = (O_0 f_0 + O_1 f_1) / L.
      red_m[half][r] = m_run;
      red_l[half][r] = l_run;
      mbar_arrive(pair_bar);
      ok = warp_all(mbar_wait(pair_bar, ku & 1, wait_ns));
      if (!ok) break;
      tc_fence_after();
      const float m0v = red_m[0][r], m1v = red_m[1][r];
      // Finite in the fixed-length form (key 0 is visible to every row).  A
      // packed sequence with more queries than keys has rows that see no key:
      // M = -inf there, and the row gets O = 0 and LSE = -inf.
      float M = fmaxf(m0v, m1v);
      bool blind = false;
      if constexpr (VL) {
        blind = !(M > -INFINITY);
        if (blind) M = 0.f;
      }
      const float f0 = ex2_approx(m0v - M), f1 = ex2_approx(m1v - M);
      const float l_tot = red_l[0][r] * f0 + red_l[1][r] * f1;
      const float inv_l = blind ? 0.f : 1.f / l_tot;
      const float w0 = blind ? 0.f : f0 * inv_l, w1 = blind ? 0.f : f1 * inv_l;
      const bool live = qrow < t.tq;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) +
                            ((static_cast<size_t>(t.b) * a.T + t.qbase + qrow) * a.Hq + t.h) * D +
                            half * (D / 2);
      uint32_t pkd[D / 4];
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o0[32], o1[32];
        const uint32_t col = half * (D / 2) + c * 32;
        tmem_ld32(tl + C::kColO + col, o0);
        tmem_ld32(tl + C::kColO + D + col, o1);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pkd[16 * c + i] = pack_bf16x2(
              fmaf(__uint_as_float(o0[2 * i]), w0, __uint_as_float(o1[2 * i]) * w1),
              fmaf(__uint_as_float(o0[2 * i + 1]), w0, __uint_as_float(o1[2 * i + 1]) * w1));
      }
      if constexpr (VL) {
        // A unit without key tiles never wrote its accumulators: they hold an
        // earlier unit's sums (which times 0 could still be NaN).
        if (blind) {
#pragma unroll
          for (int i = 0; i < D / 4; ++i) pkd[i] = 0u;
        }
      }
      // O is in registers: the next unit's first P V may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarOFree));
      if (live) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int i = 0; i < D / 16; ++i)
          dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
        if (half == 0)
          a.lse[(static_cast<size_t>(t.b) * a.Hq + t.h) * a.T + t.qbase + qrow] =
              blind ? -INFINITY : (M + log2f(l_tot)) * 0.69314718055994530942f;
      }
    }
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
                         const CUtensorMap& mv, const FwdArgs& a, const QTileSched& sched,
                         const VT& vt, cudaStream_t st) {
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
    if (dev < 64) attr_ctx[dev] = current_context_id();
  }
  attn_fwd_kernel<D, VT><<<grid, kPipeThreads * Cfg<D>::NP, smem, st>>>(mq, mk, mv, a, sched, vt);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int D, int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const FwdArgs& a, const QTileSched& sched,
                       const VarlenTable* vt, cudaStream_t st) {
  if (vt != nullptr)
    return D == 64 ? launch_fwd_t<64>(grid, mq, mk, mv, a, sched, *vt, st)
                   : launch_fwd_t<128>(grid, mq, mk, mv, a, sched, *vt, st);
  const NoVarlen none{};
  return D == 64 ? launch_fwd_t<64>(grid, mq, mk, mv, a, sched, none, st)
                 : launch_fwd_t<128>(grid, mq, mk, mv, a, sched, none, st);
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

// Fused causal grouped-query flash-attention forward for sm_103a.
//
// RustingBrain vs PyTorch/TensorFlow page, "Step 2: fused flash attention":
// one fused kernel replaces the causal softmax kernels and never writes the
// [seq_len, seq_len] score matrix.  "Step 1" names the per-row logsumexp the
// forward hands to the backward.
//
// One thread block owns one 128-row query tile of one (batch, query head) and
// walks the key/value tiles 0..diagonal in ascending order:
//   warp 0      TMA producer: Q once, then K_j / V_j into a ring of stages
//   warp 1      tcgen05 issuer: S = Q K_j^T into TMEM, then O += P V_j with P
//               read from TMEM (bf16, written over S by the softmax warps)
//   warps 2..5  softmax: thread r owns query row r (TMEM lane r); online
//               softmax in base 2 with a lazily moved row maximum, P to TMEM,
//               O rescaled in TMEM when the maximum moves, epilogue O / l and
//               LSE = ln2 * (m + log2 l)
// Two blocks share an SM (256 TMEM columns each), so one block's softmax
// overlaps the other's matrix multiplies.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_launch.h"
#include "exp2_poly.cuh"
#include "sm103_ptx.cuh"

namespace detattn {

__device__ unsigned int g_fwd_status;

namespace {

constexpr int kThreads = 320;  // producer, MMA issuer, 8 softmax warps
// The row maximum used in the exponent is only moved when the true maximum
// exceeds it by more than 2^8; until then P <= 256, which bf16 and the fp32
// accumulators hold exactly as well.  The final O / l and LSE are exact for
// any value of the stale maximum.
constexpr float kRescaleLog2 = 8.0f;
// Of every 8 consecutive pairs of scores, this many take 2^x from the FMA-pipe
// polynomial instead of the special-function unit, to balance the two.
#ifndef DETATTN_FWD_POLY_OF8
#define DETATTN_FWD_POLY_OF8 0
#endif
constexpr int kPolyOf8 = DETATTN_FWD_POLY_OF8;

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;                   // 128-byte swizzle atoms per row
  static constexpr int kTileBytes = kTileM * 128 * kAtoms;  // 128 rows x D bf16
  static constexpr int kStages = (D == 64) ? 2 : 1;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kSmemBytes = kOffV + kStages * kTileBytes + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColS = 0;    // S (fp32, 128 cols); P (bf16 pairs) of keys
                                          // 64h..64h+63 over cols 64h..64h+31
  static constexpr uint32_t kColO = 128;  // O accumulator, D cols
};

enum : int { kBarQ = 0, kBarKFull = 1, kBarVFull = 3, kBarKEmpty = 5, kBarVEmpty = 7,
             kBarS = 9, kBarP = 10, kBarO = 11, kBarDrain = 12, kNumBars = 13 };

__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mV, const FwdArgs a) {
  using C = Cfg<D>;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ uint32_t tmem_slot;
  __shared__ float red_max[2][2][kTileM];  // [tile parity][half][row] partial maxima
  __shared__ float red_l[2][kTileM];       // [half][row] partial row sums

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Heaviest query tiles (most key tiles under the causal mask) are handed out first.
  const int mt = a.n_m - 1 - static_cast<int>(blockIdx.x) / a.BHq;
  const int bh = static_cast<int>(blockIdx.x) % a.BHq;
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int hkv = h / (a.Hq / a.Hkv);
  const int m0 = mt * kTileM;
  const int n_kv = a.causal ? (mt + 1) : (a.T + kTileN - 1) / kTileN;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem) + C::kOffQ;
  const uint32_t sK0 = smem_u32(smem) + C::kOffK;
  const uint32_t sV0 = smem_u32(smem) + C::kOffV;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    mbar_init(bar(kBarS), 1);
    mbar_init(bar(kBarP), 8);
    mbar_init(bar(kBarO), 1);
    mbar_init(bar(kBarDrain), 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&mQ);
    tma_prefetch_desc(&mK);
    tma_prefetch_desc(&mV);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint64_t wait_ns = a.wait_ns;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
      mbar_arrive_expect_tx(bar(kBarQ), C::kTileBytes);
      for (int at = 0; at < C::kAtoms; ++at)
        tma_load_4d(sQ + at * 16384, &mQ, bar(kBarQ), at * 64, h, m0, b);
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % NS;
        const uint32_t ph = (j / NS) & 1;
        if (j >= NS && !(ok = mbar_wait(bar(kBarKEmpty + s), ph ^ 1, wait_ns))) break;
        mbar_arrive_expect_tx(bar(kBarKFull + s), C::kTileBytes);
        for (int at = 0; at < C::kAtoms; ++at)
          tma_load_4d(sK0 + s * C::kTileBytes + at * 16384, &mK, bar(kBarKFull + s), at * 64, hkv,
                      j * kTileN, b);
        last_k[s] = j;
        if (j >= NS && !(ok = mbar_wait(bar(kBarVEmpty + s), ph ^ 1, wait_ns))) break;
        mbar_arrive_expect_tx(bar(kBarVFull + s), C::kTileBytes);
        for (int at = 0; at < C::kAtoms; ++at)
          tma_load_4d(sV0 + s * C::kTileBytes + at * 16384, &mV, bar(kBarVFull + s), at * 64, hkv,
                      j * kTileN, b);
        last_v[s] = j;
      }
      if (!ok) {
        // Let every copy already issued land before the block's shared memory goes away.
        mbar_wait(bar(kBarQ), 0, wait_ns);
        for (int s = 0; s < NS; ++s) {
          if (last_k[s] >= 0) mbar_wait(bar(kBarKFull + s), (last_k[s] / NS) & 1, wait_ns);
          if (last_v[s] >= 0) mbar_wait(bar(kBarVFull + s), (last_v[s] / NS) & 1, wait_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t tS = tmem + C::kColS, tO = tmem + C::kColO;
      constexpr uint32_t kIdQK = idesc_bf16(kTileM, kTileN, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(kTileM, D, false, true);
      // Operand descriptors built once; the loops only add constant offsets.
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sK0, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sV0, 16384, 1024);
      ok = mbar_wait(bar(kBarQ), 0, wait_ns);
      tc_fence_after();
      for (int j = 0; j < n_kv && ok; ++j) {
        const int s = j % NS;
        const uint32_t ph = (j / NS) & 1;
        const uint64_t dK = desc_add(dK0, s * C::kTileBytes), dV = desc_add(dV0, s * C::kTileBytes);
        if (!(ok = mbar_wait(bar(kBarKFull + s), ph, wait_ns))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          constexpr uint32_t kAtom = 16384;
          const uint32_t off = (ks >> 2) * kAtom + (ks & 3) * 32;
          mma_ss(tS, desc_add(dQ, off), desc_add(dK, off), kIdQK, ks > 0);
        }
        mma_commit(bar(kBarS));
        mma_commit(bar(kBarKEmpty + s));
        if (!(ok = mbar_wait(bar(kBarP), j & 1, wait_ns))) break;
        if (!(ok = mbar_wait(bar(kBarVFull + s), ph, wait_ns))) break;
        tc_fence_after();
        // P of keys 16ks..16ks+15: half ks/4 wrote its 64 keys as 32 packed
        // columns at the start of its own 64 S columns.
#pragma unroll
        for (int ks = 0; ks < kTileN / 16; ++ks)
          mma_ts(tO, tS + (ks >> 2) * 64 + (ks & 3) * 8, desc_add(dV, ks * 2048), kIdPV,
                 (j > 0 || ks > 0) ? 1u : 0u);
        mma_commit(bar(kBarVEmpty + s));
        mma_commit(bar(kBarO));
      }
      // Every issued MMA must finish before TMEM is released.
      mma_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, wait_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    // Eight warps: warps w and w+4 share TMEM lane quarter (w & 3), i.e. the
    // same 32 query rows; "half" 0 takes key columns 0..63, half 1 64..127.
    // The two halves of a row trade their partial row maxima through shared
    // memory (one 64-thread named barrier per tile); the row sums stay split
    // until the epilogue.  Each half writes its P over its own S columns, so
    // the halves never touch each other's TMEM columns.
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int qrow = m0 + r;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t tS = tl + C::kColS + half * 64;  // this half's 64 score columns
    const float sl2 = a.scale_log2;
    const uint32_t pair_bar = 1 + quarter;          // named barrier of the two halves
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < n_kv; ++j) {
      ok = warp_all(mbar_wait(bar(kBarS), j & 1, wait_ns));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32_nowait(tS, sr[0]);
      tmem_ld32_nowait(tS + 32, sr[1]);
      tmem_wait_ld();
      reg_fence32(sr[0]);
      reg_fence32(sr[1]);

      const int kv0 = j * kTileN + half * 64;  // key of this half's first column
      const bool need_mask = a.causal ? (j == n_kv - 1) : (j * kTileN + kTileN > a.T);
      const int lim = need_mask ? (a.causal ? (qrow - kv0) : (a.T - 1 - kv0)) : (1 << 30);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c > lim) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
      }
      // Partial maximum over 64 columns in four independent chains.
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 32; ++c)
        mx4[c & 3] = fmax3(mx4[c & 3], __uint_as_float(sr[c >> 4][(2 * c) & 31]),
                           __uint_as_float(sr[c >> 4][(2 * c + 1) & 31]));
      const float mx_half = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      red_max[j & 1][half][r] = mx_half;
      named_barrier_sync(pair_bar, 64);
      const float mx = fmaxf(red_max[j & 1][0][r], red_max[j & 1][1][r]);
      const float m_new = mx * sl2;
      float alpha = 1.f;
      bool moved = false;
      if (m_new > m_run + kRescaleLog2) {
        alpha = ex2_approx(m_run - m_new);
        m_run = m_new;
        moved = true;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      const uint64_t sl2x2 = f2_make(sl2, sl2), neg_m = f2_make(-m_use, -m_use);
      uint64_t sum2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};  // four partial sums
      // P in two chunks of 32 scores (16 packed bf16 pairs each), stored over
      // this half's first 32 S columns (already read).
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = ch * 16 + i;  // pair index within the half: columns 2c, 2c+1
          const uint64_t x = f2_fma(f2_make(__uint_as_float(sr[ch][2 * i]),
                                            __uint_as_float(sr[ch][2 * i + 1])), sl2x2, neg_m);
          float x0, x1, p0, p1;
          f2_split(x, x0, x1);
          if ((c & 7) < kPolyOf8) {
            exp2_poly2(x0, x1, p0, p1);
          } else {
            p0 = ex2_approx(x0);
            p1 = ex2_approx(x1);
          }
          if (need_mask) {  // masked keys contribute exactly zero
            if (2 * c > lim) p0 = 0.f;
            if (2 * c + 1 > lim) p1 = 0.f;
          }
          sum2[i & 1] = f2_add(sum2[i & 1], f2_make(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16_nowait(tS + ch * 16, pk);
      }
      tmem_wait_st();
      if (j > 0 && __any_sync(0xffffffffu, moved)) {
        // O holds the sum over earlier tiles scaled by the old maximum: wait for
        // the last P V to land, then rescale this half's O columns in TMEM.
        ok = warp_all(mbar_wait(bar(kBarO), (j - 1) & 1, wait_ns));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t ov[32];
          const uint32_t col = C::kColO + half * (D / 2) + c * 32;
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
      if (lane == 0) mbar_arrive(bar(kBarP));
    }
    if (ok) ok = warp_all(mbar_wait(bar(kBarO), (n_kv - 1) & 1, wait_ns));
    // Row sum = half 0's part + half 1's part, in that order.
    red_l[half][r] = l_run;
    named_barrier_sync(pair_bar, 64);
    if (ok) {
      tc_fence_after();
      const float l_tot = red_l[0][r] + red_l[1][r];
      const float inv_l = 1.f / l_tot;
      const bool live = qrow < a.T;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) +
                            ((static_cast<size_t>(b) * a.T + qrow) * a.Hq + h) * D + half * (D / 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t ov[32];
        tmem_ld32(tl + C::kColO + half * (D / 2) + c * 32, ov);
        uint32_t pkd[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pkd[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l,
                               __uint_as_float(ov[2 * i + 1]) * inv_l);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
        }
      }
      if (live && half == 0)
        a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.T + qrow] =
            (m_run + log2f(l_tot)) * 0.69314718055994530942f;
    }
  }

  if (!ok) atomicOr(&g_fwd_status, 1u);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_fwd_t(int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const FwdArgs& a, cudaStream_t st) {
  const int smem = Cfg<D>::kSmemBytes;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  attn_fwd_kernel<D><<<grid, kThreads, smem, st>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int D, int grid, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const FwdArgs& a, cudaStream_t st) {
  return D == 64 ? launch_fwd_t<64>(grid, mq, mk, mv, a, st)
                 : launch_fwd_t<128>(grid, mq, mk, mv, a, st);
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

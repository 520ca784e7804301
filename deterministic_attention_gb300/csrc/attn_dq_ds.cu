// dQ of the stored-dS backward for sm_103a.
//
// RustingBrain vs PyTorch/TensorFlow page, "Where the time goes now": the
// backward's cost sits in the kernels that recompute the probabilities.  In
// this form the dK/dV step writes each dS tile it forms (bf16, dS^T layout)
// to the caller's workspace, and this kernel forms
//     dQ_i = scale * sum_j dS_ij K_j
// as a plain product on the tensor cores, without recomputing S, P or dP.
// oxide-train README, "The trainer is not bit-identical to itself after step
// 1": every dQ row is summed by one block over its key tiles in ascending
// order, with no atomics, so repeated runs give identical bits.
//
// One block per (b, query head, 128-query tile), heaviest first:
//   warp 0      TMA producer: per 64-key block, the two 64-query halves of
//               dS (MN-major A: queries contiguous) and the 64 K rows (MN-major
//               B: head dimension contiguous) into a ring of stages
//   warp 1      tcgen05.mma issuer: D[128 x D] += dS[128 x 64] K[64 x D]
//   warps 2-5   epilogue: TMEM -> scale -> bf16 dQ rows < T
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_launch.h"
#include "sm103_ptx.cuh"

namespace detattn {

__device__ unsigned int g_ds_status;

namespace {

constexpr int kDsThreads = 192;

template <int D>
struct DsCfg {
  static constexpr int kABytes = kTileM * 64 * 2;  // 128 queries x 64 keys
  static constexpr int kBBytes = 64 * D * 2;       // 64 keys x D
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = 4;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
  static_assert(kStageBytes % 1024 == 0, "stages keep the swizzle alignment");
};

enum : int { kSBarFull = 0, kSBarEmpty = 4, kSBarAcc = 8, kSBarDrain = 9, kSNumBars = 10 };

__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

template <int D>
__global__ void __launch_bounds__(kDsThreads, 1)
    attn_dq_from_ds_kernel(const __grid_constant__ CUtensorMap mDS, const __grid_constant__ CUtensorMap mK,
                           const BwdArgs a) {
  using Cf = DsCfg<D>;
  constexpr int NS = Cf::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kSNumBars];
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Unit (heaviest first): query tile mt of (b, h).
  const int u = blockIdx.x;
  const int mt = a.n_tiles - 1 - u / a.BH;
  const int bh = u % a.BH;
  const int b = bh / a.Hq, h = bh % a.Hq, hkv = h / (a.Hq / a.Hkv);
  const int n_kt = a.causal ? mt + 1 : (a.T + kTileN - 1) / kTileN;
  const int n_kb = 2 * n_kt;  // 64-key blocks
  const long pair0 = a.causal ? static_cast<long>(mt) * (mt + 1) / 2
                              : static_cast<long>(mt) * ((a.T + kTileN - 1) / kTileN);
  const long head_row0 = static_cast<long>(bh) * a.ds_pairs * 2 * kTileN;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s0 = smem_u32(smem);
  auto sA = [&](int s) { return s0 + s * Cf::kStageBytes; };
  auto sB = [&](int s) { return s0 + s * Cf::kStageBytes + Cf::kABytes; };
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), D);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(kSBarFull + s), 1);
      mbar_init(bar(kSBarEmpty + s), 1);
    }
    mbar_init(bar(kSBarAcc), 1);
    mbar_init(bar(kSBarDrain), 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&mDS);
    tma_prefetch_desc(&mK);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint64_t wait_ns = a.wait_ns;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      int last[NS];
      for (int s = 0; s < NS; ++s) last[s] = -1;
      for (int kb = 0; kb < n_kb; ++kb) {
        const int s = kb % NS;
        if (kb >= NS && !(ok = mbar_wait(bar(kSBarEmpty + s), ((kb / NS) & 1) ^ 1, wait_ns))) break;
        mbar_arrive_expect_tx(bar(kSBarFull + s), Cf::kStageBytes);
        const int kt = kb >> 1, sub = kb & 1;
        // dS rows of pair (mt, kt): half hf holds queries 64 hf .. 64 hf + 63,
        // one row per key; this block's keys are rows 64 sub .. 64 sub + 63.
        const long prow = head_row0 + (pair0 + kt) * 2 * kTileN + sub * 64;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_2d(sA(s) + hf * 8192, &mDS, bar(kSBarFull + s), 0,
                      static_cast<int>(prow + hf * kTileN));
#pragma unroll
        for (int at = 0; at < D / 64; ++at)
          tma_load_4d(sB(s) + at * 8192, &mK, bar(kSBarFull + s), at * 64, hkv, kt * kTileN + sub * 64,
                      b);
        last[s] = kb;
      }
      if (!ok)
        for (int s = 0; s < NS; ++s)
          if (last[s] >= 0) mbar_wait(bar(kSBarFull + s), (last[s] / NS) & 1, wait_ns);
    }
    // The warp meets again before the block-wide barrier below.
    __syncwarp();
  } else if (warp == 1) {
    // A: dS with queries (M) contiguous, two 64-query atoms 8 KB apart; B: K
    // with the head dimension (N) contiguous, 64-column atoms 8 KB apart.
    // Both step K (keys) by 16 rows of 128 bytes.
    constexpr uint32_t kId = idesc_bf16(kTileM, D, true, true);
    const uint64_t dA0 = sdesc_sw128(sA(0), 8192, 1024), dB0 = sdesc_sw128(sB(0), 8192, 1024);
    for (int kb = 0; kb < n_kb && ok; ++kb) {
      const int s = kb % NS;
      if (!(ok = warp_all(mbar_wait(bar(kSBarFull + s), (kb / NS) & 1, wait_ns)))) break;
      tc_fence_after();
      const uint64_t ad = desc_add(dA0, s * Cf::kStageBytes), bd = desc_add(dB0, s * Cf::kStageBytes);
      mma_ss_x4(tmem, ad, desc_add(ad, 2048), desc_add(ad, 4096), desc_add(ad, 6144), bd,
                desc_add(bd, 2048), desc_add(bd, 4096), desc_add(bd, 6144), kId, kb > 0 ? 1u : 0u);
      mma_commit(bar(kSBarEmpty + s));
    }
    mma_commit(bar(kSBarAcc));
    mma_commit(bar(kSBarDrain));
    warp_all(mbar_wait(bar(kSBarDrain), 0, wait_ns));
  } else {
    const int quarter = warp & 3;
    const int qrow = mt * kTileM + quarter * 32 + lane;
    ok = warp_all(mbar_wait(bar(kSBarAcc), 0, wait_ns));
    if (ok) {
      tc_fence_after();
      const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      uint32_t pkd[D / 2];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + c * 32, v);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pkd[16 * c + i] = pack_bf16x2(__uint_as_float(v[2 * i]) * a.scale,
                                        __uint_as_float(v[2 * i + 1]) * a.scale);
      }
      if (qrow < a.T) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dq) +
                                              ((static_cast<size_t>(b) * a.T + qrow) * a.Hq + h) * D);
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
          dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
      }
    }
  }
  if (!ok) atomicOr(&g_ds_status, 1u);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, D);
  }
}

template <int D>
cudaError_t launch_t(const CUtensorMap& mds, const CUtensorMap& mk, const BwdArgs& a, int n_units,
                     cudaStream_t st) {
  static unsigned long long attr_ctx[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long ctx = current_context_id();
  if (dev >= 64 || ctx == 0 || attr_ctx[dev] != ctx) {
    e = cudaFuncSetAttribute(attn_dq_from_ds_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DsCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_ctx[dev] = current_context_id();
  }
  attn_dq_from_ds_kernel<D><<<n_units, kDsThreads, DsCfg<D>::kSmemBytes, st>>>(mds, mk, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq_from_ds(int D, const CUtensorMap& mds, const CUtensorMap& mk,
                              const BwdArgs& a, int n_units, cudaStream_t st) {
  return D == 64 ? launch_t<64>(mds, mk, a, n_units, st) : launch_t<128>(mds, mk, a, n_units, st);
}

cudaError_t take_ds_status(cudaStream_t st, unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_ds_status, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v)
    e = cudaMemcpyToSymbolAsync(g_ds_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  *out = v;
  return e;
}

}  // namespace detattn

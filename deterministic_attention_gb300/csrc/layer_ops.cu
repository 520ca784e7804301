// Kernels around the attention in one layer of a training step, for sm_103a:
// a tcgen05 GEMM for the projections and their gradients, rotary positions
// (and their transpose for the gradients), and the AdamW update.
//
// RustingBrain vs PyTorch/TensorFlow page, "The setup": a decoder-only model
// of d_model 768 with 12 query heads over 4 KV heads of head_dim 64 and
// rotary positions; "Where the time goes now": GEMMs are most of a step.
// oxide-train README: the trainer ends its step with AdamW (LR 3e-4, weight
// decay 0.1), and "The trainer is not bit-identical to itself after step 1":
// every kernel here writes each output element once, in a fixed order, with
// no atomics, so the whole step repeats bit for bit.
//
// GEMM: C[M, N] = alpha * A[M, K] B[K, N], bf16 operands, fp32 accumulation
// in TMEM, C stored as bf16 or fp32.  Each operand is either K-major (K
// contiguous) or MN-major (M resp. N contiguous); both forms are what the
// tensor core reads from a 128-byte-swizzled tile, so a transposed operand
// costs nothing.  One block per 128 x BN tile of C, walking K in steps of 64
// in ascending order (the only order its sum is ever taken in):
//   warp 0      TMA producer: A and B tiles into a ring of stages
//   warp 1      tcgen05.mma issuer (M = 128, N = BN, K = 16 per instruction)
//   warps 2-5   epilogue: TMEM -> registers -> C, one row per thread
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "layer_launch.h"
#include "sm103_ptx.cuh"

namespace detattn {

__device__ unsigned int g_layer_status;

namespace {

constexpr int kGemmThreads = 192;
constexpr int kGemmBM = 128;
constexpr int kGemmBK = 64;

template <int BN>
struct GemmCfg {
  static constexpr int kABytes = kGemmBM * kGemmBK * 2;  // 16 KB
  static constexpr int kBBytes = BN * kGemmBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // Three stages of 32 KB, two blocks per SM, so one block's epilogue
  // overlaps the other's products.  (Measured per layer step: 204.6 us;
  // one block per SM with six stages 246 us before the split-K weight
  // gradients; 256-column blocks with four 48 KB stages 209.0 us.)
  static constexpr int kStages = 3;
  static constexpr int kBlocksPerSm = 2;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kStageBytes % 1024 == 0, "stages keep the swizzle alignment");
};

enum : int { kGBarFull = 0, kGBarEmpty = 8, kGBarAcc = 16, kGBarDrain = 17, kGNumBars = 18 };

__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

template <bool A_MN, bool B_MN, int BN, bool OUT_F32>
__global__ void __launch_bounds__(kGemmThreads, GemmCfg<BN>::kBlocksPerSm)
    gemm_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB,
                const GemmArgs g) {
  using Cf = GemmCfg<BN>;
  constexpr int NS = Cf::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kGNumBars];
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * kGemmBM;
  // This block's K range (all of K unless K is split).
  const int n_k = g.K / kGemmBK / g.k_splits;
  const int kb0 = blockIdx.z * n_k;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s0 = smem_u32(smem);
  auto sA = [&](int s) { return s0 + s * Cf::kStageBytes; };
  auto sB = [&](int s) { return s0 + s * Cf::kStageBytes + Cf::kABytes; };
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), BN);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(kGBarFull + s), 1);
      mbar_init(bar(kGBarEmpty + s), 1);
    }
    mbar_init(bar(kGBarAcc), 1);
    mbar_init(bar(kGBarDrain), 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&mA);
    tma_prefetch_desc(&mB);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      int last[8];
      for (int s = 0; s < 8; ++s) last[s] = -1;
      for (int kb = 0; kb < n_k; ++kb) {
        const int s = kb % NS;
        if (kb >= NS && !(ok = mbar_wait(bar(kGBarEmpty + s), ((kb / NS) & 1) ^ 1, g.wait_ns)))
          break;
        mbar_arrive_expect_tx(bar(kGBarFull + s), Cf::kStageBytes);
        const int k0 = (kb0 + kb) * kGemmBK;
        if constexpr (A_MN) {
          // Two 64-wide atoms of M, each [64 K rows x 128 B].
          tma_load_2d(sA(s), &mA, bar(kGBarFull + s), m0, k0);
          tma_load_2d(sA(s) + 8192, &mA, bar(kGBarFull + s), m0 + 64, k0);
        } else {
          tma_load_2d(sA(s), &mA, bar(kGBarFull + s), k0, m0);
        }
        if constexpr (B_MN) {
#pragma unroll
          for (int at = 0; at < BN / 64; ++at)
            tma_load_2d(sB(s) + at * 8192, &mB, bar(kGBarFull + s), n0 + 64 * at, k0);
        } else {
          tma_load_2d(sB(s), &mB, bar(kGBarFull + s), k0, n0);
        }
        last[s] = kb;
      }
      if (!ok)
        for (int s = 0; s < NS; ++s)
          if (last[s] >= 0) mbar_wait(bar(kGBarFull + s), (last[s] / NS) & 1, g.wait_ns);
    }
    // The warp meets again before the block-wide barrier below.
    __syncwarp();
  } else if (warp == 1) {
    constexpr uint32_t kId = idesc_bf16(kGemmBM, BN, A_MN, B_MN);
    // K-major tiles step K by 32 bytes inside the swizzled row; MN-major
    // tiles by 16 rows of 128 bytes.  MN-major atoms lie 8 KB apart (LBO).
    constexpr uint32_t kStepA = A_MN ? 2048u : 32u, kStepB = B_MN ? 2048u : 32u;
    const uint64_t dA0 = sdesc_sw128(sA(0), A_MN ? 8192 : 16, 1024);
    const uint64_t dB0 = sdesc_sw128(sB(0), B_MN ? 8192 : 16, 1024);
    for (int kb = 0; kb < n_k && ok; ++kb) {
      const int s = kb % NS;
      if (!(ok = warp_all(mbar_wait(bar(kGBarFull + s), (kb / NS) & 1, g.wait_ns)))) break;
      tc_fence_after();
      const uint64_t a = desc_add(dA0, s * Cf::kStageBytes), b = desc_add(dB0, s * Cf::kStageBytes);
      mma_ss_x4(tmem, a, desc_add(a, kStepA), desc_add(a, 2 * kStepA), desc_add(a, 3 * kStepA), b,
                desc_add(b, kStepB), desc_add(b, 2 * kStepB), desc_add(b, 3 * kStepB), kId,
                kb > 0 ? 1u : 0u);
      mma_commit(bar(kGBarEmpty + s));
    }
    mma_commit(bar(kGBarAcc));
    mma_commit(bar(kGBarDrain));
    warp_all(mbar_wait(bar(kGBarDrain), 0, g.wait_ns));
  } else {
    // Epilogue: warp w reads TMEM lanes 32 (w & 3) .. + 31, i.e. rows of C,
    // one row per thread, 32 columns at a time, stored as 16-byte vectors.
    // (Staging the chunks through shared memory so that each store writes
    // one row's consecutive columns measured slower: 206.8 against 204.6 us
    // per layer step.)
    const int quarter = warp & 3;
    const int row = m0 + quarter * 32 + lane;
    ok = warp_all(mbar_wait(bar(kGBarAcc), 0, g.wait_ns));
    if (ok) {
      tc_fence_after();
      const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + c * 32, v);
        const size_t base = static_cast<size_t>(row) * g.ldc + n0 + c * 32;
        if (g.k_splits > 1) {
          float4* dst = reinterpret_cast<float4*>(
              g.partial + (static_cast<size_t>(blockIdx.z) * g.M + row) * g.N + n0 + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        } else if constexpr (OUT_F32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(g.c) + base);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(v[4 * i]) * g.alpha, __uint_as_float(v[4 * i + 1]) * g.alpha,
                                 __uint_as_float(v[4 * i + 2]) * g.alpha,
                                 __uint_as_float(v[4 * i + 3]) * g.alpha);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g.c) + base);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            auto f = [&](int j) { return __uint_as_float(v[8 * i + j]) * g.alpha; };
            dst[i] = make_uint4(pack_bf16x2(f(0), f(1)), pack_bf16x2(f(2), f(3)),
                                pack_bf16x2(f(4), f(5)), pack_bf16x2(f(6), f(7)));
          }
        }
      }
    }
  }
  if (!ok) atomicOr(&g_layer_status, 1u);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }
}

template <bool A_MN, bool B_MN, int BN, bool OUT_F32>
cudaError_t launch_gemm_t(const CUtensorMap& ma, const CUtensorMap& mb, const GemmArgs& g,
                          cudaStream_t st) {
  using Cf = GemmCfg<BN>;
  static unsigned long long attr_ctx[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long ctx = current_context_id();
  if (dev >= 64 || ctx == 0 || attr_ctx[dev] != ctx) {
    e = cudaFuncSetAttribute(gemm_kernel<A_MN, B_MN, BN, OUT_F32>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_ctx[dev] = current_context_id();
  }
  const dim3 grid(g.N / BN, g.M / kGemmBM, g.k_splits);
  gemm_kernel<A_MN, B_MN, BN, OUT_F32><<<grid, kGemmThreads, Cf::kSmemBytes, st>>>(ma, mb, g);
  return cudaGetLastError();
}

// ------------------------------------------------------------ rotary positions
// Rotate-half rotary positions (the reading of "rotary positions" on the
// RustingBrain page): within each head, component i of the first half and
// component i of the second half turn together by the angle
// t * base^(-2i/D), t the token's position in its sequence:
//   x1' = x1 cos - x2 sin,   x2' = x2 cos + x1 sin.
// The angle is formed in fp32 as t * base^(-2i/D) and its sine and cosine
// come from sincosf.
__device__ __forceinline__ void rope_angle(int t, int i, int D, float log2_base, float* c, float* s) {
  const float inv = exp2f(-(2.0f * static_cast<float>(i) / static_cast<float>(D)) * log2_base);
  sincosf(static_cast<float>(t) * inv, s, c);
}

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void unpack8(uint4 x, float (&f)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// Splits the projection qkv [B*T, (Hq + 2 Hkv) D] (columns: Q heads, K heads,
// V heads) into q [B, T, Hq, D] and k [B, T, Hkv, D] rotated, and v copied.
// One thread per 8 pairs (i, i + D/2), i = 8c .. 8c + 7, of one head of one
// token: 16-byte loads and stores.  sign = +1 rotates by the angle, -1 by
// minus it (the transpose, for the gradients).
__device__ __forceinline__ void rotate8(float (&x1)[8], float (&x2)[8], int t, int i0, int D,
                                        float log2_base, float sign) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float c, sn;
    rope_angle(t, i0 + k, D, log2_base, &c, &sn);
    sn *= sign;
    const float a = x1[k], b = x2[k];
    x1[k] = a * c - b * sn;
    x2[k] = b * c + a * sn;
  }
}

__global__ void rope_split_kernel(const __nv_bfloat16* __restrict__ qkv, __nv_bfloat16* __restrict__ q,
                                  __nv_bfloat16* __restrict__ k, __nv_bfloat16* __restrict__ v,
                                  RopeArgs r) {
  const int H = r.Hq + 2 * r.Hkv, half = r.D / 2, nc = half / 8;
  const long n = static_cast<long>(r.B) * r.T * H * nc;
  for (long p = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; p < n;
       p += static_cast<long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(p % nc);
    const long th = p / nc;
    const int h = static_cast<int>(th % H);
    const long bt = th / H;
    const int t = static_cast<int>(bt % r.T);
    const __nv_bfloat16* src = qkv + bt * H * r.D + static_cast<long>(h) * r.D + 8 * c;
    const uint4 lo = *reinterpret_cast<const uint4*>(src);
    const uint4 hi = *reinterpret_cast<const uint4*>(src + half);
    __nv_bfloat16* dst;
    if (h < r.Hq)
      dst = q + (bt * r.Hq + h) * r.D;
    else if (h < r.Hq + r.Hkv)
      dst = k + (bt * r.Hkv + (h - r.Hq)) * r.D;
    else
      dst = v + (bt * r.Hkv + (h - r.Hq - r.Hkv)) * r.D;
    dst += 8 * c;
    if (h < r.Hq + r.Hkv) {
      float x1[8], x2[8];
      unpack8(lo, x1);
      unpack8(hi, x2);
      rotate8(x1, x2, t, 8 * c, r.D, r.log2_base, 1.0f);
      *reinterpret_cast<uint4*>(dst) = pack8(x1);
      *reinterpret_cast<uint4*>(dst + half) = pack8(x2);
    } else {
      *reinterpret_cast<uint4*>(dst) = lo;
      *reinterpret_cast<uint4*>(dst + half) = hi;
    }
  }
}

// The transpose for the gradients: dq, dk turned back by minus the angle
// and dv copied, joined into dqkv [B*T, (Hq + 2 Hkv) D].
__global__ void rope_merge_kernel(const __nv_bfloat16* __restrict__ dq, const __nv_bfloat16* __restrict__ dk,
                                  const __nv_bfloat16* __restrict__ dv, __nv_bfloat16* __restrict__ dqkv,
                                  RopeArgs r) {
  const int H = r.Hq + 2 * r.Hkv, half = r.D / 2, nc = half / 8;
  const long n = static_cast<long>(r.B) * r.T * H * nc;
  for (long p = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; p < n;
       p += static_cast<long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(p % nc);
    const long th = p / nc;
    const int h = static_cast<int>(th % H);
    const long bt = th / H;
    const int t = static_cast<int>(bt % r.T);
    const __nv_bfloat16* src;
    if (h < r.Hq)
      src = dq + (bt * r.Hq + h) * r.D;
    else if (h < r.Hq + r.Hkv)
      src = dk + (bt * r.Hkv + (h - r.Hq)) * r.D;
    else
      src = dv + (bt * r.Hkv + (h - r.Hq - r.Hkv)) * r.D;
    src += 8 * c;
    const uint4 lo = *reinterpret_cast<const uint4*>(src);
    const uint4 hi = *reinterpret_cast<const uint4*>(src + half);
    __nv_bfloat16* dst = dqkv + bt * H * r.D + static_cast<long>(h) * r.D + 8 * c;
    if (h < r.Hq + r.Hkv) {
      float y1[8], y2[8];
      unpack8(lo, y1);
      unpack8(hi, y2);
      rotate8(y1, y2, t, 8 * c, r.D, r.log2_base, -1.0f);
      *reinterpret_cast<uint4*>(dst) = pack8(y1);
      *reinterpret_cast<uint4*>(dst + half) = pack8(y2);
    } else {
      *reinterpret_cast<uint4*>(dst) = lo;
      *reinterpret_cast<uint4*>(dst + half) = hi;
    }
  }
}

// ------------------------------------------------------------ AdamW
// One update of step t (1-based) per element, in the oracle's order of
// operations: w <- w (1 - lr wd); m <- b1 m + (1 - b1) g; v <- b2 v +
// (1 - b2) g^2; w <- w - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps).
// Also writes the bf16 copy of w the next step's GEMMs read.  Four elements
// per thread (the layer's weights have multiples of 128 elements).
__device__ __forceinline__ float adamw_one(float& w, float& m, float& v, float g, const AdamArgs& a,
                                           float bc1, float bc2) {
  float wi = w * (1.0f - a.lr * a.wd);
  m = a.b1 * m + (1.0f - a.b1) * g;
  v = a.b2 * v + (1.0f - a.b2) * g * g;
  wi = wi - a.lr * (m / bc1) / (sqrtf(v / bc2) + a.eps);
  w = wi;
  return wi;
}

__global__ void adamw_kernel(float* __restrict__ w, float* __restrict__ m, float* __restrict__ v,
                             const float* __restrict__ grad, __nv_bfloat16* __restrict__ w_bf16,
                             long n, AdamArgs a) {
  const float bc1 = 1.0f - powf(a.b1, static_cast<float>(a.step));
  const float bc2 = 1.0f - powf(a.b2, static_cast<float>(a.step));
  const long n4 = n / 4;
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    float4 wi = reinterpret_cast<float4*>(w)[i], mi = reinterpret_cast<float4*>(m)[i];
    float4 vi = reinterpret_cast<float4*>(v)[i];
    const float4 gi = reinterpret_cast<const float4*>(grad)[i];
    const float r0 = adamw_one(wi.x, mi.x, vi.x, gi.x, a, bc1, bc2);
    const float r1 = adamw_one(wi.y, mi.y, vi.y, gi.y, a, bc1, bc2);
    const float r2 = adamw_one(wi.z, mi.z, vi.z, gi.z, a, bc1, bc2);
    const float r3 = adamw_one(wi.w, mi.w, vi.w, gi.w, a, bc1, bc2);
    reinterpret_cast<float4*>(w)[i] = wi;
    reinterpret_cast<float4*>(m)[i] = mi;
    reinterpret_cast<float4*>(v)[i] = vi;
    reinterpret_cast<uint2*>(w_bf16)[i] = make_uint2(pack_bf16x2(r0, r1), pack_bf16x2(r2, r3));
  }
}

// Split-K reduction: C = alpha * (partial[0] + partial[1] + ...), in
// ascending split order, four columns per thread.
template <bool OUT_F32>
__global__ void gemm_reduce_kernel(const GemmArgs g) {
  const long n4 = static_cast<long>(g.M) * g.N / 4;
  const long plane4 = n4;
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    float4 acc = reinterpret_cast<const float4*>(g.partial)[i];
    for (int z = 1; z < g.k_splits; ++z) {
      const float4 x = reinterpret_cast<const float4*>(g.partial)[z * plane4 + i];
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    const long row = (4 * i) / g.N, col = (4 * i) % g.N;
    const size_t at = static_cast<size_t>(row) * g.ldc + col;
    if constexpr (OUT_F32) {
      *reinterpret_cast<float4*>(static_cast<float*>(g.c) + at) =
          make_float4(acc.x * g.alpha, acc.y * g.alpha, acc.z * g.alpha, acc.w * g.alpha);
    } else {
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(g.c) + at) =
          make_uint2(pack_bf16x2(acc.x * g.alpha, acc.y * g.alpha),
                     pack_bf16x2(acc.z * g.alpha, acc.w * g.alpha));
    }
  }
}

int grid_of(long n, int block, int sms) {
  const long want = (n + block - 1) / block, cap = static_cast<long>(sms) * 16;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_gemm(bool a_mn, bool b_mn, bool out_f32, const CUtensorMap& ma,
                        const CUtensorMap& mb, const GemmArgs& g, cudaStream_t st) {
  constexpr int BN = kGemmBN;
  if (a_mn) {
    if (b_mn) return out_f32 ? launch_gemm_t<true, true, BN, true>(ma, mb, g, st)
                             : launch_gemm_t<true, true, BN, false>(ma, mb, g, st);
    return out_f32 ? launch_gemm_t<true, false, BN, true>(ma, mb, g, st)
                   : launch_gemm_t<true, false, BN, false>(ma, mb, g, st);
  }
  if (b_mn) return out_f32 ? launch_gemm_t<false, true, BN, true>(ma, mb, g, st)
                           : launch_gemm_t<false, true, BN, false>(ma, mb, g, st);
  return out_f32 ? launch_gemm_t<false, false, BN, true>(ma, mb, g, st)
                 : launch_gemm_t<false, false, BN, false>(ma, mb, g, st);
}

cudaError_t launch_gemm_reduce(const GemmArgs& g, bool out_f32, int sms, cudaStream_t st) {
  const long n4 = static_cast<long>(g.M) * g.N / 4;
  if (out_f32)
    gemm_reduce_kernel<true><<<grid_of(n4, 256, sms), 256, 0, st>>>(g);
  else
    gemm_reduce_kernel<false><<<grid_of(n4, 256, sms), 256, 0, st>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_rope_split(const void* qkv, void* q, void* k, void* v, const RopeArgs& r,
                              int sms, cudaStream_t st) {
  const long n = static_cast<long>(r.B) * r.T * (r.Hq + 2 * r.Hkv) * (r.D / 16);
  rope_split_kernel<<<grid_of(n, 256, sms), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(q),
      static_cast<__nv_bfloat16*>(k), static_cast<__nv_bfloat16*>(v), r);
  return cudaGetLastError();
}

cudaError_t launch_rope_merge(const void* dq, const void* dk, const void* dv, void* dqkv,
                              const RopeArgs& r, int sms, cudaStream_t st) {
  const long n = static_cast<long>(r.B) * r.T * (r.Hq + 2 * r.Hkv) * (r.D / 16);
  rope_merge_kernel<<<grid_of(n, 256, sms), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(dq), static_cast<const __nv_bfloat16*>(dk),
      static_cast<const __nv_bfloat16*>(dv), static_cast<__nv_bfloat16*>(dqkv), r);
  return cudaGetLastError();
}

cudaError_t launch_adamw(float* w, float* m, float* v, const float* grad, void* w_bf16, long n,
                         const AdamArgs& a, int sms, cudaStream_t st) {
  adamw_kernel<<<grid_of(n / 4, 256, sms), 256, 0, st>>>(w, m, v, grad,
                                                     static_cast<__nv_bfloat16*>(w_bf16), n, a);
  return cudaGetLastError();
}

cudaError_t take_layer_status(cudaStream_t st, unsigned* out) {
  unsigned val = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&val, g_layer_status, sizeof(val), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && val)
    e = cudaMemcpyToSymbolAsync(g_layer_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  *out = val;
  return e;
}

}  // namespace detattn

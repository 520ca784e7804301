// Internal interface of the layer kernels (layer_ops.cu): argument blocks and
// launch functions.  Not part of the public API.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace detattn {

constexpr int kGemmBN = 128;  // columns of C per block (rows: 128)

struct GemmArgs {
  void* c;                    // bf16 or fp32 [M, ldc] row-major
  int M, N, K;                // multiples of 128, kGemmBN and 64
  long ldc;
  float alpha;
  unsigned long long wait_ns;
  // Split K (k_splits > 1): block z of the grid's third dimension sums K
  // rows [z K / k_splits, (z + 1) K / k_splits) into fp32 partial[z] [M, N];
  // launch_gemm_reduce then adds the partials in ascending z into C.
  int k_splits;
  float* partial;
};
cudaError_t launch_gemm_reduce(const GemmArgs& g, bool out_f32, int sms, cudaStream_t st);

struct RopeArgs {
  int B, T, Hq, Hkv, D;
  float log2_base;            // log2 of the rotary base (10000)
};

struct AdamArgs {
  float lr, wd, b1, b2, eps;
  int step;                   // 1-based; the bias corrections are formed on the device
};

// a_mn / b_mn: the operand's M (resp. N) index is the contiguous one.  The
// tensor maps are 2-D bf16 maps with 128-byte swizzle: K-major A {K, M} with
// box {64, 128}; MN-major A {M, K} with box {64, 64}; K-major B {K, N} with
// box {64, kGemmBN}; MN-major B {N, K} with box {64, 64}.
cudaError_t launch_gemm(bool a_mn, bool b_mn, bool out_f32, const CUtensorMap& ma,
                        const CUtensorMap& mb, const GemmArgs& g, cudaStream_t st);
cudaError_t launch_rope_split(const void* qkv, void* q, void* k, void* v, const RopeArgs& r,
                              int sms, cudaStream_t st);
cudaError_t launch_rope_merge(const void* dq, const void* dk, const void* dv, void* dqkv,
                              const RopeArgs& r, int sms, cudaStream_t st);
cudaError_t launch_adamw(float* w, float* m, float* v, const float* grad, void* w_bf16, long n,
                         const AdamArgs& a, int sms, cudaStream_t st);
// Read-and-clear of the layer kernels' status word (bit 0: a GEMM wait ran
// out); synchronous on `st`.
cudaError_t take_layer_status(cudaStream_t st, unsigned* out);

unsigned long long current_context_id();

}  // namespace detattn

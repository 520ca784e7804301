// Deterministic gradient of an embedding lookup for sm_103a.
//
// oxide-train README, "The trainer is not bit-identical to itself after step
// 1": the trainer adds each token's gradient row into the embedding table's
// gradient with atomics, whose order changes from launch to launch, so two
// runs of one binary disagree from step 2 on.  The lookup X[t,:] = W[id_t,:]
// has the gradient
//     dW[v,:] = sum over t with id_t == v of dY[t,:]
// and here every element of dW is one fp32 sum in an order fixed by the ids
// alone, so repeated runs give identical bits.
//
// Steps (integer atomics only count and hand out slots: their results do not
// depend on the order in which they land):
//   1. count     n_v = #{t : id_t = v}                       (integer atomics)
//   2. offsets   o_v = n_0 + ... + n_{v-1}                   (one block scans)
//   3. fill      token t goes to some slot of [o_v, o_v + n_v) of `unsorted`
//   4. order     token t goes to slot o_v + #{t' in segment v : t' < t} of
//                `sorted`: each segment is in ascending token order, whatever
//                order step 3 left it in
//   5. sum       `sorted` is cut into runs of 32 entries; one warp per (run,
//                512-column slab) adds the dY rows of each id in the run in
//                ascending token order.  An id whose tokens lie inside one
//                run is final and stored in dW; an id that crosses runs
//                leaves one partial row per run it touches
//   6. rows      rows no token selects are written as zeros (right after
//                step 2); rows that crossed runs add their partials in run
//                order, one warp per (first crossed run boundary, 128
//                columns)
// The work is bound by HBM: dY is read once and every row of dW is written
// once (zero rows included), plus the partial rows of ids that cross runs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "embed_launch.h"

namespace detattn {

__device__ unsigned int g_embed_status;

namespace {

constexpr int kRun = 32;        // sorted entries per run (one per lane)
constexpr int kSlabF4 = 64;     // float4 column groups per slab (256 columns)
constexpr int kF4PerLane = kSlabF4 / 32;
constexpr int kAhead = 16;      // dY rows loaded ahead in the sum

__device__ __forceinline__ bool id_ok(int v, int V) { return v >= 0 && v < V; }

// 1. counts[v] += 1 per valid token; invalid ids are skipped here and in
// every later step, and flagged.
// Lanes of a warp holding the same id add once, through their lowest lane
// (frequent ids would otherwise queue many atomics on one address).
__global__ void embed_count_kernel(const int* __restrict__ ids, int* __restrict__ counts, int N,
                                   int V) {
  const int lane = threadIdx.x & 31;
  for (int t0 = (blockIdx.x * blockDim.x + threadIdx.x) & ~31; t0 < N;
       t0 += gridDim.x * blockDim.x) {
    const int t = t0 + lane;
    const int v = t < N ? ids[t] : -1;
    const bool good = t < N && id_ok(v, V);
    if (t < N && !good) atomicOr(&g_embed_status, 1u);
    const unsigned same = __match_any_sync(0xffffffffu, good ? v : -1);
    if (good && (same & ((1u << lane) - 1u)) == 0u) atomicAdd(counts + v, __popc(same));
  }
}

// 2. offsets[v] = sum of counts[0..v-1] for v = 0..V.  Block b takes ids
// [4096 b, 4096 b + 4096): it first adds up every count before its tile
// (coalesced, then a block reduction), then scans its own tile -- four
// adjacent counts per thread, warp shuffles over the thread totals, then
// over the warp totals.  Integer sums: the same in any order.  Also clears
// `cursor` for step 3.
constexpr int kScanTile = 4096;
__device__ __forceinline__ int block_scan_1024(int x, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += y;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  *total = warp_tot[31];
  const int r = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - x;
  __syncthreads();  // warp_tot may be reused
  return r;  // exclusive prefix of x over the block
}

__global__ void __launch_bounds__(1024) embed_scan_kernel(const int* __restrict__ counts,
                                                          int* __restrict__ offsets,
                                                          int* __restrict__ cursor, int V) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x;
  const int base = blockIdx.x * kScanTile;
  int before = 0;
  for (int v = tid; v < base; v += 1024) before += counts[v];
  int carry;
  block_scan_1024(before, warp_tot, &carry);  // carry = sum of counts[0 .. base)
  const int i0 = base + 4 * tid;
  int c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = i0 + k < V ? counts[i0 + k] : 0;
  const int s = c[0] + c[1] + c[2] + c[3];
  int tile_total;
  int run = carry + block_scan_1024(s, warp_tot, &tile_total);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (i0 + k < V) {
      offsets[i0 + k] = run;
      cursor[i0 + k] = 0;
      run += c[k];
    }
  if (base + kScanTile >= V && tid == 0) offsets[V] = carry + tile_total;
}

// 3. Each valid token takes a slot of its id's segment.
// Lanes with the same id take consecutive slots from one atomic.
__global__ void embed_fill_kernel(const int* __restrict__ ids, const int* __restrict__ offsets,
                                  int* __restrict__ cursor, int* __restrict__ unsorted, int N,
                                  int V) {
  const int lane = threadIdx.x & 31;
  for (int t0 = (blockIdx.x * blockDim.x + threadIdx.x) & ~31; t0 < N;
       t0 += gridDim.x * blockDim.x) {
    const int t = t0 + lane;
    const int v = t < N ? ids[t] : -1;
    const bool good = t < N && id_ok(v, V);
    const unsigned same = __match_any_sync(0xffffffffu, good ? v : -1);
    const int leader = __ffs(same) - 1;
    int base = 0;
    if (good && lane == leader) base = atomicAdd(cursor + v, __popc(same));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (good) unsorted[offsets[v] + base + __popc(same & ((1u << lane) - 1u))] = t;
  }
}

// 4. Token t's place in its segment is the number of the segment's tokens
// before it.  Tokens are distinct, so the places are a permutation.  One
// thread per entry of `unsorted`, which step 3 grouped by id, 256 entries
// per block.  Short segments (up to 64 tokens) are counted by each thread
// alone in global memory.  Each long segment (a frequent id) that the block
// touches is staged through shared memory in tiles, and the block's threads
// of that segment count against each tile.
constexpr int kOrderBlock = 256;
constexpr int kOrderTile = 4096;
constexpr int kOrderShort = 64;
__global__ void __launch_bounds__(kOrderBlock) embed_order_kernel(
    const int* __restrict__ ids, const int* __restrict__ offsets, const int* __restrict__ unsorted,
    int* __restrict__ sorted, int V) {
  __shared__ __align__(16) int tile[kOrderTile];
  __shared__ int long_seg[kOrderBlock];
  __shared__ int n_long;
  const int n_valid = offsets[V];
  const int e0 = blockIdx.x * kOrderBlock;
  if (e0 >= n_valid) return;
  if (threadIdx.x == 0) n_long = 0;
  __syncthreads();
  const int e = e0 + threadIdx.x;
  const bool live = e < n_valid;
  const int t = live ? unsorted[e] : 0;
  const int v = live ? ids[t] : 0;
  const int o = live ? offsets[v] : 0, n = live ? offsets[v + 1] - o : 0;
  // The first entry of each long segment in this block lists it (the list's
  // order is irrelevant: each segment's counts are its own).
  if (live && n > kOrderShort && e == max(o, e0)) long_seg[atomicAdd(&n_long, 1)] = v;
  int rank = 0;
  if (live && n <= kOrderShort) {
    int j = 0;
    for (; j + 4 <= n; j += 4) {
      const int a0 = unsorted[o + j], a1 = unsorted[o + j + 1], a2 = unsorted[o + j + 2],
                a3 = unsorted[o + j + 3];
      rank += (a0 < t) + (a1 < t) + (a2 < t) + (a3 < t);
    }
    for (; j < n; ++j) rank += unsorted[o + j] < t ? 1 : 0;
  }
  __syncthreads();
  const int nl = n_long;
  for (int li = 0; li < nl; ++li) {
    const int vs = long_seg[li];
    const int so = offsets[vs], sn = offsets[vs + 1] - so;
    const bool mine = live && v == vs;
    for (int b0 = 0; b0 < sn; b0 += kOrderTile) {
      const int nb = min(kOrderTile, sn - b0);
      __syncthreads();
      for (int j = threadIdx.x; j < kOrderTile; j += kOrderBlock)
        tile[j] = j < nb ? unsorted[so + b0 + j] : 0x7FFFFFFF;
      __syncthreads();
      if (mine) {
        const int4* t4 = reinterpret_cast<const int4*>(tile);
        int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
#pragma unroll 8
        for (int j = 0; j < (nb + 3) / 4; ++j) {
          const int4 x = t4[j];
          r0 += x.x < t;
          r1 += x.y < t;
          r2 += x.z < t;
          r3 += x.w < t;
        }
        rank += (r0 + r1) + (r2 + r3);
      }
    }
  }
  if (live) sorted[o + rank] = t;
}

__device__ __forceinline__ void add_bf16x4(float (&acc)[4], uint2 x) {
  acc[0] += __uint_as_float(x.x << 16);
  acc[1] += __uint_as_float(x.x & 0xFFFF0000u);
  acc[2] += __uint_as_float(x.y << 16);
  acc[3] += __uint_as_float(x.y & 0xFFFF0000u);
}

// 5. One warp per (run of 32 sorted entries, slab of 256 columns).  Lane l
// owns column groups slab*64 + l + 32k (k = 0, 1) of 4 floats each; entry j
// of the run is token sorted[32 r + j], read by all lanes.  The rows of one
// id are added in entry order.  Where an id's segment lies wholly inside the
// run its sum is final and goes to dW; otherwise it goes to the run's head
// partial (the segment began in an earlier run) or tail partial (it began in
// this run and goes on past it).
__global__ void __launch_bounds__(256, 2) embed_sum_kernel(EmbedArgs a) {
  const int lane = threadIdx.x & 31;
  const int n_valid = a.offsets[a.V];
  const int n_runs = (n_valid + kRun - 1) / kRun;
  const int n_f4 = a.E / 4;
  const int n_slabs = (n_f4 + kSlabF4 - 1) / kSlabF4;
  const long items = static_cast<long>(n_runs) * n_slabs;
  const long warps = static_cast<long>(gridDim.x) * (blockDim.x / 32);
  const uint2* dy = static_cast<const uint2*>(a.dy);
  for (long it = static_cast<long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5); it < items;
       it += warps) {
    const int r = static_cast<int>(it / n_slabs), slab = static_cast<int>(it % n_slabs);
    const int e0 = r * kRun, e1 = min(e0 + kRun, n_valid);
    const int n = e1 - e0;
    const int t_l = lane < n ? a.sorted[e0 + lane] : 0;
    const int v_l = lane < n ? a.ids[t_l] : -1;
    int g[kF4PerLane];
    bool gv[kF4PerLane];
#pragma unroll
    for (int k = 0; k < kF4PerLane; ++k) {
      g[k] = slab * kSlabF4 + lane + 32 * k;
      gv[k] = g[k] < n_f4;
    }
    float acc[kF4PerLane][4];
#pragma unroll
    for (int k = 0; k < kF4PerLane; ++k) acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.f;
    for (int j0 = 0; j0 < n; j0 += kAhead) {
      // Loads of up to kAhead rows, all issued before any is added.
      uint2 x[kAhead][kF4PerLane];
#pragma unroll
      for (int jj = 0; jj < kAhead; ++jj) {
        const int t = __shfl_sync(0xffffffffu, t_l, (j0 + jj) & 31);
#pragma unroll
        for (int k = 0; k < kF4PerLane; ++k)
          x[jj][k] = (j0 + jj < n && gv[k]) ? dy[static_cast<size_t>(t) * n_f4 + g[k]]
                                           : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int jj = 0; jj < kAhead; ++jj) {
        const int j = j0 + jj;
        if (j >= n) break;
        const int v = __shfl_sync(0xffffffffu, v_l, j);
        const int v_next = __shfl_sync(0xffffffffu, v_l, (j + 1) & 31);
#pragma unroll
        for (int k = 0; k < kF4PerLane; ++k) add_bf16x4(acc[k], x[jj][k]);
        if (j + 1 < n && v_next == v) continue;
        // The id's last entry in this run: store its sum.
        const int so = a.offsets[v], se = a.offsets[v + 1];
        const bool before = so < e0, after = se > e1;
        float* dst;
        if (!before && !after)
          dst = a.dw + static_cast<size_t>(v) * a.E;
        else if (before)
          dst = a.head + static_cast<size_t>(r) * a.E;
        else
          dst = a.tail + static_cast<size_t>(r) * a.E;
        float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int k = 0; k < kF4PerLane; ++k) {
          if (gv[k]) d4[g[k]] = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
          acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.f;
        }
      }
    }
  }
}

// 6a. Rows no token selects are zero: one warp per 8 consecutive rows (their
// offsets come in with one load per lane), each zero row written whole with
// lane-strided float4 stores.  Depends only on the offsets.
constexpr int kZeroRows = 8;
__global__ void __launch_bounds__(256) embed_zero_kernel(EmbedArgs a) {
  const int lane = threadIdx.x & 31;
  const int n_f4 = a.E / 4;
  const int n_blocks = (a.V + kZeroRows - 1) / kZeroRows;
  const int warps = gridDim.x * (blockDim.x / 32);
  for (int rb = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); rb < n_blocks; rb += warps) {
    const int v_l = rb * kZeroRows + (lane & (kZeroRows - 1));
    const int cnt_l = v_l < a.V ? a.offsets[v_l + 1] - a.offsets[v_l] : 1;
    for (int j = 0; j < kZeroRows; ++j) {
      const int v = rb * kZeroRows + j;
      if (v >= a.V || __shfl_sync(0xffffffffu, cnt_l, j) != 0) continue;
      float4* d4 = reinterpret_cast<float4*>(a.dw + static_cast<size_t>(v) * a.E);
      for (int g = lane; g < n_f4; g += 32) d4[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// 6b. Ids whose tokens cross runs.  Such an id crosses the boundary after its
// first run first; the item (that boundary, 128-column slab) owns its sum:
// the tail partial of the first run, then the head partials of the runs
// after it, in run order, one float4 per lane, with the partials of up to 16
// runs loaded before they are added.  A frequent id spreads over 12 such
// warps (one per slab at width 1536).
constexpr int kFixAhead = 16;
__global__ void __launch_bounds__(256) embed_fixup_kernel(EmbedArgs a) {
  const int lane = threadIdx.x & 31;
  const int n_valid = a.offsets[a.V];
  const int n_runs = (n_valid + kRun - 1) / kRun;
  const int n_f4 = a.E / 4;
  const int n_slabs = (n_f4 + 31) / 32;
  const long items = static_cast<long>(n_runs > 0 ? n_runs - 1 : 0) * n_slabs;
  const long warps = static_cast<long>(gridDim.x) * (blockDim.x / 32);
  for (long it = static_cast<long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5); it < items;
       it += warps) {
    const int rb = static_cast<int>(it / n_slabs), slab = static_cast<int>(it % n_slabs);
    // The id of the last entry of run rb, and whether it starts in rb and
    // goes on past it.
    const int v = a.ids[a.sorted[(rb + 1) * kRun - 1]];
    const int so = a.offsets[v], se = a.offsets[v + 1];
    if (so / kRun != rb || se <= (rb + 1) * kRun) continue;
    const int re = (se - 1) / kRun;
    const int g = slab * 32 + lane;
    if (g >= n_f4) continue;
    float4 acc = reinterpret_cast<const float4*>(a.tail + static_cast<size_t>(rb) * a.E)[g];
    for (int r0 = rb + 1; r0 <= re; r0 += kFixAhead) {
      float4 x[kFixAhead];
#pragma unroll
      for (int k = 0; k < kFixAhead; ++k)
        x[k] = r0 + k <= re
                   ? reinterpret_cast<const float4*>(a.head + static_cast<size_t>(r0 + k) * a.E)[g]
                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < kFixAhead; ++k) {
        if (r0 + k > re) break;
        acc.x += x[k].x;
        acc.y += x[k].y;
        acc.z += x[k].z;
        acc.w += x[k].w;
      }
    }
    reinterpret_cast<float4*>(a.dw + static_cast<size_t>(v) * a.E)[g] = acc;
  }
}

int grid_for(long threads, int block, int sms, int per_sm) {
  const long want = (threads + block - 1) / block;
  const long cap = static_cast<long>(sms) * per_sm;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_embed_grad(const EmbedArgs& a, int sms, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(a.counts, 0, sizeof(int) * static_cast<size_t>(a.V), st);
  if (e != cudaSuccess) return e;
  if (a.N > 0) {
    embed_count_kernel<<<grid_for(a.N, 256, sms, 8), 256, 0, st>>>(a.ids, a.counts, a.N, a.V);
  }
  embed_scan_kernel<<<(a.V + kScanTile - 1) / kScanTile, 1024, 0, st>>>(a.counts, a.offsets,
                                                                          a.cursor, a.V);
  {
    const long warps = (static_cast<long>(a.V) + kZeroRows - 1) / kZeroRows;
    embed_zero_kernel<<<grid_for(warps * 32, 256, sms, 8), 256, 0, st>>>(a);
  }
  if (a.N > 0) {
    embed_fill_kernel<<<grid_for(a.N, 256, sms, 8), 256, 0, st>>>(a.ids, a.offsets, a.cursor,
                                                                  a.unsorted, a.N, a.V);
    embed_order_kernel<<<(a.N + kOrderBlock - 1) / kOrderBlock, kOrderBlock, 0, st>>>(
        a.ids, a.offsets, a.unsorted, a.sorted, a.V);
    embed_sum_kernel<<<sms * 2, 256, 0, st>>>(a);
    const long n_slabs = (a.E / 4 + 31) / 32;
    const long warps = ((static_cast<long>(a.N) + kRun - 1) / kRun) * n_slabs;
    embed_fixup_kernel<<<grid_for(warps * 32, 256, sms, 8), 256, 0, st>>>(a);
  }
  return cudaGetLastError();
}

int embed_grad_launches(int N) { return N > 0 ? 7 : 2; }

cudaError_t take_embed_status(cudaStream_t st, unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_embed_status, sizeof(v), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v)
    e = cudaMemcpyToSymbolAsync(g_embed_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  *out = v;
  return e;
}

}  // namespace detattn

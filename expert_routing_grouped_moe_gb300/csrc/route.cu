// Router top-k and the grouped routing pass.
//
// Routing follows the Unsloth x NVIDIA article, section "Optimisation 3: MoE
// routing done in one grouped pass": flatten the [T,k] assignments, stable-
// sort them by expert id, one bincount, offsets from the counts, slice the
// token list by offsets -- with no per-expert data-dependent query.  On the
// GPU this is a counting sort in three kernels:
//
//   route_hist     per-CTA expert histogram of a contiguous chunk of the flat
//                  assignment list (warp __match_any_sync groups equal ids,
//                  the group leader adds __popc of the group), written
//                  expert-major: hist[g][cta]
//   route_scan     one CTA per expert: exclusive scan of hist[g][:] over the
//                  CTAs (block prefix sum), total -> counts[g]
//   route_scatter  every CTA scans counts -> offsets (and tile offsets) in
//                  shared memory, then re-walks its chunk in the same warp
//                  order: position = offsets[g] + hist-prefix + earlier warps
//                  of the CTA + rank among equal ids in earlier lanes.
//
// The walk order (CTA, then warp, then iteration, then lane) is ascending flat
// index, so equal ids keep ascending flat index: the sort is stable and the
// result is the unique one the oracle computes.
#include <cfloat>
#include <cmath>
#include <cstdint>

#include "internal.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive block-wide prefix sum of one int per thread; *total gets the sum.
__device__ int block_excl_scan(int v, int* total) {
  __shared__ int wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  const int res = (warp > 0 ? wsum[warp - 1] : 0) + x - v;
  *total = wsum[nw - 1];
  __syncthreads();
  return res;
}

// Expert id of flat assignment i (slot j = k is the shared expert, id E);
// -1 for i >= N or an id outside [0,E).
__device__ __forceinline__ int flat_id(const int32_t* __restrict__ ids, int i, int N, int k,
                                       int K, int E) {
  if (i >= N) return -1;
  const int t = i / K;
  const int j = i - t * K;
  if (j >= k) return E;
  const int e = __ldg(ids + static_cast<int64_t>(t) * k + j);
  return (e >= 0 && e < E) ? e : -2;
}

__global__ void __launch_bounds__(kRouteThreads) route_hist_kernel(
    const int32_t* __restrict__ ids, int N, int k, int K, int E, int G, int C,
    int32_t* __restrict__ hist, int* __restrict__ status) {
  extern __shared__ int cnt[];  // [kRouteWarps][G]
  for (int x = threadIdx.x; x < kRouteWarps * G; x += blockDim.x) cnt[x] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int base = blockIdx.x * kRouteChunk + warp * (32 * kRoutePerLane);
  int* my = cnt + warp * G;
  bool bad = false;
#pragma unroll
  for (int it = 0; it < kRoutePerLane; ++it) {
    const int i = base + it * 32 + lane;
    int e = flat_id(ids, i, N, k, K, E);
    bad |= (e == -2);
    const unsigned m = __match_any_sync(kFull, e);
    if (e >= 0 && lane == __ffs(m) - 1) my[e] += __popc(m);
    __syncwarp();
  }
  if (bad) atomicCAS(status, 0, kErrBadIds);
  __syncthreads();
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    int s = 0;
#pragma unroll
    for (int w = 0; w < kRouteWarps; ++w) s += cnt[w * G + e];
    hist[static_cast<int64_t>(e) * C + blockIdx.x] = s;
  }
}

__global__ void __launch_bounds__(1024) route_scan_kernel(int32_t* __restrict__ hist, int C,
                                                         int32_t* __restrict__ counts) {
  int32_t* h = hist + static_cast<int64_t>(blockIdx.x) * C;
  const int per = (C + blockDim.x - 1) / blockDim.x;
  const int lo = min(C, static_cast<int>(threadIdx.x) * per);
  const int hi = min(C, lo + per);
  int s = 0;
  for (int i = lo; i < hi; ++i) s += h[i];
  int total;
  int run = block_excl_scan(s, &total);
  for (int i = lo; i < hi; ++i) {
    const int v = h[i];
    h[i] = run;
    run += v;
  }
  if (threadIdx.x == 0) counts[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kRouteThreads) route_scatter_kernel(
    const int32_t* __restrict__ ids, int N, int k, int K, int E, int G, int C,
    const int32_t* __restrict__ hist, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ tile_off,
    int32_t* __restrict__ sorted_src, int32_t* __restrict__ dest_pos) {
  extern __shared__ int sm[];
  int* off = sm;            // [G+1]
  int* cnt = sm + (G + 1);  // [kRouteWarps][G]

  // offsets = exclusive scan of counts (every CTA, redundantly; G <= 1025)
  {
    const int per = (G + blockDim.x - 1) / blockDim.x;
    const int lo = min(G, static_cast<int>(threadIdx.x) * per);
    const int hi = min(G, lo + per);
    int s = 0, st = 0;
    for (int g = lo; g < hi; ++g) {
      const int c = __ldg(counts + g);
      s += c;
      st += (c + kTileM - 1) / kTileM;
    }
    int total, ttotal;
    int run = block_excl_scan(s, &total);
    int trun = block_excl_scan(st, &ttotal);
    for (int g = lo; g < hi; ++g) {
      const int c = __ldg(counts + g);
      off[g] = run;
      if (blockIdx.x == 0) {
        offsets[g] = run;
        tile_off[g] = trun;
      }
      run += c;
      trun += (c + kTileM - 1) / kTileM;
    }
    if (threadIdx.x == 0) {
      off[G] = total;
      if (blockIdx.x == 0) {
        offsets[G] = total;
        tile_off[G] = ttotal;
      }
    }
  }
  for (int x = threadIdx.x; x < kRouteWarps * G; x += blockDim.x) cnt[x] = 0;
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int base = blockIdx.x * kRouteChunk + warp * (32 * kRoutePerLane);
  int* my = cnt + warp * G;
  int ev[kRoutePerLane];
#pragma unroll
  for (int it = 0; it < kRoutePerLane; ++it) {
    const int i = base + it * 32 + lane;
    ev[it] = flat_id(ids, i, N, k, K, E);
    const unsigned m = __match_any_sync(kFull, ev[it]);
    if (ev[it] >= 0 && lane == __ffs(m) - 1) my[ev[it]] += __popc(m);
    __syncwarp();
  }
  __syncthreads();
  // starting position of every (warp, group) run inside this CTA's chunk
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    int run = off[g] + __ldg(hist + static_cast<int64_t>(g) * C + blockIdx.x);
#pragma unroll
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = cnt[w * G + g];
      cnt[w * G + g] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lt = lanemask_lt();
#pragma unroll
  for (int it = 0; it < kRoutePerLane; ++it) {
    const int i = base + it * 32 + lane;
    const int e = ev[it];
    const unsigned m = __match_any_sync(kFull, e);
    if (e >= 0) {
      const int pos = my[e] + __popc(m & lt);
      sorted_src[pos] = i;
      dest_pos[i] = pos;
    } else if (i < N) {
      dest_pos[i] = -1;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) my[e] += __popc(m);
    __syncwarp();
  }
  // sorted positions past the valid total (only when some ids were bad)
  for (int p = off[G] + blockIdx.x * blockDim.x + threadIdx.x; p < N;
       p += gridDim.x * blockDim.x)
    sorted_src[p] = -1;
}

// One warp per token: k rounds of warp arg-max (ties -> lower id), then the
// renormalised weights as a softmax over the selected logits.
template <int NC>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float* z = logits + static_cast<int64_t>(t) * E;
  float v[NC];
  unsigned avail = 0;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int e = c * 32 + lane;
    v[c] = e < E ? __ldg(z + e) : -INFINITY;
    if (e < E) avail |= 1u << c;
  }
  float my_val = 0.f;
  int my_id = 0;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = -1;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      if (((avail >> c) & 1u) && (bi < 0 || v[c] > bv)) {
        bv = v[c];
        bi = c * 32 + lane;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, o);
      const int oi = __shfl_xor_sync(kFull, bi, o);
      if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == r) {
      my_val = bv;
      my_id = bi;
    }
    if (bi >= 0 && (bi & 31) == lane) avail &= ~(1u << (bi >> 5));
  }
  const float m = __shfl_sync(kFull, my_val, 0);
  const float ex = lane < k ? expf(my_val - m) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  if (lane < k) {
    ids[static_cast<int64_t>(t) * k + lane] = my_id;
    w[static_cast<int64_t>(t) * k + lane] = ex / sum;
  }
}

}  // namespace

cudaError_t launch_router_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((T + 7) / 8), block(256);
  const int nc = (E + 31) / 32;
  if (nc <= 1) router_topk_kernel<1><<<grid, block, 0, s>>>(logits, T, E, k, ids, w);
  else if (nc <= 2) router_topk_kernel<2><<<grid, block, 0, s>>>(logits, T, E, k, ids, w);
  else if (nc <= 4) router_topk_kernel<4><<<grid, block, 0, s>>>(logits, T, E, k, ids, w);
  else if (nc <= 8) router_topk_kernel<8><<<grid, block, 0, s>>>(logits, T, E, k, ids, w);
  else if (nc <= 16) router_topk_kernel<16><<<grid, block, 0, s>>>(logits, T, E, k, ids, w);
  else router_topk_kernel<32><<<grid, block, 0, s>>>(logits, T, E, k, ids, w);
  return cudaGetLastError();
}

cudaError_t launch_route(const int32_t* ids, int T, int k, int E, int shared, int32_t* counts,
                         int32_t* offsets, int32_t* tile_off, int32_t* sorted_src,
                         int32_t* dest_pos, int32_t* hist, int* status, cudaStream_t s) {
  const int K = k + shared, G = E + shared;
  const int N = T * K;
  const int C = route_ctas(N > 0 ? N : 1);
  const size_t sm_hist = static_cast<size_t>(kRouteWarps) * G * sizeof(int);
  const size_t sm_scat = sm_hist + static_cast<size_t>(G + 1) * sizeof(int);
  route_hist_kernel<<<C, kRouteThreads, sm_hist, s>>>(ids, N, k, K, E, G, C, hist, status);
  route_scan_kernel<<<G, 1024, 0, s>>>(hist, C, counts);
  route_scatter_kernel<<<C, kRouteThreads, sm_scat, s>>>(ids, N, k, K, E, G, C, hist, counts,
                                                         offsets, tile_off, sorted_src,
                                                         dest_pos);
  return cudaGetLastError();
}

}  // namespace moe

// Router top-k and the grouped routing pass.
//
// Routing follows the Unsloth x NVIDIA article, section "Optimisation 3: MoE
// routing done in one grouped pass": flatten the [T,k] assignments, stable-
// sort them by expert id, one bincount, offsets from the counts, slice the
// token list by offsets -- with no per-expert data-dependent query.  On the
// GPU this is a counting sort in three kernels:
//
//   route_hist     per-CTA expert histogram of a contiguous chunk of the flat
//                  assignment list (per-warp shared-memory counters), written
//                  expert-major: hist[g][cta]
//   route_scan     one CTA per expert: exclusive scan of hist[g][:] over the
//                  CTAs (block prefix sum), total -> counts[g]
//   route_scatter  every CTA scans counts -> offsets (and tile offsets) in one
//                  warp, re-walks its chunk in the same warp order and ranks
//                  equal ids among earlier lanes with a ballot-per-bit warp
//                  match (warp multisplit); position = offsets[g] + earlier
//                  CTAs (scanned histogram) + earlier warps + rank.  The chunk
//                  is sorted in shared memory first, so sorted_src leaves the
//                  CTA as contiguous per-expert runs.
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

// Lanes of the warp holding the same value v (0 <= v < 2^nbits): one ballot
// per bit, keeping the lanes that agree on every bit (warp multisplit).
__device__ __forceinline__ unsigned warp_match(unsigned v, int nbits) {
  unsigned m = kFull;
  for (int b = 0; b < nbits; ++b) {
    const unsigned bit = (v >> b) & 1u;
    const unsigned bal = __ballot_sync(kFull, bit);
    m &= bit ? bal : ~bal;
  }
  return m;
}

__device__ __forceinline__ int bits_for(int n) {  // bits to encode 0..n-1
  return 32 - __clz(n > 1 ? n - 1 : 1);
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
template <bool SHARED>
__device__ __forceinline__ int flat_id(const int32_t* __restrict__ ids, int i, int N, int k,
                                       int K, int E) {
  if (i >= N) return -1;
  int e;
  if (SHARED) {
    const int t = i / K;
    const int j = i - t * K;
    if (j >= k) return E;
    e = __ldg(ids + static_cast<int64_t>(t) * k + j);
  } else {
    e = __ldg(ids + i);  // K == k: flat index i is the i-th id
  }
  return (e >= 0 && e < E) ? e : -2;
}

template <int PER, bool SHARED>
__global__ void __launch_bounds__(kRouteThreads) route_hist_kernel(
    const int32_t* __restrict__ ids, int N, int k, int K, int E, int G, int C,
    int32_t* __restrict__ hist, int* __restrict__ status) {
  extern __shared__ int cnt[];  // [kRouteWarps][G]
  for (int x = threadIdx.x; x < kRouteWarps * G; x += blockDim.x) cnt[x] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int base = blockIdx.x * (kRouteThreads * PER) + warp * (32 * PER);
  int* my = cnt + warp * G;
  bool bad = false;
#pragma unroll 4
  for (int it = 0; it < PER; ++it) {
    const int i = base + it * 32 + lane;
    const int e = flat_id<SHARED>(ids, i, N, k, K, E);
    bad |= (e == -2);
    if (e >= 0) atomicAdd(my + e, 1);
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

// Shared memory of the scatter kernel, in ints.
__host__ __device__ constexpr int scatter_smem_ints(int G, int chunk) {
  return (G + 1) /*off*/ + kRouteWarps * G /*cnt*/ + (G + 1) /*lbase*/ + G /*gbase*/ +
         2 * chunk /*flat index, global position*/;
}

template <int PER, bool SHARED>
__global__ void __launch_bounds__(kRouteThreads) route_scatter_kernel(
    const int32_t* __restrict__ ids, int N, int k, int K, int E, int G, int C,
    const int32_t* __restrict__ hist, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ tile_off,
    int32_t* __restrict__ sorted_src, int32_t* __restrict__ dest_pos) {
  constexpr int CH = kRouteThreads * PER;
  extern __shared__ int sm[];
  int* off = sm;                      // [G+1] global offsets
  int* cnt = off + (G + 1);           // [8][G] per-warp counts -> per-warp local starts
  int* lbase = cnt + kRouteWarps * G;  // [G+1] start of group g inside this CTA's chunk
  int* gbase = lbase + (G + 1);       // [G]   global start of this CTA's run of group g
  int* stage = gbase + G;             // [CH]  flat index at each chunk-local sorted position
  int* stage_dst = stage + CH;        // [CH]  its global sorted position
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // offsets (and tile offsets) = exclusive scans of counts, by warp 0
  if (warp == 0) {
    const int per = (G + 31) / 32;
    const int lo = min(G, lane * per), hi = min(G, lo + per);
    int s = 0, st = 0;
    for (int g = lo; g < hi; ++g) {
      const int c = __ldg(counts + g);
      s += c;
      st += (c + kTileM - 1) / kTileM;
    }
    int xs = s, xt = st;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ys = __shfl_up_sync(kFull, xs, o), yt = __shfl_up_sync(kFull, xt, o);
      if (lane >= o) {
        xs += ys;
        xt += yt;
      }
    }
    int run = xs - s, trun = xt - st;
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
    if (lane == 31) {
      off[G] = xs;
      if (blockIdx.x == 0) {
        offsets[G] = xs;
        tile_off[G] = xt;
      }
    }
  } else {
    for (int x = threadIdx.x - 32; x < kRouteWarps * G; x += blockDim.x - 32) cnt[x] = 0;
  }
  __syncthreads();

  // pass 1: per-warp counts of this warp's contiguous run of assignments
  const int base = blockIdx.x * CH + warp * (32 * PER);
  int* my = cnt + warp * G;
  int ev[PER];
#pragma unroll
  for (int it = 0; it < PER; ++it) {
    const int i = base + it * 32 + lane;
    ev[it] = flat_id<SHARED>(ids, i, N, k, K, E);
    if (ev[it] >= 0) atomicAdd(my + ev[it], 1);
  }
  __syncthreads();

  // chunk-local group starts (scan over g), per-warp starts, global run starts
  {
    const int per = (G + kRouteThreads - 1) / kRouteThreads;
    const int lo = min(G, static_cast<int>(threadIdx.x) * per), hi = min(G, lo + per);
    int s = 0;
    for (int g = lo; g < hi; ++g)
#pragma unroll
      for (int w = 0; w < kRouteWarps; ++w) s += cnt[w * G + g];
    int total;
    int run = block_excl_scan(s, &total);
    for (int g = lo; g < hi; ++g) {
      lbase[g] = run;
      gbase[g] = off[g] + __ldg(hist + static_cast<int64_t>(g) * C + blockIdx.x);
#pragma unroll
      for (int w = 0; w < kRouteWarps; ++w) {
        const int c = cnt[w * G + g];
        cnt[w * G + g] = run;
        run += c;
      }
    }
    if (threadIdx.x == 0) lbase[G] = total;
  }
  __syncthreads();

  // pass 2: stable chunk-local position; dest_pos straight to global memory
  const unsigned lt = lanemask_lt();
  const int nbits = bits_for(G);
#pragma unroll
  for (int it = 0; it < PER; ++it) {
    const int i = base + it * 32 + lane;
    const int e = ev[it];
    // lanes holding the same valid id (invalid lanes match nothing)
    const unsigned m = __ballot_sync(kFull, e >= 0) &
                       warp_match(static_cast<unsigned>(e >= 0 ? e : 0), nbits);
    if (e >= 0) {
      const int lp = my[e] + __popc(m & lt);
      const int dst = gbase[e] + (lp - lbase[e]);
      stage[lp] = i;
      stage_dst[lp] = dst;
      dest_pos[i] = dst;
    } else if (i < N) {
      dest_pos[i] = -1;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) my[e] += __popc(m);
    __syncwarp();
  }
  __syncthreads();

  // sorted_src as contiguous per-group runs (consecutive threads, consecutive addresses)
  const int n_local = lbase[G];
  for (int lp = threadIdx.x; lp < n_local; lp += blockDim.x) sorted_src[stage_dst[lp]] = stage[lp];
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

template <int PER, bool SHARED>
cudaError_t launch_route_per(const int32_t* ids, int N, int k, int K, int E, int G, int C,
                             int32_t* counts, int32_t* offsets, int32_t* tile_off,
                             int32_t* sorted_src, int32_t* dest_pos, int32_t* hist, int* status,
                             cudaStream_t s) {
  const size_t sm_hist = static_cast<size_t>(kRouteWarps) * G * sizeof(int);
  const size_t sm_scat = static_cast<size_t>(scatter_smem_ints(G, kRouteThreads * PER)) * 4;
  cudaError_t e = cudaFuncSetAttribute(route_scatter_kernel<PER, SHARED>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sm_scat));
  if (e != cudaSuccess) return e;
  route_hist_kernel<PER, SHARED><<<C, kRouteThreads, sm_hist, s>>>(ids, N, k, K, E, G, C, hist,
                                                                   status);
  route_scan_kernel<<<G, 1024, 0, s>>>(hist, C, counts);
  route_scatter_kernel<PER, SHARED><<<C, kRouteThreads, sm_scat, s>>>(
      ids, N, k, K, E, G, C, hist, counts, offsets, tile_off, sorted_src, dest_pos);
  return cudaGetLastError();
}

cudaError_t launch_route(const int32_t* ids, int T, int k, int E, int shared, int32_t* counts,
                         int32_t* offsets, int32_t* tile_off, int32_t* sorted_src,
                         int32_t* dest_pos, int32_t* hist, int* status, cudaStream_t s) {
  const int K = k + shared, G = E + shared;
  const int N = T * K;
  const int C = route_ctas(N > 0 ? N : 1);
#define MOE_ROUTE_CASE(P)                                                                  \
  case P:                                                                                  \
    return shared ? launch_route_per<P, true>(ids, N, k, K, E, G, C, counts, offsets,     \
                                              tile_off, sorted_src, dest_pos, hist, status, s) \
                  : launch_route_per<P, false>(ids, N, k, K, E, G, C, counts, offsets,    \
                                               tile_off, sorted_src, dest_pos, hist, status, s);
  switch (route_per_lane(N)) {
    MOE_ROUTE_CASE(16)
    MOE_ROUTE_CASE(8)
    default:
      return shared ? launch_route_per<4, true>(ids, N, k, K, E, G, C, counts, offsets, tile_off,
                                                sorted_src, dest_pos, hist, status, s)
                    : launch_route_per<4, false>(ids, N, k, K, E, G, C, counts, offsets,
                                                 tile_off, sorted_src, dest_pos, hist, status, s);
  }
#undef MOE_ROUTE_CASE
}

}  // namespace moe

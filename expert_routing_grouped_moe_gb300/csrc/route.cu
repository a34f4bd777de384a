// Router top-k and the grouped routing pass.
//
// Routing follows the Unsloth x NVIDIA article, section "Optimisation 3: MoE
// routing done in one grouped pass": flatten the [T,k] assignments, stable-
// sort them by expert id, one bincount, offsets from the counts, slice the
// token list by offsets -- with no per-expert data-dependent query.  On the
// GPU this is a counting sort in three kernels (two for small inputs):
//
//   route_hist     per-CTA expert histogram of a contiguous chunk of the flat
//                  assignment list (per-warp shared-memory counters), written
//                  expert-major: hist[g][cta]
//   route_scan     one CTA per expert: exclusive scan of hist[g][:] over the
//                  CTAs (block prefix sum), total -> counts[g].  Skipped when
//                  the table is small (C <= kFusedScanCtas): each scatter CTA
//                  then sums its own column prefix and the totals itself.
//   route_scatter  every CTA scans counts -> offsets (and tile offsets) in one
//                  warp, re-walks its chunk in the same warp order and ranks
//                  equal ids among earlier lanes with a ballot-per-bit warp
//                  match (warp multisplit); position = offsets[g] + earlier
//                  CTAs (scanned histogram) + earlier warps + rank.  The chunk
//                  is sorted in shared memory first, so sorted_src leaves the
//                  CTA as one contiguous run per expert, written by one warp.
//
// The walk order (CTA, then warp, then iteration, then lane) is ascending flat
// index, so equal ids keep ascending flat index: the sort is stable and the
// result is the unique one the oracle computes.
#include <cfloat>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Lanes of the warp holding the same value v (0 <= v < 2^NB): one ballot per
// bit, keeping the lanes that agree on every bit (warp multisplit).  Bits
// above the values' width are zero in every lane and cost one no-op ballot.
template <int NB>
__device__ __forceinline__ unsigned warp_match(unsigned v) {
  unsigned m = kFull;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const unsigned bit = (v >> b) & 1u;
    const unsigned bal = __ballot_sync(kFull, bit);
    m &= ~(bal ^ (0u - bit));  // lanes whose bit b equals this lane's
  }
  return m;
}

// Bits of the group ids the scatter kernel matches on (groups 0..G-1).
inline int match_bits(int G) { return G <= 64 ? 6 : G <= 128 ? 7 : G <= 256 ? 8 : 11; }

// Expert id as loaded -> routed group (>= 0), -2 for an id outside [0,E).
__device__ __forceinline__ int classify(int e, int E) { return (e >= 0 && e < E) ? e : -2; }

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

// Expert ids of this lane's PER assignments of its warp's run [base, base +
// 32*PER): ev[it] is flat index base + it*32 + lane (-1 past N, -2 bad id).
// Without a shared expert and with 16-byte aligned ids the lane loads them as
// int4 vectors, all in flight at once: ids of flat index base + (v*32 +
// lane)*4 + c, so ev[] is then in a different order (the counts do not care).
template <int PER, bool SHARED>
__device__ __forceinline__ void load_ids_any_order(const int32_t* __restrict__ ids, int base,
                                                   int lane, int N, int k, int K, int E,
                                                   bool vec, int (&ev)[PER]) {
  if (!SHARED && vec) {
#pragma unroll
    for (int v = 0; v < PER / 4; ++v) {
      const int i0 = base + (v * 32 + lane) * 4;
      if (i0 + 3 < N) {
        const int4 q = __ldg(reinterpret_cast<const int4*>(ids + i0));
        ev[4 * v + 0] = classify(q.x, E);
        ev[4 * v + 1] = classify(q.y, E);
        ev[4 * v + 2] = classify(q.z, E);
        ev[4 * v + 3] = classify(q.w, E);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          ev[4 * v + c] = i0 + c < N ? classify(__ldg(ids + i0 + c), E) : -1;
      }
    }
  } else {
#pragma unroll
    for (int it = 0; it < PER; ++it) ev[it] = flat_id<SHARED>(ids, base + it * 32 + lane, N, k, K, E);
  }
}

template <int PER, bool SHARED>
__global__ void __launch_bounds__(kRouteThreads) route_hist_kernel(
    const int32_t* __restrict__ ids, int N, int k, int K, int E, int G, int C, int vec,
    int32_t* __restrict__ hist, int* __restrict__ status) {
  extern __shared__ int cnt[];  // [kRouteWarps][G]
  for (int x = threadIdx.x; x < kRouteWarps * G; x += blockDim.x) cnt[x] = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int base = blockIdx.x * (kRouteThreads * PER) + warp * (32 * PER);
  pdl_wait();
  int ev[PER];
  load_ids_any_order<PER, SHARED>(ids, base, lane, N, k, K, E, vec != 0, ev);
  __syncthreads();
  int* my = cnt + warp * G;
  bool bad = false;
#pragma unroll
  for (int it = 0; it < PER; ++it) {
    bad |= (ev[it] == -2);
    if (ev[it] >= 0) atomicAdd(my + ev[it], 1);
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
  pdl_wait();
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

// Routing CTAs up to which the scatter kernel scans the per-CTA histogram
// itself (G * C loads per CTA) instead of a separate scan kernel.
constexpr int kFusedScanCtas = 64;

// Shared memory of the scatter kernel, in ints.
__host__ __device__ constexpr int scatter_smem_ints(int G, int chunk) {
  return (G + 1) /*off*/ + kRouteWarps * G /*cnt*/ + (G + 1) /*lbase*/ + G /*delta*/ +
         2 * G /*fused scan: totals, this CTA's prefix*/ +
         chunk /*flat index at each chunk-local sorted position*/ +
         chunk / 2 /*its group, 16 bits*/;
}

template <int PER, bool SHARED, int NB>
__global__ void __launch_bounds__(kRouteThreads, 4) route_scatter_kernel(
    const int32_t* __restrict__ ids, int N, int k, int K, int E, int G, int C,
    const int32_t* __restrict__ hist, int32_t* __restrict__ counts, int fused,
    int32_t* __restrict__ offsets, int32_t* __restrict__ tile_off,
    int32_t* __restrict__ sorted_src, int32_t* __restrict__ dest_pos) {
  // fused: hist holds raw per-CTA counts (no scan kernel ran); else hist
  // holds the exclusive prefix over CTAs and counts the totals
  constexpr int CH = kRouteThreads * PER;
  extern __shared__ int sm[];
  int* off = sm;                      // [G+1] global offsets
  int* cnt = off + (G + 1);           // [8][G] per-warp counts -> per-warp local starts
  int* lbase = cnt + kRouteWarps * G;  // [G+1] start of group g inside this CTA's chunk
  int* delta = lbase + (G + 1);       // [G]   global position - chunk-local position, group g
  int* tot = delta + G;               // [G]   fused: total of group g over all CTAs
  int* pre = tot + G;                 // [G]   fused: group g in the CTAs before this one
  int* stage = pre + G;               // [CH]  flat index at each chunk-local sorted position
  uint16_t* stage_g = reinterpret_cast<uint16_t*>(stage + CH);  // [CH] its group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();

  // this warp's ids, in walk order (all loads in flight before the scans)
  const int base = blockIdx.x * CH + warp * (32 * PER);
  int ev[PER];
#pragma unroll
  for (int it = 0; it < PER; ++it) ev[it] = flat_id<SHARED>(ids, base + it * 32 + lane, N, k, K, E);

  if (fused) {
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
      const int32_t* h = hist + static_cast<int64_t>(g) * C;
      int before = 0, all = 0;
      for (int c = 0; c < C; ++c) {
        const int v = __ldg(h + c);
        before += c < static_cast<int>(blockIdx.x) ? v : 0;
        all += v;
      }
      tot[g] = all;
      pre[g] = before;
      if (blockIdx.x == 0) counts[g] = all;
    }
    __syncthreads();
  }

  // offsets (and tile offsets) = exclusive scans of counts, by warp 0
  if (warp == 0) {
    const int per = (G + 31) / 32;
    const int lo = min(G, lane * per), hi = min(G, lo + per);
    int s = 0, st = 0;
    for (int g = lo; g < hi; ++g) {
      const int c = fused ? tot[g] : __ldg(counts + g);
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
      const int c = fused ? tot[g] : __ldg(counts + g);
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
  int* my = cnt + warp * G;
  bool valid = true;
#pragma unroll
  for (int it = 0; it < PER; ++it) {
    valid &= ev[it] >= 0;
    if (ev[it] >= 0) atomicAdd(my + ev[it], 1);
  }
  const bool all_valid = __all_sync(kFull, valid);
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
      const int before =
          fused ? pre[g] : __ldg(hist + static_cast<int64_t>(g) * C + blockIdx.x);
      delta[g] = off[g] + before - run;
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
  int32_t* dp = dest_pos + base + lane;  // dest_pos of element it: dp[it * 32]
  if (all_valid) {
    // every element of this warp's run exists and has a valid id
#pragma unroll
    for (int it = 0; it < PER; ++it) {
      const int e = ev[it];
      const unsigned m = warp_match<NB>(static_cast<unsigned>(e));
      const int lp = my[e] + __popc(m & lt);
      stage[lp] = base + it * 32 + lane;
      stage_g[lp] = static_cast<uint16_t>(e);
      dp[it * 32] = delta[e] + lp;
      __syncwarp();
      if ((m >> lane) == 1u) my[e] = lp + 1;  // the last matching lane
      __syncwarp();
    }
  } else {
#pragma unroll
    for (int it = 0; it < PER; ++it) {
      const int i = base + it * 32 + lane;
      const int e = ev[it];
      // lanes holding the same valid id (invalid lanes match nothing)
      const unsigned m = __ballot_sync(kFull, e >= 0) &
                         warp_match<NB>(static_cast<unsigned>(e >= 0 ? e : 0));
      int lp = 0;
      if (e >= 0) {
        lp = my[e] + __popc(m & lt);
        stage[lp] = i;
        stage_g[lp] = static_cast<uint16_t>(e);
        dp[it * 32] = delta[e] + lp;
      } else if (i < N) {
        dp[it * 32] = -1;
      }
      __syncwarp();
      if (e >= 0 && (m >> lane) == 1u) my[e] = lp + 1;
      __syncwarp();
    }
  }
  __syncthreads();

  // sorted_src: each group's run of this chunk is contiguous both in the
  // stage and in global memory (position q of the stage goes to delta[g] + q);
  // consecutive threads copy consecutive positions
  for (int q = threadIdx.x; q < lbase[G]; q += kRouteThreads)
    sorted_src[delta[stage_g[q]] + q] = stage[q];
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
  pdl_wait();
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

int route_kernel_count(int64_t n, int G) {
  (void)G;
  return route_ctas(n > 0 ? n : 1) <= kFusedScanCtas ? 2 : 3;
}

cudaError_t launch_router_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((T + 7) / 8), block(256);
  const int nc = (E + 31) / 32;
  if (nc <= 1) return launch_pdl(router_topk_kernel<1>, grid, block, 0, s, logits, T, E, k, ids, w);
  if (nc <= 2) return launch_pdl(router_topk_kernel<2>, grid, block, 0, s, logits, T, E, k, ids, w);
  if (nc <= 4) return launch_pdl(router_topk_kernel<4>, grid, block, 0, s, logits, T, E, k, ids, w);
  if (nc <= 8) return launch_pdl(router_topk_kernel<8>, grid, block, 0, s, logits, T, E, k, ids, w);
  if (nc <= 16)
    return launch_pdl(router_topk_kernel<16>, grid, block, 0, s, logits, T, E, k, ids, w);
  return launch_pdl(router_topk_kernel<32>, grid, block, 0, s, logits, T, E, k, ids, w);
}

template <int PER, bool SHARED, int NB>
cudaError_t launch_route_per(const int32_t* ids, int N, int k, int K, int E, int G, int C,
                             int32_t* counts, int32_t* offsets, int32_t* tile_off,
                             int32_t* sorted_src, int32_t* dest_pos, int32_t* hist, int* status,
                             cudaStream_t s) {
  const size_t sm_hist = static_cast<size_t>(kRouteWarps) * G * sizeof(int);
  const size_t sm_scat = static_cast<size_t>(scatter_smem_ints(G, kRouteThreads * PER)) * 4;
  cudaError_t e = cudaFuncSetAttribute(route_scatter_kernel<PER, SHARED, NB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sm_scat));
  if (e != cudaSuccess) return e;
  const int vec = (reinterpret_cast<uintptr_t>(ids) & 15u) == 0 ? 1 : 0;
  e = launch_pdl(route_hist_kernel<PER, SHARED>, dim3(C), dim3(kRouteThreads), sm_hist, s, ids,
                 N, k, K, E, G, C, vec, hist, status);
  const int fused = C <= kFusedScanCtas ? 1 : 0;
  if (e == cudaSuccess && !fused)
    e = launch_pdl(route_scan_kernel, dim3(G), dim3(1024), 0, s, hist, C, counts);
  if (e == cudaSuccess)
    e = launch_pdl(route_scatter_kernel<PER, SHARED, NB>, dim3(C), dim3(kRouteThreads), sm_scat,
                   s, ids, N, k, K, E, G, C, static_cast<const int32_t*>(hist), counts, fused,
                   offsets, tile_off, sorted_src, dest_pos);
  return e;
}

template <int PER, bool SHARED>
cudaError_t launch_route_nb(const int32_t* ids, int N, int k, int K, int E, int G, int C,
                            int32_t* counts, int32_t* offsets, int32_t* tile_off,
                            int32_t* sorted_src, int32_t* dest_pos, int32_t* hist, int* status,
                            cudaStream_t s) {
  switch (match_bits(G)) {
    case 6:
      return launch_route_per<PER, SHARED, 6>(ids, N, k, K, E, G, C, counts, offsets, tile_off,
                                              sorted_src, dest_pos, hist, status, s);
    case 7:
      return launch_route_per<PER, SHARED, 7>(ids, N, k, K, E, G, C, counts, offsets, tile_off,
                                              sorted_src, dest_pos, hist, status, s);
    case 8:
      return launch_route_per<PER, SHARED, 8>(ids, N, k, K, E, G, C, counts, offsets, tile_off,
                                              sorted_src, dest_pos, hist, status, s);
    default:
      return launch_route_per<PER, SHARED, 11>(ids, N, k, K, E, G, C, counts, offsets,
                                               tile_off, sorted_src, dest_pos, hist, status, s);
  }
}

cudaError_t launch_route(const int32_t* ids, int T, int k, int E, int shared, int32_t* counts,
                         int32_t* offsets, int32_t* tile_off, int32_t* sorted_src,
                         int32_t* dest_pos, int32_t* hist, int* status, cudaStream_t s) {
  const int K = k + shared, G = E + shared;
  const int N = T * K;
  const int C = route_ctas(N > 0 ? N : 1);
#define MOE_ROUTE_CASE(P)                                                                  \
  case P:                                                                                  \
    return shared ? launch_route_nb<P, true>(ids, N, k, K, E, G, C, counts, offsets,     \
                                              tile_off, sorted_src, dest_pos, hist, status, s) \
                  : launch_route_nb<P, false>(ids, N, k, K, E, G, C, counts, offsets,    \
                                               tile_off, sorted_src, dest_pos, hist, status, s);
  switch (route_per_lane(N)) {
    MOE_ROUTE_CASE(16)
    MOE_ROUTE_CASE(8)
    default:
      return shared ? launch_route_nb<4, true>(ids, N, k, K, E, G, C, counts, offsets, tile_off,
                                                sorted_src, dest_pos, hist, status, s)
                    : launch_route_nb<4, false>(ids, N, k, K, E, G, C, counts, offsets,
                                                 tile_off, sorted_src, dest_pos, hist, status, s);
  }
#undef MOE_ROUTE_CASE
}

}  // namespace moe

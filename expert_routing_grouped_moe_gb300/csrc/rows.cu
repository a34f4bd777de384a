// Row permute (gather into the expert-grouped, tile-padded layout) and
// combine (gather-reduce back to token order).  Both are pure HBM streams:
// one warp moves a row as 16-byte vectors.
//
// Permute is step 5 of the routing pass in the Unsloth x NVIDIA article,
// section "Optimisation 3" (slice the token list by offsets).  Combine is the
// top-k mixture Y[t] = sum_j w[t,j] * out(t,j), summed in fp32 in slot order
// with no atomics, so results are deterministic.
#include <algorithm>
#include <cstdint>

#include "internal.h"

namespace moe {
namespace {


// Group owning permuted tile mt: the largest g with tile_off[g] <= mt (that
// group is non-empty because mt < tile_off[G]).
__device__ __forceinline__ int group_of_tile(const int32_t* __restrict__ tile_off, int G, int mt) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(tile_off + mid) <= mt) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// One CTA per 128-row tile of the permuted layout; 8 warps x 16 rows.
__global__ void __launch_bounds__(256) permute_kernel(
    const uint4* __restrict__ src, int d8, int K, int G, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ tile_off, const int32_t* __restrict__ sorted_src,
    uint4* __restrict__ dst) {
  __shared__ int s_first, s_cnt, s_off;
  const int mt = blockIdx.x;
  if (threadIdx.x == 0) {
    if (mt >= __ldg(tile_off + G)) {
      s_cnt = -1;
    } else {
      const int g = group_of_tile(tile_off, G, mt);
      s_first = (mt - __ldg(tile_off + g)) * kTileM;
      s_off = __ldg(offsets + g);
      s_cnt = __ldg(offsets + g + 1) - s_off;
    }
  }
  __syncthreads();
  if (s_cnt < 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // each lane moves 8 vectors of a row per step (a 4 KB row of d = 2048 in one
  // step): all loads issued before the stores
  for (int r = warp * 16; r < warp * 16 + 16; ++r) {
    const int q = s_first + r;
    const int64_t p = static_cast<int64_t>(mt) * kTileM + r;
    uint4* drow = dst + p * d8;
    const uint4* srow = nullptr;
    if (q < s_cnt) srow = src + static_cast<int64_t>(__ldg(sorted_src + s_off + q) / K) * d8;
    for (int v0 = 0; v0 < d8; v0 += 256) {
      uint4 x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int v = v0 + i * 32 + lane;
        x[i] = (srow != nullptr && v < d8) ? __ldg(srow + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int v = v0 + i * 32 + lane;
        if (v < d8) drow[v] = x[i];
      }
    }
  }
}

__device__ __forceinline__ void acc_bf16x8(float (&a)[8], const uint4& x, float c) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] = fmaf(c, __uint_as_float(w[i] << 16), a[2 * i]);
    a[2 * i + 1] = fmaf(c, __uint_as_float(w[i] & 0xFFFF0000u), a[2 * i + 1]);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

constexpr int kMaxSlots = 33;

// One warp per token, 8 tokens per CTA.
__global__ void __launch_bounds__(256) combine_kernel(
    const uint4* __restrict__ rows, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ dest_pos, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ tile_off, int T, int d8, int k, int E, int shared,
    const float* __restrict__ weights, const float* __restrict__ row_scalars,
    float* __restrict__ slot_out, uint4* __restrict__ out) {
  __shared__ int64_t s_row[8][kMaxSlots];
  __shared__ float s_c[8][kMaxSlots];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const int K = k + shared;
  for (int j = lane; j < K; j += 32) {
    const int g = j < k ? __ldg(ids + static_cast<int64_t>(t) * k + j) : E;
    const int dp = __ldg(dest_pos + static_cast<int64_t>(t) * K + j);
    int64_t prow = -1;
    float c = 0.f;
    if (dp >= 0 && g >= 0 && g <= E) {
      prow = static_cast<int64_t>(__ldg(tile_off + g)) * kTileM + dp - __ldg(offsets + g);
      c = (weights != nullptr && j < k) ? __ldg(weights + static_cast<int64_t>(t) * k + j) : 1.f;
    }
    s_row[warp][j] = prow;
    s_c[warp][j] = c;
    if (slot_out != nullptr && row_scalars != nullptr && j < k)
      slot_out[static_cast<int64_t>(t) * k + j] = prow >= 0 ? __ldg(row_scalars + prow) : 0.f;
  }
  __syncwarp();
  uint4* orow = out + static_cast<int64_t>(t) * d8;
  // slot rows in groups of 8: all 8 loads of a group in flight at once
  for (int v = lane; v < d8; v += 32) {
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < K; j0 += 8) {
      uint4 x[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = j0 + jj;
        const int64_t pr = j < K ? s_row[warp][j] : -1;
        x[jj] = pr >= 0 ? __ldg(rows + pr * d8 + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (j0 + jj < K) acc_bf16x8(a, x[jj], s_c[warp][j0 + jj]);
    }
    orow[v] = make_uint4(pack2(a[0], a[1]), pack2(a[2], a[3]), pack2(a[4], a[5]),
                         pack2(a[6], a[7]));
  }
}

__global__ void sum_parts_kernel(const float* __restrict__ parts, int nparts, int64_t stride,
                                 int64_t n, float* __restrict__ out) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float s = 0.f;
    for (int q = 0; q < nparts; ++q) s += parts[q * stride + i];
    out[i] = s;
  }
}

}  // namespace

cudaError_t launch_permute(const uint16_t* src, int T, int d, int K, int G,
                           const int32_t* offsets, const int32_t* tile_off,
                           const int32_t* sorted_src, uint16_t* dst, int64_t max_rows,
                           cudaStream_t s) {
  (void)T;
  const int tiles = static_cast<int>(max_rows / kTileM);
  if (tiles == 0) return cudaSuccess;
  permute_kernel<<<tiles, 256, 0, s>>>(reinterpret_cast<const uint4*>(src), d / 8, K, G, offsets,
                                       tile_off, sorted_src, reinterpret_cast<uint4*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* rows, const int32_t* ids, const int32_t* dest_pos,
                           const int32_t* offsets, const int32_t* tile_off, int T, int d, int k,
                           int E, int shared, const float* weights, const float* row_scalars,
                           float* slot_out, uint16_t* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  combine_kernel<<<(T + 7) / 8, 256, 0, s>>>(
      reinterpret_cast<const uint4*>(rows), ids, dest_pos, offsets, tile_off, T, d / 8, k, E,
      shared, weights, row_scalars, slot_out, reinterpret_cast<uint4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_sum_parts(const float* parts, int nparts, int64_t stride, int64_t n,
                             float* out, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096));
  sum_parts_kernel<<<blocks, 256, 0, s>>>(parts, nparts, stride, n, out);
  return cudaGetLastError();
}

}  // namespace moe

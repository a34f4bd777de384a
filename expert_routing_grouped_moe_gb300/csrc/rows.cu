// Row permute (gather into expert-grouped sorted order) and combine
// (gather-reduce back to token order).  Both are pure HBM streams moving rows
// as 16-byte vectors, many loads in flight per lane before any store.
//
// Permute is step 5 of the routing pass in the Unsloth x NVIDIA article,
// section "Optimisation 3" (slice the token list by offsets): permuted row p
// is the token of sorted position p, so expert g's rows are the contiguous
// slice [offsets[g], offsets[g+1]); it is done as a scatter of each token's
// row to the sorted positions of its slots.  Combine is the top-k mixture
// Y[t] = sum_j w[t,j] * out(t,j), summed in fp32 in slot order with no
// atomics, so results are deterministic.
#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// Each warp moves one 512-column block (64 16-byte vectors, two per lane) of
// one token's row to the permuted rows of its K slots,
// dst[dest_pos[t*K + j]] = src[t]: the row is read once, and splitting rows
// into blocks puts all of a lane's loads in flight at once and gives small
// batches enough warps.
constexpr int kBlockVecs = 64;  // 16-byte vectors per warp block (512 bf16)

__global__ void __launch_bounds__(256) permute_kernel(const uint4* __restrict__ src, int T,
                                                     int d8, int K,
                                                     const int32_t* __restrict__ dest_pos,
                                                     uint4* __restrict__ dst) {
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = (d8 + kBlockVecs - 1) / kBlockVecs;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (wid >= static_cast<int64_t>(T) * nb) return;
  const int t = static_cast<int>(wid / nb);
  const int v0 = static_cast<int>(wid - static_cast<int64_t>(t) * nb) * kBlockVecs + lane;
  const uint4* srow = src + static_cast<int64_t>(t) * d8;
  uint4 x[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int v = v0 + i * 32;
    x[i] = v < d8 ? __ldg(srow + v) : make_uint4(0, 0, 0, 0);
  }
  for (int j = 0; j < K; ++j) {
    const int p = __ldg(dest_pos + static_cast<int64_t>(t) * K + j);
    if (p < 0) continue;
    uint4* drow = dst + static_cast<int64_t>(p) * d8;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int v = v0 + i * 32;
      if (v < d8) drow[v] = x[i];
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

// One warp per token, 8 tokens per CTA.  Row of slot j = dest_pos[t*K + j].
// A lane handles CS column slots (16-byte vectors 32 apart) and loads the
// rows of SB slots at a time, summed in fp32 in slot order: for K <= 2 two
// slots x 4 columns at three CTAs per SM, for K <= 4 four slots x 4 columns,
// else 8 slots x 2 columns (two CTAs per SM), so the loads in flight per SM
// do not shrink with K.
template <int SB, int CS, int MINB>
__global__ void __launch_bounds__(256, MINB) combine_kernel(
    const uint4* __restrict__ rows, const int32_t* __restrict__ dest_pos, int T, int d8, int k,
    int shared, const float* __restrict__ weights, const float* __restrict__ row_scalars,
    float* __restrict__ slot_out, uint4* __restrict__ out) {
  __shared__ int s_row[8][kMaxSlots];
  __shared__ float s_c[8][kMaxSlots];
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const int K = k + shared;
  for (int j = lane; j < K; j += 32) {
    const int dp = __ldg(dest_pos + static_cast<int64_t>(t) * K + j);
    const float wj =
        (weights != nullptr && j < k) ? __ldg(weights + static_cast<int64_t>(t) * k + j) : 1.f;
    s_row[warp][j] = dp;
    s_c[warp][j] = dp >= 0 ? wj : 0.f;
    if (slot_out != nullptr && row_scalars != nullptr && j < k)
      slot_out[static_cast<int64_t>(t) * k + j] = dp >= 0 ? __ldg(row_scalars + dp) : 0.f;
  }
  __syncwarp();
  uint4* orow = out + static_cast<int64_t>(t) * d8;
  for (int v0 = lane; v0 < d8; v0 += 32 * CS) {
    float a[CS][8];
#pragma unroll
    for (int i = 0; i < CS; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) a[i][e] = 0.f;
    for (int j0 = 0; j0 < K; j0 += SB) {
      uint4 x[SB][CS];
#pragma unroll
      for (int jj = 0; jj < SB; ++jj) {
        const int j = j0 + jj;
        const int pr = j < K ? s_row[warp][j] : -1;
#pragma unroll
        for (int i = 0; i < CS; ++i) {
          const int v = v0 + i * 32;
          x[jj][i] = (pr >= 0 && v < d8) ? __ldg(rows + static_cast<int64_t>(pr) * d8 + v)
                                         : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int jj = 0; jj < SB; ++jj)
        if (j0 + jj < K) {
#pragma unroll
          for (int i = 0; i < CS; ++i) acc_bf16x8(a[i], x[jj][i], s_c[warp][j0 + jj]);
        }
    }
#pragma unroll
    for (int i = 0; i < CS; ++i) {
      const int v = v0 + i * 32;
      if (v < d8)
        orow[v] = make_uint4(pack2(a[i][0], a[i][1]), pack2(a[i][2], a[i][3]),
                             pack2(a[i][4], a[i][5]), pack2(a[i][6], a[i][7]));
    }
  }
}

__global__ void sum_parts_kernel(const float* __restrict__ parts, int nparts, int64_t stride,
                                 int64_t n, float* __restrict__ out) {
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float s = 0.f;
    for (int q = 0; q < nparts; ++q) s += parts[q * stride + i];
    out[i] = s;
  }
}

}  // namespace

cudaError_t launch_permute(const uint16_t* src, int T, int d, int K, const int32_t* dest_pos,
                           uint16_t* dst, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int64_t warps = static_cast<int64_t>(T) * ((d / 8 + kBlockVecs - 1) / kBlockVecs);
  return launch_pdl(permute_kernel, dim3(static_cast<unsigned>((warps + 7) / 8)), dim3(256), 0, s,
                    reinterpret_cast<const uint4*>(src), T, d / 8, K, dest_pos,
                    reinterpret_cast<uint4*>(dst));
}

cudaError_t launch_combine(const uint16_t* rows, const int32_t* dest_pos, int T, int d, int k,
                           int shared, const float* weights, const float* row_scalars,
                           float* slot_out, uint16_t* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int K = k + shared;
  auto kern = K <= 2   ? combine_kernel<2, 4, 3>
              : K <= 4 ? combine_kernel<4, 4, 2>
                       : combine_kernel<8, 2, 2>;
  return launch_pdl(kern, dim3((T + 7) / 8), dim3(256), 0, s,
                    reinterpret_cast<const uint4*>(rows), dest_pos, T, d / 8, k, shared, weights,
                    row_scalars, slot_out, reinterpret_cast<uint4*>(out));
}

cudaError_t launch_sum_parts(const float* parts, int nparts, int64_t stride, int64_t n,
                             float* out, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096));
  return launch_pdl(sum_parts_kernel, dim3(blocks), dim3(256), 0, s, parts, nparts, stride, n,
                    out);
}

}  // namespace moe

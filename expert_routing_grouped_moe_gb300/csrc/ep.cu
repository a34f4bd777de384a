// Expert-parallel helpers: the two small index kernels that, with moe_route,
// moe_permute and moe_unpermute_combine, move routed rows between the rank
// that owns a token and the rank that owns its expert (experts split into
// contiguous ranges, one all-to-all each way; Unsloth x NVIDIA article,
// closing section on multi-GPU training, and the article's grouped routing).
//
// ep_row_weights    the routing weight of every sorted position, so the
//                   weight can travel with its row to the expert's rank
// ep_segment_ids    the local expert of every received row, from the count
//                   matrix of the rows received from each rank (rank-major,
//                   expert-minor), so moe_route can regroup them by expert
#include <algorithm>
#include <cstdint>

#include "../../include/moe_gb300.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void ep_row_weights_kernel(const float* __restrict__ w, const int32_t* __restrict__ dest,
                                      int T, int k, int K, float* __restrict__ row_w) {
  const int64_t n = static_cast<int64_t>(T) * K;
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int p = __ldg(dest + i);
    if (p < 0) continue;  // an assignment with a bad id has no sorted position
    const int64_t t = i / K;
    const int j = static_cast<int>(i - t * K);
    row_w[p] = j < k ? __ldg(w + t * k + j) : 1.f;
  }
}

// Every CTA scans the count matrix (P x E_loc, rank-major) in shared memory,
// then labels rows by binary search over the block starts.
constexpr int kSegThreads = 256;
__global__ void ep_segment_ids_kernel(const int32_t* __restrict__ counts, int nblk, int E_loc,
                                      int64_t n_rows, int32_t* __restrict__ ids, int* status) {
  extern __shared__ int64_t start[];  // start[b] = first row of block b; start[nblk] = total
  pdl_wait();
  // block-wide exclusive scan in chunks of the block size
  __shared__ int64_t carry;
  __shared__ int64_t wsum[kSegThreads / 32];
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = 0; base < nblk; base += kSegThreads) {
    const int b = base + threadIdx.x;
    const int64_t v = b < nblk ? max(0, __ldg(counts + b)) : 0;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int64_t before = carry;
    for (int w2 = 0; w2 < warp; ++w2) before += wsum[w2];
    if (b < nblk) start[b] = before + x - v;
    __syncthreads();
    if (threadIdx.x == kSegThreads - 1) carry = before + x;
    __syncthreads();
  }
  if (threadIdx.x == 0) start[nblk] = carry;
  __syncthreads();
  if (start[nblk] != n_rows) {
    // the counts do not describe the received rows: label nothing
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicCAS(status, 0, kErrBadIds);
    return;
  }
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n_rows;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int lo = 0, hi = nblk - 1;  // last block with start <= i (empty blocks share starts)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (start[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    ids[i] = lo % E_loc;
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_ep_row_weights(const float* topk_w, const int32_t* dest_pos, int32_t T, int32_t k,
                       int32_t shared_expert, float* row_w, moe_stream_t stream) {
  NvtxScope nvtx("moe_ep_row_weights");
  if (!topk_w || !dest_pos || !row_w) return record_error(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (T <= 0 || k <= 0 || (shared_expert != 0 && shared_expert != 1))
    return record_error(MOE_ERR_INVALID_ARG, "bad T/k/shared_expert");
  if (k > 32) return record_error(MOE_ERR_UNSUPPORTED, "k > 32");
  const int K = k + shared_expert;
  const int64_t n = static_cast<int64_t>(T) * K;
  if (n >= (int64_t(1) << 31)) return record_error(MOE_ERR_UNSUPPORTED, "too many routed rows");
  ProbeScope probe("ep_row_weights", stream);
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096));
  const cudaError_t e = launch_pdl(ep_row_weights_kernel, dim3(blocks), dim3(256), 0, stream,
                                   topk_w, dest_pos, static_cast<int>(T), static_cast<int>(k), K,
                                   row_w);
  if (e != cudaSuccess) return record_error(MOE_ERR_CUDA, cudaGetErrorString(e));
  return record_error(MOE_OK, "");
}

int moe_ep_segment_ids(const int32_t* counts, int32_t P, int32_t E_loc, int64_t n_rows,
                       int32_t* ids, moe_stream_t stream) {
  NvtxScope nvtx("moe_ep_segment_ids");
  if (!counts || (!ids && n_rows > 0)) return record_error(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (P <= 0 || E_loc <= 0 || n_rows < 0)
    return record_error(MOE_ERR_INVALID_ARG, "bad P/E_loc/n_rows");
  const int64_t nblk = static_cast<int64_t>(P) * E_loc;
  if (nblk > kMaxEpBlocks)
    return record_error(MOE_ERR_UNSUPPORTED, "P * E_loc exceeds MOE_EP_MAX_BLOCKS");
  if (n_rows >= (int64_t(1) << 31)) return record_error(MOE_ERR_UNSUPPORTED, "too many rows");
  if (n_rows == 0) return record_error(MOE_OK, "");
  int* status = nullptr;
  const int rc = device_status_word(&status);
  if (rc != MOE_OK) return rc;
  ProbeScope probe("ep_segment_ids", stream);
  const size_t smem = static_cast<size_t>(nblk + 1) * sizeof(int64_t);
  const int blocks = static_cast<int>(std::min<int64_t>((n_rows + kSegThreads - 1) / kSegThreads,
                                                        1024));
  cudaError_t e = cudaSuccess;
  if (smem > 48 * 1024)
    e = cudaFuncSetAttribute(ep_segment_ids_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (e == cudaSuccess)
    e = launch_pdl(ep_segment_ids_kernel, dim3(blocks), dim3(kSegThreads), smem, stream, counts,
                   static_cast<int>(nblk), static_cast<int>(E_loc), n_rows, ids, status);
  if (e != cudaSuccess) return record_error(MOE_ERR_CUDA, cudaGetErrorString(e));
  return record_error(MOE_OK, "");
}

}  // extern "C"

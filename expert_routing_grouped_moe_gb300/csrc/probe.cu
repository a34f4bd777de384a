// Read-stream probe: how fast this GPU streams device memory into shared
// memory with the copy engine the GEMM producers use (bulk asynchronous
// copies completing on mbarriers), with no compute behind it.  The copy peak
// that rooflines are usually quoted against mixes reads and writes; the
// grouped GEMMs mostly read, and this probe measures that ceiling.
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr uint32_t kProbeChunk = 32768;  // bytes per copy
constexpr int kProbeStages = 4;

__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// One CTA per SM: thread 0 issues 32 KB copies of chunks blockIdx.x,
// blockIdx.x + gridDim.x, ... into a 4-stage ring; thread 32 waits for each
// and frees its stage.  Every wait is bounded; a timeout records
// MOE_ERR_TIMEOUT.  The CTA exits only after all of its copies have landed
// (after a timeout, thread 0 waits a bounded time for the stages still armed).
__global__ void __launch_bounds__(64, 1) read_stream_kernel(const uint8_t* __restrict__ src,
                                                            int64_t bytes, int* status) {
  extern __shared__ uint8_t raw[];
  __shared__ uint64_t full[kProbeStages], empty[kProbeStages];
  __shared__ int abort_flag;
  __shared__ unsigned armed, armed_phase;  // stages with a copy not yet consumed, and parity
  const uint32_t ring = (smem_u32(raw) + 127u) & ~127u;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kProbeStages; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);
    }
    abort_flag = 0;
    armed = 0;
    armed_phase = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t nchunks = (bytes + kProbeChunk - 1) / kProbeChunk;
  int stage = 0;
  uint32_t phase = 0;
  if (threadIdx.x == 0) {
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
      if (!mbar_wait(empty + stage, phase ^ 1u, &abort_flag, kWaitTimeoutNs)) break;
      const int64_t off = c * kProbeChunk;
      const uint32_t n =
          static_cast<uint32_t>(bytes - off < kProbeChunk ? bytes - off : kProbeChunk);
      atomicOr(&armed, 1u << stage);
      if (phase) atomicOr(&armed_phase, 1u << stage);
      else atomicAnd(&armed_phase, ~(1u << stage));
      mbar_expect_tx(full + stage, n);
      bulk_load_1d(ring + stage * kProbeChunk, src + off, n, full + stage);
      if (++stage == kProbeStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (threadIdx.x == 32) {
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
      if (!mbar_wait(full + stage, phase, &abort_flag, kWaitTimeoutNs)) break;
      atomicAnd(&armed, ~(1u << stage));
      mbar_arrive(empty + stage);
      if (++stage == kProbeStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && abort_flag) {
    for (int i = 0; i < kProbeStages; ++i)
      if ((armed >> i) & 1u) {
        volatile int never = 0;
        mbar_wait(full + i, (armed_phase >> i) & 1u, &never, 200000000ull);
      }
    atomicCAS(status, 0, kErrTimeout);
  }
}

}  // namespace

cudaError_t launch_read_stream(const void* src, int64_t bytes, int num_sms, int* status,
                               cudaStream_t s) {
  constexpr size_t smem = kProbeStages * kProbeChunk + 128;
  cudaError_t e = cudaFuncSetAttribute(read_stream_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t nchunks = (bytes + kProbeChunk - 1) / kProbeChunk;
  const int grid = static_cast<int>(nchunks < num_sms ? nchunks : num_sms);
  read_stream_kernel<<<grid > 0 ? grid : 1, 64, smem, s>>>(static_cast<const uint8_t*>(src),
                                                           bytes, status);
  return cudaGetLastError();
}

}  // namespace moe

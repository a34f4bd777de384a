// Read-stream probe: how fast this GPU streams device memory into shared
// memory with the copy engines the GEMM producers use (asynchronous copies
// completing on mbarriers), with no compute behind them.  The copy peak that
// rooflines are usually quoted against mixes reads and writes; the grouped
// GEMMs mostly read, and this probe measures that ceiling for two access
// patterns:
//   linear  32 KB bulk copies; neighbouring CTAs read neighbouring chunks
//   tiles   the buffer as a [rows, 2048] bf16 matrix read like a GEMM operand:
//           128B-swizzled TMA boxes of 128 rows x 64 columns, each CTA walking
//           the whole K extent of its own 128-row blocks (two boxes per stage)
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr uint32_t kProbeStage = 32768;          // bytes per stage
constexpr int kProbeStages = 4;
constexpr int64_t kTileBlockBytes = 128 * 4096;  // tiles: one 128-row block
constexpr int kStagesPerBlock = 16;              // tiles: 32 K chunks, two per stage

__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Stage i of this CTA: the linear chunk, or (row block, K pair) of its row
// blocks; -1 past the end.
__device__ __forceinline__ int64_t probe_unit(int64_t i, int64_t nunits, int tiles) {
  const int64_t c =
      tiles ? (blockIdx.x + (i / kStagesPerBlock) * gridDim.x) * kStagesPerBlock +
                  i % kStagesPerBlock
            : blockIdx.x + i * gridDim.x;
  return c < nunits ? c : -1;
}

// One CTA per SM: thread 0 issues the 32 KB stages into a 4-stage ring;
// thread 32 waits for each and frees it.  Every wait is bounded; a timeout
// records MOE_ERR_TIMEOUT.  The CTA exits only after all of its copies have
// landed (after a timeout, thread 0 waits a bounded time for the stages still
// armed).
__global__ void __launch_bounds__(64, 1) read_stream_kernel(const __grid_constant__ CUtensorMap map,
                                                            const uint8_t* __restrict__ src,
                                                            int64_t bytes, int tiles,
                                                            int* status) {
  extern __shared__ uint8_t raw[];
  __shared__ uint64_t full[kProbeStages], empty[kProbeStages];
  __shared__ int abort_flag;
  __shared__ unsigned armed, armed_phase;  // stages with a copy not yet consumed, and parity
  uint8_t* ring = raw + ((1024 - (smem_u32(raw) & 1023)) & 1023);  // 128B-swizzle atoms
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
  const int64_t nunits = tiles ? (bytes / kTileBlockBytes) * kStagesPerBlock
                               : (bytes + kProbeStage - 1) / kProbeStage;
  int stage = 0;
  uint32_t phase = 0;
  if (threadIdx.x == 0) {
    for (int64_t i = 0;; ++i) {
      const int64_t c = probe_unit(i, nunits, tiles);
      if (c < 0) break;
      if (!mbar_wait(empty + stage, phase ^ 1u, &abort_flag, kWaitTimeoutNs)) break;
      atomicOr(&armed, 1u << stage);
      if (phase) atomicOr(&armed_phase, 1u << stage);
      else atomicAnd(&armed_phase, ~(1u << stage));
      uint8_t* dst = ring + stage * kProbeStage;
      if (tiles) {
        const int j = static_cast<int>(c % kStagesPerBlock);
        const int row = static_cast<int>(c / kStagesPerBlock) * 128;
        mbar_expect_tx(full + stage, kProbeStage);
        tma_load_2d(dst, &map, full + stage, 2 * j * 64, row);
        tma_load_2d(dst + kProbeStage / 2, &map, full + stage, (2 * j + 1) * 64, row);
      } else {
        const int64_t off = c * kProbeStage;
        const uint32_t n =
            static_cast<uint32_t>(bytes - off < kProbeStage ? bytes - off : kProbeStage);
        mbar_expect_tx(full + stage, n);
        bulk_load_1d(smem_u32(dst), src + off, n, full + stage);
      }
      if (++stage == kProbeStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (threadIdx.x == 32) {
    for (int64_t i = 0;; ++i) {
      if (probe_unit(i, nunits, tiles) < 0) break;
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

cudaError_t launch_read_stream(const void* src, int64_t bytes, const CUtensorMap* tiles_map,
                               int num_sms, int* status, cudaStream_t s) {
  constexpr size_t smem = kProbeStages * kProbeStage + 1024;
  cudaError_t e = cudaFuncSetAttribute(read_stream_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int tiles = tiles_map != nullptr ? 1 : 0;
  const int64_t units =
      tiles ? bytes / kTileBlockBytes : (bytes + kProbeStage - 1) / kProbeStage;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  CUtensorMap map = {};
  if (tiles) map = *tiles_map;
  read_stream_kernel<<<grid > 0 ? grid : 1, 64, smem, s>>>(
      map, static_cast<const uint8_t*>(src), bytes, tiles, status);
  return cudaGetLastError();
}

}  // namespace moe

// moe_route_noalloc: the routing pass with its scratch in library-owned device
// memory, for callers that cannot allocate device memory themselves.
//
// moe_route needs a per-(expert, CTA) histogram as scratch.  Most callers pass
// a workspace they allocated.  Some hosts give a library only raw pointers and
// a stream and own every byte of device memory through their own pool (plugin
// interfaces whose enqueue step must not allocate, serving runtimes that
// forbid allocation after start-up).  For them the histogram lives here, in a
// fixed-size array that every GPU loading this library holds until exit.
#include <mutex>

#include "../../include/moe_gb300.h"
#include "internal.h"

namespace moe {
namespace {

// Scratch for the routing histogram: moe_route_workspace_size() bytes, G groups
// times one int32 per routing CTA.  2 MiB covers, e.g., up to 256 experts with
// 8,388,608 routed rows (1M tokens x top-8).
constexpr size_t kNoAllocHistInts = size_t(1) << 19;
static __device__ __align__(256) int32_t g_route_scratch[kNoAllocHistInts];

constexpr int kMaxDev = 64;
int32_t* g_scratch_ptr[kMaxDev] = {nullptr};
std::mutex g_scratch_mu;

int set_msg(int code, const char* msg) { return record_error(code, msg); }

}  // namespace

// Host-side address of the scratch array on the current device, looked up
// once per device (the host symbol itself is not a device address).
static int scratch_on_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
    return set_msg(MOE_ERR_CUDA, "moe_route_noalloc: no usable current device");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_msg(MOE_ERR_CUDA, "moe_route_noalloc: cudaGetSymbolAddress failed");
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_route_noalloc(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t shared_expert,
                      int32_t* counts, int32_t* offsets, int32_t* tile_off, int32_t* sorted_src,
                      int32_t* dest_pos, moe_stream_t stream) {
  NvtxScope nvtx("moe_route_noalloc");
  if (!ids || !counts || !offsets || !tile_off || !sorted_src || !dest_pos)
    return set_msg(MOE_ERR_INVALID_ARG, "moe_route_noalloc: NULL pointer");
  if (T <= 0 || k <= 0 || E <= 0 || (shared_expert != 0 && shared_expert != 1) || k > E)
    return set_msg(MOE_ERR_INVALID_ARG, "moe_route_noalloc: bad T/k/E/shared_expert");
  if (E > kMaxExperts || k > 32)
    return set_msg(MOE_ERR_UNSUPPORTED, "moe_route_noalloc: E > 1024 or k > 32");
  const int64_t K = k + shared_expert, G = E + shared_expert;
  const int64_t N = static_cast<int64_t>(T) * K;
  // the same shape limit as moe_route: both accept exactly the same shapes
  if (!routed_rows_fit(T, K, G))
    return set_msg(MOE_ERR_UNSUPPORTED, "moe_route_noalloc: too many routed rows");
  const size_t need = route_ws_bytes(N, static_cast<int>(G));
  if (need > kNoAllocHistInts * sizeof(int32_t))
    return set_msg(MOE_ERR_WORKSPACE,
                   "moe_route_noalloc: routing scratch exceeds the built-in 2 MiB; "
                   "use moe_route with a caller-owned workspace");
  int32_t* scratch = nullptr;
  int rc = scratch_on_current_device(&scratch);
  if (rc != MOE_OK) return rc;
  int* status = nullptr;
  rc = device_status_word(&status);
  if (rc != MOE_OK) return set_msg(rc, "moe_route_noalloc: status word lookup failed");
  // The histogram kernel writes every scratch entry the scan reads, so the
  // previous call's contents need no clearing.  Traced by the timing probe
  // under the name "route", like moe_route.
  ProbeScope probe("route", stream);
  const cudaError_t e = launch_route(ids, T, k, E, shared_expert, counts, offsets, tile_off,
                                     sorted_src, dest_pos, scratch, status, stream);
  if (e != cudaSuccess) return set_msg(MOE_ERR_CUDA, cudaGetErrorString(e));
  return record_error(MOE_OK, "");
}

}  // extern "C"

// C ABI of the MoE-LoRA expert layer: argument checks, tensor-map encoding and
// kernel launches.  No call here allocates device memory or synchronises,
// except moe_status().  See include/moe_gb300.h for the contract of each call.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/moe_gb300.h"
#include "internal.h"

namespace moe {

// Per-device status word: kernels record data errors (bad expert ids) and
// pipeline timeouts here; moe_status() reads and clears it.
static __device__ int g_status_word;

namespace {

thread_local std::string t_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}
int ok() {
  t_err.clear();
  return MOE_OK;
}
int cuda_fail(cudaError_t e, const char* where) {
  return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

struct DevState {
  bool init = false;
  int* status = nullptr;
  int num_sms = 0;
  // second stream for the backward's weight-gradient GEMMs (created on first use)
  std::mutex aux_mu;
  cudaStream_t aux = nullptr;
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
};
constexpr int kMaxDevices = 64;
DevState g_dev[kMaxDevices];
std::mutex g_mu;

// Status-word address and SM count of the current device (looked up once).
int device_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& st = g_dev[dev];
  if (!st.init) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    st.status = static_cast<int*>(ptr);
    st.num_sms = sms;
    st.init = true;
  }
  *out = &st;
  return MOE_OK;
}

// ---- timing probe (tracing): caller-owned CUDA events around kernel launches
const char* const kKernelNames[] = {
    "route", "permute", "combine", "router_topk", "xa_gu", "gate_up", "xa_dn", "down",
    "u", "dgrad_dn", "v", "dgrad_gu", "dB_dn", "dA_dn", "dB_gu", "dA_gu", "dw_reduce",
    "dW_dn", "dW_gu", "ep_row_weights", "ep_segment_ids"};
constexpr int kNumKernels = sizeof(kKernelNames) / sizeof(kKernelNames[0]);

struct Probe {
  std::vector<void*> start, stop;
  int used = 0;
};
Probe g_probe[kNumKernels];
std::mutex g_probe_mu;
std::atomic<int> g_probe_armed{0};

int kernel_index(const char* name) {
  if (name == nullptr) return -1;
  for (int i = 0; i < kNumKernels; ++i)
    if (std::strcmp(kKernelNames[i], name) == 0) return i;
  return -1;
}

// The device's second stream and its fork/join events, created once.  Callers
// hold st->aux_mu while enqueueing work that uses them.
int aux_stream(DevState* st, cudaStream_t* out) {
  if (st->aux == nullptr) {
    cudaError_t e = cudaStreamCreateWithFlags(&st->aux, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithFlags");
    for (cudaEvent_t& ev : st->ev) {
      e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreateWithFlags");
    }
  }
  *out = st->aux;
  return MOE_OK;
}

// `waiter` waits for the work enqueued on `from` so far.
int stream_dep(cudaEvent_t ev, cudaStream_t from, cudaStream_t waiter) {
  cudaError_t e = cudaEventRecord(ev, from);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(waiter, ev, 0);
  if (e != cudaSuccess) return cuda_fail(e, "stream dependency");
  return MOE_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The same for the 256-row tiles of CTA pairs.
int64_t max_pair_tiles(int64_t T, int64_t K, int64_t G) {
  return (T * K + G * (kPairTileM - 1) + kPairTileM - 1) / kPairTileM;
}

// Which of the large row-tile GEMMs run on CTA pairs (256-row tiles, tcgen05
// cta_group::2, each CTA staging half of the B tile) instead of single CTAs
// (128-row tiles).  A pair halves the B bytes each SM stages per MMA, but a
// group's rows are padded to a multiple of 256 instead of 128: with ~256
// rows per group about half the groups carry one idle 128-row half.  So
// gate_up (whose B tile is the largest share of its staging) always pairs,
// the others when groups average at least 512 rows.  MOE_PAIR_TILES in the
// environment overrides this: "0" (none), "1" (all), or a comma-separated
// list of gate_up, down, dgrad_dn, dgrad_gu.
enum PairKernel { kPairGateUp = 1, kPairDown = 2, kPairDgradDn = 4, kPairDgradGu = 8 };
int pair_override() {
  static const int mask = [] {
    const char* v = std::getenv("MOE_PAIR_TILES");
    if (v == nullptr || *v == 0) return -1;
    if (std::strcmp(v, "0") == 0) return 0;
    if (std::strcmp(v, "1") == 0) return 15;
    int m = 0;
    if (std::strstr(v, "gate_up")) m |= kPairGateUp;
    if (std::strstr(v, "down")) m |= kPairDown;
    if (std::strstr(v, "dgrad_dn")) m |= kPairDgradDn;
    if (std::strstr(v, "dgrad_gu")) m |= kPairDgradGu;
    return m;
  }();
  return mask;
}
bool pair_tiles(const moe_dims* dm, PairKernel which, bool a_rows_by_tma) {
  const int G = dm->E + dm->shared_expert;
  if (!a_rows_by_tma || G + 1 > kTileTabInts) return false;
  const int forced = pair_override();
  if (forced >= 0) return (forced & which) != 0;
  if (which == kPairGateUp) return true;
  const int64_t rows = static_cast<int64_t>(dm->T) * (dm->k + dm->shared_expert);
  return rows >= 512 * static_cast<int64_t>(G);
}

int check_dims(const moe_dims* dm) {
  if (dm == nullptr) return fail(MOE_ERR_INVALID_ARG, "dims is NULL");
  if (dm->T <= 0 || dm->d <= 0 || dm->f <= 0 || dm->E <= 0 || dm->k <= 0 || dm->r <= 0)
    return fail(MOE_ERR_INVALID_ARG, "T, d, f, E, k, r must be positive");
  if (dm->shared_expert != 0 && dm->shared_expert != 1)
    return fail(MOE_ERR_INVALID_ARG, "shared_expert must be 0 or 1");
  if (dm->k > dm->E) return fail(MOE_ERR_INVALID_ARG, "k=%d > E=%d", dm->k, dm->E);
  if (dm->E > kMaxExperts) return fail(MOE_ERR_UNSUPPORTED, "E=%d > %d", dm->E, kMaxExperts);
  if (dm->k > 32) return fail(MOE_ERR_UNSUPPORTED, "k=%d > 32", dm->k);
  if (dm->d % 8 || dm->f % 8 || dm->r % 8)
    return fail(MOE_ERR_INVALID_ARG, "d, f and r must be multiples of 8");
  if (dm->r > 64) return fail(MOE_ERR_UNSUPPORTED, "LoRA rank r=%d > 64", dm->r);
  const int64_t K = dm->k + dm->shared_expert, G = dm->E + dm->shared_expert;
  if (!routed_rows_fit(dm->T, K, G)) return fail(MOE_ERR_UNSUPPORTED, "too many routed rows");
  return MOE_OK;
}

#define MOE_CHECK_PTR(p)                                                          \
  do {                                                                            \
    if ((p) == nullptr) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", #p);       \
    if (!aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s not 16-byte aligned", #p); \
  } while (0)

}  // namespace

// Records the start event of the next free probe slot of `name`; returns the
// slot (or -1 when the kernel is not being probed).
int probe_begin(const char* name, cudaStream_t s) {
  if (g_probe_armed.load(std::memory_order_relaxed) == 0) return -1;
  const int id = kernel_index(name);
  if (id < 0) return -1;
  std::lock_guard<std::mutex> lk(g_probe_mu);
  Probe& pr = g_probe[id];
  if (pr.used >= static_cast<int>(pr.start.size())) return -1;
  const int slot = pr.used++;
  cudaEventRecord(static_cast<cudaEvent_t>(pr.start[slot]), s);
  return id * (1 << 24) + slot;
}
void probe_end(int token, cudaStream_t s) {
  if (token < 0) return;
  std::lock_guard<std::mutex> lk(g_probe_mu);
  const Probe& pr = g_probe[token >> 24];
  cudaEventRecord(static_cast<cudaEvent_t>(pr.stop[token & ((1 << 24) - 1)]), s);
}
int device_status_word(int** out) {
  DevState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != MOE_OK) return rc;
  *out = st->status;
  return MOE_OK;
}

int record_error(int code, const char* msg) {
  t_err = msg != nullptr ? msg : "";
  return code;
}

bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows, uint32_t box_cols, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_3d(CUtensorMap* m, const void* base, uint64_t G, uint64_t rows, uint64_t cols,
                 uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {cols, rows, G};
  const cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_mn4d(CUtensorMap* m, const void* base, uint64_t G, uint64_t rows, uint64_t cols,
                   uint32_t box_rows, uint32_t chunks) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || cols % 64 != 0) return false;
  const cuuint64_t dims[4] = {64, rows, cols / 64, G};
  const cuuint64_t strides[3] = {cols * 2, 128, rows * cols * 2};
  const cuuint32_t box[4] = {64, box_rows, chunks, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_split4d(CUtensorMap* m, const void* base, uint64_t G, uint64_t half,
                      uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {cols, half, 2, G};
  const cuuint64_t strides[3] = {cols * 2, half * cols * 2, 2 * half * cols * 2};
  const cuuint32_t box[4] = {box_cols, box_rows, 2, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

struct BwdWs {
  uint16_t *us, *vs, *dh;  // hi/lo pair buffers
  float* dwp;
  // LoRA weight gradients with groups split into parts of wg_rows rows (0: no
  // split): the parts' partial sums and the arrival counters
  int wg_rows;
  float* wg_part;
  int* wg_cnt;
  size_t wg_cnt_bytes;
  size_t bytes;
};

size_t align_up(size_t x) { return (x + 1023) & ~size_t(1023); }

// Rows per part in the LoRA weight-gradient GEMMs, whose tiles otherwise sum
// over all of a group's rows.  A shared expert sees every token, K times the
// mean routed group (and a skewed router adds more large groups); their tiles
// would be many times longer than the rest and run last on a few SMs.  So
// with a shared expert the groups are summed in parts of at least 1.25 times
// the mean group size and 1024 rows (evenly loaded groups stay whole), the
// parts added in order.  0 (no split): no shared expert, or the part table
// does not fit in shared memory.  (Without a shared expert the split kernel
// measured a few us slower on balanced routing, where nothing splits.)
int wgrad_rows_per_part(int64_t N, int64_t G, bool shared) {
  if (!shared || G < 1 || G + 1 > kTileTabInts) return 0;
  int64_t rows = std::max<int64_t>(1024, (5 * N + 4 * G - 1) / (4 * G));
  rows = std::min<int64_t>((rows + 63) / 64 * 64, int64_t(1) << 30);
  return static_cast<int>(rows);
}

BwdWs bwd_layout(const moe_dims* dm, void* base) {
  const int64_t K = dm->k + dm->shared_expert, G = dm->E + dm->shared_expert;
  const size_t P = static_cast<size_t>(dm->T) * static_cast<size_t>(K);  // routed rows N
  const size_t nr = align_up(2 * P * dm->r * 2);
  const size_t ndh = align_up(2 * P * 2 * static_cast<size_t>(dm->f) * 2);
  const size_t nparts = static_cast<size_t>(kDwPartsPerTile) * ((dm->f + kDgradBN - 1) / kDgradBN);
  const size_t ndw = align_up(nparts * P * 4);
  BwdWs w{};
  uint8_t* b = static_cast<uint8_t*>(base);
  size_t o = 0;
  w.us = reinterpret_cast<uint16_t*>(b + o); o += nr;
  w.vs = reinterpret_cast<uint16_t*>(b + o); o += nr;
  w.dh = reinterpret_cast<uint16_t*>(b + o); o += ndh;
  w.dwp = reinterpret_cast<float*>(b + o); o += ndw;
  w.wg_rows = wgrad_rows_per_part(static_cast<int64_t>(P), G, dm->shared_expert != 0);
  if (w.wg_rows > 0) {
    // parts over all groups <= G + N / wg_rows; M tiles <= max(d, 2f) / 128
    const size_t parts = static_cast<size_t>(G) + (P + w.wg_rows - 1) / w.wg_rows;
    const size_t mt = (static_cast<size_t>(std::max(dm->d, 2 * dm->f)) + 127) / 128;
    w.wg_part = reinterpret_cast<float*>(b + o); o += align_up(parts * mt * 8192 * 4);
    w.wg_cnt_bytes = static_cast<size_t>(G) * mt * 8 * 4;
    w.wg_cnt = reinterpret_cast<int*>(b + o); o += align_up(w.wg_cnt_bytes);
  }
  w.bytes = o;
  return w;
}

GemmParams base_params(const moe_dims* dm, const int32_t* offsets, const int32_t* tile_off,
                       const int32_t* sorted_src, const float* topk_w, int* status) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.G = dm->E + dm->shared_expert;
  p.k = dm->k;
  p.K = dm->k + dm->shared_expert;
  p.scale = dm->lora_scale;
  p.tile_off = tile_off;
  p.offsets = offsets;
  p.sorted_src = sorted_src;
  p.topk_w = topk_w;
  p.status = status;
  p.n_btiles = 1;
  return p;
}

int run_gemm(const GemmShape& sh, GemmParams& p, int64_t row_tiles, int num_sms, cudaStream_t s,
             const char* what) {
  if (!sh.wgrad) p.max_tiles = static_cast<int>(row_tiles) * p.n_ntiles;
  ProbeScope probe(what, s);
  cudaError_t e = launch_gemm(sh, p, num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return MOE_OK;
}

#define MAP2(dst, ptr, rows, cols, br, bc)                                         \
  do {                                                                             \
    if (!make_map_2d(&(dst), (ptr), (rows), (cols), (br), (bc)))                   \
      return fail(MOE_ERR_CUDA, "tensor map encode failed (%s)", #ptr);            \
  } while (0)
#define MAP3(dst, ptr, g, rows, cols, br, bc)                                      \
  do {                                                                             \
    if (!make_map_3d(&(dst), (ptr), (g), (rows), (cols), (br), (bc)))              \
      return fail(MOE_ERR_CUDA, "tensor map encode failed (%s)", #ptr);            \
  } while (0)

// Slice i's A operand: the permuted rows `perm` [N, cols] (TMA), or
// (perm == NULL) token rows `tok` [T, cols] gathered by sorted_src (cp.async).
#define SLICE_ROWS(p, i, perm, tok, cols, bexpr, kext)                                 \
  do {                                                                               \
    if ((perm) != nullptr) {                                                         \
      MAP2((p).sl[i].a, (perm), N, (cols), 128, 64);                                 \
    } else {                                                                         \
      (p).sl[i].gather = 1;                                                          \
      (p).sl[i].gsrc = (tok);                                                        \
      (p).sl[i].gld = (cols);                                                        \
      (p).sl[i].gcols = (cols);                                                      \
      (p).gather_any = 1;                                                            \
    }                                                                                \
    bexpr;                                                                           \
    (p).sl[i].K = (kext);                                                            \
  } while (0)

#define SLICE(p, i, amap_ptr, amap_rows, amap_cols, bexpr, kext)                  \
  do {                                                                           \
    MAP2((p).sl[i].a, (amap_ptr), (amap_rows), (amap_cols), 128, 64);            \
    bexpr;                                                                       \
    (p).sl[i].K = (kext);                                                        \
  } while (0)

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return 1; }

int moe_probe_arm(const char* kernel, void* const* start_events, void* const* stop_events,
                  int32_t n) {
  const int id = kernel_index(kernel);
  if (id < 0) return fail(MOE_ERR_INVALID_ARG, "unknown kernel name");
  if (n < 0 || (n > 0 && (start_events == nullptr || stop_events == nullptr)))
    return fail(MOE_ERR_INVALID_ARG, "bad event arrays");
  std::lock_guard<std::mutex> lk(g_probe_mu);
  Probe& pr = g_probe[id];
  const bool was = !pr.start.empty();
  pr.start.assign(start_events, start_events + n);
  pr.stop.assign(stop_events, stop_events + n);
  pr.used = 0;
  const bool now = n > 0;
  if (now && !was) g_probe_armed.fetch_add(1);
  if (!now && was) g_probe_armed.fetch_sub(1);
  return ok();
}

int32_t moe_probe_count(const char* kernel) {
  const int id = kernel_index(kernel);
  if (id < 0) return -1;
  std::lock_guard<std::mutex> lk(g_probe_mu);
  return g_probe[id].used;
}

const char* moe_kernel_name(int32_t i) {
  return (i >= 0 && i < kNumKernels) ? kKernelNames[i] : nullptr;
}

const char* moe_last_error(void) { return t_err.c_str(); }

size_t moe_route_workspace_size(int32_t T, int32_t K, int32_t G) {
  if (T <= 0 || K <= 0 || G <= 0) return 0;
  return route_ws_bytes(static_cast<int64_t>(T) * K, G);
}

int32_t moe_route_kernel_count(int32_t T, int32_t K, int32_t G) {
  if (T <= 0 || K <= 0 || G <= 0) return fail(MOE_ERR_INVALID_ARG, "bad T/K/G");
  ok();
  return route_kernel_count(static_cast<int64_t>(T) * K, G);
}

int moe_status(moe_stream_t stream) {
  DevState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, st->status, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(st->status, 0, sizeof(int), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "moe_status");
  if (v != 0) return fail(v, "device status %d", v);
  return ok();
}

int moe_selftest_wait_timeout(uint32_t timeout_us, moe_stream_t stream) {
  if (timeout_us == 0 || timeout_us > 2000000u)
    return fail(MOE_ERR_INVALID_ARG, "timeout_us must be in (0, 2000000]");
  DevState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  const cudaError_t e =
      launch_wait_selftest(st->status, static_cast<uint64_t>(timeout_us) * 1000u, stream);
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test launch");
  return ok();
}

int moe_probe_read_stream(const void* src, size_t bytes, int32_t pattern, moe_stream_t stream) {
  if (src == nullptr || !aligned16(src)) return fail(MOE_ERR_INVALID_ARG, "src NULL or misaligned");
  if (pattern != MOE_PROBE_LINEAR && pattern != MOE_PROBE_TILES)
    return fail(MOE_ERR_INVALID_ARG, "pattern must be MOE_PROBE_LINEAR or MOE_PROBE_TILES");
  const size_t unit = pattern == MOE_PROBE_TILES ? size_t(128) * 4096 : 16;
  if (bytes == 0 || bytes % unit != 0 || bytes > (size_t(1) << 40))
    return fail(MOE_ERR_INVALID_ARG, "bytes must be a positive multiple of %zu", unit);
  DevState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  CUtensorMap map;
  if (pattern == MOE_PROBE_TILES && !make_map_2d(&map, src, bytes / 4096, 2048, 128, 64))
    return fail(MOE_ERR_CUDA, "tensor map encode failed (probe)");
  const cudaError_t e =
      launch_read_stream(src, static_cast<int64_t>(bytes),
                         pattern == MOE_PROBE_TILES ? &map : nullptr, st->num_sms, st->status,
                         stream);
  if (e != cudaSuccess) return cuda_fail(e, "read-stream probe launch");
  return ok();
}

int moe_router_topk(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* ids,
                    float* weights, moe_stream_t stream) {
  NvtxScope nvtx("moe_router_topk");
  if (logits == nullptr || ids == nullptr || weights == nullptr)
    return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (T <= 0 || E <= 0 || k <= 0 || k > E) return fail(MOE_ERR_INVALID_ARG, "bad T/E/k");
  if (E > kMaxExperts || k > 32) return fail(MOE_ERR_UNSUPPORTED, "E > 1024 or k > 32");
  ProbeScope probe("router_topk", stream);
  cudaError_t e = launch_router_topk(logits, T, E, k, ids, weights, stream);
  if (e != cudaSuccess) return cuda_fail(e, "router_topk launch");
  return ok();
}

namespace {
// Host checks of moe_route's arguments (before anything is launched).
int check_route_args(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t shared_expert,
                     const int32_t* counts, const int32_t* offsets, const int32_t* tile_off,
                     const int32_t* sorted_src, const int32_t* dest_pos, const void* ws,
                     size_t ws_bytes) {
  if (!ids || !counts || !offsets || !tile_off || !sorted_src || !dest_pos || !ws)
    return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (T <= 0 || k <= 0 || E <= 0 || (shared_expert != 0 && shared_expert != 1))
    return fail(MOE_ERR_INVALID_ARG, "bad T/k/E/shared_expert");
  if (k > E) return fail(MOE_ERR_INVALID_ARG, "k=%d > E=%d", k, E);
  if (E > kMaxExperts || k > 32) return fail(MOE_ERR_UNSUPPORTED, "E > 1024 or k > 32");
  const int64_t K = k + shared_expert, G = E + shared_expert;
  if (!routed_rows_fit(T, K, G)) return fail(MOE_ERR_UNSUPPORTED, "too many routed rows");
  if (!aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "ws not 16-byte aligned");
  if (ws_bytes < moe_route_workspace_size(T, static_cast<int32_t>(K), static_cast<int32_t>(G)))
    return fail(MOE_ERR_WORKSPACE, "route workspace too small");
  return MOE_OK;
}
}  // namespace

int moe_route_logits(const float* logits, int32_t T, int32_t E, int32_t k,
                     int32_t shared_expert, int32_t* ids, float* weights, int32_t* counts,
                     int32_t* offsets, int32_t* tile_off, int32_t* sorted_src, int32_t* dest_pos,
                     void* ws, size_t ws_bytes, moe_stream_t stream) {
  NvtxScope nvtx("moe_route_logits");
  if (logits == nullptr || weights == nullptr) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  int rc = check_route_args(ids, T, k, E, shared_expert, counts, offsets, tile_off, sorted_src,
                            dest_pos, ws, ws_bytes);
  if (rc) return rc;
  if ((rc = moe_router_topk(logits, T, E, k, ids, weights, stream))) return rc;
  return moe_route(ids, T, k, E, shared_expert, counts, offsets, tile_off, sorted_src, dest_pos,
                   ws, ws_bytes, stream);
}

int moe_route(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t shared_expert,
              int32_t* counts, int32_t* offsets, int32_t* tile_off, int32_t* sorted_src,
              int32_t* dest_pos, void* ws, size_t ws_bytes, moe_stream_t stream) {
  NvtxScope nvtx("moe_route");
  int rc0 = check_route_args(ids, T, k, E, shared_expert, counts, offsets, tile_off, sorted_src,
                             dest_pos, ws, ws_bytes);
  if (rc0) return rc0;
  DevState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  ProbeScope probe("route", stream);
  cudaError_t e = launch_route(ids, T, k, E, shared_expert, counts, offsets, tile_off,
                               sorted_src, dest_pos, static_cast<int32_t*>(ws), st->status,
                               stream);
  if (e != cudaSuccess) return cuda_fail(e, "route launch");
  return ok();
}

int moe_permute(const moe_bf16* src, int32_t T, int32_t d, int32_t K, const int32_t* dest_pos,
                moe_bf16* dst, moe_stream_t stream) {
  NvtxScope nvtx("moe_permute");
  MOE_CHECK_PTR(src);
  MOE_CHECK_PTR(dst);
  if (!dest_pos) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (T <= 0 || d <= 0 || K <= 0) return fail(MOE_ERR_INVALID_ARG, "bad sizes");
  if (d % 8) return fail(MOE_ERR_INVALID_ARG, "d must be a multiple of 8");
  if (K > 33) return fail(MOE_ERR_UNSUPPORTED, "more than 33 slots per token");
  if (static_cast<int64_t>(T) * K >= (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "too many routed rows");
  ProbeScope probe("permute", stream);
  cudaError_t e = launch_permute(src, T, d, K, dest_pos, dst, stream);
  if (e != cudaSuccess) return cuda_fail(e, "permute launch");
  return ok();
}

int moe_unpermute_combine(const moe_bf16* rows, const int32_t* dest_pos, int32_t T, int32_t d,
                          int32_t k, int32_t shared_expert, const float* weights,
                          const float* row_scalars, float* slot_out, moe_bf16* out,
                          moe_stream_t stream) {
  NvtxScope nvtx("moe_unpermute_combine");
  MOE_CHECK_PTR(rows);
  MOE_CHECK_PTR(out);
  if (!dest_pos) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (T <= 0 || d <= 0 || k <= 0 || (shared_expert != 0 && shared_expert != 1))
    return fail(MOE_ERR_INVALID_ARG, "bad sizes");
  if (d % 8) return fail(MOE_ERR_INVALID_ARG, "d must be a multiple of 8");
  if (k > 32) return fail(MOE_ERR_UNSUPPORTED, "k > 32");
  if ((row_scalars == nullptr) != (slot_out == nullptr))
    return fail(MOE_ERR_INVALID_ARG, "row_scalars and slot_out go together");
  ProbeScope probe("combine", stream);
  cudaError_t e = launch_combine(rows, dest_pos, T, d, k, shared_expert, weights, row_scalars,
                                 slot_out, out, stream);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return ok();
}

int moe_lora_grouped_mlp_fwd(const moe_dims* dims, const moe_bf16* Xp, const moe_bf16* X,
                             const int32_t* counts,
                             const int32_t* offsets, const int32_t* tile_off,
                             const int32_t* sorted_src, const float* topk_w,
                             const moe_bf16* W_gu, const moe_bf16* A_gu, const moe_bf16* B_gu,
                             const moe_bf16* W_dn, const moe_bf16* A_dn, const moe_bf16* B_dn,
                             moe_bf16* Yp, float* h, moe_bf16* act, moe_bf16* xa_gu,
                             moe_bf16* xa_dn, moe_stream_t stream) {
  NvtxScope nvtx("moe_lora_grouped_mlp_fwd");
  (void)counts;
  int rc = check_dims(dims);
  if (rc) return rc;
  if (Xp == nullptr && X == nullptr)
    return fail(MOE_ERR_INVALID_ARG, "pass Xp (permuted rows), X (token rows) or both");
  if (Xp) MOE_CHECK_PTR(Xp);
  if (X) MOE_CHECK_PTR(X);
  MOE_CHECK_PTR(W_gu); MOE_CHECK_PTR(A_gu); MOE_CHECK_PTR(B_gu);
  MOE_CHECK_PTR(W_dn); MOE_CHECK_PTR(A_dn); MOE_CHECK_PTR(B_dn);
  MOE_CHECK_PTR(Yp); MOE_CHECK_PTR(h); MOE_CHECK_PTR(act); MOE_CHECK_PTR(xa_gu);
  MOE_CHECK_PTR(xa_dn);
  if (!offsets || !tile_off || !sorted_src || !topk_w)
    return fail(MOE_ERR_INVALID_ARG, "NULL routing pointer");
  DevState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  const int d = dims->d, f = dims->f, r = dims->r;
  const int G = dims->E + dims->shared_expert;
  const int64_t N = static_cast<int64_t>(dims->T) * (dims->k + dims->shared_expert);
  const int64_t R = max_row_tiles(dims->T, dims->k + dims->shared_expert, G);
  const int64_t RG = (N + 127) / 128;  // tiles of the plain 128-row grid (rank-r products)
  const GemmParams base = base_params(dims, offsets, tile_off, sorted_src, topk_w, st->status);
  cudaStream_t s = stream;

  const int64_t Nf = N * f, Nr = N * r;
  {  // xa_gu pair = s * Xp A_gu^T
    GemmParams p = base;
    // token rows gathered from X when given (L2-resident), else the permuted rows
    SLICE_ROWS(p, 0, X ? nullptr : Xp, X, d, MAP3(p.sl[0].b, A_gu, G, r, d, 64, 64), d);
    p.nslices = 1; p.N = r; p.n_ntiles = (r + 63) / 64; p.out0 = xa_gu; p.ld0 = r; p.pair = Nr;
    if ((rc = run_gemm({128, false, false, Epi::kLoRAGrid}, p, RG, st->num_sms, s, "xa_gu")))
      return rc;
  }
  const bool pair_x = pair_tiles(dims, kPairGateUp, Xp != nullptr);
  const bool pair_rows = pair_tiles(dims, kPairDown, true);
  const int64_t R2 = max_pair_tiles(dims->T, dims->k + dims->shared_expert, G);
  {  // h = Xp W_gu^T + (s xa) B_gu^T (fp32) ; act pair = w * silu(gate) * up
    // (B boxes of 128 rows: one gate or up half; a CTA pair stages one each)
    GemmParams p = base;
    SLICE_ROWS(p, 0, Xp, X, d, MAP3(p.sl[0].b, W_gu, G, 2 * f, d, 128, 64), d);
    SLICE(p, 1, xa_gu, N, r, MAP3(p.sl[1].b, B_gu, G, 2 * f, r, 128, 64), r);
    SLICE(p, 2, xa_gu + Nr, N, r, MAP3(p.sl[2].b, B_gu, G, 2 * f, r, 128, 64), r);
    p.nslices = 3; p.N = f; p.n_ntiles = (f + 127) / 128; p.b_split = f;
    p.fout = h; p.ldf = 32 * ((f + 15) / 16); p.ld0 = 2 * f; p.out0 = act; p.pair = Nf;
    if (!pair_x) {  // one 4-D box per K block for both halves (the 3-D maps stay as fallback)
      GemmSlice q[3] = {p.sl[0], p.sl[1], p.sl[2]};
      if (make_map_split4d(&q[0].b, W_gu, G, f, d, 128, 64) &&
          make_map_split4d(&q[1].b, B_gu, G, f, r, 128, 64) &&
          make_map_split4d(&q[2].b, B_gu, G, f, r, 128, 64)) {
        for (int i = 0; i < 3; ++i) p.sl[i] = q[i];
        p.b4d = 1;
      }
    }
    if ((rc = run_gemm({256, false, false, Epi::kSwiGLU, pair_x}, p, pair_x ? R2 : R, st->num_sms,
                       s, "gate_up")))
      return rc;
  }
  {  // xa_dn pair = s * act A_dn^T   (act = hi + lo, already scaled by w)
    GemmParams p = base;
    SLICE(p, 0, act, N, f, MAP3(p.sl[0].b, A_dn, G, r, f, 64, 64), f);
    SLICE(p, 1, act + Nf, N, f, MAP3(p.sl[1].b, A_dn, G, r, f, 64, 64), f);
    p.nslices = 2; p.N = r; p.n_ntiles = (r + 63) / 64; p.out0 = xa_dn; p.ld0 = r; p.pair = Nr;
    if ((rc = run_gemm({128, false, false, Epi::kLoRAGrid}, p, RG, st->num_sms, s, "xa_dn")))
      return rc;
  }
  {  // Yp = act W_dn^T + xa_dn B_dn^T = w * (o)   (act and xa_dn carry w)
    GemmParams p = base;
    const uint32_t bb = pair_rows ? 128 : 256;  // B box rows: a pair stages half each
    SLICE(p, 0, act, N, f, MAP3(p.sl[0].b, W_dn, G, d, f, bb, 64), f);
    SLICE(p, 1, xa_dn, N, r, MAP3(p.sl[1].b, B_dn, G, d, r, bb, 64), r);
    p.nslices = 2; p.N = d; p.n_ntiles = (d + 255) / 256; p.out0 = Yp; p.ld0 = d;
    if ((rc = run_gemm({256, false, false, Epi::kStore, pair_rows}, p, pair_rows ? R2 : R,
                       st->num_sms, s, "down")))
      return rc;
  }
  return ok();
}

size_t moe_mlp_bwd_workspace_size(const moe_dims* dims) {
  if (check_dims(dims)) return 0;
  return bwd_layout(dims, nullptr).bytes;
}

int moe_lora_grouped_mlp_bwd(const moe_dims* dims, const moe_bf16* dYp, const moe_bf16* dY,
                             const moe_bf16* Xp, const moe_bf16* X,
                             const int32_t* counts, const int32_t* offsets,
                             const int32_t* tile_off, const int32_t* sorted_src,
                             const float* topk_w, const moe_bf16* W_gu, const moe_bf16* A_gu,
                             const moe_bf16* B_gu, const moe_bf16* W_dn, const moe_bf16* A_dn,
                             const moe_bf16* B_dn, const float* h, const moe_bf16* act,
                             const moe_bf16* xa_gu, const moe_bf16* xa_dn, moe_bf16* dXp,
                             float* dw_rows, float* dA_gu, float* dB_gu, float* dA_dn,
                             float* dB_dn, float* dW_gu, float* dW_dn, void* ws,
                             size_t ws_bytes, moe_stream_t stream) {
  NvtxScope nvtx("moe_lora_grouped_mlp_bwd");
  (void)counts;
  int rc = check_dims(dims);
  if (rc) return rc;
  if (dYp == nullptr && dY == nullptr)
    return fail(MOE_ERR_INVALID_ARG, "pass dYp (permuted rows), dY (token rows) or both");
  if (Xp == nullptr && X == nullptr)
    return fail(MOE_ERR_INVALID_ARG, "pass Xp (permuted rows), X (token rows) or both");
  if (dYp) MOE_CHECK_PTR(dYp);
  if (dY) MOE_CHECK_PTR(dY);
  if (Xp) MOE_CHECK_PTR(Xp);
  if (X) MOE_CHECK_PTR(X);
  MOE_CHECK_PTR(W_gu); MOE_CHECK_PTR(A_gu); MOE_CHECK_PTR(B_gu);
  MOE_CHECK_PTR(W_dn); MOE_CHECK_PTR(A_dn); MOE_CHECK_PTR(B_dn);
  MOE_CHECK_PTR(h); MOE_CHECK_PTR(act); MOE_CHECK_PTR(xa_gu); MOE_CHECK_PTR(xa_dn);
  MOE_CHECK_PTR(dXp); MOE_CHECK_PTR(dw_rows);
  MOE_CHECK_PTR(dA_gu); MOE_CHECK_PTR(dB_gu); MOE_CHECK_PTR(dA_dn); MOE_CHECK_PTR(dB_dn);
  MOE_CHECK_PTR(ws);
  if (dW_gu) MOE_CHECK_PTR(dW_gu);
  if (dW_dn) MOE_CHECK_PTR(dW_dn);
  if ((dW_gu || dW_dn) && (Xp == nullptr || dYp == nullptr))
    return fail(MOE_ERR_UNSUPPORTED, "full weight gradients need the permuted rows Xp and dYp");
  if (!offsets || !tile_off || !sorted_src || !topk_w)
    return fail(MOE_ERR_INVALID_ARG, "NULL routing pointer");
  const BwdWs w = bwd_layout(dims, ws);
  if (ws_bytes < w.bytes) return fail(MOE_ERR_WORKSPACE, "bwd workspace too small");
  DevState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  const int d = dims->d, f = dims->f, r = dims->r;
  const int G = dims->E + dims->shared_expert;
  const int64_t N = static_cast<int64_t>(dims->T) * (dims->k + dims->shared_expert);
  const int64_t R = max_row_tiles(dims->T, dims->k + dims->shared_expert, G);
  const int64_t RG = (N + 127) / 128;  // tiles of the plain 128-row grid (rank-r products)
  const GemmParams base = base_params(dims, offsets, tile_off, sorted_src, topk_w, st->status);
  cudaStream_t s = stream;
  const bool pair_dy = pair_tiles(dims, kPairDgradDn, dYp != nullptr);
  const bool pair_rows = pair_tiles(dims, kPairDgradGu, true);
  const int64_t R2 = max_pair_tiles(dims->T, dims->k + dims->shared_expert, G);
  // down-projection dgrad: 256-feature tiles on CTA pairs, else 192
  const int bn_dd = pair_dy ? 256 : kDgradBN;
  const int ntiles_f = (f + bn_dd - 1) / bn_dd;
  const int nparts = kDwPartsPerTile * ntiles_f;

  const int64_t Nr = N * r, N2f = N * 2 * f;
  // per-group LoRA gradients: sum over the group's rows of A^T [B_hi | B_lo],
  // A from one exact bf16 source or a hi/lo pair.  They run on the device's
  // second stream, each as soon as its inputs exist, beside the dgrad chain.
  struct WgradJob {
    const moe_bf16* a;
    const moe_bf16* a_tok;  // token rows to gather when a == NULL
    int a_pair;  // 1: a is a hi/lo pair buffer
    int M;
    const uint16_t* b;  // hi/lo pair buffer [2, N, r]
    float* out;
    int transpose;
    const char* name;
  };
  const WgradJob jobs[4] = {
      {dYp, dY, 0, d, xa_dn, dB_dn, 0, "dB_dn"},
      {act, nullptr, 1, f, w.us, dA_dn, 1, "dA_dn"},
      {w.dh, nullptr, 1, 2 * f, xa_gu, dB_gu, 0, "dB_gu"},
      {Xp, X, 0, d, w.vs, dA_gu, 1, "dA_gu"},
  };
  auto wgrad = [&](const WgradJob& j, cudaStream_t ss) -> int {
    GemmParams p = base;
    if (j.a != nullptr) {
      MAP2(p.sl[0].a, j.a, N, j.M, 64, 64);
    } else {
      p.sl[0].gather = 1;
      p.sl[0].gsrc = j.a_tok;
      p.sl[0].gld = j.M;
      p.sl[0].gcols = j.M;
      p.gather_any = 1;
    }
    p.nslices = 1;
    if (j.a_pair) {
      MAP2(p.sl[1].a, j.a + N * static_cast<int64_t>(j.M), N, j.M, 64, 64);
      p.nslices = 2;
    }
    MAP2(p.wb_hi, j.b, N, r, 64, 64);
    MAP2(p.wb_lo, j.b + Nr, N, r, 64, 64);
    p.M = j.M; p.N = r; p.n_ntiles = (j.M + 127) / 128;
    p.fout = j.out; p.fstride = static_cast<int64_t>(j.M) * r; p.transpose_out = j.transpose;
    if (w.wg_rows > 0) {
      p.wg_rows = w.wg_rows;
      p.wg_part = w.wg_part;
      p.wg_cnt = w.wg_cnt;
      p.max_tiles = static_cast<int>((G + (N + w.wg_rows - 1) / w.wg_rows) * p.n_ntiles);
    }
    return run_gemm({128, true, true, w.wg_rows > 0 ? Epi::kWgradSplit : Epi::kWgrad}, p, R,
                    st->num_sms, ss, j.name);
  };
  // full fine-tuning: per-group sum over the group's rows of A^T B with A a
  // hi/lo pair [2, N, M] (two K passes) and B one wide bf16 row matrix [N, Nb];
  // out [G, M, Nb] fp32, or [G, Nb, M] when transposed
  auto wgrad_full = [&](const moe_bf16* a_pair, int M, const moe_bf16* bmat, int Nb, float* out,
                        int transpose, const char* name, cudaStream_t ss) -> int {
    GemmParams p = base;
    MAP2(p.sl[0].a, a_pair, N, M, 64, 64);
    MAP2(p.sl[1].a, a_pair + N * static_cast<int64_t>(M), N, M, 64, 64);
    p.nslices = 2;
    MAP2(p.wb_hi, bmat, N, Nb, 64, 64);
    p.wb_lo = p.wb_hi;
    p.M = M; p.N = Nb; p.n_ntiles = (M + 127) / 128; p.n_btiles = (Nb + 255) / 256;
    p.fout = out; p.fstride = static_cast<int64_t>(M) * Nb; p.transpose_out = transpose;
    return run_gemm({256, true, true, Epi::kWgradFull}, p, R, st->num_sms, ss, name);
  };
  std::lock_guard<std::mutex> aux_lock(st->aux_mu);
  cudaStream_t aux = nullptr;
  if ((rc = aux_stream(st, &aux))) return rc;

  {  // u = dYp B_dn -> pair us = s*u
    GemmParams p = base;
    // token rows gathered from dY when given (L2-resident), else the permuted rows
    SLICE_ROWS(p, 0, dY ? nullptr : dYp, dY, d, MAP3(p.sl[0].b, B_dn, G, d, r, 64, 64), d);
    p.nslices = 1; p.N = r; p.n_ntiles = (r + 63) / 64; p.ld0 = r; p.pair = Nr;
    p.out0 = w.us;
    if (w.wg_rows > 0) {  // zero the split weight-gradient counters for the kernels after it
      p.zero = w.wg_cnt;
      p.n_zero = static_cast<int64_t>(w.wg_cnt_bytes / 4);
    }
    if ((rc = run_gemm({128, true, false, Epi::kLoRAGrid}, p, RG, st->num_sms, s, "u"))) return rc;
  }
  if ((rc = stream_dep(st->ev[0], s, aux))) return rc;
  if ((rc = wgrad(jobs[0], aux))) return rc;  // dB_dn
  if ((rc = wgrad(jobs[1], aux))) return rc;  // dA_dn
  // dW_dn[g] = sum_p dO_p^T act_p = sum_p dYp_p^T act'_p (act' carries w): [f, d] -> [d, f]
  if (dW_dn && (rc = wgrad_full(act, f, dYp, d, dW_dn, 1, "dW_dn", aux))) return rc;
  {  // g = dYp W_dn + us A_dn ; SwiGLU backward from fp32 h -> dh pair ; dw partials
    GemmParams p = base;
    SLICE_ROWS(p, 0, dYp, dY, d, MAP3(p.sl[0].b, W_dn, G, d, f, 64, 64), d);
    SLICE(p, 1, w.us, N, r, MAP3(p.sl[1].b, A_dn, G, r, f, 64, 64), r);
    SLICE(p, 2, w.us + Nr, N, r, MAP3(p.sl[2].b, A_dn, G, r, f, 64, 64), r);
    p.nslices = 3; p.N = f; p.n_ntiles = ntiles_f;
    {  // one 4-D box per K block (the 3-D maps stay as fallback); a pair's
       // CTAs stage 128 columns each
      const uint32_t chunks = (pair_dy ? bn_dd / 2 : bn_dd) / 64;
      GemmSlice q[3] = {p.sl[0], p.sl[1], p.sl[2]};
      if (make_map_mn4d(&q[0].b, W_dn, G, d, f, 64, chunks) &&
          make_map_mn4d(&q[1].b, A_dn, G, r, f, 64, chunks) &&
          make_map_mn4d(&q[2].b, A_dn, G, r, f, 64, chunks)) {
        for (int i = 0; i < 3; ++i) p.sl[i] = q[i];
        p.b4d = 1;
      }
    }
    p.fin = h; p.ldf = 32 * ((f + 15) / 16);
    p.out0 = w.dh; p.ld0 = 2 * f; p.pair = N2f; p.fout = w.dwp; p.fstride = N;
    // dh planes as TMA store targets: 16 features x 32 rows per store
    p.om_ok = make_map_2d(&p.om_hi, w.dh, N, 2 * f, 32, 16, false) &&
              make_map_2d(&p.om_lo, w.dh + N2f, N, 2 * f, 32, 16, false);
    if ((rc = run_gemm({bn_dd, true, false, Epi::kDgradDn, pair_dy}, p, pair_dy ? R2 : R,
                       st->num_sms, s, "dgrad_dn")))
      return rc;
  }
  if ((rc = stream_dep(st->ev[1], s, aux))) return rc;
  {
    ProbeScope probe("dw_reduce", aux);
    const cudaError_t e = launch_sum_parts(w.dwp, nparts, N, N, dw_rows, aux);
    if (e != cudaSuccess) return cuda_fail(e, "dw reduce");
  }
  if ((rc = wgrad(jobs[2], aux))) return rc;  // dB_gu
  // dW_gu[g] = sum_p dh_p^T Xp_p: [2f, d]
  if (dW_gu && (rc = wgrad_full(w.dh, 2 * f, Xp, d, dW_gu, 0, "dW_gu", aux))) return rc;
  {  // v = dh B_gu (dh = hi + lo) -> vs pair = s*v
    GemmParams p = base;
    SLICE(p, 0, w.dh, N, 2 * f, MAP3(p.sl[0].b, B_gu, G, 2 * f, r, 64, 64), 2 * f);
    SLICE(p, 1, w.dh + N2f, N, 2 * f, MAP3(p.sl[1].b, B_gu, G, 2 * f, r, 64, 64), 2 * f);
    p.nslices = 2; p.N = r; p.n_ntiles = (r + 63) / 64; p.ld0 = r; p.pair = Nr; p.out0 = w.vs;
    if ((rc = run_gemm({128, true, false, Epi::kLoRAGrid}, p, RG, st->num_sms, s, "v"))) return rc;
  }
  if ((rc = stream_dep(st->ev[2], s, aux))) return rc;
  if ((rc = wgrad(jobs[3], aux))) return rc;  // dA_gu
  {  // dXp = dh W_gu + vs A_gu   (high halves: dX is an output, not a row reduction)
    GemmParams p = base;
    SLICE(p, 0, w.dh, N, 2 * f, MAP3(p.sl[0].b, W_gu, G, 2 * f, d, 64, 64), 2 * f);
    SLICE(p, 1, w.vs, N, r, MAP3(p.sl[1].b, A_gu, G, r, d, 64, 64), r);
    p.nslices = 2; p.N = d; p.n_ntiles = (d + 255) / 256; p.out0 = dXp; p.ld0 = d;
    {  // one 4-D box per K block (the 3-D maps stay as fallback)
      const uint32_t chunks = pair_rows ? 2 : 4;
      GemmSlice q[2] = {p.sl[0], p.sl[1]};
      if (make_map_mn4d(&q[0].b, W_gu, G, 2 * f, d, 64, chunks) &&
          make_map_mn4d(&q[1].b, A_gu, G, r, d, 64, chunks)) {
        for (int i = 0; i < 2; ++i) p.sl[i] = q[i];
        p.b4d = 1;
      }
    }
    if ((rc = run_gemm({256, true, false, Epi::kStore, pair_rows}, p, pair_rows ? R2 : R,
                       st->num_sms, s, "dgrad_gu")))
      return rc;
  }
  // join: everything on the second stream completes before later work on s
  if ((rc = stream_dep(st->ev[3], aux, s))) return rc;
  return ok();
}

}  // extern "C"

// Internal interfaces between the C-ABI layer (api.cu) and the kernel
// translation units.  Host-side only; nothing here is exported.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

namespace moe {

// Launches a kernel with programmatic stream serialization: it may begin
// (and run up to its griddepcontrol.wait) while the previous kernel of the
// stream finishes, which hides launch latency and its own set-up.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}
// The same with the CTAs grouped into clusters of cluster_x (CTA pairs: 2).
template <typename... Params, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t s, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

constexpr int kTileM = 128;            // rows per M tile (= permuted layout granularity)
constexpr int kPairTileM = 256;        // rows per tile of a CTA pair
// Groups whose tile offsets the GEMMs keep in shared memory (G + 1 <=
// kTileTabInts); beyond that the tile scheduler searches tile_off in global
// memory, and the CTA-pair tiles (whose table is built in shared memory) are
// not used.
constexpr int kTileTabInts = 448;
constexpr int kMaxExperts = 1024;      // routed experts supported
constexpr uint64_t kWaitTimeoutNs = 4000000000ull;  // pipeline waits give up after 4 s

// Error codes recorded in the device status word (same values as moe_status_t).
constexpr int kErrBadIds = -5;
constexpr int kErrTimeout = -6;

// Upper bound on the 128-row tiles of all groups: sum_g ceil(counts[g] / 128)
// for N = T * K routed rows in G groups.  Every entry point that produces or
// consumes routing tables accepts a shape only if this many tiles of rows
// stay below 2^31 rows.
inline int64_t max_row_tiles(int64_t T, int64_t K, int64_t G) {
  return (T * K + G * (kTileM - 1) + kTileM - 1) / kTileM;
}
inline bool routed_rows_fit(int64_t T, int64_t K, int64_t G) {
  return max_row_tiles(T, K, G) * kTileM < (int64_t(1) << 31);
}

// ---- timing probe (api.cu) --------------------------------------------------
// When the probe is armed for `name` (moe_probe_arm), records a caller-owned
// CUDA event on the launch stream before and after the launches in scope.
int probe_begin(const char* name, cudaStream_t s);
void probe_end(int token, cudaStream_t s);
// NVTX range (host-side, shown by Nsight tools; a no-op without one) around
// a C-ABI call or a kernel launch.
struct NvtxScope {
  explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
  ~NvtxScope() { nvtxRangePop(); }
  NvtxScope(const NvtxScope&) = delete;
  NvtxScope& operator=(const NvtxScope&) = delete;
};
// Kernel launches in scope are traced under `name`: an NVTX range, and the
// timing probe's events when it is armed for that name.
struct ProbeScope {
  NvtxScope range;
  int token;
  cudaStream_t s;
  ProbeScope(const char* name, cudaStream_t st)
      : range(name), token(probe_begin(name, st)), s(st) {}
  ~ProbeScope() { probe_end(token, s); }
  ProbeScope(const ProbeScope&) = delete;
  ProbeScope& operator=(const ProbeScope&) = delete;
};

// ---- routing (route.cu) ----------------------------------------------------
constexpr int kRouteThreads = 256;                  // 8 warps per CTA
constexpr int kRouteWarps = kRouteThreads / 32;

// Assignments per lane, growing with the problem so that large routing
// problems use fewer, fuller CTAs (each CTA handles 256 * per-lane assignments).
inline int route_per_lane(int64_t n) {
  return n >= (int64_t(1) << 19) ? 16 : n >= (int64_t(1) << 17) ? 8 : 4;
}
inline int route_chunk(int64_t n) { return kRouteThreads * route_per_lane(n); }
inline int route_ctas(int64_t n) {
  return static_cast<int>((n + route_chunk(n) - 1) / route_chunk(n));
}
inline size_t route_ws_bytes(int64_t n, int G) {
  // per-(group, CTA) histogram, int32
  return static_cast<size_t>(G) * static_cast<size_t>(route_ctas(n > 0 ? n : 1)) * 4u;
}

cudaError_t launch_router_topk(const float* logits, int T, int E, int k, int32_t* ids,
                               float* w, cudaStream_t s);
cudaError_t launch_route(const int32_t* ids, int T, int k, int E, int shared, int32_t* counts,
                         int32_t* offsets, int32_t* tile_off, int32_t* sorted_src,
                         int32_t* dest_pos, int32_t* hist, int* status, cudaStream_t s);
// Kernels launch_route issues for n assignments and G groups: 2 when the
// per-CTA histogram is small enough for the scatter kernel to scan it itself,
// else 3 (histogram, scan, scatter).
int route_kernel_count(int64_t n, int G);

// ---- expert-parallel helpers (ep.cu) -------------------------------------------
// Blocks (rank, local expert) of a received-row count matrix: P * E_loc.
constexpr int64_t kMaxEpBlocks = 16384;

// ---- row gather / combine (rows.cu) ------------------------------------------
// Permuted rows are in sorted order: row p holds sorted position p, N = T * K rows.
cudaError_t launch_permute(const uint16_t* src, int T, int d, int K, const int32_t* dest_pos,
                           uint16_t* dst, cudaStream_t s);
cudaError_t launch_combine(const uint16_t* rows, const int32_t* dest_pos, int T, int d, int k,
                           int shared, const float* weights, const float* row_scalars,
                           float* slot_out, uint16_t* out, cudaStream_t s);
cudaError_t launch_sum_parts(const float* parts, int nparts, int64_t stride, int64_t n,
                             float* out, cudaStream_t s);

// ---- grouped GEMMs (gemm.cu) -------------------------------------------------
// Derived intermediates that feed a reduction over rows (the LoRA weight
// gradients, the routing-weight gradient) are carried as a pair of bf16
// values hi + lo (hi = bf16(v), lo = bf16(v - hi)), ~16 significant bits; a
// pair buffer holds hi at [0, P*cols) and lo at [P*cols, 2*P*cols).
enum class Epi : int {
  kSwiGLU = 0,   // h = acc (fp32, gate|up halves), act' = w*silu(gate)*up as a hi/lo pair
  kStore = 2,    // out0 = bf16(acc)
  kDgradDn = 4,  // SwiGLU backward from fp32 h (fin): dh pair (out0), dw partial (fout)
  kWgrad = 5,    // fp32 per-group weight gradient: acc[:, n] + acc[:, 64 + n]
  kWgradFull = 6,  // fp32 per-group full weight gradient: acc (B = one wide matrix)
  kLoRAGrid = 7,   // out0 = s*acc as a hi/lo pair (N <= 64), on the plain 128-row
                   // grid; up to two groups per pass, their B blocks stacked (BN = 128)
  kWgradSplit = 8,  // kWgrad with groups summed in parts of wg_rows rows, the parts'
                    // fp32 sums added in part order by the last to finish
};

constexpr int kMaxSlices = 4;
// The down-projection dgrad writes one routing-weight-gradient partial per
// 256-column tile and column half (two epilogue warps share each row).
constexpr int kDwPartsPerTile = 2;
// N tile (f features) of the down-projection dgrad with the SwiGLU-backward
// epilogue: 192 columns leave room in shared memory for a second staging tile
// per epilogue warp next to a 4-stage ring.
constexpr int kDgradBN = 192;

// One K-slice of a contraction: D += A_slice * B_slice^T over K columns.
struct GemmSlice {
  CUtensorMap a;
  CUtensorMap b;
  int K;
  int gather;                // 1: A rows are token rows gathered by sorted_src[p] / K
  const uint16_t* gsrc;      // gathered A: token-row matrix [T, gcols] bf16
  int64_t gld;               //             its leading dimension (elements)
  int gcols;                 //             its columns (K for rows mode, M for wgrad)
};

struct GemmParams {
  GemmSlice sl[kMaxSlices];  // rows mode: A/B per slice; wgrad: A sources (hi, lo)
  CUtensorMap wb_hi, wb_lo;  // wgrad: B operand hi / lo (columns [0,64) / [64,128))
  CUtensorMap om_hi, om_lo;  // SwiGLU backward: dh hi / lo planes as TMA store targets
  int om_ok;                 //   set when om_hi / om_lo are valid
  int nslices;
  int gather_any;     // some slice gathers its A rows
  int N;              // valid output columns (rows mode) / LoRA rank r (wgrad)
  int M;              // wgrad: rows of the weight gradient (d, f or 2f)
  int n_ntiles;       // N tiles per M tile (rows mode) / M tiles per group (wgrad)
  int n_btiles;       // wgrad: N tiles over the B matrix's columns (1 for the LoRA gradients)
  int b_split;        // rows offset of the second B half (gate/up pairing), 0 = none
  int b4d;            // every slice's B map is 4-D: one box per K block (MN-major
                      // 64-column chunks, or the two gate/up halves)
  int G, k, K;        // groups, top-k, slots per token
  float scale;        // LoRA scale s
  const int32_t* tile_off;
  const int32_t* offsets;
  const int32_t* sorted_src;
  const float* topk_w;
  uint16_t* out0;
  float* fout;        // fp32 output: h (SwiGLU), dw partials (dgrad), weight grad (wgrad)
  const float* fin;   // fp32 input: h (dgrad)
  int64_t ld0;        // leading dimension (elements) of out0 rows
  int64_t ldf;        // leading dimension (floats) of the fp32 h buffer (fout / fin)
  int64_t pair;       // element offset from the hi to the lo half of a pair buffer
  int64_t fstride;    // stride between dw partial slices, or group stride of fout
  int transpose_out;  // wgrad: write fout[g][n][m] instead of fout[g][m][n]
  int wg_rows;        // kWgradSplit: groups split into parts of wg_rows rows (a multiple
                      //   of 64; the part table needs G + 1 <= kTileTabInts)
  float* wg_part;     //   parts' sums: [part][M tile][N tile][8 warps][32 x 32] fp32
  int* wg_cnt;        //   arrivals per [group][M tile][N tile][warp]; zero before the launch
  int* zero;          // grid mode: n_zero words the kernel sets to 0 after its dependency
  int64_t n_zero;     //   wait, for a later launch (the split weight-gradient counters)
  int max_tiles;      // upper bound of tiles (host-known): rows mode, split wgrad
  int nrows;          // rows of the permuted buffers (N = T * K)
  int* status;
};

// Kernel shapes: BN in {128, 192, 256}; B operand K-major or MN-major; two modes.
struct GemmShape {
  int BN;
  bool b_mn;
  bool wgrad;  // wgrad: A and B both MN-major, K = group rows
  Epi epi;
  bool pair = false;  // rows mode on CTA pairs: 256-row tiles, each CTA staging half of B
};

cudaError_t launch_gemm(const GemmShape& shape, const GemmParams& p, int num_sms,
                        cudaStream_t s);
// ---- read-stream probe (probe.cu) ------------------------------------------
// Streams `bytes` from src into shared memory, one CTA per SM, and discards
// them: linear 32 KB bulk copies (tiles_map NULL; src 16-byte aligned, bytes
// a multiple of 16), or GEMM-operand tiles through tiles_map, a 128B-swizzled
// bf16 map of src as [bytes / 4096, 2048] with 128 x 64 boxes (bytes a
// multiple of 128 * 4096).
cudaError_t launch_read_stream(const void* src, int64_t bytes, const CUtensorMap* tiles_map,
                               int num_sms, int* status, cudaStream_t s);

// One thread waits on an mbarrier nothing arrives on, bounded by timeout_ns,
// then records kErrTimeout in *status (the failure path of every pipeline wait).
cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t s);

// ---- shared host state (api.cu) ----------------------------------------------
// Address of the current device's status word (looked up once per device).
int device_status_word(int** out);
// Sets the message moe_last_error() returns on this thread; returns `code`.
int record_error(int code, const char* msg);

// ---- tensor maps (api.cu) ----------------------------------------------------
// 2D bf16 map over [rows, cols] row-major; box (box_cols, box_rows); 128B
// swizzle, or none (dense box rows) with swizzle128 = false.
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows, uint32_t box_cols, bool swizzle128 = true);
// 3D bf16 map over [G, rows, cols]; box (box_cols, box_rows, 1); 128B swizzle.
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t G, uint64_t rows, uint64_t cols,
                 uint32_t box_rows, uint32_t box_cols);
// 4D views of [G, rows, cols] for one TMA box per K block (128B swizzle):
// mn: (64 columns, rows, cols / 64 chunks, G), box (64, box_rows, chunks, 1),
//     landing as `chunks` consecutive [box_rows][64] blocks; cols % 64 == 0.
// split: rows = two halves of `half` rows: (cols, half, 2, G), box
//     (box_cols, box_rows, 2, 1), landing as the two halves' blocks.
bool make_map_mn4d(CUtensorMap* m, const void* base, uint64_t G, uint64_t rows, uint64_t cols,
                   uint32_t box_rows, uint32_t chunks);
bool make_map_split4d(CUtensorMap* m, const void* base, uint64_t G, uint64_t half,
                      uint64_t cols, uint32_t box_rows, uint32_t box_cols);

}  // namespace moe

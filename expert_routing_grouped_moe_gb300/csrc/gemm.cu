// Persistent grouped GEMM on 5th-generation tensor cores (tcgen05, sm_103a).
//
// One kernel template serves every contraction of the split-LoRA SwiGLU expert
// MLP (Unsloth "Faster MoE" docs, sections "Faster LoRA MoE training" and
// "Implementation details": X W next to (X A) B, never forming B A):
//
//   rows mode   D[rows of a 128-row tile, BN cols] = sum over K-slices s of
//               A_s[rows, K_s] * B_s[group]^T ; the tile's group comes from the
//               device-side tile offsets (no host query).  Extra slices carry
//               the low-rank LoRA correction (A = the saved s*X A^T, B = the
//               other adapter matrix) and the low halves of hi/lo operand
//               pairs, all into the same fp32 accumulator.
//   grid mode   the rank-r products (N = r <= 64) on the plain 128-row grid of
//               the permuted rows: a tile whose rows belong to two groups
//               stacks the groups' B blocks into one 128-column B tile, so one
//               MMA per K step serves both (more groups: more passes over the
//               tile); no rows past a group's end are computed.
//   wgrad mode  D[M tile of a weight dimension, BN] = sum over the group's
//               rows of A[rows, M]^T B[rows, BN] -- the per-expert dA / dB
//               reductions (B = [B_hi | B_lo] of a rank-r operand, halves
//               added) and the full weight gradients (B = one wide row matrix
//               in 256-column tiles), one CTA per output tile, deterministic.
//
// Warp roles (320 threads, one CTA per SM, persistent over tiles):
//   warp 0      producer: lane 0 issues the TMA copies of 128B-swizzled A and
//               B tiles into a STAGES-deep shared-memory ring (mbarrier
//               full/empty handshake); all 32 lanes copy gathered token rows
//               with cp.async when the A rows are gathered
//   warp 1      allocates TMEM (2 x BN fp32 columns: double-buffered
//               accumulators); lane 0 issues tcgen05.mma and tcgen05.commit
//   warps 2-9   epilogue, two warps per TMEM lane quadrant (warp w reads lanes
//               32*(w%4)..), each owning half of the tile's columns: tcgen05.ld,
//               fused SwiGLU / SwiGLU backward / LoRA / weight-gradient
//               outputs.  Wide row traffic goes through a per-warp swizzled
//               shared-memory staging tile so that global loads and stores are
//               full 128-byte lines (the SwiGLU backward also stores through
//               TMA from a second tile).  The accumulator is then freed, so the
//               epilogue of one tile overlaps the mainloop of the next.
//
// Every wait is bounded (see mbar_wait): on timeout the CTA raises an abort
// flag, drains its own copies and MMAs in flight, frees TMEM, records
// MOE_ERR_TIMEOUT in the status word and returns.
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // bf16 elements per 128-byte swizzle row
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kAStageBytes = BM * BK * 2;  // 16 KB
constexpr uint32_t kChunkBytes = 64 * 128;      // one [64][64] bf16 swizzle block
constexpr uint32_t kStgTileBytes = 32 * 128;    // one staging tile: 32 rows x 128 B
constexpr uint32_t kRingMax = 192 * 1024;
constexpr uint32_t kSmemMax = 232448;           // opt-in shared memory per CTA
constexpr uint32_t kFixedSmem = 1024 /*alignment slack*/ + 256 /*barriers*/ +
                                kTileTabInts * 4 /*tile_off copy*/;

__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int BN, int EPI, bool PAIR = false, bool B_MN = false>
struct Cfg {
  // a CTA of a pair stages half of B's BN columns
  static constexpr uint32_t kBStageBytes = (PAIR ? BN / 2 : BN) * BK * 2;
  static constexpr uint32_t kStageBytes = kAStageBytes + kBStageBytes;
  static constexpr bool kGrid = EPI == static_cast<int>(Epi::kLoRAGrid);
  // staging per epilogue warp: one tile, two for the SwiGLU backward (h in,
  // dh out through TMA stores), none for the grid-mode LoRA products (whose
  // rows leave straight from registers; the ring takes the room instead)
  static constexpr uint32_t kStgBytes =
      kGrid ? 0u : (EPI == static_cast<int>(Epi::kDgradDn) ? 2 : 1) * kStgTileBytes;
  // grid-mode LoRA products with K-major B (X·Aᵀ) run two CTAs per SM (short
  // kernels of ~1.7 waves at one CTA per SM): half the shared memory and
  // registers each.  With MN-major B (the dH·B products) one CTA with the
  // full 7-stage ring measured faster.
  static constexpr int kCtasPerSm = (kGrid && !B_MN) ? 2 : 1;
  static constexpr uint32_t kSmemBudget = kCtasPerSm == 2 ? (kSmemMax / 2 - 1024) : kSmemMax;
  static constexpr uint32_t kRingFit =
      (kSmemBudget - kFixedSmem - kEpiWarps * kStgBytes) / kStageBytes * kStageBytes;
  static constexpr uint32_t kRingCap = kGrid ? kRingFit : kRingMax;
  // 4 / 4 / 6 stages for BN 256 / 192 (dgrad) / 128 (weight gradients); in grid
  // mode 3 at two CTAs per SM, 7 at one; pairs: 6 stages of 32 KB (5 with the
  // SwiGLU backward's two staging tiles)
  static constexpr int kStages = (kRingFit < kRingCap ? kRingFit : kRingCap) / kStageBytes;
  static constexpr uint32_t kTmemCols = pow2_at_least(2 * BN);  // power of two >= 32
  static constexpr size_t kSmemBytes =
      kFixedSmem + static_cast<size_t>(kStages) * kStageBytes + kEpiWarps * kStgBytes;
};

// Group owning permuted M tile mt: the largest g with tile_off[g] <= mt
// (non-empty because mt < tile_off[G]).  `tab` is the CTA's shared-memory
// copy of tile_off, or nullptr (search global memory).
__device__ __forceinline__ int group_of_tile(const int32_t* __restrict__ tile_off,
                                             const int* tab, int G, int mt) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((tab ? tab[mid] : __ldg(tile_off + mid)) <= mt) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Group owning permuted row `row` (< offsets[G]): the largest g with
// offsets[g] <= row.  `tab` is the CTA's shared-memory copy of offsets, or
// nullptr (search global memory).
__device__ __forceinline__ int group_of_row(const int32_t* __restrict__ offsets, const int* tab,
                                            int G, int row) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((tab ? tab[mid] : __ldg(offsets + mid)) <= row) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Routing weight of permuted row p (a valid sorted position; 1 for the
// shared-expert slot).
__device__ __forceinline__ float row_weight(const GemmParams& p, int64_t row) {
  const int i = __ldg(p.sorted_src + row);
  const int t = i / p.K;
  const int j = i - t * p.K;
  return j < p.k ? __ldg(p.topk_w + static_cast<int64_t>(t) * p.k + j) : 1.f;
}

// hi = bf16(v), lo = bf16(v - hi): the pair holds ~16 significant bits of v.
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    l[i] = pack_bf16x2(v[2 * i] - bf16lo(h[i]), v[2 * i + 1] - bf16hi(h[i]));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}
__device__ __forceinline__ void store8_pair(uint16_t* hi, int64_t pair, const float (&v)[8]) {
  uint4 a, b;
  split8(v, a, b);
  *reinterpret_cast<uint4*>(hi) = a;
  *reinterpret_cast<uint4*>(hi + pair) = b;
}
__device__ __forceinline__ uint4 f4_as_u4(float a, float b, float c, float d) {
  return make_uint4(__float_as_uint(a), __float_as_uint(b), __float_as_uint(c),
                    __float_as_uint(d));
}

// Logistic function with the fast reciprocal (relative error ~2^-22, far
// below the 16 significant bits the saved values keep).
__device__ __forceinline__ float sigmoidf_(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

// ------------------------------------------------------------ staging tile
// A warp's staging tile is 32 rows x 128 bytes (8 chunks of 16 B) with the
// chunk index XOR-swizzled by the row, so both a thread writing its own row
// and a warp reading 4 rows x 8 chunks touch every bank group once.
__device__ __forceinline__ uint32_t stg_at(uint32_t stg, int r, int c) {
  return stg + r * 128 + (((c ^ r) & 7) << 4);
}
__device__ __forceinline__ void sts128(uint32_t a, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// The 8 chunks of a staging row split into `nplanes` planes of `cpp` chunks
// (cpp * nplanes <= 8); plane i of row r lives at base[i] + r * ld (bytes),
// of which the first `valid` bytes exist (the rest of the plane is masked).
struct Planes {
  char* b0;
  char* b1;
  char* b2;
  char* b3;
  int64_t ld;
  int cpp_log2;
  int nplanes;
  int valid;
  int nrows = 32;  // rows of the tile that exist
};
__device__ __forceinline__ char* plane_base(const Planes& pl, int plane) {
  return plane == 0 ? pl.b0 : plane == 1 ? pl.b1 : plane == 2 ? pl.b2 : pl.b3;
}

// Coalesced store of the warp's staging tile: 4 rows x 8 chunks per step.
__device__ __forceinline__ void stg_flush(uint32_t stg, int lane, const Planes& pl) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    const int c = lane & 7;
    const int plane = c >> pl.cpp_log2;
    const int sub = c & ((1 << pl.cpp_log2) - 1);
    const uint4 v = lds128(stg_at(stg, r, c));
    if (plane < pl.nplanes && sub * 16 < pl.valid && r < pl.nrows)
      *reinterpret_cast<uint4*>(plane_base(pl, plane) + r * pl.ld + sub * 16) = v;
  }
}
// Coalesced load into registers (issue), then into the staging tile (commit).
__device__ __forceinline__ void stg_fetch(uint4 (&regs)[8], int lane, const Planes& pl) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    const int c = lane & 7;
    const int plane = c >> pl.cpp_log2;
    const int sub = c & ((1 << pl.cpp_log2) - 1);
    regs[i] = (plane < pl.nplanes && sub * 16 < pl.valid && r < pl.nrows)
                  ? __ldg(reinterpret_cast<const uint4*>(plane_base(pl, plane) + r * pl.ld +
                                                         sub * 16))
                  : make_uint4(0, 0, 0, 0);
  }
}
__device__ __forceinline__ void stg_commit(uint32_t stg, int lane, const uint4 (&regs)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) sts128(stg_at(stg, i * 4 + (lane >> 3), lane & 7), regs[i]);
}

__device__ __forceinline__ int clamp_bytes(int64_t v, int hi) {
  return v <= 0 ? 0 : (v >= hi ? hi : static_cast<int>(v));
}

// Tile coordinates shared by all roles.
struct TileInfo {
  int g;       // expert group
  int mt;      // rows mode: M tile (tile_off numbering); wgrad: M tile of the weight dimension
  int nt;      // rows mode: N tile
  int nk;      // K blocks in total
  int row0;    // first permuted row: of the tile (rows mode) / of the group (wgrad)
  int nvalid;  // rows mode: rows of the group in this tile (<= 128); wgrad: group rows
  int nkb;     // wgrad: 64-row K blocks per slice
  // wgrad with split groups: this tile's part of the group's rows, of nparts
  int part, nparts;
  // grid mode: groups g .. g + nx - 1 of this pass own rows [rlo, rhi) of the
  // tile; rows from rmid on belong to group g + 1 (B block / accumulator slot 1)
  int nx, rlo, rmid, rhi;
};

// Grid mode: tile t covers permuted rows [128 t, 128 t + 128) clipped to the
// valid rows; its rows belong to groups g0 .. g1, taken two per pass.
constexpr int kGridSlots = 2;
struct GridTile {
  int g0, g1, npass;
};
template <bool GRID>
__device__ __forceinline__ GridTile grid_tile(const GemmParams& p, int t, const int* tab) {
  GridTile gt{0, 0, 1};
  if constexpr (GRID) {
    const int nv = tab ? tab[p.G] : __ldg(p.offsets + p.G);
    const int r0 = t * BM, r1 = min(r0 + BM, nv) - 1;
    gt.g0 = group_of_row(p.offsets, tab, p.G, r0);
    gt.g1 = group_of_row(p.offsets, tab, p.G, r1);
    gt.npass = (gt.g1 - gt.g0) / kGridSlots + 1;
  }
  return gt;
}
__device__ __forceinline__ TileInfo grid_info(const GemmParams& p, int t, const GridTile& gt,
                                              int pass, const int* tab) {
  auto off = [&](int g) { return tab ? tab[g] : __ldg(p.offsets + g); };
  TileInfo ti;
  ti.g = gt.g0 + pass * kGridSlots;
  ti.nx = min(kGridSlots, gt.g1 - ti.g + 1);
  ti.mt = t;
  ti.nt = 0;
  ti.nk = 0;
  for (int s = 0; s < p.nslices; ++s) ti.nk += (p.sl[s].K + BK - 1) / BK;
  ti.row0 = t * BM;
  const int nv = off(p.G);
  ti.nvalid = min(BM, nv - ti.row0);
  ti.rlo = max(ti.row0, off(ti.g));
  ti.rmid = off(ti.g + 1);
  ti.rhi = min(ti.row0 + ti.nvalid, off(ti.g + ti.nx));
  ti.nkb = 0;
  return ti;
}

// The sequence of work units every role of a CTA walks: its tiles t =
// first + i * stride (first = blockIdx.x, stride = gridDim.x; for CTA pairs
// the pair's index and the number of pairs) and, in grid mode, each tile's
// passes.
struct Unit {
  int t, ps;
  GridTile gt;
};
template <bool GRID>
__device__ __forceinline__ Unit unit_first(const GemmParams& p, const int* tab, int num_tiles,
                                           int first) {
  Unit u{first, 0, GridTile{0, 0, 1}};
  if (GRID && u.t < num_tiles) u.gt = grid_tile<GRID>(p, u.t, tab);
  return u;
}
template <bool GRID>
__device__ __forceinline__ void unit_next(Unit& u, const GemmParams& p, const int* tab,
                                          int num_tiles, int stride) {
  if (GRID && ++u.ps < u.gt.npass) return;
  u.ps = 0;
  u.t += stride;
  if (GRID && u.t < num_tiles) u.gt = grid_tile<GRID>(p, u.t, tab);
}

// ROWS = false skips the row range (row0, nvalid) of a rows-mode tile, which
// the MMA issuer does not need.
template <bool WGRAD, bool ROWS = true, bool SPLIT = false>
__device__ __forceinline__ TileInfo tile_info(const GemmParams& p, int t, const int* tab) {
  TileInfo ti;
  if (!WGRAD) {
    ti.mt = t / p.n_ntiles;
    ti.nt = t - ti.mt * p.n_ntiles;
    ti.g = group_of_tile(p.tile_off, tab, p.G, ti.mt);
    ti.nk = 0;
    for (int s = 0; s < p.nslices; ++s) ti.nk += (p.sl[s].K + BK - 1) / BK;
    ti.row0 = 0;
    ti.nvalid = 0;
    if (ROWS) {
      // offsets follow tile_off in the table when both fit
      const int* otab = (tab && 2 * (p.G + 1) <= kTileTabInts) ? tab + p.G + 1 : nullptr;
      const int local = ti.mt - (tab ? tab[ti.g] : __ldg(p.tile_off + ti.g));
      const int off = otab ? otab[ti.g] : __ldg(p.offsets + ti.g);
      const int cnt = (otab ? otab[ti.g + 1] : __ldg(p.offsets + ti.g + 1)) - off;
      ti.row0 = off + local * BM;
      ti.nvalid = min(BM, cnt - local * BM);
    }
    ti.nkb = 0;
  } else if constexpr (SPLIT) {
    // groups split into parts of wg_rows rows: tile t = (part index * M tiles
    // + mt) * N tiles + nt, where the group's parts are numbered from tab[g]
    // (tab = parts of the earlier groups, then offsets when both fit)
    const int per_g = p.n_ntiles * p.n_btiles;
    const int pidx = t / per_g;
    const int rem = t - pidx * per_g;
    ti.mt = rem / p.n_btiles;
    ti.nt = rem - ti.mt * p.n_btiles;
    // every group in one part (no group above wg_rows): part index = group
    ti.g = tab[p.G] == p.G ? pidx : group_of_tile(nullptr, tab, p.G, pidx);
    ti.part = pidx - tab[ti.g];
    ti.nparts = tab[ti.g + 1] - tab[ti.g];
    const int* otab = 2 * (p.G + 1) <= kTileTabInts ? tab + p.G + 1 : nullptr;
    const int off = otab ? otab[ti.g] : __ldg(p.offsets + ti.g);
    const int cnt = (otab ? otab[ti.g + 1] : __ldg(p.offsets + ti.g + 1)) - off;
    ti.row0 = off + ti.part * p.wg_rows;
    ti.nvalid = min(p.wg_rows, cnt - ti.part * p.wg_rows);
    ti.nkb = (ti.nvalid + BK - 1) / BK;
    ti.nk = ti.nkb * p.nslices;
  } else {
    // tile t = (group * M tiles + mt) * N tiles + nt; `tab` holds offsets here
    const int per_g = p.n_ntiles * p.n_btiles;
    ti.g = t / per_g;
    const int rem = t - ti.g * per_g;
    ti.mt = rem / p.n_btiles;
    ti.nt = rem - ti.mt * p.n_btiles;
    ti.row0 = tab ? tab[ti.g] : __ldg(p.offsets + ti.g);
    ti.nvalid = (tab ? tab[ti.g + 1] : __ldg(p.offsets + ti.g + 1)) - ti.row0;
    ti.nkb = (ti.nvalid + BK - 1) / BK;
    ti.nk = ti.nkb * p.nslices;
  }
  return ti;
}

// ------------------------------------------------------------ CTA pairs
// A pair of CTAs (a cluster of two) computes 256-row tiles: pair tile i of
// group g covers its rows [256 i, 256 i + 256), the even CTA rows
// [256 i, 256 i + 128) and the odd one the next 128.  tab[g] = the pair tiles
// of all earlier groups (sum of ceil(count / 256)), built in shared memory
// by every CTA at start-up from the group offsets (G + 1 <= kTileTabInts);
// offsets follow at tab + G + 1 when both fit.
constexpr int kPairM = 2 * BM;

// tab[g] = sum over groups g' < g of max(min_units, ceil(count[g'] / unit)),
// g = 0..G, by all threads of the CTA (G + 1 <= 2 * blockDim.x); wsum holds
// one int per warp.  The group offsets are read from `offs` (a shared-memory
// copy, visible to every thread) or, when NULL, from global memory.
__device__ __forceinline__ void group_units_table(const GemmParams& p, int* tab, int* wsum,
                                                  int unit, int min_units,
                                                  const int* offs = nullptr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto tiles = [&](int g) {
    if (g >= p.G) return 0;
    const int c = offs ? offs[g + 1] - offs[g] : __ldg(p.offsets + g + 1) - __ldg(p.offsets + g);
    return max(min_units, (c + unit - 1) / unit);
  };
  // thread i: groups 2i and 2i + 1 (G + 1 <= 2 * blockDim.x)
  const int g0 = 2 * static_cast<int>(threadIdx.x);
  const int v0 = tiles(g0), v1 = tiles(g0 + 1);
  int x = v0 + v1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += wsum[w];
  const int excl = base + x - v0 - v1;
  if (g0 <= p.G) tab[g0] = excl;
  if (g0 + 1 <= p.G) tab[g0 + 1] = excl + v0;
}

template <bool ROWS = true>
__device__ __forceinline__ TileInfo pair_tile_info(const GemmParams& p, int t, const int* tab,
                                                   uint32_t crank) {
  TileInfo ti;
  ti.mt = t / p.n_ntiles;
  ti.nt = t - ti.mt * p.n_ntiles;
  ti.g = group_of_tile(nullptr, tab, p.G, ti.mt);
  ti.nk = 0;
  for (int s = 0; s < p.nslices; ++s) ti.nk += (p.sl[s].K + BK - 1) / BK;
  ti.row0 = 0;
  ti.nvalid = 0;
  if (ROWS) {
    const int* otab = 2 * (p.G + 1) <= kTileTabInts ? tab + p.G + 1 : nullptr;
    const int local = ti.mt - tab[ti.g];
    const int off = otab ? otab[ti.g] : __ldg(p.offsets + ti.g);
    const int cnt = (otab ? otab[ti.g + 1] : __ldg(p.offsets + ti.g + 1)) - off;
    const int first = local * kPairM + static_cast<int>(crank) * BM;
    ti.row0 = off + first;
    ti.nvalid = min(BM, cnt - first);  // <= 0: this CTA's half lies past the group's end
  }
  ti.nkb = 0;
  ti.nx = ti.rlo = ti.rmid = ti.rhi = 0;
  return ti;
}

// ------------------------------------------------------------- epilogues
// Each epilogue warp owns 32 accumulator rows (TMEM quadrant q) and one half
// (hf) of the tile's columns.  `tq` is the TMEM address of its rows' column 0,
// `row0` the permuted row of its first row, `lane` its row within the 32.

template <int BN>
__device__ __forceinline__ void epi_swiglu(const GemmParams& p, const TileInfo& ti, uint32_t tq,
                                           int hf, int64_t row0, int nrows, int lane,
                                           uint32_t stg) {
  // accumulator columns [0, BN/2) = gate, [BN/2, BN) = up of the same features;
  // this warp: features hf*BN/4 + [0, BN/4).  The saved activation is scaled
  // by the row's routing weight: act' = w * silu(gate) * up.
  const int f = p.N;
  const float w = lane < nrows ? row_weight(p, row0 + lane) : 0.f;
#pragma unroll 1
  for (int sub = 0; sub < BN / 4; sub += 16) {
    const int cg = hf * (BN / 4) + sub;
    float g[16], u[16], a[16];
    tmem_ld16(tq + cg, g);
    tmem_ld16(tq + BN / 2 + cg, u);
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = w * (g[i] * sigmoidf_(g[i]) * u[i]);
    const int j0 = ti.nt * (BN / 2) + cg;
    // h (fp32): [gate 16 | up 16]
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      sts128(stg_at(stg, lane, c), f4_as_u4(g[4 * c], g[4 * c + 1], g[4 * c + 2], g[4 * c + 3]));
      sts128(stg_at(stg, lane, 4 + c),
             f4_as_u4(u[4 * c], u[4 * c + 1], u[4 * c + 2], u[4 * c + 3]));
    }
    __syncwarp();
    {
      // h row layout: features in chunks of 16, [gate 16 | up 16] per chunk,
      // so one chunk is one 128-byte line
      float* hb = p.fout + row0 * p.ldf;
      Planes pl{reinterpret_cast<char*>(hb + 2 * j0), nullptr, nullptr, nullptr, p.ldf * 4, 3,
                1, j0 < f ? 128 : 0, nrows};
      stg_flush(stg, lane, pl);
    }
    __syncwarp();
    // act pair (bf16): [hi 16 | lo 16]
    uint4 h0, l0, h1, l1;
    split8(a, h0, l0);
    split8(a + 8, h1, l1);
    sts128(stg_at(stg, lane, 0), h0);
    sts128(stg_at(stg, lane, 1), h1);
    sts128(stg_at(stg, lane, 2), l0);
    sts128(stg_at(stg, lane, 3), l1);
    __syncwarp();
    {
      uint16_t* ab = p.out0 + row0 * static_cast<int64_t>(f) + j0;
      Planes pl{reinterpret_cast<char*>(ab), reinterpret_cast<char*>(ab + p.pair), nullptr,
                nullptr, static_cast<int64_t>(f) * 2, 1, 2,
                clamp_bytes(static_cast<int64_t>(f - j0) * 2, 32), nrows};
      stg_flush(stg, lane, pl);
    }
    __syncwarp();
  }
}

template <int BN>
__device__ __forceinline__ void epi_store(const GemmParams& p, const TileInfo& ti, uint32_t tq,
                                          int hf, int64_t row0, int nrows, int lane,
                                          uint32_t stg) {
#pragma unroll 1
  for (int c0 = hf * (BN / 2); c0 < (hf + 1) * (BN / 2); c0 += 64) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float v[16];
      tmem_ld16(tq + c0 + 16 * q4, v);
      float a[8], b[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a[i] = v[i];
        b[i] = v[8 + i];
      }
      sts128(stg_at(stg, lane, 2 * q4),
             make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                        pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7])));
      sts128(stg_at(stg, lane, 2 * q4 + 1),
             make_uint4(pack_bf16x2(b[0], b[1]), pack_bf16x2(b[2], b[3]),
                        pack_bf16x2(b[4], b[5]), pack_bf16x2(b[6], b[7])));
    }
    __syncwarp();
    const int j0 = ti.nt * BN + c0;
    Planes pl{reinterpret_cast<char*>(p.out0 + row0 * p.ld0 + j0), nullptr, nullptr, nullptr,
              p.ld0 * 2, 3, 1, clamp_bytes(static_cast<int64_t>(p.N - j0) * 2, 128), nrows};
    stg_flush(stg, lane, pl);
    __syncwarp();
  }
}

template <int BN>
__device__ __forceinline__ void epi_dgrad_dn(const GemmParams& p, const TileInfo& ti, uint32_t tq,
                                             int hf, int64_t row0, int nrows, int lane,
                                             uint32_t stg) {
  // acc = g = dY W_dn + s (dY B_dn) A_dn (unscaled by the routing weight);
  // this warp: columns hf*BN/2 + [0, BN/2) in chunks of 16
  const int f = p.N;
  const float w = lane < nrows ? row_weight(p, row0 + lane) : 0.f;
  const float* hb = p.fin + row0 * p.ldf;     // h rows: [gate 16 | up 16] per chunk, fp32
  uint16_t* db = p.out0 + row0 * p.ld0;       // dh pair [rows, 2f]
  constexpr int kSubs = (BN / 2) / 16;
  auto h_planes = [&](int j0) {
    return Planes{reinterpret_cast<char*>(const_cast<float*>(hb + 2 * j0)), nullptr, nullptr,
                  nullptr, p.ldf * 4, 3, 1, j0 < f ? 128 : 0, nrows};
  };
  const int jbase = ti.nt * BN + hf * (BN / 2);
  float dot = 0.f;
  // g of the next chunk is loaded from TMEM while this chunk is computed
  uint32_t tr[16];
  tmem_ld16_issue(tq + hf * (BN / 2), tr);
  // one 16-column chunk: h from the staging tile, g from TMEM, dh pair out
  auto process = [&](int sub) {
    const int j0 = jbase + sub * 16;
    float gt[16], up[16], gr[16];
    tmem_ld_wait16(tr);
#pragma unroll
    for (int i = 0; i < 16; ++i) gr[i] = __uint_as_float(tr[i]);
    if (sub + 1 < kSubs) tmem_ld16_issue(tq + hf * (BN / 2) + (sub + 1) * 16, tr);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 x = lds128(stg_at(stg, lane, c));
      const uint4 y = lds128(stg_at(stg, lane, 4 + c));
      gt[4 * c] = __uint_as_float(x.x); gt[4 * c + 1] = __uint_as_float(x.y);
      gt[4 * c + 2] = __uint_as_float(x.z); gt[4 * c + 3] = __uint_as_float(x.w);
      up[4 * c] = __uint_as_float(y.x); up[4 * c + 1] = __uint_as_float(y.y);
      up[4 * c + 2] = __uint_as_float(y.z); up[4 * c + 3] = __uint_as_float(y.w);
    }
    // Columns past f in a partial last chunk need no mask: this tile's
    // accumulator is exactly 0 there (W_dn and A_dn columns TMA zero-fills) and
    // the h the forward stored there is finite, so they add 0 to dot, and
    // their dh is not stored.
    float dg[16], du[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float sg = sigmoidf_(gt[i]);
      const float sl = gt[i] * sg;  // silu(gate)
      dot = fmaf(sl * up[i], gr[i], dot);
      const float da = w * gr[i];
      // d silu / d gate = sg (1 + gate (1 - sg)) = sg + silu (1 - sg)
      dg[i] = (da * up[i]) * fmaf(sl, 1.f - sg, sg);
      du[i] = da * sl;
    }
    __syncwarp();
    uint4 a0, a1, b0, b1, c0, c1, e0, e1;
    split8(dg, a0, b0);
    split8(dg + 8, a1, b1);
    split8(du, c0, e0);
    split8(du + 8, c1, e1);
    if (p.om_ok && nrows == 32 && j0 + 16 <= f) {
      // whole chunk: the four 32-row x 16-feature planes (dgate hi, dup hi,
      // dgate lo, dup lo) go out as TMA stores from the second staging tile
      const uint32_t ob = stg + kStgTileBytes;
      if (lane == 0) bulk_wait_read_all();  // the previous chunk's stores have read ob
      __syncwarp();
      const uint32_t rb = ob + lane * 32;
      sts128(rb, a0);
      sts128(rb + 16, a1);
      sts128(rb + 1024, c0);
      sts128(rb + 1024 + 16, c1);
      sts128(rb + 2048, b0);
      sts128(rb + 2048 + 16, b1);
      sts128(rb + 3072, e0);
      sts128(rb + 3072 + 16, e1);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int y = static_cast<int>(row0);
        tma_store_2d(&p.om_hi, ob, j0, y);
        tma_store_2d(&p.om_hi, ob + 1024, f + j0, y);
        tma_store_2d(&p.om_lo, ob + 2048, j0, y);
        tma_store_2d(&p.om_lo, ob + 3072, f + j0, y);
        bulk_commit();
      }
      return;
    }
    // rows past the group's end or columns past f: masked stores through the
    // staging tile
    sts128(stg_at(stg, lane, 0), a0);
    sts128(stg_at(stg, lane, 1), a1);
    sts128(stg_at(stg, lane, 2), b0);
    sts128(stg_at(stg, lane, 3), b1);
    sts128(stg_at(stg, lane, 4), c0);
    sts128(stg_at(stg, lane, 5), c1);
    sts128(stg_at(stg, lane, 6), e0);
    sts128(stg_at(stg, lane, 7), e1);
    __syncwarp();
    Planes pl{reinterpret_cast<char*>(db + j0), reinterpret_cast<char*>(db + p.pair + j0),
              reinterpret_cast<char*>(db + f + j0),
              reinterpret_cast<char*>(db + p.pair + f + j0), p.ld0 * 2, 1, 4,
              clamp_bytes(static_cast<int64_t>(f - j0) * 2, 32), nrows};
    stg_flush(stg, lane, pl);
    __syncwarp();
  };
  // h chunks are fetched two ahead (two register buffers in flight)
  uint4 pa[8], pb[8];
  stg_fetch(pa, lane, h_planes(jbase));
  stg_commit(stg, lane, pa);
  __syncwarp();
  if (kSubs > 1) stg_fetch(pa, lane, h_planes(jbase + 16));
  if (kSubs > 2) stg_fetch(pb, lane, h_planes(jbase + 32));
#pragma unroll 1
  for (int sub = 0; sub < kSubs; sub += 2) {
    process(sub);
    if (sub + 1 < kSubs) {
      stg_commit(stg, lane, pa);
      __syncwarp();
      if (sub + 3 < kSubs) stg_fetch(pa, lane, h_planes(jbase + (sub + 3) * 16));
      process(sub + 1);
    }
    if (sub + 2 < kSubs) {
      stg_commit(stg, lane, pb);
      __syncwarp();
      if (sub + 4 < kSubs) stg_fetch(pb, lane, h_planes(jbase + (sub + 4) * 16));
    }
  }
  if (lane < nrows)
    p.fout[static_cast<int64_t>(ti.nt * kDwPartsPerTile + hf) * p.fstride + row0 + lane] = dot;
}

// Grid mode: out0 = s * acc as a hi/lo pair for the rows of this pass; a
// row's accumulator is slot 0 (columns [0,64)) or, from rmid on, slot 1
// (columns [64,128)).  This warp: its 32 rows from rowq, columns hf*32 + [0,32).
__device__ __forceinline__ void epi_lora_grid(const GemmParams& p, const TileInfo& ti,
                                              uint32_t tq, int hf, int64_t rowq, int lane) {
  const int64_t row = rowq + lane;
  const bool valid = row >= ti.rlo && row < ti.rhi;
  const bool second = row >= ti.rmid;
  const bool any0 = __any_sync(0xffffffffu, valid && !second);
  const bool any1 = __any_sync(0xffffffffu, valid && second);
  const float s = p.scale;
#pragma unroll 1
  for (int c0 = hf * 32; c0 < hf * 32 + 32; c0 += 16) {
    float v16[16];
    if (any0) tmem_ld16(tq + c0, v16);
    if (any1) {
      float w16[16];
      tmem_ld16(tq + 64 + c0, w16);
      if (second) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v16[i] = w16[i];
      }
    }
#pragma unroll
    for (int h8 = 0; h8 < 2; ++h8) {
      const int j = c0 + h8 * 8;
      if (valid && j < p.N) {
        float ov[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) ov[i] = s * v16[h8 * 8 + i];
        store8_pair(p.out0 + row * p.ld0 + j, p.pair, ov);
      }
    }
  }
}

template <bool SPLIT>
__device__ __forceinline__ void epi_wgrad(const GemmParams& p, const TileInfo& ti, uint32_t tq,
                                          int hf, int q, int lane, uint32_t stg, const int* tab) {
  // columns [0,64) = A * B_hi, [64,128) = A * B_lo; this warp: n in hf*32 + [0,32)
  const int m0 = ti.mt * BM + q * 32;
  const int m = m0 + lane;
  const bool has = ti.nk > 0;
  float* fo = p.fout + static_cast<int64_t>(ti.g) * p.fstride;
  float v[32];
#pragma unroll
  for (int c0 = 0; c0 < 32; c0 += 16) {
    float vh[16], vl[16];
    if (has) {
      tmem_ld16(tq + hf * 32 + c0, vh);
      tmem_ld16(tq + 64 + hf * 32 + c0, vl);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) vh[i] = vl[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) v[c0 + i] = vh[i] + vl[i];
  }
  if (SPLIT && ti.nparts > 1) {
    // a group split into parts: this warp parks its part's 32 x 32 sums, and
    // the warp that completes the set adds the parts in part order (the same
    // sum whatever order they finish in) and stores the result
    const int wi = hf * 4 + q;
    auto slab = [&](int pidx) {
      return p.wg_part +
             ((static_cast<int64_t>(pidx) * p.n_ntiles + ti.mt) * p.n_btiles + ti.nt) * 8192 +
             wi * 1024;
    };
    const int first = tab[ti.g];  // part index of the group's part 0
    float* mine = slab(first + ti.part);
#pragma unroll
    for (int i = 0; i < 32; ++i) __stcg(mine + i * 32 + lane, v[i]);
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      int* c = p.wg_cnt +
               ((static_cast<int64_t>(ti.g) * p.n_ntiles + ti.mt) * p.n_btiles + ti.nt) * 8 + wi;
      last = atomicAdd(c, 1) == ti.nparts - 1;
      if (last) *c = 0;  // every part has arrived: zero for the next launch
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
    for (int k = 0; k < ti.nparts; ++k) {
      const float* src = slab(first + k);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] += __ldcg(src + i * 32 + lane);
    }
  }
  if (p.transpose_out) {
    // fout[g][n][m]: consecutive lanes write consecutive m (128-byte lines)
    if (m < p.M) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int n = hf * 32 + i;
        if (n < p.N) fo[static_cast<int64_t>(n) * p.M + m] = v[i];
      }
    }
  } else {
    // fout[g][m][n]: stage the warp's 32 rows x 32 columns, store whole lines
#pragma unroll
    for (int c = 0; c < 8; ++c)
      sts128(stg_at(stg, lane, c), f4_as_u4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]));
    __syncwarp();
    Planes pl{reinterpret_cast<char*>(fo + static_cast<int64_t>(m0) * p.N + hf * 32), nullptr,
              nullptr, nullptr, static_cast<int64_t>(p.N) * 4, 3, 1,
              clamp_bytes(static_cast<int64_t>(p.N - hf * 32) * 4, 128), p.M - m0};
    stg_flush(stg, lane, pl);
    __syncwarp();
  }
}

// Full weight gradient: fout[g] (+ m * N + n, or + n * M + m when
// transposed) = acc, this warp's rows m0 + [0,32) and columns
// nt*BN + hf*BN/2 + [0, BN/2).  A group without rows writes zeros.
template <int BN>
__device__ __forceinline__ void epi_wgrad_full(const GemmParams& p, const TileInfo& ti,
                                               uint32_t tq, int hf, int q, int lane,
                                               uint32_t stg) {
  const int m0 = ti.mt * BM + q * 32;
  const int m = m0 + lane;
  const bool has = ti.nk > 0;
  float* fo = p.fout + static_cast<int64_t>(ti.g) * p.fstride;
  const int nbase = ti.nt * BN + hf * (BN / 2);
#pragma unroll 1
  for (int c0 = 0; c0 < BN / 2; c0 += 32) {
    float v[32];
    if (has) {
      tmem_ld16(tq + hf * (BN / 2) + c0, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tq + hf * (BN / 2) + c0 + 16, *reinterpret_cast<float(*)[16]>(v + 16));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.f;
    }
    const int n0 = nbase + c0;
    if (p.transpose_out) {
      // fout[g][n][m]: consecutive lanes write consecutive m (128-byte lines)
      if (m < p.M) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (n0 + i < p.N) fo[static_cast<int64_t>(n0 + i) * p.M + m] = v[i];
      }
    } else {
      // fout[g][m][n]: stage the warp's 32 rows x 32 columns, store whole lines
#pragma unroll
      for (int c = 0; c < 8; ++c)
        sts128(stg_at(stg, lane, c), f4_as_u4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]));
      __syncwarp();
      Planes pl{reinterpret_cast<char*>(fo + static_cast<int64_t>(m0) * p.N + n0), nullptr,
                nullptr, nullptr, static_cast<int64_t>(p.N) * 4, 3, 1,
                clamp_bytes(static_cast<int64_t>(p.N - n0) * 4, 128), p.M - m0};
      stg_flush(stg, lane, pl);
      __syncwarp();
    }
  }
}

template <int BN, bool B_MN, bool WGRAD, int EPI, bool PAIR>
__global__ void __launch_bounds__(kThreads, Cfg<BN, EPI, PAIR, B_MN>::kCtasPerSm)
    gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<BN, EPI, PAIR, B_MN>;
  constexpr int S = C::kStages;
  constexpr bool GRID = EPI == static_cast<int>(Epi::kLoRAGrid);
  constexpr bool SPLIT = EPI == static_cast<int>(Epi::kWgradSplit);
  static_assert(!PAIR || (!WGRAD && !GRID), "CTA pairs serve the rows-mode tiles");
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned stage ring (128B swizzle atoms are 8 rows x 128 B); the
  // same offsets in both CTAs of a pair (same kernel, same dynamic size)
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* ring = smem;
  uint8_t* stage_tiles = ring + S * C::kStageBytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(stage_tiles + kEpiWarps * C::kStgBytes);
  uint64_t* empty_bar = full_bar + S;
  uint64_t* tfull_bar = empty_bar + S;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* scan_tmp = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full_bar) + 192);
  // shared-memory copy of the routing tables the tile scheduler reads:
  // tile_off then offsets (row tiles; offsets only when both fit), the pair
  // tile offsets then offsets (CTA pairs), or offsets (weight-gradient and
  // grid tiles)
  int* tile_tab = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full_bar) + 256);
  const int* tab = p.G + 1 <= kTileTabInts ? tile_tab : nullptr;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pairs: this CTA's rank in the pair; the leader (rank 0) issues the MMAs
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = crank == 0;
  const int first_unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int unit_stride = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full_bar + i, p.gather_any ? 1 + 32 : 1);  // + one arrival per producer lane
      mbar_init(empty_bar + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar + i, 1);
      // one arrival per epilogue warp (of both CTAs of a pair)
      mbar_init(tempty_bar + i, kEpiWarps * (PAIR ? 2 : 1));
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // a pair's barriers are initialised before either CTA signals the other's
  if constexpr (PAIR) cluster_sync();
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.nslices; ++s) {
      prefetch_tmap(&p.sl[s].a);
      if (!WGRAD) prefetch_tmap(&p.sl[s].b);
    }
    if (WGRAD) {
      prefetch_tmap(&p.wb_hi);
      prefetch_tmap(&p.wb_lo);
    }
    if (EPI == static_cast<int>(Epi::kDgradDn) && p.om_ok) {
      prefetch_tmap(&p.om_hi);
      prefetch_tmap(&p.om_lo);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::kTmemCols);
      tmem_relinquish();
    }
  }
  // everything above overlaps the previous kernel; from here on its outputs
  // (routing tables, permuted rows, intermediates) are read
  pdl_wait();
  if constexpr (GRID) {
    // side job: words a later launch expects at zero (the split weight-gradient
    // counters), cleared by the whole grid
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.n_zero;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
      p.zero[i] = 0;
  }
  if constexpr (PAIR) {
    // the host launches pairs only when the table fits (tab != nullptr)
    group_units_table(p, tile_tab, scan_tmp, kPairM, 0);
    if (2 * (p.G + 1) <= kTileTabInts)
      for (int i = threadIdx.x; i <= p.G; i += blockDim.x)
        tile_tab[p.G + 1 + i] = __ldg(p.offsets + i);
  } else if (SPLIT) {
    // the host splits groups only when the table fits (tab != nullptr); the
    // offsets, when they fit after it, are copied first and scanned from there
    int* otab = 2 * (p.G + 1) <= kTileTabInts ? tile_tab + p.G + 1 : nullptr;
    if (otab != nullptr) {
      for (int i = threadIdx.x; i <= p.G; i += blockDim.x) otab[i] = __ldg(p.offsets + i);
      __syncthreads();
    }
    group_units_table(p, tile_tab, scan_tmp, p.wg_rows, 1, otab);
  } else if (tab != nullptr) {
    const int32_t* src = (WGRAD || GRID) ? p.offsets : p.tile_off;
    for (int i = threadIdx.x; i <= p.G; i += blockDim.x) tile_tab[i] = __ldg(src + i);
    if (!WGRAD && !GRID && 2 * (p.G + 1) <= kTileTabInts)
      for (int i = threadIdx.x; i <= p.G; i += blockDim.x)
        tile_tab[p.G + 1 + i] = __ldg(p.offsets + i);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles =
      WGRAD  ? (SPLIT ? tile_tab[p.G] : p.G) * p.n_ntiles * p.n_btiles
      : GRID ? min((__ldg(p.offsets + p.G) + BM - 1) / BM, p.max_tiles)
      : PAIR ? min(tile_tab[p.G] * p.n_ntiles, p.max_tiles)
             : min(__ldg(p.tile_off + p.G) * p.n_ntiles, p.max_tiles);

  if (warp == 0 && (lane == 0 || p.gather_any)) {
    // ------------------------------------------------------------ producer
    // Lane 0 waits for free stages and issues the TMA tile copies (alone
    // unless rows are gathered).  A gathered A operand (token rows picked by
    // sorted_src) is copied by all 32 lanes with 16-byte cp.async into the
    // 128B-swizzled layout TMA would produce.  When any slice gathers, every
    // lane arrives on each stage's full barrier (which then expects 1 + 32
    // arrivals) once its copies so far have completed; the MMA issuer fences
    // them for the async proxy.  In a CTA pair each CTA copies its own A rows
    // and its own half of B; both count their bytes on the leader's full
    // barrier, which the leader arms with the bytes of both.
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed_bits = 0, armed_phase = 0;  // stages armed, and with which parity
    bool ok = true;
    const bool lanes_arrive = p.gather_any != 0;
    // Token rows of the permuted rows first + lane + 32*i (i < n): y[i].  Rows
    // past the group's `valid` rows repeat its first row (never stored).
    auto lane_rows = [&](int first, int valid, int n, int (&y)[4]) {
      const int r0 = __ldg(p.sorted_src + first) / p.K;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        y[i] = (i < n && r < valid) ? __ldg(p.sorted_src + first + r) / p.K : r0;
      }
    };
    int y[4] = {0, 0, 0, 0};
    for (Unit u = unit_first<GRID>(p, tab, num_tiles, first_unit); u.t < num_tiles && ok;
         unit_next<GRID>(u, p, tab, num_tiles, unit_stride)) {
      const TileInfo ti = PAIR ? pair_tile_info(p, u.t, tab, crank)
                          : GRID ? grid_info(p, u.t, u.gt, u.ps, tab)
                                 : tile_info<WGRAD, true, SPLIT>(p, u.t, tab);
      if (!WGRAD && p.gather_any) lane_rows(ti.row0, ti.nvalid, 4, y);
      int cs = 0, ckc = 0;  // rows mode: slice and K offset of the next K block
      for (int kb = 0; kb < ti.nk; ++kb) {
        int s = 0, kc = 0, row = 0;
        if (!WGRAD) {
          s = cs;
          kc = ckc;
          ckc += BK;
          if (ckc >= p.sl[cs].K) {
            ++cs;
            ckc = 0;
          }
        } else {
          s = kb / ti.nkb;
          const int b = kb - s * ti.nkb;
          row = ti.row0 + b * BK;
          if (p.sl[s].gather) lane_rows(row, ti.nvalid - b * BK, 2, y);
        }
        const bool gat = p.sl[s].gather != 0;
        int w_ok = 1;
        uint64_t* fb = full_bar + stage;
        uint8_t* sa = ring + stage * C::kStageBytes;
        uint8_t* sb = sa + kAStageBytes;
        if (lane == 0) {
          w_ok = mbar_wait(empty_bar + stage, phase ^ 1u, abort_flag, kWaitTimeoutNs);
          if (w_ok) {
            armed_bits |= 1u << stage;
            armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
            if constexpr (PAIR) {
              const CUtensorMap* mb = &p.sl[s].b;
              const uint32_t fbl = mapa_shared(smem_u32(fb), 0u);  // the leader's barrier
              if (leader) mbar_expect_tx(fb, 2u * C::kStageBytes);
              tma_load_2d_pair(sa, &p.sl[s].a, fbl, kc, ti.row0);
              // this CTA's half of the B tile: its BN / 2 columns
              const int half = static_cast<int>(crank) * (BN / 2);
              if (B_MN) {
                if (p.b4d) {
                  tma_load_4d_pair(sb, mb, fbl, 0, kc, (ti.nt * BN + half) / 64, ti.g);
                } else {
#pragma unroll
                  for (int c = 0; c < BN / 128; ++c)
                    tma_load_3d_pair(sb + c * kChunkBytes, mb, fbl, ti.nt * BN + half + c * 64, kc,
                                     ti.g);
                }
              } else if (p.b_split) {
                // gate_up: the even CTA stages the gate rows, the odd one the up rows
                tma_load_3d_pair(sb, mb, fbl, kc,
                                 ti.nt * (BN / 2) + static_cast<int>(crank) * p.b_split, ti.g);
              } else {
                tma_load_3d_pair(sb, mb, fbl, kc, ti.nt * BN + half, ti.g);
              }
            } else {
              const uint32_t b_bytes = GRID ? ti.nx * kChunkBytes : C::kBStageBytes;
              mbar_expect_tx(fb, (gat ? 0u : kAStageBytes) + b_bytes);
              if (!WGRAD) {
                const CUtensorMap* mb = &p.sl[s].b;
                if (!gat) tma_load_2d(sa, &p.sl[s].a, fb, kc, ti.row0);
                if (GRID) {
                  // one 64-row (K-major) / 64-column (MN-major) block per group
                  for (int x = 0; x < ti.nx; ++x) {
                    if (!B_MN) tma_load_3d(sb + x * kChunkBytes, mb, fb, kc, 0, ti.g + x);
                    else tma_load_3d(sb + x * kChunkBytes, mb, fb, 0, kc, ti.g + x);
                  }
                } else if (p.b4d) {
                  // the whole B tile in one box: gate/up halves or MN chunks
                  if (!B_MN) tma_load_4d(sb, mb, fb, kc, ti.nt * (BN / 2), 0, ti.g);
                  else tma_load_4d(sb, mb, fb, 0, kc, ti.nt * (BN / 64), ti.g);
                } else if (!B_MN) {
                  if (p.b_split) {
                    const int n0 = ti.nt * (BN / 2);
                    tma_load_3d(sb, mb, fb, kc, n0, ti.g);
                    tma_load_3d(sb + (BN / 2) * 128, mb, fb, kc, n0 + p.b_split, ti.g);
                  } else {
                    tma_load_3d(sb, mb, fb, kc, ti.nt * BN, ti.g);
                  }
                } else {
#pragma unroll
                  for (int c = 0; c < BN / 64; ++c)
                    tma_load_3d(sb + c * kChunkBytes, mb, fb, ti.nt * BN + c * 64, kc, ti.g);
                }
              } else {
                if (!gat) {
                  tma_load_2d(sa, &p.sl[s].a, fb, ti.mt * BM, row);
                  tma_load_2d(sa + kChunkBytes, &p.sl[s].a, fb, ti.mt * BM + 64, row);
                }
                if constexpr (EPI == static_cast<int>(Epi::kWgradFull)) {
                  // B = one wide row matrix: this tile's BN columns as 64-column chunks
#pragma unroll
                  for (int c = 0; c < BN / 64; ++c)
                    tma_load_2d(sb + c * kChunkBytes, &p.wb_hi, fb, ti.nt * BN + c * 64, row);
                } else {
                  tma_load_2d(sb, &p.wb_hi, fb, 0, row);
                  tma_load_2d(sb + kChunkBytes, &p.wb_lo, fb, 0, row);
                }
              }
            }
          }
        }
        if (lanes_arrive) w_ok = __shfl_sync(0xffffffffu, w_ok, 0);  // the stage is armed
        if (!w_ok) {
          ok = false;
          break;
        }
        if (lanes_arrive) {
          if (gat) {
            const GemmSlice& sl = p.sl[s];
            const uint32_t sa_u = smem_u32(sa);
            // Each copy instruction moves whole 128-byte row segments: eight
            // lanes per segment (lane & 7 = its 16-byte piece), so global reads
            // are coalesced and the swizzled shared-memory writes conflict-free.
            const int c = lane & 7;
            if (!WGRAD) {
              // 128 rows x 64 columns: rows 4*it + lane/8, it < 32
              const bool in = kc + c * 8 < sl.gcols;
#pragma unroll
              for (int it = 0; it < 32; ++it) {
                const int r = 4 * it + (lane >> 3);
                const int tok = __shfl_sync(0xffffffffu, y[it >> 3], r & 31);
                const uint16_t* src = sl.gsrc + static_cast<int64_t>(tok) * sl.gld + kc + c * 8;
                cp_async16(sa_u + r * 128 + (((c ^ r) & 7) << 4), in ? src : sl.gsrc,
                           in ? 16u : 0u);
              }
            } else {
              // 64 K rows x two 64-column chunks: 16 lanes per row (256 bytes),
              // rows 2*it + lane/16, it < 32
              const int ch = (lane >> 3) & 1;
              const int col = ti.mt * BM + ch * 64 + c * 8;
              const bool in = col < sl.gcols;
#pragma unroll
              for (int it = 0; it < 32; ++it) {
                const int r = 2 * it + (lane >> 4);
                const int tok = __shfl_sync(0xffffffffu, y[it >> 4], r & 31);
                const uint16_t* src = sl.gsrc + static_cast<int64_t>(tok) * sl.gld + col;
                cp_async16(sa_u + ch * kChunkBytes + r * 128 + (((c ^ r) & 7) << 4),
                           in ? src : sl.gsrc, in ? 16u : 0u);
              }
            }
          }
          cp_async_mbar_arrive_noinc(fb);
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (lanes_arrive) cp_async_wait_all();  // no copy outlives the producer
    if (!ok && lane == 0) {
      if (!PAIR || leader) {
        // drain copies still in flight into this CTA's shared memory (a
        // leader's barriers also count its partner's bytes)
        for (int i = 0; i < S; ++i)
          if ((armed_bits >> i) & 1u) {
            volatile int never = 0;
            mbar_wait(full_bar + i, (armed_phase >> i) & 1u, &never, 200000000ull);
          }
      } else if (armed_bits != 0u) {
        // a partner's copies complete on the leader's barriers: give the ones
        // in flight a fixed 2 ms to land before the CTA moves on
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1 && (WGRAD || lane == 0) && (!PAIR || leader)) {
    // --------------------------------------------------------- MMA issuer
    // Lane 0 waits and issues.  In the weight-gradient kernel the whole warp
    // runs this loop and zeroes the rows past a group's end in the group's
    // last K block; elsewhere lane 0 runs it alone.  In a CTA pair only the
    // leader issues (M = 256 over both CTAs' A rows and TMEM) and its commits
    // arrive on the barriers of both CTAs.
    constexpr int kM = PAIR ? kPairM : BM;
    constexpr uint32_t idesc_full = idesc_bf16(kM, BN, WGRAD, B_MN || WGRAD);
    constexpr uint32_t idesc_one = idesc_bf16(BM, 64, false, B_MN);  // grid pass of one group
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (Unit u = unit_first<GRID>(p, tab, num_tiles, first_unit); u.t < num_tiles && ok;
         unit_next<GRID>(u, p, tab, num_tiles, unit_stride), ++local) {
      const TileInfo ti = PAIR ? pair_tile_info<false>(p, u.t, tab, crank)
                          : GRID ? grid_info(p, u.t, u.gt, u.ps, tab)
                                 : tile_info<WGRAD, WGRAD, SPLIT>(p, u.t, tab);
      const uint32_t idesc = (GRID && ti.nx == 1) ? idesc_one : idesc_full;
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(tempty_bar + buf, (use & 1u) ^ 1u, abort_flag, kWaitTimeoutNs);
      if constexpr (WGRAD) w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
      if (!w_ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
      uint32_t accum = 0;
      int cs = 0, ckc = 0;  // rows mode: slice and K offset of the next K block
      for (int kb = 0; kb < ti.nk; ++kb) {
        int f_ok = 1;
        if (lane == 0) f_ok = mbar_wait(full_bar + stage, phase, abort_flag, kWaitTimeoutNs);
        if constexpr (WGRAD) f_ok = __shfl_sync(0xffffffffu, f_ok, 0);
        if (!f_ok) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(ring + stage * C::kStageBytes);
        const uint32_t sb = sa + kAStageBytes;
        int wg_nk16 = 4;  // weight gradients: K steps of 16 rows this block takes
        if (WGRAD) {
          const int b = kb % ti.nkb;
          const int tail = ti.nvalid - b * BK;
          if (tail < BK) {
            // the group's last block: rows [tail, 64) belong to the next group
            // (or lie past the buffer).  The MMAs stop after the K step that
            // holds row tail - 1; the rows of that step past tail are zeroed
            // in the A tile (2 chunks) and, for the LoRA gradients, in the B
            // tile too (rows past the written total may hold garbage); with
            // zero A rows the wide B tile's extra rows (finite data) add nothing
            wg_nk16 = (tail + 15) / 16;
            constexpr int kPieces = EPI == static_cast<int>(Epi::kWgradFull) ? 16 : 32;
            const int n = (wg_nk16 * 16 - tail) * kPieces;
            for (int i = lane; i < n; i += 32) {
              const int line = tail + i / kPieces;
              const int piece = i % kPieces;
              const uint32_t base = (piece >> 4) ? sb : sa;
              sts128(base + ((piece >> 3) & 1) * kChunkBytes + line * 128 + (piece & 7) * 16,
                     make_uint4(0, 0, 0, 0));
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if (lane == 0) {
          tc_fence_after();
          if (p.gather_any) fence_proxy_async_smem();  // LSU-copied A rows -> async proxy
          int nk16 = WGRAD ? wg_nk16 : 4;
          if (!WGRAD) nk16 = min(4, (p.sl[cs].K - ckc + 15) / 16);
          // descriptors of the stage's first K step; each further K step of
          // 16 moves the start address field (bits 0-13, address >> 4) by
          // 32 bytes (K-major) or 2048 bytes (MN-major: 16 rows of 128 B)
          constexpr uint32_t kAStep = (WGRAD ? 2048u : 32u) >> 4;
          constexpr uint32_t kBStep = ((B_MN || WGRAD) ? 2048u : 32u) >> 4;
          const uint64_t ad = sdesc_sw128(sa, WGRAD ? kChunkBytes : 16u, 1024);
          const uint64_t bd = sdesc_sw128(sb, (B_MN || WGRAD) ? kChunkBytes : 16u, 1024);
          auto mma = [&](uint64_t a, uint64_t b, uint32_t acc) {
            if constexpr (PAIR) tc_mma_bf16_pair(d_tmem, a, b, idesc, acc);
            else tc_mma_bf16(d_tmem, a, b, idesc, acc);
          };
          if (nk16 == 4) {
            mma(ad, bd, accum);
            mma(ad + kAStep, bd + kBStep, 1u);
            mma(ad + 2 * kAStep, bd + 2 * kBStep, 1u);
            mma(ad + 3 * kAStep, bd + 3 * kBStep, 1u);
            accum = 1;
          } else {
            for (int kk = 0; kk < nk16; ++kk) {
              mma(ad + kk * kAStep, bd + kk * kBStep, accum);
              accum = 1;
            }
          }
          if constexpr (PAIR) tc_commit_pair_mc(empty_bar + stage, 3);
          else tc_commit(empty_bar + stage);
        }
        if constexpr (WGRAD) __syncwarp();
        if (!WGRAD) {
          ckc += BK;
          if (ckc >= p.sl[cs].K) {
            ++cs;
            ckc = 0;
          }
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) {
        if constexpr (PAIR) tc_commit_pair_mc(tfull_bar + buf, 3);
        else tc_commit(tfull_bar + buf);
      }
      if constexpr (WGRAD) __syncwarp();
    }
    // all MMAs issued by this warp complete before TMEM is released
    if (lane == 0) {
      if constexpr (PAIR) tc_commit_pair(drain_bar);
      else tc_commit(drain_bar);
      volatile int never = 0;
      mbar_wait(drain_bar, 0, &never, 200000000ull);
    }
    if constexpr (WGRAD) __syncwarp();
  } else if (warp >= 2) {
    // ----------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int q = warp & 3;   // TMEM lane quadrant of this warp
    const int hf = ew >> 2;   // column half owned by this warp
    const uint32_t stg = smem_u32(stage_tiles + ew * C::kStgBytes);
    int local = 0;
    for (Unit u = unit_first<GRID>(p, tab, num_tiles, first_unit); u.t < num_tiles;
         unit_next<GRID>(u, p, tab, num_tiles, unit_stride), ++local) {
      const TileInfo ti = PAIR ? pair_tile_info(p, u.t, tab, crank)
                          : GRID ? grid_info(p, u.t, u.gt, u.ps, tab)
                                 : tile_info<WGRAD, true, SPLIT>(p, u.t, tab);
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait(tfull_bar + buf, use & 1u, abort_flag, kWaitTimeoutNs)) break;
      tc_fence_after();
      const uint32_t tq =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
      // rows of this warp that belong to the tile's group (the rest of a
      // 128-row tile runs past the group's end and is not stored)
      const int64_t row0 = static_cast<int64_t>(ti.row0) + q * 32;
      const int nrows = WGRAD ? 32 : max(0, min(32, ti.nvalid - q * 32));
      if constexpr (EPI == static_cast<int>(Epi::kWgradFull)) {
        epi_wgrad_full<BN>(p, ti, tq, hf, q, lane, stg);
      } else if constexpr (WGRAD) {
        epi_wgrad<SPLIT>(p, ti, tq, hf, q, lane, stg, tab);
      } else if constexpr (EPI == static_cast<int>(Epi::kSwiGLU)) {
        epi_swiglu<BN>(p, ti, tq, hf, row0, nrows, lane, stg);
      } else if constexpr (EPI == static_cast<int>(Epi::kStore)) {
        epi_store<BN>(p, ti, tq, hf, row0, nrows, lane, stg);
      } else if constexpr (GRID) {
        epi_lora_grid(p, ti, tq, hf, row0, lane);
      } else if constexpr (EPI == static_cast<int>(Epi::kDgradDn)) {
        epi_dgrad_dn<BN>(p, ti, tq, hf, row0, nrows, lane, stg);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // the accumulator is free: the MMA issuer waits on the leader's barrier
        if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(smem_u32(tempty_bar + buf), 0u));
        else mbar_arrive(tempty_bar + buf);
      }
    }
    // TMA stores issued by this warp complete before the CTA's shared memory
    // goes away
    if constexpr (EPI == static_cast<int>(Epi::kDgradDn)) {
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }

  __syncthreads();
  // neither CTA of a pair releases TMEM or exits while the other may still
  // signal its barriers or (the leader's MMAs) read its shared memory
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicCAS(p.status, 0, kErrTimeout);
}

// Self-test of the pipelines' failure path: one thread waits on an mbarrier
// that nothing ever arrives on, with the same bounded wait the GEMM roles use;
// when the limit passes it records MOE_ERR_TIMEOUT and returns.
__global__ void wait_selftest_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, &abort_flag, timeout_ns)) atomicCAS(status, 0, kErrTimeout);
  }
}

template <int BN, bool B_MN, bool WGRAD, int EPI, bool PAIR = false>
cudaError_t launch_one(const GemmParams& p, int num_sms, cudaStream_t s) {
  using C = Cfg<BN, EPI, PAIR, B_MN>;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  auto kern = gemm_kernel<BN, B_MN, WGRAD, EPI, PAIR>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  constexpr bool kSplit = EPI == static_cast<int>(Epi::kWgradSplit);
  const int tiles = (WGRAD && !kSplit) ? p.G * p.n_ntiles * p.n_btiles : p.max_tiles;
  if constexpr (PAIR) {
    // persistent pairs: as many clusters of two as can be resident at once
    // (one CTA per SM), looked up once per device
    static int max_pairs[64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (max_pairs[dev] <= 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (num_sms / 2));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = C::kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (n <= 0) return cudaErrorInvalidConfiguration;
      max_pairs[dev] = n < num_sms / 2 ? n : num_sms / 2;
    }
    const int pairs = tiles < max_pairs[dev] ? (tiles > 0 ? tiles : 1) : max_pairs[dev];
    return launch_pdl_cluster(kern, dim3(2 * pairs), dim3(kThreads), C::kSmemBytes, s, 2u, p);
  }
  const int slots = num_sms * C::kCtasPerSm;
  const int grid = tiles < slots ? (tiles > 0 ? tiles : 1) : slots;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), C::kSmemBytes, s, p);
}

}  // namespace

cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmShape& sh, const GemmParams& p, int num_sms, cudaStream_t s) {
  constexpr int kSw = static_cast<int>(Epi::kSwiGLU);
  constexpr int kSt = static_cast<int>(Epi::kStore);
  constexpr int kDd = static_cast<int>(Epi::kDgradDn);
  constexpr int kWg = static_cast<int>(Epi::kWgrad);
  constexpr int kWgS = static_cast<int>(Epi::kWgradSplit);
  const int e = static_cast<int>(sh.epi);
  if (p.nslices < 1 || p.nslices > kMaxSlices) return cudaErrorInvalidValue;
  if (sh.wgrad) {
    if (p.n_btiles < 1) return cudaErrorInvalidValue;
    if (sh.BN == 128 && e == kWg) return launch_one<128, true, true, kWg>(p, num_sms, s);
    if (sh.BN == 128 && e == kWgS) {
      // the part table lives in shared memory; parts are whole 64-row K blocks
      if (p.G + 1 > kTileTabInts || p.wg_rows < BK || p.wg_rows % BK != 0 || !p.wg_part ||
          !p.wg_cnt)
        return cudaErrorInvalidValue;
      return launch_one<128, true, true, kWgS>(p, num_sms, s);
    }
    if (sh.BN == 256 && e == static_cast<int>(Epi::kWgradFull))
      return launch_one<256, true, true, static_cast<int>(Epi::kWgradFull)>(p, num_sms, s);
    return cudaErrorInvalidValue;
  }
  if (sh.pair) {
    // 256-row tiles on CTA pairs; the tile table must fit in shared memory
    if (p.G + 1 > kTileTabInts || p.gather_any || sh.BN != 256) return cudaErrorInvalidValue;
    if (!sh.b_mn && e == kSw) return launch_one<256, false, false, kSw, true>(p, num_sms, s);
    if (!sh.b_mn && e == kSt) return launch_one<256, false, false, kSt, true>(p, num_sms, s);
    if (sh.b_mn && e == kSt) return launch_one<256, true, false, kSt, true>(p, num_sms, s);
    if (sh.b_mn && e == kDd) return launch_one<256, true, false, kDd, true>(p, num_sms, s);
    return cudaErrorInvalidValue;
  }
  if (sh.BN == 256 && !sh.b_mn) {
    if (e == kSw) return launch_one<256, false, false, kSw>(p, num_sms, s);
    if (e == kSt) return launch_one<256, false, false, kSt>(p, num_sms, s);
  }
  if (sh.BN == 256 && sh.b_mn) {
    if (e == kSt) return launch_one<256, true, false, kSt>(p, num_sms, s);
  }
  if (sh.BN == kDgradBN && sh.b_mn && e == kDd)
    return launch_one<kDgradBN, true, false, kDd>(p, num_sms, s);
  constexpr int kLg = static_cast<int>(Epi::kLoRAGrid);
  if (sh.BN == 128 && e == kLg) {
    if (p.N > 64) return cudaErrorInvalidValue;  // one 64-column block per group
    if (sh.b_mn) return launch_one<128, true, false, kLg>(p, num_sms, s);
    return launch_one<128, false, false, kLg>(p, num_sms, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe

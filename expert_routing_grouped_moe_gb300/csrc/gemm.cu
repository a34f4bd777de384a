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
//   wgrad mode  D[M tile of a weight dimension, 128] = sum over the group's
//               rows of A[rows, M]^T [B_hi | B_lo][rows, 128] -- the per-expert
//               dA / dB reductions, one CTA per output tile, deterministic.
//
// Warp roles (192 threads, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: 128B-swizzled A and B tiles into a STAGES-deep
//               shared-memory ring (mbarrier full/empty handshake)
//   warp 1      allocates TMEM (2 x BN fp32 columns: double-buffered
//               accumulators); lane 0 issues tcgen05.mma and tcgen05.commit
//   warps 2-5   epilogue: tcgen05.ld from TMEM (warp w reads lanes 32*(w%4)..),
//               fused SwiGLU / routing-weight scale / SwiGLU backward / LoRA
//               outputs, stores to global memory; then frees the accumulator.
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
constexpr int kThreads = 192;
constexpr uint32_t kAStageBytes = BM * BK * 2;  // 16 KB
constexpr uint32_t kChunkBytes = 64 * 128;      // one [64][64] bf16 swizzle block

template <int BN>
struct Cfg {
  static constexpr uint32_t kBStageBytes = BN * BK * 2;
  static constexpr uint32_t kStageBytes = kAStageBytes + kBStageBytes;
  static constexpr int kStages = BN >= 256 ? 4 : (BN >= 128 ? 6 : 8);
  static constexpr uint32_t kTmemCols = 2 * BN;  // power of two >= 32
  static constexpr size_t kSmemBytes =
      1024 /*alignment slack*/ + static_cast<size_t>(kStages) * kStageBytes + 256 /*barriers*/ +
      (kMaxExperts + 2) * sizeof(int);
};

__device__ __forceinline__ int group_of_tile(const int* s_tile_off, int G, int mt) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tile_off[mid] <= mt) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Routing weight of permuted row p in group g (0 for padding rows, 1 for the
// shared-expert slot).
__device__ __forceinline__ float row_weight(const GemmParams& p, const int* s_tile_off, int g,
                                            int64_t row) {
  const int q = static_cast<int>(row - static_cast<int64_t>(s_tile_off[g]) * BM);
  const int off = __ldg(p.offsets + g);
  const int cnt = __ldg(p.offsets + g + 1) - off;
  if (q >= cnt) return 0.f;
  const int i = __ldg(p.sorted_src + off + q);
  const int t = i / p.K;
  const int j = i - t * p.K;
  return j < p.k ? __ldg(p.topk_w + static_cast<int64_t>(t) * p.k + j) : 1.f;
}

__device__ __forceinline__ void store8(uint16_t* dst, const float (&v)[8]) {
  *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                              pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}
// hi = bf16(v), lo = bf16(v - hi): the pair holds ~16 significant bits of v.
__device__ __forceinline__ void store8_pair(uint16_t* hi, int64_t pair, const float (&v)[8]) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    l[i] = pack_bf16x2(v[2 * i] - bf16lo(h[i]), v[2 * i + 1] - bf16hi(h[i]));
  }
  *reinterpret_cast<uint4*>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(hi + pair) = make_uint4(l[0], l[1], l[2], l[3]);
}
__device__ __forceinline__ void load8(const uint16_t* src, float (&v)[8]) {
  const uint4 x = __ldg(reinterpret_cast<const uint4*>(src));
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16lo(w[i]);
    v[2 * i + 1] = bf16hi(w[i]);
  }
}
__device__ __forceinline__ void load8f(const float* src, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(src));
  const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8f(float* dst, const float (&v)[8]) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.f / (1.f + __expf(-z)); }

// Tile coordinates shared by all roles.
struct TileInfo {
  int g;       // expert group
  int mt;      // rows mode: permuted M tile; wgrad: M tile of the weight dimension
  int nt;      // rows mode: N tile
  int nk;      // K blocks in total
  int rt;      // wgrad: row tiles of the group (K blocks per slice = 2 * rt)
  int64_t rb;  // wgrad: first permuted row of the group
};

template <bool WGRAD>
__device__ __forceinline__ TileInfo tile_info(const GemmParams& p, const int* s_tile_off, int t) {
  TileInfo ti;
  if (!WGRAD) {
    ti.mt = t / p.n_ntiles;
    ti.nt = t - ti.mt * p.n_ntiles;
    ti.g = group_of_tile(s_tile_off, p.G, ti.mt);
    ti.nk = 0;
    for (int s = 0; s < p.nslices; ++s) ti.nk += (p.sl[s].K + BK - 1) / BK;
    ti.rt = 0;
    ti.rb = 0;
  } else {
    ti.g = t / p.n_ntiles;
    ti.mt = t - ti.g * p.n_ntiles;
    ti.nt = 0;
    ti.rt = s_tile_off[ti.g + 1] - s_tile_off[ti.g];
    ti.nk = ti.rt * (BM / BK) * p.nslices;
    ti.rb = static_cast<int64_t>(s_tile_off[ti.g]) * BM;
  }
  return ti;
}

// Slice and K offset of k-block kb (rows mode).
__device__ __forceinline__ void rows_kblock(const GemmParams& p, int kb, int& s, int& kc,
                                            int& kext) {
  s = 0;
  int nk = (p.sl[0].K + BK - 1) / BK;
  while (kb >= nk && s + 1 < p.nslices) {
    kb -= nk;
    ++s;
    nk = (p.sl[s].K + BK - 1) / BK;
  }
  kc = kb * BK;
  kext = p.sl[s].K - kc;
}

template <int BN, bool B_MN, bool WGRAD, int EPI>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned stage ring (128B swizzle atoms are 8 rows x 128 B)
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* ring = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(ring + S * C::kStageBytes);
  uint64_t* empty_bar = full_bar + S;
  uint64_t* tfull_bar = empty_bar + S;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_tile_off = reinterpret_cast<int*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full_bar + i, 1);
      mbar_init(empty_bar + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar + i, 1);
      mbar_init(tempty_bar + i, 4 * 32);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.nslices; ++s) {
      prefetch_tmap(&p.sl[s].a);
      if (!WGRAD) prefetch_tmap(&p.sl[s].b);
    }
    if (WGRAD) {
      prefetch_tmap(&p.wb_hi);
      prefetch_tmap(&p.wb_lo);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i <= p.G; i += kThreads) s_tile_off[i] = __ldg(p.tile_off + i);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles =
      WGRAD ? p.G * p.n_ntiles : min(s_tile_off[p.G] * p.n_ntiles, p.max_tiles);

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    int armed[S];
#pragma unroll
    for (int i = 0; i < S; ++i) armed[i] = -1;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      const TileInfo ti = tile_info<WGRAD>(p, s_tile_off, t);
      for (int kb = 0; kb < ti.nk; ++kb) {
        if (!mbar_wait(empty_bar + stage, phase ^ 1u, abort_flag, kWaitTimeoutNs)) {
          ok = false;
          break;
        }
        uint64_t* fb = full_bar + stage;
        uint8_t* sa = ring + stage * C::kStageBytes;
        uint8_t* sb = sa + kAStageBytes;
        mbar_expect_tx(fb, C::kStageBytes);
        armed[stage] = static_cast<int>(phase);
        if (!WGRAD) {
          int s, kc, kext;
          rows_kblock(p, kb, s, kc, kext);
          const CUtensorMap* ma = &p.sl[s].a;
          const CUtensorMap* mb = &p.sl[s].b;
          tma_load_2d(sa, ma, fb, kc, ti.mt * BM);
          if (!B_MN) {
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
          const int per = ti.rt * (BM / BK);
          const int s = kb / per;
          const int row = static_cast<int>(ti.rb) + (kb - s * per) * BK;
          tma_load_2d(sa, &p.sl[s].a, fb, ti.mt * BM, row);
          tma_load_2d(sa + kChunkBytes, &p.sl[s].a, fb, ti.mt * BM + 64, row);
          tma_load_2d(sb, &p.wb_hi, fb, 0, row);
          tma_load_2d(sb + kChunkBytes, &p.wb_lo, fb, 0, row);
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {
      // drain copies still in flight into this CTA's shared memory
      for (int i = 0; i < S; ++i)
        if (armed[i] >= 0) {
          volatile int never = 0;
          mbar_wait(full_bar + i, static_cast<uint32_t>(armed[i]), &never, 200000000ull);
        }
    }
  } else if (warp == 1 && lane == 0) {
    // --------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16(BM, BN, WGRAD, B_MN || WGRAD);
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
      const TileInfo ti = tile_info<WGRAD>(p, s_tile_off, t);
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait(tempty_bar + buf, (use & 1u) ^ 1u, abort_flag, kWaitTimeoutNs)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
      uint32_t accum = 0;
      for (int kb = 0; kb < ti.nk; ++kb) {
        if (!mbar_wait(full_bar + stage, phase, abort_flag, kWaitTimeoutNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(ring + stage * C::kStageBytes);
        const uint32_t sb = sa + kAStageBytes;
        int nk16 = 4;
        if (!WGRAD) {
          int s, kc, kext;
          rows_kblock(p, kb, s, kc, kext);
          nk16 = min(4, (kext + 15) / 16);
        }
        for (int kk = 0; kk < nk16; ++kk) {
          uint64_t ad, bd;
          if (!WGRAD) ad = sdesc_sw128(sa + kk * 32, 16, 1024);
          else ad = sdesc_sw128(sa + kk * 2048, kChunkBytes, 1024);
          if (!B_MN && !WGRAD) bd = sdesc_sw128(sb + kk * 32, 16, 1024);
          else bd = sdesc_sw128(sb + kk * 2048, kChunkBytes, 1024);
          tc_mma_bf16(d_tmem, ad, bd, idesc, accum);
          accum = 1;
        }
        tc_commit(empty_bar + stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(tfull_bar + buf);
    }
    // all MMAs issued by this thread complete before TMEM is released
    tc_commit(drain_bar);
    volatile int never = 0;
    mbar_wait(drain_bar, 0, &never, 200000000ull);
  } else if (warp >= 2) {
    // ----------------------------------------------------------- epilogue
    const int q = warp & 3;               // TMEM lane quadrant of this warp
    const int r_in_tile = q * 32 + lane;  // accumulator row
    int local = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
      const TileInfo ti = tile_info<WGRAD>(p, s_tile_off, t);
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait(tfull_bar + buf, use & 1u, abort_flag, kWaitTimeoutNs)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);

      if constexpr (WGRAD) {
        // columns [0,64) = A * B_hi, [64,128) = A * B_lo
        const int m = ti.mt * BM + r_in_tile;
        const bool has = ti.nk > 0;
        float* fo = p.fout + static_cast<int64_t>(ti.g) * p.fstride;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 16) {
          float vh[16], vl[16];
          if (has) {
            tmem_ld16(tbase + c0, vh);
            tmem_ld16(tbase + 64 + c0, vl);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) vh[i] = vl[i] = 0.f;
          }
          if (m < p.M) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int n = c0 + i;
              if (n < p.N) {
                const float v = vh[i] + vl[i];
                if (p.transpose_out) fo[static_cast<int64_t>(n) * p.M + m] = v;
                else fo[static_cast<int64_t>(m) * p.N + n] = v;
              }
            }
          }
        }
      } else {
        const int64_t row = static_cast<int64_t>(ti.mt) * BM + r_in_tile;
        if constexpr (EPI == static_cast<int>(Epi::kSwiGLU)) {
          // accumulator columns [0, BN/2) = gate, [BN/2, BN) = up of the same features
          const int f = p.N;
          float* hrow = p.fout + row * p.ld0;                         // h [rows, 2f] fp32
          uint16_t* arow = p.out0 + row * static_cast<int64_t>(f);    // act pair [rows, f]
#pragma unroll 1
          for (int c0 = 0; c0 < BN / 2; c0 += 16) {
            float g16[16], u16[16];
            tmem_ld16(tbase + c0, g16);
            tmem_ld16(tbase + BN / 2 + c0, u16);
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
              const int j = ti.nt * (BN / 2) + c0 + h8 * 8;
              if (j < f) {
                float gv[8], uv[8], av[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  gv[i] = g16[h8 * 8 + i];
                  uv[i] = u16[h8 * 8 + i];
                  av[i] = gv[i] * sigmoidf_(gv[i]) * uv[i];
                }
                store8f(hrow + j, gv);
                store8f(hrow + f + j, uv);
                store8_pair(arow + j, p.pair, av);
              }
            }
          }
        } else if constexpr (EPI == static_cast<int>(Epi::kScaleW) ||
                             EPI == static_cast<int>(Epi::kStore)) {
          const float w =
              EPI == static_cast<int>(Epi::kScaleW) ? row_weight(p, s_tile_off, ti.g, row) : 1.f;
          uint16_t* orow = p.out0 + row * p.ld0;
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 16) {
            float v16[16];
            tmem_ld16(tbase + c0, v16);
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
              const int j = ti.nt * BN + c0 + h8 * 8;
              if (j < p.N) {
                float ov[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) ov[i] = w * v16[h8 * 8 + i];
                store8(orow + j, ov);
              }
            }
          }
        } else if constexpr (EPI == static_cast<int>(Epi::kLoRA)) {
          const bool need_w = p.out1 != nullptr || p.out2 != nullptr;
          const float w = need_w ? row_weight(p, s_tile_off, ti.g, row) : 0.f;
          const float s = p.scale;
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 16) {
            float v16[16];
            tmem_ld16(tbase + c0, v16);
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
              const int j = ti.nt * BN + c0 + h8 * 8;
              if (j < p.N) {
                const int64_t o = row * p.ld0 + j;
                float ov[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) ov[i] = s * v16[h8 * 8 + i];
                store8_pair(p.out0 + o, p.pair, ov);
                if (p.out1 != nullptr) {
#pragma unroll
                  for (int i = 0; i < 8; ++i) ov[i] *= w;
                  store8_pair(p.out1 + o, p.pair, ov);
                }
                if (p.out2 != nullptr) {
                  float ah[8], al[8];
                  load8(p.aux0 + o, ah);
                  load8(p.aux0 + p.pair + o, al);
#pragma unroll
                  for (int i = 0; i < 8; ++i) ah[i] = w * (ah[i] + al[i]);
                  store8_pair(p.out2 + o, p.pair, ah);
                }
              }
            }
          }
        } else if constexpr (EPI == static_cast<int>(Epi::kDgradDn)) {
          // acc = g = dY W_dn + s (dY B_dn) A_dn (unscaled by the routing weight)
          const int f = p.N;
          const float w = row_weight(p, s_tile_off, ti.g, row);
          const float* hrow = p.fin + row * p.ld0;  // h [rows, 2f] fp32
          uint16_t* drow = p.out0 + row * p.ld0;    // dh pair [rows, 2f]
          float dot = 0.f;
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 16) {
            float v16[16];
            tmem_ld16(tbase + c0, v16);
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
              const int j = ti.nt * BN + c0 + h8 * 8;
              if (j < f) {
                float gt[8], up[8], dg[8], du[8];
                load8f(hrow + j, gt);
                load8f(hrow + f + j, up);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float gr = v16[h8 * 8 + i];
                  const float sg = sigmoidf_(gt[i]);
                  const float sl = gt[i] * sg;
                  dot = fmaf(sl * up[i], gr, dot);
                  const float da = w * gr;
                  dg[i] = da * up[i] * sg * (1.f + gt[i] * (1.f - sg));
                  du[i] = da * sl;
                }
                store8_pair(drow + j, p.pair, dg);
                store8_pair(drow + f + j, p.pair, du);
              }
            }
          }
          p.fout[static_cast<int64_t>(ti.nt) * p.fstride + row] = dot;
        }
      }
      tc_fence_before();
      mbar_arrive(tempty_bar + buf);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicCAS(p.status, 0, kErrTimeout);
}

template <int BN, bool B_MN, bool WGRAD, int EPI>
cudaError_t launch_one(const GemmParams& p, int num_sms, cudaStream_t s) {
  using C = Cfg<BN>;
  auto kern = gemm_kernel<BN, B_MN, WGRAD, EPI>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  const int tiles = WGRAD ? p.G * p.n_ntiles : p.max_tiles;
  const int grid = tiles < num_sms ? (tiles > 0 ? tiles : 1) : num_sms;
  kern<<<grid, kThreads, C::kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const GemmShape& sh, const GemmParams& p, int num_sms, cudaStream_t s) {
  constexpr int kSw = static_cast<int>(Epi::kSwiGLU);
  constexpr int kSc = static_cast<int>(Epi::kScaleW);
  constexpr int kSt = static_cast<int>(Epi::kStore);
  constexpr int kLo = static_cast<int>(Epi::kLoRA);
  constexpr int kDd = static_cast<int>(Epi::kDgradDn);
  constexpr int kWg = static_cast<int>(Epi::kWgrad);
  const int e = static_cast<int>(sh.epi);
  if (p.nslices < 1 || p.nslices > kMaxSlices) return cudaErrorInvalidValue;
  if (sh.wgrad) {
    if (sh.BN == 128 && e == kWg) return launch_one<128, true, true, kWg>(p, num_sms, s);
    return cudaErrorInvalidValue;
  }
  if (sh.BN == 256 && !sh.b_mn) {
    if (e == kSw) return launch_one<256, false, false, kSw>(p, num_sms, s);
    if (e == kSc) return launch_one<256, false, false, kSc>(p, num_sms, s);
  }
  if (sh.BN == 256 && sh.b_mn) {
    if (e == kDd) return launch_one<256, true, false, kDd>(p, num_sms, s);
    if (e == kSt) return launch_one<256, true, false, kSt>(p, num_sms, s);
  }
  if (sh.BN == 64 && e == kLo) {
    if (sh.b_mn) return launch_one<64, true, false, kLo>(p, num_sms, s);
    return launch_one<64, false, false, kLo>(p, num_sms, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe

// Persistent, warp-specialised tcgen05 GEMM used for every contraction of the MoE layer:
// the router product, the grouped expert gate/up and down projections (with their
// fused SwiGLU / gate-scaling epilogues and the LoRA K-blocks), the LoRA down-projections
// and the backward data-gradient products.
//
// Roles (256 threads, one CTA per SM; two for the LoRA weight gradients):
//   warp 0       TMA producer: 64-wide K blocks of A and of each B into a STAGES-deep ring
//   warp 1       TMEM allocator and MMA issuer (one thread issues tcgen05.mma)
//   warps 2..3   A-row gather (only when the permute is fused: cp.async of token rows)
//   warps 4..7   epilogue: tcgen05.ld of the accumulator rows (warp w reads TMEM lanes
//                32*(w%4) .. +31), fused math, global stores (bf16 outputs of the gate-scale
//                and store epilogues staged per warp in shared memory for whole-row writes)
// Two TMEM accumulator buffers let the epilogue of tile i overlap the main loop of tile i+1,
// except on 256-row tiles (two 128-row A subtiles per B stage), whose one accumulator fills
// all 512 TMEM columns.
//
// CTA pairs (CG = 2, clusters of two CTAs on the two SMs of a TPC): one M = 256 tile per
// pair, issued by the first CTA as tcgen05.mma.cta_group::2; each CTA stages its own 128 A
// rows and half of every B tile, both CTAs' TMA copies complete on the first CTA's stage
// barrier, and the first CTA's commits arrive on the stage-free and accumulator-full
// barriers of both.  Each CTA keeps two accumulators of its 128 rows, so the epilogue still
// overlaps the next tile, with half the weight bytes staged per SM.
//
// Operand tiles in shared memory use the 128-byte swizzle that TMA writes:
//   K-major  (rows x 64 K): 128-byte rows, 8-row atoms of 1024 B -> SBO = 1024; the k-th
//            16-wide MMA step starts 32 B further into the atom.
//   MN-major (64 K x 64 MN per box): 128-byte K-rows; boxes for consecutive 64-wide MN
//            chunks 8 KB apart -> LBO = 8192, SBO = 1024; the k-th MMA step starts 2 KB on.
#pragma once

#include "ptx.cuh"
#include "topk_keys.cuh"

namespace moe {

// MSUB: 128-row A subtiles per CTA tile (2: two consecutive m-tiles of one group share every
// B stage).  CTAS: CTAs resident per SM.  NACC: TMEM accumulator buffers per CTA (2 overlaps
// a tile's epilogue with the next tile's main loop; 1 when two buffers of every resident CTA
// do not fit the 512 TMEM columns, in which case a second CTA on the SM does the covering).
// CG: CTAs per MMA (2: a CTA pair issues M = 256 tcgen05.mma.cta_group::2 tiles, each CTA
// staging its own 128 A rows and half of every B tile).
template <int BN, int NB, bool A_MN, bool B_MN, int EPI, int STAGES, int MSUB = 1, int CTAS = 1,
          int CG = 1>
struct GemmCfg {
  static constexpr int A_SUB_BYTES = kBM * kBK * 2;
  static constexpr int A_BYTES = MSUB * A_SUB_BYTES;
  // B rows (K-major) or MN columns (MN-major) of one B operand staged by this CTA
  static constexpr int B_ROWS = CG == 2 ? BN / 2 : BN;
  // an MN-major B tile is always whole 64-wide TMA boxes (N below 64 is zero-filled)
  static constexpr int B_BYTES = (B_MN ? ((B_ROWS + 63) / 64) * 64 : B_ROWS) * kBK * 2;
  // CTA pairs with two K-major B operands (gate and up) run one MMA of N = 2*BN per k step:
  // its B rows 0..BN-1 (the first operand's tile) sit in the first CTA and BN..2BN-1 (the
  // second's) in the second, so each CTA stages one whole operand tile
  static constexpr bool PAIR_JOIN = CG == 2 && NB == 2 && !B_MN && 2 * BN <= 256 &&
                                    EPI != EPI_F32_BIAS && EPI != EPI_ROUTE;
  static constexpr int STAGE_BYTES = A_BYTES + NB * B_BYTES;
  // The router (EPI_F32_BIAS) with two B operands sums them into one accumulator: they are
  // the bf16 hi and lo parts of the same fp32 weights, both multiplied by the same A stage.
  static constexpr bool SUMB = ((EPI == EPI_F32_BIAS || EPI == EPI_ROUTE) && NB == 2);
  static constexpr int ACC_NB = SUMB ? 1 : NB;  // accumulators of BN columns per subtile
  static constexpr int ACC_COLS = MSUB * ACC_NB * BN;
  static constexpr int NACC = (2 * ACC_COLS * CTAS <= 512) ? 2 : 1;
  static constexpr int TMEM_COLS = (NACC * ACC_COLS <= 32)    ? 32
                                   : (NACC * ACC_COLS <= 64)  ? 64
                                   : (NACC * ACC_COLS <= 128) ? 128
                                   : (NACC * ACC_COLS <= 256) ? 256
                                                              : 512;
  // the gate-scale and store epilogues stage each warp's 32 rows in shared memory for
  // coalesced stores (the SwiGLU epilogue stores per thread: staging it was slower at c2)
  static constexpr bool STAGED_EPI = EPI == EPI_GATE_SCALE || EPI == EPI_STORE;
  static constexpr int EPI_STAGE_BYTES = STAGED_EPI ? 4 * 32 * 128 : 0;
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/ + EPI_STAGE_BYTES;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
  static_assert(NACC * ACC_COLS <= 512, "accumulators must fit in TMEM");
  static_assert(!B_MN || BN % 64 == 0, "MN-major B is read in whole 64-wide boxes");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(CG == 1 || (MSUB == 1 && CTAS == 1 && !A_MN && EPI != EPI_WGRAD),
                "CTA pairs: K-major A, one CTA per SM");
  static_assert(CG == 1 || (B_MN ? BN % 128 == 0 : (BN / 2) % 8 == 0),
                "half B tiles stay whole boxes / swizzle atoms");
};

// 32 x 32 transpose across a warp: on entry lane l holds row l (v[j] = element (l, j)), on
// exit column l (v[j] = element (j, l)).  Five butterfly stages: at stride s the lanes whose
// bit s is set trade the s-wide off-diagonal blocks with their partner lane l ^ s.
__device__ __forceinline__ void warp_transpose32(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j & s) continue;
      const float send = up ? v[j] : v[j | s];
      const float recv = __shfl_xor_sync(0xffffffffu, send, s);
      if (up) {
        v[j] = recv;
      } else {
        v[j | s] = recv;
      }
    }
  }
}

struct TileCoord {
  int g, m, n, row0, rows_valid;
};

__device__ __forceinline__ bool decode_tile(const GemmParams& P, int tile, TileCoord& tc) {
  if (P.group_off == nullptr) {
    const int total = P.m_tiles * P.n_tiles;
    if (tile >= total) return false;
    // m-major: the n-tiles of one row block run side by side, so each A tile is read from
    // DRAM once and re-read from L2 (B is small and stays L2-resident for dense problems)
    tc.g = 0;
    tc.m = tile / P.n_tiles;
    tc.n = tile - tc.m * P.n_tiles;
    tc.row0 = tc.m * kBM;
    tc.rows_valid = min(kBM, P.M - tc.row0);
    return true;
  }
  const int total = __ldg(&P.tile_off[P.G]) * P.n_tiles;
  if (tile >= total) return false;
  int lo = 0, hi = P.G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&P.tile_off[mid]) * P.n_tiles <= tile) lo = mid; else hi = mid - 1;
  }
  const int t0 = __ldg(&P.tile_off[lo]);
  const int mt = __ldg(&P.tile_off[lo + 1]) - t0;
  const int local = tile - t0 * P.n_tiles;
  tc.g = lo;
  tc.n = local / mt;
  tc.m = local - tc.n * mt;
  const int r0 = __ldg(&P.group_off[lo]);
  tc.row0 = r0 + tc.m * kBM;
  tc.rows_valid = min(kBM, __ldg(&P.group_off[lo + 1]) - tc.row0);
  return true;
}

// Grouped-over-K problems (LoRA weight gradients): tile = (group g, m-tile); the K range is
// the rows [group_off[g], group_off[g+1]) of both operands; every group has m_tiles tiles.
struct KRange {
  int k0, nrows, nkb;
};

__device__ __forceinline__ bool decode_tile_wgrad(const GemmParams& P, int tile, TileCoord& tc,
                                                  KRange& kr) {
  if (tile >= P.G * P.m_tiles * P.n_tiles) return false;
  tc.g = tile / (P.m_tiles * P.n_tiles);
  const int rem = tile - tc.g * P.m_tiles * P.n_tiles;
  tc.n = rem / P.m_tiles;
  tc.m = rem - tc.n * P.m_tiles;
  tc.row0 = tc.m * kBM;
  tc.rows_valid = min(kBM, P.M - tc.row0);
  const int lo = __ldg(&P.group_off[tc.g]);
  const int hi = __ldg(&P.group_off[tc.g + 1]);
  kr.k0 = lo;
  kr.nrows = hi > lo ? hi - lo : 0;
  kr.nkb = (kr.nrows + kBK - 1) / kBK;
  return true;
}

// Two-subtile launches (MSUB = 2): unit `pt` covers m-tiles 2*pair and 2*pair+1 of one
// (group, n-tile) in one CTA (rows_valid up to 256); the second subtile is skipped when the
// group's rows end inside the first.  pair_off is the prefix over groups of ceil(m-tiles/2).
__device__ __forceinline__ bool decode_sub_tile(const GemmParams& P, int pt, TileCoord& tc) {
  if (P.group_off == nullptr) {
    const int pairs = (P.m_tiles + 1) >> 1;
    if (pt >= pairs * P.n_tiles) return false;
    const int mp = pt / P.n_tiles;
    tc.g = 0;
    tc.n = pt - mp * P.n_tiles;
    tc.m = 2 * mp;
    tc.row0 = tc.m * kBM;
    tc.rows_valid = min(2 * kBM, P.M - tc.row0);
    return true;
  }
  const int total = __ldg(&P.pair_off[P.G]) * P.n_tiles;
  if (pt >= total) return false;
  int lo = 0, hi = P.G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&P.pair_off[mid]) * P.n_tiles <= pt) lo = mid; else hi = mid - 1;
  }
  const int p0 = __ldg(&P.pair_off[lo]);
  const int np = __ldg(&P.pair_off[lo + 1]) - p0;
  const int local = pt - p0 * P.n_tiles;
  tc.g = lo;
  tc.n = local / np;
  tc.m = 2 * (local - tc.n * np);
  tc.row0 = __ldg(&P.group_off[lo]) + tc.m * kBM;
  tc.rows_valid = min(2 * kBM, __ldg(&P.group_off[lo + 1]) - tc.row0);
  return true;
}

// Zero the K rows [valid, end) of an MN-major operand tile of `chunks` 64-wide boxes (each K
// row is one 128-byte line of a box), by the 32 lanes of one warp.
__device__ __forceinline__ void zero_k_tail(uint8_t* tile, int chunks, int valid, int end,
                                            int lane) {
  const int items = (end - valid) * 8;  // 16-byte parts of the lines to clear, per box
  for (int c = 0; c < chunks; ++c) {
    uint8_t* box = tile + c * 8192;
    for (int i = lane; i < items; i += 32) {
      const int kr = valid + (i >> 3);
      reinterpret_cast<uint4*>(box + (kr >> 3) * 1024 + (kr & 7) * 128)[i & 7] =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Store 16 consecutive bf16 values of one row, clipped to `ncols_left` columns.
__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* dst, const float (&v)[16],
                                              int ncols_left) {
  if (ncols_left >= 16) {
    uint4 a, b;
    a.x = pack_bf16x2(v[0], v[1]);   a.y = pack_bf16x2(v[2], v[3]);
    a.z = pack_bf16x2(v[4], v[5]);   a.w = pack_bf16x2(v[6], v[7]);
    b.x = pack_bf16x2(v[8], v[9]);   b.y = pack_bf16x2(v[10], v[11]);
    b.z = pack_bf16x2(v[12], v[13]); b.w = pack_bf16x2(v[14], v[15]);
    reinterpret_cast<uint4*>(dst)[0] = a;
    reinterpret_cast<uint4*>(dst)[1] = b;
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i < ncols_left) dst[i] = __float2bfloat16_rn(v[i]);
  }
}

// One epilogue warp's block of 32 rows (row r held by lane r) x CH bf16 columns, packed in
// pairs, stored to out[row_base + r][0 .. CH) (ld ldo) for rows r < rows_valid and columns
// < cols_valid (a multiple of 8).  Written row-wise into the warp's staging buffer (2*CH*32
// bytes, 128-byte swizzle: 16-byte chunk index XOR bits 7-9 of the offset, so neither the
// row-wise writes nor the column-wise reads conflict on banks), then read back so that each
// store instruction writes 32 / (CH / 8) whole row segments of 2*CH contiguous bytes.
template <int CH>
__device__ __forceinline__ void warp_store_rows(uint8_t* buf, const uint32_t (&w)[CH / 2],
                                                int lane, __nv_bfloat16* out, long ldo,
                                                long row_base, int rows_valid, int cols_valid) {
  constexpr int RB = CH * 2;    // bytes per row
  constexpr int CPR = RB / 16;  // 16-byte chunks per row
  constexpr int RPI = 32 / CPR; // rows per store instruction
  static_assert(CH == 32 || CH == 64, "staged chunk width");
#pragma unroll
  for (int j = 0; j < CPR; ++j) {
    uint32_t off = lane * RB + j * 16;
    off ^= ((off >> 7) & 7u) << 4;
    *reinterpret_cast<uint4*>(buf + off) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
  __syncwarp();
  const int j = lane % CPR;
#pragma unroll
  for (int it = 0; it < 32 / RPI; ++it) {
    const int r = it * RPI + lane / CPR;
    uint32_t off = r * RB + j * 16;
    off ^= ((off >> 7) & 7u) << 4;
    const uint4 v = *reinterpret_cast<const uint4*>(buf + off);
    if (r < rows_valid && j * 8 < cols_valid)
      *reinterpret_cast<uint4*>(out + (row_base + r) * ldo + j * 8) = v;
  }
  __syncwarp();  // the buffer is reused by the warp's next chunk
}

__device__ __forceinline__ void load_bf16x16(const __nv_bfloat16* src, float (&v)[16]) {
  const uint4 a = reinterpret_cast<const uint4*>(src)[0];
  const uint4 b = reinterpret_cast<const uint4*>(src)[1];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    float2 f = __bfloat1622float2(p);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

// Fused combine, after an epilogue warp stored its rows row_w .. row_w + wrows - 1 of the
// 256-wide n-tile strip n: each stored row counts down its token's strip counter; a warp that
// brings a counter to zero holds the token's last row of that strip and sums the token's kept
// rows (rank order j = 0 .. k-1, fp32, one bf16 rounding: the separate combine's arithmetic)
// into y.  Writers fence before counting and finishers after, so every row a finisher reads
// is visible; rows are read from L2 (written by other SMs during this kernel).
__device__ __forceinline__ void combine_finish(const GemmParams& P, int n, long row_w,
                                               int wrows, int lane) {
  __threadfence();
  __syncwarp();
  int tok = -1;
  bool fin = false;
  if (lane < wrows) {
    const int slot = __ldg(&P.row_slot[row_w + lane]);
    tok = slot / P.comb_k;
    fin = atomicSub(&P.comb_cnt[static_cast<size_t>(tok) * P.n_tiles + n], 1) == 1;
  }
  unsigned fm = __ballot_sync(0xffffffffu, fin);
  if (!fm) return;
  __threadfence();
  const __nv_bfloat16* yp = reinterpret_cast<const __nv_bfloat16*>(P.out0);
  __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(P.comb_y);
  const int col = n * 256 + lane * 8;  // one 16-byte vector of the strip per lane
  while (fm) {
    const int src = __ffs(fm) - 1;
    fm &= fm - 1;
    const int t = __shfl_sync(0xffffffffu, tok, src);
    const int r = lane < P.comb_k ? __ldcg(&P.comb_slot_row[static_cast<size_t>(t) * P.comb_k + lane]) : -1;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // the token's rows in batches of 8: all loads of a batch in flight, then summed in rank
    // order
    for (int j0 = 0; j0 < P.comb_k; j0 += 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int rj = __shfl_sync(0xffffffffu, r, (j0 + u) & 31);
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (j0 + u < P.comb_k && rj >= 0 && col < P.N)
          v[u] = __ldcg(reinterpret_cast<const uint4*>(yp + static_cast<size_t>(rj) * P.ldo + col));
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int rj = __shfl_sync(0xffffffffu, r, (j0 + u) & 31);
        if (j0 + u < P.comb_k && rj >= 0) {
          const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            acc[2 * i] += f.x;
            acc[2 * i + 1] += f.y;
          }
        }
      }
    }
    if (col < P.N) {
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * P.N + col) = o;
    }
  }
}

// CTA pairs (CG = 2) walk the two-subtile units: CTA `rank` of the pair takes the unit's
// rows rank*128 .. rank*128+127 (none of them valid when the group ends in the first half:
// that CTA still stages A rows and takes part in every barrier, and stores nothing).
template <int EPI, int MSUB, int CG>
__device__ __forceinline__ bool next_tile(const GemmParams& P, int tile, int rank, TileCoord& tc,
                                          KRange& kr) {
  if constexpr (EPI == EPI_WGRAD) {
    return decode_tile_wgrad(P, tile, tc, kr);
  } else {
    kr.k0 = 0;
    kr.nrows = 0;
    kr.nkb = 0;
    if constexpr (CG == 2) {
      if (!decode_sub_tile(P, tile, tc)) return false;
      tc.m += rank;
      tc.row0 += rank * kBM;
      tc.rows_valid = max(0, min(kBM, tc.rows_valid - rank * kBM));
      return true;
    }
    if constexpr (MSUB == 2) return decode_sub_tile(P, tile, tc);
    return decode_tile(P, tile, tc);
  }
}

// CTAS CTAs per SM: with one, a thread may use up to 255 registers; with two, 128.
template <int BN, int NB, bool A_MN, bool B_MN, int EPI, int STAGES, int MSUB, int CTAS, int CG>
__global__ void __launch_bounds__(256, CTAS) gemm_kernel(const __grid_constant__ GemmParams P) {
  using C = GemmCfg<BN, NB, A_MN, B_MN, EPI, STAGES, MSUB, CTAS, CG>;
  static_assert(MSUB == 1 || (EPI != EPI_WGRAD && !A_MN),
                "two subtiles: M-grouped or dense, K-major A");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* drain = reinterpret_cast<uint64_t*>(tmem_slot + 2);  // 8-byte aligned slot
  __shared__ int zero_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pairs: clusters of two consecutive CTAs; rank 0 issues the pair's MMAs
  const int rank = (CG == 2) ? static_cast<int>(cluster_ctarank()) : 0;
  const int unit0 = blockIdx.x / CG;     // first work unit of this CTA (pair)
  const int unit_step = gridDim.x / CG;  // number of CTAs (pairs)

  if (threadIdx.x == 0) {
    // with a gathered A operand a stage is full after the producer's expect-tx arrival
    // (B bytes) and one arrival of the gather warp that filled its A tile
    const uint32_t full_count =
        (!A_MN && EPI != EPI_WGRAD && MSUB == 1 && CG == 1 && P.gather_slot != nullptr) ? 2u
                                                                                      : 1u;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], full_count);
      mbar_init(&empty[s], 1);  // a stage is free once the MMA warp has released it
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      // every epilogue thread (one CTA), or lane 0 of each epilogue warp of both CTAs
      mbar_init(&acc_empty[a], CG == 2 ? 8 : 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    zero_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < P.nmaps; ++i) tma_prefetch_desc(&P.maps[i]);
  }
  if (warp == 1) {
    tmem_alloc<CG>(tmem_slot, C::TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  if constexpr (CG == 2) {
    cluster_sync();  // both CTAs' barriers exist before either signals the other's
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_a = l2_policy_evict_last();
    const uint64_t pol_b = P.b_policy ? l2_policy_evict_normal() : l2_policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    TileCoord tc;
    KRange kr;
    for (int tile = unit0; ok && next_tile<EPI, MSUB, CG>(P, tile, rank, tc, kr); tile += unit_step) {
      const int nseg = (EPI == EPI_WGRAD) ? 1 : P.nseg;
      for (int s = 0; ok && s < nseg; ++s) {
        const GemmSeg& sg = P.seg[s];
        const int nkb = (EPI == EPI_WGRAD) ? kr.nkb : sg.nkb;
        for (int kb = 0; kb < nkb; ++kb) {
          int w = 1;
          if (lane == 0) {
            // with CTA pairs the stage is released by the first CTA's tensor-core commit
            w = ((CG == 2) ? mbar_wait_cluster(&empty[stage], phase ^ 1, abort_flag)
                           : mbar_wait(&empty[stage], phase ^ 1, abort_flag))
                    ? 1
                    : 0;
          }
          w = __shfl_sync(0xffffffffu, w, 0);
          if (!w) { ok = false; break; }
          uint8_t* sA = smem + stage * C::STAGE_BYTES;
          const int ka = (EPI == EPI_WGRAD) ? kr.k0 + kb * kBK : sg.a_k0 + kb * kBK;
          if constexpr (CG == 2) {
            // Both CTAs' copies complete on the first CTA's stage barrier, which expects the
            // bytes of both (every box is delivered whole: rows past the tensor are zeros).
            if (lane == 0) {
              const uint32_t fb = cluster_addr(&full[stage], 0);
              uint32_t bytes = C::A_SUB_BYTES;
              if (C::PAIR_JOIN) {
                bytes += NB * C::B_BYTES;
              } else {
#pragma unroll
                for (int b = 0; b < NB; ++b) bytes += (sg.b_map[b] >= 0) ? C::B_BYTES : 0;
              }
              if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * bytes);
              tma_load_3d_pair(sA, &P.maps[sg.a_map], fb, ka, tc.row0, 0, pol_a);
              if constexpr (C::PAIR_JOIN) {
                // this CTA stages operand `rank`; in a segment without it (the LoRA block of
                // the other projection) it stages zeros instead: a box wholly before row 0,
                // which TMA fills with zeros, so the MMA adds nothing to that half
                const bool has = sg.b_map[rank] >= 0;
                const int b = has ? rank : 1 - rank;
                const int z = (P.group_off != nullptr) ? tc.g : sg.b_z[b];
                tma_load_3d_pair(sA + C::A_BYTES, &P.maps[sg.b_map[b]], fb,
                                 sg.b_k0[b] + kb * kBK, has ? tc.n * BN : -BN, z, pol_b);
              } else {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                  if (sg.b_map[b] < 0) continue;
                  uint8_t* sB = sA + C::A_BYTES + b * C::B_BYTES;
                  const int kbk = sg.b_k0[b] + kb * kBK;
                  const int z = (P.group_off != nullptr) ? tc.g : sg.b_z[b];
                  const int n0 = tc.n * BN + rank * (BN / 2);  // this CTA's half of B
                  if (!B_MN) {
                    tma_load_3d_pair(sB, &P.maps[sg.b_map[b]], fb, kbk, n0, z, pol_b);
                  } else {
#pragma unroll
                    for (int c = 0; c < C::B_ROWS / 64; ++c)
                      tma_load_3d_pair(sB + c * 8192, &P.maps[sg.b_map[b]], fb, n0 + c * 64,
                                       kbk, z, pol_b);
                  }
                }
              }
            }
            __syncwarp();
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
            continue;
          }
          if (lane == 0) {
            const int nsub = (MSUB == 2 && tc.rows_valid > kBM) ? 2 : 1;
            uint32_t bytes = sg.a_gather ? 0u : nsub * C::A_SUB_BYTES;
#pragma unroll
            for (int b = 0; b < NB; ++b) bytes += (sg.b_map[b] >= 0) ? C::B_BYTES : 0;
            mbar_arrive_expect_tx(&full[stage], bytes);
          }
          if (lane == 0) {
            if (!A_MN) {
              if (!sg.a_gather) {
                tma_load_3d(sA, &P.maps[sg.a_map], &full[stage], ka, tc.row0, 0, pol_a);
                if (MSUB == 2 && tc.rows_valid > kBM)
                  tma_load_3d(sA + C::A_SUB_BYTES, &P.maps[sg.a_map], &full[stage], ka,
                              tc.row0 + kBM, 0, pol_a);
              }
            } else {
              tma_load_3d(sA, &P.maps[sg.a_map], &full[stage], tc.row0, ka, 0, pol_a);
              tma_load_3d(sA + 8192, &P.maps[sg.a_map], &full[stage], tc.row0 + 64, ka, 0,
                          pol_a);
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              if (sg.b_map[b] < 0) continue;
              uint8_t* sB = sA + C::A_BYTES + b * C::B_BYTES;
              const int kbk = (EPI == EPI_WGRAD) ? kr.k0 + kb * kBK : sg.b_k0[b] + kb * kBK;
              const int z = (EPI == EPI_WGRAD) ? 0 : ((P.group_off != nullptr) ? tc.g : sg.b_z[b]);
              if (!B_MN) {
                tma_load_3d(sB, &P.maps[sg.b_map[b]], &full[stage], kbk, tc.n * BN, z, pol_b);
              } else {
#pragma unroll
                for (int c = 0; c < (BN + 63) / 64; ++c)
                  tma_load_3d(sB + c * 8192, &P.maps[sg.b_map[b]], &full[stage],
                              tc.n * BN + c * 64, kbk, z, pol_b);
              }
            }
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report_status(P.dev_status, MOE_ERR_TIMEOUT);
    }
  } else if (warp == 1 && (CG == 1 || rank == 0)) {
    // ------------------------------------------------------------ MMA issuer
    // (with CTA pairs only the first CTA issues: each M = 256 MMA covers both CTAs' rows)
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, A_MN, B_MN);
    // Two B operands sit back to back in the stage (K-major: the second's rows follow the
    // first's BN rows; MN-major: its 64-wide boxes follow the first's, 8 KB apart), so when
    // both are enabled one MMA of N = 2*BN covers both accumulators (columns [0, BN) and
    // [BN, 2*BN)), halving the MMA count.
    constexpr bool kJoinB = (NB == 2) && !C::SUMB && (2 * BN <= 256) && (!B_MN || BN % 64 == 0);
    constexpr uint32_t idesc2 = idesc_bf16_f32(kBM, kJoinB ? 2 * BN : BN, A_MN, B_MN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    TileCoord tc;
    KRange kr;
    for (int tile = unit0; ok && next_tile<EPI, MSUB, CG>(P, tile, rank, tc, kr); tile += unit_step) {
      int w = 1;
      if (lane == 0) {
        w = ((CG == 2) ? mbar_wait_cluster(&acc_empty[acc], acc_phase ^ 1, abort_flag)
                       : mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag))
                ? 1
                : 0;
      }
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_base = tmem_base + acc * C::ACC_COLS;
      // segment 0 writes every accumulator of the tile first (later segments add to them)
      const int nseg = (EPI == EPI_WGRAD) ? 1 : P.nseg;
      for (int s = 0; ok && s < nseg; ++s) {
        const GemmSeg& sg = P.seg[s];
        const int nkb = (EPI == EPI_WGRAD) ? kr.nkb : sg.nkb;
        for (int kb = 0; kb < nkb; ++kb) {
          if (lane == 0) {
            w = ((CG == 2) ? mbar_wait_cluster(&full[stage], phase, abort_flag)
                           : mbar_wait(&full[stage], phase, abort_flag))
                    ? 1
                    : 0;
          }
          w = __shfl_sync(0xffffffffu, w, 0);
          if (!w) { ok = false; break; }
          tc_fence_after();
          int ksteps = kBK / 16;  // 16-deep MMA steps of this k block
          if constexpr (EPI == EPI_WGRAD) {
            // rows past the group's end (the next group's rows, or memory never written)
            // must contribute nothing: the k block's MMA steps stop at the first 16-row step
            // boundary past them, and the rows in between are zeroed in both operands
            const int valid = min(kBK, kr.nrows - kb * kBK);
            ksteps = (valid + 15) / 16;
            const int end = 16 * ksteps;
            if (valid < end) {
              uint8_t* sA = smem + stage * C::STAGE_BYTES;
              zero_k_tail(sA, 2, valid, end, lane);
#pragma unroll
              for (int b = 0; b < NB; ++b)
                if (sg.b_map[b] >= 0)
                  zero_k_tail(sA + C::A_BYTES + b * C::B_BYTES, (BN + 63) / 64, valid, end, lane);
              fence_proxy_async_smem();
              __syncwarp();
            }
          }
          if constexpr (CG == 2) {
            if (lane == 0) {
              // M = 256 over the pair: A rows and B halves at the same offsets in both CTAs
              constexpr uint32_t idp = idesc_bf16_f32(2 * kBM, C::PAIR_JOIN ? 2 * BN : BN, false, B_MN);
              const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k) {
                const uint32_t accumulate = (s > 0 || kb > 0 || k > 0) ? 1u : 0u;
                const uint64_t adesc = smem_desc_sw128(a_addr + k * 32, 16, 1024);
                if constexpr (C::PAIR_JOIN) {
                  const uint64_t bdesc = smem_desc_sw128(a_addr + C::A_BYTES + k * 32, 16, 1024);
                  umma_bf16<2>(d_base, adesc, bdesc, idp, accumulate);
                } else {
#pragma unroll
                  for (int b = 0; b < NB; ++b) {
                    if (sg.b_map[b] < 0) continue;
                    const uint32_t b_addr = a_addr + C::A_BYTES + b * C::B_BYTES;
                    const uint64_t bdesc = B_MN ? smem_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                                : smem_desc_sw128(b_addr + k * 32, 16, 1024);
                    if constexpr (C::SUMB) {
                      // the router's lo weight part adds to what the hi part wrote
                      umma_bf16<2>(d_base, adesc, bdesc, idp, (accumulate || b > 0) ? 1u : 0u);
                    } else {
                      umma_bf16<2>(d_base + b * BN, adesc, bdesc, idp, accumulate);
                    }
                  }
                }
              }
              umma_commit<2>(&empty[stage]);
            }
          } else if (lane == 0) {
            const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
            const int nsub = (MSUB == 2 && tc.rows_valid > kBM) ? 2 : 1;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              if (k >= ksteps) break;
              const uint32_t accumulate = (s > 0 || kb > 0 || k > 0) ? 1u : 0u;
#pragma unroll
              for (int sub = 0; sub < MSUB; ++sub) {
                if (sub >= nsub) break;
                const uint32_t as = a_addr + sub * C::A_SUB_BYTES;
                const uint64_t adesc = A_MN ? smem_desc_sw128(as + k * 2048, 8192, 1024)
                                            : smem_desc_sw128(as + k * 32, 16, 1024);
                const uint32_t d_sub = d_base + sub * C::ACC_NB * BN;
                if (kJoinB && sg.b_map[0] >= 0 && sg.b_map[1] >= 0) {
                  const uint32_t b_addr = a_addr + C::A_BYTES;
                  const uint64_t bdesc = B_MN ? smem_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                              : smem_desc_sw128(b_addr + k * 32, 16, 1024);
                  umma_bf16(d_sub, adesc, bdesc, idesc2, accumulate);
                  continue;
                }
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                  if (sg.b_map[b] < 0) continue;
                  const uint32_t b_addr = a_addr + C::A_BYTES + b * C::B_BYTES;
                  const uint64_t bdesc = B_MN ? smem_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                              : smem_desc_sw128(b_addr + k * 32, 16, 1024);
                  if constexpr (C::SUMB) {
                    // the second B adds to what the first wrote in this k step
                    umma_bf16(d_sub, adesc, bdesc, idesc, (accumulate || b > 0) ? 1u : 0u);
                  } else {
                    umma_bf16(d_sub + b * BN, adesc, bdesc, idesc, accumulate);
                  }
                }
              }
            }
            umma_commit(&empty[stage]);
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit<CG>(&acc_full[acc]);
      __syncwarp();
      if (++acc == C::NACC) { acc = 0; acc_phase ^= 1; }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report_status(P.dev_status, MOE_ERR_TIMEOUT);
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ A-row gather
    // Only with a gathered A operand.  The two warps take alternate k blocks: each fills the
    // 128 x 64 A tile of its stage with 16-byte cp.async copies of token rows (zero fill for
    // rows past the group's end) in the 128-byte-swizzled layout TMA would produce, waits for
    // them, makes them visible to the tensor core (proxy fence) and arrives on the stage.
    if constexpr (!A_MN && EPI != EPI_WGRAD && MSUB == 1 && CG == 1) {
      if (P.gather_slot != nullptr) {
        const int gw = warp - 2;
        const int part = lane & 7;      // 16-byte chunk of a 128-byte row this lane copies
        const int rsub = lane >> 3;     // rows rsub, rsub + 4, ..., rsub + 124
        const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(P.gather_src);
        int stage = 0;
        uint32_t phase = 0;
        int q = 0;  // k blocks walked so far (all segments, all tiles)
        bool ok = true;
        TileCoord tc;
        KRange kr;
        for (int tile = unit0; ok && next_tile<EPI, MSUB, CG>(P, tile, rank, tc, kr); tile += unit_step) {
          int trow[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int rl = rsub + 4 * j;
            int t = -1;
            if (rl < tc.rows_valid) {
              const int slot = __ldg(&P.gather_slot[tc.row0 + rl]);
              t = slot >= 0 ? slot / P.gather_k : -1;
              if (t >= P.gather_rows) t = -1;
            }
            trow[j] = t;
          }
          for (int s = 0; ok && s < P.nseg; ++s) {
            const GemmSeg& sg = P.seg[s];
            for (int kb = 0; kb < sg.nkb; ++kb, ++q) {
              if ((q & 1) == gw) {
                int w = 1;
                if (lane == 0) w = mbar_wait(&empty[stage], phase ^ 1, abort_flag) ? 1 : 0;
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w) { ok = false; break; }
                if (sg.a_gather) {
                  uint8_t* sA = smem + stage * C::STAGE_BYTES;
                  const int ka = sg.a_k0 + kb * kBK + part * 8;
#pragma unroll
                  for (int j = 0; j < 32; ++j) {
                    const int rl = rsub + 4 * j;
                    const int t = trow[j];
                    const __nv_bfloat16* g = src + static_cast<size_t>(t < 0 ? 0 : t) * P.gather_ld + ka;
                    cp_async_16(sA + rl * 128 + ((part ^ (rl & 7)) << 4), g, t < 0 ? 0u : 16u);
                  }
                  cp_async_wait_all();
                  fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[stage]);
              }
              if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
          }
        }
        if (!ok && lane == 0) {
          *abort_flag = 1;
          report_status(P.dev_status, MOE_ERR_TIMEOUT);
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r_local = q * 32 + lane;
    // this warp's staging buffer (after the barrier block; gate-scale and store epilogues)
    uint8_t* epi_buf = smem + STAGES * C::STAGE_BYTES + 256 + q * (32 * 128);
    (void)epi_buf;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    TileCoord tc;
    KRange kr;
    for (int tile = unit0; next_tile<EPI, MSUB, CG>(P, tile, rank, tc, kr); tile += unit_step) {
      int w = 1;
      if (lane == 0) {
        w = ((CG == 2) ? mbar_wait_cluster(&acc_full[acc], acc_phase, abort_flag)
                       : mbar_wait(&acc_full[acc], acc_phase, abort_flag))
                ? 1
                : 0;
      }
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) { ok = false; break; }
      tc_fence_after();
      for (int sub = 0; sub < MSUB; ++sub) {
      // a missing second subtile stores nothing
      if (tc.rows_valid <= sub * kBM) break;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             acc * C::ACC_COLS + sub * C::ACC_NB * BN;
      const bool valid = r_local + sub * kBM < tc.rows_valid;
      const long row = static_cast<long>(tc.row0) + sub * kBM + r_local;
      const int col0 = tc.n * BN;
      // staged stores: this warp's rows are row_w .. row_w + 31, the first wrows of them valid
      const long row_w = static_cast<long>(tc.row0) + sub * kBM + q * 32;
      const int wrows = max(0, min(32, tc.rows_valid - sub * kBM - q * 32));

      if constexpr (EPI == EPI_F32_BIAS) {
        float* out = reinterpret_cast<float*>(P.out0);
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          tmem_ld16(t_row + c, v);
          tmem_ld_wait();
          const int col = col0 + c;
          if (valid && col < P.N) {
            float* dst = out + row * P.ldo + col;
            if (col + 16 <= P.N && (P.ldo & 3) == 0) {
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                float4 o;
                o.x = v[i] + (P.bias ? __ldg(&P.bias[col + i]) : 0.f);
                o.y = v[i + 1] + (P.bias ? __ldg(&P.bias[col + i + 1]) : 0.f);
                o.z = v[i + 2] + (P.bias ? __ldg(&P.bias[col + i + 2]) : 0.f);
                o.w = v[i + 3] + (P.bias ? __ldg(&P.bias[col + i + 3]) : 0.f);
                *reinterpret_cast<float4*>(dst + i) = o;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (col + i < P.N) dst[i] = v[i] + (P.bias ? __ldg(&P.bias[col + i]) : 0.f);
            }
          }
        }
      } else if constexpr (EPI == EPI_ROUTE) {
        // The router logits (fp32, as EPI_F32_BIAS) and, for the merge kernel, each token
        // row's tile maximum and the keys of its 16 largest (logit, expert) pairs
        // ("Day-Level Adaptation ...", section 3.3: routing scoring and top-k selection in
        // one kernel).  Pass 1 keeps the 16 largest VALUES with sorting networks (each
        // 16-column chunk sorted, then merged into the running list: independent min/max
        // pairs, no data-dependent branches); pass 2 re-reads the accumulator and emits the
        // keys of the values above the 16th largest plus, of the values equal to it, the
        // lowest-indexed ones (the tie rule).
        float* out = reinterpret_cast<float*>(P.out0);
        float best[kRouteTileK];
#pragma unroll
        for (int q2 = 0; q2 < kRouteTileK; ++q2) best[q2] = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          tmem_ld16(t_row + c, v);
          tmem_ld_wait();
          const int col = col0 + c;
          if (P.bias) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (col + i < P.N) v[i] += __ldg(&P.bias[col + i]);
          }
          if (valid && col < P.N) {
            float* dst = out + row * P.ldo + col;
            if (col + 16 <= P.N && (P.ldo & 3) == 0) {
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (col + i < P.N) dst[i] = v[i];
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (col + i >= P.N) v[i] = -INFINITY;
            sort16_desc(v);
            merge16_desc(best, v);
          }
        }
        const float mx = best[0];
        const float tau = best[kRouteTileK - 1];
        int need_eq = 0;  // values equal to tau that belong to the tile's 16
#pragma unroll
        for (int q2 = 0; q2 < kRouteTileK; ++q2) need_eq += (best[q2] == tau) ? 1 : 0;
        uint64_t* cand = reinterpret_cast<uint64_t*>(P.out1) +
                         (static_cast<size_t>(row) * P.n_tiles + tc.n) * kRouteTileK;
        int pos = 0;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          tmem_ld16(t_row + c, v);
          tmem_ld_wait();
          const int col = col0 + c;
          if (valid && col < P.N) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (col + i < P.N) {
                const float x = v[i] + (P.bias ? __ldg(&P.bias[col + i]) : 0.f);
                const bool eq = (x == tau) && need_eq > 0;
                if ((x > tau || eq) && pos < kRouteTileK) {
                  cand[pos++] = sel_key(x, col + i);
                  need_eq -= eq ? 1 : 0;
                }
              }
            }
          }
        }
        if (valid) {
          for (; pos < kRouteTileK; ++pos) cand[pos] = 0ull;  // fewer than 16 columns
          reinterpret_cast<float*>(P.out2)[static_cast<size_t>(row) * P.n_tiles + tc.n] = mx;
        }
      } else if constexpr (EPI == EPI_SWIGLU) {
        __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(P.out0);
        __nv_bfloat16* sg = reinterpret_cast<__nv_bfloat16*>(P.out1);
        __nv_bfloat16* su = reinterpret_cast<__nv_bfloat16*>(P.out2);
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float g[16], u[16];
          tmem_ld16(t_row + c, g);
          tmem_ld16(t_row + BN + c, u);
          tmem_ld_wait();
          const int col = col0 + c;
          if (valid && col < P.N) {
            const long off = row * P.ldo + col;
            if (sg) store_bf16x16(sg + off, g, P.N - col);
            if (su) store_bf16x16(su + off, u, P.N - col);
            float hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) hv[i] = silu_f(g[i]) * u[i];
            store_bf16x16(h + off, hv, P.N - col);
          }
        }
      } else if constexpr (EPI == EPI_GATE_SCALE) {
        __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(P.out0);
        float gs = 0.f;
        if (valid) gs = __ldg(&P.gate[__ldg(&P.row_slot[row])]);
        static_assert(BN % 64 == 0, "gate-scale epilogue works in 64-column chunks");
#pragma unroll 1
        for (int c = 0; c < BN; c += 64) {
          float v[4][16];
#pragma unroll
          for (int j = 0; j < 4; ++j) tmem_ld16(t_row + c + 16 * j, v[j]);
          tmem_ld_wait();
          const int col = col0 + c;
          if (col < P.N) {  // warp-uniform
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
              w[i] = pack_bf16x2(v[i >> 3][2 * (i & 7)] * gs, v[i >> 3][2 * (i & 7) + 1] * gs);
            warp_store_rows<64>(epi_buf, w, lane, y + col, P.ldo, row_w, wrows, P.N - col);
          }
        }
        if (P.comb_cnt != nullptr) combine_finish(P, tc.n, row_w, wrows, lane);
      } else if constexpr (EPI == EPI_SCALE) {
#pragma unroll 1
        for (int b = 0; b < NB; ++b) {
          __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(b == 0 ? P.out0 : P.out1);
#pragma unroll 1
          for (int c = 0; c < BN; c += 16) {
            float v[16];
            tmem_ld16(t_row + b * BN + c, v);
            tmem_ld_wait();
            const int col = col0 + c;
            if (valid && o != nullptr && col < P.N) {
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] *= P.scale;
              store_bf16x16(o + row * P.ldo + col, v, P.N - col);
            }
          }
        }
      } else if constexpr (EPI == EPI_SWIGLU_BWD) {
        // acc0 = dh; saved a_g (in0), a_u (in1) -> da_g (out0), da_u (out1); with out2, also
        // this n-tile's part of <dh, h> (h = silu(a_g) a_u recomputed in fp32) per row: the
        // gate gradient <dy, o> = <dh, h> / gate (dh = gate dy W_d (+ LoRA) is linear in dy)
        const __nv_bfloat16* ag = reinterpret_cast<const __nv_bfloat16*>(P.in0);
        const __nv_bfloat16* au = reinterpret_cast<const __nv_bfloat16*>(P.in1);
        __nv_bfloat16* dag = reinterpret_cast<__nv_bfloat16*>(P.out0);
        __nv_bfloat16* dau = reinterpret_cast<__nv_bfloat16*>(P.out1);
        float hd = 0.f;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float dh[16];
          tmem_ld16(t_row + c, dh);
          tmem_ld_wait();
          const int col = col0 + c;
          if (valid && col < P.N) {
            const long off = row * P.ldo + col;
            float g[16], u[16], o1[16], o2[16];
            load_bf16x16(ag + off, g);
            load_bf16x16(au + off, u);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float sgm = 1.0f / (1.0f + __expf(-g[i]));
              o1[i] = dh[i] * u[i] * sgm * (1.0f + g[i] * (1.0f - sgm));
              o2[i] = dh[i] * g[i] * sgm;
              hd += o2[i] * u[i];
            }
            store_bf16x16(dag + off, o1, P.N - col);
            store_bf16x16(dau + off, o2, P.N - col);
          }
        }
        if (P.out2 && valid)
          reinterpret_cast<float*>(P.out2)[row * P.n_tiles + tc.n] = hd;
      } else if constexpr (EPI == EPI_WGRAD) {
        // fp32 gradient of group g: [M, N] (ld N) or transposed [N, M] (ld M)
        static_assert(BN % 32 == 0, "weight-gradient tiles are whole 32-column blocks");
#pragma unroll 1
        for (int b = 0; b < NB; ++b) {
          float* o = reinterpret_cast<float*>(b == 0 ? P.out0 : P.out1);
          if (o == nullptr) continue;
          float* base = o + static_cast<size_t>(tc.g) * P.M * P.N;
          if (P.out_transposed) {
            // [N, M]: for each column the warp's 32 rows are 32 consecutive floats
            const int m = tc.row0 + r_local;
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
              float v[16];
              if (kr.nkb > 0) {
                tmem_ld16(t_row + b * BN + c, v);
                tmem_ld_wait();
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
              }
              const int col = col0 + c;
              if (valid && col < P.N) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  if (col + i < P.N) base[static_cast<size_t>(col + i) * P.M + m] = v[i];
              }
            }
          } else {
            // [M, N]: each 32-column block of the warp's 32 rows is transposed across the warp
            // (lane = column), so that every row leaves as one store of up to 128 contiguous
            // bytes instead of 32 rows' pieces per store
            const int m_w = tc.row0 + q * 32;
#pragma unroll 1
            for (int cb = 0; cb < BN; cb += 32) {
              const int col = col0 + cb;
              if (col >= P.N) break;  // warp-uniform
              float v[32];
              if (kr.nkb > 0) {
                float v0[16], v1[16];
                tmem_ld16(t_row + b * BN + cb, v0);
                tmem_ld16(t_row + b * BN + cb + 16, v1);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  v[i] = v0[i];
                  v[16 + i] = v1[i];
                }
              } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.f;
              }
              warp_transpose32(v, lane);
              if (col + lane < P.N) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (m_w + j < P.M) base[static_cast<size_t>(m_w + j) * P.N + col + lane] = v[j];
              }
            }
          }
        }
      } else if constexpr (EPI == EPI_STORE) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(P.out0);
        static_assert(BN % 64 == 0, "store epilogue works in 64-column chunks");
#pragma unroll 1
        for (int c = 0; c < BN; c += 64) {
          float v[4][16];
#pragma unroll
          for (int j = 0; j < 4; ++j) tmem_ld16(t_row + c + 16 * j, v[j]);
          tmem_ld_wait();
          const int col = col0 + c;
          if (col < P.N) {  // warp-uniform
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
              w[i] = pack_bf16x2(v[i >> 3][2 * (i & 7)], v[i >> 3][2 * (i & 7) + 1]);
            warp_store_rows<64>(epi_buf, w, lane, o + col, P.ldo, row_w, wrows, P.N - col);
          }
        }
      }
      }  // subtiles
      tc_fence_before();
      if constexpr (CG == 2) {
        // the accumulator buffer is free for the pair's next tile once both CTAs' four
        // epilogue warps have read their rows
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(cluster_addr(&acc_empty[acc], 0));
      } else {
        mbar_arrive(&acc_empty[acc]);
      }
      if (++acc == C::NACC) { acc = 0; acc_phase ^= 1; }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report_status(P.dev_status, MOE_ERR_TIMEOUT);
    }
  }

  // All roles are done.  On the normal path every TMA load was consumed and every MMA was
  // waited for through acc_full.  After an abort, the MMA thread waits (bounded) for its
  // own tcgen05 ops and thread 0 gives in-flight TMA copies a bounded grace period, so
  // nothing lands in shared memory or TMEM after the CTA has released them.
  __syncthreads();
  if constexpr (CG == 2) {
    // The pair's MMAs write both CTAs' TMEM: the first CTA waits (bounded) for all of them
    // before either CTA passes the pair barrier and frees its columns.  The barrier also
    // keeps both CTAs alive until every signal one sends the other has landed.
    if (rank == 0 && threadIdx.x == 32) {
      umma_commit_pair_local(drain);
      mbar_wait(drain, 0, reinterpret_cast<volatile int*>(&zero_flag));
    }
  } else {
    if (*abort_flag && threadIdx.x == 32) {
      umma_commit(drain);
      mbar_wait(drain, 0, reinterpret_cast<volatile int*>(&zero_flag));
    }
  }
  if (*abort_flag && threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
  }
  tc_fence_before();
  if constexpr (CG == 2) {
    cluster_sync();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
  }
}

// ctas_per_sm > 1 only for instantiations whose ring and TMEM both fit that many times on an
// SM (shared memory <= 227 KB / ctas_per_sm, TMEM columns <= 512 / ctas_per_sm), so that no
// CTA can wait on another's TMEM allocation.  CG = 2 launches clusters of two CTAs (one per
// SM of a pair of SMs), as many as can be resident at once.
template <int BN, int NB, bool A_MN, bool B_MN, int EPI, int STAGES, int CTAS_PER_SM = 1,
          int MSUB = 1, int CG = 1>
int launch_gemm(const GemmParams& P, cudaStream_t stream) {
  using C = GemmCfg<BN, NB, A_MN, B_MN, EPI, STAGES, MSUB, CTAS_PER_SM, CG>;
  static_assert(CTAS_PER_SM * C::TMEM_COLS <= 512, "TMEM of co-resident CTAs");
  static_assert(CTAS_PER_SM * (C::SMEM_BYTES + 1024) <= 232448, "shared memory per SM");
  static_assert(CTAS_PER_SM > 1 || C::SMEM_BYTES > 232448 / 2,
                "a single-CTA ring must be large enough to keep a second CTA off the SM");
  auto kern = gemm_kernel<BN, NB, A_MN, B_MN, EPI, STAGES, MSUB, CTAS_PER_SM, CG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return static_cast<int>(e);
  if constexpr (CG == 1) {
    kern<<<CTAS_PER_SM * num_sms(), 256, C::SMEM_BYTES, stream>>>(P);
    return static_cast<int>(cudaGetLastError());
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static int pairs_cache[64] = {0};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    int pairs = (dev >= 0 && dev < 64) ? pairs_cache[dev] : 0;
    if (pairs <= 0) {
      cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
      e = cudaOccupancyMaxActiveClusters(&pairs, kern, &cfg);
      if (e != cudaSuccess) return static_cast<int>(e);
      if (pairs <= 0) return static_cast<int>(cudaErrorInvalidConfiguration);
      pairs = min(pairs, num_sms() / 2);
      if (dev >= 0 && dev < 64) pairs_cache[dev] = pairs;
    }
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    e = cudaLaunchKernelEx(&cfg, kern, P);
    if (e != cudaSuccess) return static_cast<int>(e);
    return static_cast<int>(cudaGetLastError());
  }
}

}  // namespace moe

// Chunked gated delta-rule linear attention, forward and backward (declared in
// include/linear_attention.h).
//
// "Fine-Tuning Trillion-Parameter Sparse MoE Models: Challenges and Engineering Practices",
// section 5: normalization coefficients, gating and decay, intra-chunk query-state
// interaction and the output in fused kernels; fixed chunks with dense intra-chunk products
// and one small state recurrence between chunks.  Per sequence and head (q^, k^ L2-normed,
// alpha = exp(g)):
//     S_t = alpha_t S_{t-1} (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T,  o_t = scale S_t q^_t
//
// Chunked form (derived for this kernel).  In a chunk of C tokens with cumulative log decay
// G_i = g_1 + ... + g_i, gamma_i = exp(G_i) and state S0 at its start, let
// Gam_ij = exp(G_i - G_j) (<= 1 for j <= i).  The rows w_i = beta_i (v_i - gamma_i S0 k^_i -
// sum_{j<i} Gam_ij (k^_j . k^_i) w_j) solve
//     A W = diag(beta) V - diag(beta gamma) K^ S0^T,   A = I + tril(diag(beta)(Gam . K^K^T), -1)
// so W = U - Y S0^T with U = A^-1 diag(beta) V and Y = A^-1 diag(beta gamma) K^, and
//     O   = scale (diag(gamma) Q^ S0^T + (Gam . tril(Q^ K^T)) W)
//     S_C = gamma_C S0 + sum_j exp(G_C - G_j) w_j k^_j^T.
// U, Y and the masked Q^K^T depend only on the chunk, so they are computed for every chunk
// at once (gdr_chunk_kernel); what needs the running state is a short scan over chunks, and
// since each value row of the state evolves on its own (row r of S_t only involves v_t[r]),
// the scan is split over slices of RS value rows (gdr_scan_tc_kernel), so a few heads still
// fill the GPU.  Everything after the bf16 inputs is fp32 (the state in particular); the
// dense products of the chunk factors and of both scans run on the tensor cores with each
// fp32 operand carried as two bf16 pieces and fp32 accumulation, the masks, decays, the
// triangular inverse and the chunk-local backward on the fp32 pipes.
#include <cuda_bf16.h>
#include <math.h>

#include "../../include/linear_attention.h"
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kC = 64;    // chunk length
constexpr int kRS = 16;   // value rows of the state per scan CTA

__device__ __forceinline__ float bf(const __nv_bfloat16 v) { return __bfloat162float(v); }

// Byte offset of bf16 element (row, col) of a K-major [rows][64] block in the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_off(int row, int col) {
  return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 +
                               ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}

__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& mid) {
  hi = __float2bfloat16_rn(x);
  mid = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// Two bf16 pieces of 8 values scaled by `scale` (hi = bf16(scale x), mid = bf16(scale x - hi)),
// packed in element order as 16-byte pieces.
__device__ __forceinline__ void split8(const float (&f)[8], float scale, uint4& hi, uint4& mid) {
  uint32_t hw[4], mw[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float a = scale * f[2 * u], b = scale * f[2 * u + 1];
    const __nv_bfloat162 hb = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(hb);
    const __nv_bfloat162 mb = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hw[u] = *reinterpret_cast<const uint32_t*>(&hb);
    mw[u] = *reinterpret_cast<const uint32_t*>(&mb);
  }
  hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  mid = make_uint4(mw[0], mw[1], mw[2], mw[3]);
}

__device__ int g_gdr_status;  // first error a linear-attention kernel reported (0: none)

__device__ __forceinline__ void gdr_report(int code) { atomicCAS(&g_gdr_status, 0, code); }

// Contiguous global -> shared bulk copy (the TMA unit, no tensor map), completing `bytes` of
// transaction count on `bar`.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 bits, 4 consecutive columns: thread i of the warp gets lane (base + i).
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory image of one CTA of the tensor-core backward scan (gdr_bwd_scan_tc_kernel);
// the backward's gdr_chunk_kernel writes the tiles marked "image" exactly as they sit here.
// Tiles of chunk c in the order the scan meets them (c descending):
//   X (two buffers): sP (s P, both pieces; read as the MN-major A of P^T), sQ (s gamma Q^,
//       both pieces, MN-major A of its transpose) and dO^T of the slice (bf16, K-major B);
//   E (two buffers): E = diag(gamma_C / gamma) K^ (both pieces, K-major A) and the decays;
//   Y (one buffer, both pieces, MN-major A of Y^T).
template <int DK>
struct TcBwd {
  static constexpr int NKB = DK / 64;
  static constexpr uint32_t SP_PIECE = 8192u;                // [64 t][64 i]
  static constexpr uint32_t SQ_PIECE = NKB * 8192u;          // [64 j][64 dk] per box
  static constexpr uint32_t OT_BYTES = 2048u;                // [16 n][64 t]
  static constexpr uint32_t X_SP = 0, X_SQ = 2 * SP_PIECE, X_OT = X_SQ + 2 * SQ_PIECE;
  static constexpr uint32_t X_BYTES = X_OT + 1024u * ((OT_BYTES + 1023u) / 1024u);
  static constexpr uint32_t E_PIECE = NKB * 8192u;           // [64 i][64 dk] per block
  static constexpr uint32_t E_BYTES = 2 * E_PIECE;
  static constexpr uint32_t Y_PIECE = NKB * 8192u;
  static constexpr uint32_t Y_BYTES = 2 * Y_PIECE;
  static constexpr uint32_t B1_KB = 4096u;                   // dS pieces: [32][64] per block
  static constexpr uint32_t B2_BYTES = 4096u;                // -dW pieces: [32][64 tokens]
  static constexpr uint32_t MID_ROWS = 2048u;
  static constexpr uint32_t G_BYTES = kC * 4u;
  static constexpr uint32_t OFF_X = 0;                       // two buffers
  static constexpr uint32_t OFF_E = 2 * X_BYTES;             // two buffers
  static constexpr uint32_t OFF_Y = OFF_E + 2 * E_BYTES;
  static constexpr uint32_t OFF_B1 = OFF_Y + Y_BYTES;
  static constexpr uint32_t OFF_B2 = OFF_B1 + NKB * B1_KB;
  static constexpr uint32_t OFF_G = OFF_B2 + B2_BYTES;       // two buffers
  static constexpr uint32_t OFF_BAR = OFF_G + 2 * G_BYTES;   // 14 mbarriers, TMEM slot, flag
  static constexpr uint32_t BYTES = OFF_BAR + 128u;
  static constexpr size_t SMEM = BYTES + 1024u;
  static_assert(X_BYTES % 1024 == 0 && OFF_E % 1024 == 0 && OFF_Y % 1024 == 0 &&
                    OFF_B1 % 1024 == 0 && OFF_B2 % 1024 == 0,
                "swizzled tiles start on 1024-byte atoms");
  // M = 128 views read 8 KB past a 64-row tile (rows whose D lanes are not read): the last
  // E block, the last sP / sQ / Y box must be followed by 8 KB of shared memory
  static_assert(OFF_Y + Y_BYTES + 8192u <= BYTES, "views past Y stay in shared memory");
  static_assert(SMEM <= 227u * 1024u, "fits one CTA per SM");
  // bf16 element offsets within one chunk's images
  __device__ static uint32_t e(int s, int i, int x) {  // K-major [64][64] blocks
    return (s * E_PIECE + (x >> 6) * 8192u + sw128_off(i, x & 63)) >> 1;
  }
  __device__ static uint32_t mn(int s, int j, int x) {  // MN-major boxes (sQ, Y)
    return (s * SQ_PIECE + (x >> 6) * 8192u + sw128_off(j, x & 63)) >> 1;
  }
  __device__ static uint32_t sp(int s, int t, int i) { return (s * SP_PIECE + sw128_off(t, i)) >> 1; }
  __device__ static uint32_t ot(int n, int t) { return sw128_off(n, t) >> 1; }
};

// Barrier `id` over the first `nthreads` threads of the block; true if `pred` held in any.
__device__ __forceinline__ bool bar_sync_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbarrier.red.or.pred q, %2, %3, p;\n"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Sum of three accumulators 16 columns apart (columns taddr.., +16, +32), 4 columns each.
__device__ __forceinline__ void tmem_ld_sum3(uint32_t taddr, float (&d)[4]) {
  float a[4], b[4];
  tmem_ld4(taddr, d);
  tmem_ld4(taddr + 16, a);
  tmem_ld4(taddr + 32, b);
  tmem_ld_wait();
#pragma unroll
  for (int n = 0; n < 4; ++n) d[n] = (d[n] + a[n]) + b[n];
}

// Shared-memory image of one CTA of the tensor-core forward scan (gdr_scan_tc_kernel).  The
// forward's gdr_chunk_kernel writes the scan's chunk tiles exactly as they sit here (the
// 128-byte swizzle already applied: 16-byte piece p of a 128-byte row r at piece p ^ (r & 7),
// 8-row atoms of 1024 B), so that each tile moves with one bulk copy.  Every fp32 value of
// those tiles is carried as two bf16 pieces (hi, mid), each piece a tile of its own.
// 16 consumer warps: warp w reads TMEM lanes 32 (w % 4) .. + 31 (its quadrant) and handles
// value rows kTcCols (w / 4) .. + kTcCols - 1 of the slice, so each epilogue is spread over
// four warps per scheduler; warp 16 issues the bulk copies, warp 17 the MMAs (its lane 0),
// so that neither waits on the other or on an epilogue
constexpr int kTcThreads = 512;
constexpr int kTcCols = 4;
constexpr int kTcBlock = kTcThreads + 64;
constexpr int kTcSync = kTcThreads + 32;  // the consumer warps and the MMA warp

template <int DK>
struct TcScan {
  static constexpr int NKB = DK / 64;                        // 64-wide blocks of a dk row
  static constexpr uint32_t A1_SPLIT = NKB * 16384u;         // [Y; gamma Q^]: [128][64] per block
  static constexpr uint32_t A1_BYTES = 2 * A1_SPLIT;
  static constexpr uint32_t A3_SPLIT = NKB * 8192u;          // K^: [64 tokens][64 dk] per box
  static constexpr uint32_t A3_BYTES = 2 * A3_SPLIT;
  static constexpr uint32_t P_SPLIT = 8192u;                 // P: [64][64]
  static constexpr uint32_t P_BYTES = 2 * P_SPLIT;
  // B operands hold both pieces as one [32][64] K-major block (rows 0..15 hi, 16..31 mid):
  // one N = 32 MMA takes hi.hi and hi.mid from a single read of the A tile
  static constexpr uint32_t B1_KB = 4096u;                   // S slice: per 64-wide dk block
  static constexpr uint32_t B1_BYTES = NKB * B1_KB;
  static constexpr uint32_t BW_BYTES = 4096u;                // W, Wd: [32][64 tokens]
  static constexpr uint32_t MID_ROWS = 2048u;                // offset of the mid rows
  static constexpr uint32_t U_BYTES = kC * kRS * 4u;         // U slice [64][16] fp32
  static constexpr uint32_t G_BYTES = kC * 4u;               // log decays [64] fp32
  static constexpr uint32_t OFF_A1 = 0;                      // two buffers
  static constexpr uint32_t OFF_A3 = 2 * A1_BYTES;
  static constexpr uint32_t OFF_P = OFF_A3 + A3_BYTES;       // two buffers; 8 KB valid before
  static constexpr uint32_t OFF_B1 = OFF_P + 2 * P_BYTES;
  static constexpr uint32_t OFF_B2 = OFF_B1 + B1_BYTES;
  static constexpr uint32_t OFF_B3 = OFF_B2 + BW_BYTES;
  static constexpr uint32_t OFF_U = OFF_B3 + BW_BYTES;       // two buffers
  static constexpr uint32_t OFF_G = OFF_U + 2 * U_BYTES;     // two buffers
  static constexpr uint32_t OFF_BAR = OFF_G + 2 * G_BYTES;   // 12 mbarriers, TMEM slot, flag
  static constexpr uint32_t BYTES = OFF_BAR + 128u;
  static constexpr size_t SMEM = BYTES + 1024u;              // 1024-byte alignment slack
  static_assert(OFF_A3 % 1024 == 0 && OFF_P % 1024 == 0 && OFF_B1 % 1024 == 0 &&
                    OFF_B2 % 1024 == 0 && OFF_B3 % 1024 == 0 && OFF_U % 16 == 0,
                "swizzled tiles start on 1024-byte atoms");
  // the MN-major K^T operand reads a second 64-wide box 8 KB on even when dk = 64 (its rows
  // feed D3 lanes 64..127, which are not read): that box must lie in the buffer
  static_assert(OFF_A3 + A3_SPLIT + 16384u <= BYTES, "A3's second box stays in shared memory");
  static_assert(SMEM <= 227u * 1024u, "fits one CTA per SM");
  // bf16 element offsets within one chunk's image: piece s, row, column
  __device__ static uint32_t a1(int s, int m, int x) {
    return (s * A1_SPLIT + (x >> 6) * 16384u + sw128_off(m, x & 63)) >> 1;
  }
  __device__ static uint32_t a3(int s, int j, int x) {
    return (s * A3_SPLIT + (x >> 6) * 8192u + sw128_off(j, x & 63)) >> 1;
  }
  __device__ static uint32_t p(int s, int i, int j) {
    return (s * P_SPLIT + sw128_off(i, j)) >> 1;
  }
};

// Rows of the fp32 tiles in shared memory are padded to an odd stride, so that a warp
// reading one column of 32 rows touches 32 different banks.
template <int D>
struct Ld {
  static constexpr int v = D + 1;
};

// Shared memory of gdr_chunk_kernel (one CTA per 64-token chunk and head, two CTAs per SM).
// A1 holds, per bf16 piece and 64-wide dk block, a [128][64] K-major tile in the 128-byte
// swizzle: rows 0..63 K^, rows 64..127 Q^.  Its K^ rows serve three times: as rows of the
// A operand and as the K-major B operand of [K^; Q^] K^T, and (64-row boxes 16 KB apart) as
// the MN-major B operand of Y.  After [K^; Q^] K^T the Q^ halves of the first block of each
// piece hold the A operand of Y and then of U (A^-1 with its columns scaled, two pieces).
// The fp32 A used by the inverse later becomes the V image (the MN-major B operand of U).
template <int DK, int DV>
struct TcChunk {
  static constexpr int NKB = DK / 64;
  static constexpr uint32_t BLK = 16384u;
  static constexpr uint32_t OFF_A1 = 0;
  static constexpr uint32_t A1_BYTES = 2 * NKB * BLK;
  static constexpr uint32_t OFF_SA = A1_BYTES;               // fp32 A [64][65], then the V image
  static constexpr uint32_t SA_BYTES = 17408u;
  static constexpr uint32_t OFF_SI = OFF_SA + SA_BYTES;      // fp32 A^-1 [64][65]
  static constexpr uint32_t OFF_MISC = OFF_SI + 16640u;      // beta, G, beta * gamma [64] each
  static constexpr uint32_t OFF_BAR = OFF_MISC + 3 * kC * 4u;
  static constexpr uint32_t BYTES = OFF_BAR + 32u;
  static constexpr size_t SMEM = BYTES + 1024u;
  static constexpr uint32_t SLOT0 = OFF_A1 + 8192u;          // A operands of Y and U: hi
  static constexpr uint32_t SLOT1 = OFF_A1 + NKB * BLK + 8192u;  //                   mid
  static_assert(kC * (kC + 1) * 4u <= SA_BYTES && (DV / 64) * 8192u <= SA_BYTES,
                "A, then the V image, fit in their space");
  static_assert(SMEM + 1024u <= 114u * 1024u, "two CTAs per SM");
};

// Per chunk (grid: chunks x H x B, 256 threads): q^, k^, cumulative log decay, the WY
// factors U, Y, the masked P = Gam . tril(Q^ K^T) (diagonal included), all fp32 to the
// workspace.  Rows past the end of the sequence are zero (beta = g = 0: no effect).
// SPLIT (the forward): Y, gamma Q^, K^ and P go out instead as the tensor-core scan's
// shared-memory images (TcScan): each fp32 value as two bf16 pieces (hi, mid), per chunk
// YQs (rows 0..63 Y, 64..127 diag(gamma) Q^), Ks and Ps; U as fp32 slices of 16 value rows,
// [slice][64][16] per chunk; the log decays as fp32.
// BIMG (the backward): the fp32 factors as above plus the tensor-core backward scan's
// shared-memory images (TcBwd) of s P, s gamma Q^, E = diag(gamma_C / gamma) K^ and Y (two
// bf16 pieces each) and, per slice of 16 value rows, dO^T of the chunk (zero past the
// sequence).
//
// The three dense products run on the tensor cores with the two-piece bf16 operands of the
// scans (hi.hi + hi.mid + mid.hi, fp32 accumulation in TMEM): [K^; Q^] K^T (M = 128, N = 64,
// K = dk), then, after the triangular inverse (fp32, four threads per column),
// Y = (A^-1 diag(beta gamma)) K^ and U = (A^-1 diag(beta)) V (K = 64; V is bf16, so U takes
// two products).  The masks, decays, the inverse and every output conversion run on the
// fp32 pipes.
struct GdrBwdImages {
  __nv_bfloat16 *sP, *sQ, *E, *Y, *OT;
  float* KK;  // K^ K^T of the chunk, fp32 [64][64] (the tensor-core product, before masking)
  const __nv_bfloat16* dO;
  float scale;
};

template <int DK, int DV, bool SPLIT, bool BIMG>
__global__ void __launch_bounds__(256, 2) gdr_chunk_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const float* __restrict__ beta,
    const float* __restrict__ g, int T, int H, int nch, float* __restrict__ Y,
    float* __restrict__ U,
    float* __restrict__ Pm, float* __restrict__ Gc, float* __restrict__ Ai,
    __nv_bfloat16* __restrict__ YQs, __nv_bfloat16* __restrict__ Ks,
    __nv_bfloat16* __restrict__ Ps, GdrBwdImages img) {
  static_assert(!(SPLIT && BIMG), "one image set per launch");
  using L = TcChunk<DK, DV>;
  constexpr int NKB = L::NKB, LC = Ld<kC>::v;
  extern __shared__ uint8_t tc_smem_raw[];
  const uint32_t raw = smem_u32(tc_smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = tc_smem_raw + (sbase - raw);
  float* sA = reinterpret_cast<float*>(smem + L::OFF_SA);   // [C][LC]  A (unit lower)
  float* sI = reinterpret_cast<float*>(smem + L::OFF_SI);   // [C][LC]  A^-1
  float* sB = reinterpret_cast<float*>(smem + L::OFF_MISC);  // [C] beta
  float* sG = sB + kC;                                        // [C] cumulative log decay
  float* sBG = sG + kC;                                       // [C] beta * gamma
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 12);
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = c * kC;
  const size_t chunk_id = (static_cast<size_t>(b) * H + h) * nch + c;
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }

  // v rows: 16-byte loads issued first, held in registers until the V image is written (rows
  // past the sequence are zero)
  constexpr int VPR = DV / 8, VPER = kC * VPR / 256;  // 16-byte pieces per row / per thread
  uint4 va[VPER];
#pragma unroll
  for (int m = 0; m < VPER; ++m) {
    const int e = tid + 256 * m, i = e / VPR, pc = e - i * VPR;
    const int t = t0 + i;
    va[m] = t < T ? *reinterpret_cast<const uint4*>(
                        v + ((static_cast<size_t>(b) * T + t) * H + h) * DV + pc * 8)
                  : make_uint4(0u, 0u, 0u, 0u);
  }
  // beta and the cumulative log decay (warp 0, in token order)
  if (warp == 0) {
    float run = 0.f;
    for (int i0 = 0; i0 < kC; i0 += 32) {
      const int i = i0 + lane;
      const int t = t0 + i;
      const size_t o = (static_cast<size_t>(b) * T + t) * H + h;
      float gv = t < T ? g[o] : 0.f;
      const float bv = t < T ? beta[o] : 0.f;
#pragma unroll
      for (int s = 1; s < 32; s <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, gv, s);
        if (lane >= s) gv += y;
      }
      sB[i] = bv;
      sG[i] = run + gv;
      sBG[i] = bv * __expf(run + gv);
      run += __shfl_sync(0xffffffffu, gv, 31);
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // q, k rows, L2 normalised: a row's PPR 16-byte pieces sit in PPR consecutive threads, which
  // reduce its squared norm by shuffles; each piece of 8 values goes out whole (16-byte
  // stores) to the A1 operand and to every fp32 output and image this launch writes
  {
    constexpr int PPR = DK / 8, PER = kC * PPR / 256;
    static_assert(32 % PPR == 0 && PER * 256 == kC * PPR, "q/k tile loading");
    uint4 qa[PER], ka[PER];
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = tid + 256 * m, i = e / PPR, pc = e - i * PPR;
      const int t = t0 + i;
      const size_t o = ((static_cast<size_t>(b) * T + t) * H + h) * DK + pc * 8;
      qa[m] = t < T ? *reinterpret_cast<const uint4*>(q + o) : make_uint4(0u, 0u, 0u, 0u);
      ka[m] = t < T ? *reinterpret_cast<const uint4*>(k + o) : make_uint4(0u, 0u, 0u, 0u);
    }
    const float gC = sG[kC - 1];
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = tid + 256 * m, i = e / PPR, pc = e - i * PPR;
      const int x0 = pc * 8;
      float qf[8], kf[8];
      const uint32_t qw[4] = {qa[m].x, qa[m].y, qa[m].z, qa[m].w};
      const uint32_t kw[4] = {ka[m].x, ka[m].y, ka[m].z, ka[m].w};
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 a2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw[j]));
        const float2 b2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kw[j]));
        qf[2 * j] = a2.x; qf[2 * j + 1] = a2.y;
        kf[2 * j] = b2.x; kf[2 * j + 1] = b2.y;
        sq += a2.x * a2.x + a2.y * a2.y;
        sk += b2.x * b2.x + b2.y * b2.y;
      }
#pragma unroll
      for (int o = PPR / 2; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      const float iq = sq > 0.f ? 1.0f / sqrtf(sq) : 0.f;
      const float ik = sk > 0.f ? 1.0f / sqrtf(sk) : 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        qf[j] *= iq;
        kf[j] *= ik;
      }
      // the A1 operand: K^ row i, Q^ row 64 + i of block (piece, x0 / 64)
      uint4 hi, mid;
      split8(kf, 1.f, hi, mid);
      const uint32_t kb_off = (x0 >> 6) * L::BLK;
      *reinterpret_cast<uint4*>(smem + L::OFF_A1 + kb_off + sw128_off(i, x0 & 63)) = hi;
      *reinterpret_cast<uint4*>(smem + L::OFF_A1 + NKB * L::BLK + kb_off + sw128_off(i, x0 & 63)) = mid;
      split8(qf, 1.f, hi, mid);
      *reinterpret_cast<uint4*>(smem + L::OFF_A1 + kb_off + sw128_off(64 + i, x0 & 63)) = hi;
      *reinterpret_cast<uint4*>(smem + L::OFF_A1 + NKB * L::BLK + kb_off + sw128_off(64 + i, x0 & 63)) = mid;
      if constexpr (SPLIT) {  // gamma q^ (rows 64.. of YQs) and k^ images for the scan
        using LS = TcScan<DK>;
        __nv_bfloat16* yq = YQs + chunk_id * (LS::A1_BYTES / 2);
        __nv_bfloat16* ko = Ks + chunk_id * (LS::A3_BYTES / 2);
        split8(qf, __expf(sG[i]), hi, mid);
        *reinterpret_cast<uint4*>(yq + LS::a1(0, 64 + i, x0)) = hi;
        *reinterpret_cast<uint4*>(yq + LS::a1(1, 64 + i, x0)) = mid;
        split8(kf, 1.f, hi, mid);
        *reinterpret_cast<uint4*>(ko + LS::a3(0, i, x0)) = hi;
        *reinterpret_cast<uint4*>(ko + LS::a3(1, i, x0)) = mid;
      } else {
        if constexpr (BIMG) {  // s gamma q^ and E = (gamma_C / gamma) k^
          using LB = TcBwd<DK>;
          split8(qf, img.scale * __expf(sG[i]), hi, mid);
          *reinterpret_cast<uint4*>(img.sQ + chunk_id * LB::SQ_PIECE + LB::mn(0, i, x0)) = hi;
          *reinterpret_cast<uint4*>(img.sQ + chunk_id * LB::SQ_PIECE + LB::mn(1, i, x0)) = mid;
          split8(kf, __expf(gC - sG[i]), hi, mid);
          *reinterpret_cast<uint4*>(img.E + chunk_id * LB::E_PIECE + LB::e(0, i, x0)) = hi;
          *reinterpret_cast<uint4*>(img.E + chunk_id * LB::E_PIECE + LB::e(1, i, x0)) = mid;
        }
      }
    }
  }
  if constexpr (BIMG) {  // dO^T of every 16-row value slice: each thread gathers 8 tokens of
    // one value column (2-byte loads, the tile's rows shared through L1) into one 16-byte piece
    using LB = TcBwd<DK>;
    for (int e = tid; e < DV * (kC / 8); e += 256) {
      const int col = e % DV, tb = 8 * (e / DV);  // consecutive threads: consecutive columns
      uint32_t w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        __nv_bfloat16 p2[2];
#pragma unroll
        for (int v2 = 0; v2 < 2; ++v2) {
          const int tt = t0 + tb + 2 * u + v2;
          p2[v2] = tt < T ? img.dO[((static_cast<size_t>(b) * T + tt) * H + h) * DV + col]
                          : __float2bfloat16_rn(0.f);
        }
        w[u] = static_cast<uint32_t>(__bfloat16_as_ushort(p2[0])) |
               (static_cast<uint32_t>(__bfloat16_as_ushort(p2[1])) << 16);
      }
      *reinterpret_cast<uint4*>(img.OT + (chunk_id * (DV / kRS) + col / kRS) * (LB::OT_BYTES / 2) +
                                LB::ot(col % kRS, tb)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  bool failed = false;
  if (tid == 0) {  // D = [K^; Q^] K^T (columns 0..63)
    tc_fence_after();
    constexpr uint32_t kId = idesc_bf16_f32(128, 64, false, false);
    const uint64_t d0 = smem_desc_sw128(sbase + L::OFF_A1, 16, 1024);
#pragma unroll
    for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
          const uint32_t sa = pr == 2, sb = pr == 1;
          const uint64_t ad = d0 + (((sa * NKB + kb) * L::BLK + kk * 32) >> 4);
          const uint64_t bd = d0 + (((sb * NKB + kb) * L::BLK + kk * 32) >> 4);
          umma_bf16(tmem, ad, bd, kId, (kb | kk | pr) ? 1u : 0u);
        }
    umma_commit(bar);
  }
  // A (strictly lower part beta_i Gam_ij k^_i.k^_j, unit diagonal) into shared memory and
  // P (Gam_ij q^_i.k^_j, j <= i) out: warp w reads TMEM lanes 32 (w % 4).. (rows 0..63: A,
  // 64..127: P) and columns 32 (w / 4) .. + 31
  if (!mbar_wait(bar, 0, abort_flag)) failed = true;
  failed = __any_sync(0xffffffffu, failed);
  tc_fence_after();
  const int row = 32 * (warp & 3) + lane, j0 = 32 * (warp >> 2);
  if (!failed) {
    float d[32];
    {
      float d1[16];
      const uint32_t ta = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + j0;
      tmem_ld16(ta, d1);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) d[jj] = d1[jj];
      tmem_ld16(ta + 16, d1);
      tmem_ld_wait();
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) d[16 + jj] = d1[jj];
    }
    if (row < kC) {
      const int i = row;
      const float gi = sG[i], bi = sB[i];
      if constexpr (BIMG) {  // K^ K^T as it is, for the chunk-local backward
        float4* kko = reinterpret_cast<float4*>(img.KK + chunk_id * kC * kC + i * kC + j0);
#pragma unroll
        for (int p4 = 0; p4 < 8; ++p4)
          kko[p4] = make_float4(d[4 * p4], d[4 * p4 + 1], d[4 * p4 + 2], d[4 * p4 + 3]);
      }
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int j = j0 + jj;
        sA[i * LC + j] = j < i ? bi * __expf(gi - sG[j]) * d[jj] : (j == i ? 1.f : 0.f);
      }
    } else {
      const int i = row - kC;
      const float gi = sG[i];
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int j = j0 + jj;
        d[jj] = j <= i ? __expf(gi - sG[j]) * d[jj] : 0.f;
      }
      if constexpr (SPLIT) {
        using LS = TcScan<DK>;
        __nv_bfloat16* po = Ps + chunk_id * (LS::P_BYTES / 2);
#pragma unroll
        for (int p8 = 0; p8 < 4; ++p8) {
          uint4 hi, mid;
          split8(*reinterpret_cast<const float(*)[8]>(d + 8 * p8), 1.f, hi, mid);
          *reinterpret_cast<uint4*>(po + LS::p(0, i, j0 + 8 * p8)) = hi;
          *reinterpret_cast<uint4*>(po + LS::p(1, i, j0 + 8 * p8)) = mid;
        }
      } else {
        float4* pm = reinterpret_cast<float4*>(Pm + chunk_id * kC * kC + i * kC + j0);
#pragma unroll
        for (int p4 = 0; p4 < 8; ++p4)
          pm[p4] = make_float4(d[4 * p4], d[4 * p4 + 1], d[4 * p4 + 2], d[4 * p4 + 3]);
        if constexpr (BIMG) {
          using LB = TcBwd<DK>;
#pragma unroll
          for (int p8 = 0; p8 < 4; ++p8) {
            uint4 hi, mid;
            split8(*reinterpret_cast<const float(*)[8]>(d + 8 * p8), img.scale, hi, mid);
            *reinterpret_cast<uint4*>(img.sP + chunk_id * LB::SP_PIECE + LB::sp(0, i, j0 + 8 * p8)) = hi;
            *reinterpret_cast<uint4*>(img.sP + chunk_id * LB::SP_PIECE + LB::sp(1, i, j0 + 8 * p8)) = mid;
          }
        }
      }
    }
  }
  tc_fence_before();
  if (__syncthreads_or(failed)) failed = true;
  // X = A^-1 (A unit lower triangular) by 16 x 16 blocks.  The four diagonal blocks by
  // substitution, X_i = e_i - sum_{j<i} A_ij X_j within the block (16 steps; all blocks and
  // their 16 columns at once, four threads per column combining by shuffles; a column only
  // reads rows its own four lanes wrote, so the steps are ordered within the warp); the
  // blocks above the diagonal are zero; then the blocks below it by distance d = 1, 2, 3
  // from the diagonal (block indices, i - j = d):
  //     X_ij = -X_ii (sum_{k=j}^{i-1} A_ik X_kj)
  // each round fully parallel (the X_kj it reads are nearer the diagonal).
  if (!failed) {
    const int bb = tid >> 6, cc = (tid >> 2) & 15, part = tid & 3;
    const int jg = 16 * bb + cc;
    for (int r = 0; r < 16; ++r) {
      const int i = 16 * bb + r;
      float x = 0.f;
      for (int j = jg + part; j < i; j += 4) x -= sA[i * LC + j] * sI[j * LC + jg];
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      if (part == 0) sI[i * LC + jg] = r < cc ? 0.f : (r == cc ? 1.f : x);
      __syncwarp();
    }
    for (int e = tid; e < 6 * 256; e += 256) {  // blocks (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
      const int blk = e >> 8, w = e & 255;
      const int ib = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
      const int jb = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
      sI[(16 * ib + (w >> 4)) * LC + 16 * jb + (w & 15)] = 0.f;
    }
  }
  __syncthreads();
  if (!failed) {
    // sums of the current round: [3][16][16] fp32 over the Q^ rows of A1 (read by the first
    // MMAs only, which have completed)
    float* sT = reinterpret_cast<float*>(smem + L::OFF_A1 + 8192);
    for (int d = 1; d < 4; ++d) {
      const int np = 4 - d;  // block pairs (jb + d, jb), jb = 0 .. np - 1
      for (int e = tid; e < np * 256; e += 256) {
        const int pj = e >> 8, w = e & 255;
        const int i = 16 * (pj + d) + (w >> 4), jc = 16 * pj + (w & 15);
        float t = 0.f;
        for (int kk = 16 * pj; kk < 16 * (pj + d); ++kk) t += sA[i * LC + kk] * sI[kk * LC + jc];
        sT[e] = t;
      }
      __syncthreads();
      for (int e = tid; e < np * 256; e += 256) {
        const int pj = e >> 8, w = e & 255, ib = pj + d;
        const int i = 16 * ib + (w >> 4), cl = w & 15;
        float x = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) x -= sI[i * LC + 16 * ib + m] * sT[pj * 256 + m * 16 + cl];
        sI[i * LC + 16 * pj + cl] = x;
      }
      __syncthreads();
    }
  }
  __syncthreads();
  // the A operand of Y, A^-1 diag(beta gamma) (two pieces, K-major [64 i][64 j]), and the V
  // image (MN-major [64 j][dv] in 64-wide boxes) over A's space
  auto write_inverse_operand = [&](const float* colscale) {
    const int i = tid >> 2, jq = 16 * (tid & 3);
#pragma unroll
    for (int p8 = 0; p8 < 2; ++p8) {
      float f[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = jq + 8 * p8 + u;
        f[u] = sI[i * LC + j] * colscale[j];
      }
      uint4 hi, mid;
      split8(f, 1.f, hi, mid);
      *reinterpret_cast<uint4*>(smem + L::SLOT0 + sw128_off(i, jq + 8 * p8)) = hi;
      *reinterpret_cast<uint4*>(smem + L::SLOT1 + sw128_off(i, jq + 8 * p8)) = mid;
    }
  };
  if (!failed) {
    write_inverse_operand(sBG);
#pragma unroll
    for (int m = 0; m < VPER; ++m) {
      const int e = tid + 256 * m, j = e / VPR, pc = e - j * VPR;
      const int n = pc * 8;
      *reinterpret_cast<uint4*>(smem + L::OFF_SA + (n >> 6) * 8192 + sw128_off(j, n & 63)) = va[m];
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  const uint64_t dS0 = smem_desc_sw128(sbase + L::SLOT0, 16, 1024);
  const uint64_t dS1 = smem_desc_sw128(sbase + L::SLOT1, 16, 1024);
  if (tid == 0 && !failed) {  // Y = (A^-1 diag(beta gamma)) K^ (columns 0 .. dk - 1)
    tc_fence_after();
    constexpr uint32_t kIdY = idesc_bf16_f32(128, DK, false, true);
    const uint64_t dK = smem_desc_sw128(sbase + L::OFF_A1, L::BLK, 1024);  // MN-major boxes
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int pr = 0; pr < 3; ++pr) {
        const uint64_t ad = (pr == 2 ? dS1 : dS0) + ((kk * 32) >> 4);
        const uint64_t bd = dK + (((pr == 1 ? NKB * L::BLK : 0u) + kk * 2048) >> 4);
        umma_bf16(tmem, ad, bd, kIdY, (kk | pr) ? 1u : 0u);
      }
    umma_commit(bar);
  }
  if (!failed && !mbar_wait(bar, 1, abort_flag)) failed = true;
  // the A operand of U, A^-1 diag(beta), in the same places (Y's MMAs have read them)
  if (!failed) write_inverse_operand(sB);
  fence_proxy_async_smem();
  tc_fence_before();
  if (__syncthreads_or(failed)) failed = true;
  if (tid == 0 && !failed) {  // U = (A^-1 diag(beta)) V (columns dk .. dk + dv - 1)
    tc_fence_after();
    constexpr uint32_t kIdU = idesc_bf16_f32(128, DV, false, true);
    const uint64_t dV = smem_desc_sw128(sbase + L::OFF_SA, 8192, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int pr = 0; pr < 2; ++pr)
        umma_bf16(tmem + DK, (pr ? dS1 : dS0) + ((kk * 32) >> 4), dV + ((kk * 2048) >> 4), kIdU,
                  (kk | pr) ? 1u : 0u);
    umma_commit(bar);
  }
  // Y out (while U's MMAs run): rows i = TMEM lanes 0..63, dk columns split over two warps
  const bool yrows = (warp & 3) < 2;
  const uint32_t tl = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
  if (!failed && yrows) {
    const int i = row;
    constexpr int HX = DK / 2;
#pragma unroll 1
    for (int x0 = (warp >> 2) * HX; x0 < (warp >> 2) * HX + HX; x0 += 16) {
      float y[16];
      tmem_ld16(tl + x0, y);
      tmem_ld_wait();
#pragma unroll
      for (int p8 = 0; p8 < 2; ++p8) {
        const float(&f)[8] = *reinterpret_cast<const float(*)[8]>(y + 8 * p8);
        const int x = x0 + 8 * p8;
        uint4 hi, mid;
        if constexpr (SPLIT) {
          using LS = TcScan<DK>;
          __nv_bfloat16* yq = YQs + chunk_id * (LS::A1_BYTES / 2);
          split8(f, 1.f, hi, mid);
          *reinterpret_cast<uint4*>(yq + LS::a1(0, i, x)) = hi;
          *reinterpret_cast<uint4*>(yq + LS::a1(1, i, x)) = mid;
        } else {
          float4* yo = reinterpret_cast<float4*>(Y + chunk_id * kC * DK + i * DK + x);
          yo[0] = make_float4(f[0], f[1], f[2], f[3]);
          yo[1] = make_float4(f[4], f[5], f[6], f[7]);
          if constexpr (BIMG) {
            using LB = TcBwd<DK>;
            split8(f, 1.f, hi, mid);
            *reinterpret_cast<uint4*>(img.Y + chunk_id * LB::Y_PIECE + LB::mn(0, i, x)) = hi;
            *reinterpret_cast<uint4*>(img.Y + chunk_id * LB::Y_PIECE + LB::mn(1, i, x)) = mid;
          }
        }
      }
    }
  }
  if (!failed && !mbar_wait(bar, 0, abort_flag)) failed = true;  // U's MMAs (phase 2)
  failed = __any_sync(0xffffffffu, failed);
  tc_fence_after();
  if (!failed && yrows) {  // U out: rows i, dv columns split over two warps
    const int i = row;
    constexpr int HN = DV / 2;
#pragma unroll 1
    for (int n0 = (warp >> 2) * HN; n0 < (warp >> 2) * HN + HN; n0 += 16) {
      float u[16];
      tmem_ld16(tl + DK + n0, u);
      tmem_ld_wait();
      float4* uo;
      if constexpr (SPLIT)  // slice n0 / 16 of 16 value rows, row i
        uo = reinterpret_cast<float4*>(U + ((chunk_id * (DV / kRS) + n0 / kRS) * kC + i) * kRS);
      else
        uo = reinterpret_cast<float4*>(U + chunk_id * kC * DV + i * DV + n0);
#pragma unroll
      for (int p4 = 0; p4 < 4; ++p4)
        uo[p4] = make_float4(u[4 * p4], u[4 * p4 + 1], u[4 * p4 + 2], u[4 * p4 + 3]);
    }
  }
  static_assert(kRS == 16, "U slices are 16-column groups");
  if (tid < kC) Gc[chunk_id * kC + tid] = sG[tid];
  if (Ai && !failed)
    for (int e = tid; e < kC * kC; e += 256) Ai[chunk_id * kC * kC + e] = sI[(e / kC) * LC + (e % kC)];
  tc_fence_before();
  if (__syncthreads_or(failed) && tid == 0) gdr_report(MOE_ERR_TIMEOUT);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Scan over the chunks of one (b, h) for RS = 16 value rows of the state (grid: DV/RS x H x B,
// 16 consumer warps and a copy warp), on the tensor cores.  Per chunk, with S the slice of
// the chunk-start state:
//     D1 = [Y; diag(gamma) Q^] S^T                      (M = 128 token rows, N = 16, K = dk)
//     W  = U - D1[0:64],  Wd = diag(gamma_C / gamma) W
//     D3 = K^T Wd         ->  S^T = gamma_C S^T + D3     (M = dk, K = 64 tokens)
//     D1[64:128] += P W   ->  O = scale D1[64:128]       (K = 64 tokens)
// S_chunks (optional) receives the state at every chunk start (the backward's checkpoints).
//
// Each product is the three MMAs hi.hi + hi.mid + mid.hi of the operands' bf16 pieces,
// accumulated in fp32 in TMEM (about 16 significant bits per operand where one bf16 MMA
// keeps 8); the state and W are split by the threads that hold them.  TMEM lane x is row x
// of D3 (the state's column x, kept in registers across chunks) and row x of D1 (W's token
// row for x < 64, the output's row x - 64 above); the four warps reading a lane quadrant take
// four value rows each.  One staged [64 tokens][dk] tile of K^ serves as the MN-major A
// operand of K^T Wd (64-wide dk boxes 8 KB apart); a P tile is read as rows 64..127 of a
// 128-row A operand whose first 64 rows (the 8 KB before it) only feed D1 rows that W has
// already been read from.
//
// The chain from one chunk's state to the next is D1 -> W -> D3 -> S; P W and the output
// are off it: their MMAs are issued after K^T Wd, and D1 is double-buffered in TMEM so
// that the output rows of chunk c are read (by the warps of lane quadrants 2 and 3) while
// the warps of quadrants 0 and 1 form W of chunk c + 1.  The copy warp streams the chunk
// tiles through full / empty mbarrier pairs: [Y; gamma Q^] with the U slice and the log
// decays, and P, two buffers each; K^ one buffer, refilled as soon as K^T Wd completes.
template <int DK, int DV>
__global__ void __launch_bounds__(kTcBlock, 1) gdr_scan_tc_kernel(
    const __nv_bfloat16* __restrict__ YQs, const __nv_bfloat16* __restrict__ Ks,
    const __nv_bfloat16* __restrict__ Ps, const float* __restrict__ Us,
    const float* __restrict__ Gc, const float* __restrict__ S0, int T, int H, int nch,
    float scale, __nv_bfloat16* __restrict__ o, float* __restrict__ ST,
    float* __restrict__ Schk, float* __restrict__ Wout) {
  using L = TcScan<DK>;
  constexpr int NKB = L::NKB;
  extern __shared__ uint8_t tc_smem_raw[];
  const uint32_t raw = smem_u32(tc_smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = tc_smem_raw + (sbase - raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* d1_done = &bar[0];   // group 1 (and everything issued before it) complete
  uint64_t* d3_done = &bar[1];   // K^T Wd complete
  uint64_t* full_a = &bar[2];    // [2] [Y; gamma Q^], U slice, log decays landed
  uint64_t* full_k = &bar[4];    // K^ landed
  uint64_t* full_p = &bar[5];    // [2] P landed
  uint64_t* empty_a = &bar[7];   // [2] buffer a free (its chunk's W formed)
  uint64_t* empty_k = &bar[9];   // K^ free (K^T Wd complete)
  uint64_t* empty_p = &bar[10];  // [2] P buffer free (P W complete)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 96);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 100);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int x = 32 * (warp & 3) + (tid & 31);  // TMEM lane: token row of D1, dk column of D3
  const int n0 = kTcCols * ((warp >> 2) & 3);  // this thread's first value row of the slice
  const int r0 = blockIdx.x * kRS, h = blockIdx.y, b = blockIdx.z;
  const size_t bh = static_cast<size_t>(b) * H + h;
  static_assert(kTcCols * (kTcThreads / 128) == kRS, "four warps per quadrant cover the slice");

  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 12; ++i) mbar_init(&bar[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  // D1 buffers at columns 0 and 64 (each three accumulators of 16: hi.hi, hi.mid, mid.hi),
  // D3 at 128; summed when read
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_d3 = tmem + 128;
  bool failed = false;
  // copy warp: the last copy issued on each full barrier and the phase it completes (bits 0,
  // 1: full_a; 2: full_k; 3, 4: full_p), for the drain after an abort
  uint32_t sent = 0, par = 0;

  if (warp == kTcThreads / 32) {
    // ------------------------------------------------------------ copy warp
    if ((tid & 31) == 0) {
      auto note = [&](int i, uint32_t phase) {
        sent |= 1u << i;
        par = (par & ~(1u << i)) | (phase << i);
      };
      for (int c = 0; c < nch && !failed; ++c) {
        const int buf = c & 1;
        const uint32_t use = static_cast<uint32_t>(c >> 1);
        const size_t cid = bh * nch + c;
        if (c >= 2 && !mbar_wait(&empty_a[buf], (use - 1) & 1, abort_flag)) { failed = true; break; }
        mbar_arrive_expect_tx(&full_a[buf], L::A1_BYTES + L::U_BYTES + L::G_BYTES);
        bulk_load(smem + L::OFF_A1 + buf * L::A1_BYTES, YQs + cid * (L::A1_BYTES / 2),
                  L::A1_BYTES, &full_a[buf]);
        bulk_load(smem + L::OFF_U + buf * L::U_BYTES,
                  Us + (cid * (DV / kRS) + blockIdx.x) * (kC * kRS), L::U_BYTES, &full_a[buf]);
        bulk_load(smem + L::OFF_G + buf * L::G_BYTES, Gc + cid * kC, L::G_BYTES, &full_a[buf]);
        note(buf, use & 1);
        if (c >= 1 && !mbar_wait(empty_k, (c - 1) & 1, abort_flag)) { failed = true; break; }
        mbar_arrive_expect_tx(full_k, L::A3_BYTES);
        bulk_load(smem + L::OFF_A3, Ks + cid * (L::A3_BYTES / 2), L::A3_BYTES, full_k);
        note(2, c & 1);
        if (c >= 2 && !mbar_wait(&empty_p[buf], (use - 1) & 1, abort_flag)) { failed = true; break; }
        mbar_arrive_expect_tx(&full_p[buf], L::P_BYTES);
        bulk_load(smem + L::OFF_P + buf * L::P_BYTES, Ps + cid * (L::P_BYTES / 2), L::P_BYTES,
                  &full_p[buf]);
        note(3 + buf, use & 1);
      }
      if (failed) *abort_flag = 1;
    }
  } else if (warp == kTcThreads / 32 + 1) {
    // ------------------------------------------------------------ MMA warp (lane 0 issues)
    const bool issuer = (tid & 31) == 0;
    constexpr uint32_t kIdK32 = idesc_bf16_f32(128, 32, false, false);
    constexpr uint32_t kIdK16 = idesc_bf16_f32(128, 16, false, false);
    constexpr uint32_t kIdMN32 = idesc_bf16_f32(128, 32, true, false);
    constexpr uint32_t kIdMN16 = idesc_bf16_f32(128, 16, true, false);
    // descriptors of the operand tiles' first atoms; an operand further on adds its byte
    // offset / 16 (every address stays below 256 KB, so the 14-bit start field cannot carry)
    const uint64_t dA1 = smem_desc_sw128(sbase + L::OFF_A1, 16, 1024);
    const uint64_t dB1 = smem_desc_sw128(sbase + L::OFF_B1, 16, 1024);
    const uint64_t dP = smem_desc_sw128(sbase + L::OFF_P - 8192, 16, 1024);
    const uint64_t dB2 = smem_desc_sw128(sbase + L::OFF_B2, 16, 1024);
    const uint64_t dA3 = smem_desc_sw128(sbase + L::OFF_A3, 8192, 1024);
    const uint64_t dB3 = smem_desc_sw128(sbase + L::OFF_B3, 16, 1024);
    for (int c = 0; c < nch; ++c) {
      const int buf = c & 1;
      const uint32_t use = static_cast<uint32_t>(c >> 1);
      const uint32_t t_d1 = tmem + 64 * buf;
      if (issuer && !mbar_wait(&full_a[buf], use & 1, abort_flag)) failed = true;
      tc_fence_before();
      if (bar_sync_or(1, kTcSync, failed)) { failed = true; break; }  // B1 of this chunk
      if (issuer) {  // D1 = [Y; gamma Q^] S^T
        tc_fence_after();
        const uint64_t a0 = dA1 + ((buf * L::A1_BYTES) >> 4);
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (kb | k) ? 1u : 0u;
            const uint64_t bd = dB1 + ((kb * L::B1_KB + k * 32) >> 4);
            umma_bf16(t_d1, a0 + ((kb * 16384 + k * 32) >> 4), bd, kIdK32, acc);
            umma_bf16(t_d1 + 32, a0 + ((L::A1_SPLIT + kb * 16384 + k * 32) >> 4), bd, kIdK16, acc);
          }
        umma_commit(d1_done);
      }
      tc_fence_before();
      if (bar_sync_or(1, kTcSync, failed)) { failed = true; break; }  // W, Wd formed
      if (issuer) {
        mbar_arrive(&empty_a[buf]);  // [Y; gamma Q^], the U slice and the decays are read
        if (!mbar_wait(full_k, c & 1, abort_flag) || !mbar_wait(&full_p[buf], use & 1, abort_flag)) {
          failed = true;
          *abort_flag = 1;
        } else {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // D3 = K^T Wd
            const uint64_t bd3 = dB3 + ((k * 32) >> 4);
            umma_bf16(t_d3, dA3 + ((k * 2048) >> 4), bd3, kIdMN32, k ? 1u : 0u);
            umma_bf16(t_d3 + 32, dA3 + ((L::A3_SPLIT + k * 2048) >> 4), bd3, kIdMN16, k ? 1u : 0u);
          }
          umma_commit(d3_done);
          umma_commit(empty_k);
          const uint64_t p0 = dP + ((buf * L::P_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // D1[64:128] += P W
            const uint64_t bd2 = dB2 + ((k * 32) >> 4);
            umma_bf16(t_d1, p0 + ((k * 32) >> 4), bd2, kIdK32, 1u);
            umma_bf16(t_d1 + 32, p0 + ((L::P_SPLIT + k * 32) >> 4), bd2, kIdK16, 1u);
          }
          umma_commit(&empty_p[buf]);
        }
      }
    }
    if (failed) *abort_flag = 1;
    if (issuer && !failed) umma_commit(d1_done);  // the last chunk's P W (its output rows)
  } else {
    // ------------------------------------------------------------ consumer warps
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    // this thread's part of the state: column x for value rows n0 .. n0 + 3, in registers
    // across chunks
    const bool own_col = x < DK;
    float S[kTcCols];
#pragma unroll
    for (int n = 0; n < kTcCols; ++n)
      S[n] = (own_col && S0) ? S0[(bh * DV + r0 + n0 + n) * DK + x] : 0.f;
    auto write_state_operand = [&]() {  // S^T -> B1 (K-major [16 rows][dk], both pieces)
      if (own_col) {
        const int kb = x >> 6, col = x & 63;
#pragma unroll
        for (int n = 0; n < kTcCols; ++n) {
          __nv_bfloat16 hi, mid;
          split_bf16(S[n], hi, mid);
          const uint32_t off = L::OFF_B1 + kb * L::B1_KB + sw128_off(n0 + n, col);
          *reinterpret_cast<__nv_bfloat16*>(smem + off) = hi;
          *reinterpret_cast<__nv_bfloat16*>(smem + off + L::MID_ROWS) = mid;
        }
      }
    };
    auto out_epilogue = [&](int cc, uint32_t t_out) {  // output row x - 64 of chunk cc
      float d[kTcCols];
      tmem_ld_sum3(t_out + lane_base + n0, d);
      const int t = cc * kC + (x - 64);
      if (t < T) {
        uint2 pk;
        pk.x = pack_bf16x2(scale * d[0], scale * d[1]);
        pk.y = pack_bf16x2(scale * d[2], scale * d[3]);
        *reinterpret_cast<uint2*>(o + ((static_cast<size_t>(b) * T + t) * H + h) * DV + r0 + n0) =
            pk;
      }
    };
    write_state_operand();
    fence_proxy_async_smem();

    for (int c = 0; c < nch; ++c) {
      const int buf = c & 1;
      const uint32_t use = static_cast<uint32_t>(c >> 1);
      const size_t cid = bh * nch + c;
      const uint32_t t_d1 = tmem + 64 * buf;
      if (!mbar_wait(&full_a[buf], use & 1, abort_flag)) failed = true;
      tc_fence_before();
      // B1 holds this chunk's state; the previous chunk's TMEM reads are done
      if (bar_sync_or(1, kTcSync, failed)) { failed = true; break; }
      // the state at the chunk start (overlaps the MMAs)
      if (Schk && own_col) {
#pragma unroll
        for (int n = 0; n < kTcCols; ++n) Schk[(cid * DV + r0 + n0 + n) * DK + x] = S[n];
      }
      const float* sg = reinterpret_cast<const float*>(smem + L::OFF_G + buf * L::G_BYTES);
      const float gC = sg[kC - 1];
      const float gam_C = __expf(gC);
      if (!mbar_wait(d1_done, c & 1, abort_flag)) failed = true;
      failed = __any_sync(0xffffffffu, failed);  // the TMEM loads below are warp-collective
      tc_fence_after();
      if (!failed) {
        if ((warp & 3) < 2) {  // W and Wd for token row j = x, value rows n0..
          const int j = x;
          float d[kTcCols];
          tmem_ld_sum3(t_d1 + lane_base + n0, d);
          const float4 u4 = *reinterpret_cast<const float4*>(
              reinterpret_cast<const float*>(smem + L::OFF_U + buf * L::U_BYTES) + j * kRS + n0);
          const float uu[4] = {u4.x, u4.y, u4.z, u4.w};
          const float dec = __expf(gC - sg[j]);
          if (Wout)  // W for the backward
            *reinterpret_cast<float4*>(Wout + (cid * kC + j) * DV + r0 + n0) =
                make_float4(uu[0] - d[0], uu[1] - d[1], uu[2] - d[2], uu[3] - d[3]);
#pragma unroll
          for (int n = 0; n < kTcCols; ++n) {
            const float w = uu[n] - d[n];
            __nv_bfloat16 hi, mid;
            const uint32_t off = sw128_off(n0 + n, j);
            split_bf16(w, hi, mid);
            *reinterpret_cast<__nv_bfloat16*>(smem + L::OFF_B2 + off) = hi;
            *reinterpret_cast<__nv_bfloat16*>(smem + L::OFF_B2 + L::MID_ROWS + off) = mid;
            split_bf16(w * dec, hi, mid);
            *reinterpret_cast<__nv_bfloat16*>(smem + L::OFF_B3 + off) = hi;
            *reinterpret_cast<__nv_bfloat16*>(smem + L::OFF_B3 + L::MID_ROWS + off) = mid;
          }
        } else if (c > 0) {  // the previous chunk's output (its P W completed before D1)
          out_epilogue(c - 1, tmem + 64 * (buf ^ 1));
        }
      }
      if (failed) *abort_flag = 1;
      fence_proxy_async_smem();
      tc_fence_before();
      if (bar_sync_or(1, kTcSync, failed)) { failed = true; break; }  // W, Wd complete
      if (!mbar_wait(d3_done, c & 1, abort_flag)) failed = true;
      failed = __any_sync(0xffffffffu, failed);
      tc_fence_after();
      if (!failed && (DK == 128 || (warp & 3) < 2)) {  // column x: S^T = gamma_C S^T + K^T Wd
        float d[kTcCols];
        tmem_ld_sum3(t_d3 + lane_base + n0, d);
#pragma unroll
        for (int n = 0; n < kTcCols; ++n) S[n] = gam_C * S[n] + d[n];
        write_state_operand();
      }
      if (failed) *abort_flag = 1;
      fence_proxy_async_smem();
    }
    if (!failed) {  // the last chunk's output, once its P W completed (the MMA warp commits)
      if ((warp & 3) >= 2) {
        if (!mbar_wait(d1_done, nch & 1, abort_flag)) failed = true;
        failed = __any_sync(0xffffffffu, failed);
        tc_fence_after();
        if (!failed) out_epilogue(nch - 1, tmem + 64 * ((nch - 1) & 1));
      }
      if (failed) *abort_flag = 1;
    }
    if (failed) *abort_flag = 1;
    if (!failed && !*abort_flag && ST && own_col) {
#pragma unroll
      for (int n = 0; n < kTcCols; ++n) ST[(bh * DV + r0 + n0 + n) * DK + x] = S[n];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (tid == 0) gdr_report(MOE_ERR_TIMEOUT);
    if (tid == kTcThreads) {  // let the copies in flight land (bounded) before the CTA exits
      volatile int no_abort = 0;
      for (int i = 0; i < 5; ++i) {
        uint64_t* f = i < 2 ? &full_a[i] : (i == 2 ? full_k : &full_p[i - 3]);
        if (sent & (1u << i)) mbar_wait(f, (par >> i) & 1u, &no_abort);
      }
    }
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------- backward
//
// Gradients of <do, o> + <dS_T, S_T> (chunked form, derived for these kernels).  Per chunk,
// with dS1 the gradient of the state at the chunk's end:
//     dW  = s P^T dO + E dS1^T                       E = diag(gamma_C / gamma) K^
//     dS0 = gamma_C dS1 + s dO^T diag(gamma) Q^ - dW^T Y      (the state gradient one chunk
//                                                              earlier: a scan backwards)
// and then, locally in the chunk, with W = U - Y S0^T:
//     dP = s dO W^T (lower triangle)   dQ^ = (Gam . dP) K^ + s diag(gamma) dO S0
//     dK^ = (Gam . dP)^T Q^ + diag(gamma_C / gamma) W dS1 + diag(beta gamma) dBk + (Z + Z^T) K^
//     dBv = A^-T dW,  dBk = -A^-T dW S0,  dM = -(dBv U^T + dBk Y^T) (strictly lower)
//     dV = diag(beta) dBv,  Z = dM . beta Gam,  and the beta and log-decay gradients of every
//     place they enter (A, U, Y, P, E, gamma); dg is the reverse cumulative sum of dG.

// Backward scan over the chunks of one (b, h) for RS = 16 value rows of dS (grid: DV/RS x H x
// B, 16 consumer warps and a copy warp), on the tensor cores.  Chunks are taken last to
// first; with dS the slice of the state gradient at the chunk's end:
//     dW = (s P)^T dO + E dS^T                        (M = 64 tokens, N = 16)
//     dS = gamma_C dS + (s gamma Q^)^T dO - Y^T dW    (M = dk, K = 64 tokens)
// dW (fp32, for the chunk-local backward) and the state gradient at every chunk end go to
// global memory, dS0 at the end.  Operands and products as in the forward scan (two bf16
// pieces per fp32 operand, three MMAs per product; dO is bf16 already, so its products take
// two).  Only E dS^T and Y^T dW depend on the running state gradient: the two products with
// dO of chunk c - 1 are issued right after Y^T dW of chunk c, into the other of two TMEM
// buffers, and run while the state gradient of chunk c is formed.  TMEM: per buffer p, D_A
// (dW's five accumulators: E.dS hi.hi, hi.mid, mid.hi, sP.dO hi, mid) at columns 128 p and
// D_B (dS's: sQ.dO hi, mid, Y.dW hi.hi, hi.mid, mid.hi) at 256 + 128 p.
template <int DK, int DV>
__global__ void __launch_bounds__(kTcBlock, 1) gdr_bwd_scan_tc_kernel(
    const __nv_bfloat16* __restrict__ sPs, const __nv_bfloat16* __restrict__ sQs,
    const __nv_bfloat16* __restrict__ OTs, const __nv_bfloat16* __restrict__ Es,
    const __nv_bfloat16* __restrict__ Ys, const float* __restrict__ Gc,
    const float* __restrict__ dST, int H, int nch, float* __restrict__ dW,
    float* __restrict__ dSchk, float* __restrict__ dS0) {
  using L = TcBwd<DK>;
  constexpr int NKB = L::NKB;
  extern __shared__ uint8_t tc_smem_raw[];
  const uint32_t raw = smem_u32(tc_smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = tc_smem_raw + (sbase - raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* a_done = &bar[0];    // E dS^T (and everything issued before it) complete
  uint64_t* b_done = &bar[1];    // Y^T dW (and everything issued before it) complete
  uint64_t* full_x = &bar[2];    // [2] sP, sQ, dO^T landed
  uint64_t* full_e = &bar[4];    // [2] E, decays landed
  uint64_t* full_y = &bar[6];    // Y landed
  uint64_t* empty_x = &bar[7];   // [2] the products with dO complete
  uint64_t* empty_e = &bar[9];   // [2] E dS^T complete and the decays read
  uint64_t* empty_y = &bar[11];  // Y^T dW complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 112);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 116);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int x = 32 * (warp & 3) + (tid & 31);  // TMEM lane: token row of D_A, dk column of D_B
  const int n0 = kTcCols * ((warp >> 2) & 3);  // this thread's first value row of the slice
  const int r0 = blockIdx.x * kRS, h = blockIdx.y, b = blockIdx.z;
  const size_t bh = static_cast<size_t>(b) * H + h;

  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 12; ++i) mbar_init(&bar[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;
  // copy warp: the last copy issued on each full barrier and the phase it completes (bits 0,
  // 1: full_x; 2, 3: full_e; 4: full_y), for the drain after an abort
  uint32_t sent = 0, par = 0;

  if (warp == kTcThreads / 32) {
    // ------------------------------------------------------------ copy warp
    if ((tid & 31) == 0) {
      auto note = [&](int i, uint32_t phase) {
        sent |= 1u << i;
        par = (par & ~(1u << i)) | (phase << i);
      };
      for (int k = 0; k < nch && !failed; ++k) {  // k-th chunk met: c = nch - 1 - k
        const int buf = k & 1;
        const uint32_t use = static_cast<uint32_t>(k >> 1);
        const size_t cid = bh * nch + (nch - 1 - k);
        if (k >= 2 && !mbar_wait(&empty_x[buf], (use - 1) & 1, abort_flag)) { failed = true; break; }
        uint8_t* xb = smem + L::OFF_X + buf * L::X_BYTES;
        mbar_arrive_expect_tx(&full_x[buf], 2 * L::SP_PIECE + 2 * L::SQ_PIECE + L::OT_BYTES);
        bulk_load(xb + L::X_SP, sPs + cid * L::SP_PIECE, 2 * L::SP_PIECE, &full_x[buf]);
        bulk_load(xb + L::X_SQ, sQs + cid * L::SQ_PIECE, 2 * L::SQ_PIECE, &full_x[buf]);
        bulk_load(xb + L::X_OT, OTs + (cid * (DV / kRS) + blockIdx.x) * (L::OT_BYTES / 2),
                  L::OT_BYTES, &full_x[buf]);
        note(buf, use & 1);
        if (k >= 2 && !mbar_wait(&empty_e[buf], (use - 1) & 1, abort_flag)) { failed = true; break; }
        mbar_arrive_expect_tx(&full_e[buf], L::E_BYTES + L::G_BYTES);
        bulk_load(smem + L::OFF_E + buf * L::E_BYTES, Es + cid * L::E_PIECE, L::E_BYTES, &full_e[buf]);
        bulk_load(smem + L::OFF_G + buf * L::G_BYTES, Gc + cid * kC, L::G_BYTES, &full_e[buf]);
        note(2 + buf, use & 1);
        if (k >= 1 && !mbar_wait(empty_y, (k - 1) & 1, abort_flag)) { failed = true; break; }
        mbar_arrive_expect_tx(full_y, L::Y_BYTES);
        bulk_load(smem + L::OFF_Y, Ys + cid * L::Y_PIECE, L::Y_BYTES, full_y);
        note(4, k & 1);
      }
      if (failed) *abort_flag = 1;
    }
  } else if (warp == kTcThreads / 32 + 1) {
    // ------------------------------------------------------------ MMA warp (lane 0 issues)
    const bool issuer = (tid & 31) == 0;
    constexpr uint32_t kIdK32 = idesc_bf16_f32(128, 32, false, false);
    constexpr uint32_t kIdK16 = idesc_bf16_f32(128, 16, false, false);
    constexpr uint32_t kIdMN32 = idesc_bf16_f32(128, 32, true, false);
    constexpr uint32_t kIdMN16 = idesc_bf16_f32(128, 16, true, false);
    // descriptors of the tiles' first atoms; a tile further on adds its byte offset / 16
    const uint64_t dE = smem_desc_sw128(sbase + L::OFF_E, 16, 1024);
    const uint64_t dB1 = smem_desc_sw128(sbase + L::OFF_B1, 16, 1024);
    const uint64_t dSP = smem_desc_sw128(sbase + L::OFF_X + L::X_SP, 8192, 1024);
    const uint64_t dSQ = smem_desc_sw128(sbase + L::OFF_X + L::X_SQ, 8192, 1024);
    const uint64_t dOT = smem_desc_sw128(sbase + L::OFF_X + L::X_OT, 16, 1024);
    const uint64_t dY = smem_desc_sw128(sbase + L::OFF_Y, 8192, 1024);
    const uint64_t dB2 = smem_desc_sw128(sbase + L::OFF_B2, 16, 1024);
    // the products with dO of the k-th chunk met, into TMEM buffer k & 1
    auto issue_do_products = [&](int k) {
      const int xb = k & 1;
      if (!mbar_wait(&full_x[xb], (k >> 1) & 1, abort_flag)) return false;
      tc_fence_after();
      const uint32_t ta = tmem + 128 * xb, tb = tmem + 256 + 128 * xb;
      const uint32_t o = (xb * L::X_BYTES) >> 4;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bo = dOT + o + ((kk * 32) >> 4);
        const uint32_t acc = kk ? 1u : 0u;
        umma_bf16(ta + 48, dSP + o + ((kk * 2048) >> 4), bo, kIdMN16, acc);
        umma_bf16(ta + 64, dSP + o + ((L::SP_PIECE + kk * 2048) >> 4), bo, kIdMN16, acc);
        umma_bf16(tb, dSQ + o + ((kk * 2048) >> 4), bo, kIdMN16, acc);
        umma_bf16(tb + 16, dSQ + o + ((L::SQ_PIECE + kk * 2048) >> 4), bo, kIdMN16, acc);
      }
      umma_commit(&empty_x[xb]);
      return true;
    };
    if (issuer && !issue_do_products(0)) {
      failed = true;
      *abort_flag = 1;
    }
    for (int k = 0; k < nch; ++k) {
      const int buf = k & 1;
      const uint32_t use = static_cast<uint32_t>(k >> 1);
      const uint32_t t_a = tmem + 128 * buf, t_b = tmem + 256 + 128 * buf;
      if (issuer && !mbar_wait(&full_e[buf], use & 1, abort_flag)) failed = true;
      tc_fence_before();
      if (bar_sync_or(1, kTcSync, failed)) { failed = true; break; }  // B1 of this chunk
      if (issuer) {  // D_A += E dS^T
        tc_fence_after();
        const uint64_t e0 = dE + ((buf * L::E_BYTES) >> 4);
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (kb | kk) ? 1u : 0u;
            const uint64_t bd = dB1 + ((kb * L::B1_KB + kk * 32) >> 4);
            umma_bf16(t_a, e0 + ((kb * 8192 + kk * 32) >> 4), bd, kIdK32, acc);
            umma_bf16(t_a + 32, e0 + ((L::E_PIECE + kb * 8192 + kk * 32) >> 4), bd, kIdK16, acc);
          }
        umma_commit(a_done);
        umma_commit(&empty_e[buf]);  // the consumers read the decays before the barrier above
      }
      tc_fence_before();
      if (bar_sync_or(1, kTcSync, failed)) { failed = true; break; }  // -dW formed
      if (issuer) {
        if (!mbar_wait(full_y, k & 1, abort_flag)) {
          failed = true;
          *abort_flag = 1;
        } else {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // D_B += Y^T (-dW)
            const uint64_t bd = dB2 + ((kk * 32) >> 4);
            const uint32_t acc = kk ? 1u : 0u;
            umma_bf16(t_b + 32, dY + ((kk * 2048) >> 4), bd, kIdMN32, acc);
            umma_bf16(t_b + 64, dY + ((L::Y_PIECE + kk * 2048) >> 4), bd, kIdMN16, acc);
          }
          umma_commit(b_done);
          umma_commit(empty_y);
          if (k + 1 < nch && !issue_do_products(k + 1)) {
            failed = true;
            *abort_flag = 1;
          }
        }
      }
    }
    if (failed) *abort_flag = 1;
  } else {
    // ------------------------------------------------------------ consumer warps
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    // this thread's part of the state gradient: column x for value rows n0 .. n0 + 3
    const bool own_col = x < DK;
    float S[kTcCols];
#pragma unroll
    for (int n = 0; n < kTcCols; ++n)
      S[n] = (own_col && dST) ? dST[(bh * DV + r0 + n0 + n) * DK + x] : 0.f;
    auto write_state_operand = [&]() {  // dS -> B1 (K-major [16 rows][dk], both pieces)
      if (own_col) {
        const int kb = x >> 6, col = x & 63;
#pragma unroll
        for (int n = 0; n < kTcCols; ++n) {
          __nv_bfloat16 hi, mid;
          split_bf16(S[n], hi, mid);
          const uint32_t off = L::OFF_B1 + kb * L::B1_KB + sw128_off(n0 + n, col);
          *reinterpret_cast<__nv_bfloat16*>(smem + off) = hi;
          *reinterpret_cast<__nv_bfloat16*>(smem + off + L::MID_ROWS) = mid;
        }
      }
    };
    auto ld_sum5 = [&](uint32_t taddr, float (&d)[kTcCols]) {  // five accumulators, 16 apart
      float a[kTcCols], c2[kTcCols];
      tmem_ld4(taddr, d);
      tmem_ld4(taddr + 16, a);
      tmem_ld4(taddr + 32, c2);
      tmem_ld_wait();
#pragma unroll
      for (int n = 0; n < kTcCols; ++n) d[n] = (d[n] + a[n]) + c2[n];
      tmem_ld4(taddr + 48, a);
      tmem_ld4(taddr + 64, c2);
      tmem_ld_wait();
#pragma unroll
      for (int n = 0; n < kTcCols; ++n) d[n] += a[n] + c2[n];
    };
    write_state_operand();
    fence_proxy_async_smem();

    for (int k = 0; k < nch; ++k) {
      const int c = nch - 1 - k, buf = k & 1;
      const uint32_t use = static_cast<uint32_t>(k >> 1);
      const size_t cid = bh * nch + c;
      const uint32_t t_a = tmem + 128 * buf, t_b = tmem + 256 + 128 * buf;
      if (!mbar_wait(&full_e[buf], use & 1, abort_flag)) failed = true;
      const float gam_C = failed ? 0.f
          : __expf(reinterpret_cast<const float*>(smem + L::OFF_G + buf * L::G_BYTES)[kC - 1]);
      tc_fence_before();
      // B1 holds this chunk's state gradient; the previous chunk's TMEM reads are done
      if (bar_sync_or(1, kTcSync, failed)) { failed = true; break; }
      // the state gradient at the chunk's end (overlaps the MMAs)
      if (own_col) {
#pragma unroll
        for (int n = 0; n < kTcCols; ++n) dSchk[(cid * DV + r0 + n0 + n) * DK + x] = S[n];
      }
      if (!mbar_wait(a_done, k & 1, abort_flag)) failed = true;
      failed = __any_sync(0xffffffffu, failed);  // the TMEM loads below are warp-collective
      tc_fence_after();
      if (!failed && (warp & 3) < 2) {  // dW row i = x, value rows n0..
        const int i = x;
        float d[kTcCols];
        ld_sum5(t_a + lane_base + n0, d);
        *reinterpret_cast<float4*>(dW + (cid * kC + i) * DV + r0 + n0) =
            make_float4(d[0], d[1], d[2], d[3]);
#pragma unroll
        for (int n = 0; n < kTcCols; ++n) {
          __nv_bfloat16 hi, mid;
          const uint32_t off = L::OFF_B2 + sw128_off(n0 + n, i);
          split_bf16(-d[n], hi, mid);
          *reinterpret_cast<__nv_bfloat16*>(smem + off) = hi;
          *reinterpret_cast<__nv_bfloat16*>(smem + off + L::MID_ROWS) = mid;
        }
      }
      if (failed) *abort_flag = 1;
      fence_proxy_async_smem();
      tc_fence_before();
      if (bar_sync_or(1, kTcSync, failed)) { failed = true; break; }  // -dW complete
      if (!mbar_wait(b_done, k & 1, abort_flag)) failed = true;
      failed = __any_sync(0xffffffffu, failed);
      tc_fence_after();
      if (!failed && (DK == 128 || (warp & 3) < 2)) {  // column x: dS = gamma_C dS + D_B
        float d[kTcCols];
        ld_sum5(t_b + lane_base + n0, d);
#pragma unroll
        for (int n = 0; n < kTcCols; ++n) S[n] = gam_C * S[n] + d[n];
        write_state_operand();
      }
      if (failed) *abort_flag = 1;
      fence_proxy_async_smem();
    }
    if (failed) *abort_flag = 1;
    if (!failed && !*abort_flag && dS0 && own_col) {
#pragma unroll
      for (int n = 0; n < kTcCols; ++n) dS0[(bh * DV + r0 + n0 + n) * DK + x] = S[n];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (tid == 0) gdr_report(MOE_ERR_TIMEOUT);
    if (tid == kTcThreads) {  // let the copies in flight land (bounded) before the CTA exits
      volatile int no_abort = 0;
      for (int i = 0; i < 5; ++i) {
        uint64_t* f = i < 2 ? &full_x[i] : (i < 4 ? &full_e[i - 2] : full_y);
        if (sent & (1u << i)) mbar_wait(f, (par >> i) & 1u, &no_abort);
      }
    }
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


// Register-tiled products of the per-chunk backward, for 256 threads: thread (ti, tj) =
// (tid / 16, tid % 16) owns rows ti + 16 u (u < M / 16) and columns tj + 16 c (c < N / 16)
// of an M x N result and adds its sums to acc[u][c] (k ascending, one fp32 chain per output).
//   mm_nt4: A and B given by k-contiguous rows (shared or global, 16-byte aligned), read 16
//           bytes at a time
template <int M, int N, class FA, class FB>
__device__ __forceinline__ void mm_nt4(int K, FA Arow, FB Brow, float (&acc)[M / 16][N / 16]) {
  const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
  const float* ar[M / 16];
  const float* br[N / 16];
#pragma unroll
  for (int u = 0; u < M / 16; ++u) ar[u] = Arow(ti + 16 * u);
#pragma unroll
  for (int c = 0; c < N / 16; ++c) br[c] = Brow(tj + 16 * c);
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 a[M / 16], bb[N / 16];
#pragma unroll
    for (int u = 0; u < M / 16; ++u) a[u] = *reinterpret_cast<const float4*>(ar[u] + k);
#pragma unroll
    for (int c = 0; c < N / 16; ++c) bb[c] = *reinterpret_cast<const float4*>(br[c] + k);
#pragma unroll
    for (int u = 0; u < M / 16; ++u)
#pragma unroll
      for (int c = 0; c < N / 16; ++c)
        acc[u][c] += a[u].x * bb[c].x + a[u].y * bb[c].y + a[u].z * bb[c].z + a[u].w * bb[c].w;
  }
}

template <int M, int N>
__device__ __forceinline__ void mm_zero(float (&acc)[M / 16][N / 16]) {
#pragma unroll
  for (int u = 0; u < M / 16; ++u)
#pragma unroll
    for (int c = 0; c < N / 16; ++c) acc[u][c] = 0.f;
}

// 16 rows of a global matrix on their way to shared memory: each thread holds 16 N / 256
// elements in registers, so that the next block's loads are in flight while the current
// block is used.  Row kk, column n of the block is Bg[(k0 + kk) * ldb + n], or with TRANS
// Bg[n * ldb + k0 + kk] (consecutive threads read consecutive addresses either way).
template <int N, bool TRANS>
struct Stager {
  static constexpr int PER = 16 * N / 256;
  static_assert(PER * 256 == 16 * N, "whole elements per thread");
  float r[PER];
  __device__ __forceinline__ static void where(int e, int& kk, int& n) {
    if (TRANS) {
      n = e >> 4;
      kk = e & 15;
    } else {
      kk = e / N;
      n = e - kk * N;
    }
  }
  __device__ __forceinline__ void load(const float* __restrict__ Bg, int ldb, int k0) {
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      int kk, n;
      where(threadIdx.x + 256 * p, kk, n);
      r[p] = TRANS ? __ldg(&Bg[static_cast<size_t>(n) * ldb + k0 + kk])
                   : __ldg(&Bg[static_cast<size_t>(k0 + kk) * ldb + n]);
    }
  }
  __device__ __forceinline__ void store(float* stage) const {
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      int kk, n;
      where(threadIdx.x + 256 * p, kk, n);
      stage[kk * (N + 4) + n] = r[p];
    }
  }
};

// Float4 form of the products: thread (ti, tj) owns rows ti + 16 u and the four consecutive
// columns 64 g + 4 tj .. + 3 of every 64 (column c of the thread: bcol(tj, c)); A4(m, k)
// returns A(m, k .. k+3) and B4(k, n) returns B(k, n .. n+3) (k, n multiples of 4), so a k
// step costs one 16-byte read per row and per column group.
__device__ __forceinline__ int bcol(int tj, int c) { return (c >> 2) * 64 + 4 * tj + (c & 3); }

template <int M, int N, class FA4, class FB4>
__device__ __forceinline__ void mm_nn4(int K, FA4 A4, FB4 B4, float (&acc)[M / 16][N / 16]) {
  static_assert(N % 64 == 0, "four consecutive columns per lane, 64 per row group");
  constexpr int RA = M / 16, NG = N / 64;
  const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 a[RA];
#pragma unroll
    for (int u = 0; u < RA; ++u) a[u] = A4(ti + 16 * u, k);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      float4 bq[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) bq[g] = B4(k + kk, 64 * g + 4 * tj);
#pragma unroll
      for (int u = 0; u < RA; ++u) {
        const float av = kk == 0 ? a[u].x : kk == 1 ? a[u].y : kk == 2 ? a[u].z : a[u].w;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          acc[u][4 * g] += av * bq[g].x;
          acc[u][4 * g + 1] += av * bq[g].y;
          acc[u][4 * g + 2] += av * bq[g].z;
          acc[u][4 * g + 3] += av * bq[g].w;
        }
      }
    }
  }
}

// mm_nn4 with B in global memory, staged through shared memory 16 k rows at a time (every
// element read once by the CTA; the next block loads while the current one is used).
// stage: 16 x (N + 4) floats.  Every thread of the block must call it (it synchronises).
template <int M, int N, bool TRANS, class FA4>
__device__ __forceinline__ void mm_nn4_staged(int K, FA4 A4, const float* __restrict__ Bg,
                                              int ldb, float* stage,
                                              float (&acc)[M / 16][N / 16]) {
  Stager<N, TRANS> st;
  st.load(Bg, ldb, 0);
  for (int k0 = 0; k0 < K; k0 += 16) {
    st.store(stage);
    __syncthreads();
    if (k0 + 16 < K) st.load(Bg, ldb, k0 + 16);
    mm_nn4<M, N>(16, [&](int m, int k) { return A4(m, k0 + k); },
                 [&](int k, int n) { return *reinterpret_cast<const float4*>(stage + k * (N + 4) + n); },
                 acc);
    __syncthreads();
  }
}

// mm_nn4 with A given transposed in global memory (A(m, k) = Ag[k * lda + m]), staged the
// same way: stage holds 16 x (M + 4) floats.
template <int M, int N, class FB4>
__device__ __forceinline__ void mm_nn4_stagedA(int K, const float* __restrict__ Ag, int lda,
                                               FB4 B4, float* stage,
                                               float (&acc)[M / 16][N / 16]) {
  Stager<M, false> st;
  st.load(Ag, lda, 0);
  for (int k0 = 0; k0 < K; k0 += 16) {
    st.store(stage);
    __syncthreads();
    if (k0 + 16 < K) st.load(Ag, lda, k0 + 16);
    mm_nn4<M, N>(16,
                 [&](int m, int k) {
                   const float* col = stage + k * (M + 4) + m;
                   return make_float4(col[0], col[M + 4], col[2 * (M + 4)], col[3 * (M + 4)]);
                 },
                 [&](int k, int n) { return B4(k0 + k, n); }, acc);
    __syncthreads();
  }
}

// A4 / B4 readers: rows of a k-contiguous (A) or n-contiguous (B) matrix, 16-byte aligned
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ldg4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

// sum over the 16 lanes of a row group (tj = lane % 16), every lane gets the total
__device__ __forceinline__ float rowgroup_sum(float x) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int DK, int DV>
struct BwdLd {
  static constexpr int K = DK + 4, V = DV + 4, X = (DK > DV ? DK : DV) + 4, C = kC + 4;
};

template <int DK, int DV>
constexpr size_t bwd_chunk_smem_bytes() {
  using L = BwdLd<DK, DV>;
  return (2 * kC * L::K + 2 * kC * L::X + kC * L::V + 3 * kC * L::C + 5 * kC + 8 +
          16 * L::X) * sizeof(float);
}

// Per-chunk backward (grid: chunks x H x B, fp32 pipes): everything local to the chunk once
// dW and the state gradient at its end are known (K^ K^T comes from the factor kernel's
// tensor-core product).  dq^ and dk^ stay in registers (rows ti + 16 u,
// columns tj + 16 c of the thread) until the L2 normalisations are back-propagated and they
// are written once; every other result goes through shared memory.  Row reductions (the
// log-decay and beta gradients) are summed over the 16 lanes that own a row, in a fixed
// order (deterministic).
template <int DK, int DV>
__global__ void __launch_bounds__(256) gdr_bwd_chunk_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const float* __restrict__ beta,
    const __nv_bfloat16* __restrict__ dO, const float* __restrict__ Y, const float* __restrict__ U,
    const float* __restrict__ Pm, const float* __restrict__ Gc, const float* __restrict__ Ai,
    const float* __restrict__ Schk, const float* __restrict__ dSchk,
    const float* __restrict__ dWg, const float* __restrict__ KKg, const float* __restrict__ Wg,
    int T, int H, int nch, float scale,
    float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
    float* __restrict__ dbeta, float* __restrict__ dg) {
  using L = BwdLd<DK, DV>;
  constexpr int LK = L::K, LV = L::V, LX = L::X, LC = L::C;
  constexpr int RU = kC / 16;            // rows per thread
  constexpr int CK = DK / 16, CV = DV / 16, CC = kC / 16;  // columns per thread
  extern __shared__ float4 smb4[];
  float* sm = reinterpret_cast<float*>(smb4);
  float* sQ = sm;                   // [C][LK] q^
  float* sK = sQ + kC * LK;         // [C][LK] k^
  float* sW = sK + kC * LK;         // [C][LX] W, later dBk
  float* sX = sW + kC * LX;         // [C][LX] dO, later dY, later dBv
  float* sdW = sX + kC * LX;        // [C][LV] dW
  float* sC1 = sdW + kC * LV;       // [C][LC] Gam . dP, later Z
  float* sC2 = sC1 + kC * LC;       // [C][LC] R = dP . P + dM . M (log-decay gradient)
  float* sC3 = sC2 + kC * LC;       // [C][LC] dM . Gam . K^K^T (beta gradient)
  float* sG = sC3 + kC * LC;        // [C] cumulative log decay
  float* sB = sG + kC;              // [C] beta
  float* sdG = sB + kC;             // [C] log-decay gradient
  float* sdB = sdG + kC;            // [C] beta gradient
  float* sPart = sdB + kC;          // [C] per-row partial sums
  float* sRed = sPart + kC;         // [8] block reduction
  float* sStg = sRed + 8;           // [16][<= LX] staged rows of a global operand
  static_assert(kC + 4 <= LX, "the staging buffer holds 16 rows of any operand");
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ti = tid >> 4, tj = tid & 15;
  const size_t bh = static_cast<size_t>(b) * H + h;
  const size_t cid = bh * nch + c;
  const int t0 = c * kC;
  const float* S0 = Schk + cid * DV * DK;    // state at the chunk start
  const float* dS1 = dSchk + cid * DV * DK;  // gradient of the state at the chunk end
  const float* cU = U + cid * kC * DV;
  const float* cY = Y + cid * kC * DK;
  const float* cP = Pm + cid * kC * kC;
  const float* cA = Ai + cid * kC * kC;      // A^-1 (lower triangular, zeros above)
  auto row = [&](int i) { return ((static_cast<size_t>(b) * T + t0 + i) * H + h); };

  // the chunk's tiles, 16 bytes per load (rows of the shared tiles are 16-byte aligned)
  {  // q^ and k^: rows L2-normalised as the factor kernel does it (8 values per lane, the
     // squares summed in order, then across the row's DK / 8 lanes by an xor tree)
    constexpr int PPR = DK / 8;
    static_assert(32 % PPR == 0 && (kC * PPR) % 256 == 0, "whole rows per warp, full warps");
    for (int e = tid; e < kC * PPR; e += 256) {
      const int i = e / PPR, x0 = 8 * (e - i * PPR);
      uint4 qa = make_uint4(0u, 0u, 0u, 0u), ka = qa;
      if (t0 + i < T) {
        qa = __ldg(reinterpret_cast<const uint4*>(q + row(i) * DK + x0));
        ka = __ldg(reinterpret_cast<const uint4*>(k + row(i) * DK + x0));
      }
      const uint32_t qw[4] = {qa.x, qa.y, qa.z, qa.w};
      const uint32_t kw[4] = {ka.x, ka.y, ka.z, ka.w};
      float qf[8], kf[8], sq = 0.f, sk = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 a2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw[j]));
        const float2 b2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kw[j]));
        qf[2 * j] = a2.x; qf[2 * j + 1] = a2.y;
        kf[2 * j] = b2.x; kf[2 * j + 1] = b2.y;
        sq += a2.x * a2.x + a2.y * a2.y;
        sk += b2.x * b2.x + b2.y * b2.y;
      }
#pragma unroll
      for (int o = PPR / 2; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      const float iq = sq > 0.f ? 1.0f / sqrtf(sq) : 0.f;
      const float ik = sk > 0.f ? 1.0f / sqrtf(sk) : 0.f;
      float4* qo = reinterpret_cast<float4*>(sQ + i * LK + x0);
      float4* ko = reinterpret_cast<float4*>(sK + i * LK + x0);
      qo[0] = make_float4(qf[0] * iq, qf[1] * iq, qf[2] * iq, qf[3] * iq);
      qo[1] = make_float4(qf[4] * iq, qf[5] * iq, qf[6] * iq, qf[7] * iq);
      ko[0] = make_float4(kf[0] * ik, kf[1] * ik, kf[2] * ik, kf[3] * ik);
      ko[1] = make_float4(kf[4] * ik, kf[5] * ik, kf[6] * ik, kf[7] * ik);
    }
  }
  for (int e = tid; e < kC * DV / 4; e += 256) {
    const int i = e / (DV / 4), r = 4 * (e - i * (DV / 4));
    *reinterpret_cast<float4*>(sdW + i * LV + r) = ldg4(dWg + cid * kC * DV + 4 * e);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t0 + i < T) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(dO + row(i) * DV + r));
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
      o = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    *reinterpret_cast<float4*>(sX + i * LX + r) = o;
  }
  if (tid < kC) {
    sG[tid] = Gc[cid * kC + tid];
    sB[tid] = t0 + tid < T ? beta[row(tid)] : 0.f;
    sdG[tid] = 0.f;
    sdB[tid] = 0.f;
  }
  // gamma_C <dS1, S0> (block reduction in a fixed order)
  {
    float a = 0.f;
#pragma unroll 4
    for (int e = tid; e < DV * DK / 4; e += 256) {
      const float4 u = ldg4(dS1 + 4 * e), w = ldg4(S0 + 4 * e);
      a += u.x * w.x + u.y * w.y + u.z * w.z + u.w * w.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) sRed[warp] = a;
  }
  __syncthreads();
  const float gl = sG[kC - 1];
  // (1) W = U - Y S0^T  -> sW (the forward's W when it kept it)
  if (Wg) {
    for (int e = tid; e < kC * DV / 4; e += 256) {
      const int i = e / (DV / 4), r = 4 * (e - i * (DV / 4));
      *reinterpret_cast<float4*>(sW + i * LX + r) = ldg4(Wg + cid * kC * DV + 4 * e);
    }
  } else {
    float acc[RU][CV];
    mm_zero<kC, DV>(acc);
    mm_nn4_staged<kC, DV, true>(DK, [&](int m, int x) { return ldg4(cY + m * DK + x); }, S0, DK,
                                sStg, acc);
#pragma unroll
    for (int u = 0; u < RU; ++u)
#pragma unroll
      for (int cc = 0; cc < CV; ++cc) {
        const int i = ti + 16 * u, r = bcol(tj, cc);
        sW[i * LX + r] = __ldg(&cU[i * DV + r]) - acc[u][cc];
      }
  }
  __syncthreads();
  // (2) dP_ij = s dO_i . W_j (j <= i), kept as Gam . dP (sC1, and transposed in sC3 for
  // (4)); R_ij = dP_ij P_ij (sC2)
  {
    float acc[RU][CC];
    mm_zero<kC, kC>(acc);
    mm_nt4<kC, kC>(DV, [&](int m) { return sX + m * LX; }, [&](int n) { return sW + n * LX; },
                   acc);
#pragma unroll
    for (int u = 0; u < RU; ++u)
#pragma unroll
      for (int cc = 0; cc < CC; ++cc) {
        const int i = ti + 16 * u, j = tj + 16 * cc;
        float gd = 0.f, rr = 0.f;
        if (j <= i) {
          const float dp = scale * acc[u][cc];
          gd = __expf(sG[i] - sG[j]) * dp;
          rr = dp * __ldg(&cP[i * kC + j]);
        }
        sC1[i * LC + j] = gd;
        sC3[j * LC + i] = gd;
        sC2[i * LC + j] = rr;
      }
  }
  __syncthreads();
  // (3) dq^ = (Gam . dP) K^ + s gamma_i dO_i S0;  dG_i += s gamma_i (dO S0)_i . q^_i, and
  // (5) dY = -dW S0 from the same pass over S0 ([dO; dW] S0 as one 128-row product) -> sX
  float dqa[RU][CK];
  {
    float acc[2 * RU][CK];
    mm_zero<2 * kC, DK>(acc);
    mm_nn4_staged<2 * kC, DK, false>(
        DV,
        [&](int m, int r) {
          return ld4(m < kC ? sX + m * LX + r : sdW + (m - kC) * LV + r);
        },
        S0, DK, sStg, acc);
#pragma unroll
    for (int u = 0; u < RU; ++u)
#pragma unroll
      for (int cc = 0; cc < CK; ++cc) {
        dqa[u][cc] = acc[u][cc];
        sX[(ti + 16 * u) * LX + bcol(tj, cc)] = -acc[RU + u][cc];  // dO was read by all threads
      }
  }
#pragma unroll
  for (int u = 0; u < RU; ++u) {
    const int i = ti + 16 * u;
    const float sgi = scale * __expf(sG[i]);
    float part = 0.f;
#pragma unroll
    for (int cc = 0; cc < CK; ++cc) {
      dqa[u][cc] *= sgi;
      part += dqa[u][cc] * sQ[i * LK + bcol(tj, cc)];
    }
    part = rowgroup_sum(part);
    if (tj == 0) sdG[i] += part;
  }
  mm_nn4<kC, DK>(kC, [&](int m, int j) { return ld4(sC1 + m * LC + j); },
                 [&](int j, int n) { return ld4(sK + j * LK + n); }, dqa);
  // (4) dk^ = (Gam . dP)^T Q^ + diag(gamma_C / gamma) (W dS1); dG from E
  float dka[RU][CK];
  mm_zero<kC, DK>(dka);
  mm_nn4_staged<kC, DK, false>(DV, [&](int m, int r) { return ld4(sW + m * LX + r); }, dS1, DK,
                               sStg, dka);
#pragma unroll
  for (int u = 0; u < RU; ++u) {
    const int j = ti + 16 * u;
    const float ej = __expf(gl - sG[j]);
    float part = 0.f;
#pragma unroll
    for (int cc = 0; cc < CK; ++cc) {
      dka[u][cc] *= ej;
      part += dka[u][cc] * sK[j * LK + bcol(tj, cc)];
    }
    part = rowgroup_sum(part);
    if (tj == 0) {
      sdG[j] -= part;                    // exp(G_C - G_j): d/dG_j = -(...)
      sPart[j] = part;                   // and d/dG_C = +(...)
    }
  }
  mm_nn4<kC, DK>(kC,
                 [&](int m, int i) { return ld4(sC3 + m * LC + i); },
                 [&](int i, int n) { return ld4(sQ + i * LK + n); }, dka);
  __syncthreads();   // every row's part, the <dS1, S0> partials; dO and W are done with
  if (tid == 0) {
    float tot = 0.f;
    for (int j = 0; j < kC; ++j) tot += sPart[j];
    float sr = 0.f;
    for (int w = 0; w < 8; ++w) sr += sRed[w];
    sdG[kC - 1] += tot + __expf(gl) * sr;  // d/dG_C of every exp(G_C - G_j) and of gamma_C S0
  }
  // (6) dBk = A^-T dY -> sW; dk^ += beta gamma dBk; beta and G from Bk = beta gamma K^, and
  // (7) dBv = A^-T dW -> sX; dv = beta dBv; beta from Bv = beta V, from one pass over A^-1
  // (result columns 0 .. dk - 1 from dY, dk .. dk + dv - 1 from dW)
  {
    float acc[RU][CK + CV];
    mm_zero<kC, DK + DV>(acc);
    mm_nn4_stagedA<kC, DK + DV>(
        kC, cA, kC,
        [&](int i, int n) { return ld4(n < DK ? sX + i * LX + n : sdW + i * LV + (n - DK)); },
        sStg, acc);  // ends with a barrier: dY is no longer read when dBv replaces it
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      const int j = ti + 16 * u;
      const float gj = __expf(sG[j]);
      const float bg = sB[j] * gj;
      float part = 0.f;
#pragma unroll
      for (int cc = 0; cc < CK; ++cc) {
        const int x = bcol(tj, cc);
        sW[j * LX + x] = acc[u][cc];
        dka[u][cc] += bg * acc[u][cc];
        part += acc[u][cc] * sK[j * LK + x];
      }
      part = rowgroup_sum(part);
      if (tj == 0) {
        sdB[j] += gj * part;
        sdG[j] += bg * part;
      }
    }
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      const int j = ti + 16 * u;
      float part = 0.f;
#pragma unroll
      for (int cc = 0; cc < CV; ++cc) {
        const int r = bcol(tj, cc);
        const float a = acc[u][CK + cc];
        sX[j * LX + r] = a;
        float vj = 0.f;
        if (t0 + j < T) {
          dv[row(j) * DV + r] = sB[j] * a;
          vj = bf(v[row(j) * DV + r]);
        }
        part += a * vj;
      }
      part = rowgroup_sum(part);
      if (tj == 0) sdB[j] += part;
    }
  }
  __syncthreads();
  // (8) dM_ij = -(dBv_i . U_j + dBk_i . Y_j) for j < i; with M_ij = beta_i Gam_ij k^_i.k^_j:
  // Z_ij = dM_ij beta_i Gam_ij (-> sC1 as Z + Z^T, for dk^), dM_ij M_ij (added to R in sC2,
  // for dG) and dM_ij Gam_ij k^_i.k^_j (-> sC3, for dbeta)
  {
    float acc[RU][CC], kk[RU][CC];
    mm_zero<kC, kC>(acc);
    mm_nn4_staged<kC, kC, true>(DV, [&](int m, int r) { return ld4(sX + m * LX + r); }, cU, DV,
                                sStg, acc);
    mm_nn4_staged<kC, kC, true>(DK, [&](int m, int x) { return ld4(sW + m * LX + x); }, cY, DK,
                                sStg, acc);
#pragma unroll
    for (int u = 0; u < RU; ++u)  // K^ K^T from the factor kernel's tensor-core product
#pragma unroll
      for (int cc = 0; cc < CC; ++cc)
        kk[u][cc] = __ldg(&KKg[cid * kC * kC + (ti + 16 * u) * kC + bcol(tj, cc)]);
#pragma unroll
    for (int u = 0; u < RU; ++u)
#pragma unroll
      for (int cc = 0; cc < CC; ++cc) {
        const int i = ti + 16 * u, j = bcol(tj, cc);
        float z = 0.f, bt = 0.f;
        if (j < i) {
          const float a = acc[u][cc];
          const float gam = __expf(sG[i] - sG[j]);
          bt = -a * gam * kk[u][cc];
          z = -a * sB[i] * gam;
          sC2[i * LC + j] += bt * sB[i];
        }
        if (j <= i) {  // Z + Z^T (Z strictly lower triangular): the owner of (i, j) writes both
          sC1[i * LC + j] = z;
          sC1[j * LC + i] = z;
        }
        sC3[i * LC + j] = bt;
      }
  }
  __syncthreads();
  // (9) row and column sums of R, row sums of the beta terms; dk^ += (Z + Z^T) K^
  if (tid < kC) {
    const int i = tid;
    float rs = 0.f, cs = 0.f, db = 0.f;
    for (int j = 0; j < kC; ++j) {
      rs += sC2[i * LC + j];
      cs += sC2[j * LC + i];
      db += sC3[i * LC + j];
    }
    sdB[i] += db;
    sdG[i] += rs - cs;
  }
  mm_nn4<kC, DK>(kC,
                 [&](int i, int j) { return ld4(sC1 + i * LC + j); },
                 [&](int j, int n) { return ld4(sK + j * LK + n); }, dka);
  __syncthreads();
  // (10) dg = reverse cumulative sum of dG within the chunk (warp 0: lane l holds rows l and
  // 32 + l; suffix sums by shuffles in a fixed order, the upper half's total added to the
  // lower half); dbeta out
  if (tid < 32) {
    const int l = tid;
    float lo = sdG[l], hi = sdG[32 + l];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float a = __shfl_down_sync(0xffffffffu, lo, o);
      const float c2 = __shfl_down_sync(0xffffffffu, hi, o);
      if (l + o < 32) {
        lo += a;
        hi += c2;
      }
    }
    lo += __shfl_sync(0xffffffffu, hi, 0);
    if (t0 + l < T) {
      dg[row(l)] = lo;
      dbeta[row(l)] = sdB[l];
    }
    if (t0 + 32 + l < T) {
      dg[row(32 + l)] = hi;
      dbeta[row(32 + l)] = sdB[32 + l];
    }
  }
  // L2 normalisations: dx = (dx^ - x^ (x^ . dx^)) / ||x||, over the 16 lanes owning a row
#pragma unroll
  for (int u = 0; u < RU; ++u) {
    const int i = ti + 16 * u;
    const bool in = t0 + i < T;
    float nq = 0.f, nk = 0.f, pq = 0.f, pk = 0.f;
#pragma unroll
    for (int cc = 0; cc < CK; ++cc) {
      const int x = bcol(tj, cc);
      const float qv = in ? bf(q[row(i) * DK + x]) : 0.f;
      const float kv = in ? bf(k[row(i) * DK + x]) : 0.f;
      nq += qv * qv;
      nk += kv * kv;
      pq += dqa[u][cc] * sQ[i * LK + x];
      pk += dka[u][cc] * sK[i * LK + x];
    }
    nq = rowgroup_sum(nq);
    nk = rowgroup_sum(nk);
    pq = rowgroup_sum(pq);
    pk = rowgroup_sum(pk);
    if (in) {
      const float iq = nq > 0.f ? 1.0f / sqrtf(nq) : 0.f;
      const float ik = nk > 0.f ? 1.0f / sqrtf(nk) : 0.f;
#pragma unroll
      for (int cc = 0; cc < CK; ++cc) {
        const int x = bcol(tj, cc);
        dq[row(i) * DK + x] = (dqa[u][cc] - sQ[i * LK + x] * pq) * iq;
        dk[row(i) * DK + x] = (dka[u][cc] - sK[i * LK + x] * pk) * ik;
      }
    }
  }
}

size_t gdr_ws(int B, int T, int H, int dk, int dv) {
  const size_t nch = (T + kC - 1) / kC;
  const size_t chunks = static_cast<size_t>(B) * H * nch;
  return up256(chunks * kC * dk * 4) * 3 + up256(chunks * kC * dv * 4) +
         up256(chunks * kC * kC * 4) + up256(chunks * kC * 4);
}

template <int DK, int DV>
int gdr_launch(int B, int T, int H, const __nv_bfloat16* q, const __nv_bfloat16* k,
               const __nv_bfloat16* v, const float* beta, const float* g, const float* S0,
               float scale, __nv_bfloat16* o, float* ST, float* Schk, float* Wch, void* ws,
               cudaStream_t s) {
  const int nch = (T + kC - 1) / kC;
  const size_t chunks = static_cast<size_t>(B) * H * nch;
  // the workspace regions of gdr_ws, holding the tensor-core scan's operands: the split
  // [Y; gamma Q^] tiles (twice the bytes of one fp32 [C][dk] tile set) over the first two
  // regions, the split K^ over the third, U (fp32, slice-major), the split P over the fp32
  // P's region
  const size_t rk = up256(chunks * kC * DK * 4);
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto* YQs = reinterpret_cast<__nv_bfloat16*>(w);
  auto* Ks = reinterpret_cast<__nv_bfloat16*>(w + 2 * rk);
  float* Uw = reinterpret_cast<float*>(w + 3 * rk);
  auto* Ps = reinterpret_cast<__nv_bfloat16*>(w + 3 * rk + up256(chunks * kC * DV * 4));
  float* Gw = reinterpret_cast<float*>(w + 3 * rk + up256(chunks * kC * DV * 4) +
                                       up256(chunks * kC * kC * 4));
  constexpr size_t sm1 = TcChunk<DK, DV>::SMEM;
  auto k1 = gdr_chunk_kernel<DK, DV, true, false>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sm1));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_CHUNK, s);
  k1<<<dim3(nch, H, B), 256, sm1, s>>>(q, k, v, beta, g, T, H, nch, nullptr,
                                       Uw, nullptr, Gw, nullptr, YQs, Ks, Ps, GdrBwdImages{});
  mark_after(MOE_KERNEL_GDR_CHUNK, s);
  constexpr size_t sm2 = TcScan<DK>::SMEM;
  auto k2 = gdr_scan_tc_kernel<DK, DV>;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm2));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_SCAN, s);
  k2<<<dim3(DV / kRS, H, B), kTcBlock, sm2, s>>>(YQs, Ks, Ps, Uw, Gw, S0, T, H, nch, scale, o,
                                                   ST, Schk, Wch);  // Uw: slice-major U
  mark_after(MOE_KERNEL_GDR_SCAN, s);
  return static_cast<int>(cudaGetLastError());
}

// bytes per chunk of the backward scan's images: s P, s gamma Q^, E, Y (two bf16 pieces
// each) and dO^T of every 16-row value slice
size_t gdr_bwd_img_bytes(int dk, int dv) {
  return 2 * 8192 + 3 * static_cast<size_t>(dk / 64) * 16384 + static_cast<size_t>(dv / kRS) * 2048;
}

size_t gdr_bwd_ws(int B, int T, int H, int dk, int dv) {
  const size_t nch = (T + kC - 1) / kC;
  const size_t chunks = static_cast<size_t>(B) * H * nch;
  return gdr_ws(B, T, H, dk, dv) + up256(chunks * kC * kC * 4) + up256(chunks * kC * dv * 4) +
         up256(chunks * static_cast<size_t>(dv) * dk * 4) + up256(chunks * gdr_bwd_img_bytes(dk, dv)) +
         up256(chunks * kC * kC * 4);
}

template <int DK, int DV>
int gdr_bwd_launch(int B, int T, int H, const __nv_bfloat16* q, const __nv_bfloat16* k,
                   const __nv_bfloat16* v, const float* beta, const float* g, float scale,
                   const __nv_bfloat16* dO, const float* dST, const float* Schk, const float* Wch,
                   float* dq,
                   float* dk, float* dv, float* dbeta, float* dg, float* dS0, void* ws,
                   cudaStream_t s) {
  const int nch = (T + kC - 1) / kC;
  const size_t chunks = static_cast<size_t>(B) * H * nch;
  uint8_t* w = static_cast<uint8_t*>(ws);
  w += 2 * up256(chunks * kC * DK * 4);  // the forward's image regions, unused here
  float* Yw = reinterpret_cast<float*>(w); w += up256(chunks * kC * DK * 4);
  float* Uw = reinterpret_cast<float*>(w); w += up256(chunks * kC * DV * 4);
  float* Pw = reinterpret_cast<float*>(w); w += up256(chunks * kC * kC * 4);
  float* Gw = reinterpret_cast<float*>(w); w += up256(chunks * kC * 4);
  float* Aw = reinterpret_cast<float*>(w); w += up256(chunks * kC * kC * 4);
  float* dWw = reinterpret_cast<float*>(w); w += up256(chunks * kC * DV * 4);
  float* dSw = reinterpret_cast<float*>(w); w += up256(chunks * static_cast<size_t>(DV) * DK * 4);
  using LB = TcBwd<DK>;
  GdrBwdImages img;
  uint8_t* const img_base = w;
  img.sP = reinterpret_cast<__nv_bfloat16*>(w); w += chunks * 2 * LB::SP_PIECE;
  img.sQ = reinterpret_cast<__nv_bfloat16*>(w); w += chunks * 2 * LB::SQ_PIECE;
  img.E = reinterpret_cast<__nv_bfloat16*>(w); w += chunks * 2 * LB::E_PIECE;
  img.Y = reinterpret_cast<__nv_bfloat16*>(w); w += chunks * 2 * LB::Y_PIECE;
  img.OT = reinterpret_cast<__nv_bfloat16*>(w);
  w = img_base + up256(chunks * gdr_bwd_img_bytes(DK, DV));
  img.KK = reinterpret_cast<float*>(w);
  img.dO = dO;
  img.scale = scale;
  constexpr size_t sm1 = TcChunk<DK, DV>::SMEM;
  auto k1 = gdr_chunk_kernel<DK, DV, false, true>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sm1));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_BWD_FACTORS, s);
  k1<<<dim3(nch, H, B), 256, sm1, s>>>(q, k, v, beta, g, T, H, nch, Yw, Uw, Pw, Gw, Aw, nullptr,
                                       nullptr, nullptr, img);
  mark_after(MOE_KERNEL_GDR_BWD_FACTORS, s);
  constexpr size_t sm2 = LB::SMEM;
  auto k2 = gdr_bwd_scan_tc_kernel<DK, DV>;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm2));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_BWD_SCAN, s);
  k2<<<dim3(DV / kRS, H, B), kTcBlock, sm2, s>>>(img.sP, img.sQ, img.OT, img.E, img.Y, Gw, dST, H,
                                                 nch, dWw, dSw, dS0);
  mark_after(MOE_KERNEL_GDR_BWD_SCAN, s);
  const size_t sm3 = bwd_chunk_smem_bytes<DK, DV>();
  auto k3 = gdr_bwd_chunk_kernel<DK, DV>;
  e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm3));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_BWD, s);
  k3<<<dim3(nch, H, B), 256, sm3, s>>>(q, k, v, beta, dO, Yw, Uw, Pw, Gw, Aw, Schk, dSw,
                                       dWw, img.KK, Wch, T, H, nch, scale, dq, dk, dv, dbeta, dg);
  mark_after(MOE_KERNEL_GDR_BWD, s);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_gdr_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv) {
  if (B <= 0 || T <= 0 || H <= 0 || dk <= 0 || dv <= 0) return 0;
  return gdr_ws(B, T, H, dk, dv);
}

int moe_gdr_forward(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, const moe_bf16* q,
                    const moe_bf16* k, const moe_bf16* v, const float* beta, const float* g,
                    const float* S0, float scale, moe_bf16* o, float* S_T, float* S_chunks,
                    float* W_chunks, void* workspace, size_t workspace_bytes,
                    moe_stream_t stream) {
  if (B <= 0 || T <= 0 || H <= 0 || !q || !k || !v || !beta || !g || !o)
    return MOE_ERR_INVALID_ARG;
  if (!((dk == 64 || dk == 128) && (dv == 64 || dv == 128))) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * ((T + kC - 1) / kC) > (1ll << 24)) return MOE_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < gdr_ws(B, T, H, dk, dv)) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(q) |
       reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(W_chunks)) & 15u)
    return MOE_ERR_UNSUPPORTED;
  const auto* q_ = reinterpret_cast<const __nv_bfloat16*>(q);
  const auto* k_ = reinterpret_cast<const __nv_bfloat16*>(k);
  const auto* v_ = reinterpret_cast<const __nv_bfloat16*>(v);
  auto* o_ = reinterpret_cast<__nv_bfloat16*>(o);
  int e;
  if (dk == 128 && dv == 128)
    e = gdr_launch<128, 128>(B, T, H, q_, k_, v_, beta, g, S0, scale, o_, S_T, S_chunks, W_chunks, workspace, stream);
  else if (dk == 128)
    e = gdr_launch<128, 64>(B, T, H, q_, k_, v_, beta, g, S0, scale, o_, S_T, S_chunks, W_chunks, workspace, stream);
  else if (dv == 128)
    e = gdr_launch<64, 128>(B, T, H, q_, k_, v_, beta, g, S0, scale, o_, S_T, S_chunks, W_chunks, workspace, stream);
  else
    e = gdr_launch<64, 64>(B, T, H, q_, k_, v_, beta, g, S0, scale, o_, S_T, S_chunks, W_chunks, workspace, stream);
  count_launches(2);
  return e == 0 ? MOE_OK : MOE_ERR_CUDA;
}

int moe_gdr_device_status(int32_t* status, moe_stream_t stream) {
  if (!status) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  int v = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gdr_status, sizeof(int)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_gdr_status, &zero, sizeof(int)) != cudaSuccess)
    return MOE_ERR_CUDA;
  *status = v;
  return MOE_OK;
}

size_t moe_gdr_backward_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv) {
  if (B <= 0 || T <= 0 || H <= 0 || dk <= 0 || dv <= 0) return 0;
  return gdr_bwd_ws(B, T, H, dk, dv);
}

int moe_gdr_backward(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, const moe_bf16* q,
                     const moe_bf16* k, const moe_bf16* v, const float* beta, const float* g,
                     float scale, const moe_bf16* d_o, const float* dS_T, const float* S_chunks,
                     const float* W_chunks, float* dq, float* dk_out, float* dv_out, float* dbeta,
                     float* dg,
                     float* dS0, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (B <= 0 || T <= 0 || H <= 0 || !q || !k || !v || !beta || !g || !d_o || !S_chunks || !dq ||
      !dk_out || !dv_out || !dbeta || !dg)
    return MOE_ERR_INVALID_ARG;
  if (!((dk == 64 || dk == 128) && (dv == 64 || dv == 128))) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * ((T + kC - 1) / kC) > (1ll << 24)) return MOE_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < gdr_bwd_ws(B, T, H, dk, dv)) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(d_o) |
       reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(S_chunks) |
       reinterpret_cast<uintptr_t>(W_chunks)) & 15u)
    return MOE_ERR_UNSUPPORTED;
  const auto* q_ = reinterpret_cast<const __nv_bfloat16*>(q);
  const auto* k_ = reinterpret_cast<const __nv_bfloat16*>(k);
  const auto* v_ = reinterpret_cast<const __nv_bfloat16*>(v);
  const auto* o_ = reinterpret_cast<const __nv_bfloat16*>(d_o);
  int e;
  if (dk == 128 && dv == 128)
    e = gdr_bwd_launch<128, 128>(B, T, H, q_, k_, v_, beta, g, scale, o_, dS_T, S_chunks, W_chunks, dq, dk_out, dv_out, dbeta, dg, dS0, workspace, stream);
  else if (dk == 128)
    e = gdr_bwd_launch<128, 64>(B, T, H, q_, k_, v_, beta, g, scale, o_, dS_T, S_chunks, W_chunks, dq, dk_out, dv_out, dbeta, dg, dS0, workspace, stream);
  else if (dv == 128)
    e = gdr_bwd_launch<64, 128>(B, T, H, q_, k_, v_, beta, g, scale, o_, dS_T, S_chunks, W_chunks, dq, dk_out, dv_out, dbeta, dg, dS0, workspace, stream);
  else
    e = gdr_bwd_launch<64, 64>(B, T, H, q_, k_, v_, beta, g, scale, o_, dS_T, S_chunks, W_chunks, dq, dk_out, dv_out, dbeta, dg, dS0, workspace, stream);
  count_launches(3);
  return e == 0 ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"

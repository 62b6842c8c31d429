// Chunked gated delta-rule linear attention, forward (declared in include/linear_attention.h).
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
// the scan is split over slices of RS value rows (gdr_scan_kernel), so a few heads still
// fill the GPU.  Everything after the bf16 inputs is fp32 (the state in particular).
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

// Rows of the fp32 tiles in shared memory are padded to an odd stride, so that a warp
// reading one column of 32 rows touches 32 different banks.
template <int D>
struct Ld {
  static constexpr int v = D + 1;
};

// Per chunk (grid: chunks x H x B, 256 threads): q^, k^, cumulative log decay, the WY
// factors U, Y, the masked P = Gam . tril(Q^ K^T) (diagonal included), all fp32 to the
// workspace.  Rows past the end of the sequence are zero (beta = g = 0: no effect).
template <int DK, int DV>
__global__ void __launch_bounds__(256) gdr_chunk_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const float* __restrict__ beta,
    const float* __restrict__ g, int T, int H, int nch, float* __restrict__ Qh,
    float* __restrict__ Kh, float* __restrict__ Y, float* __restrict__ U,
    float* __restrict__ Pm, float* __restrict__ Gc, float* __restrict__ Ai) {
  constexpr int LK = Ld<DK>::v, LC = Ld<kC>::v;
  extern __shared__ float sm[];
  float* sK = sm;                    // [C][LK]
  float* sQ = sK + kC * LK;          // [C][LK]
  float* sA = sQ + kC * LK;          // [C][LC]  A (unit lower)
  float* sI = sA + kC * LC;          // [C][LC]  A^-1
  float* sB = sI + kC * LC;          // [C] beta
  float* sG = sB + kC;               // [C] cumulative log decay
  float* sBG = sG + kC;              // [C] beta * gamma
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = c * kC;
  const size_t chunk_id = (static_cast<size_t>(b) * H + h) * nch + c;

  // v rows: 16-byte loads issued first, held in registers until U needs them (rows past the
  // sequence are zero)
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
  // q, k rows, L2 normalised: every 16-byte load of the two tiles in flight at once; a row's
  // PPR pieces sit in PPR consecutive threads, which reduce its squared norm by shuffles
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
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = tid + 256 * m, i = e / PPR, pc = e - i * PPR;
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
        sQ[i * LK + pc * 8 + j] = qf[j] * iq;
        sK[i * LK + pc * 8 + j] = kf[j] * ik;
      }
    }
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
  // A (strictly lower part beta_i Gam_ij k^_i.k^_j, unit diagonal) and P (Gam_ij q^_i.k^_j,
  // j <= i).  Thread (ti, tj) computes the 4 x 4 block of rows 4 ti .. and columns 4 tj ..
  // (blocks above the diagonal are zero), 12 shared loads per 32 multiply-adds.
  {
    const int ti = tid >> 4, tj = tid & 15;
    float ak[4][4], aq[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c2 = 0; c2 < 4; ++c2) ak[a][c2] = aq[a][c2] = 0.f;
    if (tj <= ti) {
#pragma unroll 4
      for (int x = 0; x < DK; ++x) {
        float ki[4], qi[4], kj[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          ki[a] = sK[(4 * ti + a) * LK + x];
          qi[a] = sQ[(4 * ti + a) * LK + x];
          kj[a] = sK[(4 * tj + a) * LK + x];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c2 = 0; c2 < 4; ++c2) {
            ak[a][c2] += ki[a] * kj[c2];
            aq[a][c2] += qi[a] * kj[c2];
          }
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c2 = 0; c2 < 4; ++c2) {
        const int i = 4 * ti + a, j = 4 * tj + c2;
        float av = 0.f, pv = 0.f;
        if (j <= i) {
          const float gam = __expf(sG[i] - sG[j]);
          av = j < i ? sB[i] * gam * ak[a][c2] : 1.f;
          pv = gam * aq[a][c2];
        }
        sA[i * LC + j] = av;
        Pm[chunk_id * kC * kC + i * kC + j] = pv;
      }
  }
  __syncthreads();
  // A^-1 (unit lower triangular), one row per step: X_i = e_i - sum_{j<i} A_ij X_j, the 64
  // columns in parallel with 4 threads per column (each a quarter of the j range, combined by
  // shuffles within the 4 lanes).  A column only reads its own earlier rows, written by its
  // own four lanes, so the steps are ordered within the warp (the block barrier before Y
  // publishes the whole inverse).
  {
    const int col = tid >> 2, part = tid & 3;
    for (int i = 0; i < kC; ++i) {
      float x = 0.f;
      for (int j = col + part; j < i; j += 4) x -= sA[i * LC + j] * sI[j * LC + col];
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      if (part == 0) sI[i * LC + col] = i < col ? 0.f : (i == col ? 1.f : x);
      __syncwarp();
    }
  }
  // q^, k^ out for the scan; then K^ rows scaled by beta gamma in place
  for (int e = tid; e < kC * DK; e += 256) {
    const int i = e / DK, x = e - i * DK;
    Qh[chunk_id * kC * DK + e] = sQ[i * LK + x];
    Kh[chunk_id * kC * DK + e] = sK[i * LK + x];
  }
  __syncthreads();
  for (int e = tid; e < kC * DK; e += 256) {
    const int i = e / DK, x = e - i * DK;
    sK[i * LK + x] *= sBG[i];
  }
  __syncthreads();
  // Y = A^-1 (diag(beta gamma) K^): thread (ti, tx) computes rows 4 ti .. 4 ti + 3 and
  // columns tx, tx + 16, ... (A^-1 is zero above the diagonal)
  {
    constexpr int TX = DK / 16;
    const int ti = tid >> 4, tx = tid & 15;
    float acc[4][TX];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int u = 0; u < TX; ++u) acc[a][u] = 0.f;
    for (int j = 0; j <= 4 * ti + 3; ++j) {
      float ai[4], kv[TX];
#pragma unroll
      for (int a = 0; a < 4; ++a) ai[a] = sI[(4 * ti + a) * LC + j];
#pragma unroll
      for (int u = 0; u < TX; ++u) kv[u] = sK[j * LK + tx + 16 * u];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int u = 0; u < TX; ++u) acc[a][u] += ai[a] * kv[u];
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int u = 0; u < TX; ++u) Y[chunk_id * kC * DK + (4 * ti + a) * DK + tx + 16 * u] = acc[a][u];
  }
  __syncthreads();
  // V rows (beta-scaled) into the space of the K and Q tiles (no longer needed), then
  // U = A^-1 (diag(beta) V) with the same tiling
  constexpr int LV = Ld<DV>::v;
  static_assert(kC * LV <= 2 * kC * LK, "the V tile fits where the K and Q tiles were");
  float* sV = sK;  // [C][LV]
#pragma unroll
  for (int m = 0; m < VPER; ++m) {
    const int e = tid + 256 * m, i = e / VPR, pc = e - i * VPR;
    const uint32_t vw[4] = {va[m].x, va[m].y, va[m].z, va[m].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 a2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vw[j]));
      sV[i * LV + pc * 8 + 2 * j] = sB[i] * a2.x;
      sV[i * LV + pc * 8 + 2 * j + 1] = sB[i] * a2.y;
    }
  }
  __syncthreads();
  {
    constexpr int TX = DV / 16;
    const int ti = tid >> 4, tx = tid & 15;
    float acc[4][TX];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int u = 0; u < TX; ++u) acc[a][u] = 0.f;
    for (int j = 0; j <= 4 * ti + 3; ++j) {
      float ai[4], vv[TX];
#pragma unroll
      for (int a = 0; a < 4; ++a) ai[a] = sI[(4 * ti + a) * LC + j];
#pragma unroll
      for (int u = 0; u < TX; ++u) vv[u] = sV[j * LV + tx + 16 * u];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int u = 0; u < TX; ++u) acc[a][u] += ai[a] * vv[u];
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int u = 0; u < TX; ++u) U[chunk_id * kC * DV + (4 * ti + a) * DV + tx + 16 * u] = acc[a][u];
  }
  if (tid < kC) Gc[chunk_id * kC + tid] = sG[tid];
  if (Ai)
    for (int e = tid; e < kC * kC; e += 256) Ai[chunk_id * kC * kC + e] = sI[(e / kC) * LC + (e % kC)];
}

// Scan over the chunks of one (b, h) for RS value rows of the state (grid: DV/RS x H x B,
// 256 threads).  Per chunk: W = U - Y S^T, O = scale (gamma Q^ S^T + P W), then
// S = gamma_C S + sum_j exp(G_C - G_j) w_j k^_j^T.  S_chunks (optional) receives the state
// at every chunk start (the backward's checkpoints).
//
// Two phases per chunk: W and Q^ S^T (both products with the chunk-start state), then the
// output and the state update together (the update writes the other of two state buffers,
// so both read the chunk-start state without a barrier between them).  The chunk tiles do
// not depend on the state, so they stream in with cp.async while the other phase computes,
// one shared buffer per tile: Y, Q^, the U slice and the log decays (phase 1) are reloaded
// for the next chunk right after phase 1, P and K^ (phase 2) right after phase 2; phase 1
// waits only for its own group (wait_group 1: the later group may still be in flight), and
// phase 2's group is waited for before the barrier that ends phase 1 (three barriers per
// chunk).  Each thread computes blocks of outputs from float4 shared reads that
// a warp shares (a few distinct 16-byte pieces per read), so that shared-memory bandwidth
// is not what the chain of chunks waits on.
__device__ __forceinline__ void la_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void la_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void la_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// rows x D fp32 tile (global row stride D) -> shared (row stride LDS, a multiple of 4)
template <int ROWS, int D, int LDS>
__device__ __forceinline__ void tile_async(float* dst, const float* src, int src_ld, int tid) {
  constexpr int CPR = D / 4;  // 16-byte pieces per row
  for (int e = tid; e < ROWS * CPR; e += 256) {
    const int i = e / CPR, x4 = e - i * CPR;
    cp_async_16(dst + i * LDS + 4 * x4, src + static_cast<size_t>(i) * src_ld + 4 * x4, 16u);
  }
}

template <int DK>
struct ScanLd {
  static constexpr int T = DK + 4;  // streamed tiles: 16-byte rows (bank offset 4 per row)
  static constexpr int P = kC + 4;
};

template <int DK, int DV>
__global__ void __launch_bounds__(256) gdr_scan_kernel(
    const float* __restrict__ Qh, const float* __restrict__ Kh, const float* __restrict__ Y,
    const float* __restrict__ U, const float* __restrict__ Pm, const float* __restrict__ Gc,
    const float* __restrict__ S0, int T, int H, int nch, float scale,
    __nv_bfloat16* __restrict__ o, float* __restrict__ ST, float* __restrict__ Schk) {
  constexpr int LT = ScanLd<DK>::T, LP = ScanLd<DK>::P;
  constexpr int LS = ScanLd<DK>::T;  // state rows: 16-byte aligned (read as float4)
  constexpr int LW = kC + 4;         // rows of W^T (one per value row, over the chunk's tokens)
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  float* sQ = sm;                   // [C][LT]
  float* sK = sQ + kC * LT;         // [C][LT]
  float* sY = sK + kC * LT;         // [C][LT]
  float* sP = sY + kC * LT;         // [C][LP]
  float* sU = sP + kC * LP;         // [C][RS] U slice
  float* sGr = sU + kC * kRS;       // [C] log decays
  float* sSb = sGr + kC;            // 2 x [RS][LS] state rows (ping-pong over chunks)
  float* sWT = sSb + 2 * kRS * LS;  // [RS][LW]: W^T
  float* sWd = sWT + kRS * LW;      // [C][RS]: W decayed to the chunk end
  static_assert(kRS == 16 && kC == 64 && DK % 32 == 0, "thread tiling");
  const int r0 = blockIdx.x * kRS, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const size_t bh = static_cast<size_t>(b) * H + h;
  auto issue_a = [&](int c) {  // Y, Q^, U slice, log decays (phase 1)
    if (c < nch) {
      const size_t cid = bh * nch + c;
      tile_async<kC, DK, LT>(sY, Y + cid * kC * DK, DK, tid);
      tile_async<kC, DK, LT>(sQ, Qh + cid * kC * DK, DK, tid);
      tile_async<kC, kRS, kRS>(sU, U + cid * kC * DV + r0, DV, tid);
      tile_async<1, kC, kC>(sGr, Gc + cid * kC, kC, tid);
    }
    la_commit();
  };
  auto issue_b = [&](int c) {  // P, K^ (phase 2)
    if (c < nch) {
      const size_t cid = bh * nch + c;
      tile_async<kC, kC, LP>(sP, Pm + cid * kC * kC, kC, tid);
      tile_async<kC, DK, LT>(sK, Kh + cid * kC * DK, DK, tid);
    }
    la_commit();
  };
  for (int e = tid; e < kRS * DK; e += 256) {
    const int r = e / DK, x = e - r * DK;
    sSb[r * LS + x] = S0 ? S0[(bh * DV + r0 + r) * DK + x] : 0.f;
  }
  issue_a(0);
  issue_b(0);
  // Phases 1 and 2a: this thread's token rows i0 = tid / 8 and i1 = i0 + 32 and value rows
  // c0 = tid % 8 and c1 = c0 + 8 (a warp reads four token rows and eight state rows per step:
  // one shared-memory wavefront each).
  const int cq = tid & 7, i0 = tid >> 3, i1 = i0 + 32;
  const int c0 = cq, c1 = cq + 8;
  // Phase 2b: value rows rs * RPL .. + RPL - 1, float4 column group cg (a warp reads GW
  // column groups of K^ and RSEL row pieces of the decayed W per token: one wavefront each).
  constexpr int GW = DK / 32;          // column groups per warp
  constexpr int RSEL = 32 / GW;        // row selectors per warp
  constexpr int RPL = kRS / RSEL;      // rows per lane (2 for DK 128, 1 for 64)
  static_assert(RPL * RSEL == kRS && (RPL == 1 || RPL == 2), "state update tiling");
  const int lane = tid & 31, warp = tid >> 5;
  const int cg = warp * GW + lane / RSEL, rs = lane % RSEL;
  for (int c = 0; c < nch; ++c) {
    const size_t cid = bh * nch + c;
    const float* sS = sSb + (c & 1) * kRS * LS;      // state at the chunk start
    float* sSn = sSb + ((c & 1) ^ 1) * kRS * LS;     // state at the chunk end
    la_wait1();        // Y, Q^, U, decays of chunk c
    __syncthreads();   // (everyone's copies; the previous chunk is done with every tile)
    const float gC = sGr[kC - 1];
    const float gam_C = __expf(gC);
    if (Schk)
      for (int e = tid; e < kRS * DK; e += 256) {
        const int r = e / DK, x = e - r * DK;
        Schk[(cid * DV + r0 + r) * DK + x] = sS[r * LS + x];
      }
    // phase 1: Y S^T and Q^ S^T for rows i0, i1 and value rows c0, c1; W = U - Y S^T
    float oq[2][2];
    {
      float gy[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, gq[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      const float4* y0 = reinterpret_cast<const float4*>(sY + i0 * LT);
      const float4* y1 = reinterpret_cast<const float4*>(sY + i1 * LT);
      const float4* q0 = reinterpret_cast<const float4*>(sQ + i0 * LT);
      const float4* q1 = reinterpret_cast<const float4*>(sQ + i1 * LT);
      const float4* s0 = reinterpret_cast<const float4*>(sS + c0 * LS);
      const float4* s1 = reinterpret_cast<const float4*>(sS + c1 * LS);
#pragma unroll 4
      for (int x4 = 0; x4 < DK / 4; ++x4) {
        const float4 a0 = y0[x4], a1 = y1[x4], b0 = q0[x4], b1 = q1[x4];
        const float4 u0 = s0[x4], u1 = s1[x4];
        gy[0][0] += a0.x * u0.x + a0.y * u0.y + a0.z * u0.z + a0.w * u0.w;
        gy[0][1] += a0.x * u1.x + a0.y * u1.y + a0.z * u1.z + a0.w * u1.w;
        gy[1][0] += a1.x * u0.x + a1.y * u0.y + a1.z * u0.z + a1.w * u0.w;
        gy[1][1] += a1.x * u1.x + a1.y * u1.y + a1.z * u1.z + a1.w * u1.w;
        gq[0][0] += b0.x * u0.x + b0.y * u0.y + b0.z * u0.z + b0.w * u0.w;
        gq[0][1] += b0.x * u1.x + b0.y * u1.y + b0.z * u1.z + b0.w * u1.w;
        gq[1][0] += b1.x * u0.x + b1.y * u0.y + b1.z * u0.z + b1.w * u0.w;
        gq[1][1] += b1.x * u1.x + b1.y * u1.y + b1.z * u1.z + b1.w * u1.w;
      }
      const int ir[2] = {i0, i1}, cr[2] = {c0, c1};
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const float gi = sGr[ir[a]];
        const float gam_i = __expf(gi), dec_i = __expf(gC - gi);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float w = sU[ir[a] * kRS + cr[q]] - gy[a][q];
          sWT[cr[q] * LW + ir[a]] = w;
          sWd[ir[a] * kRS + cr[q]] = w * dec_i;
          oq[a][q] = gam_i * gq[a][q];
        }
      }
    }
    la_wait0();        // this thread's copies of P, K^ of chunk c have landed
    __syncthreads();   // W is complete; P, K^ are visible; Y, Q^, U and the decays are free
    issue_a(c + 1);
    // phase 2a: O = scale (gamma_i Q^_i . S_r + sum_{j<=i} P_ij w_jr)  (P is zero above the
    // diagonal; i0 <= 4 * warp + 3 and i1 < 4 * warp + 36, so whole 4-token steps suffice)
    {
      const float* p0 = sP + i0 * LP;
      const float* p1 = sP + i1 * LP;
      const float* w0 = sWT + c0 * LW;
      const float* w1 = sWT + c1 * LW;
      for (int j0 = 0; j0 <= i1; j0 += 4) {
        const float4 wa = *reinterpret_cast<const float4*>(w0 + j0);
        const float4 wb = *reinterpret_cast<const float4*>(w1 + j0);
        const float4 pb = *reinterpret_cast<const float4*>(p1 + j0);
        oq[1][0] += pb.x * wa.x + pb.y * wa.y + pb.z * wa.z + pb.w * wa.w;
        oq[1][1] += pb.x * wb.x + pb.y * wb.y + pb.z * wb.z + pb.w * wb.w;
        if (j0 <= i0) {
          const float4 pa = *reinterpret_cast<const float4*>(p0 + j0);
          oq[0][0] += pa.x * wa.x + pa.y * wa.y + pa.z * wa.z + pa.w * wa.w;
          oq[0][1] += pa.x * wb.x + pa.y * wb.y + pa.z * wb.z + pa.w * wb.w;
        }
      }
      const int ir[2] = {i0, i1}, cr[2] = {c0, c1};
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int t = c * kC + ir[a];
        if (t < T) {
          __nv_bfloat16* orow = o + ((static_cast<size_t>(b) * T + t) * H + h) * DV + r0;
#pragma unroll
          for (int q = 0; q < 2; ++q) orow[cr[q]] = __float2bfloat16_rn(scale * oq[a][q]);
        }
      }
    }
    // phase 2b (same phase: it writes the other state buffer):
    // S_r = gamma_C S_r + sum_j (gamma_C / gamma_j) w_jr k^_j
    {
      float4 acc[RPL];
#pragma unroll
      for (int v = 0; v < RPL; ++v) {
        const float4 sv = reinterpret_cast<const float4*>(sS + (rs * RPL + v) * LS)[cg];
        acc[v] = make_float4(gam_C * sv.x, gam_C * sv.y, gam_C * sv.z, gam_C * sv.w);
      }
#pragma unroll 8
      for (int j = 0; j < kC; ++j) {
        const float4 kv = reinterpret_cast<const float4*>(sK + j * LT)[cg];
        float wd[RPL];
        if constexpr (RPL == 2) {
          const float2 w2 = *reinterpret_cast<const float2*>(sWd + j * kRS + 2 * rs);
          wd[0] = w2.x;
          wd[1] = w2.y;
        } else {
          wd[0] = sWd[j * kRS + rs];
        }
#pragma unroll
        for (int v = 0; v < RPL; ++v) {
          acc[v].x += wd[v] * kv.x;
          acc[v].y += wd[v] * kv.y;
          acc[v].z += wd[v] * kv.z;
          acc[v].w += wd[v] * kv.w;
        }
      }
#pragma unroll
      for (int v = 0; v < RPL; ++v)
        reinterpret_cast<float4*>(sSn + (rs * RPL + v) * LS)[cg] = acc[v];
    }
    __syncthreads();   // P and K^ are free (the next chunk's first barrier orders the state)
    issue_b(c + 1);
  }
  __syncthreads();
  if (ST) {
    const float* sS = sSb + (nch & 1) * kRS * LS;
    for (int e = tid; e < kRS * DK; e += 256) {
      const int r = e / DK, x = e - r * DK;
      ST[(bh * DV + r0 + r) * DK + x] = sS[r * LS + x];
    }
  }
}

template <int DK>
constexpr size_t scan_smem_bytes() {
  return (3 * kC * ScanLd<DK>::T + kC * ScanLd<DK>::P + kC * kRS + kC +
          2 * kRS * ScanLd<DK>::T + kRS * (kC + 4) + kC * kRS) * sizeof(float);
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

// Backward scan over chunks for RS value rows of dS (grid: DV/RS x H x B).  Writes dW (the
// slice's columns) and the state gradient at every chunk end; dS0 at the end.  The chunk
// tiles stream in with cp.async as in the forward scan: P, K^, the dO slice and the log
// decays (needed by dW) are reloaded for the next chunk right after dW, Q^ and Y (needed by
// the state-gradient update) right after it (wait_group 1).
template <int DK, int DV>
__global__ void __launch_bounds__(256) gdr_bwd_scan_kernel(
    const float* __restrict__ Qh, const float* __restrict__ Kh, const float* __restrict__ Y,
    const float* __restrict__ Pm, const float* __restrict__ Gc,
    const __nv_bfloat16* __restrict__ dO, const float* __restrict__ dST, int T, int H, int nch,
    float scale, float* __restrict__ dW, float* __restrict__ dSchk, float* __restrict__ dS0) {
  constexpr int LT = ScanLd<DK>::T, LP = ScanLd<DK>::P;
  constexpr int LS = ScanLd<DK>::T;  // state-gradient rows: 16-byte aligned (read as float4)
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  float* sQ = sm;                   // [C][LT]
  float* sK = sQ + kC * LT;         // [C][LT]
  float* sY = sK + kC * LT;         // [C][LT]
  float* sP = sY + kC * LT;         // [C][LP]
  float* sGr = sP + kC * LP;        // [C] log decays
  __nv_bfloat16* sOb = reinterpret_cast<__nv_bfloat16*>(sGr + kC);  // [C][RS] dO slice
  float* sD = sGr + kC + kC * kRS / 2;  // [RS][LS] state gradient rows
  float* sW = sD + kRS * LS;        // [C][RS] dW slice
  float* sOg = sW + kC * kRS;       // [C][RS] s gamma_i dO
  static_assert(kRS == 16 && kC == 64 && DK % 32 == 0, "thread tiling");
  static_assert(kRS * 2 % 16 == 0, "dO slice rows are whole 16-byte pieces");
  const int r0 = blockIdx.x * kRS, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const size_t bh = static_cast<size_t>(b) * H + h;
  auto issue_a = [&](int c) {  // P, K^, dO slice, log decays
    if (c >= 0) {
      const size_t cid = bh * nch + c;
      tile_async<kC, kC, LP>(sP, Pm + cid * kC * kC, kC, tid);
      tile_async<kC, DK, LT>(sK, Kh + cid * kC * DK, DK, tid);
      tile_async<1, kC, kC>(sGr, Gc + cid * kC, kC, tid);
      constexpr int PPR = kRS * 2 / 16;  // 16-byte pieces per dO row
      for (int e = tid; e < kC * PPR; e += 256) {
        const int i = e / PPR, pc = e - i * PPR;
        const int t = c * kC + i;
        // rows past the sequence read row 0 and are zeroed when used (t >= T below)
        const size_t row = (static_cast<size_t>(b) * T + (t < T ? t : 0)) * H + h;
        cp_async_16(sOb + i * kRS + pc * 8, dO + row * DV + r0 + pc * 8, 16u);
      }
    }
    la_commit();
  };
  auto issue_b = [&](int c) {  // Q^, Y
    if (c >= 0) {
      const size_t cid = bh * nch + c;
      tile_async<kC, DK, LT>(sQ, Qh + cid * kC * DK, DK, tid);
      tile_async<kC, DK, LT>(sY, Y + cid * kC * DK, DK, tid);
    }
    la_commit();
  };
  for (int e = tid; e < kRS * DK; e += 256) {
    const int r = e / DK, x = e - r * DK;
    sD[r * LS + x] = dST ? dST[(bh * DV + r0 + r) * DK + x] : 0.f;
  }
  issue_a(nch - 1);
  issue_b(nch - 1);
  // dW phase: token rows i0 = tid / 8 and i1 = i0 + 32, value rows c0 = tid % 8, c1 = c0 + 8
  const int cq = tid & 7, i0 = tid >> 3, i1 = i0 + 32;
  const int c0 = cq, c1 = cq + 8;
  // state-gradient phase: value rows rs * RPL .. + RPL - 1, float4 column group cg
  constexpr int GW = DK / 32, RSEL = 32 / GW, RPL = kRS / RSEL;
  static_assert(RPL * RSEL == kRS && (RPL == 1 || RPL == 2), "state-gradient tiling");
  const int lane = tid & 31, warp = tid >> 5;
  const int cg = warp * GW + lane / RSEL, rs = lane % RSEL;
  for (int c = nch - 1; c >= 0; --c) {
    const size_t cid = bh * nch + c;
    la_wait1();        // P, K^, dO, decays of chunk c
    __syncthreads();
    const float gC = sGr[kC - 1];
    const float gam_C = __expf(gC);
    for (int e = tid; e < kRS * DK; e += 256) {
      const int r = e / DK, x = e - r * DK;
      dSchk[(cid * DV + r0 + r) * DK + x] = sD[r * LS + x];
    }
    // dW = s P^T dO + E dS1^T
    {
      float kd[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, pd[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      const float4* ka = reinterpret_cast<const float4*>(sK + i0 * LT);
      const float4* kb = reinterpret_cast<const float4*>(sK + i1 * LT);
      const float4* da = reinterpret_cast<const float4*>(sD + c0 * LS);
      const float4* db = reinterpret_cast<const float4*>(sD + c1 * LS);
#pragma unroll 4
      for (int x4 = 0; x4 < DK / 4; ++x4) {
        const float4 a0 = ka[x4], a1 = kb[x4], u0 = da[x4], u1 = db[x4];
        kd[0][0] += a0.x * u0.x + a0.y * u0.y + a0.z * u0.z + a0.w * u0.w;
        kd[0][1] += a0.x * u1.x + a0.y * u1.y + a0.z * u1.z + a0.w * u1.w;
        kd[1][0] += a1.x * u0.x + a1.y * u0.y + a1.z * u0.z + a1.w * u0.w;
        kd[1][1] += a1.x * u1.x + a1.y * u1.y + a1.z * u1.z + a1.w * u1.w;
      }
      // P^T dO: P[t][i] is zero for t < i, so row i0 starts at the warp's first row 4 * warp
      // and row i1 at 4 * warp + 32
      const int tw = 4 * warp;
      for (int t = tw; t < kC; ++t) {
        const bool in = c * kC + t < T;
        const float o0 = in ? bf(sOb[t * kRS + c0]) : 0.f;
        const float o1 = in ? bf(sOb[t * kRS + c1]) : 0.f;
        const float p0 = sP[t * LP + i0];
        pd[0][0] += p0 * o0;
        pd[0][1] += p0 * o1;
        if (t >= tw + 32) {
          const float p1 = sP[t * LP + i1];
          pd[1][0] += p1 * o0;
          pd[1][1] += p1 * o1;
        }
      }
      const int ir[2] = {i0, i1}, cr[2] = {c0, c1};
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int i = ir[a];
        const float gi = sGr[i];
        const float gam_i = __expf(gi), dec_i = __expf(gC - gi);
        const bool in_i = c * kC + i < T;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float w = scale * pd[a][q] + dec_i * kd[a][q];
          sW[i * kRS + cr[q]] = w;
          dW[cid * kC * DV + i * DV + r0 + cr[q]] = w;
          sOg[i * kRS + cr[q]] = in_i ? scale * gam_i * bf(sOb[i * kRS + cr[q]]) : 0.f;
        }
      }
    }
    la_wait0();        // this thread's copies of Q^, Y of chunk c have landed
    __syncthreads();   // dW is complete; Q^, Y are visible; P, K^, dO and the decays are free
    issue_a(c - 1);
    // dS0 = gamma_C dS1 + sum_j (s gamma_j dO_jr) q^_j - sum_j dW_jr Y_j  (each thread reads
    // and rewrites its own elements of the state gradient)
    {
      float4 acc[RPL];
#pragma unroll
      for (int v = 0; v < RPL; ++v) {
        const float4 sv = reinterpret_cast<const float4*>(sD + (rs * RPL + v) * LS)[cg];
        acc[v] = make_float4(gam_C * sv.x, gam_C * sv.y, gam_C * sv.z, gam_C * sv.w);
      }
#pragma unroll 8
      for (int j = 0; j < kC; ++j) {
        const float4 qv = reinterpret_cast<const float4*>(sQ + j * LT)[cg];
        const float4 yv = reinterpret_cast<const float4*>(sY + j * LT)[cg];
        float og[RPL], wv[RPL];
        if constexpr (RPL == 2) {
          const float2 o2 = *reinterpret_cast<const float2*>(sOg + j * kRS + 2 * rs);
          const float2 w2 = *reinterpret_cast<const float2*>(sW + j * kRS + 2 * rs);
          og[0] = o2.x;
          og[1] = o2.y;
          wv[0] = w2.x;
          wv[1] = w2.y;
        } else {
          og[0] = sOg[j * kRS + rs];
          wv[0] = sW[j * kRS + rs];
        }
#pragma unroll
        for (int v = 0; v < RPL; ++v) {
          acc[v].x += og[v] * qv.x - wv[v] * yv.x;
          acc[v].y += og[v] * qv.y - wv[v] * yv.y;
          acc[v].z += og[v] * qv.z - wv[v] * yv.z;
          acc[v].w += og[v] * qv.w - wv[v] * yv.w;
        }
      }
#pragma unroll
      for (int v = 0; v < RPL; ++v)
        reinterpret_cast<float4*>(sD + (rs * RPL + v) * LS)[cg] = acc[v];
    }
    __syncthreads();   // Q^ and Y are free
    issue_b(c - 1);
  }
  __syncthreads();
  if (dS0)
    for (int e = tid; e < kRS * DK; e += 256) {
      const int r = e / DK, x = e - r * DK;
      dS0[(bh * DV + r0 + r) * DK + x] = sD[r * LS + x];
    }
}

template <int DK>
constexpr size_t bwd_scan_smem_bytes() {
  return (3 * kC * ScanLd<DK>::T + kC * ScanLd<DK>::P + kC + kC * kRS / 2 + kRS * ScanLd<DK>::T +
          2 * kC * kRS) * sizeof(float);
}

// Register-tiled products of the per-chunk backward, for 256 threads: thread (ti, tj) =
// (tid / 16, tid % 16) owns rows ti + 16 u (u < M / 16) and columns tj + 16 c (c < N / 16)
// of an M x N result and adds its sums to acc[u][c] (k ascending, one fp32 chain per output).
//   mm_nn:  A(m, k) and B(k, n) element callables (B's columns are consecutive across the
//           16 lanes of a row group, A's rows are two per warp: broadcast reads)
//   mm_nt4: A and B given by k-contiguous rows (shared or global, 16-byte aligned), read 16
//           bytes at a time
template <int M, int N, class FA, class FB>
__device__ __forceinline__ void mm_nn(int K, FA A, FB B, float (&acc)[M / 16][N / 16]) {
  const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
#pragma unroll 2
  for (int k = 0; k < K; ++k) {
    float a[M / 16], bb[N / 16];
#pragma unroll
    for (int u = 0; u < M / 16; ++u) a[u] = A(ti + 16 * u, k);
#pragma unroll
    for (int c = 0; c < N / 16; ++c) bb[c] = B(k, tj + 16 * c);
#pragma unroll
    for (int u = 0; u < M / 16; ++u)
#pragma unroll
      for (int c = 0; c < N / 16; ++c) acc[u][c] += a[u] * bb[c];
  }
}

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

// mm_nn with B in global memory, staged through shared memory 16 k rows at a time (every
// element read once by the CTA, the next block loading while the current one is used):
// B(k, n) = Bg[k * ldb + n], or Bg[n * ldb + k] with TRANS.  stage: 16 x (N + 4) floats.
// Every thread of the block must call it (it synchronises).
template <int M, int N, bool TRANS, class FA>
__device__ __forceinline__ void mm_nn_staged(int K, FA A, const float* __restrict__ Bg, int ldb,
                                             float* stage, float (&acc)[M / 16][N / 16]) {
  Stager<N, TRANS> st;
  st.load(Bg, ldb, 0);
  for (int k0 = 0; k0 < K; k0 += 16) {
    st.store(stage);
    __syncthreads();
    if (k0 + 16 < K) st.load(Bg, ldb, k0 + 16);
    mm_nn<M, N>(16, [&](int m, int k) { return A(m, k0 + k); },
                [&](int k, int n) { return stage[k * (N + 4) + n]; }, acc);
    __syncthreads();
  }
}

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

// Per-chunk backward (grid: chunks x H x B): everything local to the chunk once dW and the
// state gradient at its end are known.  dq^ and dk^ stay in registers (rows ti + 16 u,
// columns tj + 16 c of the thread) until the L2 normalisations are back-propagated and they
// are written once; every other result goes through shared memory.  Row reductions (the
// log-decay and beta gradients) are summed over the 16 lanes that own a row, in a fixed
// order (deterministic).
template <int DK, int DV>
__global__ void __launch_bounds__(256) gdr_bwd_chunk_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const float* __restrict__ beta,
    const __nv_bfloat16* __restrict__ dO, const float* __restrict__ Qh,
    const float* __restrict__ Kh, const float* __restrict__ Y, const float* __restrict__ U,
    const float* __restrict__ Pm, const float* __restrict__ Gc, const float* __restrict__ Ai,
    const float* __restrict__ Schk, const float* __restrict__ dSchk,
    const float* __restrict__ dWg, int T, int H, int nch, float scale,
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
  for (int e = tid; e < kC * DK / 4; e += 256) {
    const int i = e / (DK / 4), x = 4 * (e - i * (DK / 4));
    *reinterpret_cast<float4*>(sQ + i * LK + x) = ldg4(Qh + cid * kC * DK + 4 * e);
    *reinterpret_cast<float4*>(sK + i * LK + x) = ldg4(Kh + cid * kC * DK + 4 * e);
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
  // (1) W = U - Y S0^T  -> sW
  {
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
  // (2) dP_ij = s dO_i . W_j (j <= i), kept as Gam . dP (sC1); R_ij = dP_ij P_ij (sC2)
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
        sC2[i * LC + j] = rr;
      }
  }
  __syncthreads();
  // (3) dq^ = (Gam . dP) K^ + s gamma_i dO_i S0;  dG_i += s gamma_i (dO S0)_i . q^_i
  float dqa[RU][CK];
  mm_zero<kC, DK>(dqa);
  mm_nn4_staged<kC, DK, false>(DV, [&](int m, int r) { return ld4(sX + m * LX + r); }, S0, DK,
                               sStg, dqa);
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
                 [&](int m, int i) {
                   return make_float4(sC1[i * LC + m], sC1[(i + 1) * LC + m],
                                      sC1[(i + 2) * LC + m], sC1[(i + 3) * LC + m]);
                 },
                 [&](int i, int n) { return ld4(sQ + i * LK + n); }, dka);
  __syncthreads();   // every row's part, the <dS1, S0> partials; dO and W are done with
  if (tid == 0) {
    float tot = 0.f;
    for (int j = 0; j < kC; ++j) tot += sPart[j];
    float sr = 0.f;
    for (int w = 0; w < 8; ++w) sr += sRed[w];
    sdG[kC - 1] += tot + __expf(gl) * sr;  // d/dG_C of every exp(G_C - G_j) and of gamma_C S0
  }
  // (5) dY = -dW S0 -> sX
  {
    float acc[RU][CK];
    mm_zero<kC, DK>(acc);
    mm_nn4_staged<kC, DK, false>(DV, [&](int m, int r) { return ld4(sdW + m * LV + r); }, S0,
                                 DK, sStg, acc);
#pragma unroll
    for (int u = 0; u < RU; ++u)
#pragma unroll
      for (int cc = 0; cc < CK; ++cc) sX[(ti + 16 * u) * LX + bcol(tj, cc)] = -acc[u][cc];
  }
  __syncthreads();
  // (6) dBk = A^-T dY -> sW; dk^ += beta gamma dBk; beta and G from Bk = beta gamma K^
  {
    float acc[RU][CK];
    mm_zero<kC, DK>(acc);
    mm_nn4_stagedA<kC, DK>(kC, cA, kC, [&](int i, int n) { return ld4(sX + i * LX + n); }, sStg,
                           acc);
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
  }
  __syncthreads();
  // (7) dBv = A^-T dW -> sX; dv = beta dBv; beta from Bv = beta V
  {
    float acc[RU][CV];
    mm_zero<kC, DV>(acc);
    mm_nn4_stagedA<kC, DV>(kC, cA, kC, [&](int i, int n) { return ld4(sdW + i * LV + n); },
                           sStg, acc);
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      const int j = ti + 16 * u;
      float part = 0.f;
#pragma unroll
      for (int cc = 0; cc < CV; ++cc) {
        const int r = bcol(tj, cc);
        const float a = acc[u][cc];
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
  // Z_ij = dM_ij beta_i Gam_ij (-> sC1, for dk^), dM_ij M_ij (added to R in sC2, for dG) and
  // dM_ij Gam_ij k^_i.k^_j (-> sC3, for dbeta)
  {
    float acc[RU][CC], kk[RU][CC];
    mm_zero<kC, kC>(acc);
    mm_zero<kC, kC>(kk);
    mm_nn_staged<kC, kC, true>(DV, [&](int m, int r) { return sX[m * LX + r]; }, cU, DV, sStg,
                               acc);
    mm_nn_staged<kC, kC, true>(DK, [&](int m, int x) { return sW[m * LX + x]; }, cY, DK, sStg,
                               acc);
    mm_nt4<kC, kC>(DK, [&](int m) { return sK + m * LK; }, [&](int n) { return sK + n * LK; },
                   kk);
#pragma unroll
    for (int u = 0; u < RU; ++u)
#pragma unroll
      for (int cc = 0; cc < CC; ++cc) {
        const int i = ti + 16 * u, j = tj + 16 * cc;
        float z = 0.f, bt = 0.f;
        if (j < i) {
          const float a = acc[u][cc];
          const float gam = __expf(sG[i] - sG[j]);
          bt = -a * gam * kk[u][cc];
          z = -a * sB[i] * gam;
          sC2[i * LC + j] += bt * sB[i];
        }
        sC1[i * LC + j] = z;
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
                 [&](int i, int j) {
                   const float4 r = ld4(sC1 + i * LC + j);
                   return make_float4(r.x + sC1[j * LC + i], r.y + sC1[(j + 1) * LC + i],
                                      r.z + sC1[(j + 2) * LC + i], r.w + sC1[(j + 3) * LC + i]);
                 },
                 [&](int j, int n) { return ld4(sK + j * LK + n); }, dka);
  __syncthreads();
  // (10) dg = reverse cumulative sum of dG within the chunk; dbeta out
  if (tid == 0) {
    float run = 0.f;
    for (int i = kC - 1; i >= 0; --i) {
      run += sdG[i];
      if (t0 + i < T) {
        dg[row(i)] = run;
        dbeta[row(i)] = sdB[i];
      }
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
               float scale, __nv_bfloat16* o, float* ST, float* Schk, void* ws,
               cudaStream_t s) {
  const int nch = (T + kC - 1) / kC;
  const size_t chunks = static_cast<size_t>(B) * H * nch;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* Qh = reinterpret_cast<float*>(w); w += up256(chunks * kC * DK * 4);
  float* Kh = reinterpret_cast<float*>(w); w += up256(chunks * kC * DK * 4);
  float* Yw = reinterpret_cast<float*>(w); w += up256(chunks * kC * DK * 4);
  float* Uw = reinterpret_cast<float*>(w); w += up256(chunks * kC * DV * 4);
  float* Pw = reinterpret_cast<float*>(w); w += up256(chunks * kC * kC * 4);
  float* Gw = reinterpret_cast<float*>(w);
  const size_t sm1 = (2 * kC * Ld<DK>::v + 2 * kC * Ld<kC>::v + 3 * kC) * sizeof(float);
  auto k1 = gdr_chunk_kernel<DK, DV>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sm1));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_CHUNK, s);
  k1<<<dim3(nch, H, B), 256, sm1, s>>>(q, k, v, beta, g, T, H, nch, Qh, Kh, Yw, Uw, Pw, Gw,
                                       nullptr);
  mark_after(MOE_KERNEL_GDR_CHUNK, s);
  const size_t sm2 = scan_smem_bytes<DK>();
  auto k2 = gdr_scan_kernel<DK, DV>;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm2));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_SCAN, s);
  k2<<<dim3(DV / kRS, H, B), 256, sm2, s>>>(
      Qh, Kh, Yw, Uw, Pw, Gw, S0, T, H, nch, scale, o, ST, Schk);
  mark_after(MOE_KERNEL_GDR_SCAN, s);
  return static_cast<int>(cudaGetLastError());
}

size_t gdr_bwd_ws(int B, int T, int H, int dk, int dv) {
  const size_t nch = (T + kC - 1) / kC;
  const size_t chunks = static_cast<size_t>(B) * H * nch;
  return gdr_ws(B, T, H, dk, dv) + up256(chunks * kC * kC * 4) + up256(chunks * kC * dv * 4) +
         up256(chunks * static_cast<size_t>(dv) * dk * 4);
}

template <int DK, int DV>
int gdr_bwd_launch(int B, int T, int H, const __nv_bfloat16* q, const __nv_bfloat16* k,
                   const __nv_bfloat16* v, const float* beta, const float* g, float scale,
                   const __nv_bfloat16* dO, const float* dST, const float* Schk, float* dq,
                   float* dk, float* dv, float* dbeta, float* dg, float* dS0, void* ws,
                   cudaStream_t s) {
  const int nch = (T + kC - 1) / kC;
  const size_t chunks = static_cast<size_t>(B) * H * nch;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* Qh = reinterpret_cast<float*>(w); w += up256(chunks * kC * DK * 4);
  float* Kh = reinterpret_cast<float*>(w); w += up256(chunks * kC * DK * 4);
  float* Yw = reinterpret_cast<float*>(w); w += up256(chunks * kC * DK * 4);
  float* Uw = reinterpret_cast<float*>(w); w += up256(chunks * kC * DV * 4);
  float* Pw = reinterpret_cast<float*>(w); w += up256(chunks * kC * kC * 4);
  float* Gw = reinterpret_cast<float*>(w); w += up256(chunks * kC * 4);
  float* Aw = reinterpret_cast<float*>(w); w += up256(chunks * kC * kC * 4);
  float* dWw = reinterpret_cast<float*>(w); w += up256(chunks * kC * DV * 4);
  float* dSw = reinterpret_cast<float*>(w);
  const size_t sm1 = (2 * kC * Ld<DK>::v + 2 * kC * Ld<kC>::v + 3 * kC) * sizeof(float);
  auto k1 = gdr_chunk_kernel<DK, DV>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sm1));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_BWD_FACTORS, s);
  k1<<<dim3(nch, H, B), 256, sm1, s>>>(q, k, v, beta, g, T, H, nch, Qh, Kh, Yw, Uw, Pw, Gw, Aw);
  mark_after(MOE_KERNEL_GDR_BWD_FACTORS, s);
  const size_t sm2 = bwd_scan_smem_bytes<DK>();
  auto k2 = gdr_bwd_scan_kernel<DK, DV>;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm2));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_BWD_SCAN, s);
  k2<<<dim3(DV / kRS, H, B), 256, sm2, s>>>(Qh, Kh, Yw, Pw, Gw, dO, dST, T, H, nch, scale, dWw,
                                            dSw, dS0);
  mark_after(MOE_KERNEL_GDR_BWD_SCAN, s);
  const size_t sm3 = bwd_chunk_smem_bytes<DK, DV>();
  auto k3 = gdr_bwd_chunk_kernel<DK, DV>;
  e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm3));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_BWD, s);
  k3<<<dim3(nch, H, B), 256, sm3, s>>>(q, k, v, beta, dO, Qh, Kh, Yw, Uw, Pw, Gw, Aw, Schk, dSw,
                                       dWw, T, H, nch, scale, dq, dk, dv, dbeta, dg);
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
                    void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (B <= 0 || T <= 0 || H <= 0 || !q || !k || !v || !beta || !g || !o)
    return MOE_ERR_INVALID_ARG;
  if (!((dk == 64 || dk == 128) && (dv == 64 || dv == 128))) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * ((T + kC - 1) / kC) > (1ll << 24)) return MOE_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < gdr_ws(B, T, H, dk, dv)) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(q) |
       reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u)
    return MOE_ERR_UNSUPPORTED;
  const auto* q_ = reinterpret_cast<const __nv_bfloat16*>(q);
  const auto* k_ = reinterpret_cast<const __nv_bfloat16*>(k);
  const auto* v_ = reinterpret_cast<const __nv_bfloat16*>(v);
  auto* o_ = reinterpret_cast<__nv_bfloat16*>(o);
  int e;
  if (dk == 128 && dv == 128)
    e = gdr_launch<128, 128>(B, T, H, q_, k_, v_, beta, g, S0, scale, o_, S_T, S_chunks, workspace, stream);
  else if (dk == 128)
    e = gdr_launch<128, 64>(B, T, H, q_, k_, v_, beta, g, S0, scale, o_, S_T, S_chunks, workspace, stream);
  else if (dv == 128)
    e = gdr_launch<64, 128>(B, T, H, q_, k_, v_, beta, g, S0, scale, o_, S_T, S_chunks, workspace, stream);
  else
    e = gdr_launch<64, 64>(B, T, H, q_, k_, v_, beta, g, S0, scale, o_, S_T, S_chunks, workspace, stream);
  count_launches(2);
  return e == 0 ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_gdr_backward_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv) {
  if (B <= 0 || T <= 0 || H <= 0 || dk <= 0 || dv <= 0) return 0;
  return gdr_bwd_ws(B, T, H, dk, dv);
}

int moe_gdr_backward(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, const moe_bf16* q,
                     const moe_bf16* k, const moe_bf16* v, const float* beta, const float* g,
                     float scale, const moe_bf16* d_o, const float* dS_T, const float* S_chunks,
                     float* dq, float* dk_out, float* dv_out, float* dbeta, float* dg,
                     float* dS0, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (B <= 0 || T <= 0 || H <= 0 || !q || !k || !v || !beta || !g || !d_o || !S_chunks || !dq ||
      !dk_out || !dv_out || !dbeta || !dg)
    return MOE_ERR_INVALID_ARG;
  if (!((dk == 64 || dk == 128) && (dv == 64 || dv == 128))) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * ((T + kC - 1) / kC) > (1ll << 24)) return MOE_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < gdr_bwd_ws(B, T, H, dk, dv)) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(d_o) |
       reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(S_chunks)) & 15u)
    return MOE_ERR_UNSUPPORTED;
  const auto* q_ = reinterpret_cast<const __nv_bfloat16*>(q);
  const auto* k_ = reinterpret_cast<const __nv_bfloat16*>(k);
  const auto* v_ = reinterpret_cast<const __nv_bfloat16*>(v);
  const auto* o_ = reinterpret_cast<const __nv_bfloat16*>(d_o);
  int e;
  if (dk == 128 && dv == 128)
    e = gdr_bwd_launch<128, 128>(B, T, H, q_, k_, v_, beta, g, scale, o_, dS_T, S_chunks, dq, dk_out, dv_out, dbeta, dg, dS0, workspace, stream);
  else if (dk == 128)
    e = gdr_bwd_launch<128, 64>(B, T, H, q_, k_, v_, beta, g, scale, o_, dS_T, S_chunks, dq, dk_out, dv_out, dbeta, dg, dS0, workspace, stream);
  else if (dv == 128)
    e = gdr_bwd_launch<64, 128>(B, T, H, q_, k_, v_, beta, g, scale, o_, dS_T, S_chunks, dq, dk_out, dv_out, dbeta, dg, dS0, workspace, stream);
  else
    e = gdr_bwd_launch<64, 64>(B, T, H, q_, k_, v_, beta, g, scale, o_, dS_T, S_chunks, dq, dk_out, dv_out, dbeta, dg, dS0, workspace, stream);
  count_launches(3);
  return e == 0 ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"

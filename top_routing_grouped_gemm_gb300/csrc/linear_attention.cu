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
    float* __restrict__ Pm, float* __restrict__ Gc) {
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

  // q, k rows, L2 normalised (one warp per row)
  for (int i = warp; i < kC; i += 8) {
    const int t = t0 + i;
    float sq = 0.f, sk = 0.f;
    for (int x = lane; x < DK; x += 32) {
      float qv = 0.f, kv = 0.f;
      if (t < T) {
        const size_t o = ((static_cast<size_t>(b) * T + t) * H + h) * DK + x;
        qv = bf(q[o]);
        kv = bf(k[o]);
      }
      sQ[i * LK + x] = qv;
      sK[i * LK + x] = kv;
      sq += qv * qv;
      sk += kv * kv;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    const float iq = sq > 0.f ? 1.0f / sqrtf(sq) : 0.f;
    const float ik = sk > 0.f ? 1.0f / sqrtf(sk) : 0.f;
    for (int x = lane; x < DK; x += 32) {
      sQ[i * LK + x] *= iq;
      sK[i * LK + x] *= ik;
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
  // j <= i)
  for (int e = tid; e < kC * kC; e += 256) {
    const int i = e / kC, j = e - i * kC;
    float a = 0.f, p = 0.f;
    if (j <= i) {
      float dkk = 0.f, dqk = 0.f;
#pragma unroll 8
      for (int x = 0; x < DK; ++x) {
        const float kj = sK[j * LK + x];
        dkk += sK[i * LK + x] * kj;
        dqk += sQ[i * LK + x] * kj;
      }
      const float gam = __expf(sG[i] - sG[j]);
      a = j < i ? sB[i] * gam * dkk : 1.f;
      p = gam * dqk;
    }
    sA[i * LC + j] = a;
    Pm[chunk_id * kC * kC + e] = p;
  }
  __syncthreads();
  // A^-1 by forward substitution, one column per thread (unit lower triangular)
  if (tid < kC) {
    const int col = tid;
    for (int i = 0; i < kC; ++i) {
      float x = (i == col) ? 1.f : 0.f;
      for (int j = col; j < i; ++j) x -= sA[i * LC + j] * sI[j * LC + col];
      sI[i * LC + col] = i < col ? 0.f : x;
    }
  }
  __syncthreads();
  // Y = A^-1 diag(beta gamma) K^, U = A^-1 diag(beta) V; q^, k^ out for the scan
  for (int e = tid; e < kC * DK; e += 256) {
    const int i = e / DK, x = e - i * DK;
    float y = 0.f;
    for (int j = 0; j <= i; ++j) y += sI[i * LC + j] * sBG[j] * sK[j * LK + x];
    Y[chunk_id * kC * DK + e] = y;
    Qh[chunk_id * kC * DK + e] = sQ[i * LK + x];
    Kh[chunk_id * kC * DK + e] = sK[i * LK + x];
  }
  __syncthreads();
  // V rows (beta-scaled) into the space of the K and Q tiles (no longer needed), then U
  constexpr int LV = Ld<DV>::v;
  static_assert(kC * LV <= 2 * kC * LK, "the V tile fits where the K and Q tiles were");
  float* sV = sK;  // [C][LV]
  for (int e = tid; e < kC * DV; e += 256) {
    const int i = e / DV, x = e - i * DV;
    const int t = t0 + i;
    sV[i * LV + x] = t < T ? sB[i] * bf(v[((static_cast<size_t>(b) * T + t) * H + h) * DV + x]) : 0.f;
  }
  __syncthreads();
  for (int e = tid; e < kC * DV; e += 256) {
    const int i = e / DV, x = e - i * DV;
    float u = 0.f;
    for (int j = 0; j <= i; ++j) u += sI[i * LC + j] * sV[j * LV + x];
    U[chunk_id * kC * DV + e] = u;
  }
  if (tid < kC) Gc[chunk_id * kC + tid] = sG[tid];
}

// Scan over the chunks of one (b, h) for RS value rows of the state (grid: DV/RS x H x B,
// 256 threads).  Per chunk, with its q^, k^, Y and P staged in shared memory:
// W = U - Y S^T, O = scale (gamma Q^ S^T + P W), then S = gamma_C S + sum_j exp(G_C - G_j)
// w_j k^_j^T.  S_chunks (optional) receives the state at every chunk start (the backward's
// checkpoints).
template <int DK, int DV>
__global__ void __launch_bounds__(256) gdr_scan_kernel(
    const float* __restrict__ Qh, const float* __restrict__ Kh, const float* __restrict__ Y,
    const float* __restrict__ U, const float* __restrict__ Pm, const float* __restrict__ Gc,
    const float* __restrict__ S0, int T, int H, int nch, float scale,
    __nv_bfloat16* __restrict__ o, float* __restrict__ ST, float* __restrict__ Schk) {
  constexpr int LK = Ld<DK>::v, LC = Ld<kC>::v;
  extern __shared__ float sm[];
  float* sS = sm;                   // [RS][LK] state rows
  float* sQ = sS + kRS * LK;        // [C][LK]
  float* sK = sQ + kC * LK;         // [C][LK]
  float* sY = sK + kC * LK;         // [C][LK]
  float* sP = sY + kC * LK;         // [C][LC]
  float* sW = sP + kC * LC;         // [C][RS]
  float* sG = sW + kC * kRS;        // [C]
  const int r0 = blockIdx.x * kRS, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const size_t bh = static_cast<size_t>(b) * H + h;
  for (int e = tid; e < kRS * DK; e += 256) {
    const int r = e / DK, x = e - r * DK;
    sS[r * LK + x] = S0 ? S0[(bh * DV + r0 + r) * DK + x] : 0.f;
  }
  for (int c = 0; c < nch; ++c) {
    const size_t cid = bh * nch + c;
    const float* cU = U + cid * kC * DV;
    __syncthreads();  // the previous chunk is done with the tiles
    for (int e = tid; e < kC * DK; e += 256) {
      const int i = e / DK, x = e - i * DK;
      sQ[i * LK + x] = Qh[cid * kC * DK + e];
      sK[i * LK + x] = Kh[cid * kC * DK + e];
      sY[i * LK + x] = Y[cid * kC * DK + e];
    }
    for (int e = tid; e < kC * kC; e += 256) sP[(e / kC) * LC + (e % kC)] = Pm[cid * kC * kC + e];
    if (tid < kC) sG[tid] = Gc[cid * kC + tid];
    if (Schk)
      for (int e = tid; e < kRS * DK; e += 256) {
        const int r = e / DK, x = e - r * DK;
        Schk[(cid * DV + r0 + r) * DK + x] = sS[r * LK + x];
      }
    __syncthreads();
    // W = U - Y S^T   ([C][RS])
    for (int e = tid; e < kC * kRS; e += 256) {
      const int i = e / kRS, r = e - i * kRS;
      float w = cU[i * DV + r0 + r];
      const float* yi = sY + i * LK;
      const float* sr = sS + r * LK;
#pragma unroll 8
      for (int x = 0; x < DK; ++x) w -= yi[x] * sr[x];
      sW[e] = w;
    }
    __syncthreads();
    // O = scale (gamma_i Q^_i . S_r + sum_{j<=i} P_ij w_jr)
    for (int e = tid; e < kC * kRS; e += 256) {
      const int i = e / kRS, r = e - i * kRS;
      const int t = c * kC + i;
      if (t >= T) continue;
      float a = 0.f;
      const float* qi = sQ + i * LK;
      const float* sr = sS + r * LK;
#pragma unroll 8
      for (int x = 0; x < DK; ++x) a += qi[x] * sr[x];
      a *= __expf(sG[i]);
      const float* pi = sP + i * LC;
      for (int j = 0; j <= i; ++j) a += pi[j] * sW[j * kRS + r];
      o[((static_cast<size_t>(b) * T + t) * H + h) * DV + r0 + r] = __float2bfloat16_rn(scale * a);
    }
    __syncthreads();
    // S_r = gamma_C S_r + sum_j exp(G_C - G_j) w_jr k^_j
    const float gl = sG[kC - 1];
    for (int e = tid; e < kRS * DK; e += 256) {
      const int r = e / DK, x = e - r * DK;
      float s = __expf(gl) * sS[r * LK + x];
      for (int j = 0; j < kC; ++j) s += __expf(gl - sG[j]) * sW[j * kRS + r] * sK[j * LK + x];
      sS[r * LK + x] = s;
    }
  }
  __syncthreads();
  if (ST)
    for (int e = tid; e < kRS * DK; e += 256) {
      const int r = e / DK, x = e - r * DK;
      ST[(bh * DV + r0 + r) * DK + x] = sS[r * LK + x];
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
  k1<<<dim3(nch, H, B), 256, sm1, s>>>(q, k, v, beta, g, T, H, nch, Qh, Kh, Yw, Uw, Pw, Gw);
  mark_after(MOE_KERNEL_GDR_CHUNK, s);
  const size_t sm2 = (kRS * Ld<DK>::v + 3 * kC * Ld<DK>::v + kC * Ld<kC>::v + kC * kRS + kC) *
                     sizeof(float);
  auto k2 = gdr_scan_kernel<DK, DV>;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm2));
  if (e != cudaSuccess) return static_cast<int>(e);
  mark_before(MOE_KERNEL_GDR_SCAN, s);
  k2<<<dim3(DV / kRS, H, B), 256, sm2, s>>>(
      Qh, Kh, Yw, Uw, Pw, Gw, S0, T, H, nch, scale, o, ST, Schk);
  mark_after(MOE_KERNEL_GDR_SCAN, s);
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

}  // extern "C"

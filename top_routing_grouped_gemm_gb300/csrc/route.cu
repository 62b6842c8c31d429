// Router tail and auxiliary loss.
//
// The router product itself runs on the tensor cores (gemm.cuh): W_r is split once per call
// into bf16 hi + lo parts (w = hi + lo + O(2^-18 |w|)), x is exact in bf16, and the two
// partial products accumulate in fp32, which reaches fp32-level accuracy for the logits
// (the split-precision technique of Henry, Tang and Heinecke, "Leveraging the bfloat16
// Artificial Intelligence Datatype For Higher-Precision Computations", ARITH 2019).
//
// The tail (softmax over all experts, top-k, gate renormalisation, per-block probability
// sums for the auxiliary loss) follows "Day-Level Adaptation and LoRA Fine-Tuning of
// Ultra-Large-Scale Sparse MoE Models", section 2.1 (Top-16 selection, load-balancing loss)
// and "Adapting Trillion-Parameter MoE Models for LoRA Fine-Tuning", section 2.1, eq. 1.
#include <cuda_bf16.h>
#include <math.h>

#include "moe_internal.h"
#include "route.h"

namespace moe {

namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void split_router_kernel(const float4* __restrict__ w, uint2* __restrict__ hi,
                                    uint2* __restrict__ lo, size_t n4) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = w[i];
    const float x[4] = {v.x, v.y, v.z, v.w};
    __nv_bfloat16 h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      h[j] = __float2bfloat16_rn(x[j]);
      l[j] = __float2bfloat16_rn(x[j] - __bfloat162float(h[j]));
    }
    hi[i] = *reinterpret_cast<uint2*>(h);
    lo[i] = *reinterpret_cast<uint2*>(l);
  }
}

// One warp per token; lane i holds experts lane, lane+32, ... (VPL of them).
template <int VPL>
__global__ void __launch_bounds__(256) topk_softmax_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_gate, float* __restrict__ partials) {
  constexpr int WARPS = 8;
  __shared__ float red[WARPS][VPL * 32];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t_begin = blockIdx.x * kRouteTokensPerBlock;
  const int t_end = min(t_begin + kRouteTokensPerBlock, T);
  float acc[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) acc[i] = 0.f;

  for (int t = t_begin + warp; t < t_end; t += WARPS) {
    const float* row = logits + static_cast<size_t>(t) * E;
    float v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? __ldg(&row[e]) : -INFINITY;
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i) m = fmaxf(m, v[i]);
    m = warp_max(m);
    float ex[VPL];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      ex[i] = (lane + 32 * i < E) ? expf(v[i] - m) : 0.f;
      s += ex[i];
    }
    s = warp_sum(s);
    const float inv = 1.0f / s;
#pragma unroll
    for (int i = 0; i < VPL; ++i) acc[i] += ex[i] * inv;

    // k rounds of a warp arg-max over the experts not taken yet; order (value desc,
    // index asc) is total, so every lane ends each round with the same winner.
    uint32_t taken = 0;
    int my_idx = -1;
    float my_val = 0.f;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = INT_MAX;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (be == INT_MAX || v[i] > bv)) {
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == j) {
        my_idx = be;
        my_val = bv;
      }
    }
    const float pj = (lane < k) ? expf(my_val - m) * inv : 0.f;
    const float psum = warp_sum(pj);
    if (lane < k) {
      topk_idx[static_cast<size_t>(t) * k + lane] = my_idx;
      topk_gate[static_cast<size_t>(t) * k + lane] = pj / psum;
    }
  }

#pragma unroll
  for (int i = 0; i < VPL; ++i) red[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) sum += red[w][e];
    partials[static_cast<size_t>(blockIdx.x) * E + e] = sum;
  }
}

__global__ void aux_loss_kernel(const int32_t* __restrict__ counts,
                                const float* __restrict__ partials, int n_partials, int T,
                                int k, int E, float* __restrict__ aux_out) {
  __shared__ double red[1024];
  double term = 0.0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    double P = 0.0;
    for (int b = 0; b < n_partials; ++b) P += partials[static_cast<size_t>(b) * E + e];
    const double f = static_cast<double>(counts[e]) / (static_cast<double>(T) * k);
    term += f * (P / T);
  }
  red[threadIdx.x] = term;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) aux_out[0] = static_cast<float>(E * red[0]);
}

}  // namespace

int launch_split_router(const float* w, __nv_bfloat16* hi, __nv_bfloat16* lo, size_t n,
                        cudaStream_t s) {
  const size_t n4 = n / 4;
  const int grid = static_cast<int>(std::min<size_t>((n4 + 255) / 256, 4 * 152));
  split_router_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(w),
                                           reinterpret_cast<uint2*>(hi),
                                           reinterpret_cast<uint2*>(lo), n4);
  return static_cast<int>(cudaGetLastError());
}

int launch_topk_softmax(const float* logits, int T, int E, int k, int32_t* idx, float* gate,
                        float* partials, cudaStream_t s) {
  const int grid = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  if (E <= 64)
    topk_softmax_kernel<2><<<grid, 256, 0, s>>>(logits, T, E, k, idx, gate, partials);
  else if (E <= 128)
    topk_softmax_kernel<4><<<grid, 256, 0, s>>>(logits, T, E, k, idx, gate, partials);
  else if (E <= 256)
    topk_softmax_kernel<8><<<grid, 256, 0, s>>>(logits, T, E, k, idx, gate, partials);
  else if (E <= 512)
    topk_softmax_kernel<16><<<grid, 256, 0, s>>>(logits, T, E, k, idx, gate, partials);
  else if (E <= 896)
    topk_softmax_kernel<28><<<grid, 256, 0, s>>>(logits, T, E, k, idx, gate, partials);
  else
    topk_softmax_kernel<32><<<grid, 256, 0, s>>>(logits, T, E, k, idx, gate, partials);
  return static_cast<int>(cudaGetLastError());
}

int launch_aux_loss(const int32_t* counts, const float* partials, int n_partials, int T, int k,
                    int E, float* aux_out, cudaStream_t s) {
  aux_loss_kernel<<<1, 1024, 0, s>>>(counts, partials, n_partials, T, k, E, aux_out);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace moe

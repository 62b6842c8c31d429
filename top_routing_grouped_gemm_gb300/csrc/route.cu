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
#include "topk_keys.cuh"

namespace moe {

namespace {

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

// One warp per token; lane i holds the logits of experts lane, lane+32, ... (VPL of them).
// Each warp accumulates the softmax probabilities of its tokens into its own shared-memory
// row; the block then writes one row of per-block sums (fixed order: deterministic).
// k_sel >= k keys are selected; lanes k .. k_sel-1 (the token's next preferences after its
// top-k) go to alt_idx [T, k_sel - k] when it is given.  Null topk_idx / topk_gate /
// partials skip those outputs.
template <int VPL>
__global__ void __launch_bounds__(256, VPL > 28 ? 2 : 3) topk_softmax_kernel(
    const float* __restrict__ logits, int T, int E, int k, int k_sel,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate,
    float* __restrict__ partials, int32_t* __restrict__ alt_idx) {
  constexpr int WARPS = 8;
  __shared__ float red[WARPS][VPL * 32];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < VPL; ++i) red[warp][lane + 32 * i] = 0.f;
  const int t_begin = blockIdx.x * kRouteTokensPerBlock;
  const int t_end = min(t_begin + kRouteTokensPerBlock, T);

  for (int t = t_begin + warp; t < t_end; t += WARPS) {
    const float* row = logits + static_cast<size_t>(t) * E;
    float v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? __ldg(&row[e]) : -INFINITY;
    }

    // Selection in (value desc, index asc) order on the 64-bit keys.  Each lane keeps the
    // best 4 of its own keys, sorted; a round is one warp max over the lanes' heads and the
    // winning lane pops its head.  A lane whose list runs dry rescans for the best keys
    // below its last taken one (rare: its 5th, 9th, ... win).  Key 0 marks an empty slot
    // (no real key is 0: the index field of a real key is at least 0x7FFFFFFF - 1023).
    uint64_t hk[4];
    uint64_t last = ~0ull;
    auto refill = [&]() {
#pragma unroll
      for (int q = 0; q < 4; ++q) hk[q] = 0ull;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        const uint64_t key = sel_key(v[i], e);
        if (e < E && key < last && key > hk[3]) {
          hk[3] = key;
#pragma unroll
          for (int q = 3; q > 0; --q) {
            if (hk[q] > hk[q - 1]) {
              const uint64_t tk = hk[q]; hk[q] = hk[q - 1]; hk[q - 1] = tk;
            }
          }
        }
      }
    };
    refill();
    uint64_t my_key = 0ull;
    for (int j = 0; j < k_sel; ++j) {
      const uint64_t best = warp_max_u64(hk[0]);
      if (lane == j) my_key = best;
      bool dry = false;
      if (hk[0] == best) {  // keys are unique, so exactly one lane owns the winner
        last = best;
        hk[0] = hk[1]; hk[1] = hk[2]; hk[2] = hk[3]; hk[3] = 0ull;
        dry = hk[0] == 0ull;
      }
      if (__any_sync(0xffffffffu, dry) && dry) refill();
    }
    const float m = key_value(__shfl_sync(0xffffffffu, my_key, 0));  // the largest logit
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      v[i] = (lane + 32 * i < E) ? __expf(v[i] - m) : 0.f;  // v now holds exp(l - max)
      s += v[i];
    }
    s = warp_sum(s);
    const float inv = 1.0f / s;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (lane + 32 * i < E) red[warp][lane + 32 * i] += v[i] * inv;
    const float pj = (lane < k) ? __expf(key_value(my_key) - m) * inv : 0.f;
    const float psum = warp_sum(pj);
    if (lane < k && topk_idx) {
      topk_idx[static_cast<size_t>(t) * k + lane] = key_expert(my_key);
      topk_gate[static_cast<size_t>(t) * k + lane] = pj / psum;
    }
    if (alt_idx && lane >= k && lane < k_sel)
      alt_idx[static_cast<size_t>(t) * (k_sel - k) + (lane - k)] = key_expert(my_key);
  }
  if (partials == nullptr) return;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) sum += red[w][e];
    partials[static_cast<size_t>(blockIdx.x) * E + e] = sum;
  }
}

// After the router GEMM's fused top-k epilogue: per token, the global top-k merged from the
// NT tiles' 16-key candidate lists (every global winner is a winner of its own tile, so the
// merge is exact), the softmax normaliser (the row maximum from the tiles' maxima, the sum
// from the logits), the renormalised gates, and the per-block probability sums for the
// auxiliary loss.  One warp per token,
// 8 tokens per block (the row blocks of prob_partials, as topk_softmax_kernel).
template <int VPL>
__global__ void __launch_bounds__(256, VPL > 28 ? 2 : 3) route_merge_kernel(
    const float* __restrict__ logits, const uint64_t* __restrict__ cand,
    const float* __restrict__ tile_max, int T, int E, int k, int NT,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate,
    float* __restrict__ partials) {
  constexpr int WARPS = 8;
  __shared__ float red[WARPS][VPL * 32];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < VPL; ++i) red[warp][lane + 32 * i] = 0.f;
  const int t_begin = blockIdx.x * kRouteTokensPerBlock;
  const int t_end = min(t_begin + kRouteTokensPerBlock, T);
  const int ncand = NT * kRouteTileK;

  for (int t = t_begin + warp; t < t_end; t += WARPS) {
    // every load of the token up front: this lane's candidates (at most 4 of at most
    // 8 x 16), the tiles' statistics (lane n < NT holds tile n) and its logits
    const uint64_t* ct = cand + static_cast<size_t>(t) * ncand;
    uint64_t c4[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = lane + 32 * q;
      c4[q] = (c < ncand) ? __ldg(&ct[c]) : 0ull;
    }
    float M = (lane < NT) ? __ldg(&tile_max[static_cast<size_t>(t) * NT + lane]) : -INFINITY;
    const float* row = logits + static_cast<size_t>(t) * E;
    float v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? __ldg(&row[e]) : -INFINITY;
    }
    uint64_t hk[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int q = 0; q < 4; ++q) topk_insert(hk, c4[q]);
    // softmax of the whole row: the maximum from the tiles' maxima, then exp(L - max) of
    // this lane's logits and the warp's sum
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      v[i] = (lane + 32 * i < E) ? __expf(v[i] - M) : 0.f;
      part += v[i];
    }
    const float inv = 1.0f / warp_sum(part);
    // k rounds: the warp's largest head wins; its lane pops it
    uint64_t my_key = 0ull;
    for (int j = 0; j < k; ++j) {
      const uint64_t best = warp_max_u64(hk[0]);
      if (lane == j) my_key = best;
      if (hk[0] == best) {  // keys are unique: exactly one lane owns the winner
        hk[0] = hk[1]; hk[1] = hk[2]; hk[2] = hk[3]; hk[3] = 0ull;
      }
    }
    const float pj = (lane < k) ? __expf(key_value(my_key) - M) * inv : 0.f;
    const float psum = warp_sum(pj);
    if (lane < k) {
      topk_idx[static_cast<size_t>(t) * k + lane] = key_expert(my_key);
      topk_gate[static_cast<size_t>(t) * k + lane] = pj / psum;
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) red[warp][e] += v[i] * inv;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) sum += red[w][e];
    partials[static_cast<size_t>(blockIdx.x) * E + e] = sum;
  }
}

// aux stage 1: block of 32 experts x 32 row stripes; P_e summed over the partial rows in a
// fixed order, then f_e P_e summed over the block's experts -> one value per block.
__global__ void __launch_bounds__(1024) aux_stage1_kernel(const int32_t* __restrict__ counts,
                                                          const float* __restrict__ partials,
                                                          int n_partials, int T, int k, int E,
                                                          float* __restrict__ block_terms) {
  __shared__ float sm[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + tx;
  float s = 0.f;
  if (e < E)
    for (int b = ty; b < n_partials; b += 32) s += partials[static_cast<size_t>(b) * E + e];
  sm[ty][tx] = s;
  __syncthreads();
  if (ty == 0) {
    float P = 0.f;
    for (int y = 0; y < 32; ++y) P += sm[y][tx];
    float term = 0.f;
    if (e < E) term = (static_cast<float>(counts[e]) / (static_cast<float>(T) * k)) * (P / T);
    for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
    if (tx == 0) block_terms[blockIdx.x] = term;
  }
}

__global__ void aux_stage2_kernel(const float* __restrict__ block_terms, int n_blocks, int E,
                                  float* __restrict__ aux_out) {
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int b = 0; b < n_blocks; ++b) s += block_terms[b];
    aux_out[0] = static_cast<float>(E * s);
  }
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
                        float* partials, cudaStream_t s, int n_alt, int32_t* alt_idx) {
  const int grid = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  const int ks = k + (alt_idx ? n_alt : 0);
#define MOE_TOPK(V) \
  topk_softmax_kernel<V><<<grid, 256, 0, s>>>(logits, T, E, k, ks, idx, gate, partials, alt_idx)
  if (E <= 64)
    MOE_TOPK(2);
  else if (E <= 128)
    MOE_TOPK(4);
  else if (E <= 256)
    MOE_TOPK(8);
  else if (E <= 512)
    MOE_TOPK(16);
  else if (E <= 896)
    MOE_TOPK(28);
  else
    MOE_TOPK(32);
#undef MOE_TOPK
  return static_cast<int>(cudaGetLastError());
}

int launch_route_merge(const float* logits, const uint64_t* cand, const float* tile_max, int T,
                       int E, int k, int NT, int32_t* idx, float* gate, float* partials,
                       cudaStream_t s) {
  const int grid = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
#define MOE_MERGE(V) \
  route_merge_kernel<V><<<grid, 256, 0, s>>>(logits, cand, tile_max, T, E, k, NT, idx, gate, \
                                             partials)
  if (E <= 64)
    MOE_MERGE(2);
  else if (E <= 128)
    MOE_MERGE(4);
  else if (E <= 256)
    MOE_MERGE(8);
  else if (E <= 512)
    MOE_MERGE(16);
  else if (E <= 896)
    MOE_MERGE(28);
  else
    MOE_MERGE(32);
#undef MOE_MERGE
  return static_cast<int>(cudaGetLastError());
}

int launch_aux_loss(const int32_t* counts, const float* partials, int n_partials, int T, int k,
                    int E, float* aux_out, float* block_terms, cudaStream_t s) {
  const int nb = (E + 31) / 32;
  aux_stage1_kernel<<<nb, 1024, 0, s>>>(counts, partials, n_partials, T, k, E, block_terms);
  aux_stage2_kernel<<<1, 32, 0, s>>>(block_terms, nb, E, aux_out);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace moe

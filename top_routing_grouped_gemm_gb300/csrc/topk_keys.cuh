// 64-bit selection keys of (logit, expert) shared by the top-k kernel and the router GEMM's
// fused top-k epilogue: the order of the keys is the selection order (larger logit first,
// equal logits -> lower expert index first).
#pragma once

#include <stdint.h>

namespace moe {

// Order-preserving 64-bit key of (logit, expert): larger logit -> larger key, and for equal
// logits the lower expert index -> larger key.  -0.0 and +0.0 compare equal as floats, so
// both map to the key of +0.0.  No real key is 0 (the index field is at least
// 0x7FFFFFFF - 1023), so 0 marks an empty slot.
__device__ __forceinline__ uint64_t sel_key(float v, int e) {
  uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(0x7FFFFFFF - e);
}

__device__ __forceinline__ float key_value(uint64_t key) {
  uint32_t u = static_cast<uint32_t>(key >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

__device__ __forceinline__ int key_expert(uint64_t key) {
  return 0x7FFFFFFF - static_cast<int>(static_cast<uint32_t>(key));
}

// Warp maximum of 64-bit keys as two 32-bit warp reductions: the largest high word, then
// the largest low word among the lanes holding that high word (lexicographic = unsigned
// 64-bit order).
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
  const uint32_t hi = static_cast<uint32_t>(v >> 32);
  const uint32_t m_hi = __reduce_max_sync(0xffffffffu, hi);
  const uint32_t m_lo =
      __reduce_max_sync(0xffffffffu, hi == m_hi ? static_cast<uint32_t>(v) : 0u);
  return (static_cast<uint64_t>(m_hi) << 32) | m_lo;
}

// Insert `key` into the descending list top[0 .. K-1] (fully unrolled compare-exchange
// chain, so the list stays in registers).
template <int K>
__device__ __forceinline__ void topk_insert(uint64_t (&top)[K], uint64_t key) {
  if (key <= top[K - 1]) return;
  top[K - 1] = key;
#pragma unroll
  for (int q = K - 1; q > 0; --q) {
    const uint64_t a = top[q - 1], b = top[q];
    const bool sw = b > a;
    top[q - 1] = sw ? b : a;
    top[q] = sw ? a : b;
  }
}

// Compare-exchange keeping the larger value first (min/max pairs: no branches).
__host__ __device__ __forceinline__ void cx_desc(float& a, float& b) {
  const float hi = fmaxf(a, b), lo = fminf(a, b);
  a = hi;
  b = lo;
}

// Bitonic sorting network on 16 values in registers, descending (80 compare-exchanges in 10
// stages of 8 independent ones).
__host__ __device__ __forceinline__ void sort16_desc(float (&v)[16]) {
#pragma unroll
  for (int k = 2; k <= 16; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int l = i ^ j;
        if (l > i) {
          if ((i & k) == 0 || k == 16) cx_desc(v[i], v[l]);
          else cx_desc(v[l], v[i]);
        }
      }
    }
  }
}

// best <- the 16 largest of best ∪ v (both sorted descending; result sorted descending):
// the elementwise maximum of best and reversed v is a bitonic sequence holding the 16
// largest values, which a 4-stage bitonic merger sorts.
__host__ __device__ __forceinline__ void merge16_desc(float (&best)[16], const float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) best[i] = fmaxf(best[i], v[15 - i]);
#pragma unroll
  for (int j = 8; j > 0; j >>= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int l = i ^ j;
      if (l > i) cx_desc(best[i], best[l]);
    }
  }
}

}  // namespace moe

// Dispatch (count, scan, capacity clip, arrival-ordered permutation, gather), combine,
// their backward counterparts, and the router backward.
//
// "Adapting Ultra-Large MoE Models: Engineering Practices and Optimization Pathways",
// section 3.3: a capacity limit per expert, excess tokens dropped, and the tokens each
// expert receives organised into regular GEMM batches.  "Trillion-Parameter MoE Model
// Training Adaptation: Full-Stack Optimization Practices", section 3 "Communication" and
// section 4.3: tokens are permuted by routing result, the experts run as grouped GEMMs, and
// the results are unpermuted.
//
// Determinism: positions come from sequential per-chunk counting in (token, rank) order and
// an exclusive scan over chunks, so no result depends on the order of atomic operations.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "route.h"

namespace moe {

namespace {

__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* sm, int* total) {
  // blockDim.x == 1024
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = sm[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sm[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int warp_excl = warp ? sm[warp - 1] : 0;
  *total = sm[31];
  return warp_excl + x - v;
}

// Pass 1: each warp counts one chunk of kDispatchChunk tokens, in (token, rank) order, and
// records every slot's rank among the chunk's slots routed to the same expert.  The chunk's
// expert ids are loaded up front (lane j holds rank j of every token of the chunk).
constexpr int kCountWarps = 8;
__global__ void __launch_bounds__(256) dispatch_count_kernel(
    const int32_t* __restrict__ idx, int T, int E, int k, int32_t* __restrict__ local_rank,
    int32_t* __restrict__ chunk_cnt, int32_t* dev_status) {
  extern __shared__ int cnt_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kCountWarps + warp;
  const int nch = dispatch_num_chunks(T);
  if (c >= nch) return;
  int* cnt = cnt_smem + warp * E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  const int t0 = c * kDispatchChunk;
  int ev[kDispatchChunk];
#pragma unroll
  for (int i = 0; i < kDispatchChunk; ++i) {
    const int t = t0 + i;
    ev[i] = (lane < k && t < T) ? idx[static_cast<size_t>(t) * k + lane] : -1;
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < kDispatchChunk; ++i) {
    const int t = t0 + i;
    if (t >= T) break;
    const bool act = lane < k;
    int e = ev[i];
    if (act && (e < 0 || e >= E)) {
      report_status(dev_status, MOE_ERR_BAD_INDEX);
      e = -1;
    }
    const unsigned live = __ballot_sync(0xffffffffu, act && e >= 0);
    if (act && e >= 0) {
      // a token may repeat an expert only in caller-made input; ranks then follow j order
      const unsigned grp = __match_any_sync(live, e);
      const int before = __popc(grp & ((1u << lane) - 1u));
      const int base = cnt[e];
      __syncwarp(live);
      local_rank[static_cast<size_t>(t) * k + lane] = base + before;
      if (lane == 31 - __clz(grp)) cnt[e] = base + __popc(grp);
    } else if (act) {
      local_rank[static_cast<size_t>(t) * k + lane] = -1;
    }
    __syncwarp();
  }
  for (int e = lane; e < E; e += 32) chunk_cnt[static_cast<size_t>(c) * E + e] = cnt[e];
}

// Pass 2: per expert, exclusive scan of the chunk counts (in place -> chunk bases) and the
// pre-drop totals.  Block (32 experts) x (32 parts of the chunk range).
__global__ void __launch_bounds__(1024) dispatch_scan_chunks_kernel(
    int32_t* __restrict__ chunk_cnt, int nch, int E, int32_t* __restrict__ counts) {
  __shared__ int sm[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + tx;
  const int per = (nch + 31) / 32;
  const int c0 = ty * per, c1 = min(nch, c0 + per);
  int sum = 0;
  if (e < E)
    for (int c = c0; c < c1; ++c) sum += chunk_cnt[static_cast<size_t>(c) * E + e];
  sm[ty][tx] = sum;
  __syncthreads();
  if (ty == 0 && e < E) {
    int run = 0;
    for (int p = 0; p < 32; ++p) {
      const int v = sm[p][tx];
      sm[p][tx] = run;
      run += v;
    }
    counts[e] = run;
  }
  __syncthreads();
  if (e < E) {
    int run = sm[ty][tx];
    for (int c = c0; c < c1; ++c) {
      const size_t i = static_cast<size_t>(c) * E + e;
      const int v = chunk_cnt[i];
      chunk_cnt[i] = run;
      run += v;
    }
  }
}

// Pass 3: kept counts, expert offsets, n_kept / n_dropped.  One block, thread = expert.
// pos_base[e] (may be null): slots of expert e that arrived before this batch's first token
// (held elsewhere); they occupy the first places of the expert's capacity.
__global__ void __launch_bounds__(1024) dispatch_offsets_kernel(
    const int32_t* __restrict__ counts, const int32_t* __restrict__ pos_base, int E,
    int capacity, int slots, int32_t* __restrict__ offsets,
    int32_t* __restrict__ n_kept_dropped) {
  __shared__ int sm[32];
  const int e = threadIdx.x;
  int kept = 0;
  if (e < E) {
    const int room = capacity < 0 ? counts[e]
                                  : max(0, capacity - (pos_base ? max(0, pos_base[e]) : 0));
    kept = min(counts[e], room);
  }
  int total;
  const int excl = block_exclusive_scan_1024(kept, sm, &total);
  if (e < E) offsets[e] = excl;
  if (e == 0) {
    offsets[E] = total;
    n_kept_dropped[0] = total;
    n_kept_dropped[1] = slots - total;
  }
}

// Pass 4: final rows, both index maps, and the gather x -> x_perm.  One block per token:
// warp 0 resolves the k rows, then every thread moves 16-byte vectors of x[t], read once
// and written to each kept row.
constexpr int kRowThreads = 128;
__global__ void __launch_bounds__(kRowThreads) dispatch_scatter_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ local_rank,
    const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ n_kept_dropped, const int32_t* __restrict__ pos_base,
    const float* __restrict__ gate, const uint4* __restrict__ x, int T, int d, int E, int k,
    int capacity, int32_t* __restrict__ slot_row, int32_t* __restrict__ row_slot,
    float* __restrict__ gate_perm, uint4* __restrict__ x_perm) {
  __shared__ int rows[32];
  const int t = blockIdx.x;
  const int slots = T * k;
  {
    // rows past n_kept are marked unused (disjoint from the rows written below)
    const int n_kept = n_kept_dropped[0];
    for (int r = n_kept + blockIdx.x * blockDim.x + threadIdx.x; r < slots;
         r += gridDim.x * blockDim.x)
      row_slot[r] = -1;
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int row = -1;
    if (lane < k) {
      const int slot = t * k + lane;
      const int e = idx[slot];
      const int lr = local_rank[slot];
      if (e >= 0 && e < E && lr >= 0) {
        const int pos = chunk_base[static_cast<size_t>(t / kDispatchChunk) * E + e] + lr;
        const int base = pos_base ? max(0, pos_base[e]) : 0;
        if (capacity < 0 || base + pos < capacity) row = offsets[e] + pos;
      }
      slot_row[slot] = row;
      if (row >= 0) {
        row_slot[row] = slot;
        if (gate_perm) gate_perm[row] = gate[slot];
      }
    }
    rows[lane] = row;
  }
  if (x_perm == nullptr) return;  // index maps only (the GEMM gathers the rows itself)
  __syncthreads();
  const int nvec = d / 8;
  const uint4* src = x + static_cast<size_t>(t) * nvec;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const uint4 val = src[v];
    for (int j = 0; j < k; ++j) {
      const int r = rows[j];
      if (r >= 0) x_perm[static_cast<size_t>(r) * nvec + v] = val;
    }
  }
}

// m-tiles of 128 rows per group and their prefix (tile_off), and the prefix of m-tile pairs
// (pair_off, for 256-row tiles).  Malformed offsets disable the group and are reported.
__global__ void __launch_bounds__(1024) tile_schedule_kernel(const int32_t* __restrict__ offsets,
                                                             int E, int rows_max,
                                                             int32_t* __restrict__ tile_off,
                                                             int32_t* __restrict__ pair_off,
                                                             int32_t* dev_status) {
  __shared__ int sm[32];
  const int e = threadIdx.x;
  int mt = 0;
  if (e < E) {
    const int lo = offsets[e], hi = offsets[e + 1];
    if (lo < 0 || hi < lo || hi > rows_max) {
      report_status(dev_status, MOE_ERR_BAD_INDEX);
    } else {
      mt = (hi - lo + kBM - 1) / kBM;
    }
  }
  int total;
  const int excl = block_exclusive_scan_1024(mt, sm, &total);
  if (e < E) tile_off[e] = excl;
  if (e == 0) tile_off[E] = total;
  __syncthreads();
  int total_pairs;
  const int pexcl = block_exclusive_scan_1024((mt + 1) >> 1, sm, &total_pairs);
  if (e < E) pair_off[e] = pexcl;
  if (e == 0) pair_off[E] = total_pairs;
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v, float scale) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    acc[2 * i] += scale * f.x;
    acc[2 * i + 1] += scale * f.y;
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&a)[8]) {
  uint4 o;
  o.x = pack_bf16x2(a[0], a[1]);
  o.y = pack_bf16x2(a[2], a[3]);
  o.z = pack_bf16x2(a[4], a[5]);
  o.w = pack_bf16x2(a[6], a[7]);
  return o;
}

// y[t] = sum_j y_perm[slot_row[t*k+j]] (kept slots, rank order, fp32) -> bf16.  One block
// per token, one 16-byte vector per thread: the k row loads are independent.
__global__ void __launch_bounds__(kRowThreads) combine_kernel(const uint4* __restrict__ y_perm,
                                                              const int32_t* __restrict__ slot_row,
                                                              int T, int d, int k,
                                                              uint4* __restrict__ y) {
  __shared__ int rows[32];
  const int t = blockIdx.x;
  if (threadIdx.x < 32) rows[threadIdx.x] = threadIdx.x < k ? slot_row[static_cast<size_t>(t) * k + threadIdx.x] : -1;
  __syncthreads();
  const int nvec = d / 8;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const int r = rows[j];
      if (r >= 0) add_bf16x8(acc, y_perm[static_cast<size_t>(r) * nvec + v], 1.f);
    }
    y[static_cast<size_t>(t) * nvec + v] = pack_bf16x8(acc);
  }
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per slot:  dz_perm[row] = g * dy[t];  dgate[slot] = <dy[t], y_perm[row]> / g
// (kept slots; y_perm = g * o, so this is <dy, o> up to the bf16 rounding of y_perm), else 0.
__global__ void __launch_bounds__(256) combine_bwd_kernel(
    const uint4* __restrict__ dy, const uint4* __restrict__ y_perm,
    const int32_t* __restrict__ slot_row, const float* __restrict__ gate, int T, int d, int k,
    uint4* __restrict__ dz_perm, float* __restrict__ dgate) {
  const int lane = threadIdx.x & 31;
  const size_t slot = static_cast<size_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (slot >= static_cast<size_t>(T) * k) return;
  const int r = slot_row[slot];
  if (r < 0) {
    if (lane == 0) dgate[slot] = 0.f;
    return;
  }
  const int t = static_cast<int>(slot / k);
  const int nvec = d / 8;
  const uint4* dyr = dy + static_cast<size_t>(t) * nvec;
  const float g = gate[slot];
  float dot = 0.f;
  for (int v = lane; v < nvec; v += 32) {
    float fa[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    add_bf16x8(fa, dyr[v], 1.f);
    if (y_perm) {
      float fb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      add_bf16x8(fb, y_perm[static_cast<size_t>(r) * nvec + v], 1.f);
#pragma unroll
      for (int i = 0; i < 8; ++i) dot += fa[i] * fb[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) fa[i] *= g;
    dz_perm[static_cast<size_t>(r) * nvec + v] = pack_bf16x8(fa);
  }
  if (y_perm) dot = warp_sum_f(dot);
  // without y_perm the kept slots' gate gradients come later (expert backward): zero here
  if (lane == 0 && dgate) dgate[slot] = (y_perm && g > 0.f) ? dot / g : 0.f;
}

// dgate[row_slot[r]] = (sum over the dh GEMM's n-tiles of <dh, h> of row r) / gate, for the
// kept rows r < offsets[E] (in a fixed order: deterministic).
__global__ void dgate_finalize_kernel(const float* __restrict__ part, int n_tiles,
                                      const int32_t* __restrict__ row_slot,
                                      const float* __restrict__ gate,
                                      const int32_t* __restrict__ n_rows, int rows_max,
                                      float* __restrict__ dgate) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= rows_max || r >= __ldg(n_rows)) return;
  const int slot = row_slot[r];
  if (slot < 0) return;
  float sum = 0.f;
  for (int n = 0; n < n_tiles; ++n) sum += part[static_cast<size_t>(r) * n_tiles + n];
  const float g = gate[slot];
  dgate[slot] = g > 0.f ? sum / g : 0.f;
}

// dx[t] = sum over kept slots of dx_perm rows (fp32, overwritten).  One block per token.
__global__ void __launch_bounds__(kRowThreads) dispatch_bwd_kernel(
    const uint4* __restrict__ dx_perm, const int32_t* __restrict__ slot_row, int T, int d, int k,
    float4* __restrict__ dx) {
  __shared__ int rows[32];
  const int t = blockIdx.x;
  if (threadIdx.x < 32) rows[threadIdx.x] = threadIdx.x < k ? slot_row[static_cast<size_t>(t) * k + threadIdx.x] : -1;
  __syncthreads();
  const int nvec = d / 8;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const int r = rows[j];
      if (r >= 0) add_bf16x8(acc, dx_perm[static_cast<size_t>(r) * nvec + v], 1.f);
    }
    float4* o = dx + (static_cast<size_t>(t) * nvec + v) * 2;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// Both backward paths into dx in one pass, one block per token: dx[t] = sum_j dx_perm[row_j]
// (the expert path, rank order) + sum_j c_j W_r[e_j] (the gate path, c_j as below), in the
// same order of operations as dispatch_bwd_kernel followed by route_bwd_kernel.
__global__ void __launch_bounds__(kRowThreads) dispatch_route_bwd_kernel(
    const uint4* __restrict__ dx_perm, const int32_t* __restrict__ slot_row,
    const int32_t* __restrict__ idx, const float* __restrict__ gate,
    const float* __restrict__ dgate, const float4* __restrict__ w_router, int T, int d, int E,
    int k, float4* __restrict__ dx) {
  __shared__ int rows[32];
  __shared__ float cs[32];
  __shared__ int es[32];
  const int t = blockIdx.x;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float g = 0.f, dg = 0.f;
    int e = 0, r = -1;
    if (lane < k) {
      const size_t slot = static_cast<size_t>(t) * k + lane;
      r = slot_row[slot];
      g = gate[slot];
      dg = dgate[slot];
      e = idx[slot];
      if (e < 0 || e >= E) { e = 0; g = 0.f; }
    }
    const float sgd = warp_sum_f(g * dg);
    rows[lane] = r;
    cs[lane] = g * (dg - sgd);
    es[lane] = e;
  }
  __syncthreads();
  const int nvec = d / 8;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const int r = rows[j];
      if (r >= 0) add_bf16x8(acc, dx_perm[static_cast<size_t>(r) * nvec + v], 1.f);
    }
    float4 a = make_float4(acc[0], acc[1], acc[2], acc[3]);
    float4 b = make_float4(acc[4], acc[5], acc[6], acc[7]);
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const float cj = cs[j];
      const float4 w0 = __ldg(&w_router[static_cast<size_t>(es[j]) * (d / 4) + 2 * v]);
      const float4 w1 = __ldg(&w_router[static_cast<size_t>(es[j]) * (d / 4) + 2 * v + 1]);
      a.x += cj * w0.x; a.y += cj * w0.y; a.z += cj * w0.z; a.w += cj * w0.w;
      b.x += cj * w1.x; b.y += cj * w1.y; b.z += cj * w1.z; b.w += cj * w1.w;
    }
    float4* o = dx + (static_cast<size_t>(t) * nvec + v) * 2;
    o[0] = a;
    o[1] = b;
  }
}

// dx[t] += sum_j c_j W_r[e_j],  c_j = g_j (dg_j - sum_i g_i dg_i).  One block per token.
__global__ void __launch_bounds__(kRowThreads) route_bwd_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ gate,
    const float* __restrict__ dgate, const float4* __restrict__ w_router, int T, int d, int E,
    int k, float4* __restrict__ dx) {
  __shared__ float cs[32];
  __shared__ int es[32];
  const int t = blockIdx.x;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float g = 0.f, dg = 0.f;
    int e = 0;
    if (lane < k) {
      const size_t slot = static_cast<size_t>(t) * k + lane;
      g = gate[slot];
      dg = dgate[slot];
      e = idx[slot];
      if (e < 0 || e >= E) { e = 0; g = 0.f; }
    }
    const float sgd = warp_sum_f(g * dg);
    cs[lane] = g * (dg - sgd);
    es[lane] = e;
  }
  __syncthreads();
  const int n4 = d / 4;
  for (int v = threadIdx.x; v < n4; v += blockDim.x) {
    float4 acc = dx[static_cast<size_t>(t) * n4 + v];
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const float cj = cs[j];
      const float4 w = __ldg(&w_router[static_cast<size_t>(es[j]) * n4 + v]);
      acc.x += cj * w.x;
      acc.y += cj * w.y;
      acc.z += cj * w.z;
      acc.w += cj * w.w;
    }
    dx[static_cast<size_t>(t) * n4 + v] = acc;
  }
}

// ---------------------------------------------------------------- overflow remapping
//
// "Adapting Ultra-Large MoE Models: Engineering Practices and Optimization Pathways",
// section 3.3: tokens beyond an expert's capacity are remapped or dropped.  Pass 0 is the
// plain dispatch; in round q = 1 .. rounds every slot (t, j) still unplaced proposes its
// token's preference rank j + q k (alt[t][(q-1) k + j]), and each expert takes proposals in
// arrival order into its remaining capacity.  One count / scan / decide launch triple per
// pass keeps every decision deterministic (positions from sequential chunk counting and
// scans, never from the order of atomics).

// Pass q, step 1: per 16-token chunk, the arrival rank of every proposing slot among the
// chunk's proposals to the same expert, and the chunk's per-expert proposal counts.
__global__ void __launch_bounds__(256) remap_count_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ alt,
    const int32_t* __restrict__ state, int q, int rounds, int T, int E, int k,
    int32_t* __restrict__ local_rank, int32_t* __restrict__ chunk_cnt, int32_t* dev_status) {
  extern __shared__ int cnt_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kCountWarps + warp;
  const int nch = dispatch_num_chunks(T);
  if (c >= nch) return;
  int* cnt = cnt_smem + warp * E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const int t0 = c * kDispatchChunk;
  for (int i = 0; i < kDispatchChunk; ++i) {
    const int t = t0 + i;
    if (t >= T) break;
    const bool act = lane < k;
    const size_t slot = static_cast<size_t>(t) * k + lane;
    int e = -1;
    if (act) {
      if (q == 0) {
        e = idx[slot];
      } else if (state[slot] < 0) {
        e = alt[static_cast<size_t>(t) * rounds * k + (q - 1) * k + lane];
      }
      if (e >= E || (q == 0 && e < 0)) {
        report_status(dev_status, MOE_ERR_BAD_INDEX);
        e = -1;
      }
    }
    const unsigned live = __ballot_sync(0xffffffffu, act && e >= 0);
    if (act && e >= 0) {
      const unsigned grp = __match_any_sync(live, e);
      const int before = __popc(grp & ((1u << lane) - 1u));
      const int base = cnt[e];
      __syncwarp(live);
      local_rank[slot] = base + before;
      if (lane == 31 - __clz(grp)) cnt[e] = base + __popc(grp);
    } else if (act) {
      local_rank[slot] = -1;
    }
    __syncwarp();
  }
  for (int e = lane; e < E; e += 32) chunk_cnt[static_cast<size_t>(c) * E + e] = cnt[e];
}

// Pass q, step 2: per expert, exclusive scan of the chunk counts (in place) and the pass
// total; the expert's places held before this pass (held_before) and after it (held).
// counts (pass 0 only) receives the pre-drop totals of the original selection.
__global__ void __launch_bounds__(1024) remap_scan_kernel(
    int32_t* __restrict__ chunk_cnt, int nch, int E, int q, int capacity,
    int32_t* __restrict__ held, int32_t* __restrict__ held_before,
    int32_t* __restrict__ counts) {
  __shared__ int sm[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + tx;
  const int per = (nch + 31) / 32;
  const int c0 = ty * per, c1 = min(nch, c0 + per);
  int sum = 0;
  if (e < E)
    for (int c = c0; c < c1; ++c) sum += chunk_cnt[static_cast<size_t>(c) * E + e];
  sm[ty][tx] = sum;
  __syncthreads();
  if (ty == 0 && e < E) {
    int run = 0;
    for (int pp = 0; pp < 32; ++pp) {
      const int v = sm[pp][tx];
      sm[pp][tx] = run;
      run += v;
    }
    const int h = q == 0 ? 0 : held[e];
    held_before[e] = h;
    held[e] = capacity < 0 ? h + run : min(capacity, h + run);
    if (q == 0) counts[e] = run;
  }
  __syncthreads();
  if (e < E) {
    int run = sm[ty][tx];
    for (int c = c0; c < c1; ++c) {
      const size_t i = static_cast<size_t>(c) * E + e;
      const int v = chunk_cnt[i];
      chunk_cnt[i] = run;
      run += v;
    }
  }
}

// Pass q, step 3: a proposing slot is placed iff its expert's places held before the pass
// plus its arrival position stay below the capacity; it then records the expert and its
// index among the expert's rows.  Pass 0 also initialises every slot's state.
__global__ void remap_decide_kernel(const int32_t* __restrict__ idx,
                                    const int32_t* __restrict__ alt,
                                    const int32_t* __restrict__ local_rank,
                                    const int32_t* __restrict__ chunk_base,
                                    const int32_t* __restrict__ held_before, int q, int rounds,
                                    int T, int E, int k, int capacity,
                                    int32_t* __restrict__ state,
                                    int32_t* __restrict__ slot_expert,
                                    int32_t* __restrict__ slot_index) {
  const long long slots = static_cast<long long>(T) * k;
  for (long long s = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; s < slots;
       s += static_cast<long long>(gridDim.x) * blockDim.x) {
    if (q > 0 && state[s] >= 0) continue;
    const int lr = local_rank[s];
    const int t = static_cast<int>(s / k), j = static_cast<int>(s - static_cast<long long>(t) * k);
    bool placed = false;
    int e = -1, index = -1;
    if (lr >= 0) {
      e = q == 0 ? idx[s] : alt[static_cast<size_t>(t) * rounds * k + (q - 1) * k + j];
      index = held_before[e] + chunk_base[static_cast<size_t>(t / kDispatchChunk) * E + e] + lr;
      placed = capacity < 0 || index < capacity;
    }
    if (placed) {
      state[s] = q;
      slot_expert[s] = e;
      slot_index[s] = index;
    } else if (q == 0) {
      state[s] = -1;
      slot_expert[s] = -1;
    }
  }
}

// Final rows, both index maps and the gather x -> x_perm (one block per token).
__global__ void __launch_bounds__(kRowThreads) remap_scatter_kernel(
    const int32_t* __restrict__ slot_expert, const int32_t* __restrict__ slot_index,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ n_kept_dropped,
    const uint4* __restrict__ x, int T, int d, int k, int32_t* __restrict__ slot_row,
    int32_t* __restrict__ row_slot, uint4* __restrict__ x_perm) {
  __shared__ int rows[32];
  const int t = blockIdx.x;
  const int slots = T * k;
  {
    const int n_kept = n_kept_dropped[0];
    for (int r = n_kept + blockIdx.x * blockDim.x + threadIdx.x; r < slots;
         r += gridDim.x * blockDim.x)
      row_slot[r] = -1;
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int row = -1;
    if (lane < k) {
      const int slot = t * k + lane;
      const int e = slot_expert[slot];
      if (e >= 0) row = offsets[e] + slot_index[slot];
      slot_row[slot] = row;
      if (row >= 0) row_slot[row] = slot;
    }
    rows[lane] = row;
  }
  if (x_perm == nullptr) return;
  __syncthreads();
  const int nvec = d / 8;
  const uint4* src = x + static_cast<size_t>(t) * nvec;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const uint4 val = src[v];
    for (int j = 0; j < k; ++j) {
      const int r = rows[j];
      if (r >= 0) x_perm[static_cast<size_t>(r) * nvec + v] = val;
    }
  }
}

// ---------------------------------------------------------------- expert parallelism
//
// "Trillion-Parameter MoE Model Training Adaptation: Full-Stack Optimization Practices",
// section 3 "Communication" and section 4.1: experts split evenly over the ranks of the
// expert-parallel group; tokens permuted by routing result are sent with an all-to-all to
// the ranks holding their experts, computed there as grouped GEMMs, and returned.

__global__ void zero_i32_kernel(int32_t* __restrict__ v, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    v[i] = 0;
}

// counts[e] += number of slots routed to e (integer atomics: the totals do not depend on
// their order).  Per-block shared-memory histograms, one global add per (block, expert).
__global__ void __launch_bounds__(1024) expert_histogram_kernel(
    const int32_t* __restrict__ idx, long long slots, int E, int32_t* __restrict__ counts,
    int32_t* dev_status) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < slots;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int e = idx[i];
    if (e < 0 || e >= E) {
      report_status(dev_status, MOE_ERR_BAD_INDEX);
      continue;
    }
    atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (hist[e]) atomicAdd(&counts[e], hist[e]);
}

// Rows move between the two layouts of an expert-parallel exchange.  kept[s * El + e] rows
// belong to (source s, local expert e).  Source-major layout: blocks ordered (s, e) (what
// the all-to-all delivers); expert-major layout: blocks ordered (e, s) (one contiguous
// group per expert for the grouped GEMM, sources in rank order = global arrival order).
// to_expert = 1 moves source-major -> expert-major, 0 the reverse.  One block per (s, e)
// pair (several when its rows are many); each finds its two block offsets by summing the
// kept counts before it in either order.
__global__ void __launch_bounds__(256) ep_regroup_kernel(
    const uint4* __restrict__ src, const float* __restrict__ gsrc,
    const int32_t* __restrict__ kept, int P, int El, int nvec, int to_expert, int parts,
    uint4* __restrict__ dst, float* __restrict__ gdst, int32_t* __restrict__ expert_offsets) {
  __shared__ long long red[2][8];
  const int pair = blockIdx.x / parts;
  const int part = blockIdx.x - pair * parts;
  const int s = pair / El, e = pair - s * El;
  long long off_se = 0, off_es = 0;
  for (int i = threadIdx.x; i < P * El; i += blockDim.x) {
    const int si = i / El, ei = i - si * El;
    const long long c = kept[i];
    if (i < pair) off_se += c;                       // (si, ei) before (s, e), source-major
    if (ei < e || (ei == e && si < s)) off_es += c;  // (ei, si) before (e, s), expert-major
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    off_se += __shfl_xor_sync(0xffffffffu, off_se, o);
    off_es += __shfl_xor_sync(0xffffffffu, off_es, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = off_se;
    red[1][threadIdx.x >> 5] = off_es;
  }
  __syncthreads();
  off_se = 0;
  off_es = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    off_se += red[0][w];
    off_es += red[1][w];
  }
  const int rows = kept[pair];
  if (expert_offsets && s == 0 && part == 0) {
    expert_offsets[e] = static_cast<int32_t>(off_es);
    if (e == El - 1 && threadIdx.x == 0) {
      long long total = 0;
      for (int i = 0; i < P * El; ++i) total += kept[i];
      expert_offsets[El] = static_cast<int32_t>(total);
    }
  }
  const long long from = to_expert ? off_se : off_es;
  const long long to = to_expert ? off_es : off_se;
  const long long n = static_cast<long long>(rows) * nvec;
  for (long long i = part * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(parts) * blockDim.x)
    dst[to * nvec + i] = src[from * nvec + i];
  if (gsrc && gdst)
    for (int i = part * blockDim.x + threadIdx.x; i < rows; i += parts * blockDim.x)
      gdst[to + i] = gsrc[from + i];
}

// Fused combine set-up: one warp per token counts its kept slots, sets its per-n-tile
// counters to that count, and zeroes y[t] when nothing was kept (no finisher will write it).
__global__ void __launch_bounds__(256) combine_prepare_kernel(
    const int32_t* __restrict__ slot_row, int T, int k, int n_tiles, int d,
    int32_t* __restrict__ comb_cnt, uint4* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const bool kept = lane < k && slot_row[static_cast<size_t>(t) * k + lane] >= 0;
  const int n = __popc(__ballot_sync(0xffffffffu, kept));
  for (int i = lane; i < n_tiles; i += 32) comb_cnt[static_cast<size_t>(t) * n_tiles + i] = n;
  if (n == 0) {
    const int nvec = d / 8;
    for (int v = lane; v < nvec; v += 32) y[static_cast<size_t>(t) * nvec + v] = make_uint4(0u, 0u, 0u, 0u);
  }
}

int grid_for_slots(long long slots) { return static_cast<int>((slots + 7) / 8); }

}  // namespace

int launch_dispatch(const int32_t* idx, const __nv_bfloat16* x, int T, int d, int E, int k,
                    int capacity, int32_t* counts, int32_t* offsets, int32_t* slot_row,
                    int32_t* row_slot, int32_t* n_kept_dropped, __nv_bfloat16* x_perm,
                    int32_t* local_rank, int32_t* chunk_cnt, int32_t* dev_status,
                    cudaStream_t s, const int32_t* pos_base, const float* gate,
                    float* gate_perm) {
  const int nch = dispatch_num_chunks(T);
  dispatch_count_kernel<<<(nch + kCountWarps - 1) / kCountWarps, 32 * kCountWarps,
                          kCountWarps * E * sizeof(int), s>>>(idx, T, E, k, local_rank, chunk_cnt,
                                                              dev_status);
  dispatch_scan_chunks_kernel<<<(E + 31) / 32, 1024, 0, s>>>(chunk_cnt, nch, E, counts);
  dispatch_offsets_kernel<<<1, 1024, 0, s>>>(counts, pos_base, E, capacity, T * k, offsets,
                                             n_kept_dropped);
  dispatch_scatter_kernel<<<T, kRowThreads, 0, s>>>(
      idx, local_rank, chunk_cnt, offsets, n_kept_dropped, pos_base, gate,
      reinterpret_cast<const uint4*>(x), T, d, E, k, capacity, slot_row, row_slot, gate_perm,
      reinterpret_cast<uint4*>(x_perm));
  return static_cast<int>(cudaGetLastError());
}

int launch_expert_counts(const int32_t* idx, long long slots, int E, int32_t* counts,
                         int32_t* dev_status, cudaStream_t s) {
  zero_i32_kernel<<<1, 1024, 0, s>>>(counts, E);
  const int blocks = static_cast<int>(std::min<long long>((slots + 1023) / 1024, 2 * 152));
  expert_histogram_kernel<<<std::max(blocks, 1), 1024, E * sizeof(int), s>>>(idx, slots, E,
                                                                             counts, dev_status);
  return static_cast<int>(cudaGetLastError());
}

int launch_ep_regroup(const __nv_bfloat16* src, const float* gsrc, const int32_t* kept, int P,
                      int El, int d, int to_expert, long long rows_hint, __nv_bfloat16* dst,
                      float* gdst, int32_t* expert_offsets, cudaStream_t s) {
  // enough blocks per (source, expert) pair to cover about two waves for the expected rows
  const long long pairs = static_cast<long long>(P) * El;
  const long long per_pair = std::max<long long>(1, rows_hint / std::max<long long>(1, pairs));
  const int parts = static_cast<int>(std::min<long long>(8, std::max<long long>(1, per_pair / 64)));
  ep_regroup_kernel<<<static_cast<int>(pairs * parts), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(src), gsrc, kept, P, El, d / 8, to_expert, parts,
      reinterpret_cast<uint4*>(dst), gdst, expert_offsets);
  return static_cast<int>(cudaGetLastError());
}

size_t remap_ws_bytes(int T, int k, int E, int rounds) {
  const size_t slots = static_cast<size_t>(T) * k;
  return up256(slots * 4) * 3 +                                        // local_rank, state, index
         up256(static_cast<size_t>(dispatch_num_chunks(T)) * E * 4) +  // chunk counts
         up256(static_cast<size_t>(E) * 4) * 2 +                       // held, held_before
         up256(slots * 4);                                             // slot_expert (if not given)
}

int launch_dispatch_remap(const int32_t* idx, const int32_t* alt, int rounds,
                          const __nv_bfloat16* x, int T, int d, int E, int k, int capacity,
                          int32_t* counts, int32_t* offsets, int32_t* slot_row,
                          int32_t* row_slot, int32_t* slot_expert, int32_t* n_kept_dropped,
                          __nv_bfloat16* x_perm, void* ws, int32_t* dev_status,
                          cudaStream_t s) {
  const size_t slots = static_cast<size_t>(T) * k;
  const int nch = dispatch_num_chunks(T);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* local_rank = reinterpret_cast<int32_t*>(w);  w += up256(slots * 4);
  int32_t* state = reinterpret_cast<int32_t*>(w);       w += up256(slots * 4);
  int32_t* slot_idx = reinterpret_cast<int32_t*>(w);    w += up256(slots * 4);
  int32_t* chunk_cnt = reinterpret_cast<int32_t*>(w);   w += up256(static_cast<size_t>(nch) * E * 4);
  int32_t* held = reinterpret_cast<int32_t*>(w);        w += up256(static_cast<size_t>(E) * 4);
  int32_t* held_before = reinterpret_cast<int32_t*>(w); w += up256(static_cast<size_t>(E) * 4);
  if (slot_expert == nullptr) slot_expert = reinterpret_cast<int32_t*>(w);
  const int decide_blocks = static_cast<int>(std::min<size_t>((slots + 255) / 256, 8 * 152));
  for (int q = 0; q <= rounds; ++q) {
    remap_count_kernel<<<(nch + kCountWarps - 1) / kCountWarps, 32 * kCountWarps,
                         kCountWarps * E * sizeof(int), s>>>(idx, alt, state, q, rounds, T, E, k,
                                                             local_rank, chunk_cnt, dev_status);
    remap_scan_kernel<<<(E + 31) / 32, 1024, 0, s>>>(chunk_cnt, nch, E, q, capacity, held,
                                                    held_before, counts);
    remap_decide_kernel<<<decide_blocks, 256, 0, s>>>(idx, alt, local_rank, chunk_cnt,
                                                      held_before, q, rounds, T, E, k, capacity,
                                                      state, slot_expert, slot_idx);
  }
  dispatch_offsets_kernel<<<1, 1024, 0, s>>>(held, nullptr, E, -1, T * k, offsets,
                                             n_kept_dropped);
  remap_scatter_kernel<<<T, kRowThreads, 0, s>>>(slot_expert, slot_idx, offsets, n_kept_dropped,
                                                 reinterpret_cast<const uint4*>(x), T, d, k,
                                                 slot_row, row_slot,
                                                 reinterpret_cast<uint4*>(x_perm));
  return static_cast<int>(cudaGetLastError());
}

int launch_combine_prepare(const int32_t* slot_row, int T, int k, int n_tiles, int d,
                           int32_t* comb_cnt, __nv_bfloat16* y, cudaStream_t s) {
  combine_prepare_kernel<<<(T + 7) / 8, 256, 0, s>>>(slot_row, T, k, n_tiles, d, comb_cnt,
                                                     reinterpret_cast<uint4*>(y));
  return static_cast<int>(cudaGetLastError());
}

int launch_tile_schedule(const int32_t* offsets, int E, int rows_max, int32_t* tile_off,
                         int32_t* pair_off, int32_t* dev_status, cudaStream_t s) {
  tile_schedule_kernel<<<1, 1024, 0, s>>>(offsets, E, rows_max, tile_off, pair_off,
                                          dev_status);
  return static_cast<int>(cudaGetLastError());
}

int launch_combine(const __nv_bfloat16* y_perm, const int32_t* slot_row, int T, int d, int k,
                   __nv_bfloat16* y, cudaStream_t s) {
  combine_kernel<<<T, kRowThreads, 0, s>>>(reinterpret_cast<const uint4*>(y_perm),
                                                    slot_row, T, d, k,
                                                    reinterpret_cast<uint4*>(y));
  return static_cast<int>(cudaGetLastError());
}

int launch_combine_bwd(const __nv_bfloat16* dy, const __nv_bfloat16* y_perm,
                       const int32_t* slot_row, const float* gate, int T, int d, int k,
                       __nv_bfloat16* dz_perm, float* dgate, cudaStream_t s) {
  combine_bwd_kernel<<<grid_for_slots(static_cast<long long>(T) * k), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(dy), reinterpret_cast<const uint4*>(y_perm), slot_row,
      gate, T, d, k, reinterpret_cast<uint4*>(dz_perm), dgate);
  return static_cast<int>(cudaGetLastError());
}

int launch_dgate_finalize(const float* part, int n_tiles, const int32_t* row_slot,
                          const float* gate, const int32_t* n_rows, int rows_max, float* dgate,
                          cudaStream_t s) {
  dgate_finalize_kernel<<<(rows_max + 255) / 256, 256, 0, s>>>(part, n_tiles, row_slot, gate,
                                                                n_rows, rows_max, dgate);
  return static_cast<int>(cudaGetLastError());
}

int launch_dispatch_bwd(const __nv_bfloat16* dx_perm, const int32_t* slot_row, int T, int d,
                        int k, float* dx, cudaStream_t s) {
  dispatch_bwd_kernel<<<T, kRowThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(dx_perm), slot_row, T, d, k, reinterpret_cast<float4*>(dx));
  return static_cast<int>(cudaGetLastError());
}

int launch_dispatch_route_bwd(const __nv_bfloat16* dx_perm, const int32_t* slot_row,
                              const int32_t* idx, const float* gate, const float* dgate,
                              const float* w_router, int T, int d, int E, int k, float* dx,
                              cudaStream_t s) {
  dispatch_route_bwd_kernel<<<T, kRowThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(dx_perm), slot_row, idx, gate, dgate,
      reinterpret_cast<const float4*>(w_router), T, d, E, k, reinterpret_cast<float4*>(dx));
  return static_cast<int>(cudaGetLastError());
}

int launch_route_bwd(const int32_t* idx, const float* gate, const float* dgate,
                     const float* w_router, int T, int d, int E, int k, float* dx,
                     cudaStream_t s) {
  route_bwd_kernel<<<T, kRowThreads, 0, s>>>(
      idx, gate, dgate, reinterpret_cast<const float4*>(w_router), T, d, E, k,
      reinterpret_cast<float4*>(dx));
  return static_cast<int>(cudaGetLastError());
}

}  // namespace moe

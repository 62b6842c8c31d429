// Launchers of the SIMT kernels (router tail, dispatch, combine, backward helpers).
#pragma once

#include <cuda_bf16.h>

#include <algorithm>

#include "moe_internal.h"

namespace moe {

constexpr int kRouteTokensPerBlock = 8;  // tokens per row of prob_partials
constexpr int kDispatchChunk = 16;        // tokens counted sequentially by one warp

__host__ __device__ inline int route_num_partials(int T) {
  return (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
}
__host__ __device__ inline int dispatch_num_chunks(int T) { return (T + kDispatchChunk - 1) / kDispatchChunk; }

int launch_split_router(const float* w, __nv_bfloat16* hi, __nv_bfloat16* lo, size_t n,
                        cudaStream_t s);
// n_alt > 0 with alt_idx: also the next n_alt preferences of every token (k + n_alt <= 32);
// null idx / gate / partials skip those outputs
int launch_topk_softmax(const float* logits, int T, int E, int k, int32_t* idx, float* gate,
                        float* partials, cudaStream_t s, int n_alt = 0,
                        int32_t* alt_idx = nullptr);
// After the router GEMM's fused top-k epilogue: cand [T, NT, 16] keys, tile_max [T, NT] ->
// top-k, gates, probability partials (k <= 16)
int launch_route_merge(const float* logits, const uint64_t* cand, const float* tile_max, int T,
                       int E, int k, int NT, int32_t* idx, float* gate, float* partials,
                       cudaStream_t s);
// block_terms: scratch of ceil(E/32) floats
int launch_aux_loss(const int32_t* counts, const float* partials, int n_partials, int T, int k,
                    int E, float* aux_out, float* block_terms, cudaStream_t s);

// capacity < 0 means unlimited.  pos_base [E] (may be null): slots of each expert that
// arrived before this batch (held elsewhere).  gate / gate_perm (may be null): per-slot
// gates gathered into row order.
int launch_dispatch(const int32_t* idx, const __nv_bfloat16* x, int T, int d, int E, int k,
                    int capacity, int32_t* counts, int32_t* offsets, int32_t* slot_row,
                    int32_t* row_slot, int32_t* n_kept_dropped, __nv_bfloat16* x_perm,
                    int32_t* local_rank, int32_t* chunk_cnt, int32_t* dev_status,
                    cudaStream_t s, const int32_t* pos_base = nullptr,
                    const float* gate = nullptr, float* gate_perm = nullptr);
// counts[e] = slots of idx routed to expert e (overwritten)
int launch_expert_counts(const int32_t* idx, long long slots, int E, int32_t* counts,
                         int32_t* dev_status, cudaStream_t s);
// rows (and per-row gates) between the source-major and expert-major layouts of an
// expert-parallel exchange; expert_offsets [El+1] (may be null) gets the expert-major starts
int launch_ep_regroup(const __nv_bfloat16* src, const float* gsrc, const int32_t* kept, int P,
                      int El, int d, int to_expert, long long rows_hint, __nv_bfloat16* dst,
                      float* gdst, int32_t* expert_offsets, cudaStream_t s);
// Dispatch with overflow remapping: rounds passes after the plain one; ws holds
// remap_ws_bytes(T, k, E, rounds).  slot_expert [T*k]: the expert each slot was placed on.
size_t remap_ws_bytes(int T, int k, int E, int rounds);
int launch_dispatch_remap(const int32_t* idx, const int32_t* alt, int rounds,
                          const __nv_bfloat16* x, int T, int d, int E, int k, int capacity,
                          int32_t* counts, int32_t* offsets, int32_t* slot_row,
                          int32_t* row_slot, int32_t* slot_expert, int32_t* n_kept_dropped,
                          __nv_bfloat16* x_perm, void* ws, int32_t* dev_status,
                          cudaStream_t s);
int launch_tile_schedule(const int32_t* offsets, int E, int rows_max, int32_t* tile_off,
                         int32_t* pair_off, int32_t* dev_status, cudaStream_t s);
int launch_combine(const __nv_bfloat16* y_perm, const int32_t* slot_row, int T, int d, int k,
                   __nv_bfloat16* y, cudaStream_t s);
int launch_combine_bwd(const __nv_bfloat16* dy, const __nv_bfloat16* y_perm,
                       const int32_t* slot_row, const float* gate, int T, int d, int k,
                       __nv_bfloat16* dz_perm, float* dgate, cudaStream_t s);
// dgate[row_slot[r]] = sum_n part[r][n] / gate[slot] for rows r < *n_rows (device count)
int launch_dgate_finalize(const float* part, int n_tiles, const int32_t* row_slot,
                          const float* gate, const int32_t* n_rows, int rows_max, float* dgate,
                          cudaStream_t s);
int launch_dispatch_bwd(const __nv_bfloat16* dx_perm, const int32_t* slot_row, int T, int d,
                        int k, float* dx, cudaStream_t s);
// dispatch backward and router backward in one pass (dx overwritten)
int launch_dispatch_route_bwd(const __nv_bfloat16* dx_perm, const int32_t* slot_row,
                              const int32_t* idx, const float* gate, const float* dgate,
                              const float* w_router, int T, int d, int E, int k, float* dx,
                              cudaStream_t s);
int launch_route_bwd(const int32_t* idx, const float* gate, const float* dgate,
                     const float* w_router, int T, int d, int E, int k, float* dx,
                     cudaStream_t s);

}  // namespace moe

// The C ABI of libmoe.so (declared in include/moe.h): argument checks, workspace carving,
// tensor-map encoding and the launch sequence of each step.  No entry point allocates,
// frees or synchronises.
#include <cuda_bf16.h>
#include <string.h>

#include <atomic>

#include "moe_internal.h"
#include "route.h"

using namespace moe;

namespace moe {

// Shared with the other entry-point files through moe_internal.h.
int check_problem(const moe_problem* p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (p->T <= 0 || p->d <= 0 || p->E <= 0 || p->k <= 0 || p->F <= 0 || p->r < 0)
    return MOE_ERR_INVALID_ARG;
  if (p->cap_num < 0 || p->cap_den < 0) return MOE_ERR_INVALID_ARG;
  if (p->d % 64 || p->F % 64) return MOE_ERR_UNSUPPORTED;
  if (p->k > 32 || p->k > p->E || p->E > 1024) return MOE_ERR_UNSUPPORTED;
  if (p->r && (p->r % 8 || p->r > 64)) return MOE_ERR_UNSUPPORTED;
  const long long slots = static_cast<long long>(p->T) * p->k;
  if (slots > (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  if (slots * p->d > (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// ceil(cap_num * T * k / (cap_den * E)), or -1 for an infinite capacity factor.
int capacity_of(const moe_problem* p) {
  if (p->cap_den == 0) return -1;
  const long long num = static_cast<long long>(p->cap_num) * p->T * p->k;
  const long long den = static_cast<long long>(p->cap_den) * p->E;
  const long long c = (num + den - 1) / den;
  return c > (1ll << 30) ? (1 << 30) : static_cast<int>(c);
}

size_t dispatch_ws(const moe_problem* p) {
  return up256(static_cast<size_t>(p->T) * p->k * 4) +
         up256(static_cast<size_t>(dispatch_num_chunks(p->T)) * p->E * 4);
}

// ---- instrumentation state (process-wide, see moe_set_kernel_events)
namespace {
cudaEvent_t g_ev_before[MOE_KERNEL_COUNT] = {nullptr};
cudaEvent_t g_ev_after[MOE_KERNEL_COUNT] = {nullptr};
std::atomic<long long> g_launches{0};
}  // namespace

void mark_before(int id, cudaStream_t s) {
  if (g_ev_before[id]) cudaEventRecord(g_ev_before[id], s);
}
void mark_after(int id, cudaStream_t s) {
  if (g_ev_after[id]) cudaEventRecord(g_ev_after[id], s);
}
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
long long launch_count() { return g_launches.load(std::memory_order_relaxed); }
int set_kernel_events(int kernel_id, void* event_before, void* event_after) {
  if (kernel_id < 0 || kernel_id >= MOE_KERNEL_COUNT) return MOE_ERR_INVALID_ARG;
  g_ev_before[kernel_id] = static_cast<cudaEvent_t>(event_before);
  g_ev_after[kernel_id] = static_cast<cudaEvent_t>(event_after);
  return MOE_OK;
}

}  // namespace moe

namespace {

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(int e) { return e == 0 ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)              \
  do {                             \
    const int _st = (expr);        \
    if (_st != MOE_OK) return _st; \
  } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

int lora_tile(int r) { return r <= 16 ? 16 : (r <= 32 ? 32 : 64); }

// Experts whose rows span several 128-row tiles re-read each weight tile once per tile:
// keep weights in L2 at normal priority then; with about one tile per expert they are
// streamed once and loaded evict-first.
bool weights_reused(const moe_problem* p, int rows_max) {
  const int C = capacity_of(p);
  return static_cast<long long>(rows_max) >= static_cast<long long>(kBM) * p->E &&
         (C < 0 || C > kBM);
}

// Groups average at least 1024 rows (8 m-tiles): the first-layer and down GEMMs then run on
// 256-row tiles, whose exposed epilogue (one TMEM accumulator) is small next to the time
// saved by staging each weight tile once per 256 rows.
bool big_groups(const moe_problem* p, int rows_max) {
  const int C = capacity_of(p);
  return static_cast<long long>(rows_max) >= 1024ll * p->E && (C < 0 || C >= 1024);
}

// Groups average 129..256 rows (two m-tiles, the second partly empty): staging each weight
// tile once for both m-tiles pays.
bool two_tile_groups(const moe_problem* p, int rows_max) {
  const int C = capacity_of(p);
  const long long per = rows_max / p->E;
  return per > kBM && per <= 2 * kBM && (C < 0 || C > kBM);
}

// Tile shapes of the grouped expert GEMMs.  CTA pairs stage half of every weight tile per SM
// and keep two accumulators per CTA (the epilogue of one tile overlaps the next tile's main
// loop).  Measured on GB300: groups of over 1024 rows (c4 shard: 4.3 -> 3.9 ms) take pairs
// everywhere; at 129..256 rows (c5) pairs pay for the gate/up GEMM (3253 -> 2907 us) but not
// for down (1767 vs 1775 us) or the backward dh (1710 vs 1804 us) and dx GEMMs (256-row
// tiles in one CTA 2972 vs 3173 us).  A gathered A operand takes 128-row tiles.
enum ExpertGemm { kGemmGateUp, kGemmDown, kGemmDh, kGemmDx };

int expert_tile_shape(const moe_problem* p, int rows_max, bool gather, ExpertGemm g) {
  if (gather) return kTile128;
  if (big_groups(p, rows_max)) return kTilePair;
  if (two_tile_groups(p, rows_max)) {
    if (g == kGemmGateUp) return kTilePair;
    if (g == kGemmDx) return kTile256;
  }
  return kTile128;
}

struct Carver {
  uint8_t* base;
  size_t used;
  template <class T>
  T* take(size_t count) {
    T* p = reinterpret_cast<T*>(base + used);
    used += up256(count * sizeof(T));
    return p;
  }
};

// expert tile of the router GEMM: 224 when it divides E (896 = 4 x 224: fewer, larger tiles,
// less L2 traffic per flop), else 128
int router_bn(const moe_problem* p) { return (p->E % 224 == 0) ? 224 : 128; }

size_t route_ws(const moe_problem* p) {
  const size_t nt = (p->E + router_bn(p) - 1) / router_bn(p);
  return up256(2ull * p->E * p->d * 2) + up256(static_cast<size_t>(p->T) * p->E * 4) +
         up256(static_cast<size_t>(p->T) * nt * kRouteTileK * 8) +
         up256(static_cast<size_t>(p->T) * nt * 4);
}

size_t ffn_ws(const moe_problem* p, int rows_max) {
  size_t b = 2 * up256((p->E + 1) * 4ull);
  if (p->r) b += 3 * up256(static_cast<size_t>(rows_max) * p->r * 2);
  return b;
}

GemmParams gemm_params() {
  GemmParams P;
  memset(&P, 0, sizeof(P));
  return P;
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null pointer or inconsistent sizes";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape or alignment not supported";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait ran out";
    case MOE_ERR_BAD_INDEX: return "MOE_ERR_BAD_INDEX: an index was out of range";
    default: return "unknown moe status";
  }
}

int moe_version(void) { return 10000; }

// ------------------------------------------------------------------------ routing

int moe_route_num_partials(const moe_problem* p) {
  return (p && p->T > 0) ? route_num_partials(p->T) : 0;
}

size_t moe_route_workspace_size(const moe_problem* p) {
  return check_problem(p) == MOE_OK ? route_ws(p) : 0;
}

int moe_route_from_logits(const moe_problem* p, const float* logits, int32_t* topk_idx,
                          float* topk_gate, float* prob_partials, int32_t* dev_status,
                          moe_stream_t stream) {
  (void)dev_status;
  MOE_TRY(check_problem(p));
  if (!logits || !topk_idx || !topk_gate || !prob_partials) return MOE_ERR_INVALID_ARG;
  mark_before(MOE_KERNEL_TOPK, stream);
  MOE_CUDA(launch_topk_softmax(logits, p->T, p->E, p->k, topk_idx, topk_gate, prob_partials,
                               stream));
  mark_after(MOE_KERNEL_TOPK, stream);
  count_launches(1);
  return MOE_OK;
}

namespace {

int route_impl(const moe_problem* p, const moe_bf16* x, const float* w_router, const float* bias,
               int32_t* topk_idx, float* topk_gate, float* prob_partials, float* logits,
               void* workspace, size_t workspace_bytes, int32_t* dev_status,
               moe_stream_t stream, bool fused) {
  MOE_TRY(check_problem(p));
  if (fused && p->k > kRouteTileK) return MOE_ERR_UNSUPPORTED;
  if (!x || !w_router || !topk_idx || !topk_gate || !prob_partials) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(w_router) || (logits && !al16(logits))) return MOE_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < route_ws(p)) return MOE_ERR_WORKSPACE;
  const int T = p->T, d = p->d, E = p->E;
  Carver cv{static_cast<uint8_t*>(workspace), 0};
  __nv_bfloat16* w_split = cv.take<__nv_bfloat16>(2ull * E * d);
  float* logits_ws = cv.take<float>(static_cast<size_t>(T) * E);
  float* L = logits ? logits : logits_ws;
  const int bn = router_bn(p);
  const int nt = (E + bn - 1) / bn;
  uint64_t* cand = cv.take<uint64_t>(static_cast<size_t>(T) * nt * kRouteTileK);
  float* tile_max = cv.take<float>(static_cast<size_t>(T) * nt);

  MOE_CUDA(launch_split_router(w_router, w_split, w_split + static_cast<size_t>(E) * d,
                               static_cast<size_t>(E) * d, stream));
  GemmParams P = gemm_params();
  MOE_TRY(encode_map_kmajor(&P.maps[0], x, d, T, 1, kBM));
  // the logits GEMM runs on CTA pairs (half of the bn expert rows per CTA); the fused top-k
  // variant on single CTAs
  MOE_TRY(encode_map_kmajor(&P.maps[1], w_split, d, E, 2, fused ? bn : bn / 2));
  P.nmaps = 2;
  // one K pass: each A stage is multiplied by the hi (z = 0) and lo (z = 1) weight tiles
  P.seg[0] = GemmSeg{d / kBK, 0, 0, {1, 1}, {0, 0}, {0, 1}};
  P.nseg = 1;
  P.M = T;
  P.m_tiles = (T + kBM - 1) / kBM;
  P.n_tiles = (E + bn - 1) / bn;
  P.N = E;
  P.out0 = L;
  P.ldo = E;
  P.bias = bias;
  P.b_policy = 1;  // the router weights are re-read by every token tile
  P.dev_status = dev_status;
  if (fused) {
    P.out1 = cand;
    P.out2 = tile_max;
  }
  mark_before(MOE_KERNEL_ROUTER_GEMM, stream);
  MOE_CUDA(fused ? launch_gemm_router_topk(P, bn, stream) : launch_gemm_router(P, bn, stream));
  mark_after(MOE_KERNEL_ROUTER_GEMM, stream);
  mark_before(MOE_KERNEL_TOPK, stream);
  if (fused) {
    MOE_CUDA(launch_route_merge(L, cand, tile_max, T, E, p->k, nt, topk_idx, topk_gate,
                                prob_partials, stream));
  } else {
    MOE_CUDA(launch_topk_softmax(L, T, E, p->k, topk_idx, topk_gate, prob_partials, stream));
  }
  mark_after(MOE_KERNEL_TOPK, stream);
  count_launches(3);
  return MOE_OK;
}

}  // namespace

int moe_route(const moe_problem* p, const moe_bf16* x, const float* w_router, const float* bias,
              int32_t* topk_idx, float* topk_gate, float* prob_partials, float* logits,
              void* workspace, size_t workspace_bytes, int32_t* dev_status,
              moe_stream_t stream) {
  return route_impl(p, x, w_router, bias, topk_idx, topk_gate, prob_partials, logits, workspace,
                    workspace_bytes, dev_status, stream, false);
}

int moe_route_fused_topk(const moe_problem* p, const moe_bf16* x, const float* w_router,
                         const float* bias, int32_t* topk_idx, float* topk_gate,
                         float* prob_partials, float* logits, void* workspace,
                         size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream) {
  return route_impl(p, x, w_router, bias, topk_idx, topk_gate, prob_partials, logits, workspace,
                    workspace_bytes, dev_status, stream, true);
}

// ------------------------------------------------------------------------ dispatch

size_t moe_dispatch_workspace_size(const moe_problem* p) {
  return check_problem(p) == MOE_OK ? dispatch_ws(p) : 0;
}

int moe_dispatch(const moe_problem* p, const int32_t* topk_idx, const moe_bf16* x,
                 int32_t* counts, int32_t* offsets, int32_t* slot_row, int32_t* row_slot,
                 int32_t* n_kept_dropped, moe_bf16* x_perm, void* workspace,
                 size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (!topk_idx || !counts || !offsets || !slot_row || !row_slot || !n_kept_dropped)
    return MOE_ERR_INVALID_ARG;
  if (x_perm && !x) return MOE_ERR_INVALID_ARG;
  if ((x && !al16(x)) || (x_perm && !al16(x_perm))) return MOE_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < dispatch_ws(p)) return MOE_ERR_WORKSPACE;
  Carver cv{static_cast<uint8_t*>(workspace), 0};
  int32_t* local_rank = cv.take<int32_t>(static_cast<size_t>(p->T) * p->k);
  int32_t* chunk_cnt = cv.take<int32_t>(static_cast<size_t>(dispatch_num_chunks(p->T)) * p->E);
  mark_before(MOE_KERNEL_DISPATCH, stream);
  MOE_CUDA(launch_dispatch(topk_idx, reinterpret_cast<const __nv_bfloat16*>(x), p->T, p->d,
                           p->E, p->k, capacity_of(p), counts, offsets, slot_row, row_slot,
                           n_kept_dropped, reinterpret_cast<__nv_bfloat16*>(x_perm), local_rank,
                           chunk_cnt, dev_status, stream));
  mark_after(MOE_KERNEL_DISPATCH, stream);
  count_launches(4);
  return MOE_OK;
}

int moe_dispatch_ep(const moe_problem* p, int32_t capacity, const int32_t* topk_idx,
                    const float* topk_gate, const moe_bf16* x, const int32_t* pos_base,
                    int32_t* counts, int32_t* offsets, int32_t* slot_row, int32_t* row_slot,
                    int32_t* n_kept_dropped, moe_bf16* x_perm, float* gate_perm,
                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                    moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (!topk_idx || !counts || !offsets || !slot_row || !row_slot || !n_kept_dropped)
    return MOE_ERR_INVALID_ARG;
  if ((x_perm && !x) || (gate_perm && !topk_gate)) return MOE_ERR_INVALID_ARG;
  if ((x && !al16(x)) || (x_perm && !al16(x_perm))) return MOE_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < dispatch_ws(p)) return MOE_ERR_WORKSPACE;
  Carver cv{static_cast<uint8_t*>(workspace), 0};
  int32_t* local_rank = cv.take<int32_t>(static_cast<size_t>(p->T) * p->k);
  int32_t* chunk_cnt = cv.take<int32_t>(static_cast<size_t>(dispatch_num_chunks(p->T)) * p->E);
  mark_before(MOE_KERNEL_DISPATCH, stream);
  MOE_CUDA(launch_dispatch(topk_idx, reinterpret_cast<const __nv_bfloat16*>(x), p->T, p->d,
                           p->E, p->k, capacity < 0 ? -1 : capacity, counts, offsets, slot_row,
                           row_slot, n_kept_dropped, reinterpret_cast<__nv_bfloat16*>(x_perm),
                           local_rank, chunk_cnt, dev_status, stream, pos_base, topk_gate,
                           gate_perm));
  mark_after(MOE_KERNEL_DISPATCH, stream);
  count_launches(4);
  return MOE_OK;
}

int moe_route_alternatives(const moe_problem* p, const float* logits, int32_t n_alt,
                           int32_t* alt_idx, moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (!logits || !alt_idx || n_alt <= 0) return MOE_ERR_INVALID_ARG;
  if (p->k + n_alt > 32 || p->k + n_alt > p->E) return MOE_ERR_UNSUPPORTED;
  MOE_CUDA(launch_topk_softmax(logits, p->T, p->E, p->k, nullptr, nullptr, nullptr, stream,
                               n_alt, alt_idx));
  count_launches(1);
  return MOE_OK;
}

size_t moe_dispatch_remap_workspace_size(const moe_problem* p, int32_t rounds) {
  if (check_problem(p) != MOE_OK || rounds < 0) return 0;
  return remap_ws_bytes(p->T, p->k, p->E, rounds);
}

int moe_dispatch_remap(const moe_problem* p, const int32_t* topk_idx, const int32_t* alt_idx,
                       int32_t rounds, const moe_bf16* x, int32_t* counts, int32_t* offsets,
                       int32_t* slot_row, int32_t* row_slot, int32_t* slot_expert,
                       int32_t* n_kept_dropped, moe_bf16* x_perm, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (rounds < 0) return MOE_ERR_INVALID_ARG;
  if ((rounds + 1) * p->k > 32 || (rounds + 1) * p->k > p->E) return MOE_ERR_UNSUPPORTED;
  if (!topk_idx || (rounds > 0 && !alt_idx) || !counts || !offsets || !slot_row || !row_slot ||
      !n_kept_dropped)
    return MOE_ERR_INVALID_ARG;
  if (x_perm && !x) return MOE_ERR_INVALID_ARG;
  if ((x && !al16(x)) || (x_perm && !al16(x_perm))) return MOE_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < remap_ws_bytes(p->T, p->k, p->E, rounds))
    return MOE_ERR_WORKSPACE;
  mark_before(MOE_KERNEL_DISPATCH, stream);
  MOE_CUDA(launch_dispatch_remap(topk_idx, alt_idx, rounds,
                                 reinterpret_cast<const __nv_bfloat16*>(x), p->T, p->d, p->E,
                                 p->k, capacity_of(p), counts, offsets, slot_row, row_slot,
                                 slot_expert, n_kept_dropped,
                                 reinterpret_cast<__nv_bfloat16*>(x_perm), workspace, dev_status,
                                 stream));
  mark_after(MOE_KERNEL_DISPATCH, stream);
  count_launches(3 * (rounds + 1) + 2);
  return MOE_OK;
}

int moe_expert_counts(const moe_problem* p, const int32_t* topk_idx, int32_t* counts,
                      int32_t* dev_status, moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (!topk_idx || !counts) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(launch_expert_counts(topk_idx, static_cast<long long>(p->T) * p->k, p->E, counts,
                                dev_status, stream));
  count_launches(2);
  return MOE_OK;
}

int moe_ep_regroup(const moe_bf16* src, const float* gate_src, const int32_t* kept,
                   int32_t n_sources, int32_t n_local_experts, int32_t d,
                   int32_t to_expert_major, int64_t rows_total, moe_bf16* dst,
                   float* gate_dst, int32_t* expert_offsets, moe_stream_t stream) {
  if (!kept || n_sources <= 0 || n_local_experts <= 0 || d <= 0 || rows_total < 0)
    return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(n_sources) * n_local_experts > 65536) return MOE_ERR_UNSUPPORTED;
  if ((gate_src == nullptr) != (gate_dst == nullptr)) return MOE_ERR_INVALID_ARG;
  if (rows_total > 0 && (!src || !dst)) return MOE_ERR_INVALID_ARG;
  if (d % 8 || (src && !al16(src)) || (dst && !al16(dst))) return MOE_ERR_UNSUPPORTED;
  MOE_CUDA(launch_ep_regroup(reinterpret_cast<const __nv_bfloat16*>(src), gate_src, kept,
                             n_sources, n_local_experts, d, to_expert_major ? 1 : 0, rows_total,
                             reinterpret_cast<__nv_bfloat16*>(dst), gate_dst, expert_offsets,
                             stream));
  count_launches(1);
  return MOE_OK;
}

// ------------------------------------------------------------------------ experts

size_t moe_expert_ffn_workspace_size(const moe_problem* p, int32_t rows_max) {
  return (check_problem(p) == MOE_OK && rows_max > 0) ? ffn_ws(p, rows_max) : 0;
}

}  // extern "C"

namespace {

// The expert step.  A rows come from `a_src`: the permuted rows themselves (gather = false,
// a_src = x_perm [rows, d]) or token rows gathered by slot (gather = true, a_src = x [T, d],
// row r reads x[row_slot[r] / k]).
// y_comb / slot_row (both or neither): the combine fused into the down GEMM's epilogue,
// y [T, d] written there (counters in the workspace after the plain carving).
int expert_ffn_impl(const moe_problem* p, int32_t rows_max, const moe_bf16* a_src, bool gather,
                    const int32_t* offsets, const int32_t* row_slot, const float* topk_gate,
                    const moe_bf16* w_gate, const moe_bf16* w_up, const moe_bf16* w_down,
                    const moe_lora* lora, moe_bf16* h, moe_bf16* y_perm,
                    const moe_ffn_saved* saved, void* workspace, size_t workspace_bytes,
                    int32_t* dev_status, moe_stream_t stream, const int32_t* slot_row = nullptr,
                    moe_bf16* y_comb = nullptr) {
  const moe_bf16* x_perm = a_src;
  MOE_TRY(check_problem(p));
  if (rows_max <= 0) return MOE_ERR_INVALID_ARG;
  const bool fuse_combine = y_comb != nullptr;
  if ((slot_row == nullptr) == fuse_combine) return MOE_ERR_INVALID_ARG;
  if (fuse_combine && !al16(y_comb)) return MOE_ERR_UNSUPPORTED;
  const size_t comb_bytes =
      fuse_combine ? up256(static_cast<size_t>(p->T) * ((p->d + 255) / 256) * 4) : 0;
  if (!x_perm || !offsets || !row_slot || !topk_gate || !w_gate || !w_up || !w_down || !h ||
      !y_perm)
    return MOE_ERR_INVALID_ARG;
  const bool use_lora = lora != nullptr && p->r > 0;
  if (lora && p->r == 0) return MOE_ERR_INVALID_ARG;
  if (use_lora && (!lora->A_g || !lora->B_g || !lora->A_u || !lora->B_u || !lora->A_d ||
                   !lora->B_d))
    return MOE_ERR_INVALID_ARG;
  const void* al[] = {x_perm, w_gate, w_up, w_down, h, y_perm};
  for (const void* q : al)
    if (!al16(q)) return MOE_ERR_UNSUPPORTED;
  if (use_lora) {
    const void* al2[] = {lora->A_g, lora->B_g, lora->A_u, lora->B_u, lora->A_d, lora->B_d};
    for (const void* q : al2)
      if (!al16(q)) return MOE_ERR_UNSUPPORTED;
  }
  if (saved) {
    const void* al3[] = {saved->a_gate, saved->a_up, saved->u_gate, saved->u_up, saved->u_down};
    for (const void* q : al3)
      if (q && !al16(q)) return MOE_ERR_UNSUPPORTED;
  }
  if (!workspace || workspace_bytes < ffn_ws(p, rows_max) + comb_bytes) return MOE_ERR_WORKSPACE;

  const int d = p->d, E = p->E, F = p->F, r = p->r;
  Carver cv{static_cast<uint8_t*>(workspace), 0};
  int32_t* tile_off = cv.take<int32_t>(E + 1);
  int32_t* pair_off = cv.take<int32_t>(E + 1);
  const int b_policy = weights_reused(p, rows_max) ? 1 : 0;
  const int shape_gu = expert_tile_shape(p, rows_max, gather, kGemmGateUp);
  const int shape_dn = expert_tile_shape(p, rows_max, gather, kGemmDown);
  moe_bf16 *u_g = nullptr, *u_u = nullptr, *u_d = nullptr;
  if (r) {
    u_g = cv.take<moe_bf16>(static_cast<size_t>(rows_max) * r);
    u_u = cv.take<moe_bf16>(static_cast<size_t>(rows_max) * r);
    u_d = cv.take<moe_bf16>(static_cast<size_t>(rows_max) * r);
    if (saved && saved->u_gate) u_g = saved->u_gate;
    if (saved && saved->u_up) u_u = saved->u_up;
    if (saved && saved->u_down) u_d = saved->u_down;
  }
  MOE_CUDA(launch_tile_schedule(offsets, E, rows_max, tile_off, pair_off, dev_status, stream));

  auto grouped = [&](GemmParams& P) {
    P.group_off = offsets;
    P.tile_off = tile_off;
    P.pair_off = pair_off;
    P.G = E;
    P.dev_status = dev_status;
    P.b_policy = b_policy;
  };
  // operand A of the first-layer GEMMs: permuted rows by TMA, or token rows gathered by
  // slot inside the GEMM (then the map is a placeholder of the same shape, never read)
  auto a_map = [&](CUtensorMap* m) -> int {
    return gather ? encode_map_kmajor(m, a_src, d, p->T, 1, kBM)
                  : encode_map_kmajor(m, a_src, d, rows_max, 1, kBM);
  };
  auto set_gather = [&](GemmParams& P) {
    if (gather) {
      P.gather_slot = row_slot;
      P.gather_k = p->k;
      P.gather_rows = p->T;
      P.gather_src = a_src;
      P.gather_ld = d;
    }
  };

  // LoRA down-projections of the input: u_g = s x A_g^T, u_u = s x A_u^T
  if (use_lora) {
    GemmParams P = gemm_params();
    MOE_TRY(a_map(&P.maps[0]));
    MOE_TRY(encode_map_kmajor(&P.maps[1], lora->A_g, d, r, E, lora_tile(r)));
    MOE_TRY(encode_map_kmajor(&P.maps[2], lora->A_u, d, r, E, lora_tile(r)));
    P.nmaps = 3;
    P.seg[0] = GemmSeg{d / kBK, 0, 0, {1, 2}, {0, 0}, {0, 0}, gather ? 1 : 0};
    P.nseg = 1;
    grouped(P);
    set_gather(P);
    P.n_tiles = 1;
    P.N = r;
    P.out0 = u_g;
    P.out1 = u_u;
    P.ldo = r;
    P.scale = p->lora_scale;
    MOE_CUDA(launch_gemm_lora_u2(P, r, stream));
  }
  // gate/up projections (+ LoRA K-blocks) with the SwiGLU epilogue -> h
  {
    GemmParams P = gemm_params();
    MOE_TRY(a_map(&P.maps[0]));
    MOE_TRY(encode_map_kmajor(&P.maps[1], w_gate, d, F, E, 128));
    MOE_TRY(encode_map_kmajor(&P.maps[2], w_up, d, F, E, 128));
    P.nmaps = 3;
    P.seg[0] = GemmSeg{d / kBK, 0, 0, {1, 2}, {0, 0}, {0, 0}, gather ? 1 : 0};
    P.nseg = 1;
    if (use_lora) {
      MOE_TRY(encode_map_kmajor(&P.maps[3], u_g, r, rows_max, 1, kBM));
      MOE_TRY(encode_map_kmajor(&P.maps[4], u_u, r, rows_max, 1, kBM));
      MOE_TRY(encode_map_kmajor(&P.maps[5], lora->B_g, r, F, E, 128));
      MOE_TRY(encode_map_kmajor(&P.maps[6], lora->B_u, r, F, E, 128));
      P.nmaps = 7;
      P.seg[1] = GemmSeg{(r + kBK - 1) / kBK, 3, 0, {5, -1}, {0, 0}, {0, 0}};
      P.seg[2] = GemmSeg{(r + kBK - 1) / kBK, 4, 0, {-1, 6}, {0, 0}, {0, 0}};
      P.nseg = 3;
    }
    grouped(P);
    set_gather(P);
    P.n_tiles = (F + 127) / 128;
    P.N = F;
    P.out0 = h;
    P.out1 = saved ? saved->a_gate : nullptr;
    P.out2 = saved ? saved->a_up : nullptr;
    P.ldo = F;
    mark_before(MOE_KERNEL_GATEUP_GEMM, stream);
    MOE_CUDA(launch_gemm_gateup(P, shape_gu, stream));
    mark_after(MOE_KERNEL_GATEUP_GEMM, stream);
  }
  // LoRA down-projection of h: u_d = s h A_d^T
  if (use_lora) {
    GemmParams P = gemm_params();
    MOE_TRY(encode_map_kmajor(&P.maps[0], h, F, rows_max, 1, kBM));
    MOE_TRY(encode_map_kmajor(&P.maps[1], lora->A_d, F, r, E, lora_tile(r)));
    P.nmaps = 2;
    P.seg[0] = GemmSeg{F / kBK, 0, 0, {1, -1}, {0, 0}, {0, 0}};
    P.nseg = 1;
    grouped(P);
    P.n_tiles = 1;
    P.N = r;
    P.out0 = u_d;
    P.ldo = r;
    P.scale = p->lora_scale;
    MOE_CUDA(launch_gemm_lora_u1(P, r, stream));
  }
  // down projection (+ LoRA K-block), scaled by the routing gate -> y_perm
  {
    GemmParams P = gemm_params();
    MOE_TRY(encode_map_kmajor(&P.maps[0], h, F, rows_max, 1, kBM));
    // CTA pairs: each CTA stages 128 of the tile's 256 weight rows
    const int box_n = shape_dn == kTilePair ? 128 : 256;
    MOE_TRY(encode_map_kmajor(&P.maps[1], w_down, F, d, E, box_n));
    P.nmaps = 2;
    P.seg[0] = GemmSeg{F / kBK, 0, 0, {1, -1}, {0, 0}, {0, 0}};
    P.nseg = 1;
    if (use_lora) {
      MOE_TRY(encode_map_kmajor(&P.maps[2], u_d, r, rows_max, 1, kBM));
      MOE_TRY(encode_map_kmajor(&P.maps[3], lora->B_d, r, d, E, box_n));
      P.nmaps = 4;
      P.seg[1] = GemmSeg{(r + kBK - 1) / kBK, 2, 0, {3, -1}, {0, 0}, {0, 0}};
      P.nseg = 2;
    }
    grouped(P);
    P.n_tiles = (d + 255) / 256;
    P.N = d;
    P.out0 = y_perm;
    P.ldo = d;
    P.gate = topk_gate;
    P.row_slot = row_slot;
    if (fuse_combine) {
      int32_t* comb_cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) +
                                                     ffn_ws(p, rows_max));
      MOE_CUDA(launch_combine_prepare(slot_row, p->T, p->k, P.n_tiles, d, comb_cnt,
                                      reinterpret_cast<__nv_bfloat16*>(y_comb), stream));
      P.comb_cnt = comb_cnt;
      P.comb_slot_row = slot_row;
      P.comb_y = y_comb;
      P.comb_k = p->k;
    }
    mark_before(MOE_KERNEL_DOWN_GEMM, stream);
    MOE_CUDA(launch_gemm_down(P, shape_dn, stream));
    mark_after(MOE_KERNEL_DOWN_GEMM, stream);
  }
  count_launches((use_lora ? 5 : 3) + (fuse_combine ? 1 : 0));
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_expert_ffn(const moe_problem* p, int32_t rows_max, const moe_bf16* x_perm,
                   const int32_t* offsets, const int32_t* row_slot, const float* topk_gate,
                   const moe_bf16* w_gate, const moe_bf16* w_up, const moe_bf16* w_down,
                   const moe_lora* lora, moe_bf16* h, moe_bf16* y_perm,
                   const moe_ffn_saved* saved, void* workspace, size_t workspace_bytes,
                   int32_t* dev_status, moe_stream_t stream) {
  return expert_ffn_impl(p, rows_max, x_perm, false, offsets, row_slot, topk_gate, w_gate, w_up,
                         w_down, lora, h, y_perm, saved, workspace, workspace_bytes, dev_status,
                         stream);
}

int moe_expert_ffn_gather(const moe_problem* p, int32_t rows_max, const moe_bf16* x,
                          const int32_t* offsets, const int32_t* row_slot,
                          const float* topk_gate, const moe_bf16* w_gate, const moe_bf16* w_up,
                          const moe_bf16* w_down, const moe_lora* lora, moe_bf16* h,
                          moe_bf16* y_perm, const moe_ffn_saved* saved, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream) {
  return expert_ffn_impl(p, rows_max, x, true, offsets, row_slot, topk_gate, w_gate, w_up,
                         w_down, lora, h, y_perm, saved, workspace, workspace_bytes, dev_status,
                         stream);
}

size_t moe_expert_ffn_combine_workspace_size(const moe_problem* p, int32_t rows_max) {
  if (check_problem(p) != MOE_OK || rows_max <= 0) return 0;
  return ffn_ws(p, rows_max) + up256(static_cast<size_t>(p->T) * ((p->d + 255) / 256) * 4);
}

int moe_expert_ffn_combine(const moe_problem* p, int32_t rows_max, const moe_bf16* a_src,
                           int32_t a_is_tokens, const int32_t* offsets, const int32_t* row_slot,
                           const int32_t* slot_row, const float* topk_gate,
                           const moe_bf16* w_gate, const moe_bf16* w_up,
                           const moe_bf16* w_down, const moe_lora* lora, moe_bf16* h,
                           moe_bf16* y_perm, moe_bf16* y, const moe_ffn_saved* saved,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           moe_stream_t stream) {
  if (!slot_row || !y) return MOE_ERR_INVALID_ARG;
  return expert_ffn_impl(p, rows_max, a_src, a_is_tokens != 0, offsets, row_slot, topk_gate,
                         w_gate, w_up, w_down, lora, h, y_perm, saved, workspace,
                         workspace_bytes, dev_status, stream, slot_row, y);
}

// ------------------------------------------------------------------------ combine / aux

int moe_combine(const moe_problem* p, const moe_bf16* y_perm, const int32_t* slot_row,
                moe_bf16* y, moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (!y_perm || !slot_row || !y) return MOE_ERR_INVALID_ARG;
  if (!al16(y_perm) || !al16(y)) return MOE_ERR_UNSUPPORTED;
  mark_before(MOE_KERNEL_COMBINE, stream);
  MOE_CUDA(launch_combine(reinterpret_cast<const __nv_bfloat16*>(y_perm), slot_row, p->T, p->d,
                          p->k, reinterpret_cast<__nv_bfloat16*>(y), stream));
  mark_after(MOE_KERNEL_COMBINE, stream);
  count_launches(1);
  return MOE_OK;
}

size_t moe_aux_loss_workspace_size(const moe_problem* p) {
  return check_problem(p) == MOE_OK ? up256(((p->E + 31) / 32) * sizeof(float)) : 0;
}

int moe_aux_loss(const moe_problem* p, const int32_t* counts, const float* prob_partials,
                 int32_t n_partials, float* aux_out, void* workspace, size_t workspace_bytes,
                 moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (!counts || !prob_partials || !aux_out || n_partials <= 0) return MOE_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < moe_aux_loss_workspace_size(p)) return MOE_ERR_WORKSPACE;
  MOE_CUDA(launch_aux_loss(counts, prob_partials, n_partials, p->T, p->k, p->E, aux_out,
                           static_cast<float*>(workspace), stream));
  count_launches(2);
  return MOE_OK;
}

// ------------------------------------------------------------------------ backward

int moe_combine_bwd(const moe_problem* p, const moe_bf16* dy, const moe_bf16* y_perm,
                    const int32_t* slot_row, const float* topk_gate, moe_bf16* dz_perm,
                    float* dgate, moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (!dy || !slot_row || !topk_gate || !dz_perm || (y_perm && !dgate))
    return MOE_ERR_INVALID_ARG;
  if (!al16(dy) || (y_perm && !al16(y_perm)) || !al16(dz_perm)) return MOE_ERR_UNSUPPORTED;
  count_launches(1);
  mark_before(MOE_KERNEL_COMBINE_BWD, stream);
  const int st = cuda_status(launch_combine_bwd(
      reinterpret_cast<const __nv_bfloat16*>(dy), reinterpret_cast<const __nv_bfloat16*>(y_perm),
      slot_row, topk_gate, p->T, p->d, p->k, reinterpret_cast<__nv_bfloat16*>(dz_perm), dgate,
      stream));
  mark_after(MOE_KERNEL_COMBINE_BWD, stream);
  return st;
}

size_t moe_expert_ffn_bwd_workspace_size(const moe_problem* p, int32_t rows_max) {
  if (check_problem(p) != MOE_OK || rows_max <= 0) return 0;
  size_t b = 2 * up256((p->E + 1) * 4ull) + 2 * up256(static_cast<size_t>(rows_max) * p->F * 2);
  if (p->r) b += 3 * up256(static_cast<size_t>(rows_max) * p->r * 2);
  b += up256(static_cast<size_t>(rows_max) * ((p->F + 255) / 256) * 4);  // gate-gradient parts
  return b;
}

int moe_expert_ffn_bwd(const moe_problem* p, int32_t rows_max, const moe_bf16* x_perm,
                       const int32_t* offsets, const moe_bf16* w_gate, const moe_bf16* w_up,
                       const moe_bf16* w_down, const moe_lora* lora,
                       const moe_ffn_saved* saved, const moe_bf16* h, const moe_bf16* dz_perm,
                       moe_bf16* dx_perm, const moe_lora_grad* grads,
                       const int32_t* row_slot, const float* topk_gate, float* dgate,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status,
                       moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (rows_max <= 0) return MOE_ERR_INVALID_ARG;
  if (dgate && (!row_slot || !topk_gate)) return MOE_ERR_INVALID_ARG;
  if (!x_perm || !offsets || !w_gate || !w_up || !w_down || !saved || !saved->a_gate ||
      !saved->a_up || !h || !dz_perm || !dx_perm)
    return MOE_ERR_INVALID_ARG;
  const bool use_lora = lora != nullptr && p->r > 0;
  if (lora && p->r == 0) return MOE_ERR_INVALID_ARG;
  if (use_lora) {
    if (!lora->A_g || !lora->B_g || !lora->A_u || !lora->B_u || !lora->A_d || !lora->B_d ||
        !saved->u_gate || !saved->u_up || !saved->u_down || !grads || !grads->dA_g ||
        !grads->dB_g || !grads->dA_u || !grads->dB_u || !grads->dA_d || !grads->dB_d)
      return MOE_ERR_INVALID_ARG;
    const void* al2[] = {lora->A_g, lora->B_g, lora->A_u, lora->B_u, lora->A_d, lora->B_d,
                         saved->u_gate, saved->u_up, saved->u_down};
    for (const void* q : al2)
      if (!al16(q)) return MOE_ERR_UNSUPPORTED;
  }
  const void* al[] = {x_perm, w_gate, w_up, w_down, saved->a_gate, saved->a_up, h, dz_perm,
                      dx_perm};
  for (const void* q : al)
    if (!al16(q)) return MOE_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < moe_expert_ffn_bwd_workspace_size(p, rows_max))
    return MOE_ERR_WORKSPACE;

  const int d = p->d, E = p->E, F = p->F, r = p->r;
  const float s = p->lora_scale;
  Carver cv{static_cast<uint8_t*>(workspace), 0};
  int32_t* tile_off = cv.take<int32_t>(E + 1);
  int32_t* pair_off = cv.take<int32_t>(E + 1);
  const int b_policy = weights_reused(p, rows_max) ? 1 : 0;  // as in the forward
  moe_bf16* da_g = cv.take<moe_bf16>(static_cast<size_t>(rows_max) * F);
  moe_bf16* da_u = cv.take<moe_bf16>(static_cast<size_t>(rows_max) * F);
  moe_bf16 *v_d = nullptr, *v_g = nullptr, *v_u = nullptr;
  if (r) {
    v_d = cv.take<moe_bf16>(static_cast<size_t>(rows_max) * r);
    v_g = cv.take<moe_bf16>(static_cast<size_t>(rows_max) * r);
    v_u = cv.take<moe_bf16>(static_cast<size_t>(rows_max) * r);
  }
  const int dh_tiles = (F + 255) / 256;
  float* gate_parts = cv.take<float>(static_cast<size_t>(rows_max) * dh_tiles);
  MOE_CUDA(launch_tile_schedule(offsets, E, rows_max, tile_off, pair_off, dev_status, stream));
  int launches = 1;
  // dh and dx run on CTA pairs for big groups; for two-tile groups dx (plain store epilogue)
  // takes 256-row tiles and dh (heavy SwiGLU-backward epilogue) stays on 128-row tiles
  const int shape_dh = expert_tile_shape(p, rows_max, false, kGemmDh);
  const int shape_dx = expert_tile_shape(p, rows_max, false, kGemmDx);
  auto grouped = [&](GemmParams& P) {
    P.group_off = offsets;
    P.tile_off = tile_off;
    P.pair_off = pair_off;
    P.G = E;
    P.dev_status = dev_status;
    P.b_policy = b_policy;
  };
  auto lora_v = [&](const moe_bf16* a, int K, const moe_bf16* bmat, int bk_rows,
                    moe_bf16* out) -> int {
    // out = s * (a bmat), a [rows, K] K-major, bmat[e] [K, r] (MN-major B)
    GemmParams P = gemm_params();
    MOE_TRY(encode_map_kmajor(&P.maps[0], a, K, rows_max, 1, kBM));
    MOE_TRY(encode_map_mnmajor(&P.maps[1], bmat, r, bk_rows, E));
    P.nmaps = 2;
    P.seg[0] = GemmSeg{K / kBK, 0, 0, {1, -1}, {0, 0}, {0, 0}};
    P.nseg = 1;
    grouped(P);
    P.n_tiles = 1;
    P.N = r;
    P.out0 = out;
    P.ldo = r;
    P.scale = s;
    ++launches;
    return cuda_status(launch_gemm_bwd_lora_v(P, r, stream));
  };

  // v'_d = s dz B_d
  if (use_lora) MOE_TRY(lora_v(dz_perm, d, lora->B_d, d, v_d));
  // dh = dz W_d + v'_d A_d  ->  da_g, da_u (SwiGLU backward on the saved pre-activations)
  {
    GemmParams P = gemm_params();
    MOE_TRY(encode_map_kmajor(&P.maps[0], dz_perm, d, rows_max, 1, kBM));
    MOE_TRY(encode_map_mnmajor(&P.maps[1], w_down, F, d, E));
    P.nmaps = 2;
    P.seg[0] = GemmSeg{d / kBK, 0, 0, {1, -1}, {0, 0}, {0, 0}};
    P.nseg = 1;
    if (use_lora) {
      MOE_TRY(encode_map_kmajor(&P.maps[2], v_d, r, rows_max, 1, kBM));
      MOE_TRY(encode_map_mnmajor(&P.maps[3], lora->A_d, F, r, E));
      P.nmaps = 4;
      P.seg[1] = GemmSeg{(r + kBK - 1) / kBK, 2, 0, {3, -1}, {0, 0}, {0, 0}};
      P.nseg = 2;
    }
    grouped(P);
    P.n_tiles = (F + 255) / 256;
    P.N = F;
    P.ldo = F;
    P.in0 = saved->a_gate;
    P.in1 = saved->a_up;
    P.out0 = da_g;
    P.out1 = da_u;
    P.out2 = dgate ? gate_parts : nullptr;
    ++launches;
    mark_before(MOE_KERNEL_BWD_DH_GEMM, stream);
    MOE_CUDA(launch_gemm_bwd_dh(P, shape_dh, stream));
    mark_after(MOE_KERNEL_BWD_DH_GEMM, stream);
    if (dgate) {
      MOE_CUDA(launch_dgate_finalize(gate_parts, dh_tiles, row_slot, topk_gate, offsets + E,
                                     rows_max, dgate, stream));
      ++launches;
    }
  }
  // v'_g = s da_g B_g, v'_u = s da_u B_u
  if (use_lora) {
    MOE_TRY(lora_v(da_g, F, lora->B_g, F, v_g));
    MOE_TRY(lora_v(da_u, F, lora->B_u, F, v_u));
  }
  // dx_perm = da_g W_g + da_u W_u + v'_g A_g + v'_u A_u
  {
    GemmParams P = gemm_params();
    MOE_TRY(encode_map_kmajor(&P.maps[0], da_g, F, rows_max, 1, kBM));
    MOE_TRY(encode_map_kmajor(&P.maps[1], da_u, F, rows_max, 1, kBM));
    MOE_TRY(encode_map_mnmajor(&P.maps[2], w_gate, d, F, E));
    MOE_TRY(encode_map_mnmajor(&P.maps[3], w_up, d, F, E));
    P.nmaps = 4;
    P.seg[0] = GemmSeg{F / kBK, 0, 0, {2, -1}, {0, 0}, {0, 0}};
    P.seg[1] = GemmSeg{F / kBK, 1, 0, {3, -1}, {0, 0}, {0, 0}};
    P.nseg = 2;
    if (use_lora) {
      MOE_TRY(encode_map_kmajor(&P.maps[4], v_g, r, rows_max, 1, kBM));
      MOE_TRY(encode_map_kmajor(&P.maps[5], v_u, r, rows_max, 1, kBM));
      MOE_TRY(encode_map_mnmajor(&P.maps[6], lora->A_g, d, r, E));
      MOE_TRY(encode_map_mnmajor(&P.maps[7], lora->A_u, d, r, E));
      P.nmaps = 8;
      P.seg[2] = GemmSeg{(r + kBK - 1) / kBK, 4, 0, {6, -1}, {0, 0}, {0, 0}};
      P.seg[3] = GemmSeg{(r + kBK - 1) / kBK, 5, 0, {7, -1}, {0, 0}, {0, 0}};
      P.nseg = 4;
    }
    grouped(P);
    P.n_tiles = (d + 255) / 256;
    P.N = d;
    P.ldo = d;
    P.out0 = dx_perm;
    ++launches;
    mark_before(MOE_KERNEL_BWD_DX_GEMM, stream);
    MOE_CUDA(launch_gemm_bwd_dx(P, shape_dx, stream));
    mark_after(MOE_KERNEL_BWD_DX_GEMM, stream);
  }
  // LoRA weight gradients: per expert, reductions over its rows (grouped over K)
  if (use_lora) {
    auto wgrad = [&](const moe_bf16* a, int M, const moe_bf16* b0, const moe_bf16* b1,
                     float* out0, float* out1, bool transposed) -> int {
      GemmParams P = gemm_params();
      MOE_TRY(encode_map_mnmajor(&P.maps[0], a, M, rows_max, 1));
      MOE_TRY(encode_map_mnmajor(&P.maps[1], b0, r, rows_max, 1));
      P.nmaps = 2;
      P.seg[0] = GemmSeg{0, 0, 0, {1, -1}, {0, 0}, {0, 0}};
      if (b1) {
        MOE_TRY(encode_map_mnmajor(&P.maps[2], b1, r, rows_max, 1));
        P.nmaps = 3;
        P.seg[0].b_map[1] = 2;
      }
      P.nseg = 1;
      P.group_off = offsets;
      P.G = E;
      P.M = M;
      P.m_tiles = (M + kBM - 1) / kBM;
      P.n_tiles = 1;
      P.N = r;
      P.out0 = out0;
      P.out1 = out1;
      P.out_transposed = transposed ? 1 : 0;
      P.dev_status = dev_status;
      P.b_policy = 1;  // the small B rows of an expert are re-read by each of its m-tiles
      ++launches;
      return cuda_status(launch_gemm_wgrad(P, r, b1 ? 2 : 1, stream));
    };
    // dA_g^T = x^T v'_g, dA_u^T = x^T v'_u   ([E, r, d] written transposed)
    mark_before(MOE_KERNEL_WGRAD, stream);
    MOE_TRY(wgrad(x_perm, d, v_g, v_u, grads->dA_g, grads->dA_u, true));
    // dB_d = dz^T u'_d   ([E, d, r])
    MOE_TRY(wgrad(dz_perm, d, saved->u_down, nullptr, grads->dB_d, nullptr, false));
    // dA_d^T = h^T v'_d  ([E, r, F] written transposed)
    MOE_TRY(wgrad(h, F, v_d, nullptr, grads->dA_d, nullptr, true));
    // dB_g = da_g^T u'_g, dB_u = da_u^T u'_u   ([E, F, r])
    MOE_TRY(wgrad(da_g, F, saved->u_gate, nullptr, grads->dB_g, nullptr, false));
    MOE_TRY(wgrad(da_u, F, saved->u_up, nullptr, grads->dB_u, nullptr, false));
    mark_after(MOE_KERNEL_WGRAD, stream);
  }
  count_launches(launches);
  return MOE_OK;
}

int moe_dispatch_bwd(const moe_problem* p, const moe_bf16* dx_perm, const int32_t* slot_row,
                     float* dx, moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (!dx_perm || !slot_row || !dx) return MOE_ERR_INVALID_ARG;
  if (!al16(dx_perm) || !al16(dx)) return MOE_ERR_UNSUPPORTED;
  count_launches(1);
  return cuda_status(launch_dispatch_bwd(reinterpret_cast<const __nv_bfloat16*>(dx_perm),
                                         slot_row, p->T, p->d, p->k, dx, stream));
}

int moe_route_bwd(const moe_problem* p, const int32_t* topk_idx, const float* topk_gate,
                  const float* dgate, const float* w_router, float* dx, moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (!topk_idx || !topk_gate || !dgate || !w_router || !dx) return MOE_ERR_INVALID_ARG;
  if (!al16(w_router) || !al16(dx)) return MOE_ERR_UNSUPPORTED;
  count_launches(1);
  return cuda_status(launch_route_bwd(topk_idx, topk_gate, dgate, w_router, p->T, p->d, p->E,
                                      p->k, dx, stream));
}

int moe_dispatch_route_bwd(const moe_problem* p, const moe_bf16* dx_perm,
                           const int32_t* slot_row, const int32_t* topk_idx,
                           const float* topk_gate, const float* dgate, const float* w_router,
                           float* dx, moe_stream_t stream) {
  MOE_TRY(check_problem(p));
  if (!dx_perm || !slot_row || !topk_idx || !topk_gate || !dgate || !w_router || !dx)
    return MOE_ERR_INVALID_ARG;
  if (!al16(dx_perm) || !al16(w_router) || !al16(dx)) return MOE_ERR_UNSUPPORTED;
  count_launches(1);
  mark_before(MOE_KERNEL_DISPATCH_ROUTE_BWD, stream);
  const int st = cuda_status(launch_dispatch_route_bwd(
      reinterpret_cast<const __nv_bfloat16*>(dx_perm), slot_row, topk_idx, topk_gate, dgate,
      w_router, p->T, p->d, p->E, p->k, dx, stream));
  mark_after(MOE_KERNEL_DISPATCH_ROUTE_BWD, stream);
  return st;
}

// ------------------------------------------------------------------------ instrumentation

int moe_set_kernel_events(int kernel_id, void* event_before, void* event_after) {
  return moe::set_kernel_events(kernel_id, event_before, event_after);
}

long long moe_launch_count(void) { return moe::launch_count(); }

}  // extern "C"

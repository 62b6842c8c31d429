/*
 * moe.h -- C ABI of the GB300 sparse Mixture-of-Experts layer (libmoe.so).
 *
 * The layer is the one of "Adapting Trillion-Parameter MoE Models for LoRA Fine-Tuning:
 * A Full-Stack Engineering Guide", section 2.1, equation 1:
 *
 *     y = sum_{i in TopK(x)} g_i(x) * E_i(x)
 *
 * run as the Dispatch-Compute-Combine pipeline of "Trillion-Parameter MoE Model Training
 * Adaptation: Full-Stack Optimization Practices", section 4.3 (route, permute tokens by
 * expert, grouped expert GEMMs, unpermute), with the LoRA update of the same guide,
 * section 3, equation 1 (W' = W0 + (alpha/r) B A) on each expert projection.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every function returns an int status (MOE_OK on success).  Nothing throws.
 *  - Tensor arguments are DEVICE pointers owned by the caller.  The library never
 *    allocates or frees device memory; scratch space is a caller-supplied workspace
 *    whose size the matching *_workspace_size() function returns ("Adapting Ultra-Large
 *    MoE Models: Engineering Practices and Optimization Pathways", section 3.4:
 *    pre-allocated reusable buffers).
 *  - All work is enqueued asynchronously on `stream` (a cudaStream_t); no call
 *    synchronises the device or the stream.
 *  - Host-side argument errors return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_WORKSPACE before anything is enqueued.  A failed launch returns MOE_ERR_CUDA.
 *  - Errors found on the device (an expert id out of range, a bounded wait that ran
 *    out) are written to the caller's `dev_status` word (int32, device memory, may be
 *    NULL) with first-error-wins semantics; the kernel skips the offending work instead of
 *    faulting.  The caller zeroes the word and reads it back when it chooses.
 *  - bf16 values are passed as raw 16-bit patterns (moe_bf16).  All matrices are
 *    row-major and densely packed.
 *  - Requirements (else MOE_ERR_UNSUPPORTED): d and F multiples of 64; 1 <= k <= 32;
 *    k <= E <= 1024; r == 0 or (r a multiple of 8 and r <= 64); every pointer 16-byte
 *    aligned.
 *  - Shapes: T tokens, d model width, E experts, k experts per token, F expert FFN
 *    width, r LoRA rank, N = T*k slots.  Slot (t, j) is numbered t*k + j; rank j = 0 is
 *    the largest router logit.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, inconsistent sizes      */
  MOE_ERR_UNSUPPORTED = 2,  /* shape or alignment outside the supported set             */
  MOE_ERR_WORKSPACE = 3,    /* workspace pointer null or smaller than *_workspace_size */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed                        */
  MOE_ERR_TIMEOUT = 5,      /* (device) a bounded wait inside a kernel ran out          */
  MOE_ERR_BAD_INDEX = 6     /* (device) an expert id or row index was out of range      */
};

typedef uint16_t moe_bf16;                /* raw bfloat16 bits                          */
typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t                  */

/* Problem sizes.  Capacity factor cf = cap_num / cap_den; cap_den == 0 means an infinite
 * factor (no token is ever dropped).  lora_scale is s = alpha / r. */
typedef struct moe_problem {
  int32_t T, d, E, k, F, r;
  float lora_scale;
  int32_t cap_num, cap_den;
} moe_problem;

/* LoRA factors of every expert (device pointers, bf16), or all NULL for none:
 *   A_g, A_u [E, r, d]   B_g, B_u [E, F, r]   A_d [E, r, F]   B_d [E, d, r]
 * so that the gate projection is  W_g x + s * B_g (A_g x)  and so on. */
typedef struct moe_lora {
  const moe_bf16 *A_g, *B_g, *A_u, *B_u, *A_d, *B_d;
} moe_lora;

/* Gradients of the LoRA factors (fp32, same shapes as moe_lora; overwritten). */
typedef struct moe_lora_grad {
  float *dA_g, *dB_g, *dA_u, *dB_u, *dA_d, *dB_d;
} moe_lora_grad;

/* Activations the expert forward saves for the backward (bf16, rows of x_perm order):
 *   a_gate, a_up [rows, F]  pre-activations of the gate and up projections
 *   u_gate, u_up [rows, r]  s * (x A_g^T), s * (x A_u^T)      (LoRA only)
 *   u_down       [rows, r]  s * (h A_d^T)                     (LoRA only)
 * Any pointer may be NULL when the backward will not run. */
typedef struct moe_ffn_saved {
  moe_bf16 *a_gate, *a_up, *u_gate, *u_up, *u_down;
} moe_ffn_saved;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(int status);

/* ABI version of this library (major * 10000 + minor * 100 + patch). */
int moe_version(void);

/* ==================================================================== routing
 * "Day-Level Adaptation and LoRA Fine-Tuning of Ultra-Large-Scale Sparse MoE Models",
 * section 2.1 and section 3.3 (routing scoring fused with Top-k selection);
 * "Adapting Trillion-Parameter MoE Models ...", section 2.1, equation 1 (gate g_i).
 *
 *   logits[t, e] = sum_c x[t, c] * w_router[e, c] + bias[e]        (fp32 accuracy)
 *   topk_idx[t, j]  = the k largest logits, descending; equal logits -> lower index first
 *   p[t, :]         = softmax(logits[t, :]) over all E experts (fp32)
 *   topk_gate[t, j] = p[t, topk_idx[t, j]] / sum_j' p[t, topk_idx[t, j']]
 *   prob_partials[b, e] = sum of p[t, e] over the tokens of row-block b
 *                         (moe_route_num_partials() rows; feeds moe_aux_loss)
 *
 * x [T, d] bf16; w_router [E, d] fp32; bias [E] fp32 or NULL; topk_idx [T, k] int32;
 * topk_gate [T, k] fp32; prob_partials [num_partials, E] fp32; logits [T, E] fp32 or NULL
 * (when given, the fp32 logits are written there; else they live in the workspace).
 */
int moe_route_num_partials(const moe_problem* p);
size_t moe_route_workspace_size(const moe_problem* p);
int moe_route(const moe_problem* p, const moe_bf16* x, const float* w_router,
              const float* bias, int32_t* topk_idx, float* topk_gate, float* prob_partials,
              float* logits, void* workspace, size_t workspace_bytes, int32_t* dev_status,
              moe_stream_t stream);

/* moe_route with the softmax and top-k folded into the router GEMM: its epilogue keeps, per
 * token and 224-expert tile, the tile maximum and the 16 largest (logit, expert) keys, and a
 * light kernel merges the tiles' lists (exact: every selected expert is among its tile's 16
 * largest), normalises over all E logits and renormalises the gates.  Same arguments, same
 * workspace and the same outputs as moe_route (identical topk_idx; gates and probability
 * partials equal up to fp32 summation order); k <= 16, else MOE_ERR_UNSUPPORTED.  On GB300
 * it measured slower than moe_route's separate top-k kernel (c2 64 vs 57 us, c5 139 vs
 * 132 us for router GEMM + selection), so moe_route does not use it. */
int moe_route_fused_topk(const moe_problem* p, const moe_bf16* x, const float* w_router,
                         const float* bias, int32_t* topk_idx, float* topk_gate,
                         float* prob_partials, float* logits, void* workspace,
                         size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream);

/* The selection, softmax and gate steps of moe_route alone, on caller-given fp32 logits
 * [T, E] (same outputs, same rules). */
int moe_route_from_logits(const moe_problem* p, const float* logits, int32_t* topk_idx,
                          float* topk_gate, float* prob_partials, int32_t* dev_status,
                          moe_stream_t stream);

/* ==================================================================== dispatch
 * "Adapting Ultra-Large MoE Models ...", section 3.3 (capacity factor, token dropping,
 * batch reshaping into per-expert GEMM batches); "Trillion-Parameter MoE Model Training
 * Adaptation ...", section 3 "Communication" (tokens permuted by routing result).
 *
 *   C = ceil(cf * T * k / E)   (no limit when cap_den == 0)
 *   counts[e]      slots routed to expert e before any drop
 *   pos(t, j)      number of tokens t' < t routed to the same expert (arrival order)
 *   a slot is kept iff pos < C; kept_e = min(counts[e], C)
 *   offsets[e]     exclusive prefix sum of kept_e; offsets[E] = n_kept
 *   slot_row[t*k+j] = offsets[e] + pos if kept, else -1
 *   row_slot[row]   inverse map for rows < n_kept; rows >= n_kept are set to -1
 *   n_kept_dropped  {n_kept, n_dropped}
 *   x_perm[row]     = x[row_slot[row] / k]  (rows >= n_kept are left untouched)
 * x and x_perm may both be NULL: then only the index maps are produced (for
 * moe_expert_ffn_gather, which reads the token rows itself).
 * Everything is deterministic and bit-exact.  topk_idx entries outside [0, E) set
 * MOE_ERR_BAD_INDEX in dev_status and are treated as dropped.
 * Sizes: counts [E], offsets [E+1], slot_row [T*k], row_slot [T*k] int32;
 * x [T, d] and x_perm [T*k, d] bf16.
 */
size_t moe_dispatch_workspace_size(const moe_problem* p);
int moe_dispatch(const moe_problem* p, const int32_t* topk_idx, const moe_bf16* x,
                 int32_t* counts, int32_t* offsets, int32_t* slot_row, int32_t* row_slot,
                 int32_t* n_kept_dropped, moe_bf16* x_perm, void* workspace,
                 size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream);

/* moe_dispatch without a workspace argument, for callers that cannot allocate device memory
 * (their device memory is owned by another allocator that must not be bypassed, or they are
 * handed tensor pointers with no way to call cudaMalloc).  The pages have no counterpart:
 * this is a deployment convenience of this library.  Same arguments, argument checks,
 * status codes and outputs (bit for bit) as moe_dispatch, including the index-maps-only
 * mode with x and x_perm both NULL.  The scratch is a fixed device array inside the library
 * (8 MiB per GPU that loads the library, held until the process exits); a problem needing
 * more than that (moe_dispatch_workspace_size(p) > 8 MiB) returns MOE_ERR_WORKSPACE without
 * enqueuing anything.  The first call on each device looks up the array's device address
 * (with that device current) and caches it, so make that first call before any stream
 * capture.  Every call shares the one array: calls that overlap on the GPU (e.g. on two
 * streams) race and must be serialised by the caller.  Allocates nothing (no
 * cudaMalloc/cudaFree). */
int moe_dispatch_noalloc(const moe_problem* p, const int32_t* topk_idx, const moe_bf16* x,
                         int32_t* counts, int32_t* offsets, int32_t* slot_row,
                         int32_t* row_slot, int32_t* n_kept_dropped, moe_bf16* x_perm,
                         int32_t* dev_status, moe_stream_t stream);

/* ==================================================================== overflow remapping
 * "Adapting Ultra-Large MoE Models ...", section 3.3: tokens beyond an expert's capacity are
 * handled by remapping or dropping.  The pages give no mechanism; the rule implemented:
 * token t orders all experts by the selection key (descending logit, ties -> lower index);
 * its first k are the selection, and slot j's alternatives are its preference ranks
 * j + k, j + 2k, ..., j + rounds * k (none selected, none shared by two of its slots).  Pass
 * 0 is moe_dispatch's rule; in round q = 1 .. rounds every slot still unplaced proposes its
 * q-th alternative and each expert takes the proposals in arrival order (ascending token,
 * then rank) while it holds fewer than C slots.  Slots unplaced after the last round are
 * dropped.  A remapped slot keeps its gate topk_gate[t, j] (moe_expert_ffn reads gates by
 * slot, so nothing else changes).  Within an expert the rows are in placement order: pass 0,
 * then round 1, ..., arrival order inside each.  counts stays the pre-drop histogram of the
 * original selection (what moe_aux_loss uses).
 *
 * moe_route_alternatives: alt_idx [T, n_alt] int32 = each token's preference ranks
 * k .. k + n_alt - 1 from the fp32 logits moe_route wrote (pass moe_route a logits buffer);
 * n_alt = rounds * k; k + n_alt <= min(32, E).
 * moe_dispatch_remap: outputs as moe_dispatch (x, x_perm both NULL: index maps only), plus
 * slot_expert [T*k] int32 (may be NULL): the expert each slot was placed on, -1 if dropped.
 * rounds = 0 gives moe_dispatch's result.  (rounds + 1) * k <= min(32, E).  Deterministic.
 */
int moe_route_alternatives(const moe_problem* p, const float* logits, int32_t n_alt,
                           int32_t* alt_idx, moe_stream_t stream);
size_t moe_dispatch_remap_workspace_size(const moe_problem* p, int32_t rounds);
int moe_dispatch_remap(const moe_problem* p, const int32_t* topk_idx, const int32_t* alt_idx,
                       int32_t rounds, const moe_bf16* x, int32_t* counts, int32_t* offsets,
                       int32_t* slot_row, int32_t* row_slot, int32_t* slot_expert,
                       int32_t* n_kept_dropped, moe_bf16* x_perm, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream);

/* ==================================================================== expert parallelism
 * The exchange of "Trillion-Parameter MoE Model Training Adaptation: Full-Stack Optimization
 * Practices", section 3 "Communication" (tokens permuted by routing result are sent with an
 * All-to-All to the GPUs hosting their experts, computed in grouped GEMMs, unpermuted and
 * returned) and section 4.1 (EP: the experts split evenly over the ranks, E/P contiguous
 * experts per rank).  The collectives themselves are the caller's (NCCL or any all-to-all);
 * these calls are the per-rank steps around them.
 *
 * moe_expert_counts: counts[e] = number of slots of topk_idx routed to expert e (before any
 * drop), overwritten.  Deterministic.  counts [E] int32.
 *
 * moe_dispatch_ep: moe_dispatch for one part of a larger batch (one rank's tokens, or one
 * chunk of them) when the capacity is shared with the rest of the batch in global arrival
 * order.  capacity: C of the whole batch, computed by the caller (ceil(cf * T_total * k / E));
 * negative = no limit (p's cap_num / cap_den are not used).  pos_base [E] int32 (device, may
 * be NULL = all zeros) holds, per expert, the number of its slots that arrived earlier in the
 * batch (on earlier ranks or chunks); a slot at local position pos is kept iff
 * pos_base[e] + pos < C, so kept_e = clamp(C - pos_base[e], 0, counts[e]) and offsets is
 * their exclusive scan.  With pos_base and gate_perm NULL and C = moe_dispatch's it equals
 * moe_dispatch.  gate_perm [T*k] fp32 (may be NULL): gate_perm[row] =
 * topk_gate[row_slot[row]], the gate travelling with each permuted row to the rank that
 * computes it.  Workspace: as moe_dispatch (moe_dispatch_workspace_size).
 *
 * moe_ep_regroup: moves rows (d bf16 values each) and optionally one fp32 gate per row
 * between the two layouts of the exchange.  kept [n_sources * n_local_experts] int32
 * (device): rows of (source s, local expert e) at index s * n_local_experts + e.
 * Source-major layout: blocks ordered (s, e), as an all-to-all delivers them; expert-major:
 * blocks ordered (e, s), one contiguous group per local expert for the grouped GEMM (sources
 * in rank order, i.e. global arrival order).  to_expert_major = 1 moves source-major src
 * into expert-major dst, 0 the reverse.  rows_total = the sum of kept (a launch-size hint,
 * known to the caller from the counts exchange).  expert_offsets [n_local_experts + 1]
 * (may be NULL) receives the expert-major group starts.  src and dst must not overlap.
 */
int moe_expert_counts(const moe_problem* p, const int32_t* topk_idx, int32_t* counts,
                      int32_t* dev_status, moe_stream_t stream);
int moe_dispatch_ep(const moe_problem* p, int32_t capacity, const int32_t* topk_idx,
                    const float* topk_gate, const moe_bf16* x, const int32_t* pos_base,
                    int32_t* counts, int32_t* offsets, int32_t* slot_row, int32_t* row_slot,
                    int32_t* n_kept_dropped, moe_bf16* x_perm, float* gate_perm,
                    void* workspace, size_t workspace_bytes, int32_t* dev_status,
                    moe_stream_t stream);
int moe_ep_regroup(const moe_bf16* src, const float* gate_src, const int32_t* kept,
                   int32_t n_sources, int32_t n_local_experts, int32_t d,
                   int32_t to_expert_major, int64_t rows_total, moe_bf16* dst,
                   float* gate_dst, int32_t* expert_offsets, moe_stream_t stream);

/* ==================================================================== experts
 * Grouped SwiGLU expert GEMMs with LoRA ("Trillion-Parameter MoE Model Training
 * Adaptation ...", section 4.3: grouped GEMM over experts; "Adapting Trillion-Parameter
 * MoE Models ...", section 3, equation 1: LoRA).  For every permuted row of expert e
 * (rows offsets[e] .. offsets[e+1]-1 of x_perm):
 *
 *   a_g = x W_g[e]^T + s (x A_g[e]^T) B_g[e]^T        (fp32 accumulate)
 *   a_u = x W_u[e]^T + s (x A_u[e]^T) B_u[e]^T
 *   h   = silu(a_g) * a_u                             -> h [rows, F] bf16
 *   o   = h W_d[e]^T + s (h A_d[e]^T) B_d[e]^T
 *   y_perm[row] = topk_gate[row_slot[row]] * o        -> y_perm [rows, d] bf16
 *
 * w_gate, w_up [E, F, d]; w_down [E, d, F] bf16.  lora may be NULL.  saved may be NULL.
 * offsets [E+1] int32 (device); rows_max bounds offsets[E] and sizes x_perm/h/y_perm.
 * topk_gate is indexed by slot (row_slot), as written by moe_route/moe_dispatch.
 */
size_t moe_expert_ffn_workspace_size(const moe_problem* p, int32_t rows_max);
int moe_expert_ffn(const moe_problem* p, int32_t rows_max, const moe_bf16* x_perm,
                   const int32_t* offsets, const int32_t* row_slot, const float* topk_gate,
                   const moe_bf16* w_gate, const moe_bf16* w_up, const moe_bf16* w_down,
                   const moe_lora* lora, moe_bf16* h, moe_bf16* y_perm,
                   const moe_ffn_saved* saved, void* workspace, size_t workspace_bytes,
                   int32_t* dev_status, moe_stream_t stream);

/* moe_expert_ffn with the permute fused into the first GEMMs ("Trillion-Parameter MoE Model
 * Training Adaptation ...", section 4.3: deep fusion of Permute and Grouped GEMM): operand
 * rows are gathered from the token matrix x [T, d] by slot, row r reading
 * x[row_slot[r] / k], so no permuted copy of x is written or read.  Same outputs as
 * moe_expert_ffn given x_perm = the dispatch gather of x. */
int moe_expert_ffn_gather(const moe_problem* p, int32_t rows_max, const moe_bf16* x,
                          const int32_t* offsets, const int32_t* row_slot,
                          const float* topk_gate, const moe_bf16* w_gate, const moe_bf16* w_up,
                          const moe_bf16* w_down, const moe_lora* lora, moe_bf16* h,
                          moe_bf16* y_perm, const moe_ffn_saved* saved, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream);

/* moe_expert_ffn with the unpermute fused into the down GEMM ("Trillion-Parameter MoE Model
 * Training Adaptation ...", section 4.3: deep fusion of Permute, Unpermute and Grouped GEMM):
 * y [T, d] bf16 is written by the GEMM's epilogue, bit for bit what moe_combine computes
 * from y_perm (which is still written: the epilogue reads the token's other rows from it).
 * Deterministic: every stored row counts down a per-(token, 256-column strip) counter, and
 * the warp that stores a token's last row of a strip sums that token's kept rows in rank
 * order (j = 0 .. k-1, fp32, one rounding), exactly as moe_combine does; no atomic touches
 * the sum.  a_is_tokens = 1: a_src is the token matrix x [T, d] gathered by slot (as
 * moe_expert_ffn_gather), 0: the permuted rows x_perm.  slot_row [T*k] from the dispatch.
 * Workspace: moe_expert_ffn_combine_workspace_size (the expert workspace plus one counter
 * per token and strip). */
size_t moe_expert_ffn_combine_workspace_size(const moe_problem* p, int32_t rows_max);
int moe_expert_ffn_combine(const moe_problem* p, int32_t rows_max, const moe_bf16* a_src,
                           int32_t a_is_tokens, const int32_t* offsets, const int32_t* row_slot,
                           const int32_t* slot_row, const float* topk_gate,
                           const moe_bf16* w_gate, const moe_bf16* w_up,
                           const moe_bf16* w_down, const moe_lora* lora, moe_bf16* h,
                           moe_bf16* y_perm, moe_bf16* y, const moe_ffn_saved* saved,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           moe_stream_t stream);

/* ==================================================================== combine / aux
 * Unpermute and sum ("Trillion-Parameter MoE Model Training Adaptation ...", section 3
 * "Communication": results are unpermuted and returned):
 *   y[t] = sum_{j = 0..k-1, slot_row[t*k+j] >= 0} y_perm[slot_row[t*k+j]]
 * summed in rank order in fp32, rounded once to bf16.  A token whose slots were all
 * dropped gets y[t] = 0.  y_perm [rows, d], y [T, d] bf16.
 */
int moe_combine(const moe_problem* p, const moe_bf16* y_perm, const int32_t* slot_row,
                moe_bf16* y, moe_stream_t stream);

/* Auxiliary load-balancing loss ("Day-Level Adaptation ...", section 2.1):
 *   aux = E * sum_e f_e P_e,  f_e = counts[e] / (T k) (before drops),
 *   P_e = (1/T) sum_b prob_partials[b, e].   aux_out: one fp32 in device memory.
 * The reduction runs in a fixed order (deterministic). */
size_t moe_aux_loss_workspace_size(const moe_problem* p);
int moe_aux_loss(const moe_problem* p, const int32_t* counts, const float* prob_partials,
                 int32_t n_partials, float* aux_out, void* workspace, size_t workspace_bytes,
                 moe_stream_t stream);

/* ==================================================================== backward
 * Gradient of <dy, y> with the routing decisions of the forward held fixed ("Day-Level
 * Adaptation ...", section 5: checkpoint boundaries avoid dynamic routing) and the base
 * weights and the router frozen ("Adapting Trillion-Parameter MoE Models ...", section 3:
 * only adapter parameters are trained; routing gates are not tuned).
 */

/* dz_perm[row] = g(slot) * dy[t]  (bf16, rows < n_kept);
 * dgate[t*k+j] = <dy[t], o(row)> = <dy[t], y_perm[row]> / g(slot) for kept slots, else 0.
 * dy [T, d] bf16; y_perm [rows, d] bf16 (forward output) or NULL; dgate [T*k] fp32.
 * With y_perm NULL the kept slots' gate gradients are left to moe_expert_ffn_bwd (which
 * forms them from its dh product without reading y_perm again): dgate, if given, is then
 * set to 0 for every slot. */
int moe_combine_bwd(const moe_problem* p, const moe_bf16* dy, const moe_bf16* y_perm,
                    const int32_t* slot_row, const float* topk_gate, moe_bf16* dz_perm,
                    float* dgate, moe_stream_t stream);

/* Expert backward for the rows of every expert:
 *   dh   = dz W_d + s (dz B_d) A_d;   da_g = dh * a_u * silu'(a_g);   da_u = dh * silu(a_g)
 *   dx_perm = da_g W_g + da_u W_u + s (da_g B_g) A_g + s (da_u B_u) A_u     (bf16 out)
 *   dB_d = s dz^T (h A_d^T),  dA_d = s (dz B_d)^T h,  and likewise for gate and up.
 * saved must hold a_gate and a_up (and u_* when lora is given); h is the forward's h.
 * grads may be NULL when lora is NULL.
 * dgate (optional, with row_slot [rows] and topk_gate [T*k] per slot): the gate gradients
 * of the kept slots, dgate[row_slot[r]] = <dh_r, h_r> / g = <dy[t], o_r> (dh = g dy W_d +
 * ... is linear in dy; h_r = silu(a_g) a_u recomputed in fp32 in the dh epilogue); other
 * slots are not written (see moe_combine_bwd with y_perm NULL). */
size_t moe_expert_ffn_bwd_workspace_size(const moe_problem* p, int32_t rows_max);
int moe_expert_ffn_bwd(const moe_problem* p, int32_t rows_max, const moe_bf16* x_perm,
                       const int32_t* offsets, const moe_bf16* w_gate, const moe_bf16* w_up,
                       const moe_bf16* w_down, const moe_lora* lora,
                       const moe_ffn_saved* saved, const moe_bf16* h, const moe_bf16* dz_perm,
                       moe_bf16* dx_perm, const moe_lora_grad* grads,
                       const int32_t* row_slot, const float* topk_gate, float* dgate,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status,
                       moe_stream_t stream);

/* dx[t] = sum over kept slots of dx_perm[slot_row[t*k+j]]   (fp32 [T, d], overwritten) */
int moe_dispatch_bwd(const moe_problem* p, const moe_bf16* dx_perm, const int32_t* slot_row,
                     float* dx, moe_stream_t stream);

/* Gate path through the renormalised softmax and the frozen router, accumulated:
 *   dlogit[t, e_j] = g_j (dgate_j - sum_i g_i dgate_i)   (zero off the selection)
 *   dx[t] += sum_j dlogit[t, e_j] * w_router[e_j]          (fp32 [T, d]) */
int moe_route_bwd(const moe_problem* p, const int32_t* topk_idx, const float* topk_gate,
                  const float* dgate, const float* w_router, float* dx, moe_stream_t stream);

/* moe_dispatch_bwd followed by moe_route_bwd in one pass over dx (each token's row read and
 * written once; the same order of operations, so the same bits). */
int moe_dispatch_route_bwd(const moe_problem* p, const moe_bf16* dx_perm,
                           const int32_t* slot_row, const int32_t* topk_idx,
                           const float* topk_gate, const float* dgate, const float* w_router,
                           float* dx, moe_stream_t stream);

/* ==================================================================== instrumentation
 * Profiling aids, not part of the layer.  moe_set_kernel_events() makes the library record
 * the caller's CUDA events (cudaEvent_t, passed as void*) on the launch stream immediately
 * before and after its next launches of the given kernel, so that a caller can time one
 * kernel inside a longer sequence; pass NULL events to stop.  moe_launch_count() returns
 * the number of kernels this process has launched through the library.  Both use
 * process-wide state and are not thread-safe. */
enum moe_kernel_id {
  MOE_KERNEL_ROUTER_GEMM = 0,   /* split-bf16 router product -> fp32 logits      */
  MOE_KERNEL_TOPK = 1,          /* softmax, top-k, gates, probability partials  */
  MOE_KERNEL_DISPATCH = 2,      /* the four dispatch kernels, count to gather    */
  MOE_KERNEL_GATEUP_GEMM = 3,   /* grouped gate/up GEMM with SwiGLU (+LoRA)      */
  MOE_KERNEL_DOWN_GEMM = 4,     /* grouped down GEMM with gate scaling (+LoRA)   */
  MOE_KERNEL_COMBINE = 5,       /* weighted unpermute and sum                    */
  MOE_KERNEL_BWD_DH_GEMM = 6,   /* backward dh GEMM with the SwiGLU backward      */
  MOE_KERNEL_BWD_DX_GEMM = 7,   /* backward dx_perm GEMM                         */
  MOE_KERNEL_WGRAD = 8,         /* the LoRA weight-gradient GEMMs (first to last) */
  MOE_KERNEL_GDR_CHUNK = 9,     /* linear attention: per-chunk factors           */
  MOE_KERNEL_GDR_SCAN = 10,     /* linear attention: state scan over chunks      */
  MOE_KERNEL_GDR_BWD = 11,      /* linear attention: per-chunk backward          */
  MOE_KERNEL_COMBINE_BWD = 12,  /* combine backward (dz_perm, gate gradients)    */
  MOE_KERNEL_DISPATCH_ROUTE_BWD = 13, /* dx from dx_perm and the router path      */
  MOE_KERNEL_GDR_BWD_FACTORS = 14, /* linear attention backward: chunk factors again */
  MOE_KERNEL_GDR_BWD_SCAN = 15, /* linear attention backward: state-gradient scan  */
  MOE_KERNEL_COUNT = 16
};
int moe_set_kernel_events(int kernel_id, void* event_before, void* event_after);
long long moe_launch_count(void);

/* Self-test of the bounded waits: launches one tiny kernel that waits on an mbarrier nothing
 * arrives on, gives up after timeout_ms (1..2000) and writes MOE_ERR_TIMEOUT to *dev_status,
 * exactly as a stalled pipeline stage of a GEMM would.  The kernel ends on its own; the
 * context stays usable. */
int moe_selftest_wait_timeout(int32_t* dev_status, int32_t timeout_ms, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */

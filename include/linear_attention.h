/*
 * linear_attention.h -- C ABI of the chunked gated delta-rule linear attention in
 * libmoe.so (the second workload of the hot path).
 *
 * "Fine-Tuning Trillion-Parameter Sparse MoE Models: Challenges and Engineering Practices",
 * section 5 (large fused forward and backward kernels for linear attention: normalization
 * coefficients, gating and decay, intra-chunk query-state interaction and the output; fixed
 * chunks computed with dense intra-chunk products and one small state recurrence between
 * chunks) and "Adapting Ultra-Large MoE Models: Engineering Practices and Optimization
 * Pathways", section 3.2 (state recursion and chunked computation).  The pages give no
 * equations; the operator implemented is the gated delta rule, per sequence b and head h:
 *
 *   q^_t = q_t / ||q_t||,  k^_t = k_t / ||k_t||            (L2 over the key width dk)
 *   S_t  = exp(g_t) S_{t-1} (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T     S_t [dv, dk]
 *   o_t  = scale * S_t q^_t
 *
 * Conventions as in moe.h (status codes, caller-owned device pointers, asynchronous on
 * `stream`, no allocation: scratch is the caller's workspace).  Layouts (row-major):
 *   q, k [B, T, H, dk] bf16;  v [B, T, H, dv] bf16;  beta, g [B, T, H] fp32 (beta in [0, 1],
 *   g <= 0 the log decay);  S0 [B, H, dv, dk] fp32 initial state or NULL (zero);
 *   o [B, T, H, dv] bf16;  S_T [B, H, dv, dk] fp32 final state or NULL;
 *   S_chunks [B, H, ceil(T/64), dv, dk] fp32 or NULL: the state at the start of every
 *   64-token chunk (what a backward pass restarts from);  W_chunks [B, H, ceil(T/64), 64, dv]
 *   fp32 or NULL: every chunk's W = U - Y S0^T (its tokens' values corrected by the state at
 *   the chunk start; rows past the sequence zero), which the backward then reads instead of
 *   forming it again.
 * Supported: dk and dv in {64, 128}; any T >= 1 (the last chunk may be partial).  A zero
 * q or k row is treated as a zero vector (no division by zero).  q, k, v, the workspace, the
 * forward's o, W_chunks (and the backward's d_o, S_chunks, W_chunks) must be 16-byte aligned (the kernels move
 * them in 16-byte pieces), else MOE_ERR_UNSUPPORTED.
 *
 * Precision: the state and every accumulation are fp32.  The forward scan's products run on
 * the tensor cores with each fp32 operand carried as two bf16 pieces (hi = bf16(x), mid =
 * bf16(x - hi); three MMAs hi.hi + hi.mid + mid.hi): about 2^-16 relative per product.
 */
#ifndef MOE_LINEAR_ATTENTION_H
#define MOE_LINEAR_ATTENTION_H

#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Workspace bytes of moe_gdr_forward (the per-chunk factors: about
 * 4 * (3 dk + dv + 65) bytes per token and head), 0 for non-positive sizes. */
size_t moe_gdr_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv);

/* Forward of the gated delta rule over all B x H sequences (two launches: the per-chunk
 * factors of every chunk in parallel, then the scan over chunks in slices of 16 value rows
 * of the state, on the tensor cores).  The scan's waits on its own tensor-core work are
 * bounded; one that runs out ends the scan early and records MOE_ERR_TIMEOUT for
 * moe_gdr_device_status. */
int moe_gdr_forward(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, const moe_bf16* q,
                    const moe_bf16* k, const moe_bf16* v, const float* beta, const float* g,
                    const float* S0, float scale, moe_bf16* o, float* S_T, float* S_chunks,
                    float* W_chunks, void* workspace, size_t workspace_bytes,
                    moe_stream_t stream);

/* Device-side status of the linear-attention kernels: waits for `stream`, writes the first
 * error a kernel recorded since the previous call (MOE_OK if none; MOE_ERR_TIMEOUT when a
 * bounded wait ran out, the outputs of that launch then being incomplete) to *status and
 * clears it.  Returns MOE_ERR_INVALID_ARG for a NULL status, MOE_ERR_CUDA if the stream or
 * the copy failed. */
int moe_gdr_device_status(int32_t* status, moe_stream_t stream);

/* Backward: gradients of <d_o, o> + <dS_T, S_T> with respect to q, k, v, beta, g and S0
 * (three launches: the per-chunk factors rebuilt, a backward scan over chunks for the state
 * gradient in slices of 16 value rows on the tensor cores (bounded waits as in the forward,
 * reported through moe_gdr_device_status), then every chunk's local backward in
 * parallel).
 * S_chunks: the forward's chunk-start states (required); W_chunks: the forward's W_chunks, or
 * NULL (then formed again from S_chunks).  d_o [B, T, H, dv] bf16; dS_T
 * [B, H, dv, dk] fp32 or NULL (zero).  Outputs fp32, overwritten: dq, d_k [B, T, H, dk],
 * d_v [B, T, H, dv], dbeta, dg [B, T, H], dS0 [B, H, dv, dk] (may be NULL).  Deterministic:
 * every reduction runs in a fixed order. */
size_t moe_gdr_backward_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk,
                                       int32_t dv);
int moe_gdr_backward(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, const moe_bf16* q,
                     const moe_bf16* k, const moe_bf16* v, const float* beta, const float* g,
                     float scale, const moe_bf16* d_o, const float* dS_T, const float* S_chunks,
                     const float* W_chunks,
                     float* dq, float* d_k, float* d_v, float* dbeta, float* dg, float* dS0,
                     void* workspace, size_t workspace_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LINEAR_ATTENTION_H */

// Internal declarations shared by the translation units of libmoe.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Bounded device-side waits give up after this much wall time (ns).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

inline size_t up256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Entry-point helpers shared by the files of the C ABI (defined in capi.cu).
int check_problem(const moe_problem* p);    // MOE_OK or the status an entry point returns
int capacity_of(const moe_problem* p);      // ceil(cf * T * k / E), -1 for cf = infinity
size_t dispatch_ws(const moe_problem* p);   // scratch bytes of the dispatch kernels
// Instrumentation (moe_set_kernel_events / moe_launch_count): caller events recorded
// around a kernel's launches, and the process-wide launch counter.
void mark_before(int kernel_id, cudaStream_t s);
void mark_after(int kernel_id, cudaStream_t s);
void count_launches(int n);
long long launch_count();
int set_kernel_events(int kernel_id, void* event_before, void* event_after);

// ------------------------------------------------------------------ GEMM description
//
// One persistent tcgen05 kernel serves every contraction of the layer.  A CTA owns a
// 128-row output tile (or two, on 256-row tiles) and up to two accumulators of BN columns
// each (NB operands "B" sharing one operand "A"), walks a list of K segments (each segment
// names the tensor maps and K offsets its 64-wide K blocks come from), then runs a fused
// epilogue.

constexpr int kMaxMaps = 8;
constexpr int kMaxSegs = 4;
constexpr int kBM = 128;
constexpr int kBK = 64;

// Tile shapes of the grouped expert GEMMs: 128-row tiles, 256-row tiles in one CTA, or CTA
// pairs (an M = 256 tile over two SMs).
enum TileShape { kTile128 = 0, kTile256 = 1, kTilePair = 2 };

enum Epilogue : int {
  EPI_F32_BIAS = 0,    // out_f32[row, col] = acc0 + bias[col]           (router logits)
  EPI_SWIGLU = 1,      // out_bf16 = silu(acc0) * acc1; optional save of acc0/acc1 as bf16
  EPI_GATE_SCALE = 2,  // out_bf16 = gate[row_slot[row]] * acc0            (expert down)
  EPI_SCALE = 3,       // out_bf16_i = scale * acc_i for each B operand     (LoRA u, v)
  EPI_SWIGLU_BWD = 4,  // da_g, da_u from acc0 = dh and saved a_g, a_u
  EPI_STORE = 5,       // out_bf16 = acc0                                   (dx_perm)
  EPI_WGRAD = 6,       // grouped over K: out_f32_i[g] = acc_i, plain or transposed (LoRA grads)
  EPI_ROUTE = 7,       // EPI_F32_BIAS plus, per row and n-tile, max / sum exp / top-16 keys
};

// Candidates the fused router epilogue keeps per (token, expert tile): the tile's 16 largest
// (logit, expert) keys; routing with k <= 16 merges them exactly.
constexpr int kRouteTileK = 16;

struct GemmSeg {
  int nkb;        // number of 64-wide K blocks in this segment
  int a_map;      // tensor map of operand A
  int a_k0;       // K element offset of the first block in operand A
  int b_map[2];   // tensor map of each B operand, -1 = this accumulator skips the segment
  int b_k0[2];    // K element offset in each B operand
  int b_z[2];     // third coordinate of B for dense problems (ignored when grouped)
  int a_gather;   // 1: A rows are gathered by token from P.gather_src (a_map unused)
};

struct GemmParams {
  CUtensorMap maps[kMaxMaps];
  int nmaps;
  GemmSeg seg[kMaxSegs];
  int nseg;  // segment 0 must feed every accumulator: later segments add to what it wrote
  // M grouping.  Grouped: rows of group g are [group_off[g], group_off[g+1]) and its
  // m-tiles are numbered tile_off[g] .. tile_off[g+1]-1; B's third coordinate is g.
  // Dense (group_off == nullptr): one group of M rows, m_tiles tiles.
  const int* group_off;
  const int* tile_off;
  const int* pair_off;   // 256-row tiles: prefix over groups of ceil(m-tiles / 2)
  int G;
  int M;
  int m_tiles;
  int n_tiles;     // number of BN-wide column tiles of each accumulator
  int N;           // valid columns of each accumulator (stores are clipped to N)
  // epilogue operands
  void* out0;
  void* out1;
  void* out2;
  void* out3;
  int ldo;                  // leading dimension (elements) of the outputs
  const float* bias;        // EPI_F32_BIAS
  const float* gate;        // EPI_GATE_SCALE: gate per slot
  const int* row_slot;      // EPI_GATE_SCALE: slot per row
  const void* in0;          // EPI_SWIGLU_BWD: saved a_g
  const void* in1;          // EPI_SWIGLU_BWD: saved a_u
  float scale;              // EPI_SCALE
  int out_transposed;       // EPI_WGRAD: 1 -> out[g][n][m] (ld M), 0 -> out[g][m][n] (ld N)
  // A-row gather (segments with a_gather): row r of the problem reads token row
  // gather_slot[r] / gather_k of gather_src [gather_rows, gather_ld] bf16
  const int* gather_slot;
  int gather_k;
  int gather_rows;
  const void* gather_src;
  int gather_ld;
  int b_policy;             // L2 policy of B loads: 0 evict-first (streamed), 1 normal (reused)
  // Fused combine (EPI_GATE_SCALE with comb_cnt set): comb_cnt[t * n_tiles + n] counts the
  // rows of token t whose n-tile strip is not stored yet; the epilogue warp that stores the
  // last one sums the token's kept rows (comb_slot_row, rank order, fp32) into comb_y [T, N].
  int* comb_cnt;
  const int* comb_slot_row;
  void* comb_y;
  int comb_k;
  int* dev_status;
};

// Host helpers (gemm_host.cu).
int encode_map_kmajor(CUtensorMap* map, const void* base, uint64_t k_extent, uint64_t rows,
                      uint64_t groups, uint32_t box_rows);
int encode_map_mnmajor(CUtensorMap* map, const void* base, uint64_t mn_extent,
                       uint64_t k_rows, uint64_t groups);
int num_sms();

// Kernel launchers (gemm_fwd.cu).  Return cudaError_t as int.
int launch_gemm_router(const GemmParams& P, int bn, cudaStream_t s);  // BN 128|224
int launch_gemm_router_topk(const GemmParams& P, int bn, cudaStream_t s);  // + tile top-16
// BN=128, NB=2, SwiGLU / BN=256, NB=1, gate scale; shape: a TileShape
int launch_gemm_gateup(const GemmParams& P, int shape, cudaStream_t s);
int launch_gemm_down(const GemmParams& P, int shape, cudaStream_t s);
int launch_gemm_lora_u2(const GemmParams& P, int r, cudaStream_t s); // BN=r pad, NB=2
int launch_gemm_lora_u1(const GemmParams& P, int r, cudaStream_t s); // BN=r pad, NB=1

// Fused combine: counters = kept slots per (token, n-tile), y rows of tokens with no kept slot
// zeroed (dispatch.cu)
int launch_combine_prepare(const int32_t* slot_row, int T, int k, int n_tiles, int d,
                           int32_t* comb_cnt, __nv_bfloat16* y, cudaStream_t s);

// Backward instantiations (gemm_bwd.cu).  B operands MN-major (weights used transposed).
// shape: a TileShape (the 256-row shapes walk P.pair_off units)
int launch_gemm_bwd_dh(const GemmParams& P, int shape, cudaStream_t s);  // BN=256, SwiGLU bwd
int launch_gemm_bwd_dx(const GemmParams& P, int shape, cudaStream_t s);  // BN=256, store bf16
int launch_gemm_bwd_lora_v(const GemmParams& P, int r, cudaStream_t s);  // BN=r pad, scale
// LoRA weight gradients, grouped over K (rows of each expert); A and B MN-major.
int launch_gemm_wgrad(const GemmParams& P, int r, int nb, cudaStream_t s);

}  // namespace moe

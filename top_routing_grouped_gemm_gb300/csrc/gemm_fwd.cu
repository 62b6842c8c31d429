// Forward instantiations of the tcgen05 GEMM (router, expert gate/up, expert down, LoRA).
#include "gemm.cuh"

namespace moe {

// Two B operands (the hi and lo parts of the split router weights) share each A stage and
// sum into one accumulator.  On CTA pairs (M = 256 token rows over two SMs, each staging half
// of the bn expert rows of both parts; the weight map boxes are bn / 2 rows).
int launch_gemm_router(const GemmParams& P, int bn, cudaStream_t s) {
  if (bn == 224) return launch_gemm<224, 2, false, false, EPI_F32_BIAS, 5, 1, 1, 2>(P, s);
  return launch_gemm<128, 2, false, false, EPI_F32_BIAS, 6, 1, 1, 2>(P, s);
}

// The same product with the fused top-k epilogue (candidates to P.out1, statistics to
// P.out2).
int launch_gemm_router_topk(const GemmParams& P, int bn, cudaStream_t s) {
  if (bn == 224) return launch_gemm<224, 2, false, false, EPI_ROUTE, 3>(P, s);
  return launch_gemm<128, 2, false, false, EPI_ROUTE, 4>(P, s);
}

// Tile shapes of the grouped expert GEMMs (TileShape): 128-row tiles; 256-row tiles in one
// CTA (two 128-row subtiles sharing each B stage, one TMEM accumulator: P.pair_off units);
// CTA pairs (tcgen05.mma.cta_group::2 over two SMs, M = 256: each SM stages its own 128 A rows
// and half of the weight tile, and keeps two accumulators of its 128 rows).  Neither 256-row
// shape takes a gathered A operand.
int launch_gemm_gateup(const GemmParams& P, int shape, cudaStream_t s) {
  if (shape != kTile128 && P.gather_slot != nullptr) return static_cast<int>(cudaErrorInvalidValue);
  if (shape == kTilePair) return launch_gemm<128, 2, false, false, EPI_SWIGLU, 7, 1, 1, 2>(P, s);
  if (shape == kTile256) return launch_gemm<128, 2, false, false, EPI_SWIGLU, 3, 1, 2>(P, s);
  return launch_gemm<128, 2, false, false, EPI_SWIGLU, 4>(P, s);
}

// With CTA pairs the weight maps are encoded with 128-row boxes (each CTA's half of the
// 256-row weight tile).
int launch_gemm_down(const GemmParams& P, int shape, cudaStream_t s) {
  if (shape == kTilePair) return launch_gemm<256, 1, false, false, EPI_GATE_SCALE, 6, 1, 1, 2>(P, s);
  if (shape == kTile256) return launch_gemm<256, 1, false, false, EPI_GATE_SCALE, 3, 1, 2>(P, s);
  return launch_gemm<256, 1, false, false, EPI_GATE_SCALE, 4>(P, s);
}

// The LoRA down-projections (N = r) stream their A operand through two CTAs per SM: two
// independent TMA/MMA pipelines fill shared memory faster than one deeper ring.
int launch_gemm_lora_u2(const GemmParams& P, int r, cudaStream_t s) {
  if (r <= 16) return launch_gemm<16, 2, false, false, EPI_SCALE, 5, 2>(P, s);
  if (r <= 32) return launch_gemm<32, 2, false, false, EPI_SCALE, 4, 2>(P, s);
  return launch_gemm<64, 2, false, false, EPI_SCALE, 3, 2>(P, s);
}

int launch_gemm_lora_u1(const GemmParams& P, int r, cudaStream_t s) {
  if (r <= 16) return launch_gemm<16, 1, false, false, EPI_SCALE, 5, 2>(P, s);
  if (r <= 32) return launch_gemm<32, 1, false, false, EPI_SCALE, 5, 2>(P, s);
  return launch_gemm<64, 1, false, false, EPI_SCALE, 4, 2>(P, s);
}

}  // namespace moe

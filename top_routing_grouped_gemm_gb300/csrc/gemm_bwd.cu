// Backward instantiations of the tcgen05 GEMM.  The frozen weights enter transposed, i.e. as
// MN-major B operands read straight from their forward layout (no transposed copies).
#include "gemm.cuh"

namespace moe {

// dh = dz W_d (+ v'_d A_d), epilogue: SwiGLU backward -> da_g, da_u.  Tile shapes as the
// forward GEMMs (TileShape; each CTA of a pair reads two of the tile's four 64-wide boxes).
int launch_gemm_bwd_dh(const GemmParams& P, int shape, cudaStream_t s) {
  if (shape == kTilePair) return launch_gemm<256, 1, false, true, EPI_SWIGLU_BWD, 6, 1, 1, 2>(P, s);
  if (shape == kTile256) return launch_gemm<256, 1, false, true, EPI_SWIGLU_BWD, 3, 1, 2>(P, s);
  return launch_gemm<256, 1, false, true, EPI_SWIGLU_BWD, 4>(P, s);
}

// dx_perm = da_g W_g + da_u W_u (+ v'_g A_g + v'_u A_u)
int launch_gemm_bwd_dx(const GemmParams& P, int shape, cudaStream_t s) {
  if (shape == kTilePair) return launch_gemm<256, 1, false, true, EPI_STORE, 6, 1, 1, 2>(P, s);
  if (shape == kTile256) return launch_gemm<256, 1, false, true, EPI_STORE, 3, 1, 2>(P, s);
  return launch_gemm<256, 1, false, true, EPI_STORE, 4>(P, s);
}

// v' = s (dz B_d), s (da_g B_g), s (da_u B_u): N = r (<= 64, zero-filled to 64)
int launch_gemm_bwd_lora_v(const GemmParams& P, int r, cudaStream_t s) {
  (void)r;
  return launch_gemm<64, 1, false, true, EPI_SCALE, 4, 2>(P, s);  // two CTAs per SM, as the forward LoRA products
}

// LoRA weight gradients, reduction over each expert's rows
int launch_gemm_wgrad(const GemmParams& P, int r, int nb, cudaStream_t s) {
  (void)r;
  // small tiles with short K: two CTAs per SM keep twice as many tiles in flight
  if (nb == 2) return launch_gemm<64, 2, true, true, EPI_WGRAD, 3, 2>(P, s);
  return launch_gemm<64, 1, true, true, EPI_WGRAD, 4, 2>(P, s);
}

}  // namespace moe

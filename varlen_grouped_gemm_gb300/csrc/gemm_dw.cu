// Instantiations of the two-part varlen-K weight-gradient GEMMs (a translation unit of their own: sixteen
// kernels, compiled in parallel with the others).
#include "internal.h"

namespace vgg {

// Varlen-K weight gradient with a two-part A: the per-pair gradients as a bf16 high part and the bf16
// rounding of the rest (two UMMAs per K step into one accumulator), B the expert-sorted input rows.  A
// stage holds both A tiles and B (BN = 256: 64 KB, so three stages).  A tile reduces over one expert's
// rows only (a few stages), so the epilogue's TMEM drain and stores set much of the pace.  Eight epilogue
// warps when an expert's output is large (M N >= 2^22), four otherwise, by alternating A/B runs of the
// backward at d x n (dW gate/up: M = 2n, N = d): 7168 x 2048 7.40 -> 6.12 ms, 2880 x 2880 2.46 -> 2.06 ms
// with eight; 2048 x 512 230 -> 213 us, 1536 x 256 575 -> 557 us with four.  trans: the tile is D^T of the stored output
// (dW_down[e] = dO^T A' computed as A'^T dO: M = n, N = d), written through transposed 32 x 32 blocks.
// pair: CTA pairs on 256-row tiles (padded B rows; each CTA loads 128 of B's 256 columns).
cudaError_t run_dw_dual(int BN, bool f32, bool trans, bool pair, const GemmParams& p, const Maps& m, int grid,
                        cudaStream_t s) {
  constexpr int D = X_DUAL_A, DT = X_DUAL_A | X_TRANS, DP = X_DUAL_A | X_PAIR, DTP = X_DUAL_A | X_TRANS | X_PAIR;
  if (pair && BN == 256) {
    if (trans)
      return f32 ? launch_grouped_gemm<256, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true, 2, DTP>(p, m, grid, s)
                 : launch_grouped_gemm<256, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false, 2, DTP>(p, m, grid, s);
    return f32 ? launch_grouped_gemm<256, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true, 2, DP>(p, m, grid, s)
               : launch_grouped_gemm<256, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false, 2, DP>(p, m, grid, s);
  }
  if (BN == 256 && static_cast<long long>(p.M) * p.N >= (1ll << 22)) {
    if (trans)
      return f32 ? launch_grouped_gemm<256, 3, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true, 1, DT>(p, m, grid, s)
                 : launch_grouped_gemm<256, 3, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false, 1, DT>(p, m, grid, s);
    return f32 ? launch_grouped_gemm<256, 3, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true, 1, D>(p, m, grid, s)
               : launch_grouped_gemm<256, 3, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false, 1, D>(p, m, grid, s);
  }
  if (BN == 256) {
    if (trans)
      return f32 ? launch_grouped_gemm<256, 3, 4, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true, 1, DT>(p, m, grid, s)
                 : launch_grouped_gemm<256, 3, 4, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false, 1, DT>(p, m, grid, s);
    return f32 ? launch_grouped_gemm<256, 3, 4, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true, 1, D>(p, m, grid, s)
               : launch_grouped_gemm<256, 3, 4, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false, 1, D>(p, m, grid, s);
  }
  if (trans)
    return f32 ? launch_grouped_gemm<128, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true, 1, DT>(p, m, grid, s)
               : launch_grouped_gemm<128, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false, 1, DT>(p, m, grid, s);
  return f32 ? launch_grouped_gemm<128, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true, 1, D>(p, m, grid, s)
             : launch_grouped_gemm<128, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false, 1, D>(p, m, grid, s);
}

}  // namespace vgg

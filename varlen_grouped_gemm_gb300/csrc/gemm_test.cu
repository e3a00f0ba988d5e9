// Main loops with a plain fp32 store epilogue, for the integer-exact test exports.
#include "internal.h"

namespace vgg {

// pair: CTA pairs on 256-row, 256-column tiles (each CTA loads 128 columns of B: the same B boxes).
cudaError_t run_test_m(int gathered, int b_kmajor, bool pair, const GemmParams& p, const Maps& m, int grid,
                       cudaStream_t s) {
  if (pair && !gathered && b_kmajor)
    return launch_grouped_gemm<256, 6, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE, true, 2, X_PAIR>(p, m, grid, s);
  if (pair && !gathered)
    return launch_grouped_gemm<256, 6, 4, 1, A_TMA_K, B_TMA_MN3, VAR_M, EPI_STORE, true, 2, X_PAIR>(p, m, grid, s);
  if (gathered && b_kmajor)
    return launch_grouped_gemm<128, 6, 4, 1, A_GATHER_K, B_TMA_K3, VAR_M, EPI_STORE, true>(p, m, grid, s);
  if (gathered) return launch_grouped_gemm<128, 6, 4, 1, A_GATHER_K, B_TMA_MN3, VAR_M, EPI_STORE, true>(p, m, grid, s);
  if (b_kmajor) return launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE, true>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_MN3, VAR_M, EPI_STORE, true>(p, m, grid, s);
}

// The down projection's main loop with a two-part A (high part in a0, low part in a2), K-major B.
cudaError_t run_test_m_dual(bool pair, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (pair)
    return launch_grouped_gemm<256, 4, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE, true, 2, X_DUAL_A | X_PAIR>(p, m, grid,
                                                                                                          s);
  return launch_grouped_gemm<256, 3, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE, true, 1, X_DUAL_A>(p, m, grid, s);
}

}  // namespace vgg

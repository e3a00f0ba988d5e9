// Main loops with a plain fp32 store epilogue, for the integer-exact test exports.
#include "internal.h"

namespace vgg {

cudaError_t run_test_m(int gathered, int b_kmajor, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (gathered && b_kmajor)
    return launch_grouped_gemm<128, 6, 4, 1, A_GATHER_K, B_TMA_K3, VAR_M, EPI_STORE, true>(p, m, grid, s);
  if (gathered) return launch_grouped_gemm<128, 6, 4, 1, A_GATHER_K, B_TMA_MN3, VAR_M, EPI_STORE, true>(p, m, grid, s);
  if (b_kmajor) return launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE, true>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_MN3, VAR_M, EPI_STORE, true>(p, m, grid, s);
}

// The down projection's main loop with a two-part A (high part in a0, low part in a2), K-major B.
cudaError_t run_test_m_dual(const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  return launch_grouped_gemm<256, 3, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE, true, 1, X_DUAL_A>(p, m, grid, s);
}

}  // namespace vgg

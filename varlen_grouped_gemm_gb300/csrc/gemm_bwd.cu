// Backward grouped-GEMM instantiations.
#include "internal.h"

namespace vgg {

// dA' = dO[tok] W_down[e] (W_down read MN-major), epilogue: dS partial, dH, dU, A'
// ([SM] "4.2 Epilogue 융합": one epilogue emits dH, dS and A').
cudaError_t run_dact_dswiglu(int BN, const GemmParams& p, const CUtensorMap* m, int grid, cudaStream_t s) {
  if (BN == 256) return launch_grouped_gemm<256, 4, A_CP_K, B_TMA_MN3, VAR_M, EPI_DSWIGLU>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, A_CP_K, B_TMA_MN3, VAR_M, EPI_DSWIGLU>(p, m, grid, s);
}

// dXp = [dH | dU] [W_gate[e]; W_up[e]]  (reduction over 2n, B read MN-major from two maps)
cudaError_t run_dx_store(int BN, const GemmParams& p, const CUtensorMap* m, int grid, cudaStream_t s) {
  if (BN == 256) return launch_grouped_gemm<256, 4, A_TMA_K, B_TMA_MN3, VAR_M, EPI_STORE>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, A_TMA_K, B_TMA_MN3, VAR_M, EPI_STORE>(p, m, grid, s);
}

// Varlen-K weight gradients: D[e] = sum over the expert's rows of A_row^T B_row.
cudaError_t run_varlen_k_store(int BN, const GemmParams& p, const CUtensorMap* m, int grid, cudaStream_t s) {
  if (BN == 256) return launch_grouped_gemm<256, 4, A_CP_MN, B_CP_MN, VAR_K, EPI_STORE>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, A_CP_MN, B_CP_MN, VAR_K, EPI_STORE>(p, m, grid, s);
}

// Dense A^T B with both operands MN-major (router weight gradient X^T dlogits), split K.
cudaError_t run_dense_mn_store(int BN, const GemmParams& p, const CUtensorMap* m, int grid, cudaStream_t s) {
  if (BN == 256) return launch_grouped_gemm<256, 4, A_TMA_MN, B_TMA_MN2, VAR_NONE, EPI_STORE>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, A_TMA_MN, B_TMA_MN2, VAR_NONE, EPI_STORE>(p, m, grid, s);
}

}  // namespace vgg

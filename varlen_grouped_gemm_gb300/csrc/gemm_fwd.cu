// Forward grouped-GEMM instantiations: gate/up + SwiGLU, down + combine weight, router logits.
// Template arguments: BN, pipeline stages, epilogue warps, staged stores per epilogue warp, operand
// modes, grouping mode, epilogue, fp32 output.
#include "internal.h"

namespace vgg {

// [GG] "(6) 세 번의 gg.gmm" gate and up in one pass: the B tile holds BN/2 rows of W_gate[e]
// and the same BN/2 rows of W_up[e], so the epilogue sees h and u of the same columns.
// A = X rows gathered through sorted_tok ([SM] "4.1 Gather 융합").
// cn > 1: clusters of cn CTAs on consecutive column tiles of one row tile gather a cn-th of the
// A rows each and pass them to one another through distributed shared memory.
cudaError_t run_gate_up_swiglu(int BN, int cn, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256) {
    if (cn == 4)
      return launch_grouped_gemm<256, 4, 4, 1, A_GATHER_K, B_TMA_K3_GU, VAR_M, EPI_SWIGLU, false, 4>(p, m, grid, s);
    if (cn == 2)
      return launch_grouped_gemm<256, 4, 4, 1, A_GATHER_K, B_TMA_K3_GU, VAR_M, EPI_SWIGLU, false, 2>(p, m, grid, s);
    return launch_grouped_gemm<256, 4, 4, 1, A_GATHER_K, B_TMA_K3_GU, VAR_M, EPI_SWIGLU, false>(p, m, grid, s);
  }
  return launch_grouped_gemm<128, 6, 4, 1, A_GATHER_K, B_TMA_K3_GU, VAR_M, EPI_SWIGLU, false>(p, m, grid, s);
}

// Down projection, A = sorted activation rows, epilogue scales by the combine weight.
cudaError_t run_down_scale(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256) return launch_grouped_gemm<256, 4, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_SCALE, false>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_SCALE, false>(p, m, grid, s);
}

// The down projection with A as a bf16 high part and the bf16 rounding of the rest (two UMMAs per K step
// into one accumulator); a stage holds both A tiles and B (BN = 256: 64 KB, three stages).
// A CTA pair (pair: each CTA loads 128 of the 256 columns of B) takes 48 KB stages, four of them.
cudaError_t run_down_scale_dual(int BN, bool pair, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (pair && BN == 256)
    return launch_grouped_gemm<256, 4, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_SCALE, false, 2, X_DUAL_A | X_PAIR>(p, m,
                                                                                                          grid, s);
  if (BN == 256)
    return launch_grouped_gemm<256, 3, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_SCALE, false, 1, X_DUAL_A>(p, m, grid, s);
  return launch_grouped_gemm<128, 4, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_SCALE, false, 1, X_DUAL_A>(p, m, grid, s);
}

// Router logits X[T,d] W_r[d,E] (+ bias), W_r read MN-major, fp32 out.
cudaError_t run_router_logits(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256) return launch_grouped_gemm<256, 4, 4, 1, A_TMA_K, B_TMA_MN2, VAR_NONE, EPI_STORE, true>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_MN2, VAR_NONE, EPI_STORE, true>(p, m, grid, s);
}

}  // namespace vgg

// Backward grouped-GEMM instantiations.  Template arguments as in gemm_fwd.cu; the dSwiGLU kernel,
// whose epilogue writes three outputs per tile, uses 8 epilogue warps and 2 staged stores per warp,
// paid for with one pipeline stage.
#include "internal.h"

namespace vgg {

// dA' = dO_sorted W_down[e] (W_down read MN-major), epilogue: dS partial, dH, dU, A'
// ([SM] "4.2 Epilogue 융합": one epilogue emits dH, dS and A').
// Four stages with one staged store per epilogue warp when the group table leaves room (measured
// 5-7% faster than three stages with two).
// A CTA pair (pair: each CTA loads 128 of the 256 columns of B) takes 32 KB stages, so six fit.
cudaError_t run_dact_dswiglu(int BN, bool pair, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (pair && BN == 256 && SmemLayout<256, 6, 8, 1, 1, 128>::bytes(p.groups, VAR_M) <= kMaxSmem)
    return launch_grouped_gemm<256, 6, 8, 1, A_TMA_K, B_TMA_MN3, VAR_M, EPI_DSWIGLU, false, 2, X_PAIR>(p, m, grid, s);
  if (pair && BN == 256)
    return launch_grouped_gemm<256, 5, 8, 1, A_TMA_K, B_TMA_MN3, VAR_M, EPI_DSWIGLU, false, 2, X_PAIR>(p, m, grid, s);
  if (BN == 256 && SmemLayout<256, 4, 8, 1>::bytes(p.groups, VAR_M) <= kMaxSmem)
    return launch_grouped_gemm<256, 4, 8, 1, A_TMA_K, B_TMA_MN3, VAR_M, EPI_DSWIGLU, false>(p, m, grid, s);
  if (BN == 256) return launch_grouped_gemm<256, 3, 8, 2, A_TMA_K, B_TMA_MN3, VAR_M, EPI_DSWIGLU, false>(p, m, grid, s);
  return launch_grouped_gemm<128, 4, 8, 2, A_TMA_K, B_TMA_MN3, VAR_M, EPI_DSWIGLU, false>(p, m, grid, s);
}

// dXp = [dH | dU] [W_gate[e]; W_up[e]]  (reduction over 2n, B read MN-major from two maps)
cudaError_t run_dx_store(int BN, bool pair, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (pair && BN == 256)
    return launch_grouped_gemm<256, 6, 4, 1, A_TMA_K, B_TMA_MN3, VAR_M, EPI_STORE, false, 2, X_PAIR>(p, m, grid, s);
  if (BN == 256) return launch_grouped_gemm<256, 4, 4, 1, A_TMA_K, B_TMA_MN3, VAR_M, EPI_STORE, false>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_MN3, VAR_M, EPI_STORE, false>(p, m, grid, s);
}

// Varlen-K weight gradient with both operands read by TMA from expert-sorted rows; the rows past the
// group's end in its last stage are cleared in shared memory before the last UMMAs.  A tile reduces
// over one expert's rows only (a few stages), so the ring's depth sets the bytes in flight: 4 stages
// and one staged store per epilogue warp measured faster than 3 stages with two.
cudaError_t run_dw_tiled(int BN, bool f32, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256)
    return f32 ? launch_grouped_gemm<256, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true>(p, m, grid, s)
               : launch_grouped_gemm<256, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false>(p, m, grid, s);
  return f32 ? launch_grouped_gemm<128, 6, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true>(p, m, grid, s)
             : launch_grouped_gemm<128, 6, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false>(p, m, grid, s);
}

// The same with the tile written transposed (dW_down[e] = dO^T A' computed as A'^T dO: M = n, N = d, each 32 x 32
// block transposed while it is staged), for the single-part A' of the e4m3 and block-scaled backward.
cudaError_t run_dw_tiled_trans(int BN, bool f32, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256)
    return f32 ? launch_grouped_gemm<256, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true, 1, X_TRANS>(p, m, grid, s)
               : launch_grouped_gemm<256, 4, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false, 1, X_TRANS>(p, m, grid, s);
  return f32 ? launch_grouped_gemm<128, 6, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, true, 1, X_TRANS>(p, m, grid, s)
             : launch_grouped_gemm<128, 6, 8, 1, A_TMA_MN, B_TMA_MN2, VAR_K, EPI_STORE, false, 1, X_TRANS>(p, m, grid, s);
}

// Varlen-K with one operand gathered through a token index (cp.async, zero past the group's end).
cudaError_t run_dw_gate_up(int BN, bool f32, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256)
    return f32 ? launch_grouped_gemm<256, 4, 4, 1, A_TMA_MN, B_GATHER_MN, VAR_K, EPI_STORE, true>(p, m, grid, s)
               : launch_grouped_gemm<256, 4, 4, 1, A_TMA_MN, B_GATHER_MN, VAR_K, EPI_STORE, false>(p, m, grid, s);
  return f32 ? launch_grouped_gemm<128, 6, 4, 1, A_TMA_MN, B_GATHER_MN, VAR_K, EPI_STORE, true>(p, m, grid, s)
             : launch_grouped_gemm<128, 6, 4, 1, A_TMA_MN, B_GATHER_MN, VAR_K, EPI_STORE, false>(p, m, grid, s);
}

cudaError_t run_dw_down(int BN, bool f32, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256)
    return f32 ? launch_grouped_gemm<256, 4, 4, 1, A_GATHER_MN, B_TMA_MN2, VAR_K, EPI_STORE, true>(p, m, grid, s)
               : launch_grouped_gemm<256, 4, 4, 1, A_GATHER_MN, B_TMA_MN2, VAR_K, EPI_STORE, false>(p, m, grid, s);
  return f32 ? launch_grouped_gemm<128, 6, 4, 1, A_GATHER_MN, B_TMA_MN2, VAR_K, EPI_STORE, true>(p, m, grid, s)
             : launch_grouped_gemm<128, 6, 4, 1, A_GATHER_MN, B_TMA_MN2, VAR_K, EPI_STORE, false>(p, m, grid, s);
}

// Dense A^T B with both operands MN-major (router weight gradient X^T dlogits), split K, fp32 out.
cudaError_t run_dense_mn_store(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256) return launch_grouped_gemm<256, 4, 4, 1, A_TMA_MN, B_TMA_MN2, VAR_NONE, EPI_STORE, true>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, 4, 1, A_TMA_MN, B_TMA_MN2, VAR_NONE, EPI_STORE, true>(p, m, grid, s);
}

}  // namespace vgg

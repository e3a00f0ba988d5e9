// Declarations shared by the translation units of the library (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm.cuh"

namespace vgg {

// ---- tensor maps (host) -------------------------------------------------------------------
// Operand loads, bf16, 128-byte swizzle: 2-D view [rows][inner] with a row stride, box {64, box_rows};
// 3-D view [groups][rows][inner], box {64, box_rows, 1}.  box_rows = 1 gives the gather map.
bool make_map_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t row_stride_elems,
                 uint32_t box_rows);
bool make_map_3d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t groups,
                 uint32_t box_rows);
// Epilogue stores: box {32 columns, 32 rows}; fp32 with 128-byte swizzle, bf16 with 64-byte swizzle.
// MN-major operand as chunks of 64 columns: 3-D view {64, rows, cols/64} of a [rows][cols] matrix and
// 4-D view {64, rows, cols/64, groups} of a [groups][rows][cols] tensor; box {64, 64, box_chunks(, 1)}.
bool make_chunked_map_2d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_chunks);
bool make_chunked_map_3d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t groups,
                         uint32_t box_chunks);
bool make_store_map_2d(CUtensorMap* m, void* ptr, bool fp32, uint64_t cols, uint64_t rows, uint64_t row_stride_elems);
bool make_store_map_3d(CUtensorMap* m, void* ptr, bool fp32, uint64_t cols, uint64_t rows, uint64_t depth);

// ---- grouped GEMM instantiations (BN chosen at run time: 128 or 256) -------------------------
// forward
cudaError_t run_gate_up_swiglu(int BN, int cn, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_gate_up_swiglu_e4m3(int BN, int cn, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_down_scale_e4m3(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_dx_store_e4m3(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_dact_dswiglu_e4m3(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t launch_quantize_rows_pair_e4m3(const __nv_bfloat16* M0, const __nv_bfloat16* M1, long long rows,
                                           const int32_t* rows_limit, int cols, uint8_t* q, float* scales,
                                           cudaStream_t s);
cudaError_t launch_transpose_into_bf16(const __nv_bfloat16* in, int E, int R, int C, __nv_bfloat16* out, int ld,
                                       int col0, cudaStream_t s);
cudaError_t launch_quantize_rows_e4m3(const __nv_bfloat16* M, long long rows, const int32_t* rows_limit, int cols,
                                      uint8_t* q, float* scales, cudaStream_t s);
cudaError_t run_down_scale(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
// block-scaled (1 x 32) e4m3 GEMMs: the tile width (the gate/up pair: kMxBN / 2 output columns of each), and for the
// plain ones the width for N output columns: 192, or 128 when 192-column tiles would compute more than a quarter
// of N in columns past N and 128-column tiles fewer (n = 256: 384 columns for 256)
constexpr int kMxBN = 192;
inline int mx_tile_cols(int N) {
  const int w192 = (N + kMxBN - 1) / kMxBN * kMxBN - N, w128 = (N + 127) / 128 * 128 - N;
  return (4 * w192 > N && w128 < w192) ? 128 : kMxBN;
}
cudaError_t run_gate_up_swiglu_mx(int cn, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_down_scale_mx(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_dact_dswiglu_mx(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_dx_store_mx(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t launch_quantize_rows_mx(const __nv_bfloat16* M, long long rows, const int32_t* rows_limit, int cols,
                                    uint8_t* q, uint8_t* sf, int sf_ld, cudaStream_t s);
// Scale blocks of a gathered operand per row tile of the varlen-M GEMMs over `off` (tiles in group order, at most
// tiles_cap of them) and stage of K, from row-major [src_rows][sf_ld] scales and the gather index idx[idx_rows].
cudaError_t launch_mx_tile_scales(const uint8_t* sf, int sf_ld, int src_rows, const int32_t* idx, int idx_rows,
                                  const int32_t* off, int G, int kst, long long tiles_cap, uint8_t* blocks,
                                  cudaStream_t s);
cudaError_t launch_quantize_weight_mx(const __nv_bfloat16* W, int E, int R, int C, uint8_t* q, uint8_t* blocks,
                                      int rpt, int roff, int ntile, int kst, int nblk, cudaStream_t s);
// Block-scaled operands of the weight gradients (blocks along tokens): kp = the padded stage offsets (pairs),
// then per job the source's columns as K-major code rows with their scale blocks.
struct MxColJob {
  const __nv_bfloat16* src;     // [src_rows][ld] bf16: rows at the sorted positions, or gathered through idx
  const __nv_bfloat16* src_lo;  // low part in the same layout (the value is src + src_lo), or null
  const int32_t* idx;           // sorted position -> source row (negative: no row), or null (the position)
  long long src_rows;
  long long ld;
  int C;            // columns of src (code rows written: row0 .. row0 + C - 1)
  int row0;
  uint8_t* q;       // codes [rows][kq]
  uint8_t* sf;      // scale blocks [rows / tw][kst] x ceil(tw / 128) 512-byte blocks
  int tw;           // operand rows per scale tile (the GEMM's row tile 128, or its column tile 128 / 192)
};
constexpr int kMxColJobs = 6;
struct MxColJobs {
  MxColJob job[kMxColJobs];
};
cudaError_t launch_mx_stage_offsets(const int32_t* off, int E, int32_t* kp, int* err, cudaStream_t s);
// pos_cap: the length of the pair arrays (sorted positions at or past it are an offsets error)
cudaError_t launch_quantize_cols_mx(const MxColJobs& jobs, int njobs, const int32_t* off, const int32_t* kp, int E,
                                    long long pos_cap, long long kq, int kst, int* err, cudaStream_t s);
cudaError_t run_dw_mx(int BN, bool f32, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_down_scale_dual(int BN, bool pair, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_router_logits(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
// backward
cudaError_t run_dact_dswiglu(int BN, bool pair, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_dx_store(int BN, bool pair, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_dw_gate_up(int BN, bool f32, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_dw_down(int BN, bool f32, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_dw_tiled(int BN, bool f32, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_dw_tiled_trans(int BN, bool f32, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
cudaError_t run_dw_dual(int BN, bool f32, bool trans, bool pair, const GemmParams& p, const Maps& m, int grid,
                        cudaStream_t s);
cudaError_t run_dense_mn_store(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);
// test exports
cudaError_t run_test_m(int gathered, int b_kmajor, bool pair, const GemmParams& p, const Maps& m, int grid,
                       cudaStream_t s);
cudaError_t run_test_m_dual(bool pair, const GemmParams& p, const Maps& m, int grid, cudaStream_t s);

// Expert-sorted copies of two [T, d] bf16 tensors (rows without a pair zeroed), and optionally of per-token
// e4m3 code rows c with their scales cs (rows without a pair: zero codes, scale 1).  With poff the two bf16
// copies are padded per group to multiples of 16 rows (cap_pad rows); the code rows are not.  out_a == nullptr:
// the code rows alone.
cudaError_t launch_gather_rows(const int32_t* offsets, const int32_t* poff, long long cap_pad, int E,
                               const int32_t* sorted_tok, const int32_t* tok_ptr,
                               const int32_t* tok_pairs, long long cap, int T, int d, const __nv_bfloat16* a,
                               const __nv_bfloat16* b, __nv_bfloat16* out_a, __nv_bfloat16* out_b,
                               const uint8_t* c, const float* cs, uint8_t* out_c, float* out_cs, int* err,
                               int num_sms, unsigned long long timeout_ns, cudaStream_t s);

// poff[g] = sum over the groups before g of their row counts rounded up to 16; poff[E] the total.
cudaError_t launch_pad_offsets(const int32_t* offsets, int E, int32_t* poff, int* err, cudaStream_t s);

// Zero rows [offsets[E], min(offsets[E] + 16, cap)) of up to six [cap, cols] bf16 buffers (past the last pair;
// null entries are skipped).
cudaError_t launch_zero_tail_rows(const int32_t* offsets, int E, long long cap, int cols,
                                  __nv_bfloat16* const (&bufs)[6], cudaStream_t s);

// ---- routing / permutation -----------------------------------------------------------------
// Top-K and combine weights; with part != nullptr the logits are first summed from `split` partials
// (plus bias) and written.
cudaError_t launch_topk_softmax(float* logits, const float* part, int split, const float* bias, int T, int E, int K,
                                int32_t* ids, float* w, float* scores, cudaStream_t s);

struct PermuteWs {
  int32_t* hist;       // [E * nb]
  int32_t* tokblk;     // [nb + 1]
  int* barrier;        // [1] grid-barrier counter of the one-launch grouping (right after tokblk)
  uint32_t* member;    // [T * ceil(E/32)] final pair bitmap (token rounding)
  int32_t* plain_off;  // [E + 1]
  int32_t* plain_cnt;  // [E]
  int32_t* plain_tok;  // [T * K]
  float* scoresT;      // [E * T] scores transposed (token rounding)
};
// Tokens per grouping block: the smallest of 32, 64, 128, 256 whose [E x blocks] histogram and block
// bases stay within 65536 counts ((E + 1) x blocks), else 256.  Small token counts get more, smaller
// blocks; for T <= 32768 and E <= 512 everything fits the fixed scratch of moe_permute_noalloc.
inline int perm_tok_block(int T, int E) {
  for (int tb = 32; tb < 256; tb *= 2)
    if (static_cast<long long>(E + 1) * ((T + tb - 1) / tb) <= 65536) return tb;
  return 256;
}
size_t permute_ws_bytes(int T, int E, int K, int m_tile);
PermuteWs carve_permute_ws(void* ws, int T, int E, int K, int m_tile);

cudaError_t launch_permute(const int32_t* topk_ids, const float* topk_w, const float* logits, const float* scores,
                           int T, int E, int K, int m_tile, long long cap, int32_t* counts, int32_t* offsets,
                           int32_t* sorted_tok, float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs,
                           int32_t* P_out, const PermuteWs& w, int* err, unsigned long long timeout_ns,
                           cudaStream_t s);

// Capacity (drop/pad) dispatch: the kept pairs of expert e in slots [e C, (e + 1) C), offsets e C.
// Uses the token-rounding workspace layout (m_tile > 0).
cudaError_t launch_permute_capacity(const int32_t* topk_ids, const float* topk_w, int T, int E, int K, int C,
                                    int policy, long long cap, int32_t* counts, int32_t* offsets, int32_t* sorted_tok,
                                    float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs, int32_t* P_out,
                                    const PermuteWs& w, int* err, unsigned long long timeout_ns, cudaStream_t s);

// ---- combine / reductions --------------------------------------------------------------------
cudaError_t launch_combine(const __nv_bfloat16* Y, const int32_t* tok_ptr, const int32_t* tok_pairs, int T, int d,
                           long long cap, __nv_bfloat16* O, int* err, cudaStream_t s);

cudaError_t launch_transpose_bf16(const __nv_bfloat16* in, int rows, int cols, __nv_bfloat16* out, cudaStream_t s);

// Per token: dS of its pairs (sum of the per-column-tile partials), the router-logit gradient
// (fp32, and as bf16 high and low parts dL_bf16[T][E], dL_lo[T][E]), and dX = sum of the pairs' dX
// rows + dlogits W_r^T.
cudaError_t launch_token_backward(const float* part, int part_ld, const int32_t* tok_ptr, const int32_t* tok_pairs,
                                  const int32_t* offsets, int E, const float* sorted_w, const int32_t* topk_ids,
                                  const float* topk_w, int K, const __nv_bfloat16* dXp, const __nv_bfloat16* WrT,
                                  int T, int d, long long cap, float* dS, float* dlogits, __nv_bfloat16* dL_bf16,
                                  __nv_bfloat16* dL_lo, __nv_bfloat16* dX, int* err, cudaStream_t s);

cudaError_t launch_splitk_reduce(const float* part, int splits, long long n, float* out, cudaStream_t s);

cudaError_t launch_wait_timeout_probe(int* err, unsigned long long timeout_ns, cudaStream_t s);

}  // namespace vgg

struct moe_ctx;
namespace vgg {
// Context fields needed outside api.cu.
int ctx_device(const moe_ctx* ctx);
int* ctx_error_word(moe_ctx* ctx);

// moe_permute's plain grouping (m_tile = 0) with the scratch taken from `scratch` (scratch_ints ints) rather
// than a workspace; returns a moe_status (the checks and the launch of moe_permute, MOE_ERR_UNSUPPORTED when
// the scratch is too small for T and E).
int permute_plain_with_scratch(moe_ctx* ctx, const int32_t* topk_ids, const float* topk_w, int T, int E, int K,
                               long long cap, int32_t* counts, int32_t* offsets, int32_t* sorted_tok, float* sorted_w,
                               int32_t* tok_ptr, int32_t* tok_pairs, int32_t* P_out, int32_t* scratch,
                               long long scratch_ints, cudaStream_t s);

}  // namespace vgg

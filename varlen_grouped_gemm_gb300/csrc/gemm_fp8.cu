// Gate/up + SwiGLU grouped GEMM with e4m3 operands: the gathered token rows of X and the W_gate /
// W_up pair are e4m3 codes of per-row-scaled rows, accumulated in fp32 by the kind::f8f6f4 UMMA; the
// epilogue multiplies by the token's and the output channel's scale before SwiGLU.
// [GG] "한계": the fine-grained FP8 grouped GEMM named there as the next 2x after bf16.
#include <cuda_fp8.h>

#include "internal.h"

namespace vgg {

cudaError_t run_gate_up_swiglu_e4m3(int BN, int cn, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256) {
    if (cn == 2)
      return launch_grouped_gemm<256, 4, 4, 1, A_GATHER_K, B_TMA_K3_GU, VAR_M, EPI_SWIGLU_Q, false, 2>(p, m, grid, s);
    return launch_grouped_gemm<256, 4, 4, 1, A_GATHER_K, B_TMA_K3_GU, VAR_M, EPI_SWIGLU_Q, false>(p, m, grid, s);
  }
  return launch_grouped_gemm<128, 6, 4, 1, A_GATHER_K, B_TMA_K3_GU, VAR_M, EPI_SWIGLU_Q, false>(p, m, grid, s);
}

// Down projection with e4m3 operands (A rows and W_down rows quantized per row); the epilogue multiplies
// by the A row's scale, the output channel's scale and the combine weight.
cudaError_t run_down_scale_e4m3(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  // 8 epilogue warps: with half as many stages per tile as the bf16 form the epilogue sets the pace
  // (4 warps: 91 us at c2, 8: 67 us); three stages when the group table leaves no room for four
  if (BN == 256 && SmemLayout<256, 4, 8, 1>::bytes(p.groups, VAR_M) <= kMaxSmem)
    return launch_grouped_gemm<256, 4, 8, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_SCALE_Q, false>(p, m, grid, s);
  if (BN == 256) return launch_grouped_gemm<256, 3, 8, 2, A_TMA_K, B_TMA_K3, VAR_M, EPI_SCALE_Q, false>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_SCALE_Q, false>(p, m, grid, s);
}

// The backward's dX GEMM with e4m3 operands: A = each pair's [dH | dU] row, B = [W_gate; W_up]^T (d rows
// of 2n), both quantized per row; the epilogue multiplies by the two scales and stores dXp in bf16.
cudaError_t run_dx_store_e4m3(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256 && SmemLayout<256, 4, 8, 1>::bytes(p.groups, VAR_M) <= kMaxSmem)
    return launch_grouped_gemm<256, 4, 8, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE_Q, false>(p, m, grid, s);
  if (BN == 256) return launch_grouped_gemm<256, 3, 8, 2, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE_Q, false>(p, m, grid, s);
  return launch_grouped_gemm<128, 6, 8, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE_Q, false>(p, m, grid, s);
}

// out[e][c][col0 + r] = in[e][r][c] for in [E][R][C] bf16 and out rows of ld elements (32 x 32 tiles
// through shared memory): [W_gate; W_up]^T per expert for the e4m3 dX GEMM.
__global__ void transpose_into_bf16_kernel(const __nv_bfloat16* __restrict__ in, int R, int C,
                                           __nv_bfloat16* __restrict__ out, int ld, int col0) {
  __shared__ __nv_bfloat16 tile[32][33];
  const long long e = blockIdx.z;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const __nv_bfloat16* src = in + e * R * C;
  __nv_bfloat16* dst = out + e * static_cast<long long>(C) * ld;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < R && c < C) tile[i][threadIdx.x] = src[static_cast<long long>(r) * C + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < R && c < C) dst[static_cast<long long>(c) * ld + col0 + r] = tile[threadIdx.x][i];
  }
}

cudaError_t launch_transpose_into_bf16(const __nv_bfloat16* in, int E, int R, int C, __nv_bfloat16* out, int ld,
                                       int col0, cudaStream_t s) {
  if (E <= 0 || R <= 0 || C <= 0) return cudaSuccess;
  transpose_into_bf16_kernel<<<dim3((C + 31) / 32, (R + 31) / 32, E), dim3(32, 8), 0, s>>>(in, R, C, out, ld, col0);
  return cudaGetLastError();
}

// Per-row e4m3 quantization: s = max|row| / 448 (1 for a zero row), codes = e4m3(x / s), the division
// in fp32 and the conversion rounding to nearest even and saturating at +-448.  One warp per row, 8
// elements (16 bytes) per lane and step.  Rows of up to 32 x 8 x VR columns stay in registers between the
// two passes; longer rows (VR = 0) are read twice (the second time from L1/L2).
__device__ __forceinline__ uint2 e4m3x8(const uint4 x, float s) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
  uint32_t w[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float2 a = __bfloat1622float2(h[2 * j]);
    const float2 b = __bfloat1622float2(h[2 * j + 1]);
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(a.x, s), __fdiv_rn(a.y, s)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(b.x, s), __fdiv_rn(b.y, s)), __NV_SATFINITE, __NV_E4M3);
    w[j] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint2(w[0], w[1]);
}

__device__ __forceinline__ float amax8(const uint4 x, float m) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = __bfloat1622float2(h[j]);
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return m;
}

template <int VR>
__global__ void __launch_bounds__(256) quantize_rows_e4m3_kernel(const __nv_bfloat16* __restrict__ M, long long rows,
                                                                 const int32_t* __restrict__ rows_limit, int cols,
                                                                 uint8_t* __restrict__ q,
                                                                 float* __restrict__ scales) {
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows || (rows_limit && r >= __ldg(rows_limit))) return;
  const uint4* src = reinterpret_cast<const uint4*>(M + r * cols);
  uint2* dst = reinterpret_cast<uint2*>(q + r * cols);
  const int vecs = cols / 8;
  float amax = 0.0f;
  uint4 x[VR > 0 ? VR : 1];
  if (VR > 0) {
#pragma unroll
    for (int i = 0; i < VR; ++i) {
      const int v = lane + 32 * i;
      x[i] = v < vecs ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < VR; ++i) amax = amax8(x[i], amax);
  } else {
    for (int v = lane; v < vecs; v += 32) amax = amax8(__ldg(src + v), amax);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (lane == 0) scales[r] = s;
  if (VR > 0) {
#pragma unroll
    for (int i = 0; i < VR; ++i) {
      const int v = lane + 32 * i;
      if (v < vecs) dst[v] = e4m3x8(x[i], s);
    }
  } else {
    for (int v = lane; v < vecs; v += 32) dst[v] = e4m3x8(__ldg(src + v), s);
  }
}

// rows_limit (device, optional): only rows below *rows_limit are quantized.
cudaError_t launch_quantize_rows_e4m3(const __nv_bfloat16* M, long long rows, const int32_t* rows_limit, int cols,
                                      uint8_t* q, float* scales, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;
  const unsigned g = static_cast<unsigned>(blocks);
  if (cols <= 256) quantize_rows_e4m3_kernel<1><<<g, 256, 0, s>>>(M, rows, rows_limit, cols, q, scales);
  else if (cols <= 512) quantize_rows_e4m3_kernel<2><<<g, 256, 0, s>>>(M, rows, rows_limit, cols, q, scales);
  else if (cols <= 1024) quantize_rows_e4m3_kernel<4><<<g, 256, 0, s>>>(M, rows, rows_limit, cols, q, scales);
  else if (cols <= 2048) quantize_rows_e4m3_kernel<8><<<g, 256, 0, s>>>(M, rows, rows_limit, cols, q, scales);
  else quantize_rows_e4m3_kernel<0><<<g, 256, 0, s>>>(M, rows, rows_limit, cols, q, scales);
  return cudaGetLastError();
}

// The backward's dSwiGLU GEMM with e4m3 operands: A = dO's rows (sorted), B = W_down^T (n rows of d), both
// quantized per row; the epilogue applies both scales to dA' and runs the dSwiGLU epilogue.
cudaError_t run_dact_dswiglu_e4m3(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 256 && SmemLayout<256, 4, 8, 1>::bytes(p.groups, VAR_M) <= kMaxSmem)
    return launch_grouped_gemm<256, 4, 8, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_DSWIGLU_Q, false>(p, m, grid, s);
  if (BN == 256) return launch_grouped_gemm<256, 3, 8, 2, A_TMA_K, B_TMA_K3, VAR_M, EPI_DSWIGLU_Q, false>(p, m, grid, s);
  return launch_grouped_gemm<128, 4, 8, 2, A_TMA_K, B_TMA_K3, VAR_M, EPI_DSWIGLU_Q, false>(p, m, grid, s);
}

// Per-row e4m3 quantization of the rows [M0[r] | M1[r]] (two bf16 matrices of `cols` columns each, side by
// side), the rows below *rows_limit: one scale per row over both halves, codes [rows, 2 cols].  One warp
// per row; the row is read twice (the second time from L1/L2).
__global__ void __launch_bounds__(256) quantize_rows_pair_e4m3_kernel(const __nv_bfloat16* __restrict__ M0,
                                                                      const __nv_bfloat16* __restrict__ M1,
                                                                      long long rows,
                                                                      const int32_t* __restrict__ rows_limit,
                                                                      int cols, uint8_t* __restrict__ q,
                                                                      float* __restrict__ scales) {
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows || (rows_limit && r >= __ldg(rows_limit))) return;
  const int vh = cols / 8;  // 16-byte vectors per half
  const uint4* s0 = reinterpret_cast<const uint4*>(M0 + r * cols);
  const uint4* s1 = reinterpret_cast<const uint4*>(M1 + r * cols);
  uint2* dst = reinterpret_cast<uint2*>(q + r * 2 * cols);
  float amax = 0.0f;
  for (int v = lane; v < 2 * vh; v += 32) amax = amax8(__ldg(v < vh ? s0 + v : s1 + (v - vh)), amax);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (lane == 0) scales[r] = sc;
  for (int v = lane; v < 2 * vh; v += 32) dst[v] = e4m3x8(__ldg(v < vh ? s0 + v : s1 + (v - vh)), sc);
}

cudaError_t launch_quantize_rows_pair_e4m3(const __nv_bfloat16* M0, const __nv_bfloat16* M1, long long rows,
                                           const int32_t* rows_limit, int cols, uint8_t* q, float* scales,
                                           cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  quantize_rows_pair_e4m3_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(M0, M1, rows, rows_limit, cols,
                                                                                     q, scales);
  return cudaGetLastError();
}

}  // namespace vgg

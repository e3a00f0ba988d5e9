// Top-K token choice and combine weights from the router logits.
//
// [DEP] "1) Router": each token's top-k experts (index and score, [BN, k]).
// [EP] "여러 Expert의 결과도 같은 토큰으로 돌아오기": the combine weights are the
// softmax renormalised over the chosen experts, kept apart from the selection.
//
// One warp per token.  Lane l holds experts l, l+32, ... in registers; each of
// the K rounds is a warp arg-max with the order (value descending, expert
// ascending), so equal logits go to the lower expert.  The full softmax over E
// (needed by token rounding) is written only when asked for.
#include <cfloat>
#include <climits>

#include "internal.h"

namespace vgg {

template <int VPL>
__global__ void __launch_bounds__(256) topk_softmax_kernel(const float* __restrict__ logits, int T, int E, int K,
                                                           int32_t* __restrict__ ids, float* __restrict__ w,
                                                           float* __restrict__ scores) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = logits + static_cast<long long>(t) * E;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(row + e) : -FLT_MAX;
  }
  uint32_t taken = 0;
  float vmax = 0.0f, my_ex = 0.0f, sum = 0.0f;
  int my_id = 0;
  for (int k = 0; k < K; ++k) {
    float bv = -FLT_MAX;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (k == 0) vmax = bv;
    const float ex = expf(bv - vmax);
    sum += ex;  // same order in every lane: k ascending
    if (lane == k) {
      my_id = be;
      my_ex = ex;
    }
  }
  if (lane < K) {
    ids[static_cast<long long>(t) * K + lane] = my_id;
    w[static_cast<long long>(t) * K + lane] = my_ex / sum;
  }
  if (scores) {
    // full softmax for token rounding's priorities: the fast exponential and one reciprocal (the
    // selection compares these values among themselves; relative error ~1e-6)
    float z = 0.0f;
    float ex[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      ex[i] = (e < E) ? __expf(v[i] - vmax) : 0.0f;
      z += ex[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float inv = 1.0f / z;
    float* srow = scores + static_cast<long long>(t) * E;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) srow[e] = ex[i] * inv;
    }
  }
}

cudaError_t launch_topk_softmax(const float* logits, int T, int E, int K, int32_t* ids, float* w, float* scores,
                                cudaStream_t s) {
  const int blocks = (T + 7) / 8;
  if (E <= 32) topk_softmax_kernel<1><<<blocks, 256, 0, s>>>(logits, T, E, K, ids, w, scores);
  else if (E <= 64) topk_softmax_kernel<2><<<blocks, 256, 0, s>>>(logits, T, E, K, ids, w, scores);
  else if (E <= 128) topk_softmax_kernel<4><<<blocks, 256, 0, s>>>(logits, T, E, K, ids, w, scores);
  else if (E <= 256) topk_softmax_kernel<8><<<blocks, 256, 0, s>>>(logits, T, E, K, ids, w, scores);
  else if (E <= 512) topk_softmax_kernel<16><<<blocks, 256, 0, s>>>(logits, T, E, K, ids, w, scores);
  else topk_softmax_kernel<32><<<blocks, 256, 0, s>>>(logits, T, E, K, ids, w, scores);
  return cudaGetLastError();
}

}  // namespace vgg

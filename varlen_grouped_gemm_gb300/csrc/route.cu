// Top-K token choice and combine weights from the router logits.
//
// [DEP] "1) Router": each token's top-k experts (index and score, [BN, k]).
// [EP] "여러 Expert의 결과도 같은 토큰으로 돌아오기": the combine weights are the
// softmax renormalised over the chosen experts, kept apart from the selection.
//
// One warp per token.  Lane l holds experts l, l+32, ... in registers as order-preserving unsigned keys
// of the logits (-0 folded into +0 first, so that equal logits have equal keys); each of the K rounds is
// a warp arg-max with the order (key descending, expert ascending), so equal logits go to the lower
// expert.  Within a lane the slots are in ascending expert order, so a strict comparison keeps the
// lowest expert among equal keys; a taken slot (and a slot past E) holds key 0, below every logit.
// The full softmax over E (needed by token rounding) is written only when asked for.
#include <cfloat>
#include <climits>

#include "internal.h"

namespace vgg {

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t b = __float_as_uint(x + 0.0f);  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// With split > 1 the router GEMM left `split` partial sums of the logits in part[split][T][E]: they are
// added in split order with the bias and the result is written to logits first.
template <int VPL>
__global__ void __launch_bounds__(256) topk_softmax_kernel(float* __restrict__ logits, const float* __restrict__ part,
                                                           int split, const float* __restrict__ bias, int T, int E,
                                                           int K, int32_t* __restrict__ ids, float* __restrict__ w,
                                                           float* __restrict__ scores) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float* row = logits + static_cast<long long>(t) * E;
  float v[VPL];
  if (part) {
    const long long plane = static_cast<long long>(T) * E;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        float a = __ldg(part + static_cast<long long>(t) * E + e);
        for (int sp = 1; sp < split; ++sp) a += __ldg(part + sp * plane + static_cast<long long>(t) * E + e);
        if (bias) a += __ldg(bias + e);
        v[i] = a;
        row[e] = a;
      } else {
        v[i] = -FLT_MAX;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? __ldg(row + e) : -FLT_MAX;
    }
  }
  uint32_t key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) key[i] = (lane + 32 * i < E) ? order_key(v[i]) : 0u;
  float vmax = 0.0f, my_ex = 0.0f, sum = 0.0f;
  int my_id = 0;
  for (int k = 0; k < K; ++k) {
    uint32_t bk = 0u;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const bool better = key[i] > bk;
      bk = better ? key[i] : bk;
      bi = better ? i : bi;
    }
    int be = bk ? lane + 32 * bi : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint32_t ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ok > bk || (ok == bk && oe < be)) {
        bk = ok;
        be = oe;
      }
    }
    if ((be & 31) == lane) {
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (i == (be >> 5)) key[i] = 0u;
    }
    const float bv = key_value(bk);
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

cudaError_t launch_topk_softmax(float* logits, const float* part, int split, const float* bias, int T, int E, int K,
                                int32_t* ids, float* w, float* scores, cudaStream_t s) {
  const int blocks = (T + 7) / 8;
#define VGG_TOPK(V) topk_softmax_kernel<V><<<blocks, 256, 0, s>>>(logits, part, split, bias, T, E, K, ids, w, scores)
  if (E <= 32) VGG_TOPK(1);
  else if (E <= 64) VGG_TOPK(2);
  else if (E <= 128) VGG_TOPK(4);
  else if (E <= 256) VGG_TOPK(8);
  else if (E <= 512) VGG_TOPK(16);
  else VGG_TOPK(32);
#undef VGG_TOPK
  return cudaGetLastError();
}

}  // namespace vgg

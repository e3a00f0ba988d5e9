// Grouping of the (token, expert) pairs by expert, and token rounding.
//
// [GG] "(1)-(3) 토큰 정렬": topk_ids flattened and sorted by expert so that each
// expert's tokens form one contiguous slice; bincount gives the counts.
// [DEP] table "Ragged vs Padding": the ragged layout carries offsets/indices.
// [EP] "토큰을 Expert로 보내고 원래 위치로 돌려받기": each result is tracked back
// to its token (here: tok_ptr / tok_pairs, per token in ascending expert).
//
// The stable order is a counting sort keyed by expert.  Tokens are cut into
// blocks of 256; inside a block every expert gets a 256-bit bitmap of the
// tokens that chose it (8 words in shared memory).  The rank of token t among
// the earlier tokens of its block that chose e is a popcount over that bitmap,
// so no atomics decide any position and the result is the same on every run:
//   1. hist:    per (expert, block) counts            -> hist[e][b]
//   2. scan:    one exclusive scan over hist in expert-major order gives the
//               first sorted position of every (e, b) block, the offsets and
//               the per-token pair base of every block
//   3. scatter: sorted position = base[e][b] + in-block rank.
// Token rounding ([SM] "5 기여 ③ Token Rounding 라우팅") runs the plain grouping
// first, then per expert selects the final token set (tr_select_kernel) into a
// [T x E] membership bitmap, and groups again from that bitmap.
#include <climits>

#include "internal.h"

namespace vgg {

constexpr int kTokBlock = 256;

__device__ __forceinline__ int block_exclusive_scan_256(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (blockDim.x >> 5)) ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    s_warp[lane] = wi - w;
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  const int res = s_warp[warp] + incl - v;
  total = s_warp[32];
  __syncthreads();
  return res;
}

// Collect the experts of token t (ascending) into e_out / w_out; returns the count.
// From top-K ids (plain) or from the membership bitmap (token rounding).
template <bool FROM_MEMBER>
__device__ __forceinline__ int token_experts(int t, const int32_t* ids, const float* topk_w, const uint32_t* member,
                                             const float* logits, int E, int K, int* e_out, float* w_out,
                                             int max_out, int* err) {
  int cnt = 0;
  if (!FROM_MEMBER) {
    for (int k = 0; k < K; ++k) {
      const int e = ids[static_cast<long long>(t) * K + k];
      const float w = topk_w ? topk_w[static_cast<long long>(t) * K + k] : 0.0f;
      if (e < 0 || e >= E) {
        set_error(err, DERR_BAD_EXPERT);
        continue;
      }
      bool dup = false;
      for (int q = 0; q < cnt; ++q) dup |= (e_out[q] == e);
      if (dup) {
        set_error(err, DERR_DUP_EXPERT);
        continue;
      }
      // insertion into ascending order
      int q = cnt;
      while (q > 0 && e_out[q - 1] > e) {
        e_out[q] = e_out[q - 1];
        w_out[q] = w_out[q - 1];
        --q;
      }
      e_out[q] = e;
      w_out[q] = w;
      ++cnt;
    }
  } else {
    const int W = (E + 31) >> 5;
    // weights of the token's own top-K and the denominator of a padded pair's weight
    float lmax = 0.0f, denom = 0.0f;
    if (logits) {
      lmax = logits[static_cast<long long>(t) * E + ids[static_cast<long long>(t) * K]];
      for (int k = 0; k < K; ++k) denom += expf(logits[static_cast<long long>(t) * E + ids[static_cast<long long>(t) * K + k]] - lmax);
    }
    for (int wi = 0; wi < W; ++wi) {
      uint32_t word = member[static_cast<long long>(t) * W + wi];
      while (word) {
        const int bit = __ffs(word) - 1;
        word &= word - 1;
        const int e = wi * 32 + bit;
        float w = -1.0f;
        for (int k = 0; k < K; ++k)
          if (ids[static_cast<long long>(t) * K + k] == e) w = topk_w[static_cast<long long>(t) * K + k];
        if (w < 0.0f) w = logits ? expf(logits[static_cast<long long>(t) * E + e] - lmax) / denom : 0.0f;
        if (cnt < max_out) {
          e_out[cnt] = e;
          w_out[cnt] = w;
        }
        ++cnt;
      }
    }
  }
  return cnt;
}

template <bool FROM_MEMBER>
__global__ void __launch_bounds__(kTokBlock) perm_hist_kernel(const int32_t* __restrict__ ids,
                                                             const uint32_t* __restrict__ member, int T, int E,
                                                             int K, int nb, int32_t* __restrict__ hist,
                                                             int32_t* __restrict__ tokblk, int* err) {
  extern __shared__ uint32_t bits[];  // [E][8]
  __shared__ int s_warp[33];
  const int b = blockIdx.x, tid = threadIdx.x;
  for (int i = tid; i < E * 8; i += kTokBlock) bits[i] = 0;
  __syncthreads();
  const int t = b * kTokBlock + tid;
  int cnt = 0;
  if (t < T) {
    if (!FROM_MEMBER) {
      int es[8];
      float ws[8];
      cnt = token_experts<false>(t, ids, nullptr, nullptr, nullptr, E, K, es, ws, 8, err);
      for (int q = 0; q < cnt; ++q) atomicOr(&bits[es[q] * 8 + (tid >> 5)], 1u << (tid & 31));
    } else {
      const int W = (E + 31) >> 5;
      for (int wi = 0; wi < W; ++wi) {
        uint32_t word = member[static_cast<long long>(t) * W + wi];
        while (word) {
          const int bit = __ffs(word) - 1;
          word &= word - 1;
          atomicOr(&bits[(wi * 32 + bit) * 8 + (tid >> 5)], 1u << (tid & 31));
          ++cnt;
        }
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kTokBlock) {
    int s = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += __popc(bits[e * 8 + w]);
    hist[static_cast<long long>(e) * nb + b] = s;
  }
  int total;
  block_exclusive_scan_256(cnt, s_warp, total);
  if (tid == 0) tokblk[b] = total;
}

// One block of 1024 threads: exclusive scan of hist (expert-major) in place,
// offsets/counts, and the exclusive scan of the per-block token pair counts.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ hist, int E, int nb,
                                                         int32_t* __restrict__ tokblk, int32_t* __restrict__ counts,
                                                         int32_t* __restrict__ offsets, int32_t* __restrict__ P_out,
                                                         long long cap, int* err) {
  __shared__ int s_warp[33];
  __shared__ int s_tok[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long N = static_cast<long long>(E) * nb;
  const long long chunk = (N + 1023) / 1024;
  const long long lo = tid * chunk, hi = min(N, lo + chunk);
  int local = 0;
  for (long long i = lo; i < hi; ++i) local += hist[i];
  // block exclusive scan of `local`
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = s_warp[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    s_warp[lane] = wi - w;
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  int run = s_warp[warp] + incl - local;
  for (long long i = lo; i < hi; ++i) {
    const int v = hist[i];
    hist[i] = run;
    run += v;
  }
  const int total = s_warp[32];
  // per-block token pair bases (nb <= 256 -> a few warps)
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < nb; base += 32) {
      const int i = base + lane;
      const int v = (i < nb) ? tokblk[i] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (i < nb) tokblk[i] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) {
      tokblk[nb] = carry;
      s_tok[0] = carry;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += 1024) offsets[e] = hist[static_cast<long long>(e) * nb];
  if (tid == 0) {
    offsets[E] = total;
    if (P_out) *P_out = total;
    if (total > cap || s_tok[0] != total) set_error(err, DERR_CAPACITY);
  }
  __syncthreads();
  if (counts)
    for (int e = tid; e < E; e += 1024) counts[e] = (e + 1 < E ? hist[static_cast<long long>(e + 1) * nb] : total) - hist[static_cast<long long>(e) * nb];
}

template <bool FROM_MEMBER>
__global__ void __launch_bounds__(kTokBlock) perm_scatter_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ topk_w, const uint32_t* __restrict__ member,
    const float* __restrict__ logits, int T, int E, int K, int nb, const int32_t* __restrict__ base,
    const int32_t* __restrict__ tokbase, long long cap, int32_t* __restrict__ sorted_tok,
    float* __restrict__ sorted_w, int32_t* __restrict__ tok_ptr, int32_t* __restrict__ tok_pairs, int* err) {
  extern __shared__ uint32_t bits[];  // [E][8]
  __shared__ int s_warp[33];
  // pairs per token: K without rounding; rounding may pad a token into more experts
  constexpr int kMaxPairs = FROM_MEMBER ? 32 : 8;
  const int b = blockIdx.x, tid = threadIdx.x;
  for (int i = tid; i < E * 8; i += kTokBlock) bits[i] = 0;
  __syncthreads();
  const int t = b * kTokBlock + tid;
  int es[kMaxPairs];
  float ws[kMaxPairs];
  int cnt = 0;
  if (t < T) {
    cnt = token_experts<FROM_MEMBER>(t, ids, topk_w, member, logits, E, K, es, ws, kMaxPairs, err);
    if (cnt > kMaxPairs) {
      set_error(err, DERR_CAPACITY);
      cnt = kMaxPairs;
    }
    for (int q = 0; q < cnt; ++q) atomicOr(&bits[es[q] * 8 + (tid >> 5)], 1u << (tid & 31));
  }
  __syncthreads();
  int total;
  const int tprefix = block_exclusive_scan_256(cnt, s_warp, total);
  const long long tp = static_cast<long long>(tokbase[b]) + tprefix;
  if (t < T && tok_ptr) tok_ptr[t] = static_cast<int32_t>(tp);
  if (t == T - 1 && tok_ptr) tok_ptr[T] = static_cast<int32_t>(tp + cnt);
  const int w_self = tid >> 5;
  const uint32_t lt_mask = (1u << (tid & 31)) - 1u;
  for (int q = 0; q < cnt; ++q) {
    const int e = es[q];
    int rank = __popc(bits[e * 8 + w_self] & lt_mask);
    for (int w = 0; w < w_self; ++w) rank += __popc(bits[e * 8 + w]);
    const long long j = static_cast<long long>(base[static_cast<long long>(e) * nb + b]) + rank;
    if (j >= cap || tp + q >= cap) {
      set_error(err, DERR_CAPACITY);
      continue;
    }
    sorted_tok[j] = t;
    if (sorted_w) sorted_w[j] = ws[q];
    if (tok_pairs) tok_pairs[tp + q] = static_cast<int32_t>(j);
  }
}

// Token rounding, one CTA per expert: choose the final token set of expert e
// and mark it in the membership bitmap.  Priority of a token for e is
// (score descending, token ascending); the selection is a radix select of the
// need-th largest score among the candidates, ties at the threshold resolved
// by ascending token.  Keys (score bits) are staged in shared memory.
constexpr int kTrThreads = 1024;
constexpr int kTrMaxT = 32768;

__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = s_warp[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    s_warp[lane] = wi - w;
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  const int res = s_warp[warp] + incl - v;
  total = s_warp[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kTrThreads) tr_select_kernel(const float* __restrict__ scores, int T, int E,
                                                              int m_tile, const int32_t* __restrict__ plain_off,
                                                              const int32_t* __restrict__ plain_tok,
                                                              long long plain_cap, uint32_t* __restrict__ member,
                                                              int* err) {
  extern __shared__ uint32_t tr_smem[];
  uint32_t* keys = tr_smem;               // [T]; 0xFFFFFFFF = not a candidate
  uint32_t* routed = tr_smem + T;         // [ceil(T/32)]
  __shared__ int hist[256];
  __shared__ int s_warp[33];
  __shared__ int s_digit, s_remaining;
  const int e = blockIdx.x, tid = threadIdx.x;
  const int W = (E + 31) >> 5;
  const int TW = (T + 31) >> 5;
  const int off = plain_off[e];
  const int c = plain_off[e + 1] - off;
  if (off < 0 || c < 0 || off + c > plain_cap || c > T) {
    if (tid == 0) set_error(err, DERR_BAD_OFFSETS);
    return;
  }
  int r = m_tile * ((c + m_tile / 2) / m_tile);
  r = min(r, m_tile * (T / m_tile));
  for (int i = tid; i < TW; i += kTrThreads) routed[i] = 0;
  __syncthreads();
  for (int i = tid; i < c; i += kTrThreads) {
    const int t = plain_tok[off + i];
    if (t >= 0 && t < T) atomicOr(&routed[t >> 5], 1u << (t & 31));
  }
  __syncthreads();
  const uint32_t ebit = 1u << (e & 31);
  const int ew = e >> 5;
  const bool drop = r < c;
  if (!drop) {  // every routed token stays
    for (int i = tid; i < c; i += kTrThreads) {
      const int t = plain_tok[off + i];
      if (t >= 0 && t < T) atomicOr(&member[static_cast<long long>(t) * W + ew], ebit);
    }
  }
  const int need = drop ? r : r - c;
  if (need == 0) return;
  for (int t = tid; t < T; t += kTrThreads) {
    const bool is_routed = (routed[t >> 5] >> (t & 31)) & 1u;
    const bool cand = drop ? is_routed : !is_routed;
    keys[t] = cand ? __float_as_uint(scores[static_cast<long long>(t) * E + e]) : 0xFFFFFFFFu;
  }
  __syncthreads();
  uint32_t prefix = 0, mask = 0;
  int remaining = need;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kTrThreads) hist[i] = 0;
    __syncthreads();
    for (int t = tid; t < T; t += kTrThreads) {
      const uint32_t k = keys[t];
      if (k != 0xFFFFFFFFu && (k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int cum = 0, digit = 0;
      for (int dgt = 255; dgt >= 0; --dgt) {
        if (cum + hist[dgt] >= remaining) {
          digit = dgt;
          break;
        }
        cum += hist[dgt];
      }
      s_digit = digit;
      s_remaining = remaining - cum;
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(s_digit) << shift;
    mask |= 255u << shift;
    remaining = s_remaining;
    __syncthreads();
  }
  // keys above the threshold are all taken; at the threshold the `remaining` lowest tokens.
  const int per = (T + kTrThreads - 1) / kTrThreads;
  const int t0 = tid * per, t1 = min(T, t0 + per);
  int ties = 0;
  for (int t = t0; t < t1; ++t) ties += (keys[t] == prefix);
  int tot;
  int before = block_exclusive_scan_1024(ties, s_warp, tot);
  for (int t = t0; t < t1; ++t) {
    const uint32_t k = keys[t];
    if (k == 0xFFFFFFFFu) continue;
    bool take = k > prefix;
    if (k == prefix) take = (before++ < remaining);
    if (take) atomicOr(&member[static_cast<long long>(t) * W + ew], ebit);
  }
}

size_t permute_ws_bytes(int T, int E, int K, int m_tile) {
  const long long nb = (T + kTokBlock - 1) / kTokBlock;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t b = al(sizeof(int32_t) * E * nb) + al(sizeof(int32_t) * (nb + 1));
  if (m_tile > 0) {
    b += al(sizeof(uint32_t) * static_cast<size_t>(T) * ((E + 31) / 32));
    b += al(sizeof(int32_t) * (E + 1)) + al(sizeof(int32_t) * E) + al(sizeof(int32_t) * static_cast<size_t>(T) * K);
  }
  return b;
}

PermuteWs carve_permute_ws(void* ws, int T, int E, int K, int m_tile) {
  const long long nb = (T + kTokBlock - 1) / kTokBlock;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint8_t* p = static_cast<uint8_t*>(ws);
  PermuteWs w{};
  w.hist = reinterpret_cast<int32_t*>(p);
  p += al(sizeof(int32_t) * E * nb);
  w.tokblk = reinterpret_cast<int32_t*>(p);
  p += al(sizeof(int32_t) * (nb + 1));
  if (m_tile > 0) {
    w.member = reinterpret_cast<uint32_t*>(p);
    p += al(sizeof(uint32_t) * static_cast<size_t>(T) * ((E + 31) / 32));
    w.plain_off = reinterpret_cast<int32_t*>(p);
    p += al(sizeof(int32_t) * (E + 1));
    w.plain_cnt = reinterpret_cast<int32_t*>(p);
    p += al(sizeof(int32_t) * E);
    w.plain_tok = reinterpret_cast<int32_t*>(p);
  }
  return w;
}

cudaError_t launch_permute(const int32_t* topk_ids, const float* topk_w, const float* logits, const float* scores,
                           int T, int E, int K, int m_tile, long long cap, int32_t* counts, int32_t* offsets,
                           int32_t* sorted_tok, float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs,
                           int32_t* P_out, const PermuteWs& w, int* err, cudaStream_t s) {
  const int nb = (T + kTokBlock - 1) / kTokBlock;
  const size_t bits_smem = static_cast<size_t>(E) * 8 * sizeof(uint32_t);
  cudaError_t st;
  if (m_tile <= 0) {
    perm_hist_kernel<false><<<nb, kTokBlock, bits_smem, s>>>(topk_ids, nullptr, T, E, K, nb, w.hist, w.tokblk, err);
    perm_scan_kernel<<<1, 1024, 0, s>>>(w.hist, E, nb, w.tokblk, counts, offsets, P_out, cap, err);
    perm_scatter_kernel<false><<<nb, kTokBlock, bits_smem, s>>>(topk_ids, topk_w, nullptr, nullptr, T, E, K, nb,
                                                                w.hist, w.tokblk, cap, sorted_tok, sorted_w, tok_ptr,
                                                                tok_pairs, err);
    return cudaGetLastError();
  }
  // plain grouping into the workspace (only the expert-grouped tokens are needed)
  const long long plain_cap = static_cast<long long>(T) * K;
  perm_hist_kernel<false><<<nb, kTokBlock, bits_smem, s>>>(topk_ids, nullptr, T, E, K, nb, w.hist, w.tokblk, err);
  perm_scan_kernel<<<1, 1024, 0, s>>>(w.hist, E, nb, w.tokblk, w.plain_cnt, w.plain_off, nullptr, plain_cap, err);
  perm_scatter_kernel<false><<<nb, kTokBlock, bits_smem, s>>>(topk_ids, nullptr, nullptr, nullptr, T, E, K, nb,
                                                              w.hist, w.tokblk, plain_cap, w.plain_tok, nullptr,
                                                              nullptr, nullptr, err);
  if ((st = cudaGetLastError()) != cudaSuccess) return st;
  // final token sets
  const size_t mbytes = sizeof(uint32_t) * static_cast<size_t>(T) * ((E + 31) / 32);
  if ((st = cudaMemsetAsync(w.member, 0, mbytes, s)) != cudaSuccess) return st;
  const size_t tr_smem = sizeof(uint32_t) * (static_cast<size_t>(T) + (T + 31) / 32);
  st = cudaFuncSetAttribute(tr_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                            static_cast<int>(sizeof(uint32_t) * (kTrMaxT + kTrMaxT / 32)));
  if (st != cudaSuccess) return st;
  tr_select_kernel<<<E, kTrThreads, tr_smem, s>>>(scores, T, E, m_tile, w.plain_off, w.plain_tok, plain_cap,
                                                 w.member, err);
  // group the final pairs
  perm_hist_kernel<true><<<nb, kTokBlock, bits_smem, s>>>(topk_ids, w.member, T, E, K, nb, w.hist, w.tokblk, err);
  perm_scan_kernel<<<1, 1024, 0, s>>>(w.hist, E, nb, w.tokblk, counts, offsets, P_out, cap, err);
  perm_scatter_kernel<true><<<nb, kTokBlock, bits_smem, s>>>(topk_ids, topk_w, w.member, logits, T, E, K, nb,
                                                             w.hist, w.tokblk, cap, sorted_tok, sorted_w, tok_ptr,
                                                             tok_pairs, err);
  return cudaGetLastError();
}

}  // namespace vgg

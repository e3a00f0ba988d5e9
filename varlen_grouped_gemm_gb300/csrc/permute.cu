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
//   2. scan:    one warp per expert scans its blocks in place (the expert's
//               pairs before each block) and totals them; one block scans the
//               totals into the offsets and the per-block token pair bases
//   3. scatter: sorted position = offsets[e] + hist[e][b] + in-block rank.
// Token rounding ([SM] "5 기여 ③ Token Rounding 라우팅") runs the plain grouping
// first, then per expert selects the final token set (tr_select_kernel) into a
// [T x E] membership bitmap, and groups again from that bitmap.  The capacity
// dispatch ([DEP] "Drop/Padding 방식") does the same with cap_select_kernel and
// scatters the kept pairs into slots e*C + (rank in token order).
#include <climits>

#include "internal.h"

namespace vgg {


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
    // the token's K choices (K <= 8) loaded together, then inserted in ascending expert order
    int ek[8];
    float wk[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      ek[k] = k < K ? __ldg(ids + static_cast<long long>(t) * K + k) : 0;
      wk[k] = (k < K && topk_w) ? __ldg(topk_w + static_cast<long long>(t) * K + k) : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k >= K) break;
      const int e = ek[k];
      const float w = wk[k];
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
    // the token's top-K (ids and weights, loaded once); a pair outside it (a padded one) gets
    // exp(l_e - l_max) / sum over the top-K of exp(l_k - l_max), the denominator taken on first need
    int ek[8];
    float wk[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      ek[k] = k < K ? __ldg(ids + static_cast<long long>(t) * K + k) : -1;
      wk[k] = k < K ? __ldg(topk_w + static_cast<long long>(t) * K + k) : 0.0f;
    }
    float lmax = 0.0f, denom = 0.0f;
    bool have_denom = false;
    for (int wi = 0; wi < W; ++wi) {
      uint32_t word = member[static_cast<long long>(t) * W + wi];
      while (word) {
        const int bit = __ffs(word) - 1;
        word &= word - 1;
        const int e = wi * 32 + bit;
        float w = -1.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (ek[k] == e) w = wk[k];
        if (w < 0.0f && logits) {
          if (!have_denom) {
            lmax = logits[static_cast<long long>(t) * E + ek[0]];
            for (int k = 0; k < K; ++k) denom += expf(logits[static_cast<long long>(t) * E + ek[k]] - lmax);
            have_denom = true;
          }
          w = expf(logits[static_cast<long long>(t) * E + e] - lmax) / denom;
        } else if (w < 0.0f) {
          w = 0.0f;
        }
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

template <bool FROM_MEMBER, int TB>
__global__ void __launch_bounds__(TB) perm_hist_kernel(const int32_t* __restrict__ ids,
                                                      const uint32_t* __restrict__ member, int T, int E, int K,
                                                      int nb, int32_t* __restrict__ hist,
                                                      int32_t* __restrict__ tokblk, int* err) {
  constexpr int NW = TB / 32;  // membership words per expert
  extern __shared__ uint32_t bits[];  // [E][NW]
  __shared__ int s_warp[33];
  const int b = blockIdx.x, tid = threadIdx.x;
  for (int i = tid; i < E * NW; i += TB) bits[i] = 0;
  __syncthreads();
  const int t = b * TB + tid;
  int cnt = 0;
  if (t < T) {
    if (!FROM_MEMBER) {
      int es[8];
      float ws[8];
      cnt = token_experts<false>(t, ids, nullptr, nullptr, nullptr, E, K, es, ws, 8, err);
      for (int q = 0; q < cnt; ++q) atomicOr(&bits[es[q] * NW + (tid >> 5)], 1u << (tid & 31));
    } else {
      const int W = (E + 31) >> 5;
      for (int wi = 0; wi < W; ++wi) {
        uint32_t word = member[static_cast<long long>(t) * W + wi];
        while (word) {
          const int bit = __ffs(word) - 1;
          word &= word - 1;
          atomicOr(&bits[(wi * 32 + bit) * NW + (tid >> 5)], 1u << (tid & 31));
          ++cnt;
        }
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += TB) {
    int s = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += __popc(bits[e * NW + w]);
    hist[static_cast<long long>(e) * nb + b] = s;
  }
  int total;
  block_exclusive_scan_256(cnt, s_warp, total);
  if (tid == 0) tokblk[b] = total;
}

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

// Scan, level 1: one warp per expert turns its per-block counts hist[e][*] into in-expert exclusive
// prefixes (block order = token order) and writes the expert's total.
__global__ void __launch_bounds__(256) perm_escan_kernel(int32_t* __restrict__ hist, int E, int nb,
                                                         int32_t* __restrict__ counts) {
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (e >= E) return;
  int32_t* h = hist + static_cast<long long>(e) * nb;
  int carry = 0;
  for (int b0 = 0; b0 < nb; b0 += 32) {
    const int b = b0 + lane;
    const int v = b < nb ? h[b] : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (b < nb) h[b] = carry + x - v;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  if (lane == 0) counts[e] = carry;
}

// Scan, level 2 (one block): offsets = exclusive scan of the expert totals, offsets[E] = P, and the
// exclusive scan of the per-block token pair counts.
__global__ void __launch_bounds__(1024) perm_scan_kernel(const int32_t* __restrict__ counts, int E,
                                                         int32_t* __restrict__ tokblk, int nb,
                                                         int32_t* __restrict__ offsets, int32_t* __restrict__ P_out,
                                                         long long cap, int* err) {
  __shared__ int s_warp[33];
  __shared__ int s_tok;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int carry = 0;
  for (int base = 0; base < E; base += 1024) {  // E <= 1024: one pass
    const int e = base + tid;
    const int v = e < E ? counts[e] : 0;
    int total;
    const int ex = block_exclusive_scan_1024(v, s_warp, total);
    if (e < E) offsets[e] = carry + ex;
    carry += total;
  }
  if (warp == 0) {
    int tcarry = 0;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      const int i = b0 + lane;
      const int v = (i < nb) ? tokblk[i] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (i < nb) tokblk[i] = tcarry + x - v;
      tcarry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) {
      tokblk[nb] = tcarry;
      s_tok = tcarry;
    }
  }
  __syncthreads();
  if (tid == 0) {
    offsets[E] = carry;
    if (P_out) *P_out = carry;
    if (carry > cap || s_tok != carry) set_error(err, DERR_CAPACITY);
  }
}

void launch_scan(int32_t* hist, int E, int nb, int32_t* tokblk, int32_t* counts, int32_t* offsets, int32_t* P_out,
                 long long cap, int* err, cudaStream_t s) {
  perm_escan_kernel<<<(E + 7) / 8, 256, 0, s>>>(hist, E, nb, counts);
  perm_scan_kernel<<<1, 1024, 0, s>>>(counts, E, tokblk, nb, offsets, P_out, cap, err);
}

template <bool FROM_MEMBER, int TB>
__global__ void __launch_bounds__(TB) perm_scatter_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ topk_w, const uint32_t* __restrict__ member,
    const float* __restrict__ logits, int T, int E, int K, int nb, const int32_t* __restrict__ base,
    const int32_t* __restrict__ eoff,
    const int32_t* __restrict__ tokbase, long long cap, int32_t* __restrict__ sorted_tok,
    float* __restrict__ sorted_w, int32_t* __restrict__ tok_ptr, int32_t* __restrict__ tok_pairs, int* err,
    int slot_stride) {
  constexpr int NW = TB / 32;
  extern __shared__ uint32_t bits[];  // [E][NW]
  __shared__ int s_warp[33];
  // pairs per token: K without rounding; rounding may pad a token into more experts
  constexpr int kMaxPairs = FROM_MEMBER ? 32 : 8;
  const int b = blockIdx.x, tid = threadIdx.x;
  for (int i = tid; i < E * NW; i += TB) bits[i] = 0;
  __syncthreads();
  const int t = b * TB + tid;
  int es[kMaxPairs];
  float ws[kMaxPairs];
  int cnt = 0;
  if (t < T) {
    cnt = token_experts<FROM_MEMBER>(t, ids, topk_w, member, logits, E, K, es, ws, kMaxPairs, err);
    if (cnt > kMaxPairs) {
      set_error(err, DERR_CAPACITY);
      cnt = kMaxPairs;
    }
    for (int q = 0; q < cnt; ++q) atomicOr(&bits[es[q] * NW + (tid >> 5)], 1u << (tid & 31));
  }
  __syncthreads();
  int total;
  const int tprefix = block_exclusive_scan_256(cnt, s_warp, total);
  const long long tp = static_cast<long long>(tokbase[b]) + tprefix;
  if (t < T && tok_ptr) tok_ptr[t] = static_cast<int32_t>(tp);
  if (t == T - 1 && tok_ptr) tok_ptr[T] = static_cast<int32_t>(tp + cnt);
  const int w_self = tid >> 5;
  const uint32_t lt_mask = (1u << (tid & 31)) - 1u;
  // base: the pair's rank among its expert's pairs before this token block; eoff: the expert's first
  // position (capacity layout: expert e's kept pairs fill slots [e * slot_stride, ...) in token order).
  // The lookups of a token's pairs are issued together before any is used.
  long long first[kMaxPairs];
#pragma unroll
  for (int q = 0; q < kMaxPairs; ++q) {
    if (q < cnt) {
      const int e = es[q];
      first[q] = static_cast<long long>(__ldg(base + static_cast<long long>(e) * nb + b)) +
                 (slot_stride > 0 ? static_cast<long long>(e) * slot_stride : __ldg(eoff + e));
    }
  }
#pragma unroll
  for (int q = 0; q < kMaxPairs; ++q) {
    if (q >= cnt) break;
    const int e = es[q];
    int rank = __popc(bits[e * NW + w_self] & lt_mask);
    for (int w = 0; w < w_self; ++w) rank += __popc(bits[e * NW + w]);
    const long long j = first[q] + rank;
    if (j >= cap || tp + q >= cap) {
      set_error(err, DERR_CAPACITY);
      continue;
    }
    sorted_tok[j] = t;
    if (sorted_w) sorted_w[j] = ws[q];
    if (tok_pairs) tok_pairs[tp + q] = static_cast<int32_t>(j);
  }
}

// Grid-wide barrier of a cooperative launch (every block resident): thread 0 of each block arrives on
// `counter` (zeroed before the launch) and waits, bounded by timeout_ns, until `target` arrivals.  The
// block's writes before the barrier are visible to every block after it.  Returns false, with
// MOE_DEV_TIMEOUT recorded, when the wait gave up.
__device__ bool grid_barrier(int* counter, int target, unsigned long long timeout_ns, int* err, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(counter, 1);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0;; ++i) {
      int v;
      asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
      if (v >= target) break;
      if ((i & 15u) == 15u && globaltimer_ns() - t0 > timeout_ns) {
        set_error(err, DERR_TIMEOUT);
        ok = 0;
        break;
      }
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// The whole grouping in one cooperative launch (one block per TB tokens, all resident), with the results of
// perm_hist + perm_escan + perm_scan + perm_scatter: (1) a block's membership bits per expert, its per-expert
// counts hist[e][b] and its pair count; grid barrier; (2) one warp per expert turns hist[e][*] into in-expert
// exclusive prefixes over the blocks (block order = token order) and writes the expert's total; grid barrier;
// (3) every block scans the expert totals (offsets; block 0 writes them, offsets[E] = P and the capacity
// check) and sums the pair counts of the blocks before it, then scatters its pairs with the bits it kept in
// shared memory.  Data written by other blocks during the launch is read with L1-bypassing loads.
template <bool FROM_MEMBER, int TB>
__global__ void __launch_bounds__(TB) perm_fused_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ topk_w, const uint32_t* __restrict__ member,
    const float* __restrict__ logits, int T, int E, int K, int nb, int32_t* hist, int32_t* tokblk, int* barrier,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ P_out, long long cap,
    int32_t* __restrict__ sorted_tok, float* __restrict__ sorted_w, int32_t* __restrict__ tok_ptr,
    int32_t* __restrict__ tok_pairs, int* err, int slot_stride, unsigned long long timeout_ns) {
  constexpr int NW = TB / 32;
  constexpr int kMaxPairs = FROM_MEMBER ? 32 : 8;
  extern __shared__ uint32_t fsm[];  // bits [E][NW], then the expert offsets [E + 1]
  uint32_t* bits = fsm;
  int* s_eoff = reinterpret_cast<int*>(fsm + E * NW);
  __shared__ int s_warp[33];
  __shared__ int s_ok, s_tokbase, s_toktotal;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // (1) this block's tokens
  for (int i = tid; i < E * NW; i += TB) bits[i] = 0;
  __syncthreads();
  const int t = b * TB + tid;
  int es[kMaxPairs];
  float ws[kMaxPairs];
  int cnt = 0;
  if (t < T) {
    cnt = token_experts<FROM_MEMBER>(t, ids, topk_w, member, logits, E, K, es, ws, kMaxPairs, err);
    if (cnt > kMaxPairs) {
      set_error(err, DERR_CAPACITY);
      cnt = kMaxPairs;
    }
    for (int q = 0; q < cnt; ++q) atomicOr(&bits[es[q] * NW + warp], 1u << lane);
  }
  __syncthreads();
  for (int e = tid; e < E; e += TB) {
    int n = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) n += __popc(bits[e * NW + w]);
    hist[static_cast<long long>(e) * nb + b] = n;
  }
  int btotal;
  const int tprefix = block_exclusive_scan_256(cnt, s_warp, btotal);
  if (tid == 0) tokblk[b] = btotal;
  if (!grid_barrier(barrier, nb, timeout_ns, err, &s_ok)) return;
  // (2) in-expert prefixes over the blocks
  for (int e = b * NW + warp; e < E; e += nb * NW) {
    int32_t* h = hist + static_cast<long long>(e) * nb;
    int carry = 0;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      const int bb = b0 + lane;
      const int v = bb < nb ? __ldcg(h + bb) : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (bb < nb) h[bb] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) counts[e] = carry;
  }
  if (!grid_barrier(barrier, 2 * nb, timeout_ns, err, &s_ok)) return;
  // (3) expert offsets, this block's first pair, the scatter
  int ecarry = 0;
  for (int base = 0; base < E; base += TB) {
    const int e = base + tid;
    const int v = e < E ? __ldcg(counts + e) : 0;
    int tot;
    const int ex = block_exclusive_scan_256(v, s_warp, tot);
    if (e < E) s_eoff[e] = ecarry + ex;
    ecarry += tot;
  }
  int tb_before = 0, tb_all = 0;
  for (int i = tid; i < nb; i += TB) {
    const int v = __ldcg(tokblk + i);
    if (i < b) tb_before += v;
    tb_all += v;
  }
  {
    int tot;
    block_exclusive_scan_256(tb_before, s_warp, tot);
    if (tid == 0) s_tokbase = tot;
    block_exclusive_scan_256(tb_all, s_warp, tot);
    if (tid == 0) s_toktotal = tot;
  }
  if (tid == 0) s_eoff[E] = ecarry;
  __syncthreads();
  if (b == 0) {
    for (int e = tid; e <= E; e += TB) offsets[e] = s_eoff[e];
    if (tid == 0) {
      if (P_out) *P_out = ecarry;
      if (ecarry > cap || s_toktotal != ecarry) set_error(err, DERR_CAPACITY);
    }
  }
  const long long tp = static_cast<long long>(s_tokbase) + tprefix;
  if (t < T && tok_ptr) tok_ptr[t] = static_cast<int32_t>(tp);
  if (t == T - 1 && tok_ptr) tok_ptr[T] = static_cast<int32_t>(tp + cnt);
  const uint32_t lt_mask = (1u << lane) - 1u;
  long long first[kMaxPairs];
#pragma unroll
  for (int q = 0; q < kMaxPairs; ++q) {
    if (q < cnt) {
      const int e = es[q];
      first[q] = static_cast<long long>(__ldcg(hist + static_cast<long long>(e) * nb + b)) +
                 (slot_stride > 0 ? static_cast<long long>(e) * slot_stride : s_eoff[e]);
    }
  }
#pragma unroll
  for (int q = 0; q < kMaxPairs; ++q) {
    if (q >= cnt) break;
    const int e = es[q];
    int rank = __popc(bits[e * NW + warp] & lt_mask);
    for (int w = 0; w < warp; ++w) rank += __popc(bits[e * NW + w]);
    const long long j = first[q] + rank;
    if (j >= cap || tp + q >= cap) {
      set_error(err, DERR_CAPACITY);
      continue;
    }
    sorted_tok[j] = t;
    if (sorted_w) sorted_w[j] = ws[q];
    if (tok_pairs) tok_pairs[tp + q] = static_cast<int32_t>(j);
  }
}

// out[c][r] = in[r][c] for fp32 [rows x cols], 32x32 tiles through shared memory: the token
// rounding select reads one expert's scores for all tokens, a column of the [T x E] scores.
__global__ void transpose_f32_kernel(const float* __restrict__ in, int rows, int cols, float* __restrict__ out) {
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = in[static_cast<long long>(r) * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) out[static_cast<long long>(c) * rows + r] = tile[threadIdx.x][i];
  }
}

// Token rounding, one CTA per expert: choose the final token set of expert e
// and mark it in the membership bitmap.  Priority of a token for e is
// (score descending, token ascending); the selection is a radix select of the
// need-th largest score among the candidates, ties at the threshold resolved
// by ascending token.  Keys (score bits; positive floats order as integers)
// are read from the transposed scores, L2-resident, by each pass that needs
// them, so a CTA's shared memory holds only the short lists (two CTAs fit an
// SM).  The first digit (bits 31..21) is histogrammed
// over all candidates; the keys of the bin holding the threshold are then
// compacted into a short list that the two remaining digits (20..10, 9..0)
// scan, so only one pass touches every token.
constexpr int kTrThreads = 1024;
constexpr int kTrMaxT = 32768;
constexpr int kTrListCap = 8192;  // compacted keys of the threshold bin; a larger bin rescans all keys

// The digit of the remaining-th largest from a filled histogram of digit (k >> shift) & (NB - 1): thread i owns
// bins [NB / kTrThreads i, ...); a block-wide suffix scan of the threads' counts (from the highest bins down) finds
// the owner of the bin where the count from the top reaches `remaining`, which walks its bins downwards.  Updates
// prefix, mask, remaining; returns the count of the chosen bin.
template <int NB>
__device__ int tr_pick(const int* hist, uint32_t& prefix, uint32_t& mask, int shift, int& remaining, int* s_res) {
  static_assert(NB % kTrThreads == 0, "whole bins per thread");
  constexpr int PER = NB / kTrThreads;
  constexpr int NW = kTrThreads / 32;
  __shared__ int s_wsum[NW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int sl = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) sl += hist[PER * tid + i];
  // suffix sum within the warp (lanes above), then over the warps above
  int suf = sl;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += y;
  }
  if (lane == 0) s_wsum[warp] = suf;  // the warp's total
  __syncthreads();
  int above = 0;
  for (int w = warp + 1; w < NW; ++w) above += s_wsum[w];
  suf += above;  // count of the bins from this thread's first bin to the top
  if (tid == 0 && suf < remaining) {  // fewer candidates than asked for (outside the contract): the lowest bin
    s_res[0] = 0;
    s_res[1] = remaining - suf;
    s_res[2] = 0;
  }
  if (suf >= remaining && suf - sl < remaining) {  // exactly one thread: the bin is among its own
    int cum = suf - sl, digit = PER * tid, cnt = 0;
    for (int i = PER - 1; i >= 0; --i) {
      const int h = hist[PER * tid + i];
      if (cum + h >= remaining) {
        digit = PER * tid + i;
        cnt = h;
        break;
      }
      cum += h;
    }
    s_res[0] = digit;
    s_res[1] = remaining - cum;
    s_res[2] = cnt;
  }
  __syncthreads();
  prefix |= static_cast<uint32_t>(s_res[0]) << shift;
  mask |= static_cast<uint32_t>(NB - 1) << shift;
  remaining = s_res[1];
  const int cnt = s_res[2];
  __syncthreads();
  return cnt;
}

// Add digit dg (NB = not counted) of each thread's key to hist, once per group of equal digits in the warp.
template <int NB>
__device__ __forceinline__ void tr_count(int* hist, uint32_t dg) {
  const unsigned grp = __match_any_sync(0xffffffffu, dg);
  if (dg != static_cast<uint32_t>(NB) && (threadIdx.x & 31) == __ffs(grp) - 1) atomicAdd(&hist[dg], __popc(grp));
}

// Histogram of digit (k >> shift) & (NB - 1) over keys key(i), i < n, matching `prefix` on `mask` (0xFFFFFFFF =
// not a candidate), then tr_pick.
template <int NB, class KeyAt>
__device__ int tr_digit(KeyAt key, int n, uint32_t& prefix, uint32_t& mask, int shift, int& remaining, int* hist,
                        int* s_res) {
  const int tid = threadIdx.x;
  for (int i = tid; i < NB; i += kTrThreads) hist[i] = 0;
  __syncthreads();
  for (int i0 = 0; i0 < n; i0 += kTrThreads) {
    const int i = i0 + tid;
    uint32_t dg = NB;
    if (i < n) {
      const uint32_t k = key(i);
      if (k != 0xFFFFFFFFu && (k & mask) == prefix) dg = (k >> shift) & (NB - 1);
    }
    tr_count<NB>(hist, dg);
  }
  __syncthreads();
  return tr_pick<NB>(hist, prefix, mask, shift, remaining, s_res);
}


// The `need` largest keys key(i), i < n (0xFFFFFFFF = not a candidate), ties at the threshold going to the
// lowest indices: a radix select (one 11-bit digit over all keys, the threshold bin compacted into `list` for
// the two remaining digits), then take(i) for every selected index i.  Block-wide; 1 <= need <= the number of
// candidates.  key(i) is evaluated once per pass (the caller's source: global memory, L2-resident here).
template <class KeyAt, class Take>
__device__ void select_take(KeyAt key, int n, int need, uint32_t* list, int* hist, int* s_res, Take take) {
  __shared__ int s_wties[kTrThreads / 32];
  const int tid = threadIdx.x;
  uint32_t prefix = 0, mask = 0;
  int remaining = need;
  const int lane = tid & 31;
  tr_digit<2048>(key, n, prefix, mask, 21, remaining, hist, s_res);
  // compact the keys of the threshold bin (warp-aggregated appends; order is irrelevant here)
  if (tid == 0) s_res[3] = 0;
  __syncthreads();
  for (int t0 = 0; t0 < n; t0 += kTrThreads) {
    const int t = t0 + tid;
    const uint32_t k = t < n ? key(t) : 0xFFFFFFFFu;
    const bool in = k != 0xFFFFFFFFu && (k & mask) == prefix;
    const unsigned bal = __ballot_sync(0xffffffffu, in);
    int base = 0;
    if (lane == 0 && bal) base = atomicAdd(&s_res[3], __popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    const int pos = base + __popc(bal & ((1u << lane) - 1u));
    if (in && pos < kTrListCap) list[pos] = k;
  }
  __syncthreads();
  const int nlist = s_res[3];
  int ties;
  const auto listed = [list](int i) { return list[i]; };
  if (nlist <= kTrListCap) {
    tr_digit<2048>(listed, nlist, prefix, mask, 10, remaining, hist, s_res);
    ties = tr_digit<1024>(listed, nlist, prefix, mask, 0, remaining, hist, s_res);
  } else {
    tr_digit<2048>(key, n, prefix, mask, 10, remaining, hist, s_res);
    ties = tr_digit<1024>(key, n, prefix, mask, 0, remaining, hist, s_res);
  }
  // keys above the threshold are all taken; at the threshold the `remaining` lowest indices.
  if (ties == remaining) {  // every tie is taken: no order needed
    for (int t = tid; t < n; t += kTrThreads) {
      const uint32_t k = key(t);
      if (k != 0xFFFFFFFFu && k >= prefix) take(t);
    }
    return;
  }
  // Equal keys beyond the need: indices in chunks of kTrThreads; a tie's rank in index order is the
  // ties of earlier chunks, of earlier warps of this chunk and of lower lanes.
  const int warp_id = tid >> 5;
  int tie_base = 0;
  for (int base = 0; base < n; base += kTrThreads) {
    const int t = base + tid;
    const uint32_t k = t < n ? key(t) : 0xFFFFFFFFu;
    const bool cand = k != 0xFFFFFFFFu;
    const bool tie = cand && k == prefix;
    const unsigned bal = __ballot_sync(0xffffffffu, tie);
    if (lane == 0) s_wties[warp_id] = __popc(bal);
    __syncthreads();
    int before = tie_base + __popc(bal & ((1u << lane) - 1u)), chunk_ties = 0;
    for (int w = 0; w < kTrThreads / 32; ++w) {
      const int cw = s_wties[w];
      if (w < warp_id) before += cw;
      chunk_ties += cw;
    }
    if (cand && (k > prefix || (tie && before < remaining))) take(t);
    tie_base += chunk_ties;
    __syncthreads();
  }
}

// Token rounding's padding: the `need` largest scores among the tokens not routed to the expert (col:
// the expert's scores, token-contiguous; routed: bitmap of its routed tokens), ties to the lower token;
// take(t) for each.  A candidate's key is its score's bits, read from col (global memory: the transposed
// scores, L2-resident after the transpose) at every pass rather than staged, so that the CTA's shared
// memory is small enough for two CTAs per SM.  The first digit is counted over all candidates; when the
// threshold bin fits the list, one pass takes every key above that bin and compacts the bin's keys with
// their tokens, and the rest runs on the list.  Otherwise select_take runs over all the candidates.
template <class Take>
__device__ void select_take_unrouted(const float* col, const uint32_t* routed, int T, int need, uint32_t* list,
                                     int* list_tok, int* hist, int* s_res, Take take) {
  const int tid = threadIdx.x, lane = tid & 31;
  const auto key = [col, routed](int t) -> uint32_t {
    return ((routed[t >> 5] >> (t & 31)) & 1u) ? 0xFFFFFFFFu : __float_as_uint(__ldg(col + t));
  };
  for (int i = tid; i < 2048; i += kTrThreads) hist[i] = 0;
  __syncthreads();
#pragma unroll 4
  for (int t0 = 0; t0 < T; t0 += kTrThreads) {
    const int t = t0 + tid;
    uint32_t dg = 2048;
    if (t < T) {
      const uint32_t k = key(t);
      if (k != 0xFFFFFFFFu) dg = k >> 21;
    }
    tr_count<2048>(hist, dg);
  }
  __syncthreads();
  uint32_t prefix = 0, mask = 0;
  int remaining = need;
  const int bin_cnt = tr_pick<2048>(hist, prefix, mask, 21, remaining, s_res);
  if (bin_cnt > kTrListCap) {  // a crowded bin: the general select over all the candidates
    select_take(key, T, need, list, hist, s_res, take);
    return;
  }
  const uint32_t bin = prefix >> 21;
  if (tid == 0) s_res[3] = 0;
  __syncthreads();
  for (int t0 = 0; t0 < T; t0 += kTrThreads) {
    const int t = t0 + tid;
    const uint32_t k = t < T ? key(t) : 0xFFFFFFFFu;
    const bool cand = k != 0xFFFFFFFFu;
    if (cand && (k >> 21) > bin) take(t);  // above the threshold bin: always in
    const bool in = cand && (k >> 21) == bin;
    const unsigned bal = __ballot_sync(0xffffffffu, in);
    int base = 0;
    if (lane == 0 && bal) base = atomicAdd(&s_res[3], __popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    const int pos = base + __popc(bal & ((1u << lane) - 1u));
    if (in && pos < kTrListCap) {
      list[pos] = k;
      list_tok[pos] = t;
    }
  }
  __syncthreads();
  const int nlist = min(s_res[3], kTrListCap);
  const auto listed = [list](int i) { return list[i]; };
  tr_digit<2048>(listed, nlist, prefix, mask, 10, remaining, hist, s_res);
  const int ties = tr_digit<1024>(listed, nlist, prefix, mask, 0, remaining, hist, s_res);
  // prefix is now the threshold key: the list's keys above it are in, and `remaining` of its ties,
  // the lowest tokens first
  for (int i = tid; i < nlist; i += kTrThreads) {
    const uint32_t k = list[i];
    if (k > prefix) {
      take(list_tok[i]);
    } else if (k == prefix && ties == remaining) {
      take(list_tok[i]);
    } else if (k == prefix && ties <= 256) {
      int rank = 0;
      const int ti = list_tok[i];
      for (int q = 0; q < nlist; ++q) rank += (list[q] == prefix && list_tok[q] < ti) ? 1 : 0;
      if (rank < remaining) take(ti);
    }
  }
  if (ties == remaining || ties <= 256) return;
  // many equal keys at the threshold: rank the ties in token order over all the candidates
  __shared__ int s_wt[kTrThreads / 32];
  const int warp_id = tid >> 5;
  int tie_base = 0;
  for (int base = 0; base < T; base += kTrThreads) {
    const int t = base + tid;
    const bool tie = t < T && key(t) == prefix;
    const unsigned bal = __ballot_sync(0xffffffffu, tie);
    if (lane == 0) s_wt[warp_id] = __popc(bal);
    __syncthreads();
    int before = tie_base + __popc(bal & ((1u << lane) - 1u)), chunk_ties = 0;
    for (int w = 0; w < kTrThreads / 32; ++w) {
      const int cw = s_wt[w];
      if (w < warp_id) before += cw;
      chunk_ties += cw;
    }
    if (tie && before < remaining) take(t);
    tie_base += chunk_ties;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kTrThreads, 2) tr_select_kernel(const float* __restrict__ scoresT, int T, int E,
                                                              int m_tile, const int32_t* __restrict__ plain_off,
                                                              const int32_t* __restrict__ plain_tok,
                                                              long long plain_cap, uint32_t* __restrict__ member,
                                                              int* err) {
  extern __shared__ uint32_t tr_smem[];
  uint32_t* routed = tr_smem;             // [ceil(T/32)]
  uint32_t* list = routed + ((T + 31) >> 5);  // [kTrListCap] keys of the threshold bin
  int* list_tok = reinterpret_cast<int*>(list + kTrListCap);  // [kTrListCap] their tokens
  __shared__ int hist[2048];
  __shared__ int s_res[4];
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
  const float* col = scoresT + static_cast<long long>(e) * T;  // this expert's scores, token-contiguous
  if (drop) {
    // the candidates are the c routed tokens, in token order: select among them alone
    const int32_t* toks = plain_tok + off;
    select_take(
        [toks, col, T](int i) -> uint32_t {
          const int t = __ldg(toks + i);
          return (t >= 0 && t < T) ? __float_as_uint(__ldg(col + t)) : 0xFFFFFFFFu;
        },
        c, need, list, hist, s_res,
        [&](int i) { atomicOr(&member[static_cast<long long>(plain_tok[off + i]) * W + ew], ebit); });
    return;
  }
  select_take_unrouted(col, routed, T, need, list, list_tok, hist, s_res, [&](int t) {
    atomicOr(&member[static_cast<long long>(t) * W + ew], ebit);
  });
}

// Capacity dispatch ([DEP] "Drop/Padding 방식"), one CTA per expert: of the expert's routed pairs
// (token order) keep the first C ("position") or the C with the largest routing probability, ties
// to the lower token ("probs"), and mark them in the membership bitmap.
__global__ void __launch_bounds__(kTrThreads) cap_select_kernel(const int32_t* __restrict__ plain_off,
                                                               const int32_t* __restrict__ plain_tok,
                                                               const float* __restrict__ plain_w, long long plain_cap,
                                                               int T, int E, int C, int policy,
                                                               uint32_t* __restrict__ member, int* err) {
  extern __shared__ uint32_t cs_smem[];
  uint32_t* list = cs_smem;  // [kTrListCap]
  __shared__ int hist[2048];
  __shared__ int s_res[4];
  const int e = blockIdx.x, tid = threadIdx.x;
  const int W = (E + 31) >> 5;
  const int off = plain_off[e];
  const int c = plain_off[e + 1] - off;
  if (off < 0 || c < 0 || off + c > plain_cap || c > T) {
    if (tid == 0) set_error(err, DERR_BAD_OFFSETS);
    return;
  }
  const uint32_t ebit = 1u << (e & 31);
  const int ew = e >> 5;
  auto keep = [&](int i) {
    const int t = plain_tok[off + i];
    if (t >= 0 && t < T) atomicOr(&member[static_cast<long long>(t) * W + ew], ebit);
  };
  if (c <= C || policy == 0) {  // everything fits, or the first C in token order
    const int nk = min(c, C);
    for (int i = tid; i < nk; i += kTrThreads) keep(i);
    return;
  }
  // the keys: the routing probabilities of the expert's pairs in token order (positive floats order as their bits)
  const float* pw = plain_w + off;
  select_take([pw](int i) -> uint32_t { return __float_as_uint(__ldg(pw + i)); }, c, C, list, hist, s_res, keep);
}

// offsets of the capacity layout: expert e owns slots [e C, (e + 1) C); every slot is a row of the GEMMs.
__global__ void slot_offsets_kernel(int32_t* offsets, int E, int C, int32_t* P_out) {
  for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = e * C;
  if (threadIdx.x == 0 && P_out) *P_out = E * C;
}

size_t permute_ws_bytes(int T, int E, int K, int m_tile) {
  const int tb = perm_tok_block(T, E);
  const long long nb = (T + tb - 1) / tb;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t b = al(sizeof(int32_t) * E * nb) + al(sizeof(int32_t) * (nb + 2));
  if (m_tile > 0) {
    b += al(sizeof(uint32_t) * static_cast<size_t>(T) * ((E + 31) / 32));
    b += al(sizeof(int32_t) * (E + 1)) + al(sizeof(int32_t) * E) + al(sizeof(int32_t) * static_cast<size_t>(T) * K);
    b += al(sizeof(float) * static_cast<size_t>(T) * E);
  }
  return b;
}

PermuteWs carve_permute_ws(void* ws, int T, int E, int K, int m_tile) {
  const int tb = perm_tok_block(T, E);
  const long long nb = (T + tb - 1) / tb;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint8_t* p = static_cast<uint8_t*>(ws);
  PermuteWs w{};
  w.hist = reinterpret_cast<int32_t*>(p);
  p += al(sizeof(int32_t) * E * nb);
  w.tokblk = reinterpret_cast<int32_t*>(p);
  w.barrier = w.tokblk + nb + 1;
  p += al(sizeof(int32_t) * (nb + 2));
  if (m_tile > 0) {
    w.member = reinterpret_cast<uint32_t*>(p);
    p += al(sizeof(uint32_t) * static_cast<size_t>(T) * ((E + 31) / 32));
    w.plain_off = reinterpret_cast<int32_t*>(p);
    p += al(sizeof(int32_t) * (E + 1));
    w.plain_cnt = reinterpret_cast<int32_t*>(p);
    p += al(sizeof(int32_t) * E);
    w.plain_tok = reinterpret_cast<int32_t*>(p);
    p += al(sizeof(int32_t) * static_cast<size_t>(T) * K);
    w.scoresT = reinterpret_cast<float*>(p);
  }
  return w;
}

// Launch a grouping kernel (template <bool FROM_MEMBER, int TB>) with TB threads per block.
#define VGG_PERM_LAUNCH(KERNEL, FM, tb, nb, smem, s, ...)                        \
  do {                                                                           \
    switch (tb) {                                                                \
      case 32: KERNEL<FM, 32><<<nb, 32, smem, s>>>(__VA_ARGS__); break;          \
      case 64: KERNEL<FM, 64><<<nb, 64, smem, s>>>(__VA_ARGS__); break;          \
      case 128: KERNEL<FM, 128><<<nb, 128, smem, s>>>(__VA_ARGS__); break;       \
      default: KERNEL<FM, 256><<<nb, 256, smem, s>>>(__VA_ARGS__); break;        \
    }                                                                            \
  } while (0)

// The one-launch grouping (perm_fused_kernel) as a cooperative launch.  Returns
// cudaErrorCooperativeLaunchTooLarge, launching nothing, when its blocks cannot all be resident at once.
template <bool FM, int TB>
cudaError_t launch_fused_grouping(int nb, const int32_t* ids, const float* topk_w, const uint32_t* member,
                                  const float* logits, int T, int E, int K, const PermuteWs& w, int32_t* counts,
                                  int32_t* offsets, int32_t* P_out, long long cap, int32_t* sorted_tok,
                                  float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs, int* err, int slot_stride,
                                  unsigned long long timeout_ns, cudaStream_t s) {
  auto kern = perm_fused_kernel<FM, TB>;
  const size_t smem = sizeof(uint32_t) * (static_cast<size_t>(E) * (TB / 32) + E + 1);
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t st;
  if ((st = cudaGetDevice(&dev)) != cudaSuccess) return st;
  if ((st = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return st;
  if ((st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, TB, smem)) != cudaSuccess) return st;
  if (static_cast<long long>(per_sm) * sms < nb) return cudaErrorCooperativeLaunchTooLarge;
  if ((st = cudaMemsetAsync(w.barrier, 0, sizeof(int), s)) != cudaSuccess) return st;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(nb, 1, 1);
  cfg.blockDim = dim3(TB, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ids, topk_w, member, logits, T, E, K, nb, w.hist, w.tokblk, w.barrier, counts,
                            offsets, P_out, cap, sorted_tok, sorted_w, tok_ptr, tok_pairs, err, slot_stride,
                            timeout_ns);
}

// Group the pairs (from top-K ids, or from the membership bitmap with FM) into counts, offsets, the
// expert-major order and the per-token return map: one cooperative launch when its blocks fit on the GPU at
// once, else the four launches perm_hist, perm_escan, perm_scan, perm_scatter (the same results).
template <bool FM>
cudaError_t group_pairs(int tb, int nb, size_t bits_smem, const int32_t* ids, const float* topk_w,
                        const uint32_t* member, const float* logits, int T, int E, int K, const PermuteWs& w,
                        int32_t* counts, int32_t* offsets, int32_t* P_out, long long cap, int32_t* sorted_tok,
                        float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs, int* err, int slot_stride,
                        unsigned long long timeout_ns, cudaStream_t s) {
  cudaError_t st;
  switch (tb) {
    case 32: st = launch_fused_grouping<FM, 32>(nb, ids, topk_w, member, logits, T, E, K, w, counts, offsets, P_out, cap,
                                                sorted_tok, sorted_w, tok_ptr, tok_pairs, err, slot_stride, timeout_ns, s);
             break;
    case 64: st = launch_fused_grouping<FM, 64>(nb, ids, topk_w, member, logits, T, E, K, w, counts, offsets, P_out, cap,
                                                sorted_tok, sorted_w, tok_ptr, tok_pairs, err, slot_stride, timeout_ns, s);
             break;
    case 128: st = launch_fused_grouping<FM, 128>(nb, ids, topk_w, member, logits, T, E, K, w, counts, offsets, P_out,
                                                  cap, sorted_tok, sorted_w, tok_ptr, tok_pairs, err, slot_stride,
                                                  timeout_ns, s);
              break;
    default: st = launch_fused_grouping<FM, 256>(nb, ids, topk_w, member, logits, T, E, K, w, counts, offsets, P_out,
                                                 cap, sorted_tok, sorted_w, tok_ptr, tok_pairs, err, slot_stride,
                                                 timeout_ns, s);
             break;
  }
  if (st != cudaErrorCooperativeLaunchTooLarge) return st;
  VGG_PERM_LAUNCH(perm_hist_kernel, FM, tb, nb, bits_smem, s, ids, member, T, E, K, nb, w.hist, w.tokblk, err);
  launch_scan(w.hist, E, nb, w.tokblk, counts, offsets, P_out, cap, err, s);
  VGG_PERM_LAUNCH(perm_scatter_kernel, FM, tb, nb, bits_smem, s, ids, topk_w, member, logits, T, E, K, nb, w.hist,
                  offsets, w.tokblk, cap, sorted_tok, sorted_w, tok_ptr, tok_pairs, err, slot_stride);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* topk_ids, const float* topk_w, const float* logits, const float* scores,
                           int T, int E, int K, int m_tile, long long cap, int32_t* counts, int32_t* offsets,
                           int32_t* sorted_tok, float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs,
                           int32_t* P_out, const PermuteWs& w, int* err, unsigned long long timeout_ns,
                           cudaStream_t s) {
  const int tb = perm_tok_block(T, E);
  const int nb = (T + tb - 1) / tb;
  const size_t bits_smem = static_cast<size_t>(E) * (tb / 32) * sizeof(uint32_t);
  cudaError_t st;
  if (m_tile <= 0)
    return group_pairs<false>(tb, nb, bits_smem, topk_ids, topk_w, nullptr, nullptr, T, E, K, w, counts, offsets, P_out,
                              cap, sorted_tok, sorted_w, tok_ptr, tok_pairs, err, 0, timeout_ns, s);
  // plain grouping into the workspace (only the expert-grouped tokens are needed)
  const long long plain_cap = static_cast<long long>(T) * K;
  if ((st = group_pairs<false>(tb, nb, bits_smem, topk_ids, nullptr, nullptr, nullptr, T, E, K, w, w.plain_cnt,
                               w.plain_off, nullptr, plain_cap, w.plain_tok, nullptr, nullptr, nullptr, err, 0,
                               timeout_ns, s)) != cudaSuccess)
    return st;
  // final token sets
  const size_t mbytes = sizeof(uint32_t) * static_cast<size_t>(T) * ((E + 31) / 32);
  if ((st = cudaMemsetAsync(w.member, 0, mbytes, s)) != cudaSuccess) return st;
  const size_t tr_smem = sizeof(uint32_t) * (static_cast<size_t>(T + 31) / 32 + 2 * kTrListCap);
  st = cudaFuncSetAttribute(tr_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                            static_cast<int>(sizeof(uint32_t) * (kTrMaxT / 32 + 2 * kTrListCap)));
  if (st != cudaSuccess) return st;
  transpose_f32_kernel<<<dim3((E + 31) / 32, (T + 31) / 32), dim3(32, 8), 0, s>>>(scores, T, E, w.scoresT);
  tr_select_kernel<<<E, kTrThreads, tr_smem, s>>>(w.scoresT, T, E, m_tile, w.plain_off, w.plain_tok, plain_cap,
                                                 w.member, err);
  // group the final pairs
  return group_pairs<true>(tb, nb, bits_smem, topk_ids, topk_w, w.member, logits, T, E, K, w, counts, offsets, P_out,
                           cap, sorted_tok, sorted_w, tok_ptr, tok_pairs, err, 0, timeout_ns, s);
}

cudaError_t launch_permute_capacity(const int32_t* topk_ids, const float* topk_w, int T, int E, int K, int C,
                                    int policy, long long cap, int32_t* counts, int32_t* offsets, int32_t* sorted_tok,
                                    float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs, int32_t* P_out,
                                    const PermuteWs& w, int* err, unsigned long long timeout_ns, cudaStream_t s) {
  const int tb = perm_tok_block(T, E);
  const int nb = (T + tb - 1) / tb;
  const size_t bits_smem = static_cast<size_t>(E) * (tb / 32) * sizeof(uint32_t);
  const long long plain_cap = static_cast<long long>(T) * K;
  cudaError_t st;
  // plain grouping of the top-K pairs with their probabilities (into the workspace)
  if ((st = group_pairs<false>(tb, nb, bits_smem, topk_ids, topk_w, nullptr, nullptr, T, E, K, w, w.plain_cnt,
                               w.plain_off, nullptr, plain_cap, w.plain_tok, w.scoresT, nullptr, nullptr, err, 0,
                               timeout_ns, s)) != cudaSuccess)
    return st;
  // kept pairs
  const size_t mbytes = sizeof(uint32_t) * static_cast<size_t>(T) * ((E + 31) / 32);
  if ((st = cudaMemsetAsync(w.member, 0, mbytes, s)) != cudaSuccess) return st;
  const size_t sel_smem = sizeof(uint32_t) * kTrListCap;
  st = cudaFuncSetAttribute(cap_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                            static_cast<int>(sizeof(uint32_t) * kTrListCap));
  if (st != cudaSuccess) return st;
  cap_select_kernel<<<E, kTrThreads, sel_smem, s>>>(w.plain_off, w.plain_tok, w.scoresT, plain_cap, T, E, C, policy,
                                                    w.member, err);
  // group the kept pairs into slots e C + (rank in token order); empty slots hold token -1, weight 0
  const size_t slots = static_cast<size_t>(E) * C;
  if ((st = cudaMemsetAsync(sorted_tok, 0xFF, sizeof(int32_t) * slots, s)) != cudaSuccess) return st;
  if ((st = cudaMemsetAsync(sorted_w, 0, sizeof(float) * slots, s)) != cudaSuccess) return st;
  if ((st = group_pairs<true>(tb, nb, bits_smem, topk_ids, topk_w, w.member, nullptr, T, E, K, w, counts, offsets,
                              nullptr, cap, sorted_tok, sorted_w, tok_ptr, tok_pairs, err, C, timeout_ns, s)) !=
      cudaSuccess)
    return st;
  slot_offsets_kernel<<<1, 256, 0, s>>>(offsets, E, C, P_out);
  return cudaGetLastError();
}

}  // namespace vgg

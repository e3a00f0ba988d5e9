// Memory-bound per-token kernels: the weighted combine of the forward, the
// per-token part of the backward (dS reduction, router-logit gradient, dX
// K-reduction), and two small helpers (transpose, split-K reduction).
//
// [EP] "여러 Expert의 결과도 같은 토큰으로 돌아오기": a token's expert outputs are
// summed back into the token's own slot with the combine weights.
// [DEP] "3) Combine": weighted sum of the k expert outputs per token.
// [SM] "7 한계 & 의의": the per-pair output Y is materialised and reduced
// without float atomics, for determinism and precision.
//
// The combine is one CTA per token, the per-token backward one warp per token; a token's pairs are
// visited in ascending expert order (tok_pairs), 16-byte vector loads per thread, fp32 accumulation.
#include "internal.h"

namespace vgg {

constexpr int kCombineThreads = 128;
constexpr int kMaxTokPairs = 64;

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], uint4 q) {
  float2 a = unpack_bf16x2(q.x), b = unpack_bf16x2(q.y), c = unpack_bf16x2(q.z), d = unpack_bf16x2(q.w);
  acc[0] += a.x; acc[1] += a.y; acc[2] += b.x; acc[3] += b.y;
  acc[4] += c.x; acc[5] += c.y; acc[6] += d.x; acc[7] += d.y;
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  return o;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __nv_bfloat16* __restrict__ Y,
                                                                  const int32_t* __restrict__ tok_ptr,
                                                                  const int32_t* __restrict__ tok_pairs, int T, int d,
                                                                  long long cap, __nv_bfloat16* __restrict__ O,
                                                                  int* err) {
  __shared__ int s_j[kMaxTokPairs];
  __shared__ int s_cnt;
  const int t = blockIdx.x;
  if (threadIdx.x == 0) {
    const long long p0 = tok_ptr[t], p1 = tok_ptr[t + 1];
    int cnt = static_cast<int>(p1 - p0);
    if (p0 < 0 || p1 > cap || cnt < 0 || cnt > kMaxTokPairs) {
      set_error(err, p1 > cap || p0 < 0 || cnt < 0 ? DERR_BAD_OFFSETS : DERR_CAPACITY);
      cnt = 0;
    }
    s_cnt = cnt;
  }
  __syncthreads();
  const int cnt = s_cnt;
  const long long p0 = tok_ptr[t];
  for (int r = threadIdx.x; r < cnt; r += kCombineThreads) {
    int j = tok_pairs[p0 + r];
    if (j < 0 || j >= cap) {
      set_error(err, DERR_BAD_OFFSETS);
      j = -1;
    }
    s_j[r] = j;
  }
  __syncthreads();
  const int nv = d >> 3;
  for (int c = threadIdx.x; c < nv; c += kCombineThreads) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int r = 0;
    for (; r + 4 <= cnt; r += 4) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = s_j[r + u];
        q[u] = j >= 0 ? ldg_nc_v4(Y + static_cast<long long>(j) * d + 8 * c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) add_bf16x8(acc, q[u]);
    }
    for (; r < cnt; ++r) {
      const int j = s_j[r];
      if (j >= 0) add_bf16x8(acc, ldg_nc_v4(Y + static_cast<long long>(j) * d + 8 * c));
    }
    *reinterpret_cast<uint4*>(O + static_cast<long long>(t) * d + 8 * c) = pack8(acc);
  }
}

cudaError_t launch_combine(const __nv_bfloat16* Y, const int32_t* tok_ptr, const int32_t* tok_pairs, int T, int d,
                           long long cap, __nv_bfloat16* O, int* err, cudaStream_t s) {
  if (T > 0) combine_kernel<<<T, kCombineThreads, 0, s>>>(Y, tok_ptr, tok_pairs, T, d, cap, O, err);
  return cudaGetLastError();
}

// out[c][r] = in[r][c], bf16, 32x32 tiles through shared memory.
__global__ void transpose_bf16_kernel(const __nv_bfloat16* __restrict__ in, int rows, int cols,
                                      __nv_bfloat16* __restrict__ out) {
  __shared__ __nv_bfloat16 tile[32][33];
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

cudaError_t launch_transpose_bf16(const __nv_bfloat16* in, int rows, int cols, __nv_bfloat16* out, cudaStream_t s) {
  dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
  transpose_bf16_kernel<<<grid, block, 0, s>>>(in, rows, cols, out);
  return cudaGetLastError();
}

// Per token t (one warp; 8 tokens per CTA):
//   dS[j]       = sum over column tiles of the dSwiGLU epilogue's partial <dA'_j, A_j>
//   dlogits[t]  = [k in F(t)] w_k dS_k - [k in TopK(t)] w_k * sum_{i in F(t)} w_i dS_i
//   dX[t]       = sum_j dXp[j] (ascending expert) + sum_e dlogits[t,e] W_r[:,e]
// The CTA stages the group offsets in shared memory once (the expert of a pair is a binary search
// there); each warp keeps its token's dlogits row in shared memory, so the only CTA-wide barrier is the
// one after the offsets.
constexpr int kTbWarps = 8;
constexpr int kTbNz = kMaxTokPairs + 8;  // nonzero dlogits of a token: its pairs' experts and its top-K

// Expert of sorted pair j: the e with off[e] <= j < off[e+1].
__device__ __forceinline__ int expert_of_smem(const int* off, int E, int j) {
  int lo = 0, hi = E;  // invariant: off[lo] <= j < off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= j) lo = mid;
    else hi = mid;
  }
  return lo;
}

size_t token_backward_smem(int E) {
  return sizeof(float) * kTbWarps * E + sizeof(int) * (E + 1) +
         kTbWarps * (sizeof(int) * kMaxTokPairs + (sizeof(int) + sizeof(float)) * kTbNz);
}

__global__ void __launch_bounds__(256) token_backward_kernel(
    const float* __restrict__ part, int part_ld, const int32_t* __restrict__ tok_ptr,
    const int32_t* __restrict__ tok_pairs, const int32_t* __restrict__ offsets, int E,
    const float* __restrict__ sorted_w, const int32_t* __restrict__ topk_ids, const float* __restrict__ topk_w, int K,
    const __nv_bfloat16* __restrict__ dXp, const __nv_bfloat16* __restrict__ WrT, int T, int d, long long cap,
    float* __restrict__ dS, float* __restrict__ dlogits, __nv_bfloat16* __restrict__ dL_bf16,
    __nv_bfloat16* __restrict__ dL_lo, __nv_bfloat16* __restrict__ dX, int* err) {
  extern __shared__ __align__(16) uint8_t tb_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* s_dl = reinterpret_cast<float*>(tb_smem) + warp * E;
  int* s_off = reinterpret_cast<int*>(tb_smem + sizeof(float) * kTbWarps * E);
  int* s_j = s_off + (E + 1) + warp * kMaxTokPairs;
  int* s_nz_e = s_off + (E + 1) + kTbWarps * kMaxTokPairs + warp * kTbNz;
  float* s_nz_v = reinterpret_cast<float*>(s_off + (E + 1) + kTbWarps * (kMaxTokPairs + kTbNz)) + warp * kTbNz;
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = __ldg(offsets + i);
  __syncthreads();
  const int t = blockIdx.x * kTbWarps + warp;
  if (t >= T) return;
  const long long p0 = __ldg(tok_ptr + t), p1 = __ldg(tok_ptr + t + 1);
  int cnt = static_cast<int>(p1 - p0);
  if (p0 < 0 || p1 > cap || cnt < 0 || cnt > kMaxTokPairs) {
    if (lane == 0) set_error(err, DERR_BAD_OFFSETS);
    cnt = 0;
  }
  for (int e = lane; e < E; e += 32) s_dl[e] = 0.0f;
  __syncwarp();
  float g = 0.0f;
  for (int r = lane; r < cnt; r += 32) {
    const int j = __ldg(tok_pairs + p0 + r);
    if (j < 0 || j >= cap) {
      set_error(err, DERR_BAD_OFFSETS);
      s_j[r] = -1;
      continue;
    }
    s_j[r] = j;
    float ds = 0.0f;
    for (int q = 0; q < part_ld; ++q) ds += __ldg(part + static_cast<long long>(j) * part_ld + q);
    dS[j] = ds;
    const float c = __ldg(sorted_w + j) * ds;
    s_dl[expert_of_smem(s_off, E, j)] += c;  // the experts of one token are distinct
    g += c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
  __syncwarp();
  if (lane < K) {
    const int e = __ldg(topk_ids + static_cast<long long>(t) * K + lane);
    if (e >= 0 && e < E) s_dl[e] -= __ldg(topk_w + static_cast<long long>(t) * K + lane) * g;
  }
  __syncwarp();
  int nnz = 0;
  const long long rowE = static_cast<long long>(t) * E;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    const float v = e < E ? s_dl[e] : 0.0f;
    if (e < E) {
      dlogits[rowE + e] = v;
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      dL_bf16[rowE + e] = hi;
      dL_lo[rowE + e] = __float2bfloat16_rn(v - __bfloat162float(hi));
    }
    const unsigned m = __ballot_sync(0xffffffffu, v != 0.0f);
    if (v != 0.0f) {
      const int pos = nnz + __popc(m & ((1u << lane) - 1u));
      if (pos < kTbNz) {
        s_nz_e[pos] = e;
        s_nz_v[pos] = v;
      }
    }
    nnz += __popc(m);
  }
  if (nnz > kTbNz) {  // cannot happen: the nonzeros are the token's pair experts and its top-K
    if (lane == 0) set_error(err, DERR_BAD_OFFSETS);
    nnz = kTbNz;
  }
  __syncwarp();
  const int nv = d >> 3;
  // Per 8 columns: the pair rows in batches of eight loads in flight (one memory round trip for a token
  // of up to eight pairs), added in pair order; then the router part, eight W_r^T rows (L2-resident) per
  // round trip, in nonzero order.
  constexpr int kB = 8;
  for (int c = lane; c < nv; c += 32) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int r0 = 0; r0 < cnt; r0 += kB) {
      uint4 q[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int j = r0 + u < cnt ? s_j[r0 + u] : -1;
        q[u] = j >= 0 ? ldg_nc_v4(dXp + static_cast<long long>(j) * d + 8 * c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kB; ++u)
        if (r0 + u < cnt && s_j[r0 + u] >= 0) add_bf16x8(acc, q[u]);
    }
    for (int i0 = 0; i0 < nnz; i0 += kB) {
      uint4 q[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u)
        q[u] = i0 + u < nnz ? *reinterpret_cast<const uint4*>(WrT + static_cast<long long>(s_nz_e[i0 + u]) * d + 8 * c)
                            : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        if (i0 + u >= nnz) break;
        const float v = s_nz_v[i0 + u];
        const float2 a = unpack_bf16x2(q[u].x), b = unpack_bf16x2(q[u].y), cc = unpack_bf16x2(q[u].z),
                     dd = unpack_bf16x2(q[u].w);
        acc[0] += v * a.x; acc[1] += v * a.y; acc[2] += v * b.x; acc[3] += v * b.y;
        acc[4] += v * cc.x; acc[5] += v * cc.y; acc[6] += v * dd.x; acc[7] += v * dd.y;
      }
    }
    *reinterpret_cast<uint4*>(dX + static_cast<long long>(t) * d + 8 * c) = pack8(acc);
  }
}

cudaError_t launch_token_backward(const float* part, int part_ld, const int32_t* tok_ptr, const int32_t* tok_pairs,
                                  const int32_t* offsets, int E, const float* sorted_w, const int32_t* topk_ids,
                                  const float* topk_w, int K, const __nv_bfloat16* dXp, const __nv_bfloat16* WrT,
                                  int T, int d, long long cap, float* dS, float* dlogits, __nv_bfloat16* dL_bf16,
                                  __nv_bfloat16* dL_lo, __nv_bfloat16* dX, int* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const size_t smem = token_backward_smem(E);
  cudaError_t e = cudaFuncSetAttribute(token_backward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  token_backward_kernel<<<(T + kTbWarps - 1) / kTbWarps, 32 * kTbWarps, smem, s>>>(
      part, part_ld, tok_ptr, tok_pairs, offsets, E, sorted_w, topk_ids, topk_w, K, dXp, WrT, T, d, cap, dS, dlogits,
      dL_bf16, dL_lo, dX, err);
  return cudaGetLastError();
}

// out[i] = sum_s part[s][i], s ascending.
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, long long n,
                                     float* __restrict__ out) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float a = 0.0f;
    for (int s = 0; s < splits; ++s) a += part[s * n + i];
    out[i] = a;
  }
}

cudaError_t launch_splitk_reduce(const float* part, int splits, long long n, float* out, cudaStream_t s) {
  const long long want = (n + 255) / 256;
  const int blocks = static_cast<int>(want < 4096 ? want : 4096);
  if (n > 0) splitk_reduce_kernel<<<blocks, 256, 0, s>>>(part, splits, n, out);
  return cudaGetLastError();
}

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait gives up,
// records the timeout code and the kernel returns normally.
__global__ void wait_timeout_probe_kernel(int* err, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, timeout_ns, err);
  __syncthreads();
}

cudaError_t launch_wait_timeout_probe(int* err, unsigned long long timeout_ns, cudaStream_t s) {
  wait_timeout_probe_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace vgg

namespace vgg {

// Rows [offsets[E], cap) of the backward's per-pair buffers are never written by the GEMMs.  The varlen-K
// weight-gradient GEMM multiplies the rows of its last expert's last 16-row UMMA K step, up to 15 rows past
// offsets[E], by zero rows of B, so those must hold finite values: zero them (rows further on are loaded into
// shared memory with the stage but never multiplied; the varlen-M GEMMs drop the accumulator rows they touch).
struct TailBufs {
  __nv_bfloat16* p[6];
};

__global__ void zero_tail_rows_kernel(const int32_t* __restrict__ offsets, int E, long long cap, int cols,
                                      TailBufs bufs) {
  const long long P = offsets[E];
  if (P < 0 || P >= cap) return;
  const long long n = min(cap - P, 16ll) * cols / 8;  // 16-byte vectors per buffer
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long off = P * cols + 8 * i;
#pragma unroll
    for (int k = 0; k < 6; ++k)
      if (bufs.p[k]) *reinterpret_cast<uint4*>(bufs.p[k] + off) = z;
  }
}

cudaError_t launch_zero_tail_rows(const int32_t* offsets, int E, long long cap, int cols,
                                  __nv_bfloat16* const (&bufs)[6], cudaStream_t s) {
  TailBufs b;
  for (int k = 0; k < 6; ++k) b.p[k] = bufs[k];
  zero_tail_rows_kernel<<<8, 256, 0, s>>>(offsets, E, cap, cols, b);
  return cudaGetLastError();
}

}  // namespace vgg

namespace vgg {

// out_a[j'] = a[sorted_tok[j]], out_b[j'] = b[sorted_tok[j]] for the sorted positions j of the pairs, zero
// rows elsewhere: the backward's expert-sorted copies of X and dO, read by TMA boxes in the weight-gradient
// and dA' GEMMs.  With poff the copies are padded per group (j' = j + poff[g] - offsets[g], cap_pad rows):
// every group's rows are followed by zero rows up to a multiple of 16, so a varlen-K GEMM's last UMMA K step
// reads zeros past the group's end; rows past poff[E] are left unwritten.  Without poff j' = j (cap rows).  Token-major with bulk (TMA) transfers: lane 0 of each warp reads
// token t's rows of a and b once (chunks of up to 4 KB, global -> shared) and writes them to the sorted
// positions of all of t's pairs (tok_pairs), so a and b stream from memory once instead of once per
// pair (row-major gathers re-read them from DRAM when they do not fit in L2).  Positions that hold no
// pair (the tail [P, cap) and the empty slots of the capacity layout) are then written from a zeroed
// chunk.  One token in flight per warp, three CTAs per SM.
//
// CODES: a third source travels with b, the tokens' e4m3 code rows c ([T, d] bytes) and their scales cs
// ([T]): out_c[j] = c[sorted_tok[j]], out_cs[j] = cs[sorted_tok[j]]; positions without a pair get zero
// codes and scale 1 (a zero row's quantization).  A third buffer per warp: two CTAs per SM.
constexpr int kGrWarps = 8;
static_assert(kMaxTokPairs <= 64, "gather_rows: at most two pair positions per lane");
constexpr int kGrChunk = 2048;  // bf16 elements per bulk copy

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}

// The group of sorted position j: the largest g with off[g] <= j (empty groups skipped), 0 <= g < E.
__device__ __forceinline__ int group_of(const int32_t* __restrict__ off, int E, long long j) {
  int lo = 0, hi = E;  // off[lo] <= j < off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(off + mid) <= j) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Padded group offsets: poff[g] = sum over earlier groups of their row counts rounded up to 16 (poff[E] =
// the padded total).  One block.
__global__ void __launch_bounds__(1024) pad_offsets_kernel(const int32_t* __restrict__ off, int E,
                                                           int32_t* __restrict__ poff, int* err) {
  __shared__ int wsum[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < E; base += 1024) {
    const int g = base + tid;
    int r = 0;
    if (g < E) {
      r = __ldg(off + g + 1) - __ldg(off + g);
      if (r < 0) {
        set_error(err, DERR_BAD_OFFSETS);
        r = 0;
      }
      r = (r + 15) & ~15;
    }
    int incl = r;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = wsum[lane], wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      wsum[lane] = wi - w;  // exclusive prefix of the warps
    }
    __syncthreads();
    const int excl = carry + wsum[warp] + incl - r;
    if (g < E) poff[g] = excl;
    __syncthreads();
    if (tid == 1023 || g == E - 1) carry = excl + r;
    __syncthreads();
  }
  if (tid == 0) poff[E] = carry;
}

cudaError_t launch_pad_offsets(const int32_t* offsets, int E, int32_t* poff, int* err, cudaStream_t s) {
  pad_offsets_kernel<<<1, 1024, 0, s>>>(offsets, E, poff, err);
  return cudaGetLastError();
}

template <bool CODES>
__global__ void __launch_bounds__(kGrWarps * 32) gather_rows_bulk_kernel(
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ poff, long long cap_pad, int E,
    const int32_t* __restrict__ sorted_tok,
    const int32_t* __restrict__ tok_ptr, const int32_t* __restrict__ tok_pairs, long long cap, int T, int d,
    const __nv_bfloat16* __restrict__ a, const __nv_bfloat16* __restrict__ b, __nv_bfloat16* __restrict__ out_a,
    __nv_bfloat16* __restrict__ out_b, const uint8_t* __restrict__ c, const float* __restrict__ cs,
    uint8_t* __restrict__ out_c, float* __restrict__ out_cs, int* err, unsigned long long timeout_ns) {
  extern __shared__ __align__(128) uint8_t gr_smem[];  // zero chunk, then per warp two chunks (+ a code chunk)
  __shared__ uint64_t bars[kGrWarps];
  __shared__ int abort_flag;
  constexpr uint32_t kChunkBytes = kGrChunk * 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < static_cast<int>(kChunkBytes / 16); i += blockDim.x)
    reinterpret_cast<uint4*>(gr_smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int w = 0; w < kGrWarps; ++w) mbar_init(&bars[w], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();  // the zero chunk is read by bulk stores
  __syncthreads();
  // A warp takes one token at a time: lane 0 loads the token's rows (one bulk copy per tensor and chunk)
  // and every lane stores them to one (or two) of the token's pair positions, so the stores of a token
  // are issued in parallel and the position lookups overlap the load.
  constexpr uint32_t kWarpBytes = 2 * kChunkBytes + (CODES ? kGrChunk : 0);
  const bool bf = out_a != nullptr;  // the bf16 copies (without them: the code rows alone)
  const uint32_t zero = smem_u32(gr_smem);
  const uint32_t buf = zero + kChunkBytes + kWarpBytes * warp;
  const long long P = offsets[E];
  const long long gw = static_cast<long long>(blockIdx.x) * kGrWarps + warp;
  const long long nw = static_cast<long long>(gridDim.x) * kGrWarps;
  uint32_t phase = 0;
  bool ok = true;
  for (long long t = gw; t < T && ok; t += nw) {
    const long long q0 = __ldg(tok_ptr + t), q1 = __ldg(tok_ptr + t + 1);
    if (q0 < 0 || q1 > cap || q1 < q0 || q1 - q0 > kMaxTokPairs) {
      if (lane == 0) set_error(err, DERR_BAD_OFFSETS);
      continue;
    }
    const int cnt = static_cast<int>(q1 - q0);
    if (cnt == 0) continue;
    // lane 0 issues chunk c0's loads of the token's rows into the warp's buffer
    auto load_chunk = [&](int c0) {
      const uint32_t bytes = 2u * static_cast<uint32_t>(min(kGrChunk, d - c0));
      bulk_wait_read<0>();  // this lane's previous stores have read the warp's buffer
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[warp], (bf ? 2 * bytes : 0) + (CODES ? bytes / 2 : 0));
        if (bf) {
          bulk_g2s(buf, a + t * d + c0, bytes, &bars[warp]);
          bulk_g2s(buf + kChunkBytes, b + t * d + c0, bytes, &bars[warp]);
        }
        if (CODES) bulk_g2s(buf + 2 * kChunkBytes, c + t * d + c0, bytes / 2, &bars[warp]);
      }
    };
    load_chunk(0);
    // the pair positions (and their rows in the padded copies) are looked up while the first chunk loads
    long long jl[2] = {-1, -1}, jp[2] = {-1, -1};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = lane + 32 * h;
      if (r < cnt) {
        const long long j = __ldg(tok_pairs + q0 + r);
        if (j < 0 || j >= cap || (poff && j >= P)) {
          set_error(err, DERR_BAD_OFFSETS);
        } else {
          jl[h] = j;
          if (poff) {
            const int g = group_of(offsets, E, j);
            jp[h] = j + (__ldg(poff + g) - __ldg(offsets + g));
          } else {
            jp[h] = j;
          }
        }
      }
    }
    if (CODES && cs) {  // per-row scales (the block-scaled form takes its scales elsewhere: cs == nullptr)
      const float sc = __ldg(cs + t);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if (jl[h] >= 0) out_cs[jl[h]] = sc;
    }
    for (int c0 = 0; c0 < d; c0 += kGrChunk) {
      const uint32_t bytes = 2u * static_cast<uint32_t>(min(kGrChunk, d - c0));
      if (c0 > 0) load_chunk(c0);
      const int landed = mbar_wait(&bars[warp], phase, &abort_flag, timeout_ns, err) ? 1 : 0;
      if (!__all_sync(0xffffffffu, landed)) {
        ok = false;
        break;
      }
      phase ^= 1u;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (jl[h] >= 0) {
          if (bf) {
            bulk_s2g(out_a + jp[h] * d + c0, buf, bytes);
            bulk_s2g(out_b + jp[h] * d + c0, buf + kChunkBytes, bytes);
          }
          if (CODES) bulk_s2g(out_c + jl[h] * d + c0, buf + 2 * kChunkBytes, bytes / 2);
        }
      }
      bulk_commit();
    }
  }
  // rows without a pair: the tail and the empty slots of the capacity layout, and with the padded layout the
  // rows that round every group up to a multiple of 16
  auto zero_row = [&](long long q) {
    for (int c0 = 0; c0 < d; c0 += kGrChunk) {
      const uint32_t bytes = 2u * static_cast<uint32_t>(min(kGrChunk, d - c0));
      bulk_s2g(out_a + q * d + c0, zero, bytes);
      bulk_s2g(out_b + q * d + c0, zero, bytes);
    }
    bulk_commit();
  };
  if (!bf) {
  } else if (poff) {
    // empty slots of the capacity layout (rare), then the padding rows of every group: at most 15 per group,
    // one per thread.  Rows past the padded total are never read (a group's last UMMA K step ends on its
    // padded boundary) and stay unwritten.
    const long long tid = gw * 32 + lane, nt = nw * 32;
    for (long long j = tid; j < P && ok; j += nt) {
      if (sorted_tok[j] >= 0) continue;
      const int g = group_of(offsets, E, j);
      zero_row(j + (__ldg(poff + g) - __ldg(offsets + g)));
    }
    for (long long k = tid; k < 15ll * E && ok; k += nt) {
      const int g = static_cast<int>(k / 15), i = static_cast<int>(k % 15);
      const long long row = __ldg(poff + g) + (__ldg(offsets + g + 1) - __ldg(offsets + g)) + i;
      if (row < __ldg(poff + g + 1)) zero_row(row);
    }
  } else {
    for (long long j = gw * 32 + lane; j < cap && ok; j += nw * 32)
      if (j >= P || sorted_tok[j] < 0) zero_row(j);
  }
  // the code rows keep the unpadded layout
  if (CODES) {
    for (long long j = gw * 32 + lane; j < cap && ok; j += nw * 32) {
      if (j < P && sorted_tok[j] >= 0) continue;
      if (out_cs) out_cs[j] = 1.0f;
      for (int c0 = 0; c0 < d; c0 += kGrChunk) {
        const uint32_t bytes = 2u * static_cast<uint32_t>(min(kGrChunk, d - c0));
        bulk_s2g(out_c + j * d + c0, zero, bytes / 2);
      }
      bulk_commit();
    }
  }
  if (!ok && lane == 0) {  // a load that never completed: let copies in flight land before leaving
    volatile int never = 0;
    mbar_wait(&bars[warp], phase, &never, 20000000ull, nullptr);
  }
  bulk_wait0();
}

cudaError_t launch_gather_rows(const int32_t* offsets, const int32_t* poff, long long cap_pad, int E,
                               const int32_t* sorted_tok, const int32_t* tok_ptr,
                               const int32_t* tok_pairs, long long cap, int T, int d, const __nv_bfloat16* a,
                               const __nv_bfloat16* b, __nv_bfloat16* out_a, __nv_bfloat16* out_b,
                               const uint8_t* c, const float* cs, uint8_t* out_c, float* out_cs, int* err,
                               int num_sms, unsigned long long timeout_ns, cudaStream_t s) {
  const bool codes = c != nullptr;
  if (!out_a && !codes) return cudaErrorInvalidValue;  // nothing to copy
  const size_t smem = static_cast<size_t>(kGrChunk) * (2 + kGrWarps * (codes ? 5 : 4));
  const void* fn = codes ? reinterpret_cast<const void*>(gather_rows_bulk_kernel<true>)
                         : reinterpret_cast<const void*>(gather_rows_bulk_kernel<false>);
  cudaError_t st = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (st != cudaSuccess) return st;
  const long long want = (T + kGrWarps - 1) / kGrWarps;
  const long long per_sm = codes ? 2 : 3;
  const int blocks = static_cast<int>(want < per_sm * num_sms ? want : per_sm * num_sms);
  if (blocks > 0) {
    if (codes)
      gather_rows_bulk_kernel<true><<<blocks, kGrWarps * 32, smem, s>>>(
          offsets, poff, cap_pad, E, sorted_tok, tok_ptr, tok_pairs, cap, T, d, a, b, out_a, out_b, c, cs, out_c, out_cs, err,
          timeout_ns);
    else
      gather_rows_bulk_kernel<false><<<blocks, kGrWarps * 32, smem, s>>>(
          offsets, poff, cap_pad, E, sorted_tok, tok_ptr, tok_pairs, cap, T, d, a, b, out_a, out_b, nullptr, nullptr, nullptr,
          nullptr, err, timeout_ns);
  }
  return cudaGetLastError();
}

}  // namespace vgg

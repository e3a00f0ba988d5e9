// Block-scaled e4m3 form of the forward: 1 x 32 blocks along the reduction dimension, one power-of-two
// scale (UE8M0 byte) per block, the kind::mxf8f6f4 UMMA applying both operands' scales block by block.
// [GG] "한계": the fine-grained FP8 grouped GEMM credited there with a further 2x over bf16.
//
// Block rule: e = the smallest integer with max|block| <= 448 2^e (in [-127, 127]; 0 for an all-zero
// block), codes = e4m3(x 2^-e) rounded to nearest even; the scaling is exact and no code saturates.
//
// Scale layouts:
//   row-major  [rows][4 ceil(cols / 128)] bytes (the per-token X scales, gathered by the GEMM 4 bytes per row
//              and stage); entries past cols / 32 hold 127 (scale 1);
//   blocks     512 bytes per 128 operand rows and 128 codes of K, the layout tcgen05.cp reads: row r, 32-code
//              block k at byte (r % 32) 16 + (r / 32) 4 + k.  The weights' blocks follow the GEMMs' 192-column
//              tiles, two blocks (1024 bytes) per tile and stage: W_gate / W_up [E][ceil(n / 96)][ceil(d / 128)],
//              tile rows 0..95 = W_gate rows 96 t.., rows 96..191 = W_up rows 96 t.. (one gate/up column tile);
//              W_down [E][ceil(d / BN)][ceil(n / 128)], tile rows = W_down rows BN t.. (BN = mx_tile_cols(d):
//              192, or 128 with one block per tile and stage); the activations A
//              (written by the SwiGLU epilogue): one block per row tile and stage, [row tile][ceil(n / 128)].
//              Entries with no operand row or past K hold 127.
#include "internal.h"

namespace vgg {

// One warp per row, one lane per 32-element block (64-byte loads, 32-byte code stores).
__global__ void __launch_bounds__(256) quantize_rows_mx_kernel(const __nv_bfloat16* __restrict__ M, long long rows,
                                                               const int32_t* __restrict__ rows_limit, int cols,
                                                               uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                               int sf_ld) {
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows || (rows_limit && r >= __ldg(rows_limit))) return;
  const int nb = cols / 32;
  for (int b = lane; b < sf_ld; b += 32) {
    if (b >= nb) {
      sf[r * sf_ld + b] = 127;
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(M + r * cols + 32 * b);
    float v[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 x = __ldg(src + j);
      const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack_bf16x2(wv[i]);
        v[8 * j + 2 * i] = f.x;
        v[8 * j + 2 * i + 1] = f.y;
      }
    }
    uint32_t w[8];
    const int e = mx_block32(v, w);
    uint4* dst = reinterpret_cast<uint4*>(q + r * cols + 32 * b);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    sf[r * sf_ld + b] = static_cast<uint8_t>(e + 127);
  }
}

cudaError_t launch_quantize_rows_mx(const __nv_bfloat16* M, long long rows, const int32_t* rows_limit, int cols,
                                    uint8_t* q, uint8_t* sf, int sf_ld, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;
  quantize_rows_mx_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(M, rows, rows_limit, cols, q, sf, sf_ld);
  return cudaGetLastError();
}

// Weights [E][R][C]: codes in place of the values, scales into [E][ntile][kst] groups of nblk 512-byte blocks in
// which operand row `row` is tile row roff + row % rpt (block (tile row) / 128) of column tile row / rpt (the
// block buffer is set to 127 first).
__global__ void __launch_bounds__(256) quantize_weight_mx_kernel(const __nv_bfloat16* __restrict__ W, int E, int R,
                                                                 int C, uint8_t* __restrict__ q,
                                                                 uint8_t* __restrict__ blocks, int rpt, int roff,
                                                                 int ntile, int kst, int nblk) {
  const long long wr = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // e * R + row
  const int lane = threadIdx.x & 31;
  if (wr >= static_cast<long long>(E) * R) return;
  const int e = static_cast<int>(wr / R), row = static_cast<int>(wr % R);
  const int t = row / rpt, tr = roff + row % rpt, br = tr & 127;
  uint8_t* blk = blocks + (static_cast<long long>(e) * ntile + t) * kst * (512ll * nblk) + (tr >> 7) * 512 +
                 (br & 31) * 16 + (br >> 5) * 4;
  for (int b = lane; b < C / 32; b += 32) {
    const uint4* src = reinterpret_cast<const uint4*>(W + wr * C + 32 * b);
    float v[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 x = __ldg(src + j);
      const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack_bf16x2(wv[i]);
        v[8 * j + 2 * i] = f.x;
        v[8 * j + 2 * i + 1] = f.y;
      }
    }
    uint32_t w[8];
    const int ex = mx_block32(v, w);
    uint4* dst = reinterpret_cast<uint4*>(q + wr * C + 32 * b);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    blk[(b >> 2) * (512ll * nblk) + (b & 3)] = static_cast<uint8_t>(ex + 127);
  }
}

cudaError_t launch_quantize_weight_mx(const __nv_bfloat16* W, int E, int R, int C, uint8_t* q, uint8_t* blocks,
                                      int rpt, int roff, int ntile, int kst, int nblk, cudaStream_t s) {
  const long long warps = static_cast<long long>(E) * R;
  if (warps <= 0) return cudaSuccess;
  quantize_weight_mx_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, s>>>(W, E, R, C, q, blocks, rpt, roff,
                                                                                 ntile, kst, nblk);
  return cudaGetLastError();
}

// The scale blocks of a gathered operand, in the varlen-M GEMMs' row-tile order: for every row tile of every
// group (tiles of 128 sorted rows, groups in order) and stage of K, the 512-byte block whose row r holds the 4
// scale bytes of sorted row off[g] + 128 m + r, taken from the source row idx[that row] of the row-major
// [rows][sf_ld] scales (zeros for a row past the group's end or without a source row).  One block per row tile:
// warp 0 finds the tile's group from a prefix of the groups' tile counts, then thread t copies the words of row
// t % 128 for the stages k = t / 128, t / 128 + 2, ...
__global__ void __launch_bounds__(256) mx_tile_scales_kernel(const uint8_t* __restrict__ sf, int sf_ld, int src_rows,
                                                             const int32_t* __restrict__ idx, int idx_rows,
                                                             const int32_t* __restrict__ off, int G, int kst,
                                                             uint8_t* __restrict__ blocks) {
  __shared__ int s_row0, s_end;
  const long long tile = blockIdx.x;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int running = 0, row0 = -1, end = 0;
    for (int base = 0; base < G && row0 < 0; base += 32) {
      const int g = base + lane;
      const int o = g < G ? __ldg(off + g) : 0, o1 = g < G ? __ldg(off + g + 1) : 0;
      const int cnt = g < G ? (o1 - o + 127) / 128 : 0;
      int incl = cnt;
#pragma unroll
      for (int k = 1; k < 32; k <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, k);
        if (lane >= k) incl += y;
      }
      const int first = running + incl - cnt;
      const unsigned hit = __ballot_sync(0xffffffffu, g < G && tile >= first && tile < first + cnt);
      if (hit) {
        const int src = __ffs(hit) - 1;
        row0 = __shfl_sync(0xffffffffu, o + static_cast<int>(tile - first) * 128, src);
        end = __shfl_sync(0xffffffffu, o1, src);
      }
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s_row0 = row0;
      s_end = end;
    }
  }
  __syncthreads();
  if (s_row0 < 0) return;  // past the last tile
  const int r = threadIdx.x & 127;
  const int row = s_row0 + r;
  const int src = (row < s_end && row < idx_rows) ? __ldg(idx + row) : -1;
  const bool ok = src >= 0 && src < src_rows;
  uint8_t* dst = blocks + tile * kst * 512ll + (r & 31) * 16 + (r >> 5) * 4;
  const uint32_t* srow = reinterpret_cast<const uint32_t*>(sf + static_cast<long long>(ok ? src : 0) * sf_ld);
  for (int k = threadIdx.x >> 7; k < kst; k += 2)
    *reinterpret_cast<uint32_t*>(dst + k * 512ll) = ok ? __ldg(srow + k) : 0u;
}

cudaError_t launch_mx_tile_scales(const uint8_t* sf, int sf_ld, int src_rows, const int32_t* idx, int idx_rows,
                                  const int32_t* off, int G, int kst, long long tiles_cap, uint8_t* blocks,
                                  cudaStream_t s) {
  if (tiles_cap <= 0 || G <= 0) return cudaSuccess;
  mx_tile_scales_kernel<<<static_cast<unsigned>(tiles_cap), 256, 0, s>>>(sf, sf_ld, src_rows, idx, idx_rows, off, G,
                                                                         kst, blocks);
  return cudaGetLastError();
}

// Gate/up + SwiGLU on block-scaled operands: gathered X codes (scales gathered 4 bytes per row and stage), the
// W_gate / W_up pair, 96 + 96 output columns per tile (two 192-column accumulators and four stages of scales
// fill 432 of the 512 TMEM columns); the epilogue writes H, U (fp32, when cached) and A as block-scaled codes
// with their scale blocks.
cudaError_t run_gate_up_swiglu_mx(int cn, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (cn == 2)
    return launch_grouped_gemm<kMxBN, 4, 4, 1, A_GATHER_K, B_TMA_K3_GU, VAR_M, EPI_SWIGLU, false, 2, X_MX>(p, m, grid, s);
  return launch_grouped_gemm<kMxBN, 4, 4, 1, A_GATHER_K, B_TMA_K3_GU, VAR_M, EPI_SWIGLU, false, 1, X_MX>(p, m, grid, s);
}

// Down projection on block-scaled A (rows of the SwiGLU epilogue's codes, scale blocks per row tile) and
// W_down, BN = mx_tile_cols(d) output columns per tile; the epilogue scales each row by its combine weight (Yw,
// bf16).
cudaError_t run_down_scale_mx(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 128)
    return launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_SCALE, false, 1, X_MX>(p, m, grid, s);
  return launch_grouped_gemm<kMxBN, 4, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_SCALE, false, 1, X_MX>(p, m, grid, s);
}

// The backward's dSwiGLU GEMM on block-scaled operands: A = the sorted dO code rows (TMA), B = W_down^T [E][n][d]
// codes; the dSwiGLU epilogue (dS partials, dH, dU, A' and their bf16 low parts) also writes [dH | dU] as
// block-scaled codes with their scale blocks for the dX GEMM.  Eight epilogue warps, 32 columns at a time.
cudaError_t run_dact_dswiglu_mx(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 128)
    return launch_grouped_gemm<128, 4, 8, 2, A_TMA_K, B_TMA_K3, VAR_M, EPI_DSWIGLU, false, 1, X_MX>(p, m, grid, s);
  return launch_grouped_gemm<kMxBN, 4, 8, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_DSWIGLU, false, 1, X_MX>(p, m, grid, s);
}

// The dX GEMM on block-scaled operands: A = [dH | dU] codes [cap][2n], B = [W_gate; W_up]^T [E][d][2n] codes;
// plain bf16 store of dXp (four epilogue warps: 64-column stores of the 192-column tile).
cudaError_t run_dx_store_mx(int BN, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 128)
    return launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE, false, 1, X_MX>(p, m, grid, s);
  return launch_grouped_gemm<kMxBN, 4, 4, 1, A_TMA_K, B_TMA_K3, VAR_M, EPI_STORE, false, 1, X_MX>(p, m, grid, s);
}

// ---- the weight gradients on block-scaled operands -----------------------------------------------------------
// dW_gate[e] = dH_e^T X_e, dW_up[e] = dU_e^T X_e, dW_down[e] = dO_e^T A'_e reduce over the expert's tokens, so
// their blocks run along tokens: 1 x 32 blocks of one column over 32 consecutive tokens of one expert.  Every
// operand is written transposed, K-major ([column][token] codes), with each expert's tokens starting on a
// whole 128-token stage (zero codes fill the stage past the expert's last token; an all-zero block has
// scale byte 127).

// Stage offsets of the padded reduction: kp[g] = sum over the groups before g of their row counts rounded up to
// 128, counted in code pairs (the GEMM's K unit: 64 pairs per stage).  One block.
__global__ void __launch_bounds__(1024) mx_stage_offsets_kernel(const int32_t* __restrict__ off, int E,
                                                                int32_t* __restrict__ kp, int* err) {
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
      r = (r + 127) / 128 * 64;
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
      const int w = wsum[lane];
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      wsum[lane] = wi - w;
    }
    __syncthreads();
    const int excl = carry + wsum[warp] + incl - r;
    if (g < E) kp[g] = excl;
    __syncthreads();
    if (tid == 1023) carry = excl + r;
    __syncthreads();
  }
  if (tid == 0) kp[E] = carry;
}

cudaError_t launch_mx_stage_offsets(const int32_t* off, int E, int32_t* kp, int* err, cudaStream_t s) {
  mx_stage_offsets_kernel<<<1, 1024, 0, s>>>(off, E, kp, err);
  return cudaGetLastError();
}

// One block per (stage of 128 padded tokens, 64 columns, job): the 128 x 64 tile of the job's source (gathered
// rows, or the sorted rows themselves; high + low part when given) is staged in shared memory as fp32, then
// thread (column c, 32-token block k) quantizes the column's 32 values, writes their 32 codes to row
// row0 + c of the job's code matrix and the scale byte into the job's block of that row's tile and stage.
constexpr int kMxColThreads = 256;
__global__ void __launch_bounds__(kMxColThreads) quantize_cols_mx_kernel(MxColJobs jobs, const int32_t* __restrict__ off,
                                                                        const int32_t* __restrict__ kp, int E,
                                                                        long long pos_cap, long long kq, int kst,
                                                                        int* err) {
  __shared__ float tile[128][64];
  const MxColJob& jb = jobs.job[blockIdx.z];
  const int c0 = blockIdx.y * 64;
  if (c0 >= jb.C) return;
  const int stage = blockIdx.x;
  const int t0 = stage * 64;  // first pair of the stage
  if (t0 >= __ldg(kp + E)) return;  // past the padded reduction
  // the group whose padded range holds the stage: the largest g with kp[g] <= t0
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(kp + mid) <= t0) lo = mid;
    else hi = mid;
  }
  const int g = lo;
  const int j0 = 2 * (t0 - __ldg(kp + g));  // position of the stage's first token within the group
  const int base = __ldg(off + g), cnt = __ldg(off + g + 1) - base;
  const int tid = threadIdx.x;
  // load: 8 threads per row (8 columns each), 32 rows per pass
  {
    const int q8 = tid & 7;
    const int col = c0 + 8 * q8;
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      const int i = pass * 32 + (tid >> 3);
      const int j = j0 + i;
      long long srow = -1;
      if (j < cnt) {
        const long long pos = static_cast<long long>(base) + j;
        if (pos < 0 || pos >= pos_cap) {
          set_error(err, DERR_BAD_OFFSETS);
        } else {
          srow = jb.idx ? static_cast<long long>(__ldg(jb.idx + pos)) : pos;
          if (srow >= jb.src_rows) {
            set_error(err, DERR_BAD_OFFSETS);
            srow = -1;
          }
        }
      }
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = 0.0f;
      if (srow >= 0 && col < jb.C) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(jb.src + srow * jb.ld + col));
        const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack_bf16x2(xv[e]);
          v[2 * e] = f.x;
          v[2 * e + 1] = f.y;
        }
        if (jb.src_lo) {
          const uint4 y = __ldg(reinterpret_cast<const uint4*>(jb.src_lo + srow * jb.ld + col));
          const uint32_t yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(yv[e]);
            v[2 * e] += f.x;
            v[2 * e + 1] += f.y;
          }
        }
      }
      *reinterpret_cast<float4*>(&tile[i][8 * q8]) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(&tile[i][8 * q8 + 4]) = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
  __syncthreads();
  const int c = tid & 63, kb = tid >> 6;
  if (c0 + c >= jb.C) return;
  float v[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) v[t] = tile[kb * 32 + t][c];
  uint32_t w[8];
  const int e = mx_block32(v, w);
  const long long r = static_cast<long long>(jb.row0) + c0 + c;  // operand row of the code matrix
  uint4* dst = reinterpret_cast<uint4*>(jb.q + r * kq + static_cast<long long>(stage) * 128 + kb * 32);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  const int nblk = (jb.tw + 127) / 128;
  const long long tl = r / jb.tw;
  const int tr = static_cast<int>(r - tl * jb.tw), br = tr & 127;
  jb.sf[(tl * kst + stage) * (512ll * nblk) + (tr >> 7) * 512 + (br & 31) * 16 + (br >> 5) * 4 + kb] =
      static_cast<uint8_t>(e + 127);
}

cudaError_t launch_quantize_cols_mx(const MxColJobs& jobs, int njobs, const int32_t* off, const int32_t* kp, int E,
                                    long long pos_cap, long long kq, int kst, int* err, cudaStream_t s) {
  if (njobs <= 0 || njobs > kMxColJobs || kst <= 0) return njobs > kMxColJobs ? cudaErrorInvalidValue : cudaSuccess;
  int chunks = 0;
  for (int i = 0; i < njobs; ++i) chunks = chunks > (jobs.job[i].C + 63) / 64 ? chunks : (jobs.job[i].C + 63) / 64;
  quantize_cols_mx_kernel<<<dim3(kst, chunks, njobs), kMxColThreads, 0, s>>>(jobs, off, kp, E, pos_cap, kq, kst,
                                                                              err);
  return cudaGetLastError();
}

// The weight-gradient GEMMs on block-scaled operands: A = [M][K] codes, B = [N][K] codes (varlen-K over the
// padded per-expert stages), plain store of the [E][M][N] gradient (rows past out_rows_split to the second
// output), bf16 or fp32.
cudaError_t run_dw_mx(int BN, bool f32, const GemmParams& p, const Maps& m, int grid, cudaStream_t s) {
  if (BN == 128)
    return f32 ? launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_K3, VAR_K, EPI_STORE, true, 1, X_MX>(p, m, grid, s)
               : launch_grouped_gemm<128, 6, 4, 1, A_TMA_K, B_TMA_K3, VAR_K, EPI_STORE, false, 1, X_MX>(p, m, grid, s);
  return f32 ? launch_grouped_gemm<kMxBN, 4, 4, 1, A_TMA_K, B_TMA_K3, VAR_K, EPI_STORE, true, 1, X_MX>(p, m, grid, s)
             : launch_grouped_gemm<kMxBN, 4, 4, 1, A_TMA_K, B_TMA_K3, VAR_K, EPI_STORE, false, 1, X_MX>(p, m, grid, s);
}

}  // namespace vgg

// Persistent grouped GEMM for sm_103a on the 5th-generation tensor cores.
//
//   D[128 x BN] (+)= A[128 x K] * B[K x BN]    bf16 operands, fp32 accumulation in TMEM
//
// One CTA per SM walks a static round-robin list of output tiles.  Warp roles:
//   warps 0-3  epilogue: tcgen05.ld of the accumulator (row i of the tile = TMEM lane i),
//              fused elementwise work, global stores;
//   warps 4-7  cp.async producers for operands whose rows are gathered through an
//              index (token gather fused into the operand load) or whose reduction
//              length varies per group (zero-filled past the group's end);
//   warp  8    TMA producer (one thread) for dense operands; owns the TMEM allocation;
//   warp  9    UMMA issuer (one thread).
// Shared memory holds STAGES ring slots of A (128 x 64) and B (BN x 64) in the
// 128-byte-swizzled layout that both TMA and the UMMA descriptors use.  TMEM
// holds two BN-column accumulators so that the epilogue of tile i overlaps the
// main loop of tile i+1 ([SM] "4.3 MMA ↔ IO 오버랩": TMEM split in two halves,
// one accumulating while the other drains).
//
// Grouping ("varlen") modes:
//   VAR_M    groups = experts, rows of group g are sorted rows [off[g], off[g+1]);
//            K and N fixed ([GG] "Variable-M batched matmul").
//   VAR_K    groups = experts, the reduction runs over the group's rows; M and N
//            fixed; an empty group writes zeros ([SM] "4 기여 ②": varlen-K).
//   VAR_NONE one dense problem, K optionally split across CTAs (partials per split).
#pragma once

#include <climits>

#include "ptx.cuh"

namespace vgg {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 320;
constexpr int kMaxGroups = 1024;

enum AMode { A_TMA_K = 0, A_CP_K = 1, A_CP_MN = 2, A_TMA_MN = 3 };
enum BMode { B_TMA_K3 = 0, B_TMA_K3_GU = 1, B_TMA_MN3 = 2, B_TMA_MN2 = 3, B_CP_MN = 4 };
enum VarMode { VAR_M = 0, VAR_K = 1, VAR_NONE = 2 };
enum EpiKind { EPI_STORE = 0, EPI_SWIGLU = 1, EPI_SCALE = 2, EPI_DSWIGLU = 3 };

// A row-gathered (or row-predicated) operand read with cp.async.
struct GatherSrc {
  const __nv_bfloat16* ptr0;
  const __nv_bfloat16* ptr1;  // columns >= split are read from ptr1 at (col - split)
  const int* idx;             // sorted position -> source row; null = identity
  long long ld;               // row stride in elements
  int split;                  // column split between ptr0 and ptr1
  int cols;                   // valid columns of the operand's MN extent
  long long rows;             // rows of the source; a gathered row index outside [0, rows) is an error
};

struct GemmParams {
  int M, N, K;
  int groups;
  const int* offsets;  // [groups + 1], device
  int rows_cap;        // offsets[groups] must not exceed this
  int split_k;         // VAR_NONE: number of K splits
  int a_ksplit;        // TMA A: k < a_ksplit from map 0, else map 1 at k - a_ksplit
  int b_ksplit;        // TMA B: same for B
  GatherSrc ga, gb;
  void* out0;
  void* out1;
  void* out2;
  long long ld_out;
  long long group_stride_out;  // VAR_K: per group; VAR_NONE: per K split
  int out_rows_split;          // VAR_K: output rows >= split go to out1 at row - split
  int out_fp32;
  const float* row_scale;  // VAR_M: per sorted row (combine weight)
  const float* in0;  // dSwiGLU epilogue: H, U (fp32)
  const float* in1;
  long long ld_in;
  float* part;  // dSwiGLU epilogue: per-row partial dot products [rows][part_ld]
  int part_ld;
  const float* col_bias;
  int* err;
  unsigned long long timeout_ns;
};

template <int BN, int STAGES>
struct SmemLayout {
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOffset = STAGES * kStageBytes;
  static constexpr int kNumBars = 3 * STAGES + 5;
  static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
  static constexpr size_t bytes(int groups) {
    return 1024 + static_cast<size_t>(kMiscOffset) + 16 + 8 * static_cast<size_t>(groups + 2);
  }
};

struct Tile {
  int g;        // group
  int m0;       // first row of the tile (relative to the group for VAR_M)
  int n0;       // first output column (for the gate/up pair: first column of each half)
  int nt;       // column-tile index
  int rows;     // VAR_M: valid rows in this tile; otherwise rows of M left from m0
  int k_begin;  // VAR_K: first sorted row of the group; VAR_NONE: first k of the split
  int k_len;    // reduction length handled by this tile
  int split;    // VAR_NONE: K split index
};

template <int BN, int BMODE, int VAR>
struct Sched {
  static constexpr int kColsPerTile = (BMODE == B_TMA_K3_GU) ? BN / 2 : BN;
  int ntiles, mtiles, per_group, total, ks_len;
  const int* s_off;
  const int* s_tile;

  __device__ void init(const GemmParams& p, const int* off, const int* tile) {
    s_off = off;
    s_tile = tile;
    ntiles = (p.N + kColsPerTile - 1) / kColsPerTile;
    mtiles = (p.M + BM - 1) / BM;
    if (VAR == VAR_M) {
      total = tile[p.groups];
    } else if (VAR == VAR_K) {
      per_group = mtiles * ntiles;
      total = per_group * p.groups;
    } else {
      per_group = mtiles * ntiles;
      total = per_group * p.split_k;
      ks_len = ((p.K + p.split_k - 1) / p.split_k + BK - 1) / BK * BK;
    }
  }

  // Tiles are visited in increasing order by each CTA, so the group cursor only moves forward.
  __device__ void decode(const GemmParams& p, int t, int& gcur, Tile& tl) const {
    if (VAR == VAR_M) {
      while (s_tile[gcur + 1] <= t) ++gcur;
      const int g = gcur;
      const int rows_g = s_off[g + 1] - s_off[g];
      const int mt_g = (rows_g + BM - 1) / BM;
      const int l = t - s_tile[g];
      const int mt = l % mt_g, nt = l / mt_g;
      tl.g = g;
      tl.m0 = mt * BM;
      tl.nt = nt;
      tl.n0 = nt * kColsPerTile;
      tl.rows = min(BM, rows_g - tl.m0);
      tl.k_begin = 0;
      tl.k_len = p.K;
      tl.split = 0;
    } else if (VAR == VAR_K) {
      const int g = t / per_group;
      const int l = t - g * per_group;
      const int mt = l % mtiles, nt = l / mtiles;
      tl.g = g;
      tl.m0 = mt * BM;
      tl.nt = nt;
      tl.n0 = nt * kColsPerTile;
      tl.rows = min(BM, p.M - tl.m0);
      tl.k_begin = s_off[g];
      tl.k_len = s_off[g + 1] - s_off[g];
      tl.split = 0;
    } else {
      const int sp = t / per_group;
      const int l = t - sp * per_group;
      const int mt = l % mtiles, nt = l / mtiles;
      tl.g = 0;
      tl.m0 = mt * BM;
      tl.nt = nt;
      tl.n0 = nt * kColsPerTile;
      tl.rows = min(BM, p.M - tl.m0);
      tl.k_begin = sp * ks_len;
      tl.k_len = max(0, min(p.K, (sp + 1) * ks_len) - tl.k_begin);
      tl.split = sp;
    }
  }
};

// Byte offset of the 16-byte piece (row r, piece c16) of a 128-byte-swizzled [rows x 128 B] block.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c16) {
  return static_cast<uint32_t>(r * 128 + ((c16 ^ (r & 7)) << 4));
}

// -------------------------------------------------------------------------- epilogue helpers

__device__ __forceinline__ void store_row_chunk(void* base, long long elem_off, const float (&v)[32], int ncols,
                                                int fp32) {
  if (fp32) {
    float* o = reinterpret_cast<float*>(base) + elem_off;
    if (ncols >= 32) {
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < ncols) o[i] = v[i];
    }
  } else {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(base) + elem_off;
    if (ncols >= 32) {
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        uint4 q;
        q.x = pack_bf16x2(v[i], v[i + 1]);
        q.y = pack_bf16x2(v[i + 2], v[i + 3]);
        q.z = pack_bf16x2(v[i + 4], v[i + 5]);
        q.w = pack_bf16x2(v[i + 6], v[i + 7]);
        *reinterpret_cast<uint4*>(o + i) = q;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < ncols) o[i] = __float2bfloat16_rn(v[i]);
    }
  }
}

__device__ __forceinline__ void load_f32_chunk(const float* src, float (&v)[32], int ncols) {
  if (ncols >= 32) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 q = *reinterpret_cast<const float4*>(src + i);
      v[i] = q.x; v[i + 1] = q.y; v[i + 2] = q.z; v[i + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = (i < ncols) ? src[i] : 0.0f;
  }
}

__device__ __forceinline__ void load_bf16_chunk(const __nv_bfloat16* src, float (&v)[32], int ncols) {
  if (ncols >= 32) {
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      uint4 q = *reinterpret_cast<const uint4*>(src + i);
      float2 a = unpack_bf16x2(q.x), b = unpack_bf16x2(q.y), c = unpack_bf16x2(q.z), d = unpack_bf16x2(q.w);
      v[i] = a.x; v[i + 1] = a.y; v[i + 2] = b.x; v[i + 3] = b.y;
      v[i + 4] = c.x; v[i + 5] = c.y; v[i + 6] = d.x; v[i + 7] = d.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = (i < ncols) ? __bfloat162float(src[i]) : 0.0f;
  }
}

// -------------------------------------------------------------------------- the kernel

template <int BN, int STAGES, int AMODE, int BMODE, int VAR, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1) {
  using L = SmemLayout<BN, STAGES>;
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(EPI != EPI_SWIGLU || BMODE == B_TMA_K3_GU, "SwiGLU epilogue needs the gate/up pair layout");
  constexpr bool kACp = (AMODE == A_CP_K || AMODE == A_CP_MN);
  constexpr bool kBCp = (BMODE == B_CP_MN);
  constexpr bool kAnyCp = kACp || kBCp;
  constexpr bool kATma = !kACp;
  constexpr bool kBTma = !kBCp;
  constexpr bool kAMn = (AMODE == A_CP_MN || AMODE == A_TMA_MN);
  constexpr bool kBMn = (BMODE == B_TMA_MN3 || BMODE == B_TMA_MN2 || BMODE == B_CP_MN);
  constexpr uint32_t kTxBytes = (kATma ? L::kABytes : 0) + (kBTma ? L::kBBytes : 0);
  constexpr uint32_t kTmemCols = (2 * BN <= 128) ? 128 : (2 * BN <= 256 ? 256 : 512);
  constexpr uint32_t kIdesc = idesc_bf16(BM, BN, kAMn ? 1 : 0, kBMn ? 1 : 0);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + STAGES;
  uint64_t* tfull_bar = bars + 2 * STAGES;
  uint64_t* tempty_bar = bars + 2 * STAGES + 2;
  uint64_t* drain_bar = bars + 2 * STAGES + 4;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::kMiscOffset);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kMiscOffset + 4);
  int* s_bad = reinterpret_cast<int*>(smem + L::kMiscOffset + 8);
  int* s_off = reinterpret_cast<int*>(smem + L::kMiscOffset + 16);
  int* s_tile = s_off + (p.groups + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], (kAnyCp ? 128u : 0u) + (kATma || kBTma ? 1u : 0u));
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 128);
    }
    mbar_init(drain_bar, 1);
    *s_abort = 0;
    *s_bad = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(s_tmem, kTmemCols);
    if (lane == 0) {
      if (kATma) {
        tma_prefetch_desc(&tmA0);
        tma_prefetch_desc(&tmA1);
      }
      if (kBTma) {
        tma_prefetch_desc(&tmB0);
        tma_prefetch_desc(&tmB1);
      }
    }
  }
  // group offsets into shared memory (validated: start at 0, monotone, within capacity)
  if (VAR != VAR_NONE) {
    for (int g = tid; g <= p.groups; g += kThreads) s_off[g] = __ldg(p.offsets + g);
  } else if (tid == 0) {
    s_off[0] = 0;
    s_off[1] = p.M;
  }
  __syncthreads();
  if (VAR != VAR_NONE && warp == 0) {
    int running = 0, bad = 0;
    for (int base = 0; base < p.groups; base += 32) {
      const int g = base + lane;
      int cnt = 0;
      if (g < p.groups) {
        const int rows_g = s_off[g + 1] - s_off[g];
        if (rows_g < 0) bad = 1;
        if (VAR == VAR_M)
          cnt = max(0, (rows_g + BM - 1) / BM) * ((p.N + Sched<BN, BMODE, VAR>::kColsPerTile - 1) /
                                                  Sched<BN, BMODE, VAR>::kColsPerTile);
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (g < p.groups) s_tile[g] = running + incl - cnt;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (s_off[0] != 0 || s_off[p.groups] > p.rows_cap) bad = 1;
      s_tile[p.groups] = bad ? 0 : running;
      if (bad) {
        *s_bad = 1;
        set_error(p.err, DERR_BAD_OFFSETS);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  Sched<BN, BMODE, VAR> sch;
  sch.init(p, s_off, s_tile);
  if (*s_bad) sch.total = 0;

  if (warp == 8) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && (kATma || kBTma)) {
      int it = 0, gcur = 0;
      bool aborted = false;
      for (int t = blockIdx.x; t < sch.total && !aborted; t += gridDim.x) {
        Tile tl;
        sch.decode(p, t, gcur, tl);
        const int nk = (tl.k_len + BK - 1) / BK;
        for (int ks = 0; ks < nk; ++ks, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&empty_bar[s], ph ^ 1, s_abort, p.timeout_ns, p.err)) {
            aborted = true;
            break;
          }
          uint8_t* sa = smem + s * L::kStageBytes;
          uint8_t* sb = sa + L::kABytes;
          mbar_arrive_expect_tx(&full_bar[s], kTxBytes);
          const int kg = tl.k_begin + ks * BK;
          if (AMODE == A_TMA_K) {
            const int row = (VAR == VAR_M ? s_off[tl.g] : 0) + tl.m0;
            if (kg < p.a_ksplit) tma_load_2d(sa, &tmA0, &full_bar[s], kg, row);
            else tma_load_2d(sa, &tmA1, &full_bar[s], kg - p.a_ksplit, row);
          } else if (AMODE == A_TMA_MN) {
#pragma unroll
            for (int c = 0; c < BM / 64; ++c) tma_load_2d(sa + c * (BK * 128), &tmA0, &full_bar[s], tl.m0 + 64 * c, kg);
          }
          if (BMODE == B_TMA_K3) {
            tma_load_3d(sb, &tmB0, &full_bar[s], kg, tl.n0, tl.g);
          } else if (BMODE == B_TMA_K3_GU) {
            tma_load_3d(sb, &tmB0, &full_bar[s], kg, tl.n0, tl.g);
            tma_load_3d(sb + (BN / 2) * 128, &tmB1, &full_bar[s], kg, tl.n0, tl.g);
          } else if (BMODE == B_TMA_MN3) {
            const bool first = kg < p.b_ksplit;
            const int kc = first ? kg : kg - p.b_ksplit;
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_3d(sb + c * (BK * 128), first ? &tmB0 : &tmB1, &full_bar[s], tl.n0 + 64 * c, kc, tl.g);
          } else if (BMODE == B_TMA_MN2) {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c) tma_load_2d(sb + c * (BK * 128), &tmB0, &full_bar[s], tl.n0 + 64 * c, kg);
          }
        }
      }
      if (aborted) {
        // let copies already in flight land before the CTA goes away
        volatile int never = 0;
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          mbar_wait(&full_bar[j % STAGES], (j / STAGES) & 1, &never, 20000000ull, nullptr);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------------- cp.async producers
    if (kAnyCp) {
      const int ptid = tid - 128;
      int it = 0, gcur = 0;
      bool aborted = false;
      for (int t = blockIdx.x; t < sch.total && !aborted; t += gridDim.x) {
        Tile tl;
        sch.decode(p, t, gcur, tl);
        const int nk = (tl.k_len + BK - 1) / BK;
        // A gathered along M: the tile's 8 rows handled by this thread are fixed for the whole tile
        long long arow[8];
        bool aval[8];
        if (AMODE == A_CP_K) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = (ptid >> 3) + 16 * i;
            aval[i] = r < tl.rows;
            const int srow = s_off[tl.g] + tl.m0 + r;
            arow[i] = aval[i] ? (p.ga.idx ? __ldg(p.ga.idx + srow) : srow) : 0;
            if (arow[i] < 0 || arow[i] >= p.ga.rows) {
              if (aval[i]) set_error(p.err, DERR_BAD_OFFSETS);
              aval[i] = false;
              arow[i] = 0;
            }
          }
        }
        for (int ks = 0; ks < nk; ++ks, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&empty_bar[s], ph ^ 1, s_abort, p.timeout_ns, p.err)) {
            aborted = true;
            break;
          }
          const uint32_t sa = smem_u32(smem + s * L::kStageBytes);
          const uint32_t sb = sa + L::kABytes;
          const int c16 = ptid & 7;
          if (AMODE == A_CP_K) {
            const int kc = ks * BK + c16 * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = (ptid >> 3) + 16 * i;
              const __nv_bfloat16* src = p.ga.ptr0 + arow[i] * p.ga.ld + kc;
              cp_async_16(sa + sw128_offset(r, c16), aval[i] ? src : p.ga.ptr0, aval[i] ? 16u : 0u);
            }
          } else if (AMODE == A_CP_MN) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int chunk = i >> 2;
              const int r = (ptid >> 3) + 16 * (i & 3);
              const int kr = ks * BK + r;
              const int col = tl.m0 + 64 * chunk + c16 * 8;
              bool ok = kr < tl.k_len && col < p.ga.cols;
              const __nv_bfloat16* src = p.ga.ptr0;
              if (ok) {
                const int srow = tl.k_begin + kr;
                const long long row = p.ga.idx ? __ldg(p.ga.idx + srow) : srow;
                if (row < 0 || row >= p.ga.rows) {
                  set_error(p.err, DERR_BAD_OFFSETS);
                  ok = false;
                } else {
                  src = (col < p.ga.split) ? p.ga.ptr0 + row * p.ga.ld + col
                                           : p.ga.ptr1 + row * p.ga.ld + (col - p.ga.split);
                }
              }
              cp_async_16(sa + chunk * (BK * 128) + sw128_offset(r, c16), src, ok ? 16u : 0u);
            }
          }
          if (BMODE == B_CP_MN) {
#pragma unroll
            for (int i = 0; i < 4 * (BN / 64); ++i) {
              const int chunk = i >> 2;
              const int r = (ptid >> 3) + 16 * (i & 3);
              const int kr = ks * BK + r;
              const int col = tl.n0 + 64 * chunk + c16 * 8;
              bool ok = kr < tl.k_len && col < p.gb.cols;
              const __nv_bfloat16* src = p.gb.ptr0;
              if (ok) {
                const int srow = tl.k_begin + kr;
                const long long row = p.gb.idx ? __ldg(p.gb.idx + srow) : srow;
                if (row < 0 || row >= p.gb.rows) {
                  set_error(p.err, DERR_BAD_OFFSETS);
                  ok = false;
                } else {
                  src = (col < p.gb.split) ? p.gb.ptr0 + row * p.gb.ld + col
                                           : p.gb.ptr1 + row * p.gb.ld + (col - p.gb.split);
                }
              }
              cp_async_16(sb + chunk * (BK * 128) + sw128_offset(r, c16), src, ok ? 16u : 0u);
            }
          }
          cp_async_mbar_arrive_noinc(&full_bar[s]);
        }
      }
      cp_async_wait_all();
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- UMMA issuer
    if (lane == 0) {
      int it = 0, acc = 0, gcur = 0;
      bool aborted = false;
      for (int t = blockIdx.x; t < sch.total && !aborted; t += gridDim.x, ++acc) {
        Tile tl;
        sch.decode(p, t, gcur, tl);
        const int nk = (tl.k_len + BK - 1) / BK;
        const int buf = acc & 1;
        if (!mbar_wait(&tempty_bar[buf], ((acc >> 1) & 1) ^ 1, s_abort, p.timeout_ns, p.err)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int ks = 0; ks < nk; ++ks, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&full_bar[s], ph, s_abort, p.timeout_ns, p.err)) {
            aborted = true;
            break;
          }
          if (kAnyCp) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * L::kStageBytes);
          const uint32_t sb = sa + L::kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = kAMn ? sdesc_sw128(sa + kk * 2048, BK * 128, 1024) : sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = kBMn ? sdesc_sw128(sb + kk * 2048, BK * 128, 1024) : sdesc_sw128(sb + kk * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, kIdesc, (ks | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&empty_bar[s]);
        }
        if (aborted) break;
        umma_commit(&tfull_bar[buf]);
      }
      if (aborted) {
        umma_commit(drain_bar);
        volatile int never = 0;
        mbar_wait(drain_bar, 0, &never, 20000000ull, nullptr);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 0-3)
    int acc = 0, gcur = 0;
    const int row_local = warp * 32 + lane;
    for (int t = blockIdx.x; t < sch.total; t += gridDim.x, ++acc) {
      Tile tl;
      sch.decode(p, t, gcur, tl);
      const int buf = acc & 1;
      if (!mbar_wait(&tfull_bar[buf], (acc >> 1) & 1, s_abort, p.timeout_ns, p.err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + buf * BN;
      const bool row_ok = row_local < tl.rows;
      const bool have_acc = tl.k_len > 0;

      if (EPI == EPI_SWIGLU) {
        const long long orow = s_off[tl.g] + tl.m0 + row_local;
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t rh[32], ru[32];
          tmem_ld32(tbase + c, rh);
          tmem_ld32(tbase + BN / 2 + c, ru);
          tmem_ld_wait();
          const int col = tl.n0 + c;
          const int ncols = p.N - col;
          if (row_ok && ncols > 0) {
            float h[32], u[32], a[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              h[i] = __uint_as_float(rh[i]);
              u[i] = __uint_as_float(ru[i]);
              a[i] = h[i] * sigmoidf_(h[i]) * u[i];
            }
            const long long off = orow * p.ld_out + col;
            store_row_chunk(p.out0, off, h, ncols, 1);  // H, U stay fp32 for the backward
            store_row_chunk(p.out1, off, u, ncols, 1);
            store_row_chunk(p.out2, off, a, ncols, 0);  // A is the bf16 operand of the down projection
          }
        }
      } else if (EPI == EPI_SCALE) {
        const long long orow = s_off[tl.g] + tl.m0 + row_local;
        const float w = row_ok ? __ldg(p.row_scale + orow) : 0.0f;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(tbase + c, r);
          tmem_ld_wait();
          const int col = tl.n0 + c;
          const int ncols = p.N - col;
          if (row_ok && ncols > 0) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = w * __uint_as_float(r[i]);
            store_row_chunk(p.out0, orow * p.ld_out + col, v, ncols, 0);
          }
        }
      } else if (EPI == EPI_DSWIGLU) {
        const long long orow = s_off[tl.g] + tl.m0 + row_local;
        const float w = row_ok ? __ldg(p.row_scale + orow) : 0.0f;
        float ds = 0.0f;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(tbase + c, r);
          tmem_ld_wait();
          const int col = tl.n0 + c;
          const int ncols = p.N - col;
          if (row_ok && ncols > 0) {
            float h[32], u[32], dh[32], du[32], ap[32];
            load_f32_chunk(p.in0 + orow * p.ld_in + col, h, ncols);
            load_f32_chunk(p.in1 + orow * p.ld_in + col, u, ncols);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float dap = __uint_as_float(r[i]);  // dA' = dO . W_down (unweighted)
              const float sg = sigmoidf_(h[i]);
              const float sl = h[i] * sg;
              const float a = sl * u[i];
              ds += dap * a;
              const float da = w * dap;
              du[i] = da * sl;
              dh[i] = da * u[i] * sg * (1.0f + h[i] * (1.0f - sg));
              ap[i] = w * a;
            }
            const long long off = orow * p.ld_out + col;
            store_row_chunk(p.out0, off, dh, ncols, 0);
            store_row_chunk(p.out1, off, du, ncols, 0);
            store_row_chunk(p.out2, off, ap, ncols, 0);
          }
        }
        if (row_ok) p.part[orow * p.part_ld + tl.nt] = ds;
      } else {  // EPI_STORE
        long long obase;
        void* optr = p.out0;
        const int m = tl.m0 + row_local;
        if (VAR == VAR_M) {
          obase = (s_off[tl.g] + tl.m0 + row_local) * p.ld_out;
        } else if (VAR == VAR_K) {
          obase = static_cast<long long>(tl.g) * p.group_stride_out;
          if (m >= p.out_rows_split) {
            optr = p.out1;
            obase += static_cast<long long>(m - p.out_rows_split) * p.ld_out;
          } else {
            obase += static_cast<long long>(m) * p.ld_out;
          }
        } else {
          obase = static_cast<long long>(tl.split) * p.group_stride_out + static_cast<long long>(m) * p.ld_out;
        }
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(tbase + c, r);
          tmem_ld_wait();
          const int col = tl.n0 + c;
          const int ncols = p.N - col;
          if (row_ok && ncols > 0) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v[i] = have_acc ? __uint_as_float(r[i]) : 0.0f;
              if (p.col_bias && i < ncols) v[i] += __ldg(p.col_bias + col + i);
            }
            store_row_chunk(optr, obase + col, v, ncols, p.out_fp32);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem_base, kTmemCols);
}

template <int BN, int STAGES, int AMODE, int BMODE, int VAR, int EPI>
cudaError_t launch_grouped_gemm(const GemmParams& p, const CUtensorMap* maps, int grid, cudaStream_t stream) {
  auto kern = grouped_gemm_kernel<BN, STAGES, AMODE, BMODE, VAR, EPI>;
  const size_t smem = SmemLayout<BN, STAGES>::bytes(p.groups);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, kThreads, smem, stream>>>(p, maps[0], maps[1], maps[2], maps[3]);
  return cudaGetLastError();
}

}  // namespace vgg

// Persistent grouped GEMM for sm_103a on the 5th-generation tensor cores.
//
//   D[128 x BN] (+)= A[128 x K] * B[K x BN]    bf16 operands (kind::f16) or, for the e4m3 epilogues,
//                                              e4m3 operands (kind::f8f6f4); fp32 accumulation in TMEM
//
// One CTA per SM walks a static round-robin list of output tiles.  Warp roles:
//   warps 0..EW-1  epilogue (4 or 8): tcgen05.ld of the accumulator (row i of the tile = TMEM
//              lane i), fused elementwise work, results staged in shared memory per 32-row
//              block and written by TMA stores;
//   warp  EW   TMA producer (lane 0) for the tiled operands; owns the TMEM allocation.  Loads
//              issued by one thread complete one after another, so the ring's stages are dealt
//              round-robin to up to 4 producer threads (this one and extra warps placed last);
//   warp  EW+1 UMMA issuer (lane 0);
//   gather warps (8 for a gathered K-major A, else 4) present when an operand's rows are gathered
//              through a token index: they copy those rows with cp.async (16 B per thread,
//              zero-filled past the end) straight into the swizzled stage, so the permuted
//              activations are never written ([SM] "4.1 Gather 융합"); the index lookups run two
//              stages ahead;
//   relay warp present with clusters of CN CTAs on neighbouring column tiles of one row tile:
//              each CTA gathers 128/CN of the rows and the relay copies its slice into the
//              peers' shared memory (distributed shared memory), so the gathered activations
//              are read from L2 once per cluster instead of once per CTA.
// Shared memory holds STAGES ring slots of A (128 rows x 128 bytes) and B (BN rows x 128 bytes: 64
// bf16 or 128 e4m3 values of K) in the 128-byte-swizzled layout that TMA writes and the UMMA
// descriptors read.  TMEM holds two BN-column accumulators so that the epilogue of tile i overlaps
// the main loop of tile i+1 ([SM] "4.3 MMA ↔ IO 오버랩": TMEM split in two halves, one accumulating
// while the other drains).
//
// Grouping ("varlen") modes:
//   VAR_M    groups = experts, rows of group g are sorted rows [off[g], off[g+1]);
//            K and N fixed ([GG] "Variable-M batched matmul").
//   VAR_K    groups = experts, the reduction runs over the group's rows; M and N
//            fixed; rows past the group's end enter as zeros (the gathered operand's
//            out-of-range fill, or cleared in shared memory when both operands are tiled);
//            an empty group writes zeros ([SM] "4 기여 ②").
//   VAR_NONE one dense problem, K optionally split across CTAs (partials per split).
#pragma once

#include <climits>

#include "ptx.cuh"

namespace vgg {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kMaxThreads = 384;  // up to 8 epilogue warps + producer + issuer, or 4 + 2 + 4 gather warps
constexpr int kMaxGroups = 1024;
constexpr size_t kMaxSmem = 232448;  // dynamic shared memory per CTA (227 KB)
constexpr int kStgBuf = 4096;    // one staged store: 32 rows x 128 B
constexpr int kPrefetchStages = 4;  // tiled operands are prefetched into L2 this many stages ahead

enum AMode { A_TMA_K = 0, A_GATHER_K = 1, A_TMA_MN = 2, A_GATHER_MN = 3 };
enum BMode { B_TMA_K3 = 0, B_TMA_K3_GU = 1, B_TMA_MN3 = 2, B_TMA_MN2 = 3, B_GATHER_MN = 4 };
enum VarMode { VAR_M = 0, VAR_K = 1, VAR_NONE = 2 };
// EPI_SWIGLU_Q, EPI_SCALE_Q, EPI_STORE_Q: the SwiGLU, the combine-weight and the plain (varlen-M, bf16)
// epilogues of the e4m3 form (operands are e4m3 codes of per-row-scaled rows; the accumulator is
// multiplied by the A row's scale and the output channel's scale first).
// EPI_DSWIGLU_Q: the dSwiGLU epilogue of the e4m3 form (the accumulator times q_row[row] q_col[column]).
// Extra forms (bit flags):
//   X_DUAL_A  the A operand arrives as a bf16 high part (maps a0/a1) and the bf16 rounding of the rest
//             (maps a2/a3, the same coordinates); every K step issues two UMMAs into one accumulator, so
//             the product carries about 16 significant bits of A.  The weight-gradient GEMMs take the
//             per-pair gradients (fp32 in the dSwiGLU epilogue) this way, the down projection the
//             activations A (fp32 in the SwiGLU epilogue).
//   X_TRANS   varlen-K plain store of the transposed tile: the tile's rows (TMEM lanes) are output
//             columns, its accumulator columns output rows; each 32 x 32 block is transposed while it is
//             staged for the TMA store.
//   X_PAIR    a CTA pair (cluster of 2, cta_group::2) computes a 256-row tile: each CTA loads its 128 rows of A
//             and half of B's columns, both CTAs' TMA loads complete on the even CTA's barriers, the even CTA
//             issues the M = 256 UMMAs, and each CTA drains its own 128 TMEM rows (varlen-K with padded B).
//   X_MX      block-scaled e4m3 operands (kind::mxf8f6f4): every 32 codes of an operand row along K carry
//             one power-of-two scale (UE8M0 byte).  A stage holds, after its A and B tiles, the 4 scale
//             bytes of each of A's 128 rows and of B's rows (one 512-byte block per 128 rows, the last one
//             padded) for its 128 codes of K in the layout tcgen05.cp reads
//             (row r, 32-code block k at byte (r % 32) 16 + (r / 32) 4 + k); the issuer copies them into
//             TMEM columns of that stage (past the two accumulators) before the stage's UMMAs.  The producer
//             brings every stage's scale bytes as whole 512-byte blocks laid out that way in global memory:
//             A's per row tile (for gathered rows, laid out per sorted row tile before the GEMM), B's per
//             column tile.
//             BN = 128 or 192, so that both accumulators and every stage's scales fit the 512 TMEM columns.  The
//             SwiGLU epilogue of this form emits A itself as block-scaled codes (a thread's 32 columns of
//             its row are one block) with the scale blocks the down projection reads, and the dSwiGLU
//             epilogue emits [dH | dU] the same way for the dX GEMM (o_q, o_sf).
//             Varlen-K (the weight gradients): both operands are K-major code matrices [rows][K] whose groups
//             each start on a whole stage (128 codes; the reduction padded per group with zero codes), one
//             [N][K] matrix for B, and the scale blocks of both indexed by the stage of the whole reduction.
enum XFlags { X_DUAL_A = 1, X_TRANS = 2, X_PAIR = 4, X_MX = 8 };
enum EpiKind {
  EPI_STORE = 0, EPI_SWIGLU = 1, EPI_SCALE = 2, EPI_DSWIGLU = 3, EPI_SWIGLU_Q = 4, EPI_SCALE_Q = 5, EPI_STORE_Q = 6,
  EPI_DSWIGLU_Q = 7
};

struct GemmParams {
  int M, N, K;
  int groups;
  const int* offsets;  // [groups + 1], device
  int rows_cap;        // offsets[groups] must not exceed this
  int split_k;         // VAR_NONE: number of K splits
  int a_ksplit;        // A_TMA_K: k < a_ksplit from map a0, else map a1 at k - a_ksplit
  int a_colsplit;      // A_TMA_MN: columns < split from map a0, else a1 at col - split
  int a_kwrap;         // A_TMA_MN: reduction rows k >= a_kwrap are read at k - a_kwrap (A repeated along K)
  int b_ksplit;        // B_TMA_MN3: k < b_ksplit from map b0, else b1 at k - b_ksplit
  int b_chunked;       // B_TMA_MN2: the map is the chunked 3-D view (one load per stage)
  int l2_prefetch;     // prefetch the tiled operands of later stages into L2
  const int* a_idx;    // gathered A: sorted position -> source row
  int a_rows;          // rows of the gathered A source
  const __nv_bfloat16* a_src;  // gathered A source [a_rows][a_ld]
  long long a_ld;
  const int* b_idx;
  int b_rows;
  // Optional row bases of the tiled operands (device, [groups + 1]): VAR_M A rows of group g start at
  // a_offsets[g], VAR_K B rows (the reduction) at b_offsets[g], instead of offsets[g].  The backward's
  // expert-sorted copies use them: every expert padded to a multiple of 16 rows with zero rows.
  const int* a_offsets;
  const int* b_offsets;
  const __nv_bfloat16* b_src;
  long long b_ld;
  // epilogue
  void* out0;  // direct-store pointers (used for a partially filled 32-row block)
  void* out1;
  void* out2;
  void* out3;  // dSwiGLU: bf16 low parts of dH, dU, A' (NULL: not written)
  void* out4;
  void* out5;
  long long ld_out;
  int out_rows_split;  // VAR_K: output rows >= split go to the second output at row - split
  const float* row_scale;  // VAR_M: per sorted row (combine weight); e4m3 SwiGLU: per source row of A
  const float* in0;        // dSwiGLU: H, U (fp32); e4m3 SwiGLU: W_gate, W_up scales [groups][ld_in];
  const float* in1;        // e4m3 combine-weight epilogue: A row scales [rows], W scales [groups][ld_in]
  long long ld_in;
  float* part;  // dSwiGLU epilogue: per-row partial dot products [rows][part_ld]
  int part_ld;
  const float* col_bias;
  const float* q_row;  // e4m3 dSwiGLU: A row scales [rows], B row scales [groups][q_ld]
  const float* q_col;
  int q_ld;
  // block-scaled form (X_MX): scale bytes of A (512-byte blocks [row tile][sf_kst], row tiles of the varlen-M
  // order), of B (ceil(BN / 128) 512-byte blocks per stage: [groups][column tile][sf_kst]) and of
  // the SwiGLU epilogue's block-scaled A (o_sf: [row tile][o_sf_kst] blocks); sf_kst = stages of K
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  int sf_kst;
  uint8_t* o_sf;
  int o_sf_kst;
  uint8_t* o_q;        // the dSwiGLU epilogue's block-scaled [dH | dU] codes [rows][o_q_ld] (o_sf: their blocks)
  long long o_q_ld;
  int* err;
  unsigned long long timeout_ns;
};

// One UMMA of the stage's K step: bf16 operands (K = 16) or e4m3 operands (K = 32); either way the
// step covers 32 bytes of every 128-byte operand row.
template <bool F8>
__device__ __forceinline__ void umma_step(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  if constexpr (F8) umma_e4m3(d_tmem, adesc, bdesc, idesc, accumulate);
  else umma_bf16(d_tmem, adesc, bdesc, idesc, accumulate);
}

// Tensor maps: a0/a1 and b0/b1 feed the operands (a2/a3: the low parts of a dual A), o0..o5 are the
// TMA-store targets.
struct Maps {
  CUtensorMap a0, a1, a2, a3, b0, b1, o0, o1, o2, o3, o4, o5;
};

// EW epilogue warps with DEPTH staged stores each; NA A tiles per stage (2: high and low parts); BNL rows of
// B per stage in this CTA (half of BN for a CTA pair); SF bytes of block scales per stage (X_MX, a multiple
// of 1024 so that every stage stays 1024-byte aligned).
template <int BN, int STAGES, int EW, int DEPTH, int NA = 1, int BNL = BN, int SF = 0>
struct SmemLayout {
  static constexpr int kA1Bytes = BM * BK * 2;
  static constexpr int kABytes = NA * kA1Bytes;
  static constexpr int kBBytes = BNL * BK * 2;
  static constexpr int kSfBytes = SF;
  static constexpr int kStageBytes = kABytes + kBBytes + SF;
  static constexpr int kStgOffset = STAGES * kStageBytes;
  static constexpr int kBarOffset = kStgOffset + EW * DEPTH * kStgBuf;
  static constexpr int kNumBars = 3 * STAGES + 5;
  static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
  // The grouped modes read the group offsets from global memory (a few cached loads per tile);
  // varlen-M keeps its per-group tile starts in shared memory.
  static constexpr size_t bytes(int groups, int var) {
    return 1024 + static_cast<size_t>(kMiscOffset) + 16 +
           (var == VAR_M ? 4 * static_cast<size_t>(groups + 1) : var == VAR_NONE ? 8 : 0);
  }
};

// Block-scaled form: B's scale blocks per stage (one 512-byte block per 128 rows of B), and the scale bytes of one
// stage (A's block, then B's), padded to 1024.
__host__ __device__ constexpr int mx_b_blocks(int BN) { return (BN + 127) / 128; }
__host__ __device__ constexpr int mx_stage_bytes(int BN, int XF) {
  return (XF & X_MX) ? ((512 + 512 * mx_b_blocks(BN) + 1023) / 1024) * 1024 : 0;
}

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

// With CN > 1 (varlen-M only) the CN CTAs of a cluster take the same (group, row tile) with
// consecutive column tiles: a work unit is (group, row tile, group of CN column tiles) and the CTA
// of cluster rank r computes column tile CN * unit_col + r (past the last one it computes nothing
// that is stored, but still takes part in loading the shared operand).
// With PAIR (varlen-K) the two CTAs of a cluster take the same tile of 256 rows, rank r rows 128 r ..
template <int BN, int BMODE, int VAR, int CN = 1, bool PAIR = false>
struct Sched {
  static constexpr int kColsPerTile = (BMODE == B_TMA_K3_GU) ? BN / 2 : BN;
  static constexpr int kRowsPerTile = PAIR ? 2 * BM : BM;  // a CTA pair computes 256-row tiles
  int ntiles, mtiles, per_group, total, ks_len;
  int first, stride, rank;  // this CTA's first unit, the unit stride, its rank in the cluster
  const int* s_off;
  const int* s_tile;

  __device__ void init(const GemmParams& p, const int* off, const int* tile) {
    s_off = off;
    s_tile = tile;
    rank = (CN > 1) ? static_cast<int>(blockIdx.x % CN) : 0;
    first = static_cast<int>(blockIdx.x / CN);
    stride = static_cast<int>(gridDim.x / CN);
    ntiles = (p.N + kColsPerTile - 1) / kColsPerTile;
    mtiles = PAIR ? (p.M + 2 * BM - 1) / (2 * BM) : (p.M + BM - 1) / BM;
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
      const int mt_g = (rows_g + kRowsPerTile - 1) / kRowsPerTile;
      const int l = t - s_tile[g];
      const int mt = l % mt_g, nt = PAIR ? l / mt_g : (l / mt_g) * CN + rank;
      tl.g = g;
      tl.m0 = PAIR ? mt * 2 * BM + BM * rank : mt * BM;  // a pair: rows past the group read as absent
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
      tl.m0 = PAIR ? mt * 2 * BM + BM * rank : mt * BM;
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

// A (tile, k-stage) position of the persistent loop; only tiles with a non-empty reduction have stages.
struct Pos {
  int t, ks, nk;
  Tile tl;
};

template <class S>
__device__ __forceinline__ void pos_next(const S& sch, const GemmParams& p, int& gcur, Pos& q) {
  if (q.ks + 1 < q.nk) {
    ++q.ks;
    return;
  }
  q.ks = 0;
  for (q.t += sch.stride; q.t < sch.total; q.t += sch.stride) {
    sch.decode(p, q.t, gcur, q.tl);
    q.nk = (q.tl.k_len + BK - 1) / BK;
    if (q.nk > 0) return;
  }
}

template <class S>
__device__ __forceinline__ Pos pos_first(const S& sch, const GemmParams& p, int& gcur) {
  Pos q;
  q.t = sch.first - sch.stride;
  q.ks = 0;
  q.nk = 0;
  pos_next(sch, p, gcur, q);
  return q;
}

// Byte offset of the 16-byte piece (row r, piece c16) of a 128-byte-swizzled [rows x 128 B] block.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c16) {
  return static_cast<uint32_t>(r * 128 + ((c16 ^ (r & 7)) << 4));
}

// -------------------------------------------------------------------------- epilogue helpers

// Direct per-thread store of 32 consecutive columns of one row (used for a partial 32-row block).
__device__ __forceinline__ void store_row32(void* base, long long elem_off, const float (&v)[32], int ncols, bool fp32) {
  if (fp32) {
    float* o = reinterpret_cast<float*>(base) + elem_off;
    if (ncols >= 32) {
#pragma unroll
      for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
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

__device__ __forceinline__ void load_f32_row32(const float* src, float (&v)[32], int ncols) {
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

// Write this thread's 32 values as row r of the warp's staging block, in the swizzled layout of
// the store map: fp32 rows of 128 B (128-byte swizzle), bf16 rows of 64 B (64-byte swizzle).
__device__ __forceinline__ void stage_row32(uint8_t* stg, int r, const float (&v)[32], bool fp32) {
  if (fp32) {
    uint8_t* row = stg + r * 128;
#pragma unroll
    for (int p = 0; p < 8; ++p)
      *reinterpret_cast<float4*>(row + ((p ^ (r & 7)) << 4)) = make_float4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3]);
  } else {
    uint8_t* row = stg + r * 64;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      uint4 q;
      q.x = pack_bf16x2(v[8 * p], v[8 * p + 1]);
      q.y = pack_bf16x2(v[8 * p + 2], v[8 * p + 3]);
      q.z = pack_bf16x2(v[8 * p + 4], v[8 * p + 5]);
      q.w = pack_bf16x2(v[8 * p + 6], v[8 * p + 7]);
      *reinterpret_cast<uint4*>(row + ((p ^ ((r >> 1) & 3)) << 4)) = q;
    }
  }
}

// 64 bf16 values as one 128-byte row (128-byte swizzle).
__device__ __forceinline__ void stage_row64_bf16(uint8_t* stg, int r, const float (&v)[64]) {
  uint8_t* row = stg + r * 128;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    uint4 q;
    q.x = pack_bf16x2(v[8 * p], v[8 * p + 1]);
    q.y = pack_bf16x2(v[8 * p + 2], v[8 * p + 3]);
    q.z = pack_bf16x2(v[8 * p + 4], v[8 * p + 5]);
    q.w = pack_bf16x2(v[8 * p + 6], v[8 * p + 7]);
    *reinterpret_cast<uint4*>(row + ((p ^ (r & 7)) << 4)) = q;
  }
}

// Target of one epilogue store: a TMA map and coordinates for full 32-row blocks, a pointer
// and row offset for the direct path.
struct OutRef {
  const CUtensorMap* map;
  void* ptr;
  long long row_off;  // element offset of this thread's row (direct path)
  int c_row;          // TMA row coordinate of the warp's first row
  int c_z;            // TMA third coordinate (group / split), -1 = 2-D map
};

// -------------------------------------------------------------------------- the kernel

// Producer threads for a ring of `stages` with `spare` warps left: the largest of 4, 3, 2 that
// divides the stage count and fits, else 1.
__host__ __device__ constexpr int gemm_producers(int stages, int spare) {
  return (stages % 4 == 0 && spare >= 3)   ? 4
         : (stages % 3 == 0 && spare >= 2) ? 3
         : (stages % 2 == 0 && spare >= 1) ? 2
                                           : 1;
}

// Warp roles of one instantiation.  The gate/up GEMM gathers its A rows with 8 cp.async warps (the
// copy rate grows with the number of issuing warps: about 16, 25 and 33 B/ns per SM with 4, 8 and 16
// warps) and runs 512 threads, so its roles stay within 128 registers per thread.
template <int STAGES, int EW, int AMODE, int BMODE, int CN, int XF = 0>
struct WarpPlan {
  static constexpr bool kAGather = (AMODE == A_GATHER_K || AMODE == A_GATHER_MN);
  static constexpr bool kGather = kAGather || BMODE == B_GATHER_MN;
  static constexpr int kGW = (AMODE == A_GATHER_K) ? 8 : (kGather ? 4 : 0);  // gather warps
  static constexpr int kMaxWarps = (AMODE == A_GATHER_K) ? 16 : kMaxThreads / 32;
  static constexpr int kBase = EW + 2 + kGW + ((CN > 1 && !(XF & X_PAIR)) ? 1 : 0);  // + the relay warp
  static constexpr int kNP = gemm_producers(STAGES, kMaxWarps - kBase);
  static constexpr int kThreads = (kBase + kNP - 1) * 32;
};

template <int BN, int STAGES, int EW, int DEPTH, int AMODE, int BMODE, int VAR, int EPI, bool OUTF32, int CN = 1,
          int XF = 0>
__global__ void __launch_bounds__(WarpPlan<STAGES, EW, AMODE, BMODE, CN, XF>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ Maps mp) {
  using WP = WarpPlan<STAGES, EW, AMODE, BMODE, CN, XF>;
  constexpr bool kDual = (XF & X_DUAL_A) != 0;
  constexpr bool kTrans = (XF & X_TRANS) != 0;
  constexpr bool kPair = (XF & X_PAIR) != 0;
  constexpr bool kMx = (XF & X_MX) != 0;
  constexpr int kSfStage = mx_stage_bytes(BN, XF);
  using L = SmemLayout<BN, STAGES, EW, DEPTH, kDual ? 2 : 1, kPair ? BN / 2 : BN, kSfStage>;
  static_assert(EW == 4 || EW == 8, "4 or 8 epilogue warps");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert((EPI != EPI_SWIGLU && EPI != EPI_SWIGLU_Q) || BMODE == B_TMA_K3_GU,
                "SwiGLU epilogue needs the gate/up pair layout");
  // The e4m3 form moves 128-byte operand rows like the bf16 form: the host describes e4m3 rows to TMA
  // and to the gather as 16-bit units (two codes each), so K, the coordinates and the swizzled layout
  // are those of the bf16 form with K counted in code pairs; only the UMMA kind changes.
  constexpr bool kF8 =
      (EPI == EPI_SWIGLU_Q || EPI == EPI_SCALE_Q || EPI == EPI_STORE_Q || EPI == EPI_DSWIGLU_Q) || kMx;
  static_assert(!kMx || ((BN == 128 || BN == 192) && VAR == VAR_M && (AMODE == A_GATHER_K || AMODE == A_TMA_K) &&
                         (BMODE == B_TMA_K3 || BMODE == B_TMA_K3_GU) && (CN == 1 || CN == 2) &&
                         (EPI == EPI_SWIGLU || EPI == EPI_SCALE || EPI == EPI_STORE || EPI == EPI_DSWIGLU)) ||
                    ((BN == 128 || BN == 192) && VAR == VAR_K && AMODE == A_TMA_K && BMODE == B_TMA_K3 && CN == 1 &&
                     EPI == EPI_STORE),
                "block-scaled form: BN = 128 or 192, K-major operands, varlen-M plain epilogue kinds or a varlen-K store");
  static_assert(!kMx || 2 * BN + STAGES * (4 + 4 * mx_b_blocks(BN)) <= 512, "block-scaled form: TMEM columns");
  static_assert(EPI != EPI_STORE_Q || !OUTF32, "the e4m3 plain epilogue stores bf16");
  static_assert(!kF8 || ((AMODE == A_GATHER_K || AMODE == A_TMA_K) && (BMODE == B_TMA_K3 || BMODE == B_TMA_K3_GU) &&
                         (VAR == VAR_M || kMx)),
                "e4m3 form: K-major operands, varlen-M (the block-scaled form also varlen-K)");
  static_assert(!kDual || ((AMODE == A_TMA_MN || AMODE == A_TMA_K) && !kF8), "dual A: a tiled bf16 A");
  static_assert(!kTrans || (VAR == VAR_K && EPI == EPI_STORE), "transposed store: varlen-K plain epilogue");
  constexpr bool kAMn = (AMODE == A_TMA_MN || AMODE == A_GATHER_MN);
  constexpr bool kBMn = (BMODE == B_TMA_MN3 || BMODE == B_TMA_MN2 || BMODE == B_GATHER_MN);
  constexpr bool kAGather = (AMODE == A_GATHER_K || AMODE == A_GATHER_MN);
  constexpr bool kBGather = (BMODE == B_GATHER_MN);
  constexpr bool kGather = kAGather || kBGather;
  constexpr int kProdWarp = EW;        // TMA producer, owns TMEM
  constexpr int kMmaWarp = EW + 1;     // UMMA issuer
  constexpr int kGatherWarp0 = EW + 2; // cp.async gather warps when an operand is gathered
  constexpr int kGW = WP::kGW;
  constexpr int kRStep = kGW * 4;      // row stride between a gather thread's rows
  // Clusters of CN CTAs along N share the gathered A tile: each CTA gathers rows
  // [rank * kSlice, (rank + 1) * kSlice) and a relay thread copies them to the peers.
  static_assert(CN == 1 || (CN == 2 || CN == 4), "cluster of 1, 2 or 4");
  static_assert(CN == 1 || kPair || (AMODE == A_GATHER_K && VAR == VAR_M && !kBGather), "clusters share a gathered A");
  static_assert(!kPair || (CN == 2 && !kF8 && BN == 256 &&
                            ((VAR == VAR_K && AMODE == A_TMA_MN && BMODE == B_TMA_MN2) ||
                             (VAR == VAR_M && AMODE == A_TMA_K && (BMODE == B_TMA_K3 || BMODE == B_TMA_MN3)))),
                "CTA pair: BN = 256, tiled bf16 operands (varlen-K: MN-major A, chunked B; varlen-M: K-major A)");
  constexpr bool kRelay = (CN > 1) && !kPair;
  constexpr int kSlice = BM / CN;               // A rows gathered by each CTA of a cluster
  constexpr uint32_t kSliceBytes = kSlice * 128;
  constexpr int kRelayWarp = EW + 2 + kGW;
  // TMA loads issued by one thread complete one after another; stages are spread round-robin over
  // kNP producer threads (lane 0 of the producer warp and of kNP - 1 extra warps placed last), so
  // that several stages are in flight at once.  kNP divides STAGES: a stage always has the same
  // producer.
  constexpr int kNP = WP::kNP;
  constexpr int kXProdWarp0 = WP::kBase;  // extra producer warps
  constexpr int kThreads = WP::kThreads;
  static_assert(kThreads <= 512 && (kGW == 0 || kSlice % (kRStep > 0 ? kRStep : 1) == 0), "threads / gather rows");
  // a pair's even CTA expects both CTAs' loads on its barrier
  // (block-scaled form: the producer also brings B's scale block and, for a tiled A, A's)
  constexpr uint32_t kTxBytes =
      kPair ? 2 * (L::kABytes + L::kBBytes)
            : (kAGather ? (CN - 1) * kSliceBytes : L::kABytes) + (kBGather ? 0 : L::kBBytes) +
                  (kMx ? 512 * mx_b_blocks(BN) + 512 : 0);
  constexpr uint32_t kTmemCols = kMx ? 512 : (2 * BN <= 128) ? 128 : (2 * BN <= 256 ? 256 : 512);
  constexpr int kSfCols = 4 + 4 * mx_b_blocks(BN);  // TMEM columns of one stage's scales (A: 4, B: 4 per block)
  constexpr uint32_t kIdesc =
      kF8 ? idesc_e4m3(BM, BN, kAMn ? 1 : 0, kBMn ? 1 : 0) : idesc_bf16(kPair ? 2 * BM : BM, BN, kAMn ? 1 : 0, kBMn ? 1 : 0);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + STAGES;
  uint64_t* tfull_bar = bars + 2 * STAGES;
  uint64_t* tempty_bar = bars + 2 * STAGES + 2;
  uint64_t* drain_bar = bars + 2 * STAGES + 4;
  uint64_t* gath_bar = bars + 2 * STAGES + 5;  // [STAGES] own A slice gathered (relay mode)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::kMiscOffset);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kMiscOffset + 4);
  int* s_bad = reinterpret_cast<int*>(smem + L::kMiscOffset + 8);
  int* s_off_sm = reinterpret_cast<int*>(smem + L::kMiscOffset + 16);  // dense mode: {0, M}
  const int* s_off = (VAR == VAR_NONE) ? s_off_sm : p.offsets;
  int* s_tile = s_off_sm;  // varlen-M: first tile of every group, [groups + 1]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // relay mode: the producer's expect_tx and the relay's arrival; else the producer and,
      // with a gathered operand, the 128 gather threads
      mbar_init(&full_bar[s], kRelay ? 2 : 1 + (kGather ? kGW * 32 : 0));
      mbar_init(&empty_bar[s], kPair ? 1 : CN);  // every CTA of the cluster releases the stage (a pair: one UMMA commit)
      if (kRelay) mbar_init(&gath_bar[s], kGW * 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], (kPair ? 2 : 1) * EW * 32);  // a pair: both CTAs' epilogues drain the tile
    }
    mbar_init(drain_bar, 1);
    *s_abort = 0;
    *s_bad = 0;
    fence_mbar_init();
  }
  if (warp == kProdWarp) {
    if (!kPair) tmem_alloc(s_tmem, kTmemCols);  // a pair allocates collectively once both CTAs are up
    if (lane == 0) {
      if (!kAGather) tma_prefetch_desc(&mp.a0);
      if (!kBGather) tma_prefetch_desc(&mp.b0);
    }
  }
  // group offsets into shared memory (validated: start at 0, monotone, within capacity)
  if (VAR == VAR_NONE && tid == 0) {
    s_off_sm[0] = 0;
    s_off_sm[1] = p.M;
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
        if (kMx && VAR == VAR_K && (s_off[g] % BK) != 0) bad = 1;  // groups start on whole stages (and scale blocks)
        if (VAR == VAR_M) {
          // a pair: 256-row tiles, every column tile; clusters along N: CN column tiles per unit
          constexpr int kCpt = Sched<BN, BMODE, VAR>::kColsPerTile, kRpt = kPair ? 2 * BM : BM, kCn = kPair ? 1 : CN;
          cnt = max(0, (rows_g + kRpt - 1) / kRpt) * (((p.N + kCpt - 1) / kCpt + kCn - 1) / kCn);
        }
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (VAR == VAR_M && g < p.groups) s_tile[g] = running + incl - cnt;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (s_off[0] != 0 || s_off[p.groups] > p.rows_cap) bad = 1;
      if (VAR == VAR_M) s_tile[p.groups] = bad ? 0 : running;
      if (bad) {
        *s_bad = 1;
        set_error(p.err, DERR_BAD_OFFSETS);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (CN > 1) cluster_sync();  // the peers' barriers are initialised before anything targets them
  if (kPair) {
    if (warp == kProdWarp) tmem_alloc_pair(s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();
  }
  const uint32_t tmem_base = *s_tmem;
  const uint32_t cta_rank = kPair ? cluster_ctarank() : 0;

  Sched<BN, BMODE, VAR, CN, kPair> sch;
  sch.init(p, s_off, s_tile);
  // block-scaled form: row tiles before group g = s_tile[g] / column units per group (the tile order of every
  // varlen-M GEMM over the same offsets), which indexes the scale blocks of a tiled A and of the SwiGLU output
  const int mx_ncu = ((p.N + Sched<BN, BMODE, VAR>::kColsPerTile - 1) / Sched<BN, BMODE, VAR>::kColsPerTile + CN - 1) / CN;
  if (*s_bad) sch.total = 0;
  if (kPair && VAR == VAR_K && !p.b_offsets) {  // the varlen-K pair reads padded B rows only
    if (threadIdx.x == 0) set_error(p.err, DERR_BAD_OFFSETS);
    sch.total = 0;
  }

  if (warp == kProdWarp || (warp >= kXProdWarp0 && warp < kXProdWarp0 + kNP - 1)) {
    // ---------------------------------------------------------------- TMA producers (lane 0 each)
    const int pj = (warp == kProdWarp) ? 0 : warp - kXProdWarp0 + 1;  // this thread's stages: it % kNP == pj
    if (lane == 0) {
      // An expert's weight tile is read by the CTAs on the expert's row tiles at about the same
      // time: normal L2 priority lets the later ones hit (evict-first measured up to 25% slower).
      const uint64_t pol_stream = l2_policy_evict_normal();
      // Loads (or, with l2 = true, L2 prefetches) of the tiled operands of one stage.
      auto tiled = [&](const Tile& x, int kstage, uint8_t* sa, uint8_t* sb, uint64_t* bar, bool l2) {
        const int kg = x.k_begin + kstage * BK;
        if (kPair) {
          // this CTA's 128 rows of the pair's M = 256 tile (x.m0 carries the rank) and its half of B's
          // columns (the host's B boxes are half as wide); every copy completes on the even CTA's full barrier
          const uint32_t lb = l2 ? 0u : pair_leader_addr(bar);
          const int rk = static_cast<int>(cta_rank);
          if (AMODE == A_TMA_K) {
            const int row = (p.a_offsets ? __ldg(p.a_offsets + x.g) : s_off[x.g]) + x.m0;
            const bool first = kg < p.a_ksplit;
            const int kc = first ? kg : kg - p.a_ksplit;
            if (l2) {
              tma_prefetch_l2_2d(first ? &mp.a0 : &mp.a1, kc, row);
              if (kDual) tma_prefetch_l2_2d(first ? &mp.a2 : &mp.a3, kc, row);
            } else {
              tma_load_2d_pair(sa, first ? &mp.a0 : &mp.a1, lb, kc, row);
              if (kDual) tma_load_2d_pair(sa + L::kA1Bytes, first ? &mp.a2 : &mp.a3, lb, kc, row);
            }
          } else {
            const int ka = kg >= p.a_kwrap ? kg - p.a_kwrap : kg;
#pragma unroll
            for (int c = 0; c < BM / 64; ++c) {
              const int col = x.m0 + 64 * c;
              const bool first = col < p.a_colsplit;
              const int cc = first ? col : col - p.a_colsplit;
              if (l2) {
                tma_prefetch_l2_2d(first ? &mp.a0 : &mp.a1, cc, ka);
                if (kDual) tma_prefetch_l2_2d(first ? &mp.a2 : &mp.a3, cc, ka);
              } else {
                tma_load_2d_pair(sa + c * (BK * 128), first ? &mp.a0 : &mp.a1, lb, cc, ka);
                if (kDual) tma_load_2d_pair(sa + L::kA1Bytes + c * (BK * 128), first ? &mp.a2 : &mp.a3, lb, cc, ka);
              }
            }
          }
          if (BMODE == B_TMA_K3) {  // 3-D weights {K, N, groups}: BN / 2 rows of N
            const int n = x.n0 + (BN / 2) * rk;
            if (l2) tma_prefetch_l2_3d(&mp.b0, kg, n, x.g);
            else tma_load_3d_pair(sb, &mp.b0, lb, kg, n, x.g);
          } else if (BMODE == B_TMA_MN3) {  // 4-D view {64 columns, K rows, N/64 chunks, groups}: BN / 128 chunks
            const bool first = kg < p.b_ksplit;
            const int kc = first ? kg : kg - p.b_ksplit;
            const int chunk = x.n0 / 64 + (BN / 128) * rk;
            if (l2) tma_prefetch_l2_4d(first ? &mp.b0 : &mp.b1, 0, kc, chunk, x.g);
            else tma_load_4d_pair(sb, first ? &mp.b0 : &mp.b1, lb, 0, kc, chunk, x.g);
          } else {
            // padded B rows: the group's reduction rows start at b_offsets[g]; 3-D view {64 columns, rows,
            // N/64 chunks} with boxes of BN/128 chunks
            const int kgb = __ldg(p.b_offsets + x.g) + kstage * BK;
            const int chunk = x.n0 / 64 + (BN / 128) * rk;
            if (l2) tma_prefetch_l2_3d(&mp.b0, 0, kgb, chunk);
            else tma_load_3d_pair(sb, &mp.b0, lb, 0, kgb, chunk);
          }
          return;
        }
        if (AMODE == A_TMA_K) {
          const int row = (VAR == VAR_M ? (p.a_offsets ? __ldg(p.a_offsets + x.g) : s_off[x.g]) : 0) + x.m0;
          const CUtensorMap* mp_a = kg < p.a_ksplit ? &mp.a0 : &mp.a1;
          const int kc = kg < p.a_ksplit ? kg : kg - p.a_ksplit;
          if (l2) tma_prefetch_l2_2d(mp_a, kc, row);
          else tma_load_2d(sa, mp_a, bar, kc, row);
          if (kDual) {  // the low part, same coordinates, into the stage's second A tile
            const CUtensorMap* mp_l = kg < p.a_ksplit ? &mp.a2 : &mp.a3;
            if (l2) tma_prefetch_l2_2d(mp_l, kc, row);
            else tma_load_2d(sa + L::kA1Bytes, mp_l, bar, kc, row);
          }
        } else if (AMODE == A_TMA_MN) {
#pragma unroll
          for (int c = 0; c < BM / 64; ++c) {
            const int col = x.m0 + 64 * c;
            const bool first = col < p.a_colsplit;
            const CUtensorMap* mp_a = first ? &mp.a0 : &mp.a1;
            const int cc = first ? col : col - p.a_colsplit;
            const int ka = kg >= p.a_kwrap ? kg - p.a_kwrap : kg;
            if (l2) tma_prefetch_l2_2d(mp_a, cc, ka);
            else tma_load_2d(sa + c * (BK * 128), mp_a, bar, cc, ka);
            if (kDual) {  // the low part, same coordinates, into the stage's second A tile
              const CUtensorMap* mp_l = first ? &mp.a2 : &mp.a3;
              if (l2) tma_prefetch_l2_2d(mp_l, cc, ka);
              else tma_load_2d(sa + L::kA1Bytes + c * (BK * 128), mp_l, bar, cc, ka);
            }
          }
        }
        if (kMx && !l2) {
          // the stage's scale blocks: A's (its row tile's block for this stage of K, tiled or gathered rows
          // alike), then B's (a cluster CTA past the last column tile loads the last tile's block; its results
          // are not stored)
          uint8_t* sf = sb + L::kBBytes;
          const int nt = min(x.nt, sch.ntiles - 1);
          constexpr int kSfb = 512 * mx_b_blocks(BN);
          if (VAR == VAR_K) {
            // varlen-K: both operands' blocks are indexed by the stage of the whole (padded) reduction, every
            // group starting on a whole stage: A's [row tile][stage], B's [column tile][stage]
            const long long kgl = x.k_begin / BK + kstage;
            bulk_load(sf, p.a_sf + ((x.m0 / BM) * static_cast<long long>(p.sf_kst) + kgl) * 512, 512, bar);
            bulk_load(sf + 512, p.b_sf + (static_cast<long long>(nt) * p.sf_kst + kgl) * kSfb, kSfb, bar);
          } else {
            const long long rt = s_tile[x.g] / mx_ncu + x.m0 / BM;
            bulk_load(sf, p.a_sf + (rt * p.sf_kst + kstage) * 512, 512, bar);
            bulk_load(sf + 512, p.b_sf + ((static_cast<long long>(x.g) * sch.ntiles + nt) * p.sf_kst + kstage) * kSfb,
                      kSfb, bar);
          }
        }
        if (BMODE == B_TMA_K3) {  // varlen-K: one [N][K] matrix, the group's reduction rows along K
          const int bz = (VAR == VAR_K) ? 0 : x.g;
          if (l2) tma_prefetch_l2_3d(&mp.b0, kg, x.n0, bz);
          else tma_load_3d_hint(sb, &mp.b0, bar, kg, x.n0, bz, pol_stream);
        } else if (BMODE == B_TMA_K3_GU) {
          if (l2) {
            tma_prefetch_l2_3d(&mp.b0, kg, x.n0, x.g);
            tma_prefetch_l2_3d(&mp.b1, kg, x.n0, x.g);
          } else {
            tma_load_3d_hint(sb, &mp.b0, bar, kg, x.n0, x.g, pol_stream);
            tma_load_3d_hint(sb + (BN / 2) * 128, &mp.b1, bar, kg, x.n0, x.g, pol_stream);
          }
        } else if (BMODE == B_TMA_MN3) {
          // 4-D view {64 columns, K rows, N/64 chunks, groups}: every 64-column chunk of the stage in one box
          const bool first = kg < p.b_ksplit;
          const int kc = first ? kg : kg - p.b_ksplit;
          if (l2) tma_prefetch_l2_4d(first ? &mp.b0 : &mp.b1, 0, kc, x.n0 / 64, x.g);
          else tma_load_4d_hint(sb, first ? &mp.b0 : &mp.b1, bar, 0, kc, x.n0 / 64, x.g, pol_stream);
        } else if (BMODE == B_TMA_MN2) {
          // varlen-K with padded B rows: the group's reduction rows start at b_offsets[g] in B
          const int kgb = (VAR == VAR_K && p.b_offsets) ? __ldg(p.b_offsets + x.g) + kstage * BK : kg;
          if (p.b_chunked) {  // 3-D view {64 columns, rows, N/64 chunks}
            if (l2) tma_prefetch_l2_3d(&mp.b0, 0, kgb, x.n0 / 64);
            else tma_load_3d(sb, &mp.b0, bar, 0, kgb, x.n0 / 64);
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c) {
              if (l2) tma_prefetch_l2_2d(&mp.b0, x.n0 + 64 * c, kgb);
              else tma_load_2d(sb + c * (BK * 128), &mp.b0, bar, x.n0 + 64 * c, kgb);
            }
          }
        }
      };
      int it = 0, gcur = 0;
      bool aborted = false;
      Pos q = pos_first(sch, p, gcur);
      while (q.t < sch.total && !aborted) {
        if (it % kNP != pj) {  // another producer's stage
          ++it;
          pos_next(sch, p, gcur, q);
          continue;
        }
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!mbar_wait(&empty_bar[s], ph ^ 1, s_abort, p.timeout_ns, p.err)) {
          aborted = true;
          break;
        }
        uint8_t* sa = smem + s * L::kStageBytes;
        uint8_t* sb = sa + L::kABytes;
        if (kTxBytes > 0) {
          if (!kPair || cta_rank == 0) mbar_arrive_expect_tx(&full_bar[s], kTxBytes);
          tiled(q.tl, q.ks, sa, sb, &full_bar[s], false);
          // L2 prefetch of the stages ahead of this one within the tile
          if (!p.l2_prefetch) {
          } else if (q.ks == 0) {
            for (int k2 = 1; k2 <= kPrefetchStages && k2 < q.nk; ++k2) tiled(q.tl, k2, sa, sb, nullptr, true);
          } else if (q.ks + kPrefetchStages < q.nk) {
            tiled(q.tl, q.ks + kPrefetchStages, sa, sb, nullptr, true);
          }
        } else {
          mbar_arrive(&full_bar[s]);
        }
        ++it;
        pos_next(sch, p, gcur, q);
      }
      if (aborted && kPair) {
        // the copies count on the even CTA's barriers: give those in flight 20 ms to land
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 20000000ull) {
        }
      } else if (aborted) {
        // let this thread's copies already in flight land before the CTA goes away
        volatile int never = 0;
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          if (j % kNP == pj) mbar_wait(&full_bar[j % STAGES], (j / STAGES) & 1, &never, 20000000ull, nullptr);
      } else if (CN > 1) {
        // every CTA's release of this thread's last stages has arrived here, so no peer still
        // targets this CTA's barriers when it leaves
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          if (j % kNP == pj) mbar_wait(&empty_bar[j % STAGES], (j / STAGES) & 1, s_abort, p.timeout_ns, p.err);
      }
    }
  } else if (kGather && warp >= kGatherWarp0 && warp < kGatherWarp0 + kGW) {
    // ---------------------------------------------------------------- cp.async gather producers
    // Thread ptid owns the 16-byte piece c16 of rows rsub + kRStep i of every stage.  The token
    // indices of a position are loaded two positions ahead of its copies.
    const int ptid = tid - kGatherWarp0 * 32;
    const int c16 = ptid & 7;
    const int rsub = ptid >> 3;
    constexpr int kRowsPer = kSlice / (kRStep > 0 ? kRStep : 1);  // A rows per thread and stage
    const int slice0 = sch.rank * kSlice;  // first tile row gathered by this CTA
    const uint64_t pol_keep = l2_policy_evict_last();  // gathered rows are re-read by many tiles
    auto fetch = [&](const Pos& x, int (&r)[8], const Pos& prev, const int (&pr)[8]) {
      if (AMODE == A_GATHER_K) {
        if (x.t == prev.t) {
#pragma unroll
          for (int i = 0; i < kRowsPer; ++i) r[i] = pr[i];
        } else {
#pragma unroll
          for (int i = 0; i < kRowsPer; ++i) {
            const int rr = slice0 + rsub + kRStep * i;
            r[i] = rr < x.tl.rows ? __ldg(p.a_idx + s_off[x.tl.g] + x.tl.m0 + rr) : -1;
          }
        }
      } else {
        const int* idx = kAGather ? p.a_idx : p.b_idx;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kr = x.ks * BK + rsub + 16 * j;
          r[j] = kr < x.tl.k_len ? __ldg(idx + x.tl.k_begin + kr) : -1;
        }
      }
    };
    int it = 0, gcur = 0;
    bool aborted = false;
    int r0[8], r1[8], r2[8];
    Pos q0 = pos_first(sch, p, gcur), q1 = q0, q2 = q0;
    Pos none;
    none.t = -1;
    if (q0.t < sch.total) fetch(q0, r0, none, r0);
    pos_next(sch, p, gcur, q1);
    if (q1.t < sch.total) fetch(q1, r1, q0, r0);
    q2 = q1;
    pos_next(sch, p, gcur, q2);
    if (q2.t < sch.total) fetch(q2, r2, q1, r1);
    while (q0.t < sch.total && !aborted) {
      const int s = it % STAGES;
      const uint32_t ph = (it / STAGES) & 1;
      if (!mbar_wait(&empty_bar[s], ph ^ 1, s_abort, p.timeout_ns, p.err)) {
        aborted = true;
        break;
      }
      const uint32_t sa = smem_u32(smem + s * L::kStageBytes);
      const uint32_t sb = sa + L::kABytes;
      if (AMODE == A_GATHER_K) {
        const int kc = q0.tl.k_begin + q0.ks * BK + c16 * 8;
        const bool k_in = kc < p.K;  // a last stage past K (K a multiple of 8 units) reads zeros
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
          const long long row = r0[i];
          bool ok = row >= 0 && k_in;
          if (ok && row >= p.a_rows) {
            set_error(p.err, DERR_BAD_OFFSETS);
            ok = false;
          }
          cp_async_16_hint(sa + sw128_offset(slice0 + rsub + kRStep * i, c16), ok ? p.a_src + row * p.a_ld + kc : p.a_src,
                           ok ? 16u : 0u, pol_keep);
        }
      } else if (AMODE == A_GATHER_MN) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int chunk = i >> 2, j = i & 3;
          const int col = q0.tl.m0 + 64 * chunk + c16 * 8;
          const long long row = r0[j];
          bool ok = row >= 0 && col < p.M;
          if (ok && row >= p.a_rows) {
            set_error(p.err, DERR_BAD_OFFSETS);
            ok = false;
          }
          cp_async_16_hint(sa + chunk * (BK * 128) + sw128_offset(rsub + 16 * j, c16),
                           ok ? p.a_src + row * p.a_ld + col : p.a_src, ok ? 16u : 0u, pol_keep);
        }
      }
      if (BMODE == B_GATHER_MN) {
#pragma unroll
        for (int i = 0; i < 4 * (BN / 64); ++i) {
          const int chunk = i >> 2, j = i & 3;
          const int col = q0.tl.n0 + 64 * chunk + c16 * 8;
          const long long row = r0[j];
          bool ok = row >= 0 && col < p.N;
          if (ok && row >= p.b_rows) {
            set_error(p.err, DERR_BAD_OFFSETS);
            ok = false;
          }
          cp_async_16_hint(sb + chunk * (BK * 128) + sw128_offset(rsub + 16 * j, c16),
                           ok ? p.b_src + row * p.b_ld + col : p.b_src, ok ? 16u : 0u, pol_keep);
        }
      }
      cp_async_mbar_arrive_noinc(kRelay ? &gath_bar[s] : &full_bar[s]);
      ++it;
      // rotate the index pipeline
      q0 = q1;
      q1 = q2;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        r0[i] = r1[i];
        r1[i] = r2[i];
      }
      if (q2.t < sch.total) {
        const Pos prev = q2;
        pos_next(sch, p, gcur, q2);
        if (q2.t < sch.total) fetch(q2, r2, prev, r1);
      }
    }
    cp_async_wait_all();
  } else if (kRelay && warp == kRelayWarp) {
    // ---------------------------------------------------------------- relay (one thread)
    // Once this CTA's slice of a stage has landed, make it visible to the async proxy, copy it
    // into the same stage of every peer (completing bytes on the peer's full barrier) and mark
    // it ready here.  The peers' stage is free: this CTA's gather warps waited on the stage's
    // empty barrier, which every CTA of the cluster releases.
    if (lane == 0) {
      const uint32_t me = cluster_ctarank();
      int it = 0, gcur = 0;
      Pos q = pos_first(sch, p, gcur);
      while (q.t < sch.total) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!mbar_wait(&gath_bar[s], ph, s_abort, p.timeout_ns, p.err)) break;
        fence_proxy_async_smem();
        const uint32_t src = smem_u32(smem + s * L::kStageBytes) + me * kSliceBytes;
        const uint32_t fb = smem_u32(&full_bar[s]);
#pragma unroll
        for (int r = 1; r < CN; ++r) {
          const uint32_t peer = (me + r) % CN;
          bulk_copy_to_peer(mapa_shared(src, peer), src, kSliceBytes, mapa_shared(fb, peer));
        }
        mbar_arrive(&full_bar[s]);
        ++it;
        pos_next(sch, p, gcur, q);
      }
    }
  } else if (warp == kMmaWarp && (!kPair || cta_rank == 0)) {
    // ---------------------------------------------------------------- UMMA issuer (lane 0)
    // (a pair: the even CTA's, for both CTAs)
    // With both operands tiled in the varlen-K mode, the last stage of a group reads rows of the
    // next group (or the zeroed tail): its UMMAs stop at the K step (16 rows) that holds the group's
    // last row, and the whole warp clears the rows of that step past the group's end in B before
    // lane 0 issues them.
    constexpr bool kZeroTail = (VAR == VAR_K) && !kGather && !kMx;  // block-scaled groups are whole stages
    if (!kZeroTail) {
      // lane 0 alone: no warp-wide step between a stage's arrival and its UMMAs
      if (lane == 0) {
        int it = 0, acc = 0, gcur = 0;
        bool aborted = false;
        for (int t = sch.first; t < sch.total && !aborted; t += sch.stride, ++acc) {
          Tile tl;
          sch.decode(p, t, gcur, tl);
          const int nk = (tl.k_len + BK - 1) / BK;
          const int buf = acc & 1;
          // a pair: the odd CTA's epilogue released the accumulator with cluster-scope arrivals
          if (!(kPair ? mbar_wait_cluster(&tempty_bar[buf], ((acc >> 1) & 1) ^ 1, s_abort, p.timeout_ns, p.err)
                      : mbar_wait(&tempty_bar[buf], ((acc >> 1) & 1) ^ 1, s_abort, p.timeout_ns, p.err)))
            break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          for (int ks = 0; ks < nk; ++ks, ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            if (!mbar_wait(&full_bar[s], ph, s_abort, p.timeout_ns, p.err)) {
              aborted = true;
              break;
            }
            const uint32_t sa = smem_u32(smem + s * L::kStageBytes);
            const uint32_t sb = sa + L::kABytes;
            if (kGather) fence_proxy_async_smem();  // cp.async writes -> UMMA operand reads
            tc_fence_after();
            // block-scaled form: this stage's scale blocks into its own TMEM columns (their previous readers, the
            // UMMAs of the stage's last use, completed before the stage was refilled); tcgen05.cp and the UMMAs
            // after it run in issue order
            const uint32_t sf_t = tmem_base + 2 * BN + s * kSfCols;
            if (kMx) {
              const uint32_t sf_s = sb + L::kBBytes;
              tmem_cp_32x128b_x4(sf_t, sdesc_plain(sf_s, 128, 128));
#pragma unroll
              for (int a = 0; a < mx_b_blocks(BN); ++a)
                tmem_cp_32x128b_x4(sf_t + 4 + 4 * a, sdesc_plain(sf_s + 512 + 512 * a, 128, 128));
            }
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad =
                  kAMn ? sdesc_sw128(sa + kk * 2048, BK * 128, 1024) : sdesc_sw128(sa + kk * 32, 16, 1024);
              const uint64_t bd =
                  kBMn ? sdesc_sw128(sb + kk * 2048, BK * 128, 1024) : sdesc_sw128(sb + kk * 32, 16, 1024);
              // dual A: the low part of A times the same B, into the same accumulator
              const uint64_t adl = kAMn ? sdesc_sw128(sa + L::kA1Bytes + kk * 2048, BK * 128, 1024)
                                        : sdesc_sw128(sa + L::kA1Bytes + kk * 32, 16, 1024);
              if (kMx) {  // K step kk = 32-code block kk of the stage: byte kk of every scale word
                umma_mx(d_tmem, ad, bd, idesc_mx(BM, BN, 0, 0, kk, kk), sf_t, sf_t + 4, (ks | kk) != 0 ? 1u : 0u);
              } else if (kPair) {  // same offsets in both CTAs: each holds its rows of A and its columns of B
                umma_bf16_pair(d_tmem, ad, bd, kIdesc, (ks | kk) != 0 ? 1u : 0u);
                if (kDual) umma_bf16_pair(d_tmem, adl, bd, kIdesc, 1u);
              } else {
                umma_step<kF8>(d_tmem, ad, bd, kIdesc, (ks | kk) != 0 ? 1u : 0u);
                if (kDual) umma_step<kF8>(d_tmem, adl, bd, kIdesc, 1u);
              }
            }
            if (kPair) umma_commit_pair_mc(&empty_bar[s], 3);  // both CTAs' stage s is free
            else if (CN > 1) umma_commit_mc(&empty_bar[s], static_cast<uint16_t>((1u << CN) - 1u));
            else umma_commit(&empty_bar[s]);
          }
          if (aborted) break;
          if (kPair) umma_commit_pair_mc(&tfull_bar[buf], 3);  // both CTAs' halves of the accumulator are ready
          else umma_commit(&tfull_bar[buf]);
        }
        if (*s_abort) {
          if (kPair) umma_commit_pair_mc(drain_bar, 1);
          else umma_commit(drain_bar);
          volatile int never = 0;
          mbar_wait(drain_bar, 0, &never, 20000000ull, nullptr);
        }
      }
    } else {
    int it = 0, acc = 0, gcur = 0;
    bool aborted = false;
    for (int t = sch.first; t < sch.total && !aborted; t += sch.stride, ++acc) {
      Tile tl;
      sch.decode(p, t, gcur, tl);
      const int nk = (tl.k_len + BK - 1) / BK;
      const int buf = acc & 1;
      // lane 0 waits, the warp follows its verdict (the other lanes block in the shuffle)
      int ok = 0;
      if (lane == 0)  // a pair: the odd CTA's epilogue released it with cluster-scope arrivals
        ok = kPair ? mbar_wait_cluster(&tempty_bar[buf], ((acc >> 1) & 1) ^ 1, s_abort, p.timeout_ns, p.err)
                   : mbar_wait(&tempty_bar[buf], ((acc >> 1) & 1) ^ 1, s_abort, p.timeout_ns, p.err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      for (int ks = 0; ks < nk; ++ks, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        ok = 0;
        if (lane == 0) ok = mbar_wait(&full_bar[s], ph, s_abort, p.timeout_ns, p.err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          aborted = true;
          break;
        }
        const uint32_t sa = smem_u32(smem + s * L::kStageBytes);
        const uint32_t sb = sa + L::kABytes;
        int nkk = BK / 16;  // UMMA K steps of this stage
        if (kZeroTail) {
          const int kv = tl.k_len - ks * BK;  // valid rows of this stage
          if (kv < BK) {
            // the group's last stage stops at the K step that holds its last row; only the rows of that
            // step past the group's end are cleared
            nkk = (kv + 15) / 16;
            const int kend = nkk * 16;
            if (kv < kend && !p.b_offsets) {  // padded B rows are zero there already
              uint8_t* b_gen = smem + s * L::kStageBytes + L::kABytes;
              const int pieces = (kend - kv) * 8;
              for (int c = 0; c < BN / 64; ++c)
                for (int i = lane; i < pieces; i += 32)
                  *reinterpret_cast<uint4*>(b_gen + c * (BK * 128) + (kv + (i >> 3)) * 128 + (i & 7) * 16) =
                      make_uint4(0, 0, 0, 0);
              fence_proxy_async_smem();
              __syncwarp();
            }
          }
        }
        if (lane == 0) {
          if (kGather) fence_proxy_async_smem();  // cp.async writes -> UMMA operand reads
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk >= nkk) break;
            const uint64_t ad = kAMn ? sdesc_sw128(sa + kk * 2048, BK * 128, 1024) : sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = kBMn ? sdesc_sw128(sb + kk * 2048, BK * 128, 1024) : sdesc_sw128(sb + kk * 32, 16, 1024);
            // dual A: the low part times the same B, into the same accumulator
            const uint64_t adl = kAMn ? sdesc_sw128(sa + L::kA1Bytes + kk * 2048, BK * 128, 1024)
                                      : sdesc_sw128(sa + L::kA1Bytes + kk * 32, 16, 1024);
            if (kPair) {  // same offsets in both CTAs' shared memory: each holds its rows of A, its columns of B
              umma_bf16_pair(d_tmem, ad, bd, kIdesc, (ks | kk) != 0 ? 1u : 0u);
              if (kDual) umma_bf16_pair(d_tmem, adl, bd, kIdesc, 1u);
            } else {
              umma_step<kF8>(d_tmem, ad, bd, kIdesc, (ks | kk) != 0 ? 1u : 0u);
              if (kDual) umma_step<kF8>(d_tmem, adl, bd, kIdesc, 1u);
            }
          }
          if (kPair) umma_commit_pair_mc(&empty_bar[s], 3);  // both CTAs' stage s is free
          else if (CN > 1) umma_commit_mc(&empty_bar[s], static_cast<uint16_t>((1u << CN) - 1u));
          else umma_commit(&empty_bar[s]);
        }
        __syncwarp();
      }
      if (aborted) break;
      if (lane == 0) {
        if (kPair) umma_commit_pair_mc(&tfull_bar[buf], 3);  // both CTAs' halves of the accumulator are ready
        else umma_commit(&tfull_bar[buf]);
      }
      __syncwarp();
    }
    if (aborted && lane == 0) {
      if (kPair) umma_commit_pair_mc(drain_bar, 1);
      else umma_commit(drain_bar);
      volatile int never = 0;
      mbar_wait(drain_bar, 0, &never, 20000000ull, nullptr);
    }
    }
  } else if (warp < EW) {
    // ---------------------------------------------------------------- epilogue (warps 0..EW-1)
    // Warp w reads TMEM lanes 32 (w % 4) .. +31 (its 32 rows) and, with 8 warps, one half of
    // the tile's columns (w / 4).  Results leave through a ring of DEPTH staged TMA stores.
    const int quarter = warp & 3;
    const int half = (EW == 8) ? (warp >> 2) : 0;
    uint8_t* stg_base = smem + L::kStgOffset + warp * (DEPTH * kStgBuf);
    int stg_i = 0;
    int acc = 0, gcur = 0;
    const int row_local = quarter * 32 + lane;
    auto next_stage_buf = [&]() -> uint8_t* {
      uint8_t* stg = stg_base + (stg_i % DEPTH) * kStgBuf;
      ++stg_i;
      if (lane == 0) bulk_wait_read<DEPTH - 1>();  // the store that last used this buffer has read it
      __syncwarp();
      return stg;
    };
    auto issue_store = [&](const OutRef& o, const uint8_t* stg, int col) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (o.c_z < 0) tma_store_2d(o.map, stg, col, o.c_row);
        else tma_store_3d(o.map, stg, col, o.c_row, o.c_z);
        bulk_commit();
      }
    };
    // 32 columns (fp32, or bf16 through a 64-byte-swizzled box)
    auto emit32 = [&](const OutRef& o, const float (&v)[32], int col, int ncols, bool full, bool row_ok, bool fp32) {
      if (ncols <= 0) return;
      if (full) {
        uint8_t* stg = next_stage_buf();
        stage_row32(stg, lane, v, fp32);
        issue_store(o, stg, col);
      } else if (row_ok) {
        store_row32(o.ptr, o.row_off + col, v, ncols, fp32);
      }
    };
    // 64 bf16 columns through one 128-byte-swizzled box
    auto emit64 = [&](const OutRef& o, const float (&v)[64], int col, int ncols, bool full, bool row_ok) {
      if (ncols <= 0) return;
      if (full) {
        uint8_t* stg = next_stage_buf();
        stage_row64_bf16(stg, lane, v);
        issue_store(o, stg, col);
      } else if (row_ok) {
        float lo[32], hi[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          lo[i] = v[i];
          hi[i] = v[32 + i];
        }
        store_row32(o.ptr, o.row_off + col, lo, ncols, false);
        if (ncols > 32) store_row32(o.ptr, o.row_off + col + 32, hi, ncols - 32, false);
      }
    };
    for (int t = sch.first; t < sch.total; t += sch.stride, ++acc) {
      Tile tl;
      sch.decode(p, t, gcur, tl);
      const int buf = acc & 1;
      if (!mbar_wait(&tfull_bar[buf], (acc >> 1) & 1, s_abort, p.timeout_ns, p.err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * BN;
      const bool row_ok = row_local < tl.rows;
      // a 32-row block goes out by TMA when all of its rows belong to this output
      const bool full = (VAR == VAR_M) ? (quarter * 32 + 32 <= tl.rows) : true;
      const bool have_acc = tl.k_len > 0;
      constexpr int kCols = (EW == 8) ? BN / 2 : BN;  // accumulator columns handled by this warp
      const int c_lo = half * kCols;

      if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_Q || EPI == EPI_SCALE || EPI == EPI_SCALE_Q || EPI == EPI_DSWIGLU ||
          EPI == EPI_DSWIGLU_Q) {
        const long long orow = s_off[tl.g] + tl.m0 + row_local;
        const int crow = s_off[tl.g] + tl.m0 + quarter * 32;
        const long long roff = orow * p.ld_out;
        const OutRef o0{&mp.o0, p.out0, roff, crow, -1}, o1{&mp.o1, p.out1, roff, crow, -1},
            o2{&mp.o2, p.out2, roff, crow, -1};
        const OutRef o3{&mp.o3, p.out3, roff, crow, -1}, o4{&mp.o4, p.out4, roff, crow, -1},
            o5{&mp.o5, p.out5, roff, crow, -1};
        if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_Q) {
          // columns [0, BN/2) hold h, [BN/2, BN) hold u of the same output columns
          constexpr int kHalf = (EW == 8) ? BN / 4 : BN / 2;
          float sx = 1.0f;  // e4m3 form: the scale of the row's token (an empty slot's row gets 0)
          if (EPI == EPI_SWIGLU_Q && row_ok) {
            const int tok = __ldg(p.a_idx + orow);
            sx = (tok >= 0 && tok < p.a_rows) ? __ldg(p.row_scale + tok) : 0.0f;
          }
#pragma unroll 1
          for (int c = half * kHalf; c < (half + 1) * kHalf; c += 32) {
            uint32_t rh[32], ru[32];
            tmem_ld32(tbase + c, rh);
            tmem_ld32(tbase + BN / 2 + c, ru);
            tmem_ld_wait();
            const int col = tl.n0 + c;
            const int ncols = p.N - col;
            float h[32], u[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              h[i] = __uint_as_float(rh[i]);
              u[i] = __uint_as_float(ru[i]);
            }
            if (EPI == EPI_SWIGLU_Q) {
              // lane i holds the scales of column col + i; the warp's rows share them by shuffle
              const long long so = static_cast<long long>(tl.g) * p.ld_in + col + lane;
              const float gl = lane < ncols ? __ldg(p.in0 + so) : 0.0f;
              const float ul = lane < ncols ? __ldg(p.in1 + so) : 0.0f;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                h[i] *= sx * __shfl_sync(0xffffffffu, gl, i);
                u[i] *= sx * __shfl_sync(0xffffffffu, ul, i);
              }
            }
            if (p.out0) {  // H, U stay fp32 for the backward; a forward-only call passes neither
              emit32(o0, h, col, ncols, full, row_ok, true);
              emit32(o1, u, col, ncols, full, row_ok, true);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = h[i] * sigmoidf_(h[i]) * u[i];  // A, in place of h
            if (kMx) {
              // A as block-scaled e4m3: this row's 32 columns are one block; its codes go straight to A's rows,
              // its scale byte into the row tile's scale block for the down projection (stage col / 128, byte
              // (col / 32) % 4); a row's last stage past n holds scale 1 (byte 127)
              uint32_t w[8];
              const int e = mx_block32(h, w);
              if (row_ok && ncols >= 32) {
                uint8_t* dst = static_cast<uint8_t*>(p.out2) + orow * p.ld_out + col;
                *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
                const long long rt = s_tile[tl.g] / mx_ncu + tl.m0 / BM;
                uint8_t* sfw = p.o_sf + (rt * p.o_sf_kst + col / 128) * 512 + lane * 16 + quarter * 4;
                sfw[(col >> 5) & 3] = static_cast<uint8_t>(e + 127);
                if (col + 32 == p.N && ((p.N >> 5) & 3) != 0)
                  for (int k = (p.N >> 5) & 3; k < 4; ++k) sfw[k] = 127;
              }
              continue;
            }
            emit32(o2, h, col, ncols, full, row_ok, false);  // A: bf16 operand of the down projection
            if (p.out3) {  // and the bf16 rounding of what A's bf16 value leaves (the down projection's low part)
#pragma unroll
              for (int i = 0; i < 32; ++i) h[i] -= bf16_round(h[i]);
              emit32(o3, h, col, ncols, full, row_ok, false);
            }
          }
        } else if (EPI == EPI_SCALE || EPI == EPI_SCALE_Q) {
          float w = row_ok ? __ldg(p.row_scale + orow) : 0.0f;
          if (EPI == EPI_SCALE_Q && row_ok) w *= __ldg(p.in0 + orow);  // the A row's e4m3 scale
#pragma unroll 1
          for (int c = c_lo; c < c_lo + kCols; c += 64) {
            uint32_t r0[32], r1[32];
            tmem_ld32(tbase + c, r0);
            tmem_ld32(tbase + c + 32, r1);
            tmem_ld_wait();
            float v[64];
            if (EPI == EPI_SCALE_Q) {
              // lane i holds the scales of columns c + i and c + 32 + i; the warp's rows share them
              const int col = tl.n0 + c + lane;
              const long long so = static_cast<long long>(tl.g) * p.ld_in + col;
              const float s0 = col < p.N ? __ldg(p.in1 + so) : 0.0f;
              const float s1 = col + 32 < p.N ? __ldg(p.in1 + so + 32) : 0.0f;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                v[i] = w * __shfl_sync(0xffffffffu, s0, i) * __uint_as_float(r0[i]);
                v[32 + i] = w * __shfl_sync(0xffffffffu, s1, i) * __uint_as_float(r1[i]);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                v[i] = w * __uint_as_float(r0[i]);
                v[32 + i] = w * __uint_as_float(r1[i]);
              }
            }
            emit64(o0, v, tl.n0 + c, p.N - tl.n0 - c, full, row_ok);
          }
        } else {  // EPI_DSWIGLU, EPI_DSWIGLU_Q
          const float w = row_ok ? __ldg(p.row_scale + orow) : 0.0f;
          const float sq = (EPI == EPI_DSWIGLU_Q && row_ok) ? __ldg(p.q_row + orow) : 1.0f;  // e4m3: A row scale
          float ds = 0.0f;
#pragma unroll 1
          for (int c = c_lo; c < c_lo + kCols; c += 32) {
            uint32_t r[32];
            tmem_ld32(tbase + c, r);
            tmem_ld_wait();
            const int col = tl.n0 + c;
            const int ncols = p.N - col;
            if (ncols <= 0) continue;
            if (EPI == EPI_DSWIGLU_Q) {
              // lane i holds column col + i's B scale; the warp's rows share it
              const float cs = lane < ncols ? __ldg(p.q_col + static_cast<long long>(tl.g) * p.q_ld + col + lane) : 0.0f;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                r[i] = __float_as_uint(__uint_as_float(r[i]) * sq * __shfl_sync(0xffffffffu, cs, i));
            }
            float h[32], u[32];
            if (row_ok) {
              load_f32_row32(p.in0 + orow * p.ld_in + col, h, ncols);
              load_f32_row32(p.in1 + orow * p.ld_in + col, u, ncols);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) h[i] = u[i] = 0.0f;
            }
            float dh[32], du[32], ap[32];
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
            if (kMx && row_ok && ncols >= 32) {
              // [dH | dU] as block-scaled e4m3 for the dX GEMM, from the exact fp32 values: this row's 32 columns
              // of dH (row columns col..) and of dU (n + col..) are one block each; their scale bytes go into
              // the row tile's blocks over the 2n columns
              const long long rt = s_tile[tl.g] / mx_ncu + tl.m0 / BM;
              uint8_t* sfr = p.o_sf + rt * p.o_sf_kst * 512ll + lane * 16 + quarter * 4;
              uint32_t qw[8];
              const int eh = mx_block32(dh, qw);
              uint8_t* dst = p.o_q + orow * p.o_q_ld + col;
              *reinterpret_cast<uint4*>(dst) = make_uint4(qw[0], qw[1], qw[2], qw[3]);
              *reinterpret_cast<uint4*>(dst + 16) = make_uint4(qw[4], qw[5], qw[6], qw[7]);
              sfr[(col >> 7) * 512 + ((col >> 5) & 3)] = static_cast<uint8_t>(eh + 127);
              const int eu = mx_block32(du, qw);
              const int cu = p.N + col;
              dst = p.o_q + orow * p.o_q_ld + cu;
              *reinterpret_cast<uint4*>(dst) = make_uint4(qw[0], qw[1], qw[2], qw[3]);
              *reinterpret_cast<uint4*>(dst + 16) = make_uint4(qw[4], qw[5], qw[6], qw[7]);
              sfr[(cu >> 7) * 512 + ((cu >> 5) & 3)] = static_cast<uint8_t>(eu + 127);
            }
            emit32(o0, dh, col, ncols, full, row_ok, false);
            emit32(o1, du, col, ncols, full, row_ok, false);
            emit32(o2, ap, col, ncols, full, row_ok, false);
            if (p.out3) {
              // the bf16 rounding of what the high parts left (the weight-gradient GEMMs' low operands)
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                dh[i] -= bf16_round(dh[i]);
                du[i] -= bf16_round(du[i]);
                ap[i] -= bf16_round(ap[i]);
              }
              emit32(o3, dh, col, ncols, full, row_ok, false);
              emit32(o4, du, col, ncols, full, row_ok, false);
              emit32(o5, ap, col, ncols, full, row_ok, false);
            }
          }
          // one partial per (row, column tile, column half)
          if (row_ok) p.part[orow * p.part_ld + tl.nt * (EW / 4) + half] = ds;
        }
      } else {  // EPI_STORE
        const int m = tl.m0 + row_local;
        const int mw = tl.m0 + quarter * 32;
        OutRef o{&mp.o0, p.out0, 0, 0, -1};
        if (VAR == VAR_M) {
          o.row_off = (s_off[tl.g] + static_cast<long long>(m)) * p.ld_out;
          o.c_row = s_off[tl.g] + mw;
        } else if (VAR == VAR_K) {
          // output [groups][rows][N]: rows < split go to out0 (min(M, split) rows per group), the rest to
          // out1 (M - split rows per group)
          o.c_z = tl.g;
          if (mw >= p.out_rows_split) {
            o.map = &mp.o1;
            o.ptr = p.out1;
            o.c_row = mw - p.out_rows_split;
            o.row_off = (static_cast<long long>(tl.g) * (p.M - p.out_rows_split) + (m - p.out_rows_split)) * p.ld_out;
          } else {
            o.c_row = mw;
            o.row_off = (static_cast<long long>(tl.g) * min(p.M, p.out_rows_split) + m) * p.ld_out;
          }
        } else {
          o.c_z = tl.split;
          o.c_row = mw;
        }
        if (VAR == VAR_K && mw >= p.M) {
          // rows past the output (the odd CTA of a pair on the last row tile): nothing to store
        } else if (kTrans) {
          // Each 32 x 32 block leaves transposed: block row i = accumulator column col + i (an output
          // row), block column = this thread's tile row (output column mw + lane).  Staged in the swizzled
          // layout of the store map (fp32 rows of 128 B, bf16 rows of 64 B); the TMA store clips rows and
          // columns past the output's extent.
#pragma unroll 1
          for (int c = c_lo; c < c_lo + kCols; c += 32) {
            uint32_t r[32];
            tmem_ld32(tbase + c, r);
            tmem_ld_wait();
            const int col = tl.n0 + c;
            if (col >= p.N) continue;  // a block wholly past the output (N a multiple of 64)
            uint8_t* stg = next_stage_buf();
            if (OUTF32) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                *reinterpret_cast<float*>(stg + i * 128 + ((((lane >> 2) ^ (i & 7)) << 4) | ((lane & 3) << 2))) =
                    have_acc ? __uint_as_float(r[i]) : 0.0f;
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                *reinterpret_cast<__nv_bfloat16*>(stg + i * 64 + ((((lane >> 3) ^ ((i >> 1) & 3)) << 4) | ((lane & 7) << 1))) =
                    __float2bfloat16_rn(have_acc ? __uint_as_float(r[i]) : 0.0f);
            }
            issue_store(OutRef{&mp.o0, nullptr, 0, col, tl.g}, stg, mw);
          }
        } else if (OUTF32) {
#pragma unroll 1
          for (int c = c_lo; c < c_lo + kCols; c += 32) {
            uint32_t r[32];
            tmem_ld32(tbase + c, r);
            tmem_ld_wait();
            const int col = tl.n0 + c;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v[i] = have_acc ? __uint_as_float(r[i]) : 0.0f;
              if (p.col_bias && col + i < p.N) v[i] += __ldg(p.col_bias + col + i);
            }
            emit32(o, v, col, p.N - col, full, row_ok, true);
          }
        } else {
          // e4m3 form: the A row's scale (per sorted row of the group) times the output channel's scale
          float sr = 1.0f;
          if (EPI == EPI_STORE_Q && VAR == VAR_M && row_ok) sr = __ldg(p.row_scale + s_off[tl.g] + m);
#pragma unroll 1
          for (int c = c_lo; c < c_lo + kCols; c += 64) {
            uint32_t r0[32], r1[32];
            tmem_ld32(tbase + c, r0);
            tmem_ld32(tbase + c + 32, r1);
            tmem_ld_wait();
            const int col = tl.n0 + c;
            float v[64];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v[i] = have_acc ? __uint_as_float(r0[i]) : 0.0f;
              v[32 + i] = have_acc ? __uint_as_float(r1[i]) : 0.0f;
              if (p.col_bias) {
                if (col + i < p.N) v[i] += __ldg(p.col_bias + col + i);
                if (col + 32 + i < p.N) v[32 + i] += __ldg(p.col_bias + col + 32 + i);
              }
            }
            if (EPI == EPI_STORE_Q) {
              // lane i holds the scales of columns col + i and col + 32 + i; the warp's rows share them
              const long long so = static_cast<long long>(tl.g) * p.ld_in + col + lane;
              const float s0 = col + lane < p.N ? __ldg(p.in1 + so) : 0.0f;
              const float s1 = col + 32 + lane < p.N ? __ldg(p.in1 + so + 32) : 0.0f;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                v[i] *= sr * __shfl_sync(0xffffffffu, s0, i);
                v[32 + i] *= sr * __shfl_sync(0xffffffffu, s1, i);
              }
            }
            emit64(o, v, col, p.N - col, full, row_ok);
          }
        }
      }
      tc_fence_before();
      if (kPair && cta_rank != 0) mbar_arrive_remote(mapa_shared(smem_u32(&tempty_bar[buf]), 0));
      else mbar_arrive(&tempty_bar[buf]);
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (CN > 1) cluster_sync();  // peers finished with this CTA's shared memory
  if (warp == kProdWarp) {
    if (kPair) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// grid: CTAs wanted (at most one per SM); with CN > 1 it is rounded to whole clusters and capped
// at the clusters that can be resident at once.
template <int BN, int STAGES, int EW, int DEPTH, int AMODE, int BMODE, int VAR, int EPI, bool OUTF32, int CN = 1,
          int XF = 0>
cudaError_t launch_grouped_gemm(const GemmParams& p, const Maps& maps, int grid, cudaStream_t stream) {
  auto kern = grouped_gemm_kernel<BN, STAGES, EW, DEPTH, AMODE, BMODE, VAR, EPI, OUTF32, CN, XF>;
  const size_t smem = SmemLayout<BN, STAGES, EW, DEPTH, (XF & X_DUAL_A) ? 2 : 1, (XF & X_PAIR) ? BN / 2 : BN,
                                 mx_stage_bytes(BN, XF)>::bytes(p.groups, VAR);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (grid <= 0) return cudaSuccess;
  const int threads = WarpPlan<STAGES, EW, AMODE, BMODE, CN, XF>::kThreads;
  if (CN == 1) {
    kern<<<grid, threads, smem, stream>>>(p, maps);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CN;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(CN, 1, 1);
  int max_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  int clusters = (grid + CN - 1) / CN;
  if (max_clusters > 0 && clusters > max_clusters) clusters = max_clusters;
  cfg.gridDim = dim3(clusters * CN, 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, p, maps);
}

}  // namespace vgg

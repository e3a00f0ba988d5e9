// Host side of the C ABI declared in include/moe.h: argument checks, tensor
// maps, workspace carving and the launch sequence of every entry point.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"
#include "moe.h"

// Per-kernel timing: when enabled, every internal launch is bracketed by a
// pair of CUDA events on the launching stream; moe_profile_read drains them.
struct ProfRecord {
  int kernel;
  cudaEvent_t beg, end;
};

struct moe_ctx {
  int device;
  int num_sms;
  int* d_err;
  unsigned long long timeout_ns;
  bool prof = false;
  int l2_prefetch = 0;  // L2 prefetch of later stages (measured slower; kept switchable)
  int cta_pair = 0;     // CTA pairs on the 256-row tiles of the tiled varlen-M GEMMs (dX, dA', two-part down)
  int cta_pair_dw = 0;  // CTA pairs on the varlen-K weight-gradient GEMMs (both measured slower; switchable)
  // The backward's per-token chain (router gradient, dX reduction, dW_r) runs on a second stream beside the
  // weight-gradient GEMMs, forked from and joined back into the caller's stream.
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;

  std::vector<cudaEvent_t> pool;
  size_t pool_next = 0;
  std::vector<ProfRecord> pending;
  std::vector<std::string> names;
  std::vector<double> total_ms;
  std::vector<long long> launches;
};

namespace vgg {

int ctx_device(const moe_ctx* ctx) { return ctx->device; }
int* ctx_error_word(moe_ctx* ctx) { return ctx->d_err; }

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static bool ensure_encode() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

static bool encode(CUtensorMap* m, CUtensorMapDataType dt, uint32_t rank, const void* ptr, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  if (!ensure_encode()) return false;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(m, dt, rank, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t row_stride_elems,
                 uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_elems * 2};
  cuuint32_t box[2] = {64, box_rows};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_map_3d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t groups,
                 uint32_t box_rows) {
  cuuint64_t dims[3] = {inner, rows, groups};
  cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_chunked_map_2d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_chunks) {
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, 64, box_chunks};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_chunked_map_3d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t groups,
                         uint32_t box_chunks) {
  cuuint64_t dims[4] = {64, rows, cols / 64, groups};
  cuuint64_t strides[3] = {cols * 2, 128, cols * rows * 2};
  cuuint32_t box[4] = {64, 64, box_chunks, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Box rows are 128 bytes (fp32: 32 columns; bf16: 64 columns) with the 128-byte swizzle, or for
// bf16 with box_cols = 32, 64 bytes with the 64-byte swizzle.
static CUtensorMapSwizzle store_swizzle(bool fp32, uint32_t box_cols) {
  return (fp32 || box_cols == 64) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
}

bool make_store_map_2d(CUtensorMap* m, void* ptr, bool fp32, uint64_t cols, uint64_t rows, uint64_t row_stride_elems,
                       uint32_t box_cols) {
  const uint64_t es = fp32 ? 4 : 2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_elems * es};
  cuuint32_t box[2] = {fp32 ? 32u : box_cols, 32};
  return encode(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides,
                box, store_swizzle(fp32, box_cols));
}

bool make_store_map_3d(CUtensorMap* m, void* ptr, bool fp32, uint64_t cols, uint64_t rows, uint64_t depth,
                       uint32_t box_cols) {
  const uint64_t es = fp32 ? 4 : 2;
  cuuint64_t dims[3] = {cols, rows, depth};
  cuuint64_t strides[2] = {cols * es, cols * rows * es};
  cuuint32_t box[3] = {fp32 ? 32u : box_cols, 32, 1};
  return encode(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides,
                box, store_swizzle(fp32, box_cols));
}

namespace {

constexpr size_t kAlign = 256;
inline size_t al(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

inline int gemm_bn(int N) { return N > 128 ? 256 : 128; }

// Launch shape of a varlen-M GEMM over cap sorted rows in E groups with N output columns.  With BN = 256
// (and pairs allowed) a CTA pair computes each 256-row tile, each CTA loading BN / 2 of B's columns.
struct VmShape {
  bool pair;
  int b_cols;  // columns of B per TMA box
  int grid;    // CTAs
};
inline VmShape vm_shape(const moe_ctx* ctx, int BN, bool allow, long long cap, int E, int N) {
  VmShape sh;
  sh.pair = allow && ctx->cta_pair && BN == 256;
  sh.b_cols = sh.pair ? BN / 2 : BN;
  const long long tiles = static_cast<long long>(ceil_div(cap, sh.pair ? 2 * BM : BM) + E) * ceil_div(N, BN);
  sh.grid = static_cast<int>(sh.pair ? std::min<long long>(2 * tiles, ctx->num_sms / 2 * 2)
                                     : std::min<long long>(tiles, ctx->num_sms));
  return sh;
}

// Launch shape of a two-part varlen-K weight-gradient GEMM ([G][M][N] output).  With padded B rows
// and BN = 256 a CTA pair computes each 256-row tile (each CTA loads BN / 2 of B's columns);
// otherwise one CTA per 128-row tile.
struct DwShape {
  bool pair;
  int b_chunks;  // 64-column chunks of B per TMA box
  int grid;      // CTAs
};
inline DwShape dw_shape(const moe_ctx* ctx, int BN, bool padded, int G, int M, int N) {
  DwShape sh;
  sh.pair = padded && BN == 256 && ctx->cta_pair_dw;
  sh.b_chunks = (sh.pair ? BN / 2 : BN) / 64;
  const long long tiles = static_cast<long long>(G) * ceil_div(M, sh.pair ? 2 * BM : BM) * ceil_div(N, BN);
  const long long ctas = sh.pair ? 2 * tiles : tiles;
  sh.grid = static_cast<int>(std::min<long long>(ctas, sh.pair ? ctx->num_sms / 2 * 2 : ctx->num_sms));
  return sh;
}

constexpr int kMaxSplitK = 16;

struct BwdWs {
  __nv_bfloat16 *dH, *dU, *Ap, *dXp, *WrT, *Xs, *dOs;
  __nv_bfloat16 *dH_lo, *dU_lo, *Ap_lo;  // bf16 rounding of what dH, dU, A' leave of the fp32 values
  int32_t* poff;  // [E + 1] group offsets of the padded sorted copies Xs, dOs (groups rounded up to 16 rows)
  __nv_bfloat16* dL;  // [2][Tp][E], Tp = T rounded up to 64: dlogits as a bf16 high part and the bf16
                      // rounding of the rest; rows [T, Tp) of both halves are zero
  float* part;
  float* wr_part;
};

// Column tile of the dSwiGLU GEMM (dA' = dO W_down, N = n), which also sets the number of dS partials per pair:
// 256 columns, or 128 when 256-column tiles would give fewer than eight waves over the SMs (c2, n = 512: 768
// tiles on 152 SMs; 186 -> 166 us with 128 columns, while at 2560 tiles and more 256 columns stay 4-28% faster).
// The workspace holds the partials of 128-column tiles either way.
inline int dact_bn(int n, long long cap, int E, int num_sms) {
  if (n <= 128) return 128;
  const long long tiles256 = static_cast<long long>(ceil_div(cap, BM) + E) * ceil_div(n, 256);
  return tiles256 >= 8ll * num_sms ? 256 : 128;
}
inline int dact_part_ld_max(int n) { return ceil_div(n, 128) * 2; }

// Rows of the padded sorted copies: every group rounded up to a multiple of 16 rows.
inline long long padded_rows(long long cap, int E) { return cap + 15ll * E; }

size_t bwd_ws_bytes(int T, int d, int E, int n, long long cap) {
  const int part_ld = dact_part_ld_max(n);
  const long long cp = padded_rows(cap, E);
  return 6 * al(sizeof(__nv_bfloat16) * cap * n) + al(sizeof(__nv_bfloat16) * cap * d) +
         2 * al(sizeof(__nv_bfloat16) * cp * d) + al(sizeof(int32_t) * (E + 1)) +
         al(sizeof(float) * cap * part_ld) + al(sizeof(__nv_bfloat16) * 2 * static_cast<size_t>(ceil_div(T, 64)) * 64 * E) +
         al(sizeof(__nv_bfloat16) * static_cast<size_t>(E) * d) +
         al(sizeof(float) * static_cast<size_t>(kMaxSplitK) * d * E);
}

// Store maps of the dSwiGLU epilogue's low parts (o3..o5), like those of dH, dU, A'.
bool make_lo_maps(Maps& m, const BwdWs& w, int n, long long cap) {
  return make_store_map_2d(&m.o3, w.dH_lo, false, n, cap, n, 32) && make_store_map_2d(&m.o4, w.dU_lo, false, n, cap, n, 32) &&
         make_store_map_2d(&m.o5, w.Ap_lo, false, n, cap, n, 32);
}

BwdWs carve_bwd(void* ws, int T, int d, int E, int n, long long cap) {
  const int part_ld = dact_part_ld_max(n);
  uint8_t* p = static_cast<uint8_t*>(ws);
  BwdWs w{};
  auto take = [&](size_t bytes) {
    uint8_t* r = p;
    p += al(bytes);
    return r;
  };
  w.dH = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * cap * n));
  w.dU = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * cap * n));
  w.Ap = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * cap * n));
  w.dH_lo = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * cap * n));
  w.dU_lo = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * cap * n));
  w.Ap_lo = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * cap * n));
  w.dXp = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * cap * d));
  w.Xs = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * padded_rows(cap, E) * d));
  w.dOs = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * padded_rows(cap, E) * d));
  w.poff = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (E + 1)));
  w.part = reinterpret_cast<float*>(take(sizeof(float) * cap * part_ld));
  w.dL = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * 2 * static_cast<size_t>(ceil_div(T, 64)) * 64 * E));
  w.WrT = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * static_cast<size_t>(E) * d));
  w.wr_part = reinterpret_cast<float*>(take(sizeof(float) * static_cast<size_t>(kMaxSplitK) * d * E));
  return w;
}

GemmParams base_params(moe_ctx* ctx) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.split_k = 1;
  p.a_ksplit = INT_MAX;
  p.a_colsplit = INT_MAX;
  p.a_kwrap = INT_MAX;
  p.b_ksplit = INT_MAX;
  p.out_rows_split = INT_MAX;
  p.err = ctx->d_err;
  p.timeout_ns = ctx->timeout_ns;
  p.l2_prefetch = ctx->l2_prefetch;
  return p;
}

Maps zero_maps() {
  Maps m;
  std::memset(&m, 0, sizeof(m));
  return m;
}

bool shapes_ok(int T, int d, int E, int n, int K) {
  return T >= 1 && T <= 65536 && d >= 64 && d % 64 == 0 && n >= 64 && n % 64 == 0 && K >= 1 && K <= 8 && E >= K &&
         E <= kMaxGroups && E % 8 == 0;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

constexpr size_t kProfPool = 4096;

void prof_drain(moe_ctx* ctx) {
  for (const ProfRecord& r : ctx->pending) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.end) == cudaSuccess && cudaEventElapsedTime(&ms, r.beg, r.end) == cudaSuccess) {
      ctx->total_ms[r.kernel] += ms;
      ctx->launches[r.kernel] += 1;
    }
  }
  ctx->pending.clear();
  ctx->pool_next = 0;
}

int prof_kernel_id(moe_ctx* ctx, const char* name) {
  for (size_t i = 0; i < ctx->names.size(); ++i)
    if (ctx->names[i] == name) return static_cast<int>(i);
  ctx->names.emplace_back(name);
  ctx->total_ms.push_back(0.0);
  ctx->launches.push_back(0);
  return static_cast<int>(ctx->names.size() - 1);
}

// Brackets one launch with events when profiling is on.
struct ProfScope {
  moe_ctx* ctx;
  cudaStream_t s;
  ProfRecord rec{};
  bool on = false;
  ProfScope(moe_ctx* c, const char* name, cudaStream_t st) : ctx(c), s(st) {
    if (!ctx->prof) return;
    if (ctx->pool_next + 2 > ctx->pool.size()) prof_drain(ctx);
    rec.kernel = prof_kernel_id(ctx, name);
    rec.beg = ctx->pool[ctx->pool_next++];
    rec.end = ctx->pool[ctx->pool_next++];
    on = cudaEventRecord(rec.beg, s) == cudaSuccess;
  }
  ~ProfScope() {
    if (on && cudaEventRecord(rec.end, s) == cudaSuccess) ctx->pending.push_back(rec);
  }
};

}  // namespace
}  // namespace vgg

using namespace vgg;

#define VGG_REQUIRE(cond)                  \
  do {                                     \
    if (!(cond)) return MOE_ERR_INVALID_ARG; \
  } while (0)
#define VGG_CUDA(call)                          \
  do {                                          \
    cudaError_t e_ = (call);                    \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)
// A timed launch: `name` is the kernel's label in moe_profile_read.
#define VGG_LAUNCH(name, call)                    \
  do {                                            \
    ProfScope ps_(ctx, name, s);                  \
    cudaError_t e_ = (call);                      \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA;   \
  } while (0)

// Down projection of the sorted activation rows A, each row scaled by its combine weight (Yw).  With A_lo
// (the bf16 rounding of what A's bf16 value leaves of the fp32 activation) the GEMM takes A as two parts.
static int down_projection(moe_ctx* ctx, const void* A, const void* A_lo, const void* W_down, int d, int E, int n,
                           long long cap, const int32_t* offsets, const float* sorted_w, void* Yw, cudaStream_t s) {
  GemmParams p = base_params(ctx);
  p.N = d;
  p.K = n;
  p.groups = E;
  p.offsets = offsets;
  p.rows_cap = static_cast<int>(cap);
  p.out0 = Yw;
  p.ld_out = d;
  p.row_scale = sorted_w;
  const int BN = gemm_bn(d);
  const VmShape sh = vm_shape(ctx, BN, A_lo != nullptr, cap, E, d);
  Maps m = zero_maps();
  if (!make_map_2d(&m.a0, A, n, cap, n, BM) || !make_map_3d(&m.b0, W_down, n, d, E, sh.b_cols) ||
      !make_store_map_2d(&m.o0, Yw, false, d, cap, d, 64) || (A_lo && !make_map_2d(&m.a2, A_lo, n, cap, n, BM)))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.a3 = m.a2;
  m.b1 = m.b0;
  if (A_lo) VGG_LAUNCH("down_scale", run_down_scale_dual(BN, sh.pair, p, m, sh.grid, s));
  else VGG_LAUNCH("down_scale", run_down_scale(BN, p, m, sh.grid, s));
  return MOE_OK;
}

// The plain grouping of moe_permute (m_tile = 0) with its hist / block-base scratch taken from `scratch`
// (scratch_ints ints) instead of a workspace: the same argument checks and launch as moe_permute.
int vgg::permute_plain_with_scratch(moe_ctx* ctx, const int32_t* topk_ids, const float* topk_w, int T, int E, int K,
                                    long long cap, int32_t* counts, int32_t* offsets, int32_t* sorted_tok,
                                    float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs, int32_t* P_out,
                                    int32_t* scratch, long long scratch_ints, cudaStream_t s) {
  VGG_REQUIRE(ctx && topk_ids && topk_w && counts && offsets && sorted_tok && sorted_w && tok_ptr && tok_pairs &&
              scratch);
  VGG_REQUIRE(shapes_ok(T, 64, E, 64, K));
  VGG_REQUIRE(cap >= moe_pair_capacity(T, E, K, 0) && cap < INT_MAX);
  const int tb = perm_tok_block(T, E);
  const int nb = (T + tb - 1) / tb;
  if (static_cast<long long>(E + 1) * nb + 2 > scratch_ints) return MOE_ERR_UNSUPPORTED;
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  PermuteWs w{};
  w.hist = scratch;
  w.tokblk = scratch + static_cast<long long>(E) * nb;
  w.barrier = w.tokblk + nb + 1;
  VGG_LAUNCH("permute", launch_permute(topk_ids, topk_w, nullptr, nullptr, T, E, K, 0, cap, counts, offsets,
                                       sorted_tok, sorted_w, tok_ptr, tok_pairs, P_out, w, ctx->d_err, ctx->timeout_ns,
                                       s));
  return MOE_OK;
}

extern "C" {

int moe_create(moe_ctx** out, int device) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return MOE_ERR_INVALID_ARG;
  if (cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
  if (!ensure_encode()) return MOE_ERR_CUDA;
  moe_ctx* c = new (std::nothrow) moe_ctx;
  if (!c) return MOE_ERR_CUDA;
  c->device = device;
  c->num_sms = sms;
  c->timeout_ns = 2000000000ull;
  int prio_lo = 0, prio_hi = 0;
  if (cudaMalloc(&c->d_err, 16) != cudaSuccess || cudaMemset(c->d_err, 0, 16) != cudaSuccess ||
      cudaDeviceGetStreamPriorityRange(&prio_lo, &prio_hi) != cudaSuccess ||
      cudaStreamCreateWithPriority(&c->side, cudaStreamNonBlocking, prio_hi) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->join, cudaEventDisableTiming) != cudaSuccess) {
    if (c->join) cudaEventDestroy(c->join);
    if (c->fork) cudaEventDestroy(c->fork);
    if (c->side) cudaStreamDestroy(c->side);
    if (c->d_err) cudaFree(c->d_err);
    delete c;
    return MOE_ERR_CUDA;
  }
  *out = c;
  return MOE_OK;
}

int moe_destroy(moe_ctx* ctx) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  for (cudaEvent_t e : ctx->pool) cudaEventDestroy(e);
  cudaEventDestroy(ctx->join);
  cudaEventDestroy(ctx->fork);
  cudaStreamDestroy(ctx->side);
  cudaFree(ctx->d_err);
  delete ctx;
  return MOE_OK;
}

const char* moe_status_str(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported device or configuration";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE: return "device-side data error (see moe_get_error)";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side bounded wait timed out";
    default: return "unknown status";
  }
}

int moe_get_error(moe_ctx* ctx, int* device_error) {
  if (!ctx || !device_error) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  *device_error = 0;
  VGG_CUDA(cudaDeviceSynchronize());
  int code = 0;
  VGG_CUDA(cudaMemcpy(&code, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost));
  VGG_CUDA(cudaMemset(ctx->d_err, 0, 16));
  *device_error = code;
  if (code == 0) return MOE_OK;
  return code == DERR_TIMEOUT ? MOE_ERR_DEVICE_TIMEOUT : MOE_ERR_DEVICE;
}

int moe_set_wait_timeout(moe_ctx* ctx, unsigned long long timeout_ns) {
  if (!ctx || timeout_ns == 0) return MOE_ERR_INVALID_ARG;
  ctx->timeout_ns = timeout_ns;
  return MOE_OK;
}

int moe_set_cta_pairs(moe_ctx* ctx, int varlen_m, int varlen_k) {
  if (!ctx || (varlen_m != 0 && varlen_m != 1) || (varlen_k != 0 && varlen_k != 1)) return MOE_ERR_INVALID_ARG;
  ctx->cta_pair = varlen_m;
  ctx->cta_pair_dw = varlen_k;
  return MOE_OK;
}

constexpr int kMaxRouteSplit = 4;

// Split of the router GEMM's reduction over d when it has fewer tiles than SMs (the partials
// are summed, with the bias, by the top-K kernel).
static int route_split(int T, int d, int E, int num_sms) {
  const int tiles = ceil_div(T, BM) * ceil_div(E, gemm_bn(E));
  int split = std::min(kMaxRouteSplit, std::max(1, num_sms / std::max(tiles, 1)));
  return std::max(1, std::min(split, d / (8 * BK)));
}

static size_t route_ws_bytes(int T, int E) {
  return sizeof(float) * static_cast<size_t>(kMaxRouteSplit) * T * E;
}

long long moe_pair_capacity(int T, int E, int K, int m_tile) {
  long long cap = static_cast<long long>(T) * K;
  if (m_tile > 0) cap += static_cast<long long>(E) * (m_tile / 2);
  return cap;
}

long long moe_expert_capacity(int T, int E, int K, double capacity_factor) {
  if (T < 1 || E < 1 || K < 1 || !(capacity_factor > 0.0) || capacity_factor > 1e6) return 0;
  // the factor times the mean load T K / E, evaluated left to right in double, rounded up
  return static_cast<long long>(std::ceil(capacity_factor * T * K / E));
}

size_t moe_workspace_bytes(int T, int d, int E, int n, int K, int m_tile) {
  if (!shapes_ok(T, d, E, n, K)) return 0;
  const long long cap = moe_pair_capacity(T, E, K, m_tile);
  return std::max({permute_ws_bytes(T, E, K, m_tile), bwd_ws_bytes(T, d, E, n, cap), route_ws_bytes(T, E)}) + kAlign;
}

int moe_route(moe_ctx* ctx, const void* X, const void* W_r, const float* bias, int T, int d, int E, int K,
              float* logits, float* scores, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
              moe_stream_t stream) {
  VGG_REQUIRE(ctx && X && W_r && logits && topk_ids && topk_w);
  VGG_REQUIRE(shapes_ok(T, d, E, 64, K));
  VGG_REQUIRE(aligned16(X) && aligned16(W_r) && aligned16(logits));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int split = route_split(T, d, E, ctx->num_sms);
  // without room in the caller's workspace the GEMM writes the logits (plus bias) itself
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0 ||
      ws_bytes < sizeof(float) * static_cast<size_t>(split) * T * E)
    split = 1;
  float* part = split > 1 ? static_cast<float*>(ws) : nullptr;
  GemmParams p = base_params(ctx);
  p.M = T;
  p.N = E;
  p.K = d;
  p.groups = 1;
  p.split_k = split;
  p.out0 = split > 1 ? part : logits;
  p.ld_out = E;
  p.col_bias = split > 1 ? nullptr : bias;
  const int BN = gemm_bn(E);
  Maps m = zero_maps();
  if (!make_map_2d(&m.a0, X, d, T, d, BM) || !make_map_2d(&m.b0, W_r, E, d, E, 64) ||
      !make_store_map_3d(&m.o0, split > 1 ? part : logits, true, E, T, split, 32))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.b1 = m.b0;
  const int tiles = ceil_div(T, BM) * ceil_div(E, BN);
  VGG_LAUNCH("router_logits", run_router_logits(BN, p, m, std::min(tiles * split, ctx->num_sms), s));
  VGG_LAUNCH("topk_softmax", launch_topk_softmax(logits, part, split, bias, T, E, K, topk_ids, topk_w, scores, s));
  return MOE_OK;
}

int moe_permute(moe_ctx* ctx, const int32_t* topk_ids, const float* topk_w, const float* logits,
                const float* scores, int T, int E, int K, int m_tile, long long cap, int32_t* counts,
                int32_t* offsets, int32_t* sorted_tok, float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs,
                int32_t* P_out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  VGG_REQUIRE(ctx && topk_ids && topk_w && counts && offsets && sorted_tok && sorted_w && tok_ptr && tok_pairs &&
              ws);
  VGG_REQUIRE(shapes_ok(T, 64, E, 64, K));
  VGG_REQUIRE(m_tile >= 0 && (m_tile == 0 || m_tile % 64 == 0));
  VGG_REQUIRE(cap >= moe_pair_capacity(T, E, K, m_tile) && cap < INT_MAX);
  VGG_REQUIRE(ws_bytes >= permute_ws_bytes(T, E, K, m_tile));
  VGG_REQUIRE((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) == 0);
  if (m_tile > 0) {
    VGG_REQUIRE(scores && logits);
    if (T > 32768) return MOE_ERR_UNSUPPORTED;
  }
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  PermuteWs w = carve_permute_ws(ws, T, E, K, m_tile);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VGG_LAUNCH("permute", launch_permute(topk_ids, topk_w, logits, scores, T, E, K, m_tile, cap, counts, offsets,
                                       sorted_tok, sorted_w, tok_ptr, tok_pairs, P_out, w, ctx->d_err, ctx->timeout_ns,
                                       s));
  return MOE_OK;
}

int moe_permute_capacity(moe_ctx* ctx, const int32_t* topk_ids, const float* topk_w, int T, int E, int K, int C,
                         int policy, long long cap, int32_t* counts, int32_t* offsets, int32_t* sorted_tok,
                         float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs, int32_t* P_out, void* ws,
                         size_t ws_bytes, moe_stream_t stream) {
  VGG_REQUIRE(ctx && topk_ids && topk_w && counts && offsets && sorted_tok && sorted_w && tok_ptr && tok_pairs &&
              P_out && ws);
  VGG_REQUIRE(shapes_ok(T, 64, E, 64, K));
  VGG_REQUIRE(C >= 1 && (policy == 0 || policy == 1));
  VGG_REQUIRE(cap >= static_cast<long long>(E) * C && cap < INT_MAX);
  VGG_REQUIRE(ws_bytes >= permute_ws_bytes(T, E, K, 1));
  VGG_REQUIRE((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) == 0);
  if (T > 32768) return MOE_ERR_UNSUPPORTED;
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  PermuteWs w = carve_permute_ws(ws, T, E, K, 1);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VGG_LAUNCH("permute", launch_permute_capacity(topk_ids, topk_w, T, E, K, C, policy, cap, counts, offsets,
                                                sorted_tok, sorted_w, tok_ptr, tok_pairs, P_out, w, ctx->d_err,
                                                ctx->timeout_ns, s));
  return MOE_OK;
}

size_t moe_capacity_workspace_bytes(int T, int d, int E, int n, int K, int C) {
  if (!shapes_ok(T, d, E, n, K) || C < 1) return 0;
  const long long cap = static_cast<long long>(E) * C;
  return std::max({permute_ws_bytes(T, E, K, 1), bwd_ws_bytes(T, d, E, n, cap), route_ws_bytes(T, E)}) + kAlign;
}

int moe_grouped_gemm_fwd(moe_ctx* ctx, const void* X, const void* W_gate, const void* W_up, const void* W_down,
                         int T, int d, int E, int n, long long cap, const int32_t* offsets,
                         const int32_t* sorted_tok, const float* sorted_w, void* H, void* U, void* A, void* Yw,
                         void* ws, size_t ws_bytes, moe_stream_t stream) {
  VGG_REQUIRE(ctx && X && W_gate && W_up && W_down && offsets && sorted_tok && sorted_w && A && Yw && ws);
  VGG_REQUIRE((H == nullptr) == (U == nullptr));  // both NULL: forward only, no backward cache
  VGG_REQUIRE(shapes_ok(T, d, E, n, 1));
  VGG_REQUIRE(cap >= 1 && cap < INT_MAX);
  // the workspace holds A's low part between the two GEMMs
  VGG_REQUIRE(ws_bytes >= sizeof(__nv_bfloat16) * static_cast<size_t>(cap) * n);
  VGG_REQUIRE((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) == 0);
  VGG_REQUIRE(aligned16(X) && aligned16(W_gate) && aligned16(W_up) && aligned16(W_down) && aligned16(H) &&
              aligned16(U) && aligned16(A) && aligned16(Yw));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* A_lo = ws;
  // gate/up + SwiGLU: A = X rows gathered by sorted_tok, B = the W_gate / W_up pair
  {
    GemmParams p = base_params(ctx);
    p.N = n;
    p.K = d;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.a_idx = sorted_tok;
    p.a_rows = T;
    p.a_src = static_cast<const __nv_bfloat16*>(X);
    p.a_ld = d;
    p.out0 = H;
    p.out1 = U;
    p.out2 = A;
    p.out3 = A_lo;
    p.ld_out = n;
    const int BN = n > 64 ? 256 : 128;
    Maps m = zero_maps();
    if (!make_map_3d(&m.b0, W_gate, d, n, E, BN / 2) || !make_map_3d(&m.b1, W_up, d, n, E, BN / 2) ||
        (H && (!make_store_map_2d(&m.o0, H, true, n, cap, n, 32) || !make_store_map_2d(&m.o1, U, true, n, cap, n, 32))) ||
        !make_store_map_2d(&m.o2, A, false, n, cap, n, 32) || !make_store_map_2d(&m.o3, A_lo, false, n, cap, n, 32))
      return MOE_ERR_CUDA;
    const int tiles = (ceil_div(cap, BM) + E) * ceil_div(n, BN / 2);
    // pairs of CTAs on neighbouring column tiles share the gathered X rows (each gathers half)
    const int cn = ceil_div(n, BN / 2) >= 2 ? 2 : 1;
    VGG_LAUNCH("gate_up_swiglu", run_gate_up_swiglu(BN, cn, p, m, std::min(tiles, ctx->num_sms), s));
  }
  return down_projection(ctx, A, A_lo, W_down, d, E, n, cap, offsets, sorted_w, Yw, s);
}

int moe_quantize_rows_e4m3(moe_ctx* ctx, const void* M, long long rows, int cols, void* q, float* scales,
                           moe_stream_t stream) {
  VGG_REQUIRE(ctx && M && q && scales);
  VGG_REQUIRE(rows >= 0 && rows <= (1ll << 31) && cols >= 16 && cols % 16 == 0);
  VGG_REQUIRE(aligned16(M) && aligned16(q));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VGG_LAUNCH("quantize_e4m3", launch_quantize_rows_e4m3(static_cast<const __nv_bfloat16*>(M), rows, nullptr, cols,
                                                        static_cast<uint8_t*>(q), scales, s));
  return MOE_OK;
}

int moe_grouped_gemm_fwd_e4m3(moe_ctx* ctx, const void* Xq, const float* x_scale, const void* Wg_q,
                              const float* wg_scale, const void* Wu_q, const float* wu_scale, const void* W_down,
                              const void* Wd_q, const float* wd_scale, int T, int d, int E, int n, long long cap,
                              const int32_t* offsets, const int32_t* sorted_tok, const float* sorted_w, void* H,
                              void* U, void* A, void* Aq, float* a_scale, void* Yw, moe_stream_t stream) {
  VGG_REQUIRE(ctx && Xq && x_scale && Wg_q && wg_scale && Wu_q && wu_scale && offsets && sorted_tok && sorted_w &&
              A && Yw);
  VGG_REQUIRE((H == nullptr) == (U == nullptr));  // both NULL: forward only, no backward cache
  VGG_REQUIRE(shapes_ok(T, d, E, n, 1));
  // the down projection: bf16 (W_down) or e4m3 (Wd_q, wd_scale with the Aq, a_scale buffers)
  const bool down8 = Wd_q != nullptr;
  VGG_REQUIRE(down8 ? (wd_scale && Aq && a_scale && aligned16(Wd_q) && aligned16(Aq)) : W_down != nullptr);
  VGG_REQUIRE(cap >= 1 && cap < INT_MAX);
  VGG_REQUIRE(aligned16(Xq) && aligned16(Wg_q) && aligned16(Wu_q) && aligned16(W_down) && aligned16(H) &&
              aligned16(U) && aligned16(A) && aligned16(Yw));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    // e4m3 rows are handed to TMA and to the gather as rows of d / 2 16-bit units (code pairs): the
    // 128-byte stage rows, swizzle and coordinates are those of the bf16 form
    const int dk = d / 2;
    GemmParams p = base_params(ctx);
    p.N = n;
    p.K = dk;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.a_idx = sorted_tok;
    p.a_rows = T;
    p.a_src = static_cast<const __nv_bfloat16*>(Xq);
    p.a_ld = dk;
    p.out0 = H;
    p.out1 = U;
    p.out2 = A;
    p.ld_out = n;
    p.row_scale = x_scale;
    p.in0 = wg_scale;
    p.in1 = wu_scale;
    p.ld_in = n;
    const int BN = n > 64 ? 256 : 128;
    Maps m = zero_maps();
    if (!make_map_3d(&m.b0, Wg_q, dk, n, E, BN / 2) || !make_map_3d(&m.b1, Wu_q, dk, n, E, BN / 2) ||
        (H && (!make_store_map_2d(&m.o0, H, true, n, cap, n, 32) || !make_store_map_2d(&m.o1, U, true, n, cap, n, 32))) ||
        !make_store_map_2d(&m.o2, A, false, n, cap, n, 32))
      return MOE_ERR_CUDA;
    const int tiles = (ceil_div(cap, BM) + E) * ceil_div(n, BN / 2);
    const int cn = ceil_div(n, BN / 2) >= 2 ? 2 : 1;
    VGG_LAUNCH("gate_up_swiglu_e4m3", run_gate_up_swiglu_e4m3(BN, cn, p, m, std::min(tiles, ctx->num_sms), s));
  }
  if (!down8) return down_projection(ctx, A, nullptr, W_down, d, E, n, cap, offsets, sorted_w, Yw, s);
  // A's rows (those below offsets[E]) to e4m3, then the e4m3 down projection
  VGG_LAUNCH("quantize_a_e4m3", launch_quantize_rows_e4m3(static_cast<const __nv_bfloat16*>(A), cap, offsets + E, n,
                                                          static_cast<uint8_t*>(Aq), a_scale, s));
  {
    const int nk = n / 2;  // code pairs, as in the gate/up form
    GemmParams p = base_params(ctx);
    p.N = d;
    p.K = nk;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.out0 = Yw;
    p.ld_out = d;
    p.row_scale = sorted_w;
    p.in0 = a_scale;
    p.in1 = wd_scale;
    p.ld_in = d;
    const int BN = gemm_bn(d);
    Maps m = zero_maps();
    if (!make_map_2d(&m.a0, Aq, nk, cap, nk, BM) || !make_map_3d(&m.b0, Wd_q, nk, d, E, BN) ||
        !make_store_map_2d(&m.o0, Yw, false, d, cap, d, 64))
      return MOE_ERR_CUDA;
    m.a1 = m.a0;
    m.b1 = m.b0;
    const int tiles = (ceil_div(cap, BM) + E) * ceil_div(d, BN);
    VGG_LAUNCH("down_scale_e4m3", run_down_scale_e4m3(BN, p, m, std::min(tiles, ctx->num_sms), s));
  }
  return MOE_OK;
}

long long moe_mx_sf_cols(int cols) { return cols > 0 ? 4ll * ceil_div(cols, 128) : 0; }

long long moe_mx_weight_sf_bytes(int E, int d, int n, int which) {
  if (E < 1 || d < 64 || n < 64 || d % 64 || n % 64) return 0;
  // one group of mx_b_blocks(BN) blocks per column tile of BN rows and stage of K (the gate/up pair: kMxBN / 2 rows
  // of each; the plain GEMMs: BN = mx_tile_cols of their output width)
  const auto grp = [](int BN) { return 512ll * mx_b_blocks(BN); };
  if (which == 0) return grp(kMxBN) * E * ceil_div(n, kMxBN / 2) * ceil_div(d, 128);
  const int bd = mx_tile_cols(d), bn = mx_tile_cols(n);
  if (which == 1) return grp(bd) * E * ceil_div(d, bd) * ceil_div(n, 128);
  if (which == 2) return grp(bn) * E * ceil_div(n, bn) * ceil_div(d, 128);      // W_down^T [E][n][d]
  if (which == 3) return grp(bd) * E * ceil_div(d, bd) * ceil_div(2 * n, 128);  // [W_gate; W_up]^T [E][d][2n]
  return 0;
}

long long moe_mx_act_sf_bytes(long long cap, int E, int n) {
  if (cap < 1 || E < 1 || n < 64 || n % 64) return 0;
  return 512ll * (ceil_div(cap, BM) + E) * ceil_div(n, 128);
}

namespace vgg {
// The block-scaled weight gradients' workspace: the padded stage offsets, then the K-major code matrices of the
// two GEMMs' operands ([dH | dU]^T [2n][kq], X^T [d][kq], dO^T [d][kq], A'^T [n][kq]; kq = the padded reduction's
// capacity in tokens) and their scale blocks (A operands per 128-row tile, B operands per column tile of the
// GEMM, each per 128-token stage).  With base == nullptr only the size is computed.
struct MxDwWs {
  int32_t* kp;
  uint8_t *gu_a, *gu_b, *dn_a, *dn_b;
  uint8_t *gu_a_sf, *gu_b_sf, *dn_a_sf, *dn_b_sf;
  long long kq;
  int kst, bn_gu, bn_dn;
  size_t bytes;
};
static MxDwWs carve_mx_dw(void* base, int d, int E, int n, long long cap) {
  MxDwWs w{};
  w.kq = (cap + 127ll * E + 127) / 128 * 128;
  w.kst = static_cast<int>(w.kq / 128);
  w.bn_gu = mx_tile_cols(d);
  w.bn_dn = mx_tile_cols(n);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    uint8_t* ptr = base ? static_cast<uint8_t*>(base) + o : nullptr;
    o += al(bytes);
    return ptr;
  };
  const size_t kq = static_cast<size_t>(w.kq), kst = static_cast<size_t>(w.kst);
  w.kp = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (E + 1)));
  w.gu_a = take(2 * static_cast<size_t>(n) * kq);
  w.gu_b = take(static_cast<size_t>(d) * kq);
  w.dn_a = take(static_cast<size_t>(d) * kq);
  w.dn_b = take(static_cast<size_t>(n) * kq);
  w.gu_a_sf = take(512 * kst * ceil_div(2 * n, BM));
  w.gu_b_sf = take(512 * kst * ceil_div(d, w.bn_gu) * mx_b_blocks(w.bn_gu));
  w.dn_a_sf = take(512 * kst * ceil_div(d, BM));
  w.dn_b_sf = take(512 * kst * ceil_div(n, w.bn_dn) * mx_b_blocks(w.bn_dn));
  w.bytes = o;
  return w;
}
}  // namespace vgg

size_t moe_mx_dw_ws_bytes(int d, int E, int n, long long cap) {
  if (cap < 1 || E < 1 || E > kMaxGroups || d < 64 || d % 64 || n < 64 || n % 64) return 0;
  return carve_mx_dw(nullptr, d, E, n, cap).bytes;
}

int moe_quantize_rows_mx(moe_ctx* ctx, const void* M, long long rows, int cols, void* q, void* sf,
                         moe_stream_t stream) {
  VGG_REQUIRE(ctx && M && q && sf);
  VGG_REQUIRE(rows >= 0 && rows <= (1ll << 31) && cols >= 64 && cols % 64 == 0);
  VGG_REQUIRE(aligned16(M) && aligned16(q) && (reinterpret_cast<uintptr_t>(sf) & 3u) == 0);
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VGG_LAUNCH("quantize_mx", launch_quantize_rows_mx(static_cast<const __nv_bfloat16*>(M), rows, nullptr, cols,
                                                    static_cast<uint8_t*>(q), static_cast<uint8_t*>(sf),
                                                    static_cast<int>(moe_mx_sf_cols(cols)), s));
  return MOE_OK;
}

int moe_quantize_weights_mx(moe_ctx* ctx, const void* W_gate, const void* W_up, const void* W_down, int E, int d,
                            int n, void* Wg_q, void* Wu_q, void* gu_sf, void* Wd_q, void* dn_sf,
                            moe_stream_t stream) {
  VGG_REQUIRE(ctx && W_gate && W_up && W_down && Wg_q && Wu_q && gu_sf && Wd_q && dn_sf);
  VGG_REQUIRE(E >= 1 && E <= kMaxGroups && d >= 64 && d % 64 == 0 && n >= 64 && n % 64 == 0);
  VGG_REQUIRE(aligned16(W_gate) && aligned16(W_up) && aligned16(W_down) && aligned16(Wg_q) && aligned16(Wu_q) &&
              aligned16(gu_sf) && aligned16(Wd_q) && aligned16(dn_sf));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // every entry of the blocks that no operand row or column fills holds scale 1
  VGG_CUDA(cudaMemsetAsync(gu_sf, 127, static_cast<size_t>(moe_mx_weight_sf_bytes(E, d, n, 0)), s));
  VGG_CUDA(cudaMemsetAsync(dn_sf, 127, static_cast<size_t>(moe_mx_weight_sf_bytes(E, d, n, 1)), s));
  const int kd = ceil_div(d, 128), kn = ceil_div(n, 128), nb = mx_b_blocks(kMxBN), hb = kMxBN / 2;
  VGG_LAUNCH("quantize_mx_weights",
             launch_quantize_weight_mx(static_cast<const __nv_bfloat16*>(W_gate), E, n, d, static_cast<uint8_t*>(Wg_q),
                                       static_cast<uint8_t*>(gu_sf), hb, 0, ceil_div(n, hb), kd, nb, s));
  VGG_LAUNCH("quantize_mx_weights",
             launch_quantize_weight_mx(static_cast<const __nv_bfloat16*>(W_up), E, n, d, static_cast<uint8_t*>(Wu_q),
                                       static_cast<uint8_t*>(gu_sf), hb, hb, ceil_div(n, hb), kd, nb, s));
  const int bd = mx_tile_cols(d);
  VGG_LAUNCH("quantize_mx_weights",
             launch_quantize_weight_mx(static_cast<const __nv_bfloat16*>(W_down), E, d, n, static_cast<uint8_t*>(Wd_q),
                                       static_cast<uint8_t*>(dn_sf), bd, 0, ceil_div(d, bd), kn, mx_b_blocks(bd), s));
  return MOE_OK;
}

int moe_grouped_gemm_fwd_mx(moe_ctx* ctx, const void* Xq, const void* x_sf, const void* Wg_q, const void* Wu_q,
                            const void* gu_sf, const void* Wd_q, const void* dn_sf, int T, int d, int E, int n,
                            long long cap, const int32_t* offsets, const int32_t* sorted_tok, const float* sorted_w,
                            void* H, void* U, void* x_sf_tiles, void* Aq, void* a_sf, void* Yw, moe_stream_t stream) {
  VGG_REQUIRE(ctx && Xq && x_sf && Wg_q && Wu_q && gu_sf && Wd_q && dn_sf && offsets && sorted_tok && sorted_w &&
              x_sf_tiles && Aq && a_sf && Yw);
  VGG_REQUIRE((H == nullptr) == (U == nullptr));  // both NULL: forward only, no backward cache
  VGG_REQUIRE(shapes_ok(T, d, E, n, 1));
  VGG_REQUIRE(cap >= 1 && cap < INT_MAX);
  VGG_REQUIRE(aligned16(Xq) && (reinterpret_cast<uintptr_t>(x_sf) & 3u) == 0 && aligned16(Wg_q) &&
              aligned16(Wu_q) && aligned16(gu_sf) && aligned16(Wd_q) && aligned16(dn_sf) && aligned16(H) &&
              aligned16(U) && aligned16(x_sf_tiles) && aligned16(Aq) && aligned16(a_sf) && aligned16(Yw));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int dk = d / 2, nk = n / 2;  // e4m3 rows as 16-bit units (code pairs) for TMA and the gather
  // the gathered X rows' scales, laid out per sorted row tile and stage of K as the GEMM's producer loads them
  VGG_LAUNCH("mx_tile_scales",
             launch_mx_tile_scales(static_cast<const uint8_t*>(x_sf), static_cast<int>(moe_mx_sf_cols(d)), T,
                                   sorted_tok, static_cast<int>(cap), offsets, E, ceil_div(d, 128),
                                   ceil_div(cap, BM) + E, static_cast<uint8_t*>(x_sf_tiles), s));
  {
    GemmParams p = base_params(ctx);
    p.N = n;
    p.K = dk;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.a_idx = sorted_tok;
    p.a_rows = T;
    p.a_src = static_cast<const __nv_bfloat16*>(Xq);
    p.a_ld = dk;
    p.out0 = H;
    p.out1 = U;
    p.out2 = Aq;
    p.ld_out = n;
    p.a_sf = static_cast<const uint8_t*>(x_sf_tiles);
    p.b_sf = static_cast<const uint8_t*>(gu_sf);
    p.sf_kst = ceil_div(d, 128);
    p.o_sf = static_cast<uint8_t*>(a_sf);
    p.o_sf_kst = ceil_div(n, 128);
    Maps m = zero_maps();
    if (!make_map_3d(&m.b0, Wg_q, dk, n, E, kMxBN / 2) || !make_map_3d(&m.b1, Wu_q, dk, n, E, kMxBN / 2) ||
        (H && (!make_store_map_2d(&m.o0, H, true, n, cap, n, 32) || !make_store_map_2d(&m.o1, U, true, n, cap, n, 32))))
      return MOE_ERR_CUDA;
    const int tiles = (ceil_div(cap, BM) + E) * ceil_div(n, kMxBN / 2);
    // pairs of CTAs on neighbouring column tiles share the gathered X rows (each gathers half the codes)
    const int cn = ceil_div(n, kMxBN / 2) >= 2 ? 2 : 1;
    VGG_LAUNCH("gate_up_swiglu_mx", run_gate_up_swiglu_mx(cn, p, m, std::min(tiles, ctx->num_sms), s));
  }
  {
    GemmParams p = base_params(ctx);
    p.N = d;
    p.K = nk;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.out0 = Yw;
    p.ld_out = d;
    p.row_scale = sorted_w;
    p.a_sf = static_cast<const uint8_t*>(a_sf);
    p.b_sf = static_cast<const uint8_t*>(dn_sf);
    p.sf_kst = ceil_div(n, 128);
    const int BN = mx_tile_cols(d);
    Maps m = zero_maps();
    if (!make_map_2d(&m.a0, Aq, nk, cap, nk, BM) || !make_map_3d(&m.b0, Wd_q, nk, d, E, BN) ||
        !make_store_map_2d(&m.o0, Yw, false, d, cap, d, 64))
      return MOE_ERR_CUDA;
    m.a1 = m.a0;
    m.b1 = m.b0;
    const int tiles = (ceil_div(cap, BM) + E) * ceil_div(d, BN);
    VGG_LAUNCH("down_scale_mx", run_down_scale_mx(BN, p, m, std::min(tiles, ctx->num_sms), s));
  }
  return MOE_OK;
}

int moe_combine(moe_ctx* ctx, const void* Yw, const int32_t* tok_ptr, const int32_t* tok_pairs, int T, int d,
                long long cap, void* O, moe_stream_t stream) {
  VGG_REQUIRE(ctx && Yw && tok_ptr && tok_pairs && O);
  VGG_REQUIRE(T >= 1 && T <= 65536 && d >= 8 && d % 8 == 0 && cap >= 1);
  VGG_REQUIRE(aligned16(Yw) && aligned16(O));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VGG_LAUNCH("combine", launch_combine(static_cast<const __nv_bfloat16*>(Yw), tok_ptr, tok_pairs, T, d, cap,
                                       static_cast<__nv_bfloat16*>(O), ctx->d_err, s));
  return MOE_OK;
}

// Block-scaled dSwiGLU and dX GEMMs of the backward (moe_backward_mx): weight codes and scale blocks, the sorted dO
// code rows, dO's scale blocks per sorted row tile, and the [dH | dU] codes and scale blocks.
struct MxBwd {
  const void* Wdt_q;
  const void* wdt_sf;
  const void* Wgu_q;
  const void* wgu_sf;
  void* dOq;
  void* do_sf_tiles;
  void* HUq;
  void* hu_sf;
  void* dw_ws;  // the block-scaled weight gradients' workspace (moe_mx_dw_ws_bytes), or null: two-part bf16
};

// The backward; with Wgu_q the dX GEMM runs on e4m3 operands (moe_backward_e4m3), with mx both activation-gradient
// GEMMs on block-scaled operands (moe_backward_mx).
static int backward_impl(moe_ctx* ctx, const void* dO, const void* X, const void* W_r, const void* W_gate,
                         const void* W_up, const void* W_down, int T, int d, int E, int n, int K, int m_tile,
                         long long cap, const int32_t* topk_ids, const float* topk_w, const int32_t* offsets,
                         const int32_t* sorted_tok, const float* sorted_w, const int32_t* tok_ptr,
                         const int32_t* tok_pairs, const void* H, const void* U, void* dX, void* dW_gate,
                         void* dW_up, void* dW_down, int dW_fp32, float* dS, float* dlogits, float* dW_r, void* ws,
                         size_t ws_bytes, moe_stream_t stream, const void* Wgu_q, const float* wgu_scale, void* HUq,
                         float* hu_scale, const void* Wdt_q, const float* wdt_scale, void* dOq, float* do_scale,
                         const MxBwd* mx = nullptr) {
  VGG_REQUIRE(ctx && dO && X && W_r && W_gate && W_up && W_down && topk_ids && topk_w && offsets && sorted_tok &&
              sorted_w && tok_ptr && tok_pairs && H && U && dX && dW_gate && dW_up && dW_down && dS && dlogits &&
              dW_r && ws);
  VGG_REQUIRE(shapes_ok(T, d, E, n, K));
  // cap: the pair arrays' length (moe_pair_capacity, or E*C for the capacity dispatch); the device checks
  // offsets[E] <= cap
  VGG_REQUIRE(m_tile >= 0 && cap >= 1 && cap < INT_MAX);
  VGG_REQUIRE(ws_bytes >= bwd_ws_bytes(T, d, E, n, cap));
  VGG_REQUIRE((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) == 0);
  VGG_REQUIRE(aligned16(dO) && aligned16(X) && aligned16(W_r) && aligned16(W_gate) && aligned16(W_up) &&
              aligned16(W_down) && aligned16(H) && aligned16(U) && aligned16(dX) && aligned16(dW_gate) &&
              aligned16(dW_up) && aligned16(dW_down) && aligned16(dW_r));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  BwdWs w = carve_bwd(ws, T, d, E, n, cap);
  const bool f32 = dW_fp32 != 0;
  const int bn6 = dact_bn(n, cap, E, ctx->num_sms);
  // one dS partial per (column tile, epilogue column half); the block-scaled form tiles n by mx_tile_cols(n)
  const int part_ld = (mx ? ceil_div(n, mx_tile_cols(n)) : ceil_div(n, bn6)) * 2;
  if (cap > static_cast<long long>(T) * K) {
    __nv_bfloat16* const tail[6] = {w.dH, w.dU, w.Ap, w.dH_lo, w.dU_lo, w.Ap_lo};
    VGG_LAUNCH("zero_tail", launch_zero_tail_rows(offsets, E, cap, n, tail, s));
  }
  // e4m3 dSwiGLU GEMM: dO quantized once per token (a token's pairs share its row, so its codes are those of
  // every pair) into the dX partials' region, which is free until the dX GEMM; the gather below copies the
  // code rows and scales to the sorted positions.  When that region is too small (a capacity layout with
  // cap < T) the sorted rows are quantized instead.
  const size_t tok_codes = al(static_cast<size_t>(T) * d);
  const bool dact_tok = Wdt_q && tok_codes + sizeof(float) * T <= sizeof(__nv_bfloat16) * cap * d;
  uint8_t* tq = reinterpret_cast<uint8_t*>(w.dXp);
  float* ts = reinterpret_cast<float*>(tq + tok_codes);
  if (dact_tok)
    VGG_LAUNCH("quantize_do_e4m3", launch_quantize_rows_e4m3(static_cast<const __nv_bfloat16*>(dO), T, nullptr, d, tq,
                                                            ts, s));
  // block-scaled form: dO in 1 x 32 blocks per token (codes and row-major scales) into the same region; the gather
  // below copies the code rows to the sorted positions and mx_tile_scales lays the scales out per sorted row tile
  const int mx_sfc = static_cast<int>(moe_mx_sf_cols(d));
  uint8_t* mq = reinterpret_cast<uint8_t*>(w.dXp);
  uint8_t* msf = mq + tok_codes;
  if (mx) {
    if (tok_codes + static_cast<size_t>(T) * mx_sfc > sizeof(__nv_bfloat16) * cap * d) return MOE_ERR_UNSUPPORTED;
    VGG_LAUNCH("quantize_mx", launch_quantize_rows_mx(static_cast<const __nv_bfloat16*>(dO), T, nullptr, d, mq, msf,
                                                      mx_sfc, s));
  }
  // expert-sorted copies of X and dO (and of dO's codes): every backward GEMM then reads whole TMA boxes.  The
  // bf16 copies are padded per expert to multiples of 16 rows (zero rows), except when the e4m3 dSwiGLU GEMM
  // quantizes the sorted dO rows themselves (a capacity layout with fewer slots than tokens).
  // With the block-scaled weight gradients (which read X and dO through the token index) only the code rows are
  // copied.
  const bool mx_dw = mx && mx->dw_ws;
  // The e4m3 and block-scaled forms take the weight gradients' operands rounded once to bf16: their
  // activation-gradient GEMMs already carry e4m3 rounding, and the single-part GEMMs run half the UMMAs.  The
  // bf16 backward keeps the two-part operands of the precision bound; the dSwiGLU epilogue writes the low
  // parts for them (and for the block-scaled weight gradients' quantization) only.
  const bool variant = Wgu_q || Wdt_q || mx;
  const bool dw_single = variant && !mx_dw;
  const bool lo_parts = !dw_single;
  const bool padded = !mx_dw && (mx || !(Wdt_q && !dact_tok));
  const long long cap_pad = padded ? padded_rows(cap, E) : cap;
  const int32_t* poff = padded ? w.poff : nullptr;
  if (padded) VGG_LAUNCH("pad_offsets", launch_pad_offsets(offsets, E, w.poff, ctx->d_err, s));
  VGG_LAUNCH("gather_rows", launch_gather_rows(offsets, poff, cap_pad, E, sorted_tok, tok_ptr, tok_pairs, cap, T, d,
                                               static_cast<const __nv_bfloat16*>(X),
                                               static_cast<const __nv_bfloat16*>(dO), mx_dw ? nullptr : w.Xs,
                                               mx_dw ? nullptr : w.dOs,
                                               mx ? mq : (dact_tok ? tq : nullptr), dact_tok ? ts : nullptr,
                                               static_cast<uint8_t*>(mx ? mx->dOq : dOq), mx ? nullptr : do_scale,
                                               ctx->d_err, ctx->num_sms, ctx->timeout_ns, s));
  // dA' = dO[tok] W_down[e]; epilogue: dS partials, dH, dU, A' = w A
  if (mx) {
    // block-scaled: A = the sorted dO code rows, its scale blocks per sorted row tile; B = W_down^T codes; the
    // epilogue also writes [dH | dU] block-scaled for the dX GEMM
    VGG_LAUNCH("mx_tile_scales", launch_mx_tile_scales(msf, mx_sfc, T, sorted_tok, static_cast<int>(cap), offsets, E,
                                                       ceil_div(d, 128), ceil_div(cap, BM) + E,
                                                       static_cast<uint8_t*>(mx->do_sf_tiles), s));
    GemmParams p = base_params(ctx);
    p.N = n;
    p.K = d / 2;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.in0 = static_cast<const float*>(H);
    p.in1 = static_cast<const float*>(U);
    p.ld_in = n;
    p.out0 = w.dH;
    p.out1 = w.dU;
    p.out2 = w.Ap;
    p.out3 = lo_parts ? w.dH_lo : nullptr;
    p.out4 = lo_parts ? w.dU_lo : nullptr;
    p.out5 = lo_parts ? w.Ap_lo : nullptr;
    p.ld_out = n;
    p.row_scale = sorted_w;
    p.part = w.part;
    p.part_ld = part_ld;
    p.a_sf = static_cast<const uint8_t*>(mx->do_sf_tiles);
    p.b_sf = static_cast<const uint8_t*>(mx->wdt_sf);
    p.sf_kst = ceil_div(d, 128);
    p.o_q = static_cast<uint8_t*>(mx->HUq);
    p.o_q_ld = 2ll * n;
    p.o_sf = static_cast<uint8_t*>(mx->hu_sf);
    p.o_sf_kst = ceil_div(2 * n, 128);
    const int BN = mx_tile_cols(n);
    Maps m = zero_maps();
    if (!make_map_2d(&m.a0, mx->dOq, d / 2, cap, d / 2, BM) || !make_map_3d(&m.b0, mx->Wdt_q, d / 2, n, E, BN) ||
        !make_store_map_2d(&m.o0, w.dH, false, n, cap, n, 32) || !make_store_map_2d(&m.o1, w.dU, false, n, cap, n, 32) ||
        !make_store_map_2d(&m.o2, w.Ap, false, n, cap, n, 32) || (lo_parts && !make_lo_maps(m, w, n, cap)))
      return MOE_ERR_CUDA;
    m.a1 = m.a0;
    m.b1 = m.b0;
    const int tiles = (ceil_div(cap, BM) + E) * ceil_div(n, BN);
    VGG_LAUNCH("dact_dswiglu_mx", run_dact_dswiglu_mx(BN, p, m, std::min(tiles, ctx->num_sms), s));
  } else if (Wdt_q) {
    // e4m3: the sorted dO code rows (gathered above, else the sorted rows below offsets[E] quantized here),
    // B = W_down^T quantized per row by moe_quantize_dact_weights_e4m3; rows handed to TMA as 16-bit units
    if (!dact_tok)
      VGG_LAUNCH("quantize_do_e4m3", launch_quantize_rows_e4m3(w.dOs, cap, offsets + E, d,
                                                              static_cast<uint8_t*>(dOq), do_scale, s));
    GemmParams p = base_params(ctx);
    p.N = n;
    p.K = d / 2;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.in0 = static_cast<const float*>(H);
    p.in1 = static_cast<const float*>(U);
    p.ld_in = n;
    p.out0 = w.dH;
    p.out1 = w.dU;
    p.out2 = w.Ap;
    p.out3 = lo_parts ? w.dH_lo : nullptr;
    p.out4 = lo_parts ? w.dU_lo : nullptr;
    p.out5 = lo_parts ? w.Ap_lo : nullptr;
    p.ld_out = n;
    p.row_scale = sorted_w;
    p.part = w.part;
    p.part_ld = part_ld;
    p.q_row = do_scale;
    p.q_col = wdt_scale;
    p.q_ld = n;
    Maps m = zero_maps();
    if (!make_map_2d(&m.a0, dOq, d / 2, cap, d / 2, BM) || !make_map_3d(&m.b0, Wdt_q, d / 2, n, E, bn6) ||
        !make_store_map_2d(&m.o0, w.dH, false, n, cap, n, 32) || !make_store_map_2d(&m.o1, w.dU, false, n, cap, n, 32) ||
        !make_store_map_2d(&m.o2, w.Ap, false, n, cap, n, 32) || (lo_parts && !make_lo_maps(m, w, n, cap)))
      return MOE_ERR_CUDA;
    m.a1 = m.a0;
    m.b1 = m.b0;
    const int tiles = (ceil_div(cap, BM) + E) * ceil_div(n, bn6);
    VGG_LAUNCH("dact_dswiglu_e4m3", run_dact_dswiglu_e4m3(bn6, p, m, std::min(tiles, ctx->num_sms), s));
  } else {
    GemmParams p = base_params(ctx);
    p.N = n;
    p.K = d;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.in0 = static_cast<const float*>(H);
    p.in1 = static_cast<const float*>(U);
    p.ld_in = n;
    p.out0 = w.dH;
    p.out1 = w.dU;
    p.out2 = w.Ap;
    p.out3 = lo_parts ? w.dH_lo : nullptr;
    p.out4 = lo_parts ? w.dU_lo : nullptr;
    p.out5 = lo_parts ? w.Ap_lo : nullptr;
    p.ld_out = n;
    p.row_scale = sorted_w;
    p.part = w.part;
    p.part_ld = part_ld;
    p.a_offsets = poff;  // dO's sorted copy may be padded per expert
    const VmShape sh = vm_shape(ctx, bn6, true, cap, E, n);
    Maps m = zero_maps();
    if (!make_map_2d(&m.a0, w.dOs, d, cap_pad, d, BM) || !make_chunked_map_3d(&m.b0, W_down, n, d, E, sh.b_cols / 64) ||
        !make_store_map_2d(&m.o0, w.dH, false, n, cap, n, 32) || !make_store_map_2d(&m.o1, w.dU, false, n, cap, n, 32) ||
        !make_store_map_2d(&m.o2, w.Ap, false, n, cap, n, 32) || (lo_parts && !make_lo_maps(m, w, n, cap)))
      return MOE_ERR_CUDA;
    m.a1 = m.a0;
    m.b1 = m.b0;
    VGG_LAUNCH("dact_dswiglu", run_dact_dswiglu(bn6, sh.pair, p, m, sh.grid, s));
  }
  // dXp = [dH | dU] [W_gate[e]; W_up[e]]
  if (mx) {
    // block-scaled: A = [dH | dU] codes from the dSwiGLU epilogue with their scale blocks, B = [W_gate; W_up]^T
    GemmParams p = base_params(ctx);
    p.N = d;
    p.K = n;  // 2n codes
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.out0 = w.dXp;
    p.ld_out = d;
    p.a_sf = static_cast<const uint8_t*>(mx->hu_sf);
    p.b_sf = static_cast<const uint8_t*>(mx->wgu_sf);
    p.sf_kst = ceil_div(2 * n, 128);
    const int BN = mx_tile_cols(d);
    Maps m = zero_maps();
    if (!make_map_2d(&m.a0, mx->HUq, n, cap, n, BM) || !make_map_3d(&m.b0, mx->Wgu_q, n, d, E, BN) ||
        !make_store_map_2d(&m.o0, w.dXp, false, d, cap, d, 64))
      return MOE_ERR_CUDA;
    m.a1 = m.a0;
    m.b1 = m.b0;
    const int tiles = (ceil_div(cap, BM) + E) * ceil_div(d, BN);
    VGG_LAUNCH("dx_gemm_mx", run_dx_store_mx(BN, p, m, std::min(tiles, ctx->num_sms), s));
  } else if (Wgu_q) {
    // e4m3: each pair's row [dH | dU] quantized (the rows below offsets[E]), B = [W_gate; W_up]^T quantized per
    // row by moe_quantize_dx_weights_e4m3; rows are handed to TMA as 16-bit units (code pairs)
    VGG_LAUNCH("quantize_hu_e4m3", launch_quantize_rows_pair_e4m3(w.dH, w.dU, cap, offsets + E, n,
                                                                  static_cast<uint8_t*>(HUq), hu_scale, s));
    GemmParams p = base_params(ctx);
    p.N = d;
    p.K = n;  // 2n codes
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.out0 = w.dXp;
    p.ld_out = d;
    p.row_scale = hu_scale;
    p.in1 = wgu_scale;
    p.ld_in = d;
    const int BN = gemm_bn(d);
    Maps m = zero_maps();
    if (!make_map_2d(&m.a0, HUq, n, cap, n, BM) || !make_map_3d(&m.b0, Wgu_q, n, d, E, BN) ||
        !make_store_map_2d(&m.o0, w.dXp, false, d, cap, d, 64))
      return MOE_ERR_CUDA;
    m.a1 = m.a0;
    m.b1 = m.b0;
    const int tiles = (ceil_div(cap, BM) + E) * ceil_div(d, BN);
    VGG_LAUNCH("dx_gemm_e4m3", run_dx_store_e4m3(BN, p, m, std::min(tiles, ctx->num_sms), s));
  } else {
    GemmParams p = base_params(ctx);
    p.N = d;
    p.K = 2 * n;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.a_ksplit = n;
    p.b_ksplit = n;
    p.out0 = w.dXp;
    p.ld_out = d;
    const int BN = gemm_bn(d);
    const VmShape sh = vm_shape(ctx, BN, true, cap, E, d);
    Maps m = zero_maps();
    if (!make_map_2d(&m.a0, w.dH, n, cap, n, BM) || !make_map_2d(&m.a1, w.dU, n, cap, n, BM) ||
        !make_chunked_map_3d(&m.b0, W_gate, d, n, E, sh.b_cols / 64) ||
        !make_chunked_map_3d(&m.b1, W_up, d, n, E, sh.b_cols / 64) || !make_store_map_2d(&m.o0, w.dXp, false, d, cap, d, 64))
      return MOE_ERR_CUDA;
    VGG_LAUNCH("dx_gemm", run_dx_store(BN, sh.pair, p, m, sh.grid, s));
  }
  // The per-token chain (wr_transpose, token_backward, dW_r) reads what the GEMMs above wrote and writes only
  // its own outputs and workspace regions, so it runs on the side stream while the weight-gradient GEMMs below
  // run on the caller's; the caller's stream waits for it before returning.  A token_backward block fits on an
  // SM beside a weight-gradient CTA (shared memory, threads, registers), and the side stream has the higher
  // priority, so its blocks take the room the persistent GEMM leaves.
  // With per-launch profiling on, the chain stays on the caller's stream: a kernel's events then bracket that
  // kernel alone, not its overlap with the weight-gradient GEMMs.
  const cudaStream_t s_main = s;
  const bool fork = !ctx->prof;
  if (fork) {
    if (cudaEventRecord(ctx->fork, s_main) != cudaSuccess || cudaStreamWaitEvent(ctx->side, ctx->fork, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    s = ctx->side;
  }
  // per token: dS, router-logit gradient, dX
  VGG_LAUNCH("wr_transpose", launch_transpose_bf16(static_cast<const __nv_bfloat16*>(W_r), d, E, w.WrT, s));
  const int Tp = ceil_div(T, 64) * 64;
  __nv_bfloat16* dL_lo = w.dL + static_cast<size_t>(Tp) * E;
  if (Tp > T) {  // zero rows past the last token in both halves
    if (cudaMemsetAsync(w.dL + static_cast<size_t>(T) * E, 0, sizeof(__nv_bfloat16) * (Tp - T) * E, s) != cudaSuccess ||
        cudaMemsetAsync(dL_lo + static_cast<size_t>(T) * E, 0, sizeof(__nv_bfloat16) * (Tp - T) * E, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  VGG_LAUNCH("token_backward", launch_token_backward(w.part, part_ld, tok_ptr, tok_pairs, offsets, E, sorted_w,
                                                     topk_ids, topk_w, K, w.dXp, w.WrT, T, d, cap, dS, dlogits, w.dL,
                                                     dL_lo, static_cast<__nv_bfloat16*>(dX), ctx->d_err, s));
  // dW_r = X^T dlogits, split over tokens.  dlogits enters as X^T hi + X^T lo with hi = bf16(dlogits) and
  // lo = bf16(dlogits - hi), about 16 significant bits: a single bf16 rounding of dlogits costs up to a few
  // percent on the columns of heavily loaded experts, whose gradient sums thousands of tokens' rounding
  // errors.  One launch reduces over 2 Tp rows: [hi; lo] against X read twice (rows k >= Tp wrap to k - Tp).
  {
    GemmParams p = base_params(ctx);
    p.M = d;
    p.N = E;
    p.K = 2 * Tp;
    p.groups = 1;
    p.a_kwrap = Tp;
    const int BN = gemm_bn(E);
    const int tiles = ceil_div(d, BM) * ceil_div(E, BN);
    int split = std::max(1, std::min(ctx->num_sms / std::max(tiles, 1), kMaxSplitK));
    split = std::max(1, std::min(split, ceil_div(2 * Tp, 8 * BK)));
    p.split_k = split;
    p.ld_out = E;
    p.out0 = w.wr_part;
    Maps m = zero_maps();
    if (!make_map_2d(&m.a0, X, d, T, d, 64) || !make_map_2d(&m.b0, w.dL, E, 2 * static_cast<uint64_t>(Tp), E, 64) ||
        !make_store_map_3d(&m.o0, w.wr_part, true, E, d, split, 32))
      return MOE_ERR_CUDA;
    m.a1 = m.a0;
    m.b1 = m.b0;
    VGG_LAUNCH("dwr_gemm", run_dense_mn_store(BN, p, m, std::min(tiles * split, ctx->num_sms), s));
    VGG_LAUNCH("dwr_reduce", launch_splitk_reduce(w.wr_part, split, static_cast<long long>(d) * E, dW_r, s));
  }
  if (fork && cudaEventRecord(ctx->join, s) != cudaSuccess) return MOE_ERR_CUDA;
  s = s_main;
  if (mx_dw) {
    // block-scaled weight gradients: blocks of 32 tokens of one expert along each operand column.  One launch
    // writes the four operands transposed (K-major codes over the per-expert stages) with their scale blocks,
    // from dH, dU and A' (high + low parts) at the sorted positions and from X and dO through the token index.
    const MxDwWs v = carve_mx_dw(mx->dw_ws, d, E, n, cap);
    VGG_LAUNCH("mx_stage_offsets", launch_mx_stage_offsets(offsets, E, v.kp, ctx->d_err, s));
    MxColJobs jobs{};
    jobs.job[0] = MxColJob{w.dH, w.dH_lo, nullptr, cap, n, n, 0, v.gu_a, v.gu_a_sf, BM};
    jobs.job[1] = MxColJob{w.dU, w.dU_lo, nullptr, cap, n, n, n, v.gu_a, v.gu_a_sf, BM};
    jobs.job[2] = MxColJob{static_cast<const __nv_bfloat16*>(X), nullptr, sorted_tok, T, d, d, 0, v.gu_b, v.gu_b_sf,
                           v.bn_gu};
    jobs.job[3] = MxColJob{static_cast<const __nv_bfloat16*>(dO), nullptr, sorted_tok, T, d, d, 0, v.dn_a, v.dn_a_sf,
                           BM};
    jobs.job[4] = MxColJob{w.Ap, w.Ap_lo, nullptr, cap, n, n, 0, v.dn_b, v.dn_b_sf, v.bn_dn};
    // scale bytes of operand rows that no job writes (past M or N in a tile) hold 127 (scale 1)
    VGG_CUDA(cudaMemsetAsync(v.gu_a_sf, 127, static_cast<size_t>(static_cast<uint8_t*>(mx->dw_ws) + v.bytes - v.gu_a_sf),
                             s));
    VGG_LAUNCH("quantize_cols_mx", launch_quantize_cols_mx(jobs, 5, offsets, v.kp, E, cap, v.kq, v.kst, ctx->d_err,
                                                           s));
    // [dW_gate; dW_up][e] = [dH | dU]^T X over the expert's stages (M = 2n, N = d)
    {
      GemmParams p = base_params(ctx);
      p.M = 2 * n;
      p.N = d;
      p.K = static_cast<int>(v.kq / 2);
      p.groups = E;
      p.offsets = v.kp;
      p.rows_cap = static_cast<int>(v.kq / 2);
      p.out0 = dW_gate;
      p.out1 = dW_up;
      p.out_rows_split = n;
      p.ld_out = d;
      p.a_sf = v.gu_a_sf;
      p.b_sf = v.gu_b_sf;
      p.sf_kst = v.kst;
      Maps m = zero_maps();
      if (!make_map_2d(&m.a0, v.gu_a, v.kq / 2, 2 * n, v.kq / 2, BM) ||
          !make_map_3d(&m.b0, v.gu_b, v.kq / 2, d, 1, v.bn_gu) ||
          !make_store_map_3d(&m.o0, dW_gate, f32, d, n, E, 64) || !make_store_map_3d(&m.o1, dW_up, f32, d, n, E, 64))
        return MOE_ERR_CUDA;
      m.a1 = m.a0;
      m.b1 = m.b0;
      const long long tiles = static_cast<long long>(E) * ceil_div(2 * n, BM) * ceil_div(d, v.bn_gu);
      VGG_LAUNCH("dw_gate_up_mx", run_dw_mx(v.bn_gu, f32, p, m, static_cast<int>(std::min<long long>(tiles, ctx->num_sms)), s));
    }
    // dW_down[e] = dO^T A' over the expert's stages (M = d, N = n)
    {
      GemmParams p = base_params(ctx);
      p.M = d;
      p.N = n;
      p.K = static_cast<int>(v.kq / 2);
      p.groups = E;
      p.offsets = v.kp;
      p.rows_cap = static_cast<int>(v.kq / 2);
      p.out0 = dW_down;
      p.ld_out = n;
      p.a_sf = v.dn_a_sf;
      p.b_sf = v.dn_b_sf;
      p.sf_kst = v.kst;
      Maps m = zero_maps();
      if (!make_map_2d(&m.a0, v.dn_a, v.kq / 2, d, v.kq / 2, BM) ||
          !make_map_3d(&m.b0, v.dn_b, v.kq / 2, n, 1, v.bn_dn) || !make_store_map_3d(&m.o0, dW_down, f32, n, d, E, 64))
        return MOE_ERR_CUDA;
      m.a1 = m.a0;
      m.b1 = m.b0;
      const long long tiles = static_cast<long long>(E) * ceil_div(d, BM) * ceil_div(n, v.bn_dn);
      VGG_LAUNCH("dw_down_mx", run_dw_mx(v.bn_dn, f32, p, m, static_cast<int>(std::min<long long>(tiles, ctx->num_sms)), s));
    }
    if (fork && cudaStreamWaitEvent(s_main, ctx->join, 0) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  // varlen-K weight gradients: [dW_gate; dW_up][e] = [dH | dU]^T X[tok], with [dH | dU] as high and low
  // bf16 parts (about 16 significant bits of the fp32 gradients)
  {
    GemmParams p = base_params(ctx);
    p.M = 2 * n;
    p.N = d;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.a_colsplit = n;
    p.b_chunked = 1;
    p.b_offsets = poff;
    p.out0 = dW_gate;
    p.out1 = dW_up;
    p.out_rows_split = n;
    p.ld_out = d;
    const int BN = gemm_bn(d);
    const DwShape sh = dw_shape(ctx, BN, poff != nullptr && !dw_single, E, 2 * n, d);
    Maps m = zero_maps();
    if (!make_map_2d(&m.a0, w.dH, n, cap, n, 64) || !make_map_2d(&m.a1, w.dU, n, cap, n, 64) ||
        (!dw_single && (!make_map_2d(&m.a2, w.dH_lo, n, cap, n, 64) || !make_map_2d(&m.a3, w.dU_lo, n, cap, n, 64))) ||
        !make_chunked_map_2d(&m.b0, w.Xs, d, cap_pad, sh.b_chunks) ||
        !make_store_map_3d(&m.o0, dW_gate, f32, d, n, E, 64) || !make_store_map_3d(&m.o1, dW_up, f32, d, n, E, 64))
      return MOE_ERR_CUDA;
    m.b1 = m.b0;
    if (dw_single) VGG_LAUNCH("dw_gate_up", run_dw_tiled(BN, f32, p, m, sh.grid, s));
    else VGG_LAUNCH("dw_gate_up", run_dw_dual(BN, f32, false, sh.pair, p, m, sh.grid, s));
  }
  // dW_down[e] = dO[tok]^T A' (the combine weight is folded into A' = w A), computed as its transpose
  // A'^T dO[tok] with A' as high and low bf16 parts (tile rows = columns of dW_down) and stored through
  // transposed blocks
  {
    GemmParams p = base_params(ctx);
    p.M = n;
    p.N = d;
    p.groups = E;
    p.offsets = offsets;
    p.rows_cap = static_cast<int>(cap);
    p.out0 = dW_down;
    p.ld_out = n;
    const int BN = gemm_bn(d);
    const DwShape sh = dw_shape(ctx, BN, poff != nullptr && !dw_single, E, n, d);
    Maps m = zero_maps();
    p.b_chunked = 1;
    p.b_offsets = poff;
    if (!make_map_2d(&m.a0, w.Ap, n, cap, n, 64) || (!dw_single && !make_map_2d(&m.a2, w.Ap_lo, n, cap, n, 64)) ||
        !make_chunked_map_2d(&m.b0, w.dOs, d, cap_pad, sh.b_chunks) ||
        !make_store_map_3d(&m.o0, dW_down, f32, n, d, E, 32))
      return MOE_ERR_CUDA;
    m.a1 = m.a0;
    m.a3 = m.a2;
    m.b1 = m.b0;
    if (dw_single) VGG_LAUNCH("dw_down", run_dw_tiled_trans(BN, f32, p, m, sh.grid, s));
    else VGG_LAUNCH("dw_down", run_dw_dual(BN, f32, true, sh.pair, p, m, sh.grid, s));
  }
  if (fork && cudaStreamWaitEvent(s, ctx->join, 0) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_backward(moe_ctx* ctx, const void* dO, const void* X, const void* W_r, const void* W_gate,
                 const void* W_up, const void* W_down, int T, int d, int E, int n, int K, int m_tile, long long cap,
                 const int32_t* topk_ids, const float* topk_w, const int32_t* offsets, const int32_t* sorted_tok,
                 const float* sorted_w, const int32_t* tok_ptr, const int32_t* tok_pairs, const void* H,
                 const void* U, void* dX, void* dW_gate, void* dW_up, void* dW_down, int dW_fp32, float* dS,
                 float* dlogits, float* dW_r, void* ws, size_t ws_bytes, moe_stream_t stream) {
  return backward_impl(ctx, dO, X, W_r, W_gate, W_up, W_down, T, d, E, n, K, m_tile, cap, topk_ids, topk_w, offsets,
                       sorted_tok, sorted_w, tok_ptr, tok_pairs, H, U, dX, dW_gate, dW_up, dW_down, dW_fp32, dS,
                       dlogits, dW_r, ws, ws_bytes, stream, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                       nullptr, nullptr);
}

int moe_backward_e4m3(moe_ctx* ctx, const void* dO, const void* X, const void* W_r, const void* W_gate,
                      const void* W_up, const void* W_down, const void* Wgu_q, const float* wgu_scale,
                      const void* Wdt_q, const float* wdt_scale, int T, int d, int E, int n, int K, int m_tile,
                      long long cap, const int32_t* topk_ids, const float* topk_w, const int32_t* offsets,
                      const int32_t* sorted_tok, const float* sorted_w, const int32_t* tok_ptr,
                      const int32_t* tok_pairs, const void* H, const void* U, void* HUq, float* hu_scale, void* dOq,
                      float* do_scale, void* dX, void* dW_gate, void* dW_up, void* dW_down, int dW_fp32, float* dS,
                      float* dlogits, float* dW_r, void* ws, size_t ws_bytes, moe_stream_t stream) {
  // each e4m3 GEMM is optional: a NULL weight code array keeps that GEMM in bf16
  VGG_REQUIRE(!Wgu_q || (wgu_scale && HUq && hu_scale && aligned16(Wgu_q) && aligned16(HUq)));
  VGG_REQUIRE(!Wdt_q || (wdt_scale && dOq && do_scale && aligned16(Wdt_q) && aligned16(dOq)));
  return backward_impl(ctx, dO, X, W_r, W_gate, W_up, W_down, T, d, E, n, K, m_tile, cap, topk_ids, topk_w, offsets,
                       sorted_tok, sorted_w, tok_ptr, tok_pairs, H, U, dX, dW_gate, dW_up, dW_down, dW_fp32, dS,
                       dlogits, dW_r, ws, ws_bytes, stream, Wgu_q, wgu_scale, HUq, hu_scale, Wdt_q, wdt_scale, dOq,
                       do_scale);
}

int moe_backward_mx(moe_ctx* ctx, const void* dO, const void* X, const void* W_r, const void* W_gate, const void* W_up,
                    const void* W_down, const void* Wdt_q, const void* wdt_sf, const void* Wgu_q, const void* wgu_sf,
                    int T, int d, int E, int n, int K, int m_tile, long long cap, const int32_t* topk_ids,
                    const float* topk_w, const int32_t* offsets, const int32_t* sorted_tok, const float* sorted_w,
                    const int32_t* tok_ptr, const int32_t* tok_pairs, const void* H, const void* U, void* dOq,
                    void* do_sf_tiles, void* HUq, void* hu_sf, void* dX, void* dW_gate, void* dW_up, void* dW_down,
                    int dW_fp32, float* dS, float* dlogits, float* dW_r, void* ws, size_t ws_bytes, void* dw_ws,
                    size_t dw_ws_bytes, moe_stream_t stream) {
  VGG_REQUIRE(Wdt_q && wdt_sf && Wgu_q && wgu_sf && dOq && do_sf_tiles && HUq && hu_sf);
  VGG_REQUIRE(aligned16(Wdt_q) && aligned16(wdt_sf) && aligned16(Wgu_q) && aligned16(wgu_sf) && aligned16(dOq) &&
              aligned16(do_sf_tiles) && aligned16(HUq) && aligned16(hu_sf));
  // the block-scaled weight gradients: a workspace of moe_mx_dw_ws_bytes, 256-byte aligned (null: two-part bf16)
  VGG_REQUIRE(!dw_ws || ((reinterpret_cast<uintptr_t>(dw_ws) & (kAlign - 1)) == 0 &&
                         dw_ws_bytes >= moe_mx_dw_ws_bytes(d, E, n, cap) && moe_mx_dw_ws_bytes(d, E, n, cap) > 0));
  const MxBwd mx{Wdt_q, wdt_sf, Wgu_q, wgu_sf, dOq, do_sf_tiles, HUq, hu_sf, dw_ws};
  return backward_impl(ctx, dO, X, W_r, W_gate, W_up, W_down, T, d, E, n, K, m_tile, cap, topk_ids, topk_w, offsets,
                       sorted_tok, sorted_w, tok_ptr, tok_pairs, H, U, dX, dW_gate, dW_up, dW_down, dW_fp32, dS,
                       dlogits, dW_r, ws, ws_bytes, stream, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                       nullptr, nullptr, &mx);
}

int moe_quantize_bwd_weights_mx(moe_ctx* ctx, const void* W_gate, const void* W_up, const void* W_down, int E, int d,
                                int n, void* tmp, void* Wdt_q, void* wdt_sf, void* Wgu_q, void* wgu_sf,
                                moe_stream_t stream) {
  VGG_REQUIRE(ctx && W_gate && W_up && W_down && tmp && Wdt_q && wdt_sf && Wgu_q && wgu_sf);
  VGG_REQUIRE(E >= 1 && E <= kMaxGroups && d >= 64 && d % 64 == 0 && n >= 64 && n % 64 == 0);
  VGG_REQUIRE(aligned16(W_gate) && aligned16(W_up) && aligned16(W_down) && aligned16(tmp) && aligned16(Wdt_q) &&
              aligned16(wdt_sf) && aligned16(Wgu_q) && aligned16(wgu_sf));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  __nv_bfloat16* t = static_cast<__nv_bfloat16*>(tmp);
  const int bn = mx_tile_cols(n), bd = mx_tile_cols(d);
  VGG_CUDA(cudaMemsetAsync(wdt_sf, 127, static_cast<size_t>(moe_mx_weight_sf_bytes(E, d, n, 2)), s));
  VGG_CUDA(cudaMemsetAsync(wgu_sf, 127, static_cast<size_t>(moe_mx_weight_sf_bytes(E, d, n, 3)), s));
  // W_down^T [E][n][d], blocks along d
  VGG_LAUNCH("quantize_mx_weights", launch_transpose_into_bf16(static_cast<const __nv_bfloat16*>(W_down), E, d, n, t,
                                                               d, 0, s));
  VGG_LAUNCH("quantize_mx_weights", launch_quantize_weight_mx(t, E, n, d, static_cast<uint8_t*>(Wdt_q),
                                                              static_cast<uint8_t*>(wdt_sf), bn, 0, ceil_div(n, bn),
                                                              ceil_div(d, 128), mx_b_blocks(bn), s));
  // [W_gate; W_up]^T [E][d][2n], blocks along 2n (the transposes follow the quantization above on the stream)
  VGG_LAUNCH("quantize_mx_weights", launch_transpose_into_bf16(static_cast<const __nv_bfloat16*>(W_gate), E, n, d, t,
                                                               2 * n, 0, s));
  VGG_LAUNCH("quantize_mx_weights", launch_transpose_into_bf16(static_cast<const __nv_bfloat16*>(W_up), E, n, d, t,
                                                               2 * n, n, s));
  VGG_LAUNCH("quantize_mx_weights", launch_quantize_weight_mx(t, E, d, 2 * n, static_cast<uint8_t*>(Wgu_q),
                                                              static_cast<uint8_t*>(wgu_sf), bd, 0, ceil_div(d, bd),
                                                              ceil_div(2 * n, 128), mx_b_blocks(bd), s));
  return MOE_OK;
}

int moe_quantize_dact_weights_e4m3(moe_ctx* ctx, const void* W_down, int E, int n, int d, void* tmp, void* Wdt_q,
                                   float* wdt_scale, moe_stream_t stream) {
  VGG_REQUIRE(ctx && W_down && tmp && Wdt_q && wdt_scale);
  VGG_REQUIRE(shapes_ok(1, d, E, n, 1));
  VGG_REQUIRE(aligned16(W_down) && aligned16(tmp) && aligned16(Wdt_q));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  __nv_bfloat16* t = static_cast<__nv_bfloat16*>(tmp);
  VGG_LAUNCH("quantize_e4m3", launch_transpose_into_bf16(static_cast<const __nv_bfloat16*>(W_down), E, d, n, t, d, 0,
                                                         s));
  VGG_LAUNCH("quantize_e4m3", launch_quantize_rows_e4m3(t, static_cast<long long>(E) * n, nullptr, d,
                                                        static_cast<uint8_t*>(Wdt_q), wdt_scale, s));
  return MOE_OK;
}

int moe_quantize_dx_weights_e4m3(moe_ctx* ctx, const void* W_gate, const void* W_up, int E, int n, int d, void* tmp,
                                 void* Wgu_q, float* wgu_scale, moe_stream_t stream) {
  VGG_REQUIRE(ctx && W_gate && W_up && tmp && Wgu_q && wgu_scale);
  VGG_REQUIRE(shapes_ok(1, d, E, n, 1));
  VGG_REQUIRE(aligned16(W_gate) && aligned16(W_up) && aligned16(tmp) && aligned16(Wgu_q));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  __nv_bfloat16* t = static_cast<__nv_bfloat16*>(tmp);
  VGG_LAUNCH("quantize_e4m3", launch_transpose_into_bf16(static_cast<const __nv_bfloat16*>(W_gate), E, n, d, t, 2 * n,
                                                         0, s));
  VGG_LAUNCH("quantize_e4m3", launch_transpose_into_bf16(static_cast<const __nv_bfloat16*>(W_up), E, n, d, t, 2 * n, n,
                                                         s));
  VGG_LAUNCH("quantize_e4m3", launch_quantize_rows_e4m3(t, static_cast<long long>(E) * d, nullptr, 2 * n,
                                                        static_cast<uint8_t*>(Wgu_q), wgu_scale, s));
  return MOE_OK;
}

int moe_test_gemm_varlen_m(moe_ctx* ctx, const void* A, const int32_t* idx, const void* B, int B_kmajor, int G,
                           int rows_a, int K, int N, long long cap, const int32_t* offsets, float* D,
                           moe_stream_t stream) {
  VGG_REQUIRE(ctx && A && B && offsets && D);
  VGG_REQUIRE(G >= 1 && G <= kMaxGroups && rows_a >= 1 && K >= 64 && K % 64 == 0 && N >= 8 && N % 8 == 0);
  VGG_REQUIRE(cap >= 1 && cap < INT_MAX && aligned16(A) && aligned16(B) && aligned16(D));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  GemmParams p = base_params(ctx);
  p.N = N;
  p.K = K;
  p.groups = G;
  p.offsets = offsets;
  p.rows_cap = static_cast<int>(cap);
  p.a_idx = idx;
  p.a_rows = rows_a;
  p.a_src = static_cast<const __nv_bfloat16*>(A);
  p.a_ld = K;
  p.out0 = D;
  p.ld_out = N;
  Maps m = zero_maps();
  if (!idx && !make_map_2d(&m.a0, A, K, rows_a, K, BM)) return MOE_ERR_CUDA;
  m.a1 = m.a0;
  if (B_kmajor) {
    if (!make_map_3d(&m.b0, B, K, N, G, 128)) return MOE_ERR_CUDA;
  } else {
    if (N % 64 || !make_chunked_map_3d(&m.b0, B, N, K, G, 2)) return MOE_ERR_CUDA;
  }
  m.b1 = m.b0;
  if (!make_store_map_2d(&m.o0, D, true, N, cap, N, 32)) return MOE_ERR_CUDA;
  // 128-column tiles, or CTA pairs on 256-column tiles (each CTA loads the same 128-column B boxes)
  const VmShape sh = vm_shape(ctx, idx ? 128 : 256, true, cap, G, N);
  const int tiles = (ceil_div(cap, BM) + G) * ceil_div(N, 128);
  return cuda_status(run_test_m(idx != nullptr, B_kmajor, sh.pair, p, m,
                                sh.pair ? sh.grid : std::min(tiles, ctx->num_sms), static_cast<cudaStream_t>(stream)));
}

int moe_test_gemm_varlen_m_dual(moe_ctx* ctx, const void* A_hi, const void* A_lo, const void* B, int G, int rows_a,
                                int K, int N, long long cap, const int32_t* offsets, float* D, moe_stream_t stream) {
  VGG_REQUIRE(ctx && A_hi && A_lo && B && offsets && D);
  VGG_REQUIRE(G >= 1 && G <= kMaxGroups && rows_a >= 1 && K >= 64 && K % 64 == 0 && N >= 8 && N % 8 == 0);
  VGG_REQUIRE(cap >= 1 && cap < INT_MAX && rows_a >= cap && aligned16(A_hi) && aligned16(A_lo) && aligned16(B) &&
              aligned16(D));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  GemmParams p = base_params(ctx);
  p.N = N;
  p.K = K;
  p.groups = G;
  p.offsets = offsets;
  p.rows_cap = static_cast<int>(cap);
  p.out0 = D;
  p.ld_out = N;
  const VmShape sh = vm_shape(ctx, 256, true, cap, G, N);
  Maps m = zero_maps();
  if (!make_map_2d(&m.a0, A_hi, K, rows_a, K, BM) || !make_map_2d(&m.a2, A_lo, K, rows_a, K, BM) ||
      !make_map_3d(&m.b0, B, K, N, G, sh.b_cols) || !make_store_map_2d(&m.o0, D, true, N, cap, N, 32))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.a3 = m.a2;
  m.b1 = m.b0;
  return cuda_status(run_test_m_dual(sh.pair, p, m, sh.grid, static_cast<cudaStream_t>(stream)));
}

int moe_test_gemm_varlen_k(moe_ctx* ctx, const void* A, const int32_t* idx_a, int rows_a, const void* B,
                           const int32_t* idx_b, int rows_b, int G, int M, int N, long long cap,
                           const int32_t* offsets, float* D, moe_stream_t stream) {
  VGG_REQUIRE(ctx && A && B && offsets && D);
  VGG_REQUIRE(idx_a == nullptr || idx_b == nullptr);  // at most one operand is gathered
  VGG_REQUIRE(G >= 1 && G <= kMaxGroups && M >= 64 && M % 64 == 0 && N >= 64 && N % 64 == 0 && rows_a >= 1 &&
              rows_b >= 1);
  VGG_REQUIRE(cap >= 1 && cap < INT_MAX && aligned16(A) && aligned16(B) && aligned16(D));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  GemmParams p = base_params(ctx);
  p.M = M;
  p.N = N;
  p.groups = G;
  p.offsets = offsets;
  p.rows_cap = static_cast<int>(cap);
  p.a_idx = idx_a;
  p.a_rows = rows_a;
  p.a_src = static_cast<const __nv_bfloat16*>(A);
  p.a_ld = M;
  p.b_idx = idx_b;
  p.b_rows = rows_b;
  p.b_chunked = 1;
  p.b_src = static_cast<const __nv_bfloat16*>(B);
  p.b_ld = N;
  p.out0 = D;
  p.ld_out = N;
  const int BN = gemm_bn(N);
  Maps m = zero_maps();
  if ((!idx_a && !make_map_2d(&m.a0, A, M, rows_a, M, 64)) || (!idx_b && !make_chunked_map_2d(&m.b0, B, N, rows_b, BN / 64)) ||
      !make_store_map_3d(&m.o0, D, true, N, M, G, 32))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.b1 = m.b0;
  const int tiles = G * ceil_div(M, BM) * ceil_div(N, BN);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int grid = std::min(tiles, ctx->num_sms);
  if (idx_b) return cuda_status(run_dw_gate_up(BN, true, p, m, grid, s));
  if (idx_a) return cuda_status(run_dw_down(BN, true, p, m, grid, s));
  return cuda_status(run_dw_tiled(BN, true, p, m, grid, s));
}

int moe_test_gemm_varlen_k_dual(moe_ctx* ctx, const void* A_hi, const void* A_lo, int rows_a, const void* B, int rows_b,
                                int G, int M, int N, long long cap, const int32_t* offsets, const int32_t* b_offsets,
                                int trans, float* D, moe_stream_t stream) {
  VGG_REQUIRE(ctx && A_hi && A_lo && B && offsets && D);
  VGG_REQUIRE(G >= 1 && G <= kMaxGroups && M >= 64 && M % 64 == 0 && N >= 64 && N % 64 == 0 && rows_a >= 1 &&
              rows_b >= 1);
  VGG_REQUIRE(cap >= 1 && cap < INT_MAX && aligned16(A_hi) && aligned16(A_lo) && aligned16(B) && aligned16(D));
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  GemmParams p = base_params(ctx);
  p.M = M;
  p.N = N;
  p.groups = G;
  p.offsets = offsets;
  p.rows_cap = static_cast<int>(cap);
  p.b_chunked = 1;
  p.b_offsets = b_offsets;
  p.out0 = D;
  p.ld_out = N;
  const int BN = gemm_bn(N);
  const DwShape sh = dw_shape(ctx, BN, b_offsets != nullptr, G, M, N);
  Maps m = zero_maps();
  if (!make_map_2d(&m.a0, A_hi, M, rows_a, M, 64) || !make_map_2d(&m.a2, A_lo, M, rows_a, M, 64) ||
      !make_chunked_map_2d(&m.b0, B, N, rows_b, sh.b_chunks) ||
      !(trans ? make_store_map_3d(&m.o0, D, true, M, N, G, 32) : make_store_map_3d(&m.o0, D, true, N, M, G, 32)))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.a3 = m.a2;
  m.b1 = m.b0;
  return cuda_status(run_dw_dual(BN, true, trans != 0, sh.pair, p, m, sh.grid, static_cast<cudaStream_t>(stream)));
}

int moe_profile_enable(moe_ctx* ctx, int enable) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (enable && ctx->pool.empty()) {
    ctx->pool.resize(kProfPool);
    for (auto& e : ctx->pool)
      if (cudaEventCreate(&e) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (!enable) prof_drain(ctx);
  ctx->prof = enable != 0;
  return MOE_OK;
}

int moe_profile_read(moe_ctx* ctx, int max_kernels, char* names, double* total_ms, long long* launches,
                     int* n_kernels) {
  if (!ctx || max_kernels < 0 || !n_kernels) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  prof_drain(ctx);
  const int n = static_cast<int>(ctx->names.size());
  *n_kernels = n;
  for (int i = 0; i < n && i < max_kernels; ++i) {
    if (names) {
      std::strncpy(names + 32 * i, ctx->names[i].c_str(), 31);
      names[32 * i + 31] = 0;
    }
    if (total_ms) total_ms[i] = ctx->total_ms[i];
    if (launches) launches[i] = ctx->launches[i];
    ctx->total_ms[i] = 0.0;
    ctx->launches[i] = 0;
  }
  return MOE_OK;
}

int moe_test_wait_timeout(moe_ctx* ctx, unsigned long long timeout_ns, moe_stream_t stream) {
  VGG_REQUIRE(ctx && timeout_ns > 0 && timeout_ns <= 10000000000ull);
  DeviceGuard g(ctx->device);
  VGG_REQUIRE(g.ok);
  return cuda_status(launch_wait_timeout_probe(ctx->d_err, timeout_ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

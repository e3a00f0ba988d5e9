/*
 * moe.h — C ABI of the GB300 (sm_103a) MoE expert-layer hot path.
 *
 * What the calls compute, with the passages they follow (page title, section):
 *   [GG]  "DeepSeek 계열 MoE 학습 가속: Python expert loop → grouped GEMM"
 *   [EP]  "EP: Expert를 나누고 토큰 보내기"
 *   [SM]  "SonicMoE: IO·타일 인식 최적화로 MoE 학습 가속하기"
 *   [DEP] "Deep EP"
 *
 * Shapes: T tokens, d model width, E experts, n expert width, K experts per token.
 * Layouts are row-major and contiguous.  Expert weights are the stacked
 * nn.Linear (out, in) matrices ([GG] "(5) Weight stacking"):
 *   X[T,d] bf16, W_r[d,E] bf16, bias[E] fp32,
 *   W_gate[E,n,d] bf16, W_up[E,n,d] bf16, W_down[E,d,n] bf16.
 * Pairs: one (token, expert) assignment.  P = T*K without token rounding; with
 * token rounding P is computed on the device and is at most
 * moe_pair_capacity(T, E, K, m_tile).  Arrays indexed by pair are sized for
 * that capacity ("cap") and ordered by expert, tokens ascending inside an
 * expert (the "sorted" order of [GG] "(1)-(3) 토큰 정렬").
 *
 * Conventions shared by every call:
 * - All tensor pointers are DEVICE pointers owned by the caller; the library
 *   neither allocates nor frees per call.  Scratch memory comes from the
 *   caller's workspace `ws` of at least moe_workspace_bytes(...) bytes
 *   (256-byte aligned).  moe_create allocates one small device error word.
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *   default stream) and returns a host-side status.  Argument errors
 *   (NULL pointers, sizes out of range, d or n not multiples of 64,
 *   misaligned pointers) return MOE_ERR_INVALID_ARG before anything is
 *   launched; a failed launch returns MOE_ERR_CUDA.
 * - Errors found on the device (an expert id out of range, corrupt offsets,
 *   a pair count beyond capacity, a bounded wait that timed out) never trap:
 *   the kernel records a code in the context's error word and returns early.
 *   moe_get_error() synchronizes the device and reports it.
 * - Supported sizes: 1 <= K <= 8, K <= E <= 1024, T <= 65536,
 *   d and n multiples of 64, m_tile 0 or a multiple of 64.
 * - No C++ exception crosses this interface.
 */
#ifndef VGG_MOE_H
#define VGG_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx moe_ctx;
typedef void* moe_stream_t; /* cudaStream_t */

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_CUDA = 3,
  MOE_ERR_DEVICE = 4,         /* a kernel recorded a data error; see moe_get_error */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded device wait gave up */
};

/* Device-side error codes reported by moe_get_error. */
enum moe_device_error {
  MOE_DEV_OK = 0,
  MOE_DEV_BAD_EXPERT = 1,
  MOE_DEV_DUP_EXPERT = 2,
  MOE_DEV_BAD_OFFSETS = 3,
  MOE_DEV_TIMEOUT = 4,
  MOE_DEV_CAPACITY = 5,
};

/* Create a context on `device` (makes it current).  Allocates the 16-byte error word. */
int moe_create(moe_ctx** out, int device);
int moe_destroy(moe_ctx* ctx);
const char* moe_status_str(int status);

/* Synchronize the device, return the first device error code in *device_error
 * (0 = none) and clear it.  Returns MOE_OK, or MOE_ERR_DEVICE /
 * MOE_ERR_DEVICE_TIMEOUT when a code was pending, or MOE_ERR_CUDA. */
int moe_get_error(moe_ctx* ctx, int* device_error);

/* Bound of every device spin-wait, in nanoseconds (default 2 s). */
int moe_set_wait_timeout(moe_ctx* ctx, unsigned long long timeout_ns);

/*
 * CTA pairs (tcgen05 cta_group::2): a cluster of two CTAs computes each 256-row tile with M = 256
 * UMMAs issued by the even CTA, each CTA holding its 128 rows of A and half of B's 256 columns.
 * varlen_m (0/1): the tiled varlen-M GEMMs with 256-column tiles (dX, dA' with the dSwiGLU epilogue, the
 * two-part down projection); varlen_k (0/1): the two-part weight-gradient GEMMs on padded sorted rows.
 * Both default to 0: on GB300 they measured slower than one CTA per 128-row tile (the varlen-K tiles
 * are bound by their epilogue, the varlen-M ones gain nothing from halving each SM's B bytes).  Results
 * are identical either way up to fp32 summation order.  Returns MOE_ERR_INVALID_ARG for a NULL ctx or a
 * flag other than 0 or 1.
 */
int moe_set_cta_pairs(moe_ctx* ctx, int varlen_m, int varlen_k);

/* Pair capacity for the pair-indexed arrays: T*K, plus E*m_tile/2 under token rounding. */
long long moe_pair_capacity(int T, int E, int K, int m_tile);

/*
 * Slots per expert of the capacity dispatch (moe_permute_capacity):
 * C = ceil(capacity_factor * T * K / E), the factor times the mean load, evaluated left to right in
 * double precision.  [DEP] "Drop/Padding 방식" names the capacity factor but gives no formula; this
 * is the library's reading.  Returns 0 for T, E or K below 1 or a factor that is not in (0, 1e6].
 */
long long moe_expert_capacity(int T, int E, int K, double capacity_factor);

/* Workspace needed by moe_route / moe_permute / moe_grouped_gemm_fwd / moe_backward for these sizes. */
size_t moe_workspace_bytes(int T, int d, int E, int n, int K, int m_tile);

/*
 * moe_route — router logits, top-K token choice and combine weights.
 * [DEP] "1) Router": scores every expert for each token and returns the top-k
 * expert indices and scores, [BN, k] each.  [EP] "여러 Expert의 결과도 같은
 * 토큰으로 돌아오기": the combine weights are kept apart from the selection.
 *
 *   logits[t,e] = sum_i X[t,i] W_r[i,e] + bias[e]              (fp32 accumulation)
 *   topk_ids[t,:] = the K largest logits, largest first, ties to the lower expert
 *   topk_w[t,k]  = exp(l_k - l_max) / sum_{j in top-K} exp(l_j - l_max)
 *   scores[t,e]  = softmax over all E experts (only when scores != NULL)
 *
 * X[T,d], W_r[d,E] bf16; bias[E] fp32 or NULL; outputs logits[T,E] fp32,
 * scores[T,E] fp32 (NULL allowed unless token rounding follows),
 * topk_ids[T,K] int32, topk_w[T,K] fp32.
 */
int moe_route(moe_ctx* ctx, const void* X, const void* W_r, const float* bias, int T, int d, int E, int K,
              float* logits, float* scores, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
              moe_stream_t stream);

/*
 * moe_permute — group the (token, expert) pairs by expert.
 * [GG] "(1)-(3) 토큰 정렬": flatten topk_ids, sort by expert (stable: tokens
 * ascending inside an expert), bincount per expert.  [DEP] table "Ragged vs
 * Padding": the ragged layout's offset/index metadata.  [EP] "토큰을 Expert로
 * 보내고 원래 위치로 돌려받기": every result is tracked back to its token.
 *
 * With m_tile > 0 (token rounding, [SM] "5 기여 ③ Token Rounding 라우팅"):
 * each expert's count c_e becomes r_e = m_tile*floor((c_e + m_tile/2)/m_tile)
 * (at most m_tile*floor(T/m_tile)); short experts are padded with the tokens
 * not routed to them in descending scores[t,e] (ties: lower token first),
 * long ones drop routed tokens in ascending score (ties: higher token first).
 * A padded pair's weight is exp(l_e - l_max)/sum_{j in top-K} exp(l_j - l_max).
 * `scores` and `logits` are then required; otherwise they may be NULL.
 *
 * Outputs: counts[E], offsets[E+1] (exclusive scan, offsets[E] = P),
 * sorted_tok[cap] (token of each sorted pair), sorted_w[cap] (its combine
 * weight), tok_ptr[T+1] and tok_pairs[cap] (per token, the sorted positions
 * of its pairs in ascending expert), P_out (device int32 scalar).  cap must be
 * at least moe_pair_capacity(T,E,K,m_tile).
 *
 * Each grouping runs as one cooperative launch (all of its blocks resident at once, two grid barriers
 * bounded by moe_set_wait_timeout; a barrier that gives up records MOE_DEV_TIMEOUT); when the GPU cannot
 * hold all blocks at once it runs as four ordinary launches with the same results.
 */
int moe_permute(moe_ctx* ctx, const int32_t* topk_ids, const float* topk_w, const float* logits,
                const float* scores, int T, int E, int K, int m_tile, long long cap, int32_t* counts,
                int32_t* offsets, int32_t* sorted_tok, float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs,
                int32_t* P_out, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_permute_capacity — the capacity (drop/pad) dispatch variant of moe_permute.
 * [DEP] "Drop/Padding 방식": the pairs are laid out per expert as [E, C] slots;
 * each expert keeps at most C of its routed tokens and the rest are dropped,
 * an expert with fewer is padded to C.  policy 0 ("position") keeps the first
 * C routed tokens in token order, policy 1 ("probs") the C with the largest
 * routing probability topk_w (ties: lower token first).  Kept pairs keep their
 * top-K weight.  C is the caller's (moe_expert_capacity gives ceil(capacity_factor * T*K/E)).
 *
 * Outputs: counts[E] (kept pairs per expert), offsets[E+1] = e*C,
 * sorted_tok[cap] (token of every slot, -1 for an empty slot), sorted_w[cap]
 * (its weight, 0 for an empty slot), tok_ptr[T+1] and tok_pairs[cap] (per
 * token, the slots of its kept pairs in ascending expert), P_out = E*C.
 * cap >= E*C; T <= 32768; ws of at least moe_capacity_workspace_bytes(...).
 * The slots feed moe_grouped_gemm_fwd / moe_combine / moe_backward unchanged
 * (every slot is a GEMM row; an empty slot is a zero row with weight 0).
 */
int moe_permute_capacity(moe_ctx* ctx, const int32_t* topk_ids, const float* topk_w, int T, int E, int K, int C,
                         int policy, long long cap, int32_t* counts, int32_t* offsets, int32_t* sorted_tok,
                         float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs, int32_t* P_out, void* ws,
                         size_t ws_bytes, moe_stream_t stream);

/* Workspace of the whole path under the capacity dispatch (pair capacity E*C). */
size_t moe_capacity_workspace_bytes(int T, int d, int E, int n, int K, int C);

/*
 * moe_permute_noalloc — moe_permute without a workspace, for callers that cannot
 * allocate device memory at all (a caller that only receives buffers from a host
 * runtime that offers no allocator, or a loop that must not allocate once it
 * runs).  The pages describe no such entry point; it is an addition of this
 * library.
 *
 * Same grouping and outputs as moe_permute with m_tile = 0 (plain top-K), but its
 * scratch lives in a fixed device array inside the library (257 KiB, held by every
 * GPU that loads the library until the process exits), so it supports at most
 * T <= 32768 tokens and E <= 512 experts and returns MOE_ERR_UNSUPPORTED beyond
 * that.  No cudaMalloc, cudaFree or other allocating call is made.
 * The first call on a device looks up that array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any stream
 * capture.  All calls share the one array: calls that overlap on the GPU (two
 * streams, or two contexts on one device) race and must be serialized by the
 * caller.  The array needs no clearing: every call rewrites what it reads.
 * The cached address belongs to the device's primary context: a process that
 * resets a device (cudaDeviceReset) must not call this entry point on that
 * device afterwards.
 */
int moe_permute_noalloc(moe_ctx* ctx, const int32_t* topk_ids, const float* topk_w, int T, int E, int K,
                        long long cap, int32_t* counts, int32_t* offsets, int32_t* sorted_tok, float* sorted_w,
                        int32_t* tok_ptr, int32_t* tok_pairs, int32_t* P_out, moe_stream_t stream);

/*
 * moe_grouped_gemm_fwd — the expert MLP of every pair, as varlen-M grouped GEMMs.
 * [GG] "(6) 세 번의 gg.gmm" and "Variable-M batched matmul"; [SM] "MoE 연산 =
 * Grouped GEMM", "4.1 Gather 융합" (token rows gathered inside the operand
 * load, the permuted X never written), "4.2 Epilogue 융합" (SwiGLU in the
 * epilogue).  For sorted pair j of expert e with token t = sorted_tok[j]:
 *
 *   H[j] = X[t] W_gate[e]^T,  U[j] = X[t] W_up[e]^T,  A[j] = silu(H[j]) * U[j]
 *   Yw[j] = sorted_w[j] * (A[j] W_down[e]^T)
 *
 * H and U are kept in fp32 (the backward's dSwiGLU reads them; both may be NULL for a
 * forward-only call, which then writes neither); A is computed from the fp32
 * accumulators and stored rounded to bf16.  The down projection takes A as that
 * bf16 value plus the bf16 rounding of the rest (about 16 significant bits, two
 * UMMAs per K step); the low part lives in the workspace `ws` between the two
 * GEMMs (at least 2*cap*n bytes, 256-byte aligned; moe_workspace_bytes covers it).
 * Outputs H, U [cap,n] fp32, A [cap,n] bf16, Yw [cap,d] bf16.
 */
int moe_grouped_gemm_fwd(moe_ctx* ctx, const void* X, const void* W_gate, const void* W_up, const void* W_down,
                         int T, int d, int E, int n, long long cap, const int32_t* offsets,
                         const int32_t* sorted_tok, const float* sorted_w, void* H, void* U, void* A, void* Yw,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_quantize_rows_e4m3 — per-row e4m3 quantization for the FP8 gate/up GEMM.
 * [GG] "한계" (a fine-grained FP8 grouped GEMM as the next 2x over bf16; the page
 * gives no recipe, the per-row one here is this library's reading).
 *
 * M [rows, cols] bf16 (device), row-major.  For every row r:
 *   scales[r] = max_i |M[r,i]| / 448 in fp32 (1 when the row is all zeros),
 *   q[r,i]    = e4m3(M[r,i] / scales[r]), the division in fp32, rounded to
 *               nearest even and saturated at +-448 (e4m3: 4 exponent bits,
 *               bias 7, 3 mantissa bits; q holds the bit patterns, one byte each).
 * Outputs q [rows, cols] uint8 and scales [rows] fp32 (device, caller-owned).
 * Use it on X (one scale per token) and on the rows of W_gate / W_up viewed as
 * [E*n, d] (one scale per output channel).  cols % 16 == 0; M and q 16-byte
 * aligned; else MOE_ERR_INVALID_ARG.
 */
int moe_quantize_rows_e4m3(moe_ctx* ctx, const void* M, long long rows, int cols, void* q, float* scales,
                           moe_stream_t stream);

/*
 * moe_grouped_gemm_fwd_e4m3 — moe_grouped_gemm_fwd with e4m3 gate/up operands and,
 * optionally, an e4m3 down projection.
 * [GG] "한계" and "(6) 세 번의 gg.gmm"; [SM] "4.1 Gather 융합", "4.2 Epilogue 융합".
 * Xq [T,d] and x_scale [T]: moe_quantize_rows_e4m3 of X; Wg_q, Wu_q [E,n,d] and
 * wg_scale, wu_scale [E,n]: moe_quantize_rows_e4m3 of W_gate, W_up as [E*n, d].
 * For sorted pair j of expert e with token t = sorted_tok[j] and column c:
 *
 *   H[j,c] = x_scale[t] * wg_scale[e,c] * sum_i e4m3(Xq[t,i]) e4m3(Wg_q[e,c,i])
 *   U[j,c] likewise with Wu_q, wu_scale;  A[j] = silu(H[j]) * U[j] (bf16)
 *
 * Down projection, bf16 (Wd_q == NULL): Yw[j] = sorted_w[j] * (A[j] W_down[e]^T) as in
 * moe_grouped_gemm_fwd.  e4m3 (Wd_q != NULL; W_down may be NULL): Wd_q [E,d,n] and wd_scale
 * [E,d] are moe_quantize_rows_e4m3 of W_down as [E*d, n]; the rows of A below offsets[E] are
 * quantized the same way into Aq [cap,n] (uint8 codes) and a_scale [cap] (caller-owned device
 * buffers), and
 *
 *   Yw[j,c] = sorted_w[j] * a_scale[j] * wd_scale[e,c] * sum_i e4m3(Aq[j,i]) e4m3(Wd_q[e,c,i])
 *
 * Code products are accumulated in fp32 on the tensor cores (kind::f8f6f4).  A slot with
 * sorted_tok = -1 (capacity dispatch) gives zero rows.  Shape rules as moe_grouped_gemm_fwd (d and n
 * multiples of 64: a last stage of 128 codes may be half past K and reads zeros there); outputs H, U (both may be
 * NULL: forward only), A, Yw and ownership as moe_grouped_gemm_fwd; no workspace.
 * MOE_ERR_INVALID_ARG on a violated rule.
 */
int moe_grouped_gemm_fwd_e4m3(moe_ctx* ctx, const void* Xq, const float* x_scale, const void* Wg_q,
                              const float* wg_scale, const void* Wu_q, const float* wu_scale, const void* W_down,
                              const void* Wd_q, const float* wd_scale, int T, int d, int E, int n, long long cap,
                              const int32_t* offsets, const int32_t* sorted_tok, const float* sorted_w, void* H,
                              void* U, void* A, void* Aq, float* a_scale, void* Yw, moe_stream_t stream);

/*
 * Block-scaled e4m3 form ("fine-grained" FP8): [GG] "한계" credits a fine-grained FP8 grouped GEMM with
 * a further 2x over bf16; the pages give no recipe, this library's reading is the following.  Every
 * operand row is cut into blocks of 32 consecutive elements along the reduction dimension; a block has
 * one power-of-two scale 2^e, stored as the byte e + 127, with e the smallest integer in [-127, 127]
 * such that max|block| <= 448 2^e (0 for an all-zero block), and codes e4m3(x 2^-e) rounded to nearest
 * even (exact scaling, no saturation).  The GEMMs run on the kind::mxf8f6f4 tensor-core instruction,
 * which multiplies every 32-element block's code products by both operands' block scales.
 *
 * Scale layouts (bytes, device):
 *   row-major  [rows][moe_mx_sf_cols(cols)]: the scales of row r's blocks in order, then bytes of value
 *              127 up to a multiple of 4 per 128 columns;
 *   blocks     512 bytes per 128 operand rows and 128 columns of the reduction: row r, block k of the
 *              128 columns at byte (r % 32) * 16 + (r / 32) * 4 + k; rows or columns beyond the operand
 *              hold 127.  The weights' blocks come per tile of a GEMM's B rows (ceil(rows / 128) blocks)
 *              and 128 columns: W_gate / W_up [E][ceil(n/96)][ceil(d/128)] pairs of blocks, tile rows
 *              0..95 of [e][t][.] = W_gate[e] rows 96t..96t+95, tile rows 96..191 = W_up[e] rows
 *              96t..96t+95 (tile row i in block i / 128, block row i % 128); W_down [E][ceil(d/Bd)]
 *              [ceil(n/128)] over W_down[e] rows Bd t.. with Bd = w(d); the activations A: one block per
 *              128-row tile of every expert's sorted rows (tiles in expert order) and 128 columns,
 *              [tiles][ceil(n/128)].  The width w(N) of the plain GEMMs' tiles (down projection, dSwiGLU,
 *              dX) is 192, or 128 when 192-row tiles would pass N by more than N / 4 and 128-row tiles by
 *              less (w(256) = 128; w(512) = w(2048) = 192).
 */
/* Bytes per row of a row-major scale array for `cols` columns: 4 * ceil(cols / 128). */
long long moe_mx_sf_cols(int cols);
/* Bytes of the weight scale blocks: which = 0 the W_gate / W_up pair, 1 W_down (the forward); 2 W_down^T,
 * 3 [W_gate; W_up]^T (the backward's dSwiGLU and dX GEMMs, moe_quantize_bwd_weights_mx); 0 on bad arguments. */
long long moe_mx_weight_sf_bytes(int E, int d, int n, int which);
/* Bytes of the activation scale blocks for a pair capacity cap: (ceil(cap/128) + E) * ceil(n/128) * 512. */
long long moe_mx_act_sf_bytes(long long cap, int E, int n);

/*
 * moe_quantize_rows_mx — block-scaled quantization of M [rows, cols] bf16 (row-major, device) along its
 * rows: codes q [rows, cols] uint8 and row-major scales sf [rows][moe_mx_sf_cols(cols)] (caller-owned
 * device buffers).  Use it on X (blocks along d).  cols % 64 == 0; M and q 16-byte aligned; else
 * MOE_ERR_INVALID_ARG.
 */
int moe_quantize_rows_mx(moe_ctx* ctx, const void* M, long long rows, int cols, void* q, void* sf,
                         moe_stream_t stream);

/*
 * moe_quantize_weights_mx — block-scaled codes and scale blocks of the expert weights, once per weight
 * update: W_gate, W_up [E,n,d] and W_down [E,d,n] bf16 (device) to codes Wg_q, Wu_q [E,n,d], Wd_q
 * [E,d,n] uint8 (blocks along each row, i.e. along d for W_gate / W_up and along n for W_down) and the
 * scale blocks gu_sf (moe_mx_weight_sf_bytes(E,d,n,0) bytes) and dn_sf (moe_mx_weight_sf_bytes(E,d,n,1)).
 * Caller-owned device buffers, 16-byte aligned; d, n multiples of 64; else MOE_ERR_INVALID_ARG.
 */
int moe_quantize_weights_mx(moe_ctx* ctx, const void* W_gate, const void* W_up, const void* W_down, int E, int d,
                            int n, void* Wg_q, void* Wu_q, void* gu_sf, void* Wd_q, void* dn_sf,
                            moe_stream_t stream);

/*
 * moe_grouped_gemm_fwd_mx — moe_grouped_gemm_fwd on block-scaled e4m3 operands, the activations quantized
 * inside the gate/up GEMM's epilogue.  [GG] "한계" and "(6) 세 번의 gg.gmm"; [SM] "4.1 Gather 융합",
 * "4.2 Epilogue 융합".  Xq [T,d], x_sf: moe_quantize_rows_mx of X; Wg_q, Wu_q, gu_sf, Wd_q, dn_sf:
 * moe_quantize_weights_mx.  For sorted pair j of expert e, token t = sorted_tok[j], column c, with
 * dq(.) the block-scaled value (code times its block's scale):
 *
 *   H[j,c] = sum_i dq(Xq[t,i]) dq(Wg_q[e,c,i]),  U[j,c] likewise with Wu_q,
 *   A[j]   = silu(H[j]) U[j], quantized per 32-column block in fp32 into Aq [cap,n] uint8 and the
 *            activation scale blocks a_sf (moe_mx_act_sf_bytes(cap,E,n) bytes),
 *   Yw[j,c] = sorted_w[j] * sum_i dq(Aq[j,i]) dq(Wd_q[e,c,i])  (bf16).
 *
 * x_sf_tiles (moe_mx_act_sf_bytes(cap,E,d) bytes, caller-owned scratch, overwritten) receives the gathered
 * rows' scales laid out per sorted row tile, the form the gate/up GEMM loads them in.
 * Block products are accumulated in fp32 on the tensor cores.  A slot with sorted_tok = -1 (capacity
 * dispatch) gives zero rows.  H, U [cap,n] fp32 are the backward's cache (both NULL: forward only).  Rows of
 * Aq at or past offsets[E], and scale bytes of rows past an expert's last row, are not written.  Shape rules
 * as moe_grouped_gemm_fwd; every buffer caller-owned device memory, codes and scale blocks 16-byte
 * aligned; no workspace.  MOE_ERR_INVALID_ARG on a violated rule.
 */
int moe_grouped_gemm_fwd_mx(moe_ctx* ctx, const void* Xq, const void* x_sf, const void* Wg_q, const void* Wu_q,
                            const void* gu_sf, const void* Wd_q, const void* dn_sf, int T, int d, int E, int n,
                            long long cap, const int32_t* offsets, const int32_t* sorted_tok, const float* sorted_w,
                            void* H, void* U, void* x_sf_tiles, void* Aq, void* a_sf, void* Yw, moe_stream_t stream);

/*
 * moe_quantize_bwd_weights_mx — the block-scaled B operands of the backward's activation-gradient GEMMs, once per
 * weight update: W_down^T (per expert [n, d], blocks along d) into codes Wdt_q [E,n,d] and scale blocks wdt_sf
 * (moe_mx_weight_sf_bytes(E,d,n,2) bytes, [E][ceil(n/w(n))][ceil(d/128)] tiles of blocks over W_down^T's rows);
 * [W_gate; W_up]^T (per expert [d, 2n], W_gate's rows in columns 0..n-1, W_up's in n..2n-1, blocks along 2n)
 * into Wgu_q [E,d,2n] and wgu_sf (moe_mx_weight_sf_bytes(E,d,n,3) bytes, [E][ceil(d/w(d))][ceil(2n/128)] tiles);
 * w(N) the tile width stated with the scale layouts above.
 * tmp: device scratch of E*d*2n bf16 (caller-owned, overwritten).  [SM] "3 기여 ①" (dA' = dO W_down),
 * "4 기여 ②" (the dX GEMM); [GG] "한계".  16-byte aligned buffers, d and n multiples of 64, else
 * MOE_ERR_INVALID_ARG.
 */
int moe_quantize_bwd_weights_mx(moe_ctx* ctx, const void* W_gate, const void* W_up, const void* W_down, int E, int d,
                                int n, void* tmp, void* Wdt_q, void* wdt_sf, void* Wgu_q, void* wgu_sf,
                                moe_stream_t stream);

/*
 * moe_backward_mx — moe_backward with the dSwiGLU GEMM and the dX GEMM on block-scaled e4m3 operands, each
 * activation quantized where it is produced.  dO is quantized per token in 1 x 32 blocks (inside the call, in
 * the workspace), its code rows are copied to the sorted positions dOq [cap,d] (caller-owned) and their scales
 * laid out per sorted row tile into do_sf_tiles (moe_mx_act_sf_bytes(cap,E,d) bytes, caller-owned scratch);
 * with dq(.) the block-scaled value, for sorted pair j of expert e:
 *
 *   dA'[j,c] = sum_i dq(dOq[j,i]) dq(Wdt_q[e,c,i])      (the dSwiGLU epilogue as moe_backward on this dA')
 *   the epilogue also writes [dH | dU][j] quantized from its fp32 values into HUq [cap,2n] and the scale
 *   blocks hu_sf (moe_mx_act_sf_bytes(cap,E,2n) bytes), both caller-owned;
 *   dXp[j,c]  = sum_k dq(HUq[j,k]) dq(Wgu_q[e,c,k])
 *
 * Wdt_q, wdt_sf, Wgu_q, wgu_sf from moe_quantize_bwd_weights_mx.  The router gradient and dX's reduction are
 * those of moe_backward.  With dw_ws == NULL the weight gradients are moe_backward's GEMMs with dH, dU and
 * A' = w A each rounded once to bf16 from the fp32 value (no low part; the dSwiGLU epilogue then writes none).
 * With dw_ws (caller-owned device scratch of at least moe_mx_dw_ws_bytes(d,E,n,cap) bytes, 256-byte aligned,
 * overwritten) they run on block-scaled operands with the blocks along tokens: for expert e, with its sorted
 * pairs j = offsets[e] + i split into blocks of 32 consecutive i (the last one partial), every operand column
 * quantized per block by the rule above (dH, dU, A' from their fp32 values, X and dO from bf16, both read at
 * the pairs' tokens):
 *
 *   dW_gate[e][r,c] = sum_i dq(dH[j,r]) dq(X[tok_j,c])     dW_up likewise with dU
 *   dW_down[e][c,r] = sum_i dq(dO[tok_j,c]) dq(A'[j,r])
 *
 * accumulated in fp32 on the tensor cores; the expert-sorted bf16 copies of X and dO are then not made.
 * [GG] "한계" (the fine-grained FP8 grouped GEMM); [SM] "4 기여 ②" (varlen-K weight gradients).  Arguments, shape rules, workspace and ownership otherwise as
 * moe_backward; MOE_ERR_UNSUPPORTED when the pair capacity is too small to stage dO's per-token codes in the
 * workspace (cap * 2d bytes must hold T * (d + 4 ceil(d/128)) plus alignment).
 */
int moe_backward_mx(moe_ctx* ctx, const void* dO, const void* X, const void* W_r, const void* W_gate, const void* W_up,
                    const void* W_down, const void* Wdt_q, const void* wdt_sf, const void* Wgu_q, const void* wgu_sf,
                    int T, int d, int E, int n, int K, int m_tile, long long cap, const int32_t* topk_ids,
                    const float* topk_w, const int32_t* offsets, const int32_t* sorted_tok, const float* sorted_w,
                    const int32_t* tok_ptr, const int32_t* tok_pairs, const void* H, const void* U, void* dOq,
                    void* do_sf_tiles, void* HUq, void* hu_sf, void* dX, void* dW_gate, void* dW_up, void* dW_down,
                    int dW_fp32, float* dS, float* dlogits, float* dW_r, void* ws, size_t ws_bytes, void* dw_ws,
                    size_t dw_ws_bytes, moe_stream_t stream);

/*
 * moe_mx_dw_ws_bytes — bytes of the workspace that moe_backward_mx takes (dw_ws) to run the weight gradients on
 * block-scaled e4m3 operands, for a layer of hidden size d, E experts, intermediate size n and pair capacity cap
 * (0 for an invalid shape: d, n multiples of 64, 1 <= E <= 1024, cap >= 1).  It holds the four operands as
 * K-major codes over a reduction padded per expert to whole 128-token stages ((3n + 2d) x (cap + 127 E) bytes
 * at most, rounded up to 128 tokens), their scale blocks and the stage offsets.
 */
size_t moe_mx_dw_ws_bytes(int d, int E, int n, long long cap);

/*
 * moe_combine — weighted sum of every token's expert outputs, in original token order.
 * [EP] "여러 Expert의 결과도 같은 토큰으로 돌아오기" (y(A2) = 0.7 u0 + 0.3 u2 in
 * A2's own slot); [DEP] "3) Combine".  O[t] = sum over t's pairs, in ascending
 * expert, of Yw[j] (weights already applied); fp32 accumulation in a fixed
 * order (no atomics, deterministic); O[T,d] bf16.  A token without pairs gets 0.
 */
int moe_combine(moe_ctx* ctx, const void* Yw, const int32_t* tok_ptr, const int32_t* tok_pairs, int T, int d,
                long long cap, void* O, moe_stream_t stream);

/*
 * moe_backward — gradients of the layer for an upstream gradient dO[T,d].
 * [SM] "3 기여 ① 메모리 효율 알고리즘" (dS from <dA', A> instead of <dO, Y>),
 * "4.2 Epilogue 융합" (dH, dS, A' in one epilogue, dSwiGLU fused), "4 기여 ②"
 * (varlen-K grouped GEMM for dW).  Unlike [SM] "4.1 Gather 융합", the backward
 * writes expert-sorted copies of X and dO into the workspace once (every
 * backward GEMM then reads whole TMA boxes); the weight-gradient GEMMs take
 * dH, dU and A' as a bf16 high part plus the bf16 rounding of the rest (about
 * 16 significant bits of the epilogue's fp32 values), also in the workspace.
 * With dA'[j] = dO[t] W_down[e] and w = sorted_w[j]:
 *   dS[j] = <dA'[j], A[j]>           (= <dO[t], Y[j]>, the gradient of w)
 *   dA = w dA',  dU = dA * silu(H),  dH = dA * U * s(H) (1 + H (1 - s(H)))
 *   dX[t] = sum_j (dH[j] W_gate[e] + dU[j] W_up[e]) + dlogits[t] W_r^T
 *   dW_gate[e] = sum_j dH[j]^T X[t], dW_up[e] = sum_j dU[j]^T X[t],
 *   dW_down[e] = sum_j (w dO[t])^T A[j]    (zero for an expert without pairs)
 *   dlogits[t,k] = [k in F(t)] w_k dS_k - [k in TopK(t)] w_k sum_{i in F(t)} w_i dS_i
 *   dW_r = X^T dlogits
 * (F(t) = the token's final pairs; TopK(t) = its top-K; the bias is not trained.)
 *
 * Inputs: dO, X, W_r, W_gate, W_up, W_down, the routing state of moe_route and
 * moe_permute, and H, U (fp32) from moe_grouped_gemm_fwd.  Outputs: dX[T,d] bf16,
 * dW_gate/dW_up[E,n,d] and dW_down[E,d,n] (bf16, or fp32 when dW_fp32 != 0),
 * dS[cap] fp32, dlogits[T,E] fp32, dW_r[d,E] fp32.
 */
int moe_backward(moe_ctx* ctx, const void* dO, const void* X, const void* W_r, const void* W_gate,
                 const void* W_up, const void* W_down, int T, int d, int E, int n, int K, int m_tile, long long cap,
                 const int32_t* topk_ids, const float* topk_w, const int32_t* offsets, const int32_t* sorted_tok,
                 const float* sorted_w, const int32_t* tok_ptr, const int32_t* tok_pairs, const void* H,
                 const void* U, void* dX, void* dW_gate, void* dW_up, void* dW_down, int dW_fp32, float* dS,
                 float* dlogits, float* dW_r, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_quantize_dx_weights_e4m3 — the B operand of the e4m3 dX GEMM: for every expert e the matrix
 * [W_gate[e]; W_up[e]]^T (d rows of 2n: row c holds W_gate[e][:, c] then W_up[e][:, c]) quantized
 * per row as moe_quantize_rows_e4m3 does.  [GG] "한계"; [SM] "4 기여 ②" (the dX GEMM).
 * W_gate, W_up [E,n,d] bf16; tmp [E,d,2n] bf16 device scratch (caller-owned, overwritten);
 * outputs Wgu_q [E,d,2n] uint8 codes and wgu_scale [E,d] fp32.  Shape rules as moe_backward;
 * 16-byte aligned pointers; else MOE_ERR_INVALID_ARG.
 */
int moe_quantize_dx_weights_e4m3(moe_ctx* ctx, const void* W_gate, const void* W_up, int E, int n, int d, void* tmp,
                                 void* Wgu_q, float* wgu_scale, moe_stream_t stream);

/*
 * moe_quantize_dact_weights_e4m3 — the B operand of the e4m3 dSwiGLU GEMM: W_down[e]^T (n rows of d)
 * quantized per row as moe_quantize_rows_e4m3 does.  [SM] "3 기여 ①" (dA' = dO W_down).
 * W_down [E,d,n] bf16; tmp [E,n,d] bf16 device scratch (caller-owned, overwritten); outputs
 * Wdt_q [E,n,d] uint8 codes and wdt_scale [E,n] fp32.  Shape rules as moe_backward; 16-byte
 * aligned pointers; else MOE_ERR_INVALID_ARG.
 */
int moe_quantize_dact_weights_e4m3(moe_ctx* ctx, const void* W_down, int E, int n, int d, void* tmp, void* Wdt_q,
                                   float* wdt_scale, moe_stream_t stream);

/*
 * moe_backward_e4m3 — moe_backward with the dX GEMM and/or the dSwiGLU GEMM on e4m3 operands.
 * [GG] "한계" (the FP8 grouped GEMM); [SM] "3 기여 ①", "4 기여 ②".  Arguments as moe_backward, plus:
 *   Wgu_q / wgu_scale (moe_quantize_dx_weights_e4m3; NULL: bf16 dX GEMM) with the caller-owned
 *   buffers HUq [cap, 2n] uint8 and hu_scale [cap] fp32: the rows [dH[j] | dU[j]] below offsets[E]
 *   are quantized per row into them (one scale over both halves), and
 *     dXp[j,c] = hu_scale[j] * wgu_scale[e,c] * sum_k e4m3(HUq[j,k]) e4m3(Wgu_q[e,c,k]);
 *   Wdt_q / wdt_scale (moe_quantize_dact_weights_e4m3; NULL: bf16 dSwiGLU GEMM) with dOq [cap, d]
 *   uint8 and do_scale [cap] fp32: they receive the per-row quantization of the expert-sorted dO rows
 *   (dO is quantized once per token when the workspace's dX-partials region holds T*d + 4T bytes, i.e.
 *   whenever cap >= T, and the codes gathered with dO; else the sorted rows below offsets[E] are
 *   quantized; the codes are the same either way), and
 *     dA'[j,c] = do_scale[j] * wdt_scale[e,c] * sum_i e4m3(dOq[j,i]) e4m3(Wdt_q[e,c,i]),
 *   the dSwiGLU epilogue (dS = <dA', A>, dH, dU, A') running on that dA'.
 * Code products accumulate in fp32 (kind::f8f6f4); everything else as moe_backward, except that the
 * weight-gradient GEMMs take dH, dU and A' = w A each rounded once to bf16 from the fp32 value (no low
 * part: the e4m3 GEMMs already carry e4m3 rounding).  MOE_ERR_INVALID_ARG on a missing or misaligned buffer.
 */
int moe_backward_e4m3(moe_ctx* ctx, const void* dO, const void* X, const void* W_r, const void* W_gate,
                      const void* W_up, const void* W_down, const void* Wgu_q, const float* wgu_scale,
                      const void* Wdt_q, const float* wdt_scale, int T, int d, int E, int n, int K, int m_tile,
                      long long cap, const int32_t* topk_ids, const float* topk_w, const int32_t* offsets,
                      const int32_t* sorted_tok, const float* sorted_w, const int32_t* tok_ptr,
                      const int32_t* tok_pairs, const void* H, const void* U, void* HUq, float* hu_scale, void* dOq,
                      float* do_scale, void* dX, void* dW_gate, void* dW_up, void* dW_down, int dW_fp32, float* dS,
                      float* dlogits, float* dW_r, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Per-kernel timing (tracing).  With profiling enabled, every kernel the
 * library launches is bracketed by a CUDA event pair on its stream (events
 * come from a pool created by the first moe_profile_enable).  moe_profile_read
 * waits for the recorded events, returns per kernel label its accumulated
 * milliseconds and launch count since the last read (names: max_kernels x 32
 * chars, NUL-terminated), resets the totals and sets *n_kernels to the number
 * of labels seen.  A context is not thread-safe while profiling.
 */
int moe_profile_enable(moe_ctx* ctx, int enable);
int moe_profile_read(moe_ctx* ctx, int max_kernels, char* names, double* total_ms, long long* launches,
                     int* n_kernels);

/*
 * Test exports: the grouped-GEMM main loops on raw operands, fp32 results.
 * They exist so that integer-valued operands (exact in fp32 whatever the
 * summation order) can check the gather, the varlen bookkeeping and the
 * operand layouts bit for bit.
 *
 * moe_test_gemm_varlen_m: for each group e and sorted row j of it,
 *   D[j, c] = sum_k A[row(j), k] * B[e, c, k]      (B_kmajor = 1: B is [G, N, K])
 *   D[j, c] = sum_k A[row(j), k] * B[e, k, c]      (B_kmajor = 0: B is [G, K, N])
 * with row(j) = idx[j] (gathered, idx != NULL) or j.  A[rows_a, K] bf16,
 * D[cap, N] fp32; offsets[G+1].  With B_kmajor = 0, N must be a multiple of 64.  A gathered row index outside the source
 * records MOE_DEV_BAD_OFFSETS and reads zeros instead.  Tiles of 128 x 128; without idx and with
 * moe_set_cta_pairs(ctx, 1, .) CTA pairs on 256 x 256 tiles.
 *
 * moe_test_gemm_varlen_k: for each group e,
 *   D[e, m, c] = sum_{j in group e} A[rowa(j), m] * B[rowb(j), c]
 * with rowa(j) = idx_a ? idx_a[j] : j (same for b).  A[rows_a, M], B[rows_b, N] bf16,
 * D[G, M, N] fp32 (zeros for an empty group).  At most one of idx_a, idx_b is
 * non-NULL: a gathered operand is zero past a group's end; with both NULL the
 * rows of B past the group's end are cleared in shared memory (the weight-
 * gradient path).  M and N are multiples of 64.
 */
int moe_test_gemm_varlen_m(moe_ctx* ctx, const void* A, const int32_t* idx, const void* B, int B_kmajor,
                           int G, int rows_a, int K, int N, long long cap, const int32_t* offsets, float* D,
                           moe_stream_t stream);
int moe_test_gemm_varlen_k(moe_ctx* ctx, const void* A, const int32_t* idx_a, int rows_a, const void* B,
                           const int32_t* idx_b, int rows_b, int G, int M, int N, long long cap,
                           const int32_t* offsets, float* D, moe_stream_t stream);

/*
 * moe_test_gemm_varlen_m_dual: the down projection's main loop with a two-part A, for each group e and
 * sorted row j of it,
 *   D[j, c] = sum_k (A_hi[j, k] + A_lo[j, k]) * B[e, c, k]       (B is [G, N, K], K-major)
 * (two UMMAs per K step into one fp32 accumulator).  A_hi, A_lo [rows_a, K] bf16 with rows_a >= cap,
 * D[cap, N] fp32; rows outside every group are left untouched.  K a multiple of 64, N of 8.  Tiles of
 * 128 x 256 (CTA pairs on 256 x 256 with moe_set_cta_pairs(ctx, 1, .)).
 */
int moe_test_gemm_varlen_m_dual(moe_ctx* ctx, const void* A_hi, const void* A_lo, const void* B, int G, int rows_a,
                                int K, int N, long long cap, const int32_t* offsets, float* D, moe_stream_t stream);

/*
 * moe_test_gemm_varlen_k_dual: the weight-gradient form with a two-part A, for each group e,
 *   S[e, m, c] = sum_{i < M_e} (A_hi[off[e] + i, m] + A_lo[off[e] + i, m]) * B[boff[e] + i, c]
 * (two UMMAs per K step into one fp32 accumulator), M_e = off[e+1] - off[e].  A_hi, A_lo [rows_a, M],
 * B [rows_b, N] bf16.  b_offsets = NULL: boff = off, and the rows of B past a group's end are cleared in
 * shared memory; else boff = b_offsets[G+1], the padded layout of the backward's sorted copies (each group's
 * rows followed by zero rows up to the next multiple of 16, which the caller provides).  trans = 0: D[G, M, N] = S;
 * trans = 1: D[G, N, M] with D[e, c, m] = S[e, m, c] (the transposed store of dW_down).  fp32
 * out, zeros for an empty group; M and N multiples of 64.  The kernel configuration is the backward's for
 * the same N (CTA pairs with b_offsets, N > 128 and moe_set_cta_pairs(ctx, ., 1)).
 */
int moe_test_gemm_varlen_k_dual(moe_ctx* ctx, const void* A_hi, const void* A_lo, int rows_a, const void* B, int rows_b,
                                int G, int M, int N, long long cap, const int32_t* offsets, const int32_t* b_offsets,
                                int trans, float* D, moe_stream_t stream);

/* Test export: launch one CTA that waits on an mbarrier nobody arrives on, with
 * the given bound; the wait gives up, records MOE_DEV_TIMEOUT and returns. */
int moe_test_wait_timeout(moe_ctx* ctx, unsigned long long timeout_ns, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VGG_MOE_H */

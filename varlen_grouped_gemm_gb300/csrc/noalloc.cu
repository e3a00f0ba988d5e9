// moe_permute_noalloc: the expert grouping of moe_permute (plain top-K, no token rounding) for
// callers that cannot allocate device memory, not even the small workspace moe_permute takes.
// Examples: code that only receives buffers handed to it by a host runtime with no allocator
// interface, or a loop that must not call into an allocator once it is running.
//
// The grouping's scratch (per-expert, per-token-block counts and their scan, plus the per-block
// pair bases; perm_tok_block keeps them within the array for T <= 32768, E <= 512) lives in a
// file-scope device array of fixed size, which every GPU that loads this library keeps until the
// process exits.  Host code cannot pass that array's name to
// a kernel (in host code it names a host-side stand-in, not device memory), so the first call on
// each device looks up the array's device address with cudaGetSymbolAddress and caches it.
#include <mutex>

#include "internal.h"
#include "moe.h"

namespace vgg {
namespace {

constexpr int kNoAllocMaxT = 32768;                // tokens
constexpr int kNoAllocMaxE = 512;                  // experts
constexpr int kNoAllocBlocks = kNoAllocMaxT / 256;  // the array holds (E + 1) x 128 + 2 counts
// hist + block bases + their total + the one-launch grouping's barrier counter
constexpr int kNoAllocScratchInts = kNoAllocMaxE * kNoAllocBlocks + kNoAllocBlocks + 2;

// 65,666 ints = 257 KiB; contents are fully rewritten (the barrier counter zeroed) by every call before they
// are read.
__device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
int32_t* g_scratch_dev[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once per device).  The address
// belongs to the device's primary context, so it stays valid unless the process resets the device.
int32_t* scratch_for(int device) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_dev[device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_permute_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    g_scratch_dev[device] = static_cast<int32_t*>(ptr);
  }
  return g_scratch_dev[device];
}

}  // namespace
}  // namespace vgg

extern "C" int moe_permute_noalloc(moe_ctx* ctx, const int32_t* topk_ids, const float* topk_w, int T, int E, int K,
                                   long long cap, int32_t* counts, int32_t* offsets, int32_t* sorted_tok,
                                   float* sorted_w, int32_t* tok_ptr, int32_t* tok_pairs, int32_t* P_out,
                                   moe_stream_t stream) {
  using namespace vgg;
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (T > kNoAllocMaxT || E > kNoAllocMaxE) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch
  const int device = ctx_device(ctx);
  if (device < 0 || device >= kMaxDevices) return MOE_ERR_INVALID_ARG;
  // the array's address is looked up with the context's device current
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return MOE_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* scratch = scratch_for(device);
  if (prev != device) cudaSetDevice(prev);
  if (!scratch) return MOE_ERR_CUDA;
  // the checks and the launch of moe_permute's plain grouping, on the fixed array
  return permute_plain_with_scratch(ctx, topk_ids, topk_w, T, E, K, cap, counts, offsets, sorted_tok, sorted_w,
                                    tok_ptr, tok_pairs, P_out, scratch, kNoAllocScratchInts,
                                    static_cast<cudaStream_t>(stream));
}

// dflash2_head_topk_noalloc: the head GEMM + fused top-K + hidden_projection with its scratch
// in a fixed device array owned by this library, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all, or not at the moment they need the head: a
// real-time serving loop where an allocation would stall every other stream of the device, a host
// runtime whose allocator is not CUDA-aware, or plug-in hosts that hand over only the input and
// output buffers. dflash2_head_topk needs a caller workspace
// for the per-column-range top-K lists; this variant keeps those lists in `g_head_scratch`, a
// file-scope device array of kNoallocScratchBytes (8 MiB) instead.
//
// Properties a caller must know:
//  * The array exists once per device that loads the library and stays allocated until the
//    process exits.
//  * Every call on a device shares it. A call overwrites the part it uses, and the array keeps the
//    last call's contents afterwards. Calls that may overlap on the GPU (different streams, or
//    different host threads without ordering) race on the array and corrupt each other's results;
//    serialise them on one stream.
//  * Nothing in the array must start at zero: every list entry the merge step reads is written
//    earlier in the same call, so the array is never cleared.
//  * The first call on a device looks up the array's device address (cudaGetSymbolAddress with
//    that device current) and caches it; make that first call before any stream capture. The
//    cache is keyed by device index, so the address belongs to the device's primary context (the
//    CUDA runtime's) and is valid until cudaDeviceReset; after a reset, or in another driver-API
//    context, this entry point must not be called.
//  * Sizes whose lists need more than 8 MiB are rejected with DFLASH2_ERR_INVALID_ARG (e.g. up to
//    about 65,000 rows on a 152-SM GB300; 960 rows need about 4.7 MB).
//  * No cudaMalloc, cudaFree or allocating library routine is called.
#include <mutex>

#include "internal.h"

namespace dfl {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_head_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev];
std::mutex g_scratch_mu;

// Device address of g_head_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDev) return fail(DFLASH2_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_head_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(DFLASH2_ERR_CUDA, "cudaGetSymbolAddress(g_head_scratch) failed: %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DFLASH2_OK;
}

}  // namespace
}  // namespace dfl

using namespace dfl;

extern "C" int dflash2_head_topk_noalloc(const void* h, int M, int H, const void* w_head, int V, const float* bias,
                                         const void* w_proj, int R, int K, int dtype, int32_t* cand, float* unary,
                                         float* z, float* logits, void* stream) {
  if (dtype != DFLASH2_BF16 && dtype != DFLASH2_F32)
    return fail(DFLASH2_ERR_INVALID_ARG, "dtype=%d is not DFLASH2_BF16 or DFLASH2_F32", dtype);
  if (M < 1) return fail(DFLASH2_ERR_INVALID_ARG, "M=%d must be >= 1", M);
  if (H < 64 || H % 64 != 0) return fail(DFLASH2_ERR_INVALID_ARG, "H=%d must be a positive multiple of 64", H);
  if (K < 1 || K > 16 || K > V) return fail(DFLASH2_ERR_INVALID_ARG, "K=%d must be in [1, min(16, V)]", K);
  if (!h || !w_head || !cand || !unary) return fail(DFLASH2_ERR_INVALID_ARG, "a required pointer is NULL");
  if ((w_proj == nullptr) != (z == nullptr))
    return fail(DFLASH2_ERR_INVALID_ARG, "w_proj and z must be both set or both NULL");
  if (w_proj != nullptr && (R < 16 || R > 256 || R % 16 != 0))
    return fail(DFLASH2_ERR_INVALID_ARG, "R=%d must be a multiple of 16 in [16, 256]", R);
  if ((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(w_head) | reinterpret_cast<uintptr_t>(w_proj) |
       reinterpret_cast<uintptr_t>(bias)) & 15u)
    return fail(DFLASH2_ERR_INVALID_ARG, "h, w_head, w_proj and bias must be 16-byte aligned");
  const int r_eff = w_proj != nullptr ? R : 0;
  const int sms = sm_count();
  const size_t need = head_workspace(M, V, K, r_eff, sms);
  if (need > kNoallocScratchBytes)
    return fail(DFLASH2_ERR_INVALID_ARG,
                "M=%d needs %zu bytes of top-K scratch, more than the fixed %zu-byte array of the "
                "allocation-free entry point; use dflash2_head_topk with a caller workspace",
                M, need, kNoallocScratchBytes);
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != DFLASH2_OK) return rc;
  const GemmPlan plan = head_plan(M, H, V, r_eff, sms);
  const GemmProblem gp{h, w_head, w_proj, M, H, V, r_eff, dtype};
  return launch_head_topk(gp, plan, bias, K, cand, unary, z, logits, scratch, static_cast<cudaStream_t>(stream));
}

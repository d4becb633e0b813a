// moe_route_static: the router (fp32 logits + top-k + combine weights) for
// callers that cannot allocate device memory.
//
// The ordinary path keeps the router's partial sums in the workspace that
// moe_layer_create allocates.  Some callers cannot make that allocation: for
// example a serving runtime that reserves the whole device memory pool for
// its own allocator at start-up, or a step that must not call into
// cudaMalloc because it can synchronise the device or fail for lack of memory
// half-way through.  This entry point takes everything from the caller except
// that scratch, which lives in the fixed-size array below, loaded with the
// library (every GPU that loads it holds these 1 MiB until the process
// exits).  It runs the same kernels as moe_route does for up to 64 tokens
// (split-K partial sums, added in a fixed order by the top-k pass), so its
// results are the same bit for bit.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxExperts = 512;

// Split-K partial logits, [ks][T][E] fp32 with ks = router_ksplit(H) <= 8,
// T <= MOE_ROUTE_STATIC_MAX_TOKENS, E <= 512.
constexpr size_t kScratchFloats = (size_t)8 * MOE_ROUTE_STATIC_MAX_TOKENS * kMaxExperts;
static __device__ __align__(256) float g_route_scratch[kScratchFloats];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DeviceScratch {
  float* ptr = nullptr;
  unsigned long long ctx_id = 0;  // the context the address belongs to
};

std::mutex g_setup_mutex;
DeviceScratch g_scratch[kMaxDevices];

// Identifier of the current context (0 if the driver cannot tell), so that a
// context made after a device reset gets its own set-up.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
    cudaGetLastError();
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is asked of
// the runtime at set-up: once per device (and again if the device's context
// was replaced, e.g. after cudaDeviceReset), with that device current.
cudaError_t scratch_on_current_device(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  // make sure the device's context exists before asking which one it is
  e = cudaFree(nullptr);
  if (e != cudaSuccess) return e;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceScratch& d = g_scratch[dev];
  if (!d.ptr || d.ctx_id != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    d.ptr = static_cast<float*>(p);
    d.ctx_id = ctx;
  }
  *out = d.ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" moe_status moe_route_static(const void* x, int32_t T, int32_t H, int32_t E, int32_t k,
                                       const float* router_w, const float* router_b,
                                       int32_t* topk_idx, float* topk_w, void* stream) {
  if (T < 0 || H <= 0 || H % 128 != 0 || H > 16384 || E < 1 || E > kMaxExperts || k < 1 || k > 8 || k > E)
    return MOE_ERR_INVALID_ARG;
  if (T > MOE_ROUTE_STATIC_MAX_TOKENS) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if ((uintptr_t)x % 16 != 0 || (uintptr_t)router_w % 16 != 0) return MOE_ERR_INVALID_ARG;
  static_assert(MOE_ROUTE_STATIC_MAX_TOKENS <= moe::kRouterSplitMaxT,
                "the split-K router serves every token count the entry point accepts");
  float* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  // Every partial sum the top-k pass reads is written by the partial-sum pass
  // of the same call first, so nothing in the scratch has to start at zero.
  e = moe::launch_router_split(static_cast<const uint16_t*>(x), T, H, E, k, router_w, router_b,
                               moe::Scoring{0, 1.0f, nullptr}, scratch, nullptr, topk_idx, topk_w,
                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

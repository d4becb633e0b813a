// moe_route_static: the router (fp32 logits + top-k + combine weights) for
// callers that cannot allocate device memory.
//
// The ordinary path keeps the router logits in the workspace that
// moe_layer_create allocates.  Some callers cannot make that allocation: for
// example a serving runtime that reserves the whole device memory pool for
// its own allocator at start-up, or a step that must not call into
// cudaMalloc because it can synchronise the device or fail for lack of memory
// half-way through.  This entry point takes everything from the caller except
// the logits scratch, which lives in the fixed-size array below, loaded with
// the library (every GPU that loads it holds these 128 KB until the process
// exits).
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Logits scratch, [T][E] fp32 with T * E <= MOE_ROUTE_STATIC_MAX_LOGITS.
static __device__ __align__(256) float g_route_scratch[MOE_ROUTE_STATIC_MAX_LOGITS];

std::mutex g_setup_mutex;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is asked of
// the runtime once per device, with that device current.
cudaError_t scratch_on_current_device(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" moe_status moe_route_static(const void* x, int32_t T, int32_t H, int32_t E, int32_t k,
                                       const float* router_w, const float* router_b,
                                       int32_t* topk_idx, float* topk_w, void* stream) {
  if (T < 0 || H <= 0 || H % 128 != 0 || H > 16384 || E < 1 || E > 512 || k < 1 || k > 8 || k > E)
    return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * E > MOE_ROUTE_STATIC_MAX_LOGITS) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if ((uintptr_t)x % 16 != 0 || (uintptr_t)router_w % 16 != 0) return MOE_ERR_INVALID_ARG;
  float* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  // Every logit the top-k pass reads is written by the logits pass first, so
  // nothing in the scratch has to start at zero.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = moe::launch_router_logits(static_cast<const uint16_t*>(x), T, H, E, router_w, router_b,
                                scratch, 0, st);
  if (e == cudaSuccess) e = moe::launch_topk(scratch, T, E, k, moe::Scoring{0, 1.0f, nullptr}, topk_idx, topk_w, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

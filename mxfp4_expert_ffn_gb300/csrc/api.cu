// The C ABI (include/moe_ffn.h): validation, workspace, launch sequencing,
// error reporting, optional per-kernel timing and host-side fault injection.
#include <stdlib.h>
#include <string.h>

#include <new>

#include "common.cuh"
#include "internal.h"

namespace moe {
cudaError_t prepare_segments_kernel(int E);
cudaError_t prepare_ffn_simt(int H, int I);
}  // namespace moe

namespace {

using namespace moe;

// Host-side fault injection for tests: MOE_FAULT=alloc makes
// moe_layer_create fail before allocating, MOE_FAULT=launch makes
// moe_forward / moe_route fail before launching, MOE_FAULT=arg makes them
// reject their arguments.  Nothing is injected on the device.
bool fault(const char* what) {
  const char* f = getenv("MOE_FAULT");
  return f && strcmp(f, what) == 0;
}

moe_status cuda_fail(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  cudaGetLastError();  // clear the (non-sticky) error state
  return MOE_ERR_CUDA;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Carver {
  char* base;
  size_t off = 0;
  template <class T>
  T* take(size_t n) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = align_up(off + n * sizeof(T), 256);
    return p;
  }
};

// Lays out the workspace in one allocation (base = nullptr: sizing pass).
size_t carve(const moe_config& c, int num_sms, char* base, Workspace& ws) {
  const size_t T = (size_t)c.max_tokens, H = (size_t)c.hidden, I = (size_t)c.inter;
  const size_t k = (size_t)c.top_k, E = (size_t)c.n_experts, ns = (size_t)c.n_shared;
  const size_t NE = E + ns, S = T * k, P = S + ns * T;
  Carver cv{base};
  ws.xq = cv.take<uint8_t>(T * H);
  ws.xs = cv.take<uint8_t>(T * H / 32);
  ws.cnt = cv.take<int32_t>(NE);
  ws.off = cv.take<int32_t>(NE + 1);
  ws.perm = cv.take<int32_t>(S);
  ws.slot_pos = cv.take<int32_t>(S);
  ws.pos_tok = cv.take<int32_t>(P);
  ws.active = cv.take<int32_t>(NE);
  ws.n_active = cv.take<int32_t>(2);
  ws.tile_prefix = cv.take<int32_t>(NE + 1);
  // sum over experts of ceil(tokens / 16) <= slots / 16 + experts
  ws.tile_info = cv.take<int4>(P / 16 + NE + 16);
  ws.xg = cv.take<uint8_t>(P * H);
  ws.xgs = cv.take<uint8_t>(P * H / 32);
  ws.hq = cv.take<uint8_t>(P * I);
  ws.hs = cv.take<uint8_t>(P * I / 32);
  ws.o = cv.take<float>(P * H);
  ws.logits = cv.take<float>(T * E);
  const size_t split_rows = 8 * (T < (size_t)kRouterSplitMaxT ? T : (size_t)kRouterSplitMaxT);
  ws.rpart = cv.take<float>((split_rows > 4 * T ? split_rows : 4 * T) * E);
  ws.w3 = cv.take<uint16_t>(3 * E * H);
  ws.idx = cv.take<int32_t>(T * k);
  ws.w = cv.take<float>(T * k);
  ws.x = cv.take<uint16_t>(T * H);
  // the error word right before y (256 bytes apart): one copy brings back both
  ws.err = cv.take<int32_t>(1);
  ws.y = cv.take<uint16_t>(T * H);
  // split partition of the tensor-core GEMM (few units, e.g. decode): two
  // partial slots per CTA and one counter per (unit, row quadrant), units < 4 * SMs
  ws.part_bn = mma_tile_for_tokens(c.max_tokens) < 64 ? mma_tile_for_tokens(c.max_tokens) : 64;
  // (one region per GEMM: down may start while gate/up finishes)
  ws.part = cv.take<float>((size_t)2 * 2 * num_sms * 2 * ws.part_bn * 128);
  ws.split_cnt_n = 2 * 4 * kSplitUnitsPerCta * num_sms + (int)NE + 2;
  ws.split_cnt = cv.take<int32_t>((size_t)ws.split_cnt_n);
  ws.ready = ws.split_cnt + 2 * 4 * kSplitUnitsPerCta * num_sms;
  ws.ready_done = ws.ready + NE;
  ws.unit_next = ws.ready_done + 1;
  ws.prep_cnt = cv.take<int32_t>(32);  // one per token block (at most 16) and one for the blocks
  ws.comb_cnt_n = kPrepMaxTokens * (int)(H / 128) * 4;
  ws.comb_cnt = cv.take<int32_t>((size_t)ws.comb_cnt_n);
  ws.seg_cbase = cv.take<int32_t>((size_t)kSegCtas * E);
  ws.seg_counter = cv.take<int32_t>(1);
  ws.seg_routed = cv.take<int32_t>(1);
  return cv.off;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

moe_status validate_config(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  const bool ok = c->hidden >= 128 && c->hidden <= 16384 && c->hidden % 128 == 0 &&
                  c->inter >= 128 && c->inter <= 16384 && c->inter % 128 == 0 &&
                  c->n_experts >= 1 && c->n_experts <= 512 && c->top_k >= 1 && c->top_k <= 8 &&
                  c->top_k <= c->n_experts && c->n_shared >= 0 && c->n_shared <= 4 &&
                  c->max_tokens >= 1 && c->max_tokens <= 65536;
  return ok ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

moe_status validate_weights(const moe_config* c, const moe_weights* w) {
  if (!w || !w->router_w) return MOE_ERR_INVALID_ARG;
  const moe_mx_mat* routed[3] = {&w->gate, &w->up, &w->down};
  const moe_mx_mat* shared[3] = {&w->s_gate, &w->s_up, &w->s_down};
  for (int i = 0; i < 3; ++i) {
    if (!routed[i]->codes || !routed[i]->scales) return MOE_ERR_INVALID_ARG;
    if (!aligned(routed[i]->codes, 32) || !aligned(routed[i]->scales, 32)) return MOE_ERR_INVALID_ARG;
    if (c->n_shared > 0) {
      if (!shared[i]->codes || !shared[i]->scales) return MOE_ERR_INVALID_ARG;
      if (!aligned(shared[i]->codes, 32) || !aligned(shared[i]->scales, 32)) return MOE_ERR_INVALID_ARG;
    }
  }
  if (!aligned(w->router_w, 16)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

ExpertBank bank_of(const moe_layer* L) {
  ExpertBank b;
  b.gc = L->w.gate.codes;
  b.gs = L->w.gate.scales;
  b.uc = L->w.up.codes;
  b.us = L->w.up.scales;
  b.dc = L->w.down.codes;
  b.ds = L->w.down.scales;
  b.sgc = L->w.s_gate.codes;
  b.sgs = L->w.s_gate.scales;
  b.suc = L->w.s_up.codes;
  b.sus = L->w.s_up.scales;
  b.sdc = L->w.s_down.codes;
  b.sds = L->w.s_down.scales;
  b.E = L->cfg.n_experts;
  b.H = L->cfg.hidden;
  b.I = L->cfg.inter;
  return b;
}

// Makes the layer's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  cudaError_t status = cudaSuccess;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) status = cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// Records a pair of events around one launch while timing is on.
struct TimedScope {
  moe_layer* L;
  cudaStream_t st;
  int pair = -1;
  TimedScope(moe_layer* layer, cudaStream_t s, const char* name) : L(layer), st(s) {
    if (!L || !L->timing || L->ev_used >= 64) return;
    int t = 0;
    while (t < L->n_timers && strcmp(L->timers[t].name, name) != 0) ++t;
    if (t == L->n_timers) {
      if (t == kMaxTimed) return;
      L->timers[t].name = name;
      L->n_timers++;
    }
    pair = L->ev_used++;
    L->ev_pending_timer[pair] = t;
    cudaEventRecord(L->ev_pool[2 * pair], st);
  }
  ~TimedScope() {
    if (pair >= 0) cudaEventRecord(L->ev_pool[2 * pair + 1], st);
  }
};

void collect_times(moe_layer* L) {
  for (int p = 0; p < L->ev_used; ++p) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, L->ev_pool[2 * p], L->ev_pool[2 * p + 1]) == cudaSuccess) {
      L->timers[L->ev_pending_timer[p]].ms += ms;
      L->timers[L->ev_pending_timer[p]].launches += 1;
    }
  }
  cudaGetLastError();
  L->ev_used = 0;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or option";
    case MOE_ERR_OOM: return "device memory allocation failed";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_INTERNAL: return "device-side check failed (expert id out of range)";
  }
  return "unknown status";
}

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

}  // extern "C"

namespace {

// A layer computing the routed experts [e_lo, e_hi) (all of them: 0, E),
// whose routed banks hold those experts only.
moe_status create_impl(const moe_config* cfg, const moe_weights* w, int device, int e_lo, int e_hi,
                       moe_layer** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_status st = validate_config(cfg);
  if (st != MOE_OK) return st;
  if ((st = validate_weights(cfg, w)) != MOE_OK) return st;
  if (e_lo < 0 || e_hi > cfg->n_experts || e_lo >= e_hi) return MOE_ERR_INVALID_ARG;
  const bool partial = e_lo != 0 || e_hi != cfg->n_experts;
  if (fault("alloc")) return MOE_ERR_OOM;
  DeviceGuard g(device);
  if (g.status != cudaSuccess) return cuda_fail(g.status);
  moe_layer* L = new (std::nothrow) moe_layer();
  if (!L) return MOE_ERR_OOM;
  L->cfg = *cfg;
  L->w = *w;
  L->device = device;
  if (cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    delete L;
    return cuda_fail(cudaErrorInvalidDevice);
  }
  Workspace sizing;
  const size_t bytes = carve(*cfg, L->num_sms, nullptr, sizing);
  void* base = nullptr;
  if (cudaMalloc(&base, bytes) != cudaSuccess) {
    cudaGetLastError();
    delete L;
    return MOE_ERR_OOM;
  }
  carve(*cfg, L->num_sms, static_cast<char*>(base), L->ws);
  L->ws.e_lo = e_lo;
  L->ws.e_hi = e_hi;
  L->ws.base = base;
  L->ws.bytes = bytes;
  cudaError_t e = cudaMemset(base, 0, bytes);
  // pinned staging of the host entry point: the error word, then y of batches
  // of up to 16 KB (one device-to-host copy for both; larger ones are copied
  // straight to the caller, a second host copy would cost more than it saves)
  L->out_rows = (int)(16384 / ((size_t)cfg->hidden * sizeof(uint16_t)));
  if (L->out_rows > cfg->max_tokens) L->out_rows = cfg->max_tokens;
  if (e == cudaSuccess)
    e = cudaMallocHost(&L->ws.err_host, 256 + (size_t)L->out_rows * cfg->hidden * sizeof(uint16_t));
  if (e == cudaSuccess) e = prepare_segments_kernel(cfg->n_experts);
  if (e == cudaSuccess) e = prepare_ffn_simt(cfg->hidden, cfg->inter);
  if (e == cudaSuccess) e = prepare_prep_kernel(cfg->n_experts, cfg->hidden);
  if (e == cudaSuccess) {
    L->maps = mma_maps_create(*cfg, *w, L->ws);  // NULL: tensor-core path unavailable
    cudaGetLastError();
    // a range of experts runs on the tensor cores only (the SIMT kernels index
    // the banks by the global expert id)
    if (partial && !L->maps) e = cudaErrorNotSupported;
    if (e == cudaSuccess) e = router_split_weights(w->router_w, cfg->n_experts, cfg->hidden, L->ws.w3, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
      L->router_mma = router_map_weights(&L->router_map, L->ws.w3, cfg->n_experts, cfg->hidden);
  }
  if (e != cudaSuccess) {
    if (L->ws.err_host) cudaFreeHost(L->ws.err_host);
    mma_maps_destroy(L->maps);
    cudaFree(base);
    delete L;
    if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
    return cuda_fail(e);
  }
  *out = L;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_layer_create(const moe_config* cfg, const moe_weights* w, int device,
                            moe_layer** out) {
  if (!cfg) {
    if (out) *out = nullptr;
    return MOE_ERR_INVALID_ARG;
  }
  return create_impl(cfg, w, device, 0, cfg->n_experts, out);
}

moe_status moe_layer_create_range(const moe_config* cfg, const moe_weights* w, int device,
                                  int32_t expert_begin, int32_t expert_end, moe_layer** out) {
  if (!cfg) {
    if (out) *out = nullptr;
    return MOE_ERR_INVALID_ARG;
  }
  return create_impl(cfg, w, device, expert_begin, expert_end, out);
}

moe_status moe_destroy(moe_layer* L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  cudaError_t e = cudaDeviceSynchronize();
  for (int i = 0; i < 128; ++i)
    if (L->ev_pool[i]) cudaEventDestroy(L->ev_pool[i]);
  if (L->ws.err_host) cudaFreeHost(L->ws.err_host);
  cudaFree(L->ws.base);
  mma_maps_destroy(L->maps);
  delete L;
  return cuda_fail(e);
}

moe_status moe_layer_destroy(moe_layer* L) { return moe_destroy(L); }

moe_status moe_set_option(moe_layer* L, int32_t option, int64_t value) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (option == MOE_OPT_PATH) {
    if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
    if (value == 2 && !L->maps) return MOE_ERR_UNSUPPORTED;
    if (value == 1 && (L->act_format == MOE_ACT_FP4 || L->shared_format == MOE_SHARED_FP8_B32 ||
                       L->ws.e_lo != 0 || L->ws.e_hi != L->cfg.n_experts))
      return MOE_ERR_UNSUPPORTED;  // no SIMT path for these variants, nor for a range of experts
    L->path = (int)value;
    return MOE_OK;
  }
  if (option == MOE_OPT_SCORING) {
    if (value != MOE_SCORING_SOFTMAX && value != MOE_SCORING_SIGMOID) return MOE_ERR_INVALID_ARG;
    L->scoring = (int)value;
    return MOE_OK;
  }
  if (option == MOE_OPT_ROUTED_SCALE) {
    if (value < 0 || value > 0xFFFFFFFFll) return MOE_ERR_INVALID_ARG;
    const uint32_t bits = (uint32_t)value;
    float f;
    memcpy(&f, &bits, sizeof f);
    if (!(f > 0.f) || f > 3.0e38f) return MOE_ERR_INVALID_ARG;  // positive, finite (NaN fails too)
    L->routed_scale = f;
    return MOE_OK;
  }
  if (option == MOE_OPT_SHARED_FORMAT) {
    if (value != MOE_SHARED_MXFP4 && value != MOE_SHARED_FP8_B32) return MOE_ERR_INVALID_ARG;
    // FP8 shared experts: tensor-core path with FP8 activations only
    if (value == MOE_SHARED_FP8_B32 &&
        (!L->maps || L->cfg.n_shared == 0 || L->path == 1 || L->act_format == MOE_ACT_FP4))
      return MOE_ERR_UNSUPPORTED;
    if (value == L->shared_format) return MOE_OK;
    if (!mma_maps_set_shared_format(L->maps, L->cfg, L->w, value == MOE_SHARED_FP8_B32)) return MOE_ERR_UNSUPPORTED;
    L->shared_format = (int)value;
    return MOE_OK;
  }
  if (option == MOE_OPT_ACT_FORMAT) {
    if (value != MOE_ACT_FP8 && value != MOE_ACT_FP4) return MOE_ERR_INVALID_ARG;
    // FP4 activations run on the tensor cores only, for H and I multiples of 256
    if (value == MOE_ACT_FP4 && (!L->maps || !mma_act4_supported(L->cfg))) return MOE_ERR_UNSUPPORTED;
    if (value == MOE_ACT_FP4 && L->shared_format == MOE_SHARED_FP8_B32) return MOE_ERR_UNSUPPORTED;
    L->act_format = (int)value;
    return MOE_OK;
  }
  if (option == MOE_OPT_WAIT_LIMIT) {
    if (value < 0 || value > 0x7FFFFFFFll) return MOE_ERR_INVALID_ARG;
    L->wait_limit = (uint32_t)value;
    return MOE_OK;
  }
  if (option == MOE_OPT_TIMING) {
    DeviceGuard g(L->device);
    if (value && !L->ev_pool[0]) {
      for (int i = 0; i < 128; ++i)
        if (cudaEventCreate(&L->ev_pool[i]) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    }
    L->timing = value != 0;
    return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status moe_get_kernel_times(moe_layer* L, const char** names, double* ms, int64_t* launches,
                                int32_t cap, int32_t* n) {
  if (!L || !n || cap < 0 || (cap > 0 && (!names || !ms || !launches))) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  cudaError_t e = cudaDeviceSynchronize();
  collect_times(L);
  *n = L->n_timers;
  for (int i = 0; i < L->n_timers && i < cap; ++i) {
    names[i] = L->timers[i].name;
    ms[i] = L->timers[i].ms;
    launches[i] = L->timers[i].launches;
  }
  for (int i = 0; i < L->n_timers; ++i) {
    L->timers[i].ms = 0.0;
    L->timers[i].launches = 0;
  }
  return cuda_fail(e);
}

moe_status moe_sync(moe_layer* L, void* stream) {
  if (!L) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(L->ws.err_host, L->ws.err, sizeof(int32_t),
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  const int32_t bits = *L->ws.err_host;
  if (bits) {
    e = cudaMemsetAsync(L->ws.err, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    return (bits & kErrTimeout) ? MOE_ERR_TIMEOUT : MOE_ERR_INTERNAL;
  }
  return MOE_OK;
}

}  // extern "C"

namespace {

moe_status check_tokens(const moe_layer* L, int32_t T) {
  if (!L || T < 0 || T > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (fault("arg")) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

Scoring scoring_of(const moe_layer* L) {
  return Scoring{L->scoring, L->routed_scale, L->w.router_b};
}

moe_status route_impl(moe_layer* L, const void* x, int32_t T, const float* logits_in,
                      float* logits_out, int32_t* idx, float* w, cudaStream_t st) {
  const moe_config& c = L->cfg;
  cudaError_t e = cudaSuccess;
  const float* lg = logits_in;
  if (!lg && T <= kRouterSplitMaxT) {
    // small T: split-K logits (W_r streamed by ~E/8 x 8 CTAs), summed in the top-k pass
    TimedScope ts(L, st, "router_split");
    return cuda_fail(launch_router_split(static_cast<const uint16_t*>(x), T, c.hidden, c.n_experts,
                                         c.top_k, L->w.router_w, L->w.router_b, scoring_of(L),
                                         L->ws.rpart, logits_out, idx, w, st));
  }
  if (!lg && L->router_mma && L->path != 1) {
    // many tokens: tensor-core logits (three bf16 parts of W_r), K split over CTAs
    TimedScope ts(L, st, "router_mma");
    e = launch_router_mma(L->router_map, static_cast<const uint16_t*>(x), T, c.n_experts, c.hidden,
                          L->ws.rpart, L->ws.err, L->num_sms, st);
    if (e == cudaSuccess)
      e = launch_topk_sum(L->ws.rpart, router_mma_ksplit(c.hidden), L->w.router_b, T, c.n_experts,
                          c.top_k, scoring_of(L), logits_out, idx, w, st);
    return cuda_fail(e);
  }
  if (!lg) {
    float* dst = logits_out ? logits_out : L->ws.logits;
    TimedScope ts(L, st, "router_logits");
    e = launch_router_logits(static_cast<const uint16_t*>(x), T, c.hidden, c.n_experts, L->w.router_w,
                             L->scoring ? nullptr : L->w.router_b, dst, L->num_sms, st);
    lg = dst;
  } else if (logits_out && logits_out != logits_in) {
    e = cudaMemcpyAsync(logits_out, logits_in, sizeof(float) * (size_t)T * c.n_experts,
                        cudaMemcpyDeviceToDevice, st);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  {
    TimedScope ts(L, st, "topk");
    e = launch_topk(lg, T, c.n_experts, c.top_k, scoring_of(L), idx, w, st);
  }
  return cuda_fail(e);
}

// The tensor-core path is faster at every token count measured (decode T = 1
// included); SIMT is kept for MOE_OPT_PATH = 1 and for shapes without maps.
bool use_mma(const moe_layer* L, int T) {
  (void)T;
  if (!L->maps) return false;
  return L->path != 1;
}

bool act4_of(const moe_layer* L) { return L->act_format == MOE_ACT_FP4; }

// gate/up, down and combine on the tensor cores, once the segments and the
// activation codes are in the workspace.  small: up to kPrepMaxTokens tokens
// after the preparation kernel (token-major codes, every expert in one tile):
// gate/up reads all tokens' codes (dense) and, with shared experts, the down
// GEMM does the combine.
// y_f32 (expert parallelism): the fp32 sums are stored there instead of y.
moe_status ffn_tail(moe_layer* L, int32_t T, int bn, bool small, const float* w,
                    const void* residual, void* y, cudaStream_t st, float* y_f32 = nullptr) {
  const moe_config& c = L->cfg;
  const ExpertBank bank = bank_of(L);
  const int ns_tiles = c.n_shared * ((T + bn - 1) / bn);
  cudaError_t e;
  {
    TimedScope ts(L, st, "ffn_up_mma");
    e = launch_ffn_mma(*L->maps, bank, 0, bn, small ? T : 0, L->ws, L->num_sms, st, nullptr, act4_of(L), ns_tiles,
                       L->wait_limit, small);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  if (small && bn == 16 && c.n_shared > 0 && !y_f32) {
    // up to 16 tokens: the combine runs inside the down GEMM (every token has a
    // shared-expert position, so every y row has a last writer).  With wider
    // tiles a unit is the last writer of up to 64 tokens, whose combines one
    // warp would do one after the other; the combine kernel does them in
    // parallel instead.
    const CombineArgs cmb{T, c.top_k, c.n_shared, w, static_cast<const uint16_t*>(residual),
                          static_cast<uint16_t*>(y)};
    TimedScope ts(L, st, "ffn_down_mma");
    return cuda_fail(launch_ffn_mma(*L->maps, bank, 1, bn, 0, L->ws, L->num_sms, st, &cmb, act4_of(L), ns_tiles,
                                    L->wait_limit, small));
  }
  {
    TimedScope ts(L, st, "ffn_down_mma");
    e = launch_ffn_mma(*L->maps, bank, 1, bn, 0, L->ws, L->num_sms, st, nullptr, act4_of(L), ns_tiles,
                       L->wait_limit, small);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  {
    TimedScope ts(L, st, "combine");
    e = launch_combine(L->ws, T, c.hidden, c.top_k, c.n_shared, w,
                       static_cast<const uint16_t*>(residual), static_cast<uint16_t*>(y), st, y_f32);
  }
  return cuda_fail(e);
}

moe_status forward_impl(moe_layer* L, const void* x, int32_t T, const int32_t* idx,
                        const float* w, const void* residual, void* y, cudaStream_t st,
                        float* y_f32 = nullptr) {
  const moe_config& c = L->cfg;
  const ExpertBank bank = bank_of(L);
  const bool mma = use_mma(L, T);
  const int bn = mma ? mma_tile_for_tokens(T) : 0;
  cudaError_t e;
  if (mma && T <= kPrepMaxTokens) {
    {
      TimedScope ts(L, st, "prep");
      e = launch_prep(static_cast<const uint16_t*>(x), T, c.hidden, c.n_experts, c.top_k, c.n_shared,
                      bn, nullptr, nullptr, scoring_of(L), nullptr, const_cast<int32_t*>(idx), nullptr, false,
                      act4_of(L), L->ws, st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return ffn_tail(L, T, bn, true, w, residual, y, st, y_f32);
  }
  {
    TimedScope ts(L, st, "segments");
    e = launch_segments(idx, T, c.top_k, c.n_experts, c.n_shared, bn, L->ws, st);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  if (mma) {
    {
      TimedScope ts(L, st, "quantize_scatter");
      e = launch_quantize_scatter(static_cast<const uint16_t*>(x), T, c.hidden, c.top_k, c.n_shared,
                                  L->ws.slot_pos, L->ws.xg, L->ws.xgs, act4_of(L), st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return ffn_tail(L, T, bn, false, w, residual, y, st, y_f32);
  } else {
    // the FP4-activation and FP8-shared-expert variants run on the tensor cores only
    if (act4_of(L) || L->shared_format == MOE_SHARED_FP8_B32) return MOE_ERR_UNSUPPORTED;
    {
      TimedScope ts(L, st, "quantize_act");
      e = launch_quantize_act(static_cast<const uint16_t*>(x), T, c.hidden, L->ws.xq, L->ws.xs, st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    {
      TimedScope ts(L, st, "ffn_up_simt");
      e = launch_ffn_up_simt(bank, T, c.top_k, c.n_shared, L->ws, L->num_sms, st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    {
      TimedScope ts(L, st, "ffn_down_simt");
      e = launch_ffn_down_simt(bank, T, c.top_k, c.n_shared, L->ws, L->num_sms, st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
  }
  {
    TimedScope ts(L, st, "combine");
    e = launch_combine(L->ws, T, c.hidden, c.top_k, c.n_shared, w,
                       static_cast<const uint16_t*>(residual), static_cast<uint16_t*>(y), st, y_f32);
  }
  return cuda_fail(e);
}

// Route and forward in one pass.  For small batches on the tensor cores the
// router, top-k, the x codes and the segments are a single launch.
moe_status step_impl(moe_layer* L, const void* x, int32_t T, const void* residual, void* y,
                     int32_t* idx, float* w, float* logits_out, cudaStream_t st) {
  const moe_config& c = L->cfg;
  if (!idx) idx = L->ws.idx;
  if (!w) w = L->ws.w;
  if (use_mma(L, T) && T <= kPrepMaxTokens) {
    const int bn = mma_tile_for_tokens(T);
    cudaError_t e = cudaSuccess;
    // above 8 tokens the router's partial sums and the codes of x come from a
    // register-tiled launch, then selection and segments from the preparation
    // launch; up to 8 tokens (one token block) the preparation launch does it
    // all (one launch less on the decode path)
    const bool tile = T > 8 && router_tile_quantises(c.hidden);
    if (tile) {
      TimedScope ts(L, st, "router_tile");
      e = launch_router_tile(static_cast<const uint16_t*>(x), T, c.hidden, c.n_experts, L->w.router_w, L->ws.rpart,
                             L->ws.xq, L->ws.xs, act4_of(L), st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    {
      TimedScope ts(L, st, "prep");
      e = launch_prep(static_cast<const uint16_t*>(x), T, c.hidden, c.n_experts, c.top_k, c.n_shared,
                      bn, L->w.router_w, L->w.router_b, scoring_of(L), logits_out, idx, w, true, act4_of(L),
                      L->ws, st, tile);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return ffn_tail(L, T, bn, true, w, residual, y, st);
  }
  moe_status s = route_impl(L, x, T, nullptr, logits_out, idx, w, st);
  if (s != MOE_OK) return s;
  return forward_impl(L, x, T, idx, w, residual, y, st);
}

}  // namespace

extern "C" {

moe_status moe_step(moe_layer* L, const void* x, int32_t T, const void* residual, void* y,
                    int32_t* topk_idx, float* topk_w, float* logits_out, void* stream) {
  moe_status s = check_tokens(L, T);
  if (s != MOE_OK || T == 0) return s;
  if (!x || !y || x == y) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || (residual && !aligned(residual, 16)))
    return MOE_ERR_INVALID_ARG;
  if (fault("launch")) return MOE_ERR_CUDA;
  DeviceGuard g(L->device);
  if (g.status != cudaSuccess) return cuda_fail(g.status);
  return step_impl(L, x, T, residual, y, topk_idx, topk_w, logits_out,
                   static_cast<cudaStream_t>(stream));
}

moe_status moe_route(moe_layer* L, const void* x, int32_t T, const float* logits_in,
                     float* logits_out, int32_t* topk_idx, float* topk_w, void* stream) {
  moe_status s = check_tokens(L, T);
  if (s != MOE_OK || T == 0) return s;
  if (!topk_idx || !topk_w || (!logits_in && !x)) return MOE_ERR_INVALID_ARG;
  if (x && !aligned(x, 16)) return MOE_ERR_INVALID_ARG;
  if (fault("launch")) return MOE_ERR_CUDA;
  DeviceGuard g(L->device);
  if (g.status != cudaSuccess) return cuda_fail(g.status);
  return route_impl(L, x, T, logits_in, logits_out, topk_idx, topk_w,
                    static_cast<cudaStream_t>(stream));
}

moe_status moe_forward(moe_layer* L, const void* x, int32_t T, const int32_t* topk_idx,
                       const float* topk_w, const void* residual, void* y, void* stream) {
  moe_status s = check_tokens(L, T);
  if (s != MOE_OK || T == 0) return s;
  if (!x || !topk_idx || !topk_w || !y || x == y) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || (residual && !aligned(residual, 16)))
    return MOE_ERR_INVALID_ARG;
  if (fault("launch")) return MOE_ERR_CUDA;
  DeviceGuard g(L->device);
  if (g.status != cudaSuccess) return cuda_fail(g.status);
  return forward_impl(L, x, T, topk_idx, topk_w, residual, y, static_cast<cudaStream_t>(stream));
}

moe_status moe_forward_partial(moe_layer* L, const void* x, int32_t T, const int32_t* topk_idx,
                               const float* topk_w, float* y_partial, void* stream) {
  moe_status s = check_tokens(L, T);
  if (s != MOE_OK || T == 0) return s;
  if (!x || !topk_idx || !topk_w || !y_partial) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y_partial, 16)) return MOE_ERR_INVALID_ARG;
  if (fault("launch")) return MOE_ERR_CUDA;
  DeviceGuard g(L->device);
  if (g.status != cudaSuccess) return cuda_fail(g.status);
  return forward_impl(L, x, T, topk_idx, topk_w, nullptr, nullptr, static_cast<cudaStream_t>(stream), y_partial);
}

moe_status moe_combine_partials(const float* partials, int32_t n_parts, int32_t T, int32_t H,
                                const void* residual, void* y, void* stream) {
  if (n_parts < 1 || T < 0 || H <= 0 || H % 4 != 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!partials || !y || !aligned(partials, 16) || !aligned(y, 8) || (residual && !aligned(residual, 8)))
    return MOE_ERR_INVALID_ARG;
  return cuda_fail(launch_combine_parts(partials, n_parts, T, H, static_cast<const uint16_t*>(residual),
                                        static_cast<uint16_t*>(y), static_cast<cudaStream_t>(stream)));
}

moe_status moe_forward_host(moe_layer* L, const void* x_host, int32_t T, void* y_host,
                            void* stream) {
  moe_status s = check_tokens(L, T);
  if (s != MOE_OK || T == 0) return s;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  if (fault("launch")) return MOE_ERR_CUDA;
  DeviceGuard g(L->device);
  if (g.status != cudaSuccess) return cuda_fail(g.status);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)T * L->cfg.hidden * sizeof(uint16_t);
  cudaError_t e = cudaMemcpyAsync(L->ws.x, x_host, bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((s = step_impl(L, L->ws.x, T, nullptr, L->ws.y, nullptr, nullptr, nullptr, st)) != MOE_OK) return s;
  if (T > L->out_rows || reinterpret_cast<char*>(L->ws.err) + 256 != reinterpret_cast<char*>(L->ws.y)) {
    e = cudaMemcpyAsync(y_host, L->ws.y, bytes, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return moe_sync(L, stream);
  }
  // small batches: the error word and y in one copy through the pinned staging
  e = cudaMemcpyAsync(L->ws.err_host, L->ws.err, 256 + bytes, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  memcpy(y_host, reinterpret_cast<const char*>(L->ws.err_host) + 256, bytes);
  const int32_t bits = *L->ws.err_host;
  if (bits) {
    e = cudaMemsetAsync(L->ws.err, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    return (bits & kErrTimeout) ? MOE_ERR_TIMEOUT : MOE_ERR_INTERNAL;
  }
  return MOE_OK;
}

moe_status moe_stack_forward_host(moe_layer* const* Ls, int32_t n, const void* x_host, int32_t T,
                                  float norm_eps, void* y_host, void* stream) {
  if (!Ls || n < 1 || n > 64 || !x_host || !y_host || norm_eps != norm_eps) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < n; ++l) {
    moe_status s = check_tokens(Ls[l], T);
    if (s != MOE_OK) return s;
    if (Ls[l]->device != Ls[0]->device || Ls[l]->cfg.hidden != Ls[0]->cfg.hidden) return MOE_ERR_INVALID_ARG;
  }
  if (T == 0) return MOE_OK;
  if (fault("launch")) return MOE_ERR_CUDA;
  DeviceGuard g(Ls[0]->device);
  if (g.status != cudaSuccess) return cuda_fail(g.status);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int H = Ls[0]->cfg.hidden;
  const bool norm = norm_eps >= 0.f;
  const size_t bytes = (size_t)T * H * sizeof(uint16_t);
  // The residual stream: the input in layer 0's y (normalised: x_0 is only
  // read as the residual) or x (not normalised: x_0 is the layer's input),
  // then each layer's output in its own y.  A layer's y may alias its
  // residual but never its input.
  uint16_t* cur = norm ? Ls[0]->ws.y : Ls[0]->ws.x;
  cudaError_t e = cudaMemcpyAsync(cur, x_host, bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e);
  for (int l = 0; l < n; ++l) {
    moe_layer* L = Ls[l];
    const uint16_t* in = cur;
    if (norm) {
      e = launch_rmsnorm(cur, T, H, norm_eps, L->ws.x, st);
      if (e != cudaSuccess) return cuda_fail(e);
      in = L->ws.x;
    }
    uint16_t* out = (!norm && cur == L->ws.y) ? L->ws.x : L->ws.y;
    moe_status s = step_impl(L, in, T, cur, out, nullptr, nullptr, nullptr, st);
    if (s != MOE_OK) return s;
    cur = out;
  }
  e = cudaMemcpyAsync(y_host, cur, bytes, cudaMemcpyDeviceToHost, st);
  for (int l = 0; e == cudaSuccess && l < n; ++l)
    e = cudaMemcpyAsync(Ls[l]->ws.err_host, Ls[l]->ws.err, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  int32_t bits = 0;
  for (int l = 0; l < n; ++l) {
    const int32_t b = *Ls[l]->ws.err_host;
    if (b) {
      bits |= b;
      e = cudaMemsetAsync(Ls[l]->ws.err, 0, sizeof(int32_t), st);
      if (e != cudaSuccess) return cuda_fail(e);
    }
  }
  if (bits) {
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    return (bits & kErrTimeout) ? MOE_ERR_TIMEOUT : MOE_ERR_INTERNAL;
  }
  return MOE_OK;
}

moe_status moe_quantize_act(moe_layer* L, const void* x, int32_t T, uint8_t* q, uint8_t* s,
                            void* stream) {
  moe_status st = check_tokens(L, T);
  if (st != MOE_OK || T == 0) return st;
  if (!x || !q || !s || !aligned(x, 16) || !aligned(q, 8)) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  if (g.status != cudaSuccess) return cuda_fail(g.status);
  TimedScope ts(L, static_cast<cudaStream_t>(stream), "quantize_act");
  return cuda_fail(launch_quantize_act(static_cast<const uint16_t*>(x), T, L->cfg.hidden, q, s,
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_quantize_act4(moe_layer* L, const void* x, int32_t T, uint8_t* q, uint8_t* s,
                             void* stream) {
  moe_status st = check_tokens(L, T);
  if (st != MOE_OK || T == 0) return st;
  if (!x || !q || !s || !aligned(x, 16) || !aligned(q, 4)) return MOE_ERR_INVALID_ARG;
  if (L->cfg.hidden % 256 != 0) return MOE_ERR_UNSUPPORTED;
  DeviceGuard g(L->device);
  if (g.status != cudaSuccess) return cuda_fail(g.status);
  TimedScope ts(L, static_cast<cudaStream_t>(stream), "quantize_act4");
  return cuda_fail(launch_quantize_act4(static_cast<const uint16_t*>(x), T, L->cfg.hidden, q, s,
                                        static_cast<cudaStream_t>(stream)));
}

moe_status moe_segments(moe_layer* L, const int32_t* topk_idx, int32_t T, int32_t* offsets,
                        int32_t* perm, void* stream) {
  moe_status s = check_tokens(L, T);
  if (s != MOE_OK) return s;
  if (!topk_idx || !offsets || !perm) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  if (g.status != cudaSuccess) return cuda_fail(g.status);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const moe_config& c = L->cfg;
  cudaError_t e = launch_segments(topk_idx, T, c.top_k, c.n_experts, c.n_shared, 0, L->ws, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(offsets, L->ws.off, sizeof(int32_t) * (c.n_experts + 1),
                        cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && T > 0)
    e = cudaMemcpyAsync(perm, L->ws.perm, sizeof(int32_t) * (size_t)T * c.top_k,
                        cudaMemcpyDeviceToDevice, st);
  return cuda_fail(e);
}

moe_status moe_rmsnorm(const void* x, int32_t T, int32_t H, float eps, void* out, void* stream) {
  if (T < 0 || H <= 0 || H % 8 != 0 || H > 65536 || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out || !aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  return cuda_fail(launch_rmsnorm(static_cast<const uint16_t*>(x), T, H, eps,
                                  static_cast<uint16_t*>(out), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

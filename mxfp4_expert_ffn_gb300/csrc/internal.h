// Internal declarations: the layer handle and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_ffn.h"

namespace moe {

constexpr int kMaxTimed = 16;

// How routed weights are formed from the fp32 router logits l.
//  softmax (0): the bias is part of l; selection on l; w = softmax over the k
//               selected l.
//  sigmoid (1): s = sigmoid(l) with l unbiased; selection on s + bias; w = s /
//               (sum of the k selected s).  The DeepSeek-V3 style gate.
// In both, w is then multiplied by scale (the routed scaling factor).
struct Scoring {
  int sigmoid;
  float scale;
  const float* sel_bias;  // sigmoid: per-expert selection bias, or null
};


// Device workspace, sized at create time for cfg.max_tokens.
// Positions: the T*k routed slots grouped expert by expert (stable in slot
// order), then n_shared blocks of T positions for the shared experts
// (position S + s*T + t is token t of shared expert s).
struct Workspace {
  uint8_t* xq = nullptr;      // [T][H]     E4M3 codes of x
  uint8_t* xs = nullptr;      // [T][H/32]  UE8M0 scale bytes of x
  int32_t* cnt = nullptr;     // [NE]       tokens per expert (NE = E + n_shared)
  int32_t* off = nullptr;     // [NE+1]     first position of each expert
  int32_t* perm = nullptr;    // [T*k]      slot of each routed position
  int32_t* slot_pos = nullptr;// [T*k]      position of each slot (-1: invalid id)
  int32_t* pos_tok = nullptr; // [P]        token of each position
  int32_t* active = nullptr;  // [NE]       experts with tokens, routed then shared
  int32_t* n_active = nullptr;// [2]        active experts, token tiles in all
  int32_t* tile_prefix = nullptr; // [NE+1] token tiles before each active expert
  int4* tile_info = nullptr;  // [tiles]    (expert, first position, tokens, 0) per token tile
  uint8_t* xg = nullptr;      // [P][H]     E4M3 codes of x, gathered by position
  uint8_t* xgs = nullptr;     // [P][H/32]
  uint8_t* hq = nullptr;      // [P][I]     E4M3 codes of h
  uint8_t* hs = nullptr;      // [P][I/32]  UE8M0 scale bytes of h
  float* o = nullptr;         // [P][H]     expert outputs per position
  float* logits = nullptr;    // [T][E]     router logits scratch
  float* rpart = nullptr;     // split-K router partial sums ([8][min(T,64)][E] or [4][T][E])
  uint16_t* w3 = nullptr;     // [3][E][H]  router weights as three bf16 parts
  int32_t* idx = nullptr;     // [T][k]     routing scratch (host entry point)
  float* w = nullptr;         // [T][k]
  uint16_t* x = nullptr;      // [T][H]     bf16 staging (host entry point)
  uint16_t* y = nullptr;      // [T][H]
  float* part = nullptr;      // [2][2*SMs][2][part_bn][128] split-partition partial tiles (up, down)
  int32_t* split_cnt = nullptr; // [2][16*SMs] split-partition counters (up, down), then ready
  int split_cnt_n = 0;        // entries of split_cnt and ready (zeroed by the segments kernel)
  int32_t* ready = nullptr;   // [NE]       gate/up units finished per token tile (small batches)
  int32_t* ready_done = nullptr; // [1]     gate/up CTAs finished (small batches)
  int32_t* unit_next = nullptr;  // [1]     down: units taken (small batches, whole units)
  int part_bn = 0;            // token-tile width the partial slots are sized for
  int32_t* prep_cnt = nullptr;// [32]       small-batch preparation counters (zero between launches)
  int32_t* comb_cnt = nullptr;// [64][H/128][4] fused-combine counters (zeroed by the segments)
  int comb_cnt_n = 0;
  int32_t* seg_cbase = nullptr; // [kSegCtas][E] large-batch segments: per-CTA counts, then bases
  int32_t* seg_counter = nullptr; // [1]    its last-arriver counter (zero between launches)
  int32_t* seg_routed = nullptr;  // [1]    its routed slot total
  int32_t* err = nullptr;     // [1]        device error word
  int e_lo = 0, e_hi = 1 << 30; // expert ids this layer computes (expert parallelism); others
                                // in [0, E) belong to other ranks and are skipped silently
  int32_t* err_host = nullptr;// pinned: the error word, then (host entry point) y of small batches
  void* base = nullptr;       // single allocation holding all of the above
  size_t bytes = 0;
};

struct MmaMaps;

constexpr int kSegCtas = 32;  // CTAs of the large-batch segments
// The tensor-core GEMM's split partition takes launches of fewer than this
// many units per CTA (one arrival counter per unit and row quadrant).  With
// more units the plain partition is as even, and cutting units costs more
// (partial tiles through L2): measured slower at 7 and 16 units per CTA.
constexpr int kSplitUnitsPerCta = 4;

struct Timer {
  const char* name = nullptr;
  double ms = 0.0;
  int64_t launches = 0;
};

}  // namespace moe

struct moe_layer {
  moe_config cfg;
  moe_weights w;
  int device = 0;
  int num_sms = 0;
  int path = 0;
  int scoring = 0;            // MOE_SCORING_SOFTMAX / MOE_SCORING_SIGMOID
  float routed_scale = 1.0f;  // routed weights are multiplied by it
  int act_format = 0;         // MOE_ACT_FP8 / MOE_ACT_FP4
  int out_rows = 0;           // y rows the pinned staging (ws.err_host) holds after the error word
  int shared_format = 0;      // MOE_SHARED_MXFP4 / MOE_SHARED_FP8_B32
  uint32_t wait_limit = 1u << 24;  // polls per bounded wait in the tensor-core GEMMs
  bool timing = false;
  moe::Workspace ws;
  moe::MmaMaps* maps = nullptr;  // TMA descriptors of the tensor-core path
  CUtensorMap router_map;        // the bf16 router parts, for the tensor-core router
  bool router_mma = false;
  moe::Timer timers[moe::kMaxTimed];
  int n_timers = 0;
  cudaEvent_t ev_pool[2 * 64] = {};
  int ev_used = 0;
  int ev_pending_timer[64] = {};
};

namespace moe {

// Launches a kernel as a programmatic dependent of the previous work in the
// stream: it may start while that work drains and waits in pdl_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Expert weight pointers for expert id e (routed 0..E-1, shared E..E+ns-1).
struct ExpertBank {
  const uint8_t *gc, *gs, *uc, *us, *dc, *ds;       // routed banks
  const uint8_t *sgc, *sgs, *suc, *sus, *sdc, *sds; // shared banks
  int E, H, I;
};

// --- launchers (return the launch's cudaError_t) ---------------------------
cudaError_t launch_quantize_act(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* s,
                                cudaStream_t st);
cudaError_t launch_segments(const int32_t* idx, int T, int k, int E, int n_shared, int bn,
                            const Workspace& ws, cudaStream_t st);
// The codes of x at every position of each token (slot_pos for the routed
// slots, S + s*T + t for the shared experts), computed once per token.
cudaError_t launch_quantize_scatter(const uint16_t* x, int T, int H, int k, int ns, const int32_t* slot_pos,
                                    uint8_t* xg, uint8_t* xgs, bool act4, cudaStream_t st);
// The FP4-activation variant's quantiser of x by token: q [T][H/2], s [T][H/32].
cudaError_t launch_quantize_act4(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* s,
                                 cudaStream_t st);
cudaError_t launch_router_logits(const uint16_t* x, int T, int H, int E, const float* W,
                                 const float* b, float* logits, int num_sms, cudaStream_t st);
int router_ksplit(int H);
constexpr int kRouterSplitMaxT = 64;
// Split-K partial sums part[ks][T][E] (ks = router_ksplit(H)) of the router
// logits for T <= kRouterSplitMaxT tokens, and, with xq non-null, the codes
// of x (xq [T][H] E4M3, or packed E2M1 when act4; xs [T][H/32]).
cudaError_t launch_router_tile(const uint16_t* x, int T, int H, int E, const float* W, float* part,
                               uint8_t* xq, uint8_t* xs, bool act4, cudaStream_t st);
// Whether launch_router_tile can also write the codes of x for this hidden size.
bool router_tile_quantises(int H);
cudaError_t launch_router_split(const uint16_t* x, int T, int H, int E, int k, const float* W,
                                const float* b, const Scoring& sg, float* part, float* logits_out,
                                int32_t* idx, float* w, cudaStream_t st);
cudaError_t launch_topk_sum(const float* part, int ksplit, const float* b, int T, int E, int k,
                            const Scoring& sg, float* logits_out, int32_t* idx, float* w,
                            cudaStream_t st);
int router_mma_ksplit(int H);
cudaError_t router_split_weights(const float* w, int E, int H, uint16_t* w3, cudaStream_t st);
bool router_map_weights(CUtensorMap* m, const uint16_t* w3, int E, int H);
cudaError_t launch_router_mma(const CUtensorMap& w3map, const uint16_t* x, int T, int E, int H,
                              float* part, int32_t* err, int num_sms, cudaStream_t st);
cudaError_t launch_topk(const float* logits, int T, int E, int k, const Scoring& sg, int32_t* idx,
                        float* w, cudaStream_t st);
cudaError_t launch_ffn_up_simt(const ExpertBank& bank, int T, int k, int n_shared,
                               const Workspace& ws, int num_sms, cudaStream_t st);
cudaError_t launch_ffn_down_simt(const ExpertBank& bank, int T, int k, int n_shared,
                                 const Workspace& ws, int num_sms, cudaStream_t st);
cudaError_t launch_combine(const Workspace& ws, int T, int H, int k, int n_shared,
                           const float* w, const uint16_t* residual, uint16_t* y,
                           cudaStream_t st, float* y_f32 = nullptr);
// y = bf16(sum of part[r], r = 0 .. R-1 in order) (+ residual), part [R][T][H] fp32.
cudaError_t launch_combine_parts(const float* part, int R, int T, int H, const uint16_t* residual, uint16_t* y,
                                 cudaStream_t st);
MmaMaps* mma_maps_create(const moe_config& c, const moe_weights& w, const Workspace& ws);
void mma_maps_destroy(MmaMaps* m);
int mma_tile_for_tokens(int T);
// The combine fused into the down GEMM (small batches).
struct CombineArgs {
  int T, k, ns;
  const float* w;           // [T][k]
  const uint16_t* residual; // [T][H] or null
  uint16_t* y;              // [T][H]
};
// dense_T (gate/up, T <= 64 tokens, bn >= T): the activations are the codes of
// all dense_T tokens, token-major (xq/xs), and each unit's epilogue reads its
// own tokens' columns; 0: the slot-ordered copy xg/xgs by position.  cmb (down,
// bn <= 64): the combine runs inside the down GEMM (needs T <= kPrepMaxTokens).
// act4: the FP4-activation variant (xg/xq/hq hold packed E2M1 codes).
// ns_tiles: token tiles of the shared experts (n_shared x ceil(T / bn)).
// wait_limit: polls after which a pipeline wait gives up (MOE_OPT_WAIT_LIMIT).
// early: with 64-token tiles, gate/up counts its finished units per token
// tile in ws.ready and down takes whole units dynamically, each waiting for
// its tile instead of for the whole gate/up launch (the small-batch path: the
// preparation kernel zeroed the counts; at most NE tiles).
cudaError_t launch_ffn_mma(const MmaMaps& mm, const ExpertBank& bk, int mode, int bn, int dense_T,
                           const Workspace& ws, int num_sms, cudaStream_t st,
                           const CombineArgs* cmb = nullptr, bool act4 = false, int ns_tiles = 0,
                           uint32_t wait_limit = 1u << 24, bool early = false);
// Re-encodes the shared experts' maps for MXFP4 or FP8 (32 x 32 block) weights.
bool mma_maps_set_shared_format(MmaMaps* m, const moe_config& c, const moe_weights& w, bool fp8);
// FP4 activations need H and I multiples of 256 (whole 128-byte chunks).
bool mma_act4_supported(const moe_config& c);
// Small batches (T <= kPrepMaxTokens): router + top-k (route) or the given
// routing, FP8 codes of x by token (xq/xs) and the segments, in one launch.
// parts_ready (route): launch_router_tile has already written the router's
// partial sums (ws.rpart) and the codes of x; this launch adds the partials,
// selects and builds the segments.
constexpr int kPrepMaxTokens = 64;
cudaError_t prepare_prep_kernel(int E, int H);
cudaError_t launch_prep(const uint16_t* x, int T, int H, int E, int k, int ns, int bn,
                        const float* W, const float* b, const Scoring& sg, float* logits_out,
                        int32_t* idx, float* w, bool route, bool act4, const Workspace& ws,
                        cudaStream_t st, bool parts_ready = false);
cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps, uint16_t* out,
                           cudaStream_t st);

}  // namespace moe

/*
 * moe_ffn.h -- C ABI of the GB300 (sm_103a) routed MXFP4 mixture-of-experts
 * FFN layer.
 *
 * The layer (DeepSeek-V4.1-Flash MoE block geometry: 384 routed experts plus
 * one shared expert, top-6, hidden 5120, expert intermediate 2304; FreeToken
 * issue #444, "Architecture delta vs deepseek_v4") computes, per token t with
 * bf16 input x[t]:
 *
 *   logits  l = W_r x + b                       (fp32)
 *   routing idx = top-k of l (value desc, index asc), w = softmax over them
 *   x^      = FP8 E4M3 per-32 with UE8M0 scale (dynamic activation scheme,
 *             FreeToken issue #444 "Is the quantization already supported")
 *   expert  o_e = Wd_e Q8( silu(Wg_e x^) * (Wu_e x^) )   (MXFP4 weights)
 *   y       = bf16( sum_shared o_s + sum_j w_j o_idx_j )  [+ residual]
 *
 * MXFP4 matrices use one canonical layout (packed E2M1 + one UE8M0 per 32,
 * FreeToken issue #444, janit's comment item 2 "Routed expert bytes per
 * token"): a matrix with N output rows and K inputs is
 *   codes  [N][K/2] bytes, row-major; element k of a row is the low nibble of
 *          byte k/2 when k is even and the high nibble when k is odd;
 *   scales [N][K/32] bytes, UE8M0 (value 2^(s-127)) for elements 32j..32j+31.
 * A bank of E experts stacks E such matrices contiguously.
 *
 * Conventions for every call:
 *  - Pointers named x, y, residual, logits, topk_* and the weight pointers are
 *    DEVICE pointers on the layer's device unless the name ends in _host.
 *  - bf16 tensors are passed as void* holding IEEE bfloat16 bit patterns,
 *    row-major [T][H].
 *  - Calls are asynchronous on the caller's CUDA stream (cudaStream_t passed
 *    as void*, NULL = legacy default stream).  Argument errors are returned
 *    synchronously and nothing is launched.  A launch failure returns
 *    MOE_ERR_CUDA and clears the CUDA error state.  Errors the kernels record
 *    on the device (an expert id out of range) are returned by moe_sync (and
 *    by moe_forward_host, which synchronises).
 *  - A layer must not be used from two streams at the same time: calls share
 *    the layer's workspace.
 *  - No call allocates device memory except moe_layer_create.
 *  - No call exits or aborts the process.
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* NULL pointer, bad size, T > max_tokens, ... */
  MOE_ERR_UNSUPPORTED = 2, /* shape outside the supported envelope        */
  MOE_ERR_OOM = 3,         /* workspace allocation failed                 */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed        */
  MOE_ERR_TIMEOUT = 5,     /* a bounded device wait gave up               */
  MOE_ERR_INTERNAL = 6     /* a device-side check failed (index range)    */
} moe_status;

/* One MXFP4 matrix or bank of matrices in the canonical layout above. */
typedef struct {
  const uint8_t* codes;
  const uint8_t* scales;
} moe_mx_mat;

/* Shapes.  hidden and inter: multiples of 128 (128..16384); n_experts 1..512;
 * top_k 1..8 and <= n_experts; n_shared 0..4; max_tokens 1..65536 bounds T
 * of every call and sizes the workspace.  Anything else returns
 * MOE_ERR_UNSUPPORTED. */
typedef struct {
  int32_t hidden;
  int32_t inter;
  int32_t n_experts;
  int32_t top_k;
  int32_t n_shared;
  int32_t max_tokens;
} moe_config;

/* Weights, all borrowed device pointers that must outlive the layer.
 * gate/up: banks of n_experts matrices with N = inter, K = hidden;
 * down: N = hidden, K = inter.  s_gate/s_up/s_down: the shared experts, same
 * shapes, n_shared of them (ignored when n_shared = 0).
 * router_w: fp32 [n_experts][hidden]; router_b: fp32 [n_experts] or NULL.
 * Code and scale pointers must be 32-byte aligned, router_w 16-byte aligned. */
typedef struct {
  moe_mx_mat gate, up, down;
  moe_mx_mat s_gate, s_up, s_down;
  const float* router_w;
  const float* router_b;
} moe_weights;

typedef struct moe_layer moe_layer;

/* Creates a layer on `device`: validates the shapes, allocates the workspace
 * for max_tokens (the only allocation the library makes) and builds any
 * derived layout.  On failure *out is NULL and nothing is left allocated. */
moe_status moe_layer_create(const moe_config* cfg, const moe_weights* w, int device,
                            moe_layer** out);

/* Synchronises the layer's device, frees its workspace and the handle.
 * NULL returns MOE_ERR_INVALID_ARG.  The handle must not be used afterwards. */
moe_status moe_destroy(moe_layer* layer);

/* The same call under the name that pairs with moe_layer_create. */
moe_status moe_layer_destroy(moe_layer* layer);

/* Router (ai.rs, "What remains is the reference rounding itself": the gate is
 * a switch over the top-6 scores; llama.cpp discussion #28766, "Correctness").
 *  x          bf16 [T][H]
 *  logits_in  fp32 [T][E] or NULL.  When given, the logits are not computed:
 *             selection and weights use these values (so two implementations
 *             given the same logits must select identically).
 *  logits_out fp32 [T][E] or NULL: receives the logits used.
 *  topk_idx   int32 [T][k]: expert ids by rank (larger logit first, equal
 *             logits by lower index, NaN ranks as -infinity).
 *  topk_w     fp32 [T][k]: softmax over the k selected logits (sums to 1).
 * T = 0 is a no-op. */
moe_status moe_route(moe_layer* layer, const void* x, int32_t T, const float* logits_in,
                     float* logits_out, int32_t* topk_idx, float* topk_w, void* stream);

/* Expert FFN and combine for T tokens routed by (topk_idx, topk_w):
 *  y[t] = bf16( sum_shared o_s + sum_j topk_w[t][j] * o_{topk_idx[t][j]} ),
 * summed in fixed order (shared experts, then j = 0..k-1); with a residual
 * (bf16 [T][H] or NULL) y[t] = bf16(residual[t] + y[t]).  y may alias
 * residual but not x.  Expert ids outside [0, n_experts) are skipped and
 * make the next moe_sync return MOE_ERR_INTERNAL.  A repeated id in one row is
 * computed once per slot.  x, y and residual must be 16-byte aligned.  T = 0
 * is a no-op. */
moe_status moe_forward(moe_layer* layer, const void* x, int32_t T, const int32_t* topk_idx,
                       const float* topk_w, const void* residual, void* y, void* stream);

/* One layer step on device buffers: moe_route followed by moe_forward, with
 * the same results as those two calls (bit for bit: the logits are the same
 * fixed-order fp32 sums).  For small batches the router, the top-k, the FP8
 * codes of x and the expert segments run as one launch.  The cost of a
 * decode step is the bytes of the experts it selects (FreeToken issue #444,
 * janit's comment item 1: rate = bandwidth / routed bytes per token).
 *  topk_idx, topk_w  int32/fp32 [T][k] or NULL: receive the routing;
 *  logits_out        fp32 [T][E] or NULL: receives the logits.
 * x, y and residual as for moe_forward (16-byte aligned, y may alias the
 * residual but not x).  T = 0 is a no-op. */
moe_status moe_step(moe_layer* layer, const void* x, int32_t T, const void* residual, void* y,
                    int32_t* topk_idx, float* topk_w, float* logits_out, void* stream);

/* moe_route followed by moe_forward, with x and y in HOST memory: copies x to
 * the device, runs the layer and copies y back, all on `stream`; returns
 * after y_host is written (the call synchronises the stream).  For full copy
 * speed x_host and y_host should be page-locked.  T <= max_tokens. */
moe_status moe_forward_host(moe_layer* layer, const void* x_host, int32_t T, void* y_host,
                            void* stream);

/* A stack of layers over one batch of T tokens, with x and y in HOST memory
 * (the 8-layer decode stack of the pages' workloads: layers run back to
 * back, a bf16 residual add between them).  Copies x to the device, then for
 * l = 0 .. n_layers - 1
 *     x_{l+1} = bf16( x_l + moe_step(layers[l], N(x_l)) )
 * where N(v) = bf16( v / sqrt(mean(v^2) + norm_eps) ) per token (moe_rmsnorm)
 * when norm_eps >= 0, and the identity when norm_eps < 0; then copies x_n to
 * y_host.  Returns after y_host is written (the call synchronises the
 * stream).  All layers must be on one device with one hidden size, and T at
 * most each one's max_tokens (MOE_ERR_INVALID_ARG otherwise); 1 <= n_layers
 * <= 64.  Runs entirely in the layers' own workspaces (no allocation); a
 * device error any layer recorded is returned, and cleared, as by moe_sync.
 * For full copy speed x_host and y_host should be page-locked. */
moe_status moe_stack_forward_host(moe_layer* const* layers, int32_t n_layers, const void* x_host,
                                  int32_t T, float norm_eps, void* y_host, void* stream);

/* Expert parallelism: the routed experts split over ranks (FreeToken issue
 * #444, "Other engines": the model served on several GB300s).  The scheme is
 * all-gather / partial / exchange: every rank routes the whole batch with the
 * full router, computes the share of y its experts (and, on one rank, the
 * shared experts) contribute, and the shares of each token are added on the
 * token's owner in rank order.
 *
 * moe_layer_create_range: a layer that computes routed experts
 * expert_begin .. expert_end - 1 only.  The routed banks in w hold those
 * experts only (expert e at index e - expert_begin); the router weights cover
 * all cfg->n_experts experts; the shared experts, if cfg->n_shared > 0, are
 * computed by this layer (give them to one rank only).  Slots routed to other
 * experts are skipped without an error.  Tensor-core path only:
 * MOE_ERR_UNSUPPORTED where the shapes have none, and MOE_OPT_PATH = 1 is
 * refused.  0 <= expert_begin < expert_end <= n_experts (MOE_ERR_INVALID_ARG
 * otherwise). */
moe_status moe_layer_create_range(const moe_config* cfg, const moe_weights* w, int device,
                                  int32_t expert_begin, int32_t expert_end, moe_layer** out);

/* The layer's share of y in fp32, not rounded and without a residual:
 *   y_partial[t] = sum_shared o_s + sum over slots j whose expert the layer
 *                  computes of topk_w[t][j] * o_{topk_idx[t][j]}
 * (shared experts first, then j = 0..k-1).  y_partial fp32 [T][H], 16-byte
 * aligned.  Other arguments as for moe_forward. */
moe_status moe_forward_partial(moe_layer* layer, const void* x, int32_t T, const int32_t* topk_idx,
                               const float* topk_w, float* y_partial, void* stream);

/* Adds the ranks' shares of a layer: y[t] = bf16( sum over r = 0 .. n_parts-1,
 * in that order, of partials[r][t] ), then with a residual (bf16 [T][H] or
 * NULL) y[t] = bf16(residual[t] + y[t]).  partials fp32 [n_parts][T][H]
 * (16-byte aligned), y bf16 [T][H]; H a multiple of 4.  No layer is needed. */
moe_status moe_combine_partials(const float* partials, int32_t n_parts, int32_t T, int32_t H,
                                const void* residual, void* y, void* stream);

/* The activation quantiser alone: q [T][H] E4M3 codes and s [T][H/32] UE8M0
 * bytes, by the rule: per block of 32, e = the smallest integer with
 * max|x| <= 448 * 2^e (e = 0 for an all-zero block, limited to [-127, 127]),
 * s = e + 127, q = E4M3(x / 2^e) rounded to nearest, ties to even, sign kept
 * for zero results.  Inputs must be finite. */
moe_status moe_quantize_act(moe_layer* layer, const void* x, int32_t T, uint8_t* q, uint8_t* s,
                            void* stream);

/* The FP4-activation variant's quantiser (MOE_OPT_ACT_FORMAT): q [T][H/2]
 * packed E2M1 codes (element 2i in the low nibble of byte i, as the weight
 * codes) and s [T][H/32] UE8M0 bytes, by the rule: per block of 32, e = the
 * smallest integer with max|x| <= 6 * 2^e (e = 0 for an all-zero block,
 * limited to [-127, 127]), s = e + 127, code = E2M1(x / 2^e) rounded to
 * nearest, ties to the even code, sign kept for zero results.  Inputs must be
 * finite; H a multiple of 256 (MOE_ERR_UNSUPPORTED otherwise); q 4-byte
 * aligned. */
moe_status moe_quantize_act4(moe_layer* layer, const void* x, int32_t T, uint8_t* q, uint8_t* s,
                             void* stream);

/* The expert segments the forward pass builds from topk_idx [T][k]:
 * offsets [E+1] (offsets[e] = number of slots routed to experts below e) and
 * perm [T*k], the slots s = t*k + j listed expert by expert, in increasing
 * slot order within an expert. */
moe_status moe_segments(moe_layer* layer, const int32_t* topk_idx, int32_t T, int32_t* offsets,
                        int32_t* perm, void* stream);

/* Row RMS normalisation used between the layers of a stack:
 * out[t] = bf16( x[t] / sqrt(mean(x[t]^2) + eps) ), computed in fp32.
 * out may alias x.  H a multiple of 8, at most 65536. */
moe_status moe_rmsnorm(const void* x, int32_t T, int32_t H, float eps, void* out, void* stream);

/* Router without any device allocation, for callers that cannot call
 * cudaMalloc: a runtime whose device memory pool is entirely reserved by its
 * own allocator, or a step that must not make a call which can synchronise
 * the device or fail for lack of memory.  The pages describe no such entry
 * point; it has no counterpart there.
 *
 * Same result, bit for bit, as moe_route(layer, x, T, NULL, NULL, topk_idx,
 * topk_w, stream) on a layer with these shapes, router weights and the
 * default scoring (softmax, scale 1): the same split-K kernels, partial sums
 * added in the same fixed order.  No layer handle is needed: the partial
 * sums go to a fixed array of 8 * MOE_ROUTE_STATIC_MAX_TOKENS * 512 floats
 * (1 MiB) built into the library, which every GPU that loads the library
 * holds until the process exits.  T above MOE_ROUTE_STATIC_MAX_TOKENS returns
 * MOE_ERR_UNSUPPORTED; H must be a multiple of 128 (at most 16384),
 * E <= 512, 1 <= k <= min(8, E) (MOE_ERR_INVALID_ARG otherwise); x and
 * router_w 16-byte aligned; router_b fp32 [E] or NULL.
 * The first call on a device looks up the array's device address (set-up,
 * done once per device with that device current, and again when the
 * device's context has been replaced, e.g. after cudaDeviceReset); make that
 * first call before any stream capture.  All calls share the one array:
 * calls whose work overlaps on the GPU (two streams, or two host threads)
 * race on it and must be serialised by the caller.  No call allocates or
 * frees memory. */
#define MOE_ROUTE_STATIC_MAX_TOKENS 64
moe_status moe_route_static(const void* x, int32_t T, int32_t H, int32_t E, int32_t k,
                            const float* router_w, const float* router_b, int32_t* topk_idx,
                            float* topk_w, void* stream);

/* Waits for the stream and reports any device error the layer's kernels
 * recorded (MOE_ERR_INTERNAL / MOE_ERR_TIMEOUT) or CUDA reported; clears the
 * layer's recorded error. */
moe_status moe_sync(moe_layer* layer, void* stream);

/* Options (moe_set_option):
 *  MOE_OPT_PATH    0 = automatic (the tensor-core kernels when the build
 *                  has them), 1 = always the SIMT streaming kernels, 2 =
 *                  always the tensor-core kernels (MOE_ERR_UNSUPPORTED if
 *                  the build has none).
 *  MOE_OPT_TIMING  1 = record CUDA events around each kernel the layer
 *                  launches (read with moe_get_kernel_times), 0 = off.
 *  MOE_OPT_SCORING how the routed weights follow from the logits:
 *                  MOE_SCORING_SOFTMAX (default): logits include router_b,
 *                  selection on them, weights = softmax over the k selected;
 *                  MOE_SCORING_SIGMOID: logits l = router_w x without the
 *                  bias, s = sigmoid(l), selection on s + router_b (ties to
 *                  the lower index), weights = s / (sum of the k selected s).
 *                  The pages call the gate a switch over the top 6 (ai.rs,
 *                  "What remains is the reference rounding itself") without
 *                  naming the score; softmax is this library's reading, sigmoid
 *                  with a selection-only bias is the DeepSeek-V3-style variant.
 *                  sigmoid is computed by a fixed sequence of fp32 operations
 *                  (no library exp) so that selection is reproducible bit for
 *                  bit; logits_in / logits_out of moe_route are then unbiased.
 *  MOE_OPT_ROUTED_SCALE  routed weights are multiplied by this factor (the
 *                  shared experts keep weight 1): value = the IEEE-754 bits
 *                  of a positive finite float in the low 32 bits; default 1.
 *  MOE_OPT_ACT_FORMAT  MOE_ACT_FP8 (default): x and h quantised to E4M3 per
 *                  32, the checkpoint's dynamic scheme; MOE_ACT_FP4: both as
 *                  E2M1 per 32 (moe_quantize_act4's rule) and the expert
 *                  GEMMs on the FP4 x FP4 tensor-core kind -- a different,
 *                  noisier layer (the pages measure FP4 blocks of 32 losing
 *                  far more than FP8: ai.rs, "What remains is the reference
 *                  rounding itself", the table of round-trip errors), kept as
 *                  an option for compute-bound batches.  Tensor-core path
 *                  only: MOE_ERR_UNSUPPORTED when H or I is not a multiple of
 *                  256 or the layer has no tensor-core path; MOE_OPT_PATH = 1
 *                  (SIMT) is refused while it is set.
 *  MOE_OPT_SHARED_FORMAT  how the shared experts' weights (s_gate, s_up, s_down)
 *                  are stored: MOE_SHARED_MXFP4 (default) as the routed bank;
 *                  MOE_SHARED_FP8_B32: codes [n_shared][N][K] E4M3 (one byte per
 *                  element, the two NaN codes not allowed) and scales
 *                  [n_shared][N/32][K/32] UE8M0, one per block of 32 rows x 32
 *                  inputs -- the checkpoint's scheme for its FP8 dense layers
 *                  (FreeToken issue #444, "Is the quantization already
 *                  supported": weight_block_size [32, 32], scale_fmt ue8m0; ai.rs,
 *                  "The defect that never raised an error": the fp8 scale block
 *                  is 32 x 32).  The pointers given at create are read in this
 *                  format from the next call on (their sizes must match it).
 *                  Tensor-core path with FP8 activations only: MOE_ERR_UNSUPPORTED
 *                  without shared experts, with MOE_OPT_PATH = 1 or with FP4
 *                  activations (and those are refused while it is set).
 *  MOE_OPT_WAIT_LIMIT  how many times a wait inside the tensor-core expert
 *                  GEMMs polls its barrier before it gives up (default 2^24,
 *                  far longer than any copy or MMA takes); 0..2^31-1.  A wait
 *                  that gives up sets the layer's error word (moe_sync then
 *                  returns MOE_ERR_TIMEOUT), lets the copies and MMAs it had
 *                  issued finish, frees its tensor memory and ends the kernel;
 *                  that call's y is undefined and the next call starts clean.
 *                  0 makes every such wait give up at once: a test of that
 *                  error path without hanging or faulting the GPU.
 * moe_route_static always uses softmax scoring with scale 1.             */
enum { MOE_OPT_PATH = 1, MOE_OPT_TIMING = 2, MOE_OPT_SCORING = 3, MOE_OPT_ROUTED_SCALE = 4,
       MOE_OPT_ACT_FORMAT = 5, MOE_OPT_SHARED_FORMAT = 6, MOE_OPT_WAIT_LIMIT = 7 };
enum { MOE_SCORING_SOFTMAX = 0, MOE_SCORING_SIGMOID = 1 };
enum { MOE_ACT_FP8 = 0, MOE_ACT_FP4 = 1 };
enum { MOE_SHARED_MXFP4 = 0, MOE_SHARED_FP8_B32 = 1 };
moe_status moe_set_option(moe_layer* layer, int32_t option, int64_t value);

/* Per-kernel timing gathered while MOE_OPT_TIMING is on (synchronises the
 * layer's device).  Fills up to `cap` entries: names[i] points to a static
 * string, ms[i] is the summed event time and launches[i] the count.  Stores
 * the number of kernels in *n, then resets the counters. */
moe_status moe_get_kernel_times(moe_layer* layer, const char** names, double* ms,
                                int64_t* launches, int32_t cap, int32_t* n);

const char* moe_status_string(moe_status s);
int32_t moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H */

// Host side of the grouped block-scaled expert GEMM: tensor maps of the
// weight banks and activations, and the launch of the kernel of
// ffn_mma_kernel.cuh for a layer's shapes and activation format.
#define MOE_FFN_MMA_INSTANTIATE launch_ffn_mma_fp8
#define MOE_FFN_MMA_A4 0
#include "ffn_mma_kernel.cuh"

namespace moe {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    cudaGetLastError();
  }
  return fn;
}

// 3-D view {128-element chunk, row, chunk index} of a row-major [rows][K]
// matrix; a box is {128, box_rows, ch}: box_rows rows of ch consecutive
// chunks, stored in shared memory chunk-major (one swizzled tile per chunk).
// fp4: packed E2M1, expanded to one byte per element in shared memory.
bool map_3d(CUtensorMap* m, bool fp4, const void* base, uint64_t K, uint64_t rows,
            uint32_t box_rows, uint32_t ch) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !base) return false;
  const uint64_t row_bytes = fp4 ? K / 2 : K, chunk_bytes = fp4 ? 64 : 128;
  cuuint64_t dims[3] = {128, rows, K / 128};
  cuuint64_t strides[2] = {row_bytes, chunk_bytes};
  cuuint32_t box[3] = {128, box_rows, ch};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int chunks_per_stage(int K, bool allow3) {
  if (allow3 && K % 384 == 0) return 3;
  return K % 256 == 0 ? 2 : 1;
}

// gate and up banks as one 4-D tensor {128-element chunk, row, chunk index,
// matrix}: the matrix stride is the distance between the two banks, so one
// box {128, 128, ch, 2} loads the same rows of both.  Needs the distance to be
// a multiple of 32 bytes; *swap tells that the up bank comes first.
// fmt: how the banks' bytes are read -- kExpand: packed E2M1 expanded to a
// byte per element (128-element chunks); kPacked: the packed bytes as they are
// (FP4-activation variant: 128-byte chunks of 256 elements, for kind::mxf4);
// kBytes: one byte per element already (FP8 shared expert).
enum { kExpand = 0, kPacked = 1, kBytes = 2 };
bool map_4d_pair(CUtensorMap* m, const void* gate, const void* up, uint64_t K, uint64_t rows,
                 uint32_t ch, int* swap, int fmt = kExpand) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !gate || !up) return false;
  const uintptr_t g = (uintptr_t)gate, u = (uintptr_t)up;
  const uintptr_t lo = g < u ? g : u, dist = g < u ? u - g : g - u;
  if (dist == 0 || dist % 32 != 0 || dist >= (1ull << 40)) return false;
  *swap = u < g;
  cuuint64_t dims[4] = {128, rows, K / (fmt == kPacked ? 256 : 128), 2};
  cuuint64_t strides[3] = {fmt == kBytes ? K : K / 2, fmt == kExpand ? 64u : 128u, (cuuint64_t)dist};
  cuuint32_t box[4] = {128, 128, ch, 2};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, fmt == kExpand ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
             reinterpret_cast<void*>(lo), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Tensor maps of one activation format: weights (FP8 activations: FP4 codes
// expanded to a byte each; FP4 activations: packed bytes) and activations.
struct FormatMaps {
  CUtensorMap gate, up, down, s_gate, s_up, s_down;
  CUtensorMap gu_pair, s_gu_pair;  // gate + up as one 4-D tensor (when possible)
  int merged[2], swap_gu[2];
  CUtensorMap xg[3], hq[3];  // per token tile width: 16, 64, 112
  CUtensorMap xq[4];         // dense gate/up: the token-major codes, 16, 32, 48 or 64 rows per copy
  int ch_up, ch_down;
  bool ok;
  bool shared_fp8;  // the shared maps read FP8 (32 x 32 block) weights
};

struct MmaMaps {
  FormatMaps f[2];  // [0] FP8 activations, [1] FP4 activations (f[1].ok: shapes allow it)
};

static int bn_index(int bn) { return bn == 16 ? 0 : (bn == 64 ? 1 : 2); }

// Token tile width: 16 up to 16 tokens, 64 below 512 tokens (up to 64 tokens
// every expert's slots fit one tile, so its weights stream once), else 112 —
// the widest N for which the gate/up kernel's two accumulators fit TMEM twice
// (2 x 2 x 112 columns + the stages' scale factors <= 512), so the epilogue of
// one unit overlaps the MMAs of the next.
int mma_tile_for_tokens(int T) { return T <= 16 ? 16 : (T < 512 ? 64 : 112); }

// a4: packed operands (the FP4-activation variant): a chunk is 128 bytes of
// a row, 256 elements, one per stage; rows of K elements are K/2 bytes for
// weights and activations alike.
static bool format_maps(FormatMaps* m, bool a4, const moe_config& c, const moe_weights& w, const Workspace& ws) {
  // the routed banks hold the layer's own experts (all E, or its range under
  // expert parallelism)
  const uint64_t H = c.hidden, I = c.inter, ns = c.n_shared;
  const uint64_t E = (uint64_t)(ws.e_hi < c.n_experts ? ws.e_hi : c.n_experts) - (uint64_t)ws.e_lo;
  const uint64_t P = (uint64_t)c.max_tokens * (c.top_k + c.n_shared);
  m->shared_fp8 = false;
  m->ch_up = a4 ? 1 : chunks_per_stage((int)H, false);
  m->ch_down = a4 ? 1 : chunks_per_stage((int)I, true);
  // weights: a4 views [rows][K/2] bytes as 128-byte chunks; else the 4-bit expansion
  auto wmap = [&](CUtensorMap* t, const void* codes, uint64_t K, uint64_t rows, int ch) {
    return a4 ? map_3d(t, false, codes, K / 2, rows, 128, ch) : map_3d(t, true, codes, K, rows, 128, ch);
  };
  bool ok = wmap(&m->gate, w.gate.codes, H, E * I, m->ch_up) && wmap(&m->up, w.up.codes, H, E * I, m->ch_up) &&
            wmap(&m->down, w.down.codes, I, E * H, m->ch_down);
  if (ok && ns > 0)
    ok = wmap(&m->s_gate, w.s_gate.codes, H, ns * I, m->ch_up) && wmap(&m->s_up, w.s_up.codes, H, ns * I, m->ch_up) &&
         wmap(&m->s_down, w.s_down.codes, I, ns * H, m->ch_down);
  m->merged[0] = m->merged[1] = 0;
  m->swap_gu[0] = m->swap_gu[1] = 0;
  if (ok) {
    m->merged[0] = map_4d_pair(&m->gu_pair, w.gate.codes, w.up.codes, H, E * I, m->ch_up, &m->swap_gu[0],
                               a4 ? kPacked : kExpand);
    if (ns > 0)
      m->merged[1] = map_4d_pair(&m->s_gu_pair, w.s_gate.codes, w.s_up.codes, H, ns * I, m->ch_up,
                                 &m->swap_gu[1], a4 ? kPacked : kExpand);
  }
  const uint32_t bns[3] = {16, 64, 112};
  const uint64_t xk = a4 ? H / 2 : H, hk = a4 ? I / 2 : I;  // activation row bytes
  for (int i = 0; ok && i < 3; ++i)
    ok = map_3d(&m->xg[i], false, ws.xg, xk, P, bns[i], m->ch_up) &&
         map_3d(&m->hq[i], false, ws.hq, hk, P, bns[i], m->ch_down);
  const uint64_t T = (uint64_t)c.max_tokens;
  for (int i = 0; ok && i < 4; ++i) ok = map_3d(&m->xq[i], false, ws.xq, xk, T, 16 * (i + 1), m->ch_up);
  m->ok = ok;
  return ok;
}

bool mma_act4_supported(const moe_config& c) { return c.hidden % 256 == 0 && c.inter % 256 == 0; }

// The FP8-activation maps of the shared experts for their weight format: MXFP4
// (expanded, as the routed bank) or FP8 with 32 x 32 blocks (codes read as bytes).
bool mma_maps_set_shared_format(MmaMaps* mm, const moe_config& c, const moe_weights& w, bool fp8) {
  FormatMaps* m = &mm->f[0];
  const uint64_t H = c.hidden, I = c.inter, ns = c.n_shared;
  if (ns == 0) return false;
  bool ok = map_3d(&m->s_gate, !fp8, w.s_gate.codes, H, ns * I, 128, m->ch_up) &&
            map_3d(&m->s_up, !fp8, w.s_up.codes, H, ns * I, 128, m->ch_up) &&
            map_3d(&m->s_down, !fp8, w.s_down.codes, I, ns * H, 128, m->ch_down);
  if (ok)
    m->merged[1] = map_4d_pair(&m->s_gu_pair, w.s_gate.codes, w.s_up.codes, H, ns * I, m->ch_up, &m->swap_gu[1],
                               fp8 ? kBytes : kExpand);
  m->shared_fp8 = ok && fp8;
  return ok;
}

MmaMaps* mma_maps_create(const moe_config& c, const moe_weights& w, const Workspace& ws) {
  MmaMaps* m = new MmaMaps();
  if (!format_maps(&m->f[0], false, c, w, ws)) {
    delete m;
    return nullptr;
  }
  m->f[1].ok = false;
  if (mma_act4_supported(c)) format_maps(&m->f[1], true, c, w, ws);
  return m;
}

void mma_maps_destroy(MmaMaps* m) { delete m; }

cudaError_t launch_ffn_mma(const MmaMaps& maps, const ExpertBank& bk, int mode, int bn, int dense_T,
                           const Workspace& ws, int num_sms, cudaStream_t st, const CombineArgs* cmb, bool act4,
                           int ns_tiles, uint32_t wait_limit, bool early) {
  const FormatMaps& mm = maps.f[act4 ? 1 : 0];
  if (!mm.ok) return cudaErrorInvalidValue;
  MmaParams p;
  memset(&p, 0, sizeof(p));
  p.shared_fp8 = mm.shared_fp8 ? 1 : 0;
  p.ns_tiles = ns_tiles;
  p.wait_limit = wait_limit;
  const int bi = bn_index(bn);
  int ch;
  if (mode == kModeUp) {
    p.a_routed[0] = mm.merged[0] ? mm.gu_pair : mm.gate;
    p.a_routed[1] = mm.up;
    p.a_shared[0] = mm.merged[1] ? mm.s_gu_pair : mm.s_gate;
    p.a_shared[1] = mm.s_up;
    for (int i = 0; i < 2; ++i) {
      p.merged[i] = mm.merged[i];
      p.swap_gu[i] = mm.swap_gu[i];
    }
    p.b = mm.xg[bi];
    p.b16 = mm.xg[0];
    p.b64 = mm.xg[1];
    p.b_ragged = bn >= 64;
    p.b_rows = bn;
    p.sa_routed[0] = bk.gs;
    p.sa_routed[1] = bk.us;
    p.sa_shared[0] = bk.sgs;
    p.sa_shared[1] = bk.sus;
    p.sb = ws.xgs;
    if (dense_T > 0) {
      // every token's codes (token-major xq / xs), T rounded up to 16 rows per copy
      const int r16 = (dense_T + 15) / 16;
      if (r16 > 4 || 16 * r16 > bn) return cudaErrorInvalidValue;
      p.dense = 1;
      p.T = dense_T;
      p.b = mm.xq[r16 - 1];
      p.b_rows = 16 * r16;
      p.wait_tiles = 1;  // launched right after the preparation kernel
      p.pos_tok = ws.pos_tok;
      p.sb = ws.xs;
    }
    p.K = bk.H;
    p.rows = bk.I;
    p.out_cols = bk.I;
    ch = mm.ch_up;
  } else {
    p.a_routed[0] = mm.down;
    p.a_shared[0] = mm.s_down;
    p.b = mm.hq[bi];
    p.b_rows = bn;  // the ragged copies measured slower for down (442 -> 455 us at 256 tokens)
    p.sa_routed[0] = bk.ds;
    p.sa_shared[0] = bk.sds;
    p.sb = ws.hs;
    p.K = bk.I;
    p.rows = bk.H;
    p.out_cols = bk.H;
    ch = mm.ch_down;
  }
  p.E = bk.E;
  p.e_lo = ws.e_lo;
  p.n_active = ws.n_active;
  p.tile_prefix = ws.tile_prefix;
  p.tile_info = ws.tile_info;
  p.hq = ws.hq;
  p.hs = ws.hs;
  p.o = ws.o;
  const size_t part_n = (size_t)2 * num_sms * 2 * ws.part_bn * 128, cnt_n = (size_t)4 * kSplitUnitsPerCta * num_sms;
  p.part = ws.part + (mode == kModeUp ? 0 : part_n);
  p.cnt = ws.split_cnt + (mode == kModeUp ? 0 : cnt_n);
  p.split_ok = bn <= ws.part_bn && ws.split_cnt_n >= (int)(2 * cnt_n);
  if (early && bn == 64) {  // the EARLY kernel variant (see launch_bn)
    p.ready = ws.ready;
    p.ready_need = (int)(bk.I / 128) * 4;
    p.ready_done = ws.ready_done;
    p.unit_next = ws.unit_next;
    p.down_mt = (int)(bk.H / 128);
  }
  p.err = ws.err;
  if (mode == kModeDown && cmb && bn <= 64) {
    p.fuse_combine = 1;
    p.shared_first = 1;
    p.T = cmb->T;
    p.k = cmb->k;
    p.ns = cmb->ns;
    p.slot_pos = ws.slot_pos;
    p.pos_tok = ws.pos_tok;
    p.w = cmb->w;
    p.res = cmb->residual;
    p.y = cmb->y;
    p.comb_cnt = ws.comb_cnt;
  }
  return act4 ? launch_ffn_mma_fp4(p, mode, bn, ch, num_sms, st)
              : launch_ffn_mma_fp8(p, mode, bn, ch, num_sms, st);
}

}  // namespace moe

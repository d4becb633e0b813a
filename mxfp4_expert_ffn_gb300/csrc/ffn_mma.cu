// Grouped block-scaled expert GEMM on the 5th-generation tensor cores.
//
// D[w_row][token] = sum_k E2M1(W)[w_row][k] * 2^(sw-127) * E4M3(x)[token][k] * 2^(sx-127)
// with tcgen05.mma kind::mxf8f6f4 (A = weights in MXFP4, B = activations in
// FP8 E4M3, one UE8M0 scale per 32 along K for both), fp32 accumulators in
// TMEM.  The checkpoint's routed experts are FP4 with UE8M0 block scales and
// its activations are quantised dynamically to FP8 (FreeToken issue #444, "Is
// the quantization already supported"; janit's comment item 2).
//
// One persistent CTA per SM, ten warps:
//   warp 0      TMA producer: weight tiles through the 4-bit-unpacking tensor
//               map type (packed in HBM, one byte per element in shared memory,
//               as the f8f6f4 MMA reads them), activation tiles by position;
//   warp 1      MMA issuer and TMEM owner;
//   warps 2..5  epilogue (one TMEM lane quadrant each);
//   warps 6..9  scale-factor writers: per stage they copy the UE8M0 bytes of
//               the weight rows and tokens into TMEM (tcgen05.st), row r at
//               lane r / column r/32, k-block j in byte j.
// Work unit = (active expert, tile of weight rows, tile of BN tokens); for
// gate/up a tile holds 64 gate rows and the same 64 up rows (M = 128), so the
// epilogue has g and u of 64 intermediate rows and writes h = silu(g) * u as
// FP8 per 32 rows; for down a tile is 128 rows of the hidden dimension and
// the epilogue writes fp32 expert outputs per position.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace moe {

enum { kModeUp = 0, kModeDown = 1 };

struct MmaParams {
  CUtensorMap a_routed[2];   // up mode: gate, up banks; down mode: down bank in [0]
  CUtensorMap a_shared[2];
  CUtensorMap b;             // activations by position, [P][K] E4M3
  const uint8_t* sa_routed[2];
  const uint8_t* sa_shared[2];
  const uint8_t* sb;         // activation scales by position, [P][K/32]
  int E, K, rows;            // rows per expert of the weight matrices (I up, H down)
  int out_cols;              // I (h row length) in up mode, H in down mode
  const int32_t* active;
  const int32_t* n_active;
  const int32_t* off;
  const int32_t* cnt;
  const int32_t* tile_prefix;
  uint8_t* hq;
  uint8_t* hs;
  float* o;
  int32_t* err;
};

namespace {

using namespace sm100;

constexpr int kThreadsMma = 320;
constexpr uint32_t kWaitLimit = 1u << 24;

template <int BN>
struct Cfg {
  static constexpr int kStages = BN >= 128 ? 5 : (BN >= 64 ? 7 : 10);
  static constexpr int kATile = 16384;         // 128 rows x 128 bytes
  static constexpr int kBTile = BN * 128;
  static constexpr int kStageBytes = kATile + kBTile;
  static constexpr int kUbufStride = BN + 1;  // floats per u row (padded)
  static constexpr int kUbufBytes = 2 * 32 * kUbufStride * 4;
  static constexpr int kSfCols = 8;           // per stage: 4 A columns, 4 B columns
  static constexpr int kTmemCols = 2 * BN + kStages * kSfCols;
  static constexpr int kTmemAlloc = kTmemCols <= 32 ? 32 : kTmemCols <= 64 ? 64 : kTmemCols <= 128 ? 128 : kTmemCols <= 256 ? 256 : 512;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kUbufBytes;
  static_assert(kTmemCols <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct Unit {
  int e, p0, n0, m_tile, row0;
};

// Unit u -> (active expert, token tile, row tile); row tiles innermost so
// that consecutive units share the activation tile.
template <int BN>
__device__ __forceinline__ Unit decode_unit(const MmaParams& p, int u, int mt_per_expert,
                                            int row_tile, int n_act) {
  const int v = u / mt_per_expert;
  const int mt = u - v * mt_per_expert;
  int lo = 0, hi = n_act;  // largest a with tile_prefix[a] <= v
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.tile_prefix[mid] <= v) lo = mid;
    else hi = mid;
  }
  Unit r;
  r.e = p.active[lo];
  const int j = v - p.tile_prefix[lo];
  r.n0 = j * BN;
  r.p0 = p.off[r.e];
  r.m_tile = min(BN, p.cnt[r.e] - r.n0);
  r.row0 = mt * row_tile;
  return r;
}

template <int MODE, int BN>
__global__ void __launch_bounds__(kThreadsMma, 1) ffn_mma_kernel(const __grid_constant__ MmaParams p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* stage_base = smem;
  float* ubuf = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
  __shared__ __align__(8) uint64_t full_bar[C::kStages], sf_bar[C::kStages], empty_bar[C::kStages];
  __shared__ __align__(8) uint64_t accf_bar[2], acce_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_tile = MODE == kModeUp ? 64 : 128;
  const int mt_per_expert = p.rows / row_tile;
  const int n_act = *p.n_active;
  const int total = p.tile_prefix[n_act] * mt_per_expert;
  const int k_stages = p.K / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&sf_bar[s], 4);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], 4);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, C::kTmemAlloc);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t sf_col0 = 2 * BN;

  auto give_up = [&]() {
    atomicOr(p.err, kErrTimeout);
    *(volatile int*)&abort_flag = 1;
  };
  auto aborted = [&]() { return *(volatile int*)&abort_flag != 0; };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      uint32_t g = 0;
      int last_parity[C::kStages];
      for (int s = 0; s < C::kStages; ++s) last_parity[s] = -1;
      for (int u = blockIdx.x; u < total && !aborted(); u += gridDim.x) {
        const Unit un = decode_unit<BN>(p, u, mt_per_expert, row_tile, n_act);
        const bool sh = un.e >= p.E;
        const int erow = (sh ? un.e - p.E : un.e) * p.rows + un.row0;
        const CUtensorMap* a0 = sh ? &p.a_shared[0] : &p.a_routed[0];
        const CUtensorMap* a1 = sh ? &p.a_shared[1] : &p.a_routed[1];
        for (int s = 0; s < k_stages; ++s, ++g) {
          const int slot = g % C::kStages;
          const uint32_t ph = (g / C::kStages) & 1;
          if (!mbar_wait(&empty_bar[slot], ph ^ 1, kWaitLimit)) { give_up(); break; }
          uint8_t* sa = stage_base + slot * C::kStageBytes;
          uint8_t* sb = sa + C::kATile;
          mbar_expect_tx(&full_bar[slot], 8192 + BN * 128);
          if (MODE == kModeUp) {
            tma_load_2d(sa, a0, s * 128, erow, &full_bar[slot]);
            tma_load_2d(sa + 8192, a1, s * 128, erow, &full_bar[slot]);
          } else {
            tma_load_2d(sa, a0, s * 128, erow, &full_bar[slot]);
          }
          tma_load_2d(sb, &p.b, s * 128, un.p0 + un.n0, &full_bar[slot]);
          last_parity[slot] = (int)ph;
        }
      }
      // never leave with copies in flight: wait for the last load into each slot
      for (int s = 0; s < C::kStages; ++s)
        if (last_parity[s] >= 0) mbar_wait(&full_bar[s], (uint32_t)last_parity[s], kWaitLimit);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      uint32_t g = 0, it = 0;
      for (int u = blockIdx.x; u < total && !aborted(); u += gridDim.x, ++it) {
        const int buf = it & 1;
        if (!mbar_wait(&acce_bar[buf], ((it >> 1) & 1) ^ 1, kWaitLimit)) { give_up(); break; }
        fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        bool ok = true;
        for (int s = 0; s < k_stages; ++s, ++g) {
          const int slot = g % C::kStages;
          const uint32_t ph = (g / C::kStages) & 1;
          if (!mbar_wait(&full_bar[slot], ph, kWaitLimit) || !mbar_wait(&sf_bar[slot], ph, kWaitLimit)) {
            give_up();
            ok = false;
            break;
          }
          fence_after();
          const uint32_t sa = smem_u32(stage_base + slot * C::kStageBytes);
          const uint32_t sb = sa + C::kATile;
          const uint32_t sfa = tmem + sf_col0 + slot * C::kSfCols;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_mxf8f6f4(d_tmem, sw128_desc(sa + 32 * k), sw128_desc(sb + 32 * k),
                         idesc_e2m1_e4m3(128, BN, (uint32_t)k), sfa, sfa + 4, (s | k) ? 1u : 0u);
          mma_commit(&empty_bar[slot]);
        }
        if (!ok) break;
        mma_commit(&accf_bar[buf]);
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------- scale factors
    const int q = warp & 3;
    uint32_t g = 0;
    for (int u = blockIdx.x; u < total && !aborted(); u += gridDim.x) {
      const Unit un = decode_unit<BN>(p, u, mt_per_expert, row_tile, n_act);
      const bool sh = un.e >= p.E;
      const int r = 32 * q + lane;  // weight row of this lane within the tile
      const uint8_t* sa_row;
      if (MODE == kModeUp) {
        const uint8_t* base = sh ? p.sa_shared[r >= 64] : p.sa_routed[r >= 64];
        const int erow = (sh ? un.e - p.E : un.e) * p.rows + un.row0 + (r & 63);
        sa_row = base + (size_t)erow * (p.K / 32);
      } else {
        const uint8_t* base = sh ? p.sa_shared[0] : p.sa_routed[0];
        const int erow = (sh ? un.e - p.E : un.e) * p.rows + un.row0 + r;
        sa_row = base + (size_t)erow * (p.K / 32);
      }
      bool ok = true;
      for (int s = 0; s < k_stages; ++s, ++g) {
        const int slot = g % C::kStages;
        const uint32_t ph = (g / C::kStages) & 1;
        if (!mbar_wait(&empty_bar[slot], ph ^ 1, kWaitLimit)) { give_up(); ok = false; break; }
        fence_after();
        const uint32_t col = tmem + ((uint32_t)(32 * q) << 16) + sf_col0 + slot * C::kSfCols;
        tmem_st_x1(col + q, *reinterpret_cast<const uint32_t*>(sa_row + 4 * s));
#pragma unroll
        for (int c = 0; c < (BN + 31) / 32; ++c) {
          const int n = lane + 32 * c;
          uint32_t w = 0x7F7F7F7Fu;  // 1.0 for tokens outside the tile
          if (n < un.m_tile)
            w = *reinterpret_cast<const uint32_t*>(p.sb + (size_t)(un.p0 + un.n0 + n) * (p.K / 32) + 4 * s);
          tmem_st_x1(col + 4 + c, w);
        }
        tmem_st_wait();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_bar[slot]);
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    uint32_t it = 0;
    for (int u = blockIdx.x; u < total && !aborted(); u += gridDim.x, ++it) {
      const Unit un = decode_unit<BN>(p, u, mt_per_expert, row_tile, n_act);
      const int buf = it & 1;
      if (!mbar_wait(&accf_bar[buf], (it >> 1) & 1, kWaitLimit)) { give_up(); break; }
      fence_after();
      const uint32_t t_base = tmem + ((uint32_t)(32 * q) << 16) + buf * BN;
      if (MODE == kModeDown) {
        float* orow = p.o + (size_t)(un.p0 + un.n0) * p.out_cols + un.row0 + 32 * q + lane;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          uint32_t v[16];
          tmem_ld16(t_base + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c + j < un.m_tile) orow[(size_t)(c + j) * p.out_cols] = __uint_as_float(v[j]);
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[buf]);
      } else {
        float* ub = ubuf + (q & 1) * 32 * C::kUbufStride + lane * C::kUbufStride;
        if (q >= 2) {
          // u rows: park them in shared memory for the g warps
#pragma unroll 1
          for (int c = 0; c < BN; c += 16) {
            uint32_t v[16];
            tmem_ld16(t_base + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) ub[c + j] = __uint_as_float(v[j]);
          }
          fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce_bar[buf]);
          named_bar_sync(1, 128);
          named_bar_sync(1, 128);
        } else {
          named_bar_sync(1, 128);
          const int irow = un.row0 + 32 * q;  // first intermediate row of this warp
#pragma unroll 1
          for (int c = 0; c < BN; c += 16) {
            uint32_t v[16];
            tmem_ld16(t_base + c, v);
            tmem_ld_wait();
            if (c + 16 >= BN) {
              fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acce_bar[buf]);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (c + j >= un.m_tile) break;  // warp-uniform
              const float gg = __uint_as_float(v[j]);
              const float h = gg / (1.0f + expf(-gg)) * ub[c + j];
              const int ex = fp8_block_exponent(warp_max(fabsf(h)));
              const uint32_t code = e4m3x2(scale_pow2_neg(h, ex), 0.f) & 0xFFu;
              const size_t pos = (size_t)(un.p0 + un.n0 + c + j);
              p.hq[pos * p.out_cols + irow + lane] = (uint8_t)code;
              if (lane == 0) p.hs[pos * (p.out_cols / 32) + irow / 32] = (uint8_t)(ex + 127);
            }
          }
          named_bar_sync(1, 128);
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, C::kTmemAlloc);
  }
}

template <int MODE, int BN>
cudaError_t launch_one(const MmaParams& p, int num_sms, cudaStream_t st) {
  using C = Cfg<BN>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(ffn_mma_kernel<MODE, BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  ffn_mma_kernel<MODE, BN><<<num_sms, kThreadsMma, C::kSmemBytes, st>>>(p);
  return cudaGetLastError();
}

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

// Weight bank [rows][K] of packed E2M1, loaded as boxes of 128 elements x
// box_rows rows and expanded to one byte per element in shared memory.
bool map_fp4(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !base) return false;
  cuuint64_t dims[2] = {K, rows};
  cuuint64_t strides[1] = {K / 2};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activations by position [rows][K] of E4M3 bytes, boxes of 128 x box_rows.
bool map_u8(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !base) return false;
  cuuint64_t dims[2] = {K, rows};
  cuuint64_t strides[1] = {K};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

struct MmaMaps {
  CUtensorMap gate, up, down, s_gate, s_up, s_down;
  CUtensorMap xg[3], hq[3];  // per token tile width: 16, 64, 128
};

static int bn_index(int bn) { return bn == 16 ? 0 : (bn == 64 ? 1 : 2); }

int mma_tile_for_tokens(int T) { return T <= 64 ? 16 : (T < 512 ? 64 : 128); }

MmaMaps* mma_maps_create(const moe_config& c, const moe_weights& w, const Workspace& ws) {
  MmaMaps* m = new MmaMaps();
  const uint64_t H = c.hidden, I = c.inter, E = c.n_experts, ns = c.n_shared;
  const uint64_t P = (uint64_t)c.max_tokens * (c.top_k + c.n_shared);
  bool ok = map_fp4(&m->gate, w.gate.codes, H, E * I, 64) && map_fp4(&m->up, w.up.codes, H, E * I, 64) &&
            map_fp4(&m->down, w.down.codes, I, E * H, 128);
  if (ok && ns > 0)
    ok = map_fp4(&m->s_gate, w.s_gate.codes, H, ns * I, 64) &&
         map_fp4(&m->s_up, w.s_up.codes, H, ns * I, 64) &&
         map_fp4(&m->s_down, w.s_down.codes, I, ns * H, 128);
  const uint32_t bns[3] = {16, 64, 128};
  for (int i = 0; ok && i < 3; ++i)
    ok = map_u8(&m->xg[i], ws.xg, H, P, bns[i]) && map_u8(&m->hq[i], ws.hq, I, P, bns[i]);
  if (!ok) {
    delete m;
    return nullptr;
  }
  return m;
}

void mma_maps_destroy(MmaMaps* m) { delete m; }

cudaError_t launch_ffn_mma(const MmaMaps& mm, const ExpertBank& bk, int mode, int bn,
                           const Workspace& ws, int num_sms, cudaStream_t st) {
  MmaParams p;
  memset(&p, 0, sizeof(p));
  const int bi = bn_index(bn);
  if (mode == kModeUp) {
    p.a_routed[0] = mm.gate;
    p.a_routed[1] = mm.up;
    p.a_shared[0] = mm.s_gate;
    p.a_shared[1] = mm.s_up;
    p.b = mm.xg[bi];
    p.sa_routed[0] = bk.gs;
    p.sa_routed[1] = bk.us;
    p.sa_shared[0] = bk.sgs;
    p.sa_shared[1] = bk.sus;
    p.sb = ws.xgs;
    p.K = bk.H;
    p.rows = bk.I;
    p.out_cols = bk.I;
  } else {
    p.a_routed[0] = mm.down;
    p.a_shared[0] = mm.s_down;
    p.b = mm.hq[bi];
    p.sa_routed[0] = bk.ds;
    p.sa_shared[0] = bk.sds;
    p.sb = ws.hs;
    p.K = bk.I;
    p.rows = bk.H;
    p.out_cols = bk.H;
  }
  p.E = bk.E;
  p.active = ws.active;
  p.n_active = ws.n_active;
  p.off = ws.off;
  p.cnt = ws.cnt;
  p.tile_prefix = ws.tile_prefix;
  p.hq = ws.hq;
  p.hs = ws.hs;
  p.o = ws.o;
  p.err = ws.err;
  if (mode == kModeUp) {
    if (bn == 16) return launch_one<kModeUp, 16>(p, num_sms, st);
    if (bn == 64) return launch_one<kModeUp, 64>(p, num_sms, st);
    return launch_one<kModeUp, 128>(p, num_sms, st);
  }
  if (bn == 16) return launch_one<kModeDown, 16>(p, num_sms, st);
  if (bn == 64) return launch_one<kModeDown, 64>(p, num_sms, st);
  return launch_one<kModeDown, 128>(p, num_sms, st);
}

}  // namespace moe

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
//   warp 0      TMA producer.  Weights go through a 3-D view (128-element
//               chunk, row, chunk index) of the canonical [row][K] bank with
//               the 4-bit-unpacking tensor-map type, so that one TMA op moves
//               128 rows x CH chunks (16 KB of HBM for CH = 2) and lands as CH
//               standard 128-row swizzled tiles, one byte per element, as the
//               f8f6f4 MMA reads them.  Large ops matter: a TMA unit completes
//               a roughly fixed number of ops per second.
//   warp 1      MMA issuer and TMEM owner;
//   warps 2..5  epilogue (one TMEM lane quadrant each);
//   warps 6..9  scale-factor writers: per stage they copy the UE8M0 bytes of
//               the weight rows and tokens into TMEM (tcgen05.st): row r at
//               lane r, column r/32 of its group, k-block j in byte j.
// Work unit = (active expert, 128 weight rows, token tile of BN).  gate/up
// units hold 128 gate rows and the same 128 up rows in two accumulators, so
// every epilogue warp has g and u of its 32 intermediate rows: it writes
// h = silu(g) * u as FP8 with one scale per 32 rows.  down units write fp32
// expert outputs per position.
#pragma once

#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace moe {

enum { kModeUp = 0, kModeDown = 1 };

struct MmaParams {
  CUtensorMap a_routed[2];   // up mode: gate, up banks; down mode: down bank in [0]
  CUtensorMap a_shared[2];
  CUtensorMap b;             // activations by position, 3-D view of [P][K] E4M3
  CUtensorMap b16, b64;      // b_ragged: the same rows, 16 / 64 per copy
  const uint8_t* sa_routed[2];
  const uint8_t* sa_shared[2];
  const uint8_t* sb;         // activation scales by position, [P][K/32]
  int E, K, rows;            // rows per expert of the weight matrices (I up, H down)
  int e_lo;                  // the routed banks hold experts e_lo, e_lo + 1, ... (expert parallelism)
  int out_cols;              // I (h row length) in up mode, H in down mode
  const int32_t* n_active;   // [0] active experts, [1] token tiles in all
  const int32_t* tile_prefix;
  int wait_tiles;            // the tile table comes from the previous kernel itself
  const int4* tile_info;
  int n_stages;              // ring depth (runtime: fits the shared memory)
  int merged[2];             // up mode, routed / shared: gate and up load as one 4-D op
  int swap_gu[2];            // ... whose first matrix is the up bank
  uint8_t* hq;
  uint8_t* hs;
  float* o;
  float* part;               // split partition: fp32 partial tiles, 2 slots per CTA
  int32_t* cnt;              // split partition: pieces finished per (unit, row quadrant)
  int split_ok;              // part/cnt are large enough for this launch
  int dense;                 // up mode, T <= 64: B = the codes of all tokens (token-major), read by TMA
  int b_rows;                // activation rows one B copy brings (dense: T rounded up to 16; else BN)
  int b_ragged;              // gate/up tiles by position: a unit of up to 16 positions copies 16
                             // rows (b16), of up to 64 (112-token tiles) 64 rows (b64), else the
                             // tile's; each multiplies its rows rounded up to 16
  int fuse_combine;          // down mode, BN <= 64: the last writer of a token's rows combines them
  int T, k, ns;              // tokens (dense, fuse_combine), top-k, shared experts (fuse_combine)
  const int32_t* slot_pos;   // fuse_combine: position of slot t*k + j (-1: invalid id)
  const float* w;            // fuse_combine: combine weights [T][k]
  const uint16_t* res;       // fuse_combine: bf16 residual [T][H] or null
  uint16_t* y;               // fuse_combine: bf16 output [T][H]
  int32_t* comb_cnt;         // fuse_combine: writers finished per (token, 128-row tile, quadrant)
  const int32_t* pos_tok;    // dense, fuse_combine: token of each position
  int shared_fp8;            // shared experts in FP8 (E4M3, one scale per 32 x 32 block)
  uint32_t wait_limit;       // polls after which a pipeline wait gives up (then the error word)
  int ns_tiles;              // token tiles of the shared experts (the last ones of the table)
  int shared_first;          // process the shared experts' tiles first (fuse_combine: see the kernel)
  int32_t* err;
  int32_t* ready;            // small batches: gate/up units finished per token tile (gate/up counts;
                             // down waits per unit for its tile, not for the whole gate/up launch)
  int ready_need;            // down: the count that makes a tile final (gate/up units per tile x 4 warps)
  int32_t* ready_done;       // gate/up CTAs finished (each adds one as it leaves)
  int32_t* unit_next;        // down, whole units: the launch-wide counter of units taken
  int down_mt;               // 128-row tiles of the down matrix (H / 128): both kernels tell from
                             // the tile count whether down runs whole units (then the above apply)
};

namespace {

using namespace sm100;

constexpr int kThreadsMma = 352;  // 11 warps: TMA, MMA, 4 epilogue, 4 scale-factor, 2nd MMA
constexpr int kIssuer2Warp = 10;
// Polls for the waits that let copies and MMAs already issued complete before
// the CTA leaves (they always end: the hardware finishes what was issued).
constexpr uint32_t kDrainLimit = 1u << 24;
// Polls of a tile's gate/up count before down waits for the whole gate/up
// launch instead (always correct; the counts only let it start earlier).
constexpr uint32_t kReadyPolls = 1u << 16;
// Entries of the shared-memory queue that hands dynamically taken units from
// the producer to the other roles.  Writing entry i, the producer has waited
// for the MMAs of a stage of unit i - 1 - NS (or later), so the MMA issuer has
// taken unit i - 1 - NS, which means the epilogue (the last reader) has taken
// unit i - 3 - NS: with NS <= 6 no entry is overwritten before all have read it.
constexpr int kUq = 16;
constexpr int kSmemBudget = 227 * 1024 - 2048;

constexpr int pow2_cols(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }

constexpr int kMaxStages = 6;
static_assert(kUq >= kMaxStages + 4, "unit queue depth");

// A4: the FP4-activation variant (both operands packed E2M1, kind::mxf4):
// a 128-byte chunk of a row holds 256 K elements instead of 128, and its
// scales are two words (8 k-blocks) instead of one.
template <int MODE, int BN, int CH, bool A4 = false>
struct Cfg {
  static constexpr int kNA = MODE == kModeUp ? 2 : 1;     // weight matrices per unit
  static constexpr int kKC = A4 ? 256 : 128;              // K elements per 128-byte chunk
  static constexpr int kW = A4 ? 2 : 1;                   // scale words per row and chunk
  static constexpr int kATile = 128 * 128 * CH;           // one matrix, one stage
  static constexpr int kBTile = BN * 128 * CH;
  // MMA issue is split over two threads (see the kernel): gate/up one matrix
  // each; down one half of each stage's K steps each, into a second
  // accumulator that the epilogue adds in a fixed order (so every K step reads
  // the weight tile once).
  static constexpr bool kSplitK = MODE == kModeDown;
  // MMA width per tile from its token count (the 112-token tiles; narrower
  // tiles are mostly full or one instruction step wide)
  static constexpr bool kRagged = BN == 112;
  static constexpr int kAccCols = (MODE == kModeUp || kSplitK ? 2 : 1) * BN;  // g, u (up); o (down)
  static constexpr int kNAcc = (MODE == kModeUp && BN >= 128) ? 1 : 2;
  // 64-token gate/up: the activation tiles get a ring of their own (two
  // slots), so that three 64 KB weight stages still fit next to them; the
  // weight bytes in flight, not the activations (read from L2), set the pace.
  static constexpr bool kSepB = MODE == kModeUp && BN == 64 && !A4 && CH == 2;
  static constexpr int kBRing = kSepB ? 2 : 0;
  static constexpr int kStage = kNA * kATile + (kSepB ? 0 : kBTile);  // shared memory of one ring stage
  static constexpr int kStageCap0 = (kSmemBudget - 1024 - kBRing * kBTile) / kStage;
  static constexpr int kStageCap = kStageCap0 < kMaxStages ? kStageCap0 : kMaxStages;
  // Scale factors in TMEM, per stage: 4 columns per (weight matrix, chunk),
  // then per chunk the token scales (group of 32 tokens g at column g); with
  // the column split each half starts a 4-column group of its own (the MMA
  // is handed a 4-column-aligned scale address).
  static constexpr int kBCols = 4;  // token scale groups of 32 (BN <= 128)
  static constexpr int kSfCols = (kNA * 4 * CH + kBCols * CH) * kW;
  // A scales of (matrix m, chunk c, word w); B scales of (chunk c, word w, token group g)
  __host__ __device__ static constexpr int sfa_col(int m, int c, int w) { return ((m * CH + c) * kW + w) * 4; }
  __host__ __device__ static constexpr int sfb_col(int c, int w, int g) {
    return kNA * 4 * CH * kW + (c * kW + w) * kBCols + g;
  }
  // ring depth: what the shared memory holds, and what TMEM holds next to the accumulators
  static constexpr int kStageCapT = (512 - kNAcc * kAccCols) / kSfCols;
  static constexpr int kStages = kStageCap < kStageCapT ? kStageCap : kStageCapT;
  static constexpr int kTmemCols = kNAcc * kAccCols + kStages * kSfCols;
  static constexpr int kTmemAlloc = pow2_cols(kTmemCols);
  static_assert(kTmemCols <= 512, "TMEM budget");
};

// Pipeline geometry: as many stages as fit the shared memory (at most
// kMaxStages).  The bytes in flight per SM bound the bandwidth (about ten TMA
// ops in flight, a few microseconds each), so every byte of shared memory goes
// to the ring.
template <int MODE, int BN, int CH, bool A4>
void geometry(int K, int* n_stages, int* smem) {
  using C = Cfg<MODE, BN, CH, A4>;
  (void)K;
  *n_stages = C::kStages;
  *smem = 1024 + C::kStages * C::kStage + C::kBRing * C::kBTile;
}

struct Unit {
  int e, pos0, m_tile, row0;
};

// Unit u -> (token tile v, 128-row tile); row tiles innermost so consecutive
// units share the activation tile.  rot: the units start at tile rot of the
// table and wrap around (n_tiles tiles in all).
__device__ __forceinline__ int tile_of(int u, int mt_units, int rot, int n_tiles) {
  const int v = u / mt_units + rot;
  return v >= n_tiles ? v - n_tiles : v;
}
__device__ __forceinline__ Unit decode_unit(const MmaParams& p, int u, int mt_units, int rot, int n_tiles) {
  const int v = tile_of(u, mt_units, rot, n_tiles);
  const int4 t = __ldg(p.tile_info + v);
  const int r = u - (u / mt_units) * mt_units;
  return Unit{t.x, t.y, t.z, r * 128};
}

// Work partition.  Plain: whole units strided over the CTAs.  Split: when
// there are few units (a decode step), the units' K stages form one sequence
// that is cut into gridDim.x nearly equal contiguous ranges, so that every SM
// streams the same number of weight bytes.  A unit cut between CTAs is
// finished by the last of them to arrive, which adds the fp32 partial tiles in
// piece order (fixed, so results do not depend on arrival order).
struct Piece {
  int u, s0, s1;  // unit, stage range [s0, s1)
};

constexpr int kMaxPieces = 16;  // pieces per unit in the split partition
constexpr int kMaxTopK = 8, kMaxShared = 4;  // layer limits (moe_config)

// All arithmetic in 32 bits: split mode needs total < kSplitUnitsPerCta *
// gridDim.x (at most 64 stages a unit), so stage iterations times CTAs stay
// far below 2^32.
struct Sched {
  int ti, g, end;  // split: stage iterations in all, cursor, end of this CTA's range
  int total, ks, u;
  int cta, G;      // this CTA and the number of CTAs
  bool split;
  __device__ Sched(int total_, int ks_, int split_ok, int cta_, int G_)
      : total(total_), ks(ks_), cta(cta_), G(G_) {
    split = false;
    if (split_ok && total < kSplitUnitsPerCta * G) {
      ti = total * ks;
      const int split_max = (ti + G - 1) / G;
      const int plain_max = ((total + G - 1) / G) * ks;
      // worth it when the busiest CTA gets at least 5 % fewer stages, and
      // no unit is cut into more than kMaxPieces pieces
      split = ti >= G && split_max * 20 < plain_max * 19 && ks <= (kMaxPieces - 2) * (ti / G);
    }
    g = split ? begin(cta) : 0;
    end = split ? begin(cta + 1) : 0;
    u = cta;
  }
  __device__ int begin(int c) const { return (int)(((unsigned)c * (unsigned)ti) / G); }
  // the CTA whose range holds stage iteration it
  __device__ int owner(int it) const { return (int)(((unsigned)(it + 1) * G + ti - 1) / ti) - 1; }
  __device__ Piece next() {
    Piece pc{-1, 0, 0};
    if (!split) {
      if (u < total) pc = Piece{u, 0, ks};
      u += G;
      return pc;
    }
    if (g >= end) return pc;
    pc.u = g / ks;
    pc.s0 = g - pc.u * ks;
    pc.s1 = min(ks, pc.s0 + (end - g));
    g += pc.s1 - pc.s0;
    return pc;
  }
  // Unit uu is computed by CTAs first .. first + n - 1 (piece j by CTA first + j).
  __device__ void pieces(int uu, int& first, int& n) const {
    if (!split) {
      first = cta;
      n = 1;
      return;
    }
    first = owner(uu * ks);
    n = owner((uu + 1) * ks - 1) - first + 1;
  }
  // Partial slot of piece j: 2c for the first piece of CTA c's range, 2c + 1 for its last.
  __device__ int slot(int uu, int first, int j) const {
    return (j == 0 && begin(first) != uu * ks) ? 2 * first + 1 : 2 * (first + j);
  }
};

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            int32_t c2, int32_t c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// Small batches read every weight tile exactly once: their copies carry an L2
// evict-first policy, so that streaming the weights leaves the small reused
// data of the launches around them (activation codes, tile tables, h, the
// serial kernels' code) in L2.  (Where a tile is read by several token tiles
// the second read would then miss.)
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_4d_hint(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                 int32_t c2, int32_t c3, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                 int32_t c2, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// h = silu(g) * u = g / (1 + e^-g) * u with the SFU exponential and the fast
// divide: a few ulp from the correctly rounded form, far inside the FP8
// rounding of h that follows (one E4M3 step is 2^-3 relative).
__device__ __forceinline__ float swiglu(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            int32_t c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

template <int MODE, int BN, int CH, bool A4, bool EARLY>
__global__ void __launch_bounds__(kThreadsMma, 1) ffn_mma_kernel(const __grid_constant__ MmaParams p) {
  using C = Cfg<MODE, BN, CH, A4>;
  constexpr int NA = C::kNA;
  constexpr int NC = (BN + 31) / 32;  // 32-token groups of the B scale factors
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // full_bar[s]: stage s's copies have landed (the producer's expect-tx
  // arrival and the bytes of the weight and activation copies) and its scale
  // factors are in TMEM (one arrival per scale-factor warp): the MMA issuer
  // waits on this one barrier per stage.  Under load each barrier operation
  // costs ~0.1 us of shared-memory latency, so one wait instead of two or three
  // shortens the time a stage holds its slot.
  __shared__ __align__(8) uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t accf_bar[2], acce_bar[2], drain_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ uint32_t uq[kUq];  // (entry number + 1) << 16 | (unit + 1)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt_per_expert = p.rows / 128;
  const int k_stages = p.K / (C::kKC * CH);
  const int NS = p.n_stages;
  uint8_t* stage_base = smem;
  constexpr bool kSepB = C::kSepB;
  const int stage_bytes = C::kStage;
  uint8_t* bring_base = smem + NS * stage_bytes;  // kSepB: the B ring after the weight stages
  // Dense mode (gate/up for up to 64 tokens): B is the codes of all T tokens,
  // token-major as the preparation kernel wrote them, b_rows = T rounded up to
  // 16 rows by one TMA copy per stage; every expert's unit multiplies them all
  // (an MMA costs about the same at N = 16 and N = 64) and the epilogue reads
  // the accumulator columns of the unit's own tokens.  No copy of x per slot
  // is made and the expert's weights stream once.
  const bool dense = MODE == kModeUp && p.dense;
  const int BR = p.b_rows;  // activation rows per B tile (the MMA's N, except ragged tiles)
  // bytes a stage's copies bring: the weights packed (FP4: 64 bytes per
  // 128-element chunk row, unpacked into 128; A4: 128 bytes, stored as is),
  // and the activation rows (128 bytes per chunk row; the activation copy
  // lands on the stage's barrier too)
  const uint32_t tx_a = NA * 128 * (A4 ? 128 : 64) * CH;
  // Tiles by position (not dense) are often part-filled, so a unit copies
  // the smallest of 16, 64 or BN rows that holds its positions (one copy per
  // stage; its chunks then lie that many rows apart in shared memory) and
  // multiplies only its rows rounded up to 16 (less shared-memory traffic per
  // stage for the copies and the MMAs)
  const bool ragged_b = BN >= 64 && !dense && p.b_ragged;
  auto b_rows_of = [&](const Unit& un) {
    return !ragged_b ? BR : un.m_tile <= 16 ? 16 : (BN > 64 && un.m_tile <= 64) ? 64 : BR;
  };
  const uint32_t sf_col0 = C::kNAcc * C::kAccCols;

  if (threadIdx.x == 0) {
    // bring the tensor maps this CTA reads into the descriptor cache while
    // the previous kernel finishes
#pragma unroll
    for (int m = 0; m < NA; ++m) {
      prefetch_tensormap(&p.a_routed[m]);
      prefetch_tensormap(&p.a_shared[m]);
    }
    prefetch_tensormap(&p.b);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1 + 4);
      mbar_init(&empty_bar[s], 2);  // one commit per MMA-issuing thread
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 2);
      mbar_init(&acce_bar[b], 4);
      mbar_init(&drain_bar[b], 1);
    }
    for (int i = 0; i < kUq; ++i) uq[i] = 0u;
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, C::kTmemAlloc);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_slot;
  // Programmatic dependent launch.  Usually the tile table and the weights
  // were final before the previous kernel started, so they are read right
  // away and only the activations (and the outputs' readers) wait for the
  // previous kernel in pdl_wait() below; after the small-batch preparation
  // kernel the tile table is that kernel's own output, so everything waits.
  if (p.wait_tiles) pdl_wait();
  pdl_trigger();
  const int mt_units = mt_per_expert;
  const int total = p.n_active[1] * mt_units;
  // FP8 shared experts: their tiles close the table, so a unit's format follows
  // from its index (no tile-table load on the issuing thread)
  const int n_tiles = p.n_active[1];
  const int shared_tile0 = (!A4 && p.shared_fp8) ? n_tiles - p.ns_tiles : 0x7FFFFFFF;
  // With the combine fused into the down GEMM, whichever unit writes a token's
  // last output row does that token's combine.  The shared experts' tiles hold
  // every token, so they go first: the last writers are then routed units
  // spread over the launch, not the last few units holding all the tokens.
  const int rot = p.shared_first ? n_tiles - p.ns_tiles : 0;
  auto shared_fp8_unit = [&](int u) { return tile_of(u, mt_units, rot, n_tiles) >= shared_tile0; };
  const Sched sc0(total, k_stages, BN <= 64 && p.split_ok, (int)blockIdx.x, (int)gridDim.x);

  auto give_up = [&]() {
    atomicOr(p.err, kErrTimeout);
    *(volatile int*)&abort_flag = 1;
  };
  auto aborted = [&]() { return *(volatile int*)&abort_flag != 0; };
  // Down after a small batch's gate/up: the activations of a unit (h of its
  // token tile) are final once gate/up has counted every unit of that tile
  // (each epilogue warp counts its 32 rows of a unit after writing them), so
  // each role waits for its unit's tile rather than for the whole previous
  // launch.  h then reaches the tensor copies (async proxy) and the scale
  // loads.  A wait that runs out of polls falls back to the launch wait.
  // Only when down runs whole units (not the split partition of a decode
  // step, where the counting costs more than the earlier start brings); both
  // kernels decide from the same tile count.
  // The code exists only in the EARLY variant (small batches with 64-token
  // tiles): compiled into the others, even unused, it slowed them.
  const bool early_on =
      EARLY && p.ready != nullptr && n_tiles * p.down_mt >= kSplitUnitsPerCta * (int)gridDim.x;
  const bool early = MODE == kModeDown && early_on;
  auto wait_tile = [&](int u, bool& all) {
    if (all) return;
    // once every gate/up CTA has left, no later unit needs a look
    if (ld_acquire_gpu(p.ready_done) >= (int)gridDim.x) {
      fence_proxy_async_global();
      all = true;
      return;
    }
    const int32_t* r = p.ready + tile_of(u, mt_units, rot, n_tiles);
    const uint32_t lim = p.wait_limit < kReadyPolls ? p.wait_limit : kReadyPolls;
    for (uint32_t i = 0; i < lim; ++i) {
      if (ld_acquire_gpu(r) >= p.ready_need) {
        fence_proxy_async_global();
        return;
      }
      __nanosleep(64);
    }
    pdl_wait();
    all = true;
  };
  // Early down with whole units: CTAs that start while gate/up finishes
  // take more units.  The producer takes the next unit from a launch-wide
  // counter (one unit ahead, so the atomic's latency hides behind a unit's
  // copies) and hands each unit to the other roles through the queue; -1 ends
  // it.  Which CTA computes a unit changes nothing in the unit's arithmetic.
  // Each CTA's first unit is its own index; the counter hands out the rest.
  const bool dyn = early && !sc0.split && total < 0xFFFF;
  int dyn_cur = 0;
  auto uq_tag = [](uint32_t i) { return ((i & 0x7FFFu) + 1u) << 16; };
  auto next_producer = [&](Sched& sc, uint32_t& i) -> Piece {
    if (!dyn) return sc.next();
    const int u = dyn_cur < total ? dyn_cur : -1;
    if (u >= 0) dyn_cur = (int)gridDim.x + atomicAdd(p.unit_next, 1);
    *(volatile uint32_t*)&uq[i % kUq] = uq_tag(i) | (uint32_t)(u + 1);
    ++i;
    return u >= 0 ? Piece{u, 0, k_stages} : Piece{-1, 0, 0};
  };
  auto next_reader = [&](Sched& sc, uint32_t& i) -> Piece {
    if (!dyn) return sc.next();
    const uint32_t want = uq_tag(i);
    const volatile uint32_t* e = &uq[i % kUq];
    ++i;
    uint32_t v = *e, n = 0;
    while ((v & 0xFFFF0000u) != want) {
      if (++n >= p.wait_limit) {
        give_up();
        return Piece{-1, 0, 0};
      }
      v = *e;
    }
    const int u = (int)(v & 0xFFFFu) - 1;
    return u >= 0 ? Piece{u, 0, k_stages} : Piece{-1, 0, 0};
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      uint32_t g = 0;
      int last_parity[kMaxStages];
      int deferred_pos[kMaxStages], deferred_s[kMaxStages], n_deferred = 0;
      // dense mode runs after the preparation kernel and waited for it above;
      // early down waits per unit (wait_tile) before the unit's first B copy
      bool waited = dense || early, all_ready = false;
      // B copies issued before the previous kernel is waited for: as many as
      // there are slots to hold them
      const uint32_t defer_cap = kSepB ? 2u : (uint32_t)NS;
      // the activation tile of stage g, one op into the stage's own area or
      // the B ring's slot bs, landing on the stage's full barrier fs; dense:
      // rows 0.. of the token-major codes
      auto load_b = [&](int bs, int fs, int pos0, int st, int rows) {
        const int row = dense ? 0 : pos0;
        uint8_t* dst = kSepB ? bring_base + bs * C::kBTile : stage_base + fs * stage_bytes + NA * C::kATile;
        // the 16- and 64-row maps exist only for the ragged tiles (gate/up by position)
        const CUtensorMap* map = !ragged_b ? &p.b : rows == 16 ? &p.b16 : (BN > 64 && rows == 64) ? &p.b64 : &p.b;
        tma_load_3d(dst, map, 0, row, st * CH, &full_bar[fs]);
      };
      const uint64_t wpol = EARLY ? l2_evict_first_policy() : 0;
      int deferred_rows[kMaxStages];
#pragma unroll
      for (int s = 0; s < kMaxStages; ++s) last_parity[s] = -1;
      Sched sc = sc0;
      uint32_t qi = 0;
      dyn_cur = (int)blockIdx.x;
      for (Piece pc = next_producer(sc, qi); pc.u >= 0 && !aborted(); pc = next_producer(sc, qi)) {
        const Unit un = decode_unit(p, pc.u, mt_units, rot, n_tiles);
        const bool sh = un.e >= p.E;
        const int erow = (sh ? un.e - p.E : un.e - p.e_lo) * p.rows + un.row0;
        const int brows_u = b_rows_of(un);
        bool ok = true;
        const int s_end = pc.s1;
        for (int s = pc.s0; s < s_end; ++s, ++g) {
          const int slot = g % NS;
          const uint32_t ph = (g / NS) & 1;
          if (!waited && g >= defer_cap) {
            // ring full: wait for the previous kernel, then load the deferred activations
            pdl_wait();
            waited = true;
            for (int i = 0; i < n_deferred; ++i) load_b(i, i, deferred_pos[i], deferred_s[i], deferred_rows[i]);
          }
          if (!mbar_wait(&empty_bar[slot], ph ^ 1, p.wait_limit)) { give_up(); ok = false; break; }
          uint8_t* sa = stage_base + slot * stage_bytes;
          // FP8 shared weights arrive as bytes: twice the packed FP4 count
          mbar_expect_tx(&full_bar[slot], tx_a + (uint32_t)brows_u * 128u * CH +
                                              (shared_fp8_unit(pc.u) ? NA * 128 * 64 * CH : 0));
          if (NA == 2 && p.merged[sh]) {
            // gate and up rows of the stage in one op: {chunk elems, rows, chunks, matrix}
            if constexpr (EARLY)
              tma_load_4d_hint(sa, sh ? &p.a_shared[0] : &p.a_routed[0], 0, erow, s * CH, 0, &full_bar[slot], wpol);
            else
              tma_load_4d(sa, sh ? &p.a_shared[0] : &p.a_routed[0], 0, erow, s * CH, 0, &full_bar[slot]);
          } else {
#pragma unroll
            for (int m = 0; m < NA; ++m) {
              if constexpr (EARLY)
                tma_load_3d_hint(sa + m * C::kATile, sh ? &p.a_shared[m] : &p.a_routed[m], 0, erow, s * CH,
                                 &full_bar[slot], wpol);
              else
                tma_load_3d(sa + m * C::kATile, sh ? &p.a_shared[m] : &p.a_routed[m], 0, erow, s * CH,
                            &full_bar[slot]);
            }
          }
          if (early && s == pc.s0) wait_tile(pc.u, all_ready);
          if (waited) {
            if constexpr (kSepB) {
              // B slot g % 2 was last read by stage g - 2, whose MMAs
              // completing is the latest phase of that stage's empty
              // barrier (stage g + 1, its next user, is not issued yet)
              const int bs = (int)(g & 1u);
              if (g >= 2u) {
                const uint32_t g2 = g - 2u;
                if (!mbar_wait(&empty_bar[g2 % NS], (g2 / NS) & 1u, p.wait_limit)) { give_up(); ok = false; break; }
              }
              load_b(bs, slot, un.pos0, s, brows_u);
            } else {
              load_b(0, slot, un.pos0, s, brows_u);
            }
          } else {
            // while g < defer_cap the B slot and the stage slot are both g
            deferred_pos[n_deferred] = un.pos0;
            deferred_rows[n_deferred] = brows_u;
            deferred_s[n_deferred++] = s;
          }
#pragma unroll
          for (int i = 0; i < kMaxStages; ++i)
            if (i == slot) last_parity[i] = (int)ph;
        }
        if (!ok) break;
      }
      if (!waited) {
        pdl_wait();
        for (int i = 0; i < n_deferred; ++i) load_b(i, i, deferred_pos[i], deferred_s[i], deferred_rows[i]);
      }
      // never leave with copies in flight: wait for the last load into each
      // slot (the activation copies land on the same barriers)
#pragma unroll
      for (int s = 0; s < kMaxStages; ++s)
        if (last_parity[s] >= 0) mbar_wait(&full_bar[s], (uint32_t)last_parity[s], kDrainLimit);
    }
  } else if (warp == 1 || warp == kIssuer2Warp) {
    // ---------------------------------------------------------------- MMA
    // Two issuing threads.  A thread that also commits (tcgen05.commit in the
    // same loop) issues tcgen05.mma at ~105 cycles per instruction for N <=
    // 128; two such threads keep the tensor pipe at its throughput (measured:
    // ~39 cycles at N = 16, ~64 at N = 128).  Each thread commits its own
    // MMAs, so the empty and accumulator-full barriers count two arrivals.
    if (lane == 0) {
      const int j = warp == 1 ? 0 : 1;
      // N of the MMAs: the B rows (dense: all tokens), or per unit the tile's
      // tokens for the ragged wide tiles
      const int NI0 = BR;
      uint32_t g = 0, it = 0;
      Sched sc = sc0;
      uint32_t qi = 0;
      for (Piece pc = next_reader(sc, qi); pc.u >= 0 && !aborted(); pc = next_reader(sc, qi), ++it) {
        const int buf = C::kNAcc == 2 ? (int)(it & 1) : 0;
        const uint32_t ph_acc = C::kNAcc == 2 ? ((it >> 1) & 1) : (it & 1);
        const uint32_t d_tmem = tmem + buf * C::kAccCols;
        int swap = 0, NI = NI0, brows = BR;
        if (C::kRagged || ragged_b) {
          // part-filled tiles: N = the tile's tokens rounded up to the
          // instruction's step of 16, so the MMAs cost only the columns in
          // use (the epilogue reads no column past them)
          const Unit un = decode_unit(p, pc.u, mt_units, rot, n_tiles);
          NI = min(BN, (un.m_tile + 15) & ~15);
          brows = b_rows_of(un);  // its B chunks lie that many rows apart
        }
        if (NA == 2) {
          // the shared experts' tiles close the table, so no table load is
          // needed to tell them
          const int sh = tile_of(pc.u, mt_units, rot, n_tiles) >= n_tiles - p.ns_tiles;
          swap = p.merged[sh] && p.swap_gu[sh];
        }
        uint32_t idesc_base = A4 ? idesc_e2m1_e2m1(128, NI, 0) : idesc_e2m1_e4m3(128, NI, 0);
        if (shared_fp8_unit(pc.u)) idesc_base &= ~(7u << 7);  // A = E4M3 (FP8 shared expert)
        // the accumulator buffer is free once the epilogue has read it out
        if (!mbar_wait(&acce_bar[buf], ph_acc ^ 1, p.wait_limit)) { give_up(); break; }
        fence_after();
        bool ok = true;
        const int s_beg = pc.s0, s_end = pc.s1;
        for (int s = s_beg; s < s_end; ++s, ++g) {
          const int slot = g % NS;
          const uint32_t ph = (g / NS) & 1;
          if (!mbar_wait(&full_bar[slot], ph, p.wait_limit)) {
            give_up();
            ok = false;
            break;
          }
          fence_after();
          const uint32_t sa = smem_u32(stage_base + slot * stage_bytes);
          const uint32_t sb_addr = kSepB ? smem_u32(bring_base + (g & 1u) * C::kBTile) : sa + NA * C::kATile;
          // descriptors differ only in the start-address field (bits 0..13, address / 16)
          const uint64_t a_desc0 = sw128_desc(sa), b_desc0 = sw128_desc(sb_addr);
          const uint32_t sf = tmem + sf_col0 + slot * C::kSfCols;
#pragma unroll
          for (int c = 0; c < CH; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // 32 bytes of each operand row per instruction (K = 32 E4M3 / K = 64
              // packed E2M1); scale byte k of the chunk's word (A4: word k / 2,
              // bytes 2 (k % 2) and up)
              const int w = A4 ? k >> 1 : 0;
              const uint32_t sfid = A4 ? (uint32_t)(k & 1) * 2u : (uint32_t)k;
              const uint32_t idesc = idesc_base | (sfid << 4) | (sfid << 29);
              // chunk c of the B tile starts after c chunks of brows rows of 128 bytes
              const uint64_t bdesc = b_desc0 + (uint64_t)((c * brows * 128 + 32 * k) >> 4);
              const uint32_t sfb = sf + C::sfb_col(c, w, 0);
              auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfbb, uint32_t accumulate) {
                if constexpr (A4)
                  mma_mxf4(d, a, b, idesc, sfa, sfbb, accumulate);
                else
                  mma_mxf8f6f4(d, a, b, idesc, sfa, sfbb, accumulate);
              };
              if constexpr (MODE == kModeUp) {
                const int m = j, acc = swap ? 1 - m : m;  // gate -> accumulator 0, up -> 1
                mma(d_tmem + acc * BN, a_desc0 + (uint64_t)((m * C::kATile + c * 16384 + 32 * k) >> 4), bdesc,
                    sf + C::sfa_col(acc, c, w), sfb, (s != s_beg || c || k) ? 1u : 0u);
              } else {
                // K steps i = 4c + k of the stage: the first half to accumulator 0
                const int i = c * 4 + k, first = j * CH * 2;
                if ((i < CH * 2) == (j == 0))
                  mma(d_tmem + j * BN, a_desc0 + (uint64_t)((c * 16384 + 32 * k) >> 4), bdesc, sf + C::sfa_col(0, c, w),
                      sfb, (s != s_beg || i != first) ? 1u : 0u);
              }
            }
          mma_commit(&empty_bar[slot]);
        }
        if (!ok) break;
        mma_commit(&accf_bar[buf]);
      }
      // Leave only when every MMA this thread issued has completed: after a
      // wait elsewhere gave up, nothing else waits for them, and the TMEM they
      // write is freed below.  (With no MMA outstanding the commit arrives at
      // once.)
      mma_commit(&drain_bar[j]);
      mbar_wait(&drain_bar[j], 0, kDrainLimit);
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------- scale factors
    // The scale words of NB stages are fetched at once (double-buffered in
    // registers), so a global-load latency is paid per NB stages.
    constexpr int KW = C::kW;                                    // scale words per row and chunk
    constexpr int NB = 4, NW = (NA * CH + NC * CH) * KW;  // words per stage
    const int q = warp & 3;
    if (!early) pdl_wait();  // the activation scales come from the previous kernel
    uint32_t g = 0;
    bool ok = true, all_ready = false;
    Sched sc = sc0;
    uint32_t qi = 0;
    for (Piece pc = next_reader(sc, qi); ok && pc.u >= 0 && !aborted(); pc = next_reader(sc, qi)) {
      const Unit un = decode_unit(p, pc.u, mt_units, rot, n_tiles);
      const int s_end = pc.s1;
      const bool sh = un.e >= p.E;
      const size_t erow = (size_t)(sh ? un.e - p.E : un.e - p.e_lo) * p.rows + un.row0 + 32 * q + lane;
      const uint8_t* sa_row[NA];
#pragma unroll
      for (int m = 0; m < NA; ++m)
        sa_row[m] = (sh ? p.sa_shared[m] : p.sa_routed[m]) +
                    // FP8 shared: one scale per 32 x 32 block, shared by the warp's 32 rows
                    (shared_fp8_unit(pc.u) ? (erow >> 5) : erow) * (p.K / 32);
      // the scale row of B column n: dense, token n (all T tokens); else the
      // unit's position pos0 + n.  Columns without one get 2^0.
      const uint8_t* sb_row[NC];
#pragma unroll
      for (int cb = 0; cb < NC; ++cb) {
        const int n = lane + 32 * cb;
        sb_row[cb] = nullptr;
        if (dense ? n < p.T : n < un.m_tile) sb_row[cb] = p.sb + (size_t)(dense ? n : un.pos0 + n) * (p.K / 32);
      }
      // the weight scales first: their addresses are known before the token ones
      auto load = [&](uint32_t (&w)[NB][NW], int s0) {
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          if (s0 + i < s_end) {
#pragma unroll
            for (int c = 0; c < CH; ++c)
#pragma unroll
              for (int v = 0; v < KW; ++v) {
                const int kb = 4 * (KW * ((s0 + i) * CH + c) + v);  // first k-block of the word
#pragma unroll
                for (int m = 0; m < NA; ++m)
                  w[i][(m * CH + c) * KW + v] = __ldg(reinterpret_cast<const uint32_t*>(sa_row[m] + kb));
              }
          }
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          if (s0 + i < s_end) {
#pragma unroll
            for (int c = 0; c < CH; ++c)
#pragma unroll
              for (int v = 0; v < KW; ++v) {
                const int kb = 4 * (KW * ((s0 + i) * CH + c) + v);
#pragma unroll
                for (int cb = 0; cb < NC; ++cb)
                  w[i][(NA * CH + c * NC + cb) * KW + v] =
                      !sb_row[cb] ? 0x7F7F7F7Fu
                      // early down: written by the running gate/up launch, so not through
                      // the read-only cache (a line may hold an earlier tile's scales)
                      : (early && !all_ready) ? __ldcg(reinterpret_cast<const uint32_t*>(sb_row[cb] + kb))
                              : __ldg(reinterpret_cast<const uint32_t*>(sb_row[cb] + kb));
              }
          }
        }
      };
      auto store = [&](const uint32_t (&w)[NB][NW], int s0) -> bool {
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          if (s0 + i >= s_end) break;
          const int slot = g % NS;
          const uint32_t ph = (g / NS) & 1;
          if (!mbar_wait(&empty_bar[slot], ph ^ 1, p.wait_limit)) { give_up(); return false; }
          fence_after();
          const uint32_t col = tmem + ((uint32_t)(32 * q) << 16) + sf_col0 + slot * C::kSfCols;
#pragma unroll
          for (int c = 0; c < CH; ++c)
#pragma unroll
            for (int v = 0; v < KW; ++v) {
#pragma unroll
              for (int m = 0; m < NA; ++m) tmem_st_x1(col + C::sfa_col(m, c, v) + q, w[i][(m * CH + c) * KW + v]);
#pragma unroll
              for (int cb = 0; cb < NC; ++cb)
                tmem_st_x1(col + C::sfb_col(c, v, cb), w[i][(NA * CH + c * NC + cb) * KW + v]);
            }
          tmem_st_wait();
          fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full_bar[slot]);
          ++g;
        }
        return true;
      };
      uint32_t w0[NB][NW], w1[NB][NW];
      if (early) wait_tile(pc.u, all_ready);
      load(w0, pc.s0);
      for (int s0 = pc.s0; s0 < s_end; s0 += 2 * NB) {
        if (s0 + NB < s_end) load(w1, s0 + NB);
        if (!(ok = store(w0, s0))) break;
        if (s0 + NB >= s_end) break;
        if (s0 + 2 * NB < s_end) load(w0, s0 + 2 * NB);
        if (!(ok = store(w1, s0 + NB))) break;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;        // TMEM lane quadrant of this warp
    const int rl = 32 * q + lane;  // row within the 128-row tile
    // early down writes nothing the running gate/up reads (its partial tiles
    // have a region of their own)
    if (!early) pdl_wait();
    // h of one position at this lane's row, given the 32-row block maximum:
    // FP8 one code per row; FP4 (A4) two rows per byte, the even lane writing
    // its row (low nibble) and the next one's.  Lane 0 writes the scale.
    auto store_h = [&](size_t pos, const Unit& un, float h, float amax) {
      const int row = un.row0 + rl;
      if constexpr (A4) {
        const int ex = fp4_block_exponent(amax);
        const float hv = scale_pow2_neg(h, ex);
        const float hn = __shfl_down_sync(0xFFFFFFFFu, hv, 1);
        if ((lane & 1) == 0) p.hq[pos * (p.out_cols / 2) + row / 2] = (uint8_t)e2m1x2(hv, hn);
        if (lane == 0) p.hs[pos * (p.out_cols / 32) + (un.row0 + 32 * q) / 32] = (uint8_t)(ex + 127);
      } else {
        const int ex = fp8_block_exponent(amax);
        p.hq[pos * p.out_cols + row] = (uint8_t)(e4m3x2(scale_pow2_neg(h, ex), 0.f) & 0xFFu);
        if (lane == 0) p.hs[pos * (p.out_cols / 32) + (un.row0 + 32 * q) / 32] = (uint8_t)(ex + 127);
      }
    };
    // One output column (a token position) of the tile: all 32 lanes of the
    // warp take part (the h block scale is a max over the warp's 32 rows).
    auto emit = [&](const Unit& un, int col, float a, float b) {
      const size_t pos = (size_t)(un.pos0 + col);
      const int row = un.row0 + rl;  // weight row (I row for up, H row for down)
      if (MODE == kModeDown) {
        p.o[pos * p.out_cols + row] = a;
      } else {
        const float h = swiglu(a, b);
        store_h(pos, un, h, warp_max(fabsf(h)));
      }
    };
    // Sixteen columns at once (the main path): the SwiGLU values of all of them
    // first, then the sixteen 32-row maxima as interleaved shuffle trees, so
    // the shuffle latency is paid once per group rather than once per column.
    // Same operations per column as emit(), so the same bits.
    auto emit16 = [&](const Unit& un, int c, const uint32_t (&v)[16], const uint32_t (&vu)[16]) {
      const int row = un.row0 + rl;
      if constexpr (MODE == kModeDown) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (c + j >= un.m_tile) break;  // warp-uniform
          const float a = C::kSplitK ? __uint_as_float(v[j]) + __uint_as_float(vu[j]) : __uint_as_float(v[j]);
          p.o[(size_t)(un.pos0 + c + j) * p.out_cols + row] = a;
        }
      } else {
        float h[16], am[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float g = __uint_as_float(v[j]);
          h[j] = swiglu(g, __uint_as_float(vu[j]));
          am[j] = fabsf(h[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int j = 0; j < 16; ++j) am[j] = fmaxf(am[j], __shfl_xor_sync(0xFFFFFFFFu, am[j], o));
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (c + j >= un.m_tile) break;  // warp-uniform
          store_h((size_t)(un.pos0 + c + j), un, h[j], am[j]);
        }
      }
    };
    // Down mode with the combine fused (small batches): after a warp has
    // written the o rows of its unit, each of the unit's positions counts one
    // arrival for its token; the warp that brings a token's count to the
    // number of its positions (valid routed slots + shared experts) adds that
    // token's o rows for these 32 output rows in the fixed order of the
    // combine (shared experts, then slots j = 0..k-1) and writes y.
    auto combine_tail = [&](const Unit& un) {
      if constexpr (MODE == kModeDown && BN <= 64) {
        if (!p.fuse_combine) return;
        __threadfence();
        __syncwarp();
        const int n_rt = p.out_cols / 128, rt = un.row0 / 128;
        const int row = un.row0 + rl;
        const size_t S = (size_t)p.T * p.k, H = (size_t)p.out_cols;
        // the unit's positions 32 at a time, lane i0 + lane counting its token
        for (int i0 = 0; i0 < un.m_tile; i0 += 32) {
          int done = -1;
          if (i0 + lane < un.m_tile) {
            const int t = p.pos_tok[un.pos0 + i0 + lane];
            int sp[kMaxTopK];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) sp[j] = j < p.k ? p.slot_pos[t * p.k + j] : -1;
            int need = p.ns;
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) need += sp[j] >= 0;
            if (atomicAdd(&p.comb_cnt[(t * n_rt + rt) * 4 + q], 1) == need - 1) done = t;
          }
          unsigned todo = __ballot_sync(0xFFFFFFFFu, done >= 0);
          if (todo) __threadfence();
          while (todo) {
            const int t = __shfl_sync(0xFFFFFFFFu, done, __ffs(todo) - 1);
            todo &= todo - 1;
            // lane j < k holds slot j's position and weight; then every o load is in flight at once
            const int my_pp = lane < p.k ? p.slot_pos[t * p.k + lane] : -1;
            const float my_w = lane < p.k ? p.w[t * p.k + lane] : 0.f;
            float osh[kMaxShared], ov[kMaxTopK];
#pragma unroll
            for (int j = 0; j < kMaxShared; ++j)
              osh[j] = j < p.ns ? __ldcg(p.o + (S + (size_t)j * p.T + t) * H + row) : 0.f;
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
              const int pp = __shfl_sync(0xFFFFFFFFu, my_pp, j);
              ov[j] = pp >= 0 ? __ldcg(p.o + (size_t)pp * H + row) : 0.f;
            }
            // the combine's fixed order: shared experts, then slots j = 0..k-1
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxShared; ++j)
              if (j < p.ns) acc += osh[j];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
              const float wj = __shfl_sync(0xFFFFFFFFu, my_w, j);
              if (__shfl_sync(0xFFFFFFFFu, my_pp, j) >= 0) acc = fmaf(wj, ov[j], acc);
            }
            uint16_t yb = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
            if (p.res)
              yb = __bfloat16_as_ushort(__float2bfloat16_rn(bf16_bits_to_float(p.res[(size_t)t * H + row]) +
                                                            bf16_bits_to_float(yb)));
            p.y[(size_t)t * H + row] = yb;
          }
        }
      }
    };
    constexpr int kSlot = NA * BN * 128;  // floats per partial slot: [matrix][position][row]
    // The accumulator values of the unit's positions i0 .. i0 + 15 (matrix 0
    // / the first K half in v, matrix 1 / the second K half in vu): in dense
    // mode the column of each position's token, one column per load; else the
    // positions are the columns.
    auto load_cols = [&](const Unit& un, uint32_t t_base, int i0, uint32_t (&v)[16], uint32_t (&vu)[16]) {
      constexpr bool kTwo = MODE == kModeUp || C::kSplitK;
      if (dense) {
        const int tok = (lane < 16 && i0 + lane < un.m_tile) ? p.pos_tok[un.pos0 + i0 + lane] : 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t col = (uint32_t)__shfl_sync(0xFFFFFFFFu, tok, j);
          tmem_ld1(t_base + col, v[j]);
          if (kTwo) tmem_ld1(t_base + BN + col, vu[j]);
        }
      } else {
        tmem_ld16(t_base + i0, v);
        if (kTwo) tmem_ld16(t_base + BN + i0, vu);
      }
      tmem_ld_wait();
    };
    // small batches, gate/up: count this warp's 32 rows of a finished unit
    // toward its tile (down reads them by tensor copies: proxy fence first)
    auto count_tile = [&](int u) {
      if constexpr (MODE == kModeUp) {
        if (!early_on) return;
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.ready + tile_of(u, mt_units, rot, n_tiles), 1);
      }
    };
    uint32_t it = 0;
    Sched sc = sc0;
    uint32_t qi = 0;
    for (Piece pc = next_reader(sc, qi); pc.u >= 0 && !aborted(); pc = next_reader(sc, qi), ++it) {
      const Unit un = decode_unit(p, pc.u, mt_units, rot, n_tiles);
      const int buf = C::kNAcc == 2 ? (int)(it & 1) : 0;
      const uint32_t ph_acc = C::kNAcc == 2 ? ((it >> 1) & 1) : (it & 1);
      if (!mbar_wait(&accf_bar[buf], ph_acc, p.wait_limit)) { give_up(); break; }
      fence_after();
      const uint32_t t_base = tmem + ((uint32_t)(32 * q) << 16) + buf * C::kAccCols;
      int first, n;
      sc.pieces(pc.u, first, n);
      // positions of the unit, in groups of 16
      const int i_end = (un.m_tile + 15) & ~15;
      if (n == 1) {
        // the whole unit: straight from TMEM to the outputs
#pragma unroll 1
        for (int i0 = 0; i0 < i_end; i0 += 16) {
          uint32_t v[16], vu[16];
          load_cols(un, t_base, i0, v, vu);
          if (i0 + 16 >= i_end) {
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce_bar[buf]);
          }
          emit16(un, i0, v, vu);  // down split-K: the two K halves, in fixed order
        }
        count_tile(pc.u);
        combine_tail(un);
        continue;
      }
      if constexpr (BN <= 64) {
        // A piece of a unit cut between CTAs: publish the fp32 partial tile;
        // the last piece to arrive adds all of them in piece order.  Each warp
        // owns its 32 rows, so the hand-off is per warp (one counter per unit
        // and quadrant) and no warp ever waits for another.
        float* mine = p.part + (size_t)sc.slot(pc.u, first, sc.cta - first) * kSlot;
#pragma unroll 1
        for (int i0 = 0; i0 < i_end; i0 += 16) {
          uint32_t v[16], vu[16];
          load_cols(un, t_base, i0, v, vu);
          if (i0 + 16 >= i_end) {
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce_bar[buf]);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (i0 + j >= un.m_tile) break;  // warp-uniform
            if constexpr (C::kSplitK)
              mine[(i0 + j) * 128 + rl] = __uint_as_float(v[j]) + __uint_as_float(vu[j]);
            else
              mine[(i0 + j) * 128 + rl] = __uint_as_float(v[j]);
            if (MODE == kModeUp) mine[(BN + i0 + j) * 128 + rl] = __uint_as_float(vu[j]);
          }
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&p.cnt[pc.u * 4 + q], 1) == n - 1;
        if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
          __threadfence();
          const float* src[kMaxPieces];
#pragma unroll
          for (int j = 0; j < kMaxPieces; ++j)
            src[j] = p.part + (size_t)sc.slot(pc.u, first, j < n ? j : 0) * kSlot + rl;
#pragma unroll 1
          for (int col = 0; col < un.m_tile; ++col) {
            float pa[kMaxPieces], pb[kMaxPieces];
#pragma unroll
            for (int j = 0; j < kMaxPieces; ++j) {  // all loads in flight, then the fixed-order sum
              pa[j] = j < n ? __ldcg(src[j] + col * 128) : 0.f;
              pb[j] = (MODE == kModeUp && j < n) ? __ldcg(src[j] + (BN + col) * 128) : 0.f;
            }
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxPieces; ++j) {
              if (j < n) {
                a += pa[j];
                b += pb[j];
              }
            }
            emit(un, col, a, b);
          }
          if (lane == 0) p.cnt[pc.u * 4 + q] = 0;
          count_tile(pc.u);
          combine_tail(un);
        }
      }
    }
  }
  // early down: this launch completes only after gate/up's (as the launch
  // order promises the kernels after it)
  if (early && threadIdx.x == 0) pdl_wait();
  fence_before();
  __syncthreads();
  if (MODE == kModeUp && early_on && threadIdx.x == 0) {
    // every unit of this CTA is counted (its warps' counts came before the barrier)
    __threadfence();
    atomicAdd(p.ready_done, 1);
  }
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, C::kTmemAlloc);
  }
}

template <int MODE, int BN, int CH, bool A4, bool EARLY = false>
cudaError_t launch_one(MmaParams& p, int num_sms, cudaStream_t st) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(ffn_mma_kernel<MODE, BN, CH, A4, EARLY>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  int smem = 0;
  geometry<MODE, BN, CH, A4>(p.K, &p.n_stages, &smem);
  if (p.n_stages < 2) return cudaErrorInvalidConfiguration;
  cudaError_t e = launch_pdl(ffn_mma_kernel<MODE, BN, CH, A4, EARLY>, dim3(num_sms), dim3(kThreadsMma), smem, st, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int MODE, int CH, bool A4>
cudaError_t launch_bn(MmaParams& p, int bn, int num_sms, cudaStream_t st) {
  if (bn == 16) return launch_one<MODE, 16, CH, A4>(p, num_sms, st);
  // small batches with 64-token tiles (17 to 64 tokens): the variant whose
  // down starts per token tile (the code costs the other launches time even
  // unused, so it is a variant of its own)
  if (bn == 64)
    return p.ready ? launch_one<MODE, 64, CH, A4, true>(p, num_sms, st) : launch_one<MODE, 64, CH, A4, false>(p, num_sms, st);
  return launch_one<MODE, 112, CH, A4>(p, num_sms, st);
}

}  // namespace

// Launches of the kernel for one activation format (one translation unit each,
// so that the two sets of instantiations compile in parallel).  ch: chunks per
// stage, 1..3.
cudaError_t launch_ffn_mma_fp8(MmaParams& p, int mode, int bn, int ch, int num_sms, cudaStream_t st);
cudaError_t launch_ffn_mma_fp4(MmaParams& p, int mode, int bn, int ch, int num_sms, cudaStream_t st);

#ifdef MOE_FFN_MMA_INSTANTIATE
cudaError_t MOE_FFN_MMA_INSTANTIATE(MmaParams& p, int mode, int bn, int ch, int num_sms, cudaStream_t st) {
#if MOE_FFN_MMA_A4
  // FP4 activations: one 256-element chunk per stage (the TMEM left next to
  // the widest tile's double-buffered accumulators holds two stages' scales)
  if (ch != 1) return cudaErrorInvalidValue;
  return mode == kModeUp ? launch_bn<kModeUp, 1, true>(p, bn, num_sms, st)
                         : launch_bn<kModeDown, 1, true>(p, bn, num_sms, st);
#else
  // ch 3 only where it divides down's K chunks (I / 384)
  if (mode == kModeUp)
    return ch == 2 ? launch_bn<kModeUp, 2, false>(p, bn, num_sms, st)
                   : launch_bn<kModeUp, 1, false>(p, bn, num_sms, st);
  if (ch == 3) return launch_bn<kModeDown, 3, false>(p, bn, num_sms, st);
  return ch == 2 ? launch_bn<kModeDown, 2, false>(p, bn, num_sms, st)
                 : launch_bn<kModeDown, 1, false>(p, bn, num_sms, st);
#endif
}
#endif

}  // namespace moe

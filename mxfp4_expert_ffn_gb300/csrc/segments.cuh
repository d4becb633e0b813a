// Expert segments: a stable counting sort of the T*k (token, rank) slots by
// expert, the active-expert list and the token-tile table of the tensor-core
// path.  The routed MoE block (FreeToken issue #444, "Architecture delta vs
// deepseek_v4": 384 routed + 1 shared experts, top-6).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {

// A slot's expert id is local (this layer computes it), remote (a valid id in
// [0, E) outside the layer's expert range: another rank's under expert
// parallelism, skipped without an error) or invalid (skipped and reported).
__device__ __forceinline__ bool slot_local(int e, const Workspace& ws) { return e >= ws.e_lo && e < ws.e_hi; }

// Block-wide exclusive scans over the experts (thread e for expert e; needs
// blockDim.x == 1024 >= E) of the per-expert slot counts cnt_s[e], of the
// "has slots" flags and of the token tiles of width bn: writes ws.cnt/off, the
// first position off_s[e], the active list act_s (routed experts in order,
// then the shared ones) with tile prefixes tp_s[0..na], n_active and the
// routed slot total.  Ends with a barrier.
__device__ __forceinline__ void scan_experts(const int32_t* cnt_s, int E, int T, int S, int ns, int bn,
                                             const Workspace& ws, int32_t* off_s, int32_t* act_s,
                                             int32_t* tp_s, int* n_act_s, int* routed_total_s) {
  const int NE = E + ns, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    // block-wide exclusive scans over the experts (one thread each) of the counts,
    // of the "has slots" flags and of the token tiles
    __shared__ int wsum[32][3];
    const int tb = bn > 0 ? bn : 1;
    const int c = tid < E ? cnt_s[tid] : 0;
    const int f = c > 0, ntl = (c + tb - 1) / tb;
    int a = c, b = f, d = ntl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a2 = __shfl_up_sync(0xFFFFFFFFu, a, o);
      const int b2 = __shfl_up_sync(0xFFFFFFFFu, b, o);
      const int d2 = __shfl_up_sync(0xFFFFFFFFu, d, o);
      if (lane >= o) {
        a += a2;
        b += b2;
        d += d2;
      }
    }
    if (lane == 31) {
      wsum[warp][0] = a;
      wsum[warp][1] = b;
      wsum[warp][2] = d;
    }
    __syncthreads();
    if (warp == 0) {
      int x = wsum[lane][0], y = wsum[lane][1], z = wsum[lane][2];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x2 = __shfl_up_sync(0xFFFFFFFFu, x, o);
        const int y2 = __shfl_up_sync(0xFFFFFFFFu, y, o);
        const int z2 = __shfl_up_sync(0xFFFFFFFFu, z, o);
        if (lane >= o) {
          x += x2;
          y += y2;
          z += z2;
        }
      }
      wsum[lane][0] = x;  // inclusive prefix over warps
      wsum[lane][1] = y;
      wsum[lane][2] = z;
    }
    __syncthreads();
    const int pa = warp ? wsum[warp - 1][0] : 0, pb = warp ? wsum[warp - 1][1] : 0,
              pd = warp ? wsum[warp - 1][2] : 0;
    if (tid < E) {
      const int off = pa + a - c, fr = pb + b - f, tr = pd + d - ntl;
      ws.cnt[tid] = c;
      ws.off[tid] = off;
      off_s[tid] = off;
      if (c > 0) {
        act_s[fr] = tid;
        tp_s[fr] = tr;
      }
    }
    if (tid == 0) {
      const int n_routed_active = wsum[31][1];
      int tiles = wsum[31][2];
      *routed_total_s = wsum[31][0];
      for (int sh = 0; sh < ns; ++sh) {
        ws.cnt[E + sh] = T;
        ws.off[E + sh] = S + sh * T;
        if (T > 0) {
          act_s[n_routed_active + sh] = E + sh;
          tp_s[n_routed_active + sh] = tiles;
          tiles += (T + tb - 1) / tb;
        }
      }
      ws.off[NE] = S + ns * T;
      const int na = n_routed_active + (T > 0 ? ns : 0);
      *n_act_s = na;
      *ws.n_active = na;
      ws.n_active[1] = tiles;
      tp_s[na] = tiles;
    }
  }
  __syncthreads();
}

// Builds the expert segments in one CTA of 1024 threads.  Each warp owns a
// contiguous range of slots; pass 1 counts its slots per expert, pass 2 turns
// the counts into per-warp bases (warps in slot order), pass 3 places each
// slot at base + rank among the warp's equal-expert lanes.  The result is a
// stable counting sort, identical on every run.
// Needs blockDim.x == 1024 and sm = 36 * E + 2 * ns + 1 ints of shared memory; every
// thread of the CTA must call it.
// zero_counts: zero the GEMMs' split-partition (and per-tile) counters and the
// fused-combine counters here (the preparation kernel does it in its parallel
// phase instead).
__device__ __forceinline__ void segments_cta(const int32_t* __restrict__ idx, int T, int k, int E,
                                             int ns, int bn, const Workspace& ws, int32_t* sm,
                                             bool scatter_smem = false, bool zero_counts = true) {
  const int NE = E + ns;
  int32_t* wcnt = sm;                  // [32][E] per-warp counts, then running bases
  int32_t* stot = sm + 32 * E;         // [E]     slots per expert
  int32_t* off_s = stot + E;           // [E]     first position per expert
  int32_t* act_s = off_s + E;          // [NE]    active experts
  int32_t* tp_s = act_s + NE;          // [NE+1]  token tiles before each active expert
  int32_t* ps = tp_s + NE + 1;         // [S]     scatter_smem: the slot at each position
  __shared__ int n_act_s, routed_total_s;
  const int S = T * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
  if (zero_counts) {
    // the tensor-core GEMM's split-partition counters start every forward at zero
    for (int i = threadIdx.x; i < ws.split_cnt_n; i += blockDim.x) ws.split_cnt[i] = 0;
    // and so do the fused-combine counters
    for (int i = threadIdx.x; i < ws.comb_cnt_n; i += blockDim.x) ws.comb_cnt[i] = 0;
  }
  __syncthreads();
  // Each warp owns slots [lo, hi) and reads their expert ids eight rows of 32
  // at a time (all eight loads in flight before they are used).
  constexpr int kU = 8;
  const int per = (S + 31) / 32;
  const int lo = min(S, warp * per), hi = min(S, lo + per);
  for (int b0 = lo; b0 < hi; b0 += 32 * kU) {
    int er[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int s = b0 + 32 * u + lane;
      er[u] = s < hi ? idx[s] : -1;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (b0 + 32 * u >= hi) break;  // warp-uniform
      int e = er[u];
      if (b0 + 32 * u + lane < hi && (e < 0 || e >= E)) {
        raise_error(ws.err, kErrExpertRange);
        e = -1;
      } else if (!slot_local(e, ws)) {
        e = -1;
      }
      if (b0 + 32 * u + lane >= hi) e = -1;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
    stot[e] = run;
  }
  __syncthreads();
  scan_experts(stot, E, T, S, ns, bn, ws, off_s, act_s, tp_s, &n_act_s, &routed_total_s);
  const int na = n_act_s;
  for (int a = threadIdx.x; a <= na; a += blockDim.x) {
    ws.tile_prefix[a] = tp_s[a];
    if (a < na) ws.active[a] = act_s[a];
  }
  // placement: position p = the expert's first position + the slots of that
  // expert in earlier warps + the equal-expert lanes before this one
  for (int b0 = lo; b0 < hi; b0 += 32 * kU) {
    int er[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int s = b0 + 32 * u + lane;
      er[u] = s < hi ? idx[s] : -1;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (b0 + 32 * u >= hi) break;  // warp-uniform
      const int s = b0 + 32 * u + lane;
      int e = er[u];
      if (s >= hi || e < 0 || e >= E || !slot_local(e, ws)) e = -1;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
      if (e >= 0) {
        const int p = off_s[e] + wcnt[warp * E + e] + __popc(peers & ((1u << lane) - 1u));
        ws.slot_pos[s] = p;
        if (scatter_smem) {
          ps[p] = s;
        } else {
          ws.perm[p] = s;
          ws.pos_tok[p] = s / k;
        }
      } else if (s < hi) {
        ws.slot_pos[s] = -1;
      }
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + e] += __popc(peers);
      __syncwarp();
    }
  }
  if (scatter_smem) {
    // the position-ordered tables leave shared memory in coalesced rows
    __syncthreads();
    for (int p = threadIdx.x; p < routed_total_s; p += blockDim.x) {
      const int sl = ps[p];
      ws.perm[p] = sl;
      ws.pos_tok[p] = sl / k;
    }
  }
  for (int i = threadIdx.x; i < ns * T; i += blockDim.x) ws.pos_tok[S + i] = i % T;
  // token tiles of width bn for the tensor-core path: (expert, first position, tokens)
  if (bn > 0) {
    for (int a = threadIdx.x; a < na; a += blockDim.x) {
      const int x = act_s[a];
      const int c = x < E ? stot[x] : T, p0 = x < E ? off_s[x] : S + (x - E) * T, t0 = tp_s[a];
      for (int j = 0; j * bn < c; ++j) ws.tile_info[t0 + j] = make_int4(x, p0 + j * bn, min(bn, c - j * bn), 0);
    }
  }
  // positions left free by invalid expert ids still name a real token, so
  // that every position's row can be read safely
  for (int p = routed_total_s + threadIdx.x; p < S; p += blockDim.x) ws.pos_tok[p] = 0;
}


// The same segments for a small batch (T * k <= blockDim.x == 1024, E <= 1024),
// with every intermediate in shared memory: one thread per slot, counts by
// shared atomics, the rank of a slot among its expert's slots by counting
// the earlier equal slots (so the order is the stable one above, bit for bit).
// sm needs 4 * E + 2 * ns + T * k + 1 ints.
__device__ __forceinline__ void segments_small_cta(const int32_t* __restrict__ idx, int T, int k, int E,
                                                   int ns, int bn, const Workspace& ws, int32_t* sm,
                                                   bool zero_counts = true) {
  const int NE = E + ns, S = T * k, tid = threadIdx.x;
  int32_t* cnt_s = sm;             // [E]     slots per expert
  int32_t* off_s = sm + E;         // [E]     first position per expert
  int32_t* act_s = sm + 2 * E;     // [NE]    active experts, routed then shared
  int32_t* tp_s = sm + 2 * E + NE; // [NE+1]  token tiles before each active expert
  int32_t* sid = tp_s + NE + 1;    // [S]     expert of each slot (-1: invalid)
  __shared__ int n_act_s, routed_total_s;
  if (zero_counts) {
    for (int i = tid; i < ws.split_cnt_n; i += blockDim.x) ws.split_cnt[i] = 0;
    for (int i = tid; i < ws.comb_cnt_n; i += blockDim.x) ws.comb_cnt[i] = 0;
  }
  for (int e = tid; e < E; e += blockDim.x) cnt_s[e] = 0;
  __syncthreads();
  int e = -1;
  if (tid < S) {
    e = idx[tid];
    if (e < 0 || e >= E) {
      raise_error(ws.err, kErrExpertRange);
      e = -1;
    } else if (!slot_local(e, ws)) {
      e = -1;
    }
    sid[tid] = e;
    if (e >= 0) atomicAdd(&cnt_s[e], 1);
  }
  __syncthreads();
  scan_experts(cnt_s, E, T, S, ns, bn, ws, off_s, act_s, tp_s, &n_act_s, &routed_total_s);
  const int na = n_act_s;
  for (int a = tid; a <= na; a += blockDim.x) {
    ws.tile_prefix[a] = tp_s[a];
    if (a < na) ws.active[a] = act_s[a];
  }
  if (tid < S) {
    if (e >= 0) {
      int r = 0;
      for (int s2 = 0; s2 < tid; ++s2) r += sid[s2] == e;
      const int p = off_s[e] + r;
      ws.perm[p] = tid;
      ws.slot_pos[tid] = p;
      ws.pos_tok[p] = tid / k;
    } else {
      ws.slot_pos[tid] = -1;
    }
  }
  for (int i = tid; i < ns * T; i += blockDim.x) ws.pos_tok[S + i] = i % T;
  if (bn > 0) {
    for (int a = tid; a < na; a += blockDim.x) {
      const int x = act_s[a];
      const int c = x < E ? cnt_s[x] : T, p0 = x < E ? off_s[x] : S + (x - E) * T, t0 = tp_s[a];
      for (int j = 0; j * bn < c; ++j) ws.tile_info[t0 + j] = make_int4(x, p0 + j * bn, min(bn, c - j * bn), 0);
    }
  }
  for (int p = routed_total_s + tid; p < S; p += blockDim.x) ws.pos_tok[p] = 0;
}

// Expert segments of at most 32 slots when every expert's slots fit one
// token tile (T <= bn), without a CTA-wide barrier: every thread fills the
// count and first position of its experts from the slot ids, and warp 0
// places the slots (one lane each) with match and ballot operations -- the
// same stable counting sort as segments_cta, so the same outputs.
// sid: the S slot ids in shared memory, visible to every calling thread.
// The caller zeroes ws.split_cnt and ws.comb_cnt (the preparation kernel does
// it in its parallel phase, off this serial path).
__device__ __forceinline__ void segments_tiny(const int32_t* sid, int T, int k, int E, int ns,
                                              const Workspace& ws) {
  const int S = T * k, NE = E + ns, tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0, off = 0;
    for (int j = 0; j < S; ++j) {
      const int x = sid[j];
      const bool v = x >= 0 && x < E && slot_local(x, ws);
      c += v && x == e;
      off += v && x < e;
    }
    ws.cnt[e] = c;
    ws.off[e] = off;
  }
  for (int i = tid; i < ns * T; i += blockDim.x) ws.pos_tok[S + i] = i % T;
  if (tid >= 32) return;
  const unsigned full = 0xFFFFFFFFu;
  const int x = lane < S ? sid[lane] : -1;
  const bool v = lane < S && x >= 0 && x < E && slot_local(x, ws);
  if (lane < S && (x < 0 || x >= E)) raise_error(ws.err, kErrExpertRange);
  const unsigned same = __match_any_sync(full, v ? x : -1 - lane);  // lanes with this slot's expert
  const int rank = __popc(same & ((1u << lane) - 1u));            // earlier slots of that expert
  const bool leader = v && (__ffs(same) - 1 == lane);              // the expert's first slot
  int less = 0, dless = 0;  // valid slots / active experts with a lower expert id
  for (int j = 0; j < S; ++j) {
    const int xj = __shfl_sync(full, v ? x : 0x7FFFFFFF, j);
    const int lj = __shfl_sync(full, leader ? 1 : 0, j);
    less += xj < x;
    dless += lj && xj < x;
  }
  const int routed_total = __popc(__ballot_sync(full, v));
  const int n_routed = __popc(__ballot_sync(full, leader));
  if (lane < S) {
    if (v) {
      const int p = less + rank;
      ws.perm[p] = lane;
      ws.slot_pos[lane] = p;
      ws.pos_tok[p] = lane / k;
    } else {
      ws.slot_pos[lane] = -1;
    }
    if (lane >= routed_total) ws.pos_tok[lane] = 0;  // positions freed by invalid ids
  }
  if (leader) {  // active expert dless: one token tile of its slots
    ws.active[dless] = x;
    ws.tile_prefix[dless] = dless;
    ws.tile_info[dless] = make_int4(x, less, __popc(same), 0);
  }
  if (lane < ns) {  // the shared experts after the routed ones, every token once
    const int a = n_routed + lane;
    ws.cnt[E + lane] = T;
    ws.off[E + lane] = S + lane * T;
    ws.active[a] = E + lane;
    ws.tile_prefix[a] = a;
    ws.tile_info[a] = make_int4(E + lane, S + lane * T, T, 0);
  }
  if (lane == 0) {
    const int na = n_routed + ns;
    ws.off[NE] = S + ns * T;
    ws.tile_prefix[na] = na;
    ws.n_active[0] = na;
    ws.n_active[1] = na;
  }
}

// ---- Large batches: the same stable counting sort over G CTAs in two
// launches.  Slot ranges are contiguous per CTA and, inside a CTA, per warp,
// in slot order, so positions come out exactly as from segments_cta.

// Per-warp counts of this CTA's slots [c0, c1) into wcnt[32][E] (shared,
// zeroed by the caller); invalid ids are reported (when report) and skipped.
__device__ __forceinline__ void count_warp_slots(const int32_t* __restrict__ idx, int c0, int c1, int E,
                                                 int32_t* wcnt, const Workspace& ws, bool report) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (c1 - c0 + 31) / 32;
  const int lo = min(c1, c0 + warp * per), hi = min(c1, lo + per);
  for (int b0 = lo; b0 < hi; b0 += 32) {
    const int s = b0 + lane;
    int e = s < hi ? idx[s] : -1;
    if (s < hi && (e < 0 || e >= E)) {
      if (report) raise_error(ws.err, kErrExpertRange);
      e = -1;
    } else if (!slot_local(e, ws)) {
      e = -1;
    }
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + e] += __popc(peers);
  }
}

// Launch 1 of 2 (grid G, 1024 threads, 32 * E + 4 * E + 2 * ns + 2 ints of shared
// memory): per-CTA counts into ws.seg_cbase[cta][E]; the last CTA to finish
// turns them into absolute per-CTA bases, runs scan_experts and writes the
// active list, tile table and shared positions.  Also zeroes the GEMM counters.
__device__ __forceinline__ void segments_count_cta(const int32_t* __restrict__ idx, int T, int k, int E, int ns,
                                                   int bn, const Workspace& ws, int32_t* sm) {
  const int NE = E + ns, S = T * k, G = gridDim.x, cta = blockIdx.x;
  int32_t* wcnt = sm;              // [32][E]
  int32_t* stot = sm + 32 * E;     // [E]
  int32_t* off_s = stot + E;       // [E]
  int32_t* act_s = off_s + E;      // [NE]
  int32_t* tp_s = act_s + NE;      // [NE+1]
  __shared__ int n_act_s, routed_total_s, last;
  for (int i = cta * blockDim.x + threadIdx.x; i < ws.split_cnt_n; i += G * blockDim.x) ws.split_cnt[i] = 0;
  for (int i = cta * blockDim.x + threadIdx.x; i < ws.comb_cnt_n; i += G * blockDim.x) ws.comb_cnt[i] = 0;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int per = (S + G - 1) / G;
  const int c0 = min(S, cta * per), c1 = min(S, c0 + per);
  count_warp_slots(idx, c0, c1, E, wcnt, ws, true);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < 32; ++w) c += wcnt[w * E + e];
    ws.seg_cbase[cta * E + e] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    last = atomic_add_acq_rel(ws.seg_counter, 1) == G - 1;
    if (last) *ws.seg_counter = 0;
  }
  __syncthreads();
  if (!last) return;
  // the finisher: per expert, the running count over CTAs in order
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int c = 0; c < G; ++c) {
      const int n = __ldcg(ws.seg_cbase + c * E + e);
      ws.seg_cbase[c * E + e] = run;
      run += n;
    }
    stot[e] = run;
  }
  __syncthreads();
  scan_experts(stot, E, T, S, ns, bn, ws, off_s, act_s, tp_s, &n_act_s, &routed_total_s);
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    for (int c = 0; c < G; ++c) ws.seg_cbase[c * E + e] += off_s[e];
  const int na = n_act_s;
  for (int a = threadIdx.x; a <= na; a += blockDim.x) {
    ws.tile_prefix[a] = tp_s[a];
    if (a < na) ws.active[a] = act_s[a];
  }
  if (bn > 0) {
    for (int a = threadIdx.x; a < na; a += blockDim.x) {
      const int x = act_s[a];
      const int c = x < E ? stot[x] : T, p0 = x < E ? off_s[x] : S + (x - E) * T, t0 = tp_s[a];
      for (int j = 0; j * bn < c; ++j) ws.tile_info[t0 + j] = make_int4(x, p0 + j * bn, min(bn, c - j * bn), 0);
    }
  }
  if (threadIdx.x == 0) *ws.seg_routed = routed_total_s;
}

// Launch 2 of 2 (same grid, 32 * E ints of shared memory): per-warp counts
// again, per-warp bases from this CTA's base, then every slot's position.
__device__ __forceinline__ void segments_place_cta(const int32_t* __restrict__ idx, int T, int k, int E, int ns,
                                                   const Workspace& ws, int32_t* sm) {
  const int S = T * k, G = gridDim.x, cta = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* wcnt = sm;  // [32][E] counts, then bases
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int per = (S + G - 1) / G;
  const int c0 = min(S, cta * per), c1 = min(S, c0 + per);
  count_warp_slots(idx, c0, c1, E, wcnt, ws, false);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = __ldcg(ws.seg_cbase + cta * E + e);
    for (int w = 0; w < 32; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const int wper = (c1 - c0 + 31) / 32;
  const int lo = min(c1, c0 + warp * wper), hi = min(c1, lo + wper);
  for (int b0 = lo; b0 < hi; b0 += 32) {
    const int s = b0 + lane;
    int e = s < hi ? idx[s] : -1;
    if (s >= hi || e < 0 || e >= E || !slot_local(e, ws)) e = -1;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    if (e >= 0) {
      const int p = wcnt[warp * E + e] + __popc(peers & ((1u << lane) - 1u));
      ws.slot_pos[s] = p;
      ws.perm[p] = s;
      ws.pos_tok[p] = s / k;
    } else if (s < hi) {
      ws.slot_pos[s] = -1;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  // shared positions, and positions left free by invalid ids (a real token)
  for (int i = cta * blockDim.x + threadIdx.x; i < ns * T; i += G * blockDim.x) ws.pos_tok[S + i] = i % T;
  const int rt = __ldcg(ws.seg_routed);
  for (int p = rt + cta * blockDim.x + threadIdx.x; p < S; p += G * blockDim.x) ws.pos_tok[p] = 0;
}

}  // namespace moe

// Tile walk shared by the grouped GEMM kernels: a tile is (route block,
// weight-row tile); stage 1 walks route-block major (the n-tiles of a block
// reuse its activation rows), and so does stage 2 at decode sizes
// (n_group_log2 < 0); larger stage-2 walks go in groups of 2^n_group_log2
// feature tiles, route-block major inside a group (the FP32 reductions of
// concurrently running tiles stay in the group's slice of the accumulator,
// i.e. in L2, and the intermediate is read once per group).
#pragma once
#include <cstdint>
#include "common.cuh"
#include "moe_internal.h"
#include "router_warp.cuh"
#include "sm100_ptx.cuh"

namespace moe {

// Expert id of a route block, checked when the tile becomes current (the
// load was issued one tile earlier, so the check never waits on it). The
// sort writes ids in [0, E) for every block below the padded route count;
// any other value means a corrupted route list: it is reported through the
// status word (kDevBadExpert) and replaced by expert 0, so no weight access
// leaves the weight arrays.
template <class Args>
__device__ __forceinline__ int expert_checked(const Args& a, int e) {
  if (static_cast<unsigned>(e) < static_cast<unsigned>(a.E)) return e;
  if (a.status) atomicOr(a.status, kDevBadExpert);
  return 0;
}

// ---------------------------------------------------------- local layout
// At decode sizes a GEMM can derive the route layout itself: topk_ids is an
// input of the call, complete before the call's first kernel starts, so the
// CTA counts the valid routes per expert, pads each count to the route block
// and scans, before the kernel's dependency wait. The producer then knows
// the experts of its first tiles and loads their weights while the previous
// kernel (the sort and gather, or stage one) still runs. The result is the
// layout the sort writes (stable counting sort, ids outside [0, E) dropped,
// empty experts take no block): blk_expert[b] = expert of route block b, and
// the number of blocks; the producer checks the block count against the
// sort's after the wait.
// Measured on GB300 (backbone, expert-parallel and a16w4 decode sweeps): the
// local layout shortens calls of up to ~150 routes by 3-11 % and lengthens
// calls of several hundred routes by 3-6 %, so it is used up to 160 routes.
constexpr int kLocalMaxRoutes = 160;
constexpr int kLocalMaxBlocks = 1024;   // R / 16 + E <= 288 + 512 at the route limit

// Gated calls (gate.logits set): the routing comes from the router logits,
// the call's input, through the per-token selection the gating kernels use.
// All threads of the CTA; cnt: E + 1 ints of scratch shared memory (free
// before the dependency wait), followed by room for R ids when gating;
// blk_expert: kLocalMaxBlocks entries. Returns the number of route blocks.
// Contains __syncthreads.
__device__ __forceinline__ int local_block_layout(const int32_t* ids, int R, int E, int bn,
                                                  int* cnt, uint16_t* blk_expert,
                                                  const LocalGate& gate, int M) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
  for (int e = tid; e <= E; e += nt) cnt[e] = 0;
  if (gate.logits) {
    // one warp per token selects its experts; the ids go to shared memory
    int* sid = cnt + E + 1;
    const int k = R / M;
    for (int t = tid >> 5; t < M; t += nt >> 5) {
      uint32_t v[16];
      router_load<16>(gate.logits + static_cast<int64_t>(t) * gate.ld, gate.E_route, lane, v);
      int e;
      float w;
      router_select_rounds<16>(v, gate.topk_sel, lane, &e, &w);
      if (lane >= gate.topk_sel && lane < gate.topk_sel + gate.n_shared)
        e = gate.shared_id + lane - gate.topk_sel;
      if (lane < k) sid[t * k + lane] = e;
    }
    __syncthreads();
    for (int r = tid; r < R; r += nt) {
      const int v = sid[r];
      if (v >= 0 && v < E) atomicAdd(&cnt[v], 1);
    }
    ids = nullptr;
    R = 0;   // counted
  }
  __syncthreads();
  // 16-byte loads, four in flight per thread before any count is added
  // (topk_ids is 256-byte aligned: the library checks every pointer)
  const int R4 = R >> 2;
  const int4* ids4 = reinterpret_cast<const int4*>(ids);
  auto add = [&](int v) {
    if (v >= 0 && v < E) atomicAdd(&cnt[v], 1);
  };
  for (int q0 = tid; q0 < R4; q0 += 4 * nt) {
    int4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q = q0 + j * nt;
      v[j] = q < R4 ? __ldg(ids4 + q) : make_int4(-1, -1, -1, -1);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      add(v[j].x);
      add(v[j].y);
      add(v[j].z);
      add(v[j].w);
    }
  }
  for (int r = 4 * R4 + tid; r < R; r += nt) add(__ldg(ids + r));
  __syncthreads();
  if (tid < 32) {   // exclusive scan of the block counts, in place
    // lane l owns experts [l * per, (l + 1) * per): one warp scan of the lane sums
    const int per = (E + 31) >> 5, e0 = lane * per, e1 = min(e0 + per, E);
    int sum = 0;
    for (int e = e0; e < e1; ++e) sum += (cnt[e] + bn - 1) / bn;
    int x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    int run = x - sum;
    for (int e = e0; e < e1; ++e) {
      const int nb = (cnt[e] + bn - 1) / bn;
      cnt[e] = run;
      run += nb;
    }
    if (lane == 31) cnt[E] = x;
  }
  __syncthreads();
  const int nblk = cnt[E];
  for (int e = tid; e < E; e += nt)
    for (int b = cnt[e]; b < cnt[e + 1] && b < kLocalMaxBlocks; ++b)
      blk_expert[b] = static_cast<uint16_t>(e);
  __syncthreads();
  return nblk;
}

template <class Args>
__device__ __forceinline__ void tile_coords(int t, const Args& a, int& m_blk, int& n_tile) {
  if (a.stage == 1 || a.n_group_log2 < 0) {
    m_blk = t / a.n_tiles;
    n_tile = t % a.n_tiles;
  } else {
    const int g = t / (a.num_blocks << a.n_group_log2);
    const int r = t - g * (a.num_blocks << a.n_group_log2);
    m_blk = r >> a.n_group_log2;
    n_tile = (g << a.n_group_log2) + (r & ((1 << a.n_group_log2) - 1));
  }
}

// This CTA's tiles t = blockIdx.x + i * gridDim.x that hold routes, in order.
// A tile holds routes iff its route block starts below the padded route count,
// so the walk needs no memory access. Route blocks are walked from the last
// one down: shared experts are appended after the routed ones, so their
// blocks (every token's route, the largest segments) are scheduled first,
// and the longest work starts in the first wave. With kExpert (the
// producer, the only role that addresses weights) the expert id of the next
// tile is loaded one tile ahead, off its critical path; the other roles
// never load it (e = 0).
template <class Args, bool kExpert = true>
struct TileSeq {
  int t, m_blk, n_tile, e;
  bool valid;
  int nt, nm, nn, ne;
  bool nvalid;

  __device__ __forceinline__ static bool find(int& t, int& m, int& n, const Args& a, int total,
                                              int P, int bn) {
    for (; t < total; t += gridDim.x) {
      tile_coords(t, a, m, n);
      if (m * bn < P) {
        m = P / bn - 1 - m;   // last route block first
        return true;
      }
    }
    return false;
  }
  __device__ __forceinline__ void init(const Args& a, int total, int P, int bn) {
    t = blockIdx.x;
    valid = find(t, m_blk, n_tile, a, total, P, bn);
    e = kExpert && valid ? expert_checked(a, __ldg(a.block_expert + m_blk)) : 0;
    nt = t + gridDim.x;
    nvalid = valid && find(nt, nm, nn, a, total, P, bn);
    ne = kExpert && nvalid ? __ldg(a.block_expert + nm) : 0;   // checked in next()
  }
  __device__ __forceinline__ void next(const Args& a, int total, int P, int bn) {
    t = nt; m_blk = nm; n_tile = nn; valid = nvalid;
    e = kExpert && valid ? expert_checked(a, ne) : 0;
    nt = t + gridDim.x;
    nvalid = valid && find(nt, nm, nn, a, total, P, bn);
    ne = kExpert && nvalid ? __ldg(a.block_expert + nm) : 0;   // checked in next()
  }
};


// ------------------------------------------------------------ split walk
// With few tiles (decode) whole tiles leave CTAs idle in a partial last
// wave. SplitSeq instead gives every CTA an equal, contiguous share of the
// T * kblocks k-blocks of the T tiles (tiles route-block major, last route
// block first) when T < kSplitMaxWaves * G for a grid of G CTAs: CTA c takes
// k-blocks [c * L, (c + 1) * L) with L = ceil(T * kblocks / G), cut at tile
// boundaries into units (tile, K range). A tile whose K range spans CTAs
// f..l is computed in l - f + 1 parts. Stage 2 adds every part to the
// accumulator like a whole tile (its epilogue is a sum); stage 1 adds the
// parts into split slot f (at most one split tile starts in a CTA's range)
// and the part that arrives last runs the epilogue from the slot. With more
// tiles the CTAs walk whole tiles t = blockIdx.x + i * gridDim.x. Stage-1
// tiles are route-block major, so the tiles that hold routes are the first
// (P / bn) * n_tiles in either stage's numbering here.
constexpr int kSplitMaxWaves = 8;

template <class Args, bool kExpert = true>
struct SplitSeq {
  int m_blk, n_tile, e, kb0, kb1, slot, parts;   // the current unit
  bool valid;
  int nm, nn, ne, nkb0, nkb1, nslot, nparts;     // the next one
  bool nvalid;
  int pos, end;   // walk cursor: next k-block (split walk) or next tile, and the end
  int kblocks, pblk, L;
  bool split;

  __device__ __forceinline__ bool take(int& m, int& n, int& k0, int& k1, int& sl, int& np,
                                       const Args& a) {
    if (pos >= end) return false;
    int tt;
    if (split) {
      tt = pos / kblocks;
      k0 = pos - tt * kblocks;
      k1 = min(kblocks, k0 + (end - pos));
      pos += k1 - k0;
      const int f = tt * kblocks / L, l = ((tt + 1) * kblocks - 1) / L;
      np = l - f + 1;
      sl = np > 1 ? f : -1;
    } else {
      tt = pos;
      pos += gridDim.x;
      k0 = 0; k1 = kblocks; sl = -1; np = 1;
    }
    m = pblk - 1 - tt / a.n_tiles;   // last route block first
    n = tt % a.n_tiles;
    return true;
  }
  __device__ __forceinline__ void init(const Args& a, int P, int bn, int kb) {
    kblocks = kb;
    pblk = P / bn;
    const int T = pblk * a.n_tiles;
    const int G = gridDim.x;
    split = T > 0 && T < kSplitMaxWaves * G && G <= kSplitSlots;
    if (split) {
      const int N = T * kb;
      L = (N + G - 1) / G;
      pos = min(N, static_cast<int>(blockIdx.x) * L);
      end = min(N, pos + L);
    } else {
      L = 1;
      pos = blockIdx.x;
      end = T;
    }
    valid = take(m_blk, n_tile, kb0, kb1, slot, parts, a);
    e = kExpert && valid ? expert_checked(a, __ldg(a.block_expert + m_blk)) : 0;
    nvalid = valid && take(nm, nn, nkb0, nkb1, nslot, nparts, a);
    ne = kExpert && nvalid ? __ldg(a.block_expert + nm) : 0;   // checked in next()
  }
  __device__ __forceinline__ void next(const Args& a) {
    m_blk = nm; n_tile = nn; kb0 = nkb0; kb1 = nkb1; slot = nslot; parts = nparts;
    valid = nvalid;
    e = kExpert && valid ? expert_checked(a, ne) : 0;
    nvalid = valid && take(nm, nn, nkb0, nkb1, nslot, nparts, a);
    ne = kExpert && nvalid ? __ldg(a.block_expert + nm) : 0;   // checked in next()
  }
};


// Uniform access for the kernels: a TileSeq unit always covers the whole K
// range (constant 0 / kblocks, so kernels using it compile as before).
template <class Args, bool X>
__device__ __forceinline__ void seq_init(TileSeq<Args, X>& q, const Args& a, int total, int P,
                                         int bn, int) { q.init(a, total, P, bn); }
template <class Args, bool X>
__device__ __forceinline__ void seq_init(SplitSeq<Args, X>& q, const Args& a, int, int P, int bn,
                                         int kb) { q.init(a, P, bn, kb); }
template <class Args, bool X>
__device__ __forceinline__ void seq_next(TileSeq<Args, X>& q, const Args& a, int total, int P,
                                         int bn) { q.next(a, total, P, bn); }
template <class Args, bool X>
__device__ __forceinline__ void seq_next(SplitSeq<Args, X>& q, const Args& a, int, int, int) {
  q.next(a);
}
template <class Args, bool X>
__device__ __forceinline__ int seq_kb0(const TileSeq<Args, X>&) { return 0; }
template <class Args, bool X>
__device__ __forceinline__ int seq_kb0(const SplitSeq<Args, X>& q) { return q.kb0; }
template <class Args, bool X>
__device__ __forceinline__ int seq_kb1(const TileSeq<Args, X>&, int kblocks) { return kblocks; }
template <class Args, bool X>
__device__ __forceinline__ int seq_kb1(const SplitSeq<Args, X>& q, int) { return q.kb1; }

}  // namespace moe

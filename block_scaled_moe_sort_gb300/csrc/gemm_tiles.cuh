// Tile walk shared by the grouped GEMM kernels: a tile is (route block,
// weight-row tile); stage 1 walks route-block major (the n-tiles of a block
// reuse its activation rows), stage 2 in groups of 2^n_group_log2 feature tiles,
// route-block major inside a group (the FP32 reductions of concurrently
// running tiles stay in the group's slice of the accumulator, i.e. in L2,
// and the intermediate is read once per group).
#pragma once
#include <cstdint>
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

// Expert of route block m. The sort writes ids in [0, E) for every block
// below the padded route count; any other value means a corrupted route
// list: it is reported through the status word (kDevBadExpert) and replaced
// by expert 0, so no weight access leaves the weight arrays.
template <class Args>
__device__ __forceinline__ int block_expert_checked(const Args& a, int m) {
  const int e = __ldg(a.block_expert + m);
  if (static_cast<unsigned>(e) < static_cast<unsigned>(a.E)) return e;
  if (a.status) atomicOr(a.status, kDevBadExpert);
  return 0;
}

template <class Args>
__device__ __forceinline__ void tile_coords(int t, const Args& a, int& m_blk, int& n_tile) {
  if (a.stage == 1) {
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
// so the walk needs no memory access; the expert id of the next tile is
// loaded one tile ahead, off the critical path of every role.
template <class Args>
struct TileSeq {
  int t, m_blk, n_tile, e;
  bool valid;
  int nt, nm, nn, ne;
  bool nvalid;

  __device__ __forceinline__ static bool find(int& t, int& m, int& n, const Args& a, int total,
                                              int P, int bn) {
    for (; t < total; t += gridDim.x) {
      tile_coords(t, a, m, n);
      if (m * bn < P) return true;
    }
    return false;
  }
  __device__ __forceinline__ void init(const Args& a, int total, int P, int bn) {
    t = blockIdx.x;
    valid = find(t, m_blk, n_tile, a, total, P, bn);
    e = valid ? block_expert_checked(a, m_blk) : -1;
    nt = t + gridDim.x;
    nvalid = valid && find(nt, nm, nn, a, total, P, bn);
    ne = nvalid ? block_expert_checked(a, nm) : -1;
  }
  __device__ __forceinline__ void next(const Args& a, int total, int P, int bn) {
    t = nt; m_blk = nm; n_tile = nn; e = ne; valid = nvalid;
    nt = t + gridDim.x;
    nvalid = valid && find(nt, nm, nn, a, total, P, bn);
    ne = nvalid ? block_expert_checked(a, nm) : -1;
  }
};


// ------------------------------------------------------ stage-1 tail split
// With few tiles (decode) the last, partial wave of stage-1 tiles leaves most
// CTAs idle. SplitSeq walks stage-1 work units instead: with T tiles on a grid
// of G CTAs, W = T / G whole waves and r = T - W * G tiles left over, the r
// tiles are split into S = min(G / r, kblocks, kSplitMaxParts) K ranges when
// W < kSplitMaxWaves. Units [0, W * G) are whole tiles; unit W * G + v is K
// range v % S of tile W * G + v / S, whose partial sums go to slot v / S of
// the split buffer (the range that finishes last runs the epilogue). Stage-1
// tiles are route-block major, so the tiles that hold routes are the first
// (P / bn) * n_tiles.
constexpr int kSplitMaxWaves = 2;
constexpr int kSplitMaxParts = 8;

template <class Args>
struct SplitSeq {
  int t, m_blk, n_tile, e, kb0, kb1, slot;
  bool valid;
  int nt, nm, nn, ne, nkb0, nkb1, nslot;
  bool nvalid;
  int wg, S, U, kblocks;

  __device__ __forceinline__ bool locate(int u, int& m, int& n, int& k0, int& k1, int& sl,
                                         const Args& a) const {
    if (u >= U) return false;
    int tt;
    if (u < wg) {
      tt = u; k0 = 0; k1 = kblocks; sl = -1;
    } else {
      const int v = u - wg, part = v % S;
      tt = wg + v / S;
      k0 = part * kblocks / S;
      k1 = (part + 1) * kblocks / S;
      sl = v / S;
    }
    m = tt / a.n_tiles;
    n = tt % a.n_tiles;
    return true;
  }
  __device__ __forceinline__ void init(const Args& a, int P, int bn, int kb) {
    kblocks = kb;
    const int T = (P / bn) * a.n_tiles;
    const int G = gridDim.x;
    const int W = T / G, r = T - W * G;
    int parts = 1;
    if (W < kSplitMaxWaves && r > 0 && r <= kSplitSlots) parts = min(min(G / r, kblocks), kSplitMaxParts);
    if (parts > 1) { S = parts; wg = W * G; U = wg + r * parts; } else { S = 1; wg = T; U = T; }
    t = blockIdx.x;
    valid = locate(t, m_blk, n_tile, kb0, kb1, slot, a);
    e = valid ? block_expert_checked(a, m_blk) : -1;
    nt = t + gridDim.x;
    nvalid = valid && locate(nt, nm, nn, nkb0, nkb1, nslot, a);
    ne = nvalid ? block_expert_checked(a, nm) : -1;
  }
  __device__ __forceinline__ void next(const Args& a) {
    t = nt; m_blk = nm; n_tile = nn; e = ne; kb0 = nkb0; kb1 = nkb1; slot = nslot;
    valid = nvalid;
    nt = t + gridDim.x;
    nvalid = valid && locate(nt, nm, nn, nkb0, nkb1, nslot, a);
    ne = nvalid ? block_expert_checked(a, nm) : -1;
  }
};


// Uniform access for the kernels: a TileSeq unit always covers the whole K
// range (constant 0 / kblocks, so kernels using it compile as before).
template <class Args>
__device__ __forceinline__ void seq_init(TileSeq<Args>& q, const Args& a, int total, int P, int bn,
                                         int) { q.init(a, total, P, bn); }
template <class Args>
__device__ __forceinline__ void seq_init(SplitSeq<Args>& q, const Args& a, int, int P, int bn,
                                         int kb) { q.init(a, P, bn, kb); }
template <class Args>
__device__ __forceinline__ void seq_next(TileSeq<Args>& q, const Args& a, int total, int P,
                                         int bn) { q.next(a, total, P, bn); }
template <class Args>
__device__ __forceinline__ void seq_next(SplitSeq<Args>& q, const Args& a, int, int, int) {
  q.next(a);
}
template <class Args>
__device__ __forceinline__ int seq_kb0(const TileSeq<Args>&) { return 0; }
template <class Args>
__device__ __forceinline__ int seq_kb0(const SplitSeq<Args>& q) { return q.kb0; }
template <class Args>
__device__ __forceinline__ int seq_kb1(const TileSeq<Args>&, int kblocks) { return kblocks; }
template <class Args>
__device__ __forceinline__ int seq_kb1(const SplitSeq<Args>& q, int) { return q.kb1; }

}  // namespace moe

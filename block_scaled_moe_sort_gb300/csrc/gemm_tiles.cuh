// Tile walk shared by the grouped GEMM kernels: a tile is (route block,
// weight-row tile); stage 1 walks route-block major (the n-tiles of a block
// reuse its activation rows), stage 2 feature-tile major (the FP32
// reductions of concurrently running tiles stay in one slice of the
// accumulator, i.e. in L2).
#pragma once
#include <cstdint>

namespace moe {

template <class Args>
__device__ __forceinline__ void tile_coords(int t, const Args& a, int& m_blk, int& n_tile) {
  if (a.stage == 1) {
    m_blk = t / a.n_tiles;
    n_tile = t % a.n_tiles;
  } else {
    n_tile = t / a.num_blocks;
    m_blk = t % a.num_blocks;
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
    e = valid ? __ldg(a.block_expert + m_blk) : -1;
    nt = t + gridDim.x;
    nvalid = valid && find(nt, nm, nn, a, total, P, bn);
    ne = nvalid ? __ldg(a.block_expert + nm) : -1;
  }
  __device__ __forceinline__ void next(const Args& a, int total, int P, int bn) {
    t = nt; m_blk = nm; n_tile = nn; e = ne; valid = nvalid;
    nt = t + gridDim.x;
    nvalid = valid && find(nt, nm, nn, a, total, P, bn);
    ne = nvalid ? __ldg(a.block_expert + nm) : -1;
  }
};

}  // namespace moe

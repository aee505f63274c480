// Route sort of the fused MoE layer: a stable counting sort of the
// token-expert routes by expert id, each expert's segment padded to a
// multiple of block_m ("the sorter" of AITER #5609 "Add DeepSeek V4.1 Flash
// TP4 gfx950 MoE tuning", Performance on the measured runtime; its block size
// must equal the GEMM block, Commands run).
//
// One CTA of 32 warps. Each warp owns a contiguous slice of the routes, so
// stability falls out of (warp order, then order inside the warp):
//   pass 1  per-warp expert histogram: __match_any_sync groups the lanes that
//           hold the same expert; the group leader adds the group size to
//           the warp's private counter row in shared memory;
//   scan    per expert, exclusive prefix over warps, then an exclusive scan
//           of the padded totals over experts gives the segment starts;
//   pass 2  the same walk again; a route's position is its expert's start +
//           its warp's prefix + its rank among equal lanes below it.
#include <cstdint>
#include "common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kSortWarps = 32;
constexpr int kSortThreads = kSortWarps * 32;

__global__ void __launch_bounds__(kSortThreads, 1)
    sort_routes_kernel(const int32_t* __restrict__ ids, const float* __restrict__ wts, int R,
                       int E, int bm, int64_t p_max, int32_t* __restrict__ sorted_route,
                       float* __restrict__ sorted_w, int32_t* __restrict__ block_expert,
                       int32_t* __restrict__ expert_off, int32_t* __restrict__ num_padded,
                       int32_t* __restrict__ route_pos, int32_t* __restrict__ status) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                          // [kSortWarps][E]
  int32_t* off = sm + kSortWarps * E;         // [E + 1]
  int32_t* tot = off + E + 1;                 // [E]
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0 && status) status[0] = 0;
  for (int i = tid; i < kSortWarps * E; i += kSortThreads) cnt[i] = 0;
  __syncthreads();

  const int chunk = (R + kSortWarps - 1) / kSortWarps;
  const int r0 = min(R, w * chunk), r1 = min(R, r0 + chunk);
  int32_t* my = cnt + w * E;

  for (int base = r0; base < r1; base += 32) {
    const int r = base + lane;
    const bool in = r < r1;
    const int e = in ? __ldg(ids + r) : -1;
    const bool valid = in && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid && lane == __ffs(peers) - 1) my[e] += __popc(peers);
  }
  __syncthreads();

  for (int e = tid; e < E; e += kSortThreads) {
    int s = 0;
    for (int ww = 0; ww < kSortWarps; ++ww) {
      const int c = cnt[ww * E + e];
      cnt[ww * E + e] = s;
      s += c;
    }
    tot[e] = s;
  }
  __syncthreads();
  if (w == 0) {
    int running = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int v = e < E ? (tot[e] + bm - 1) / bm * bm : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (e < E) off[e] = running + x - v;
      running += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) off[E] = running;
  }
  __syncthreads();
  const int P = off[E];

  for (int base = r0; base < r1; base += 32) {
    const int r = base + lane;
    const bool in = r < r1;
    const int e = in ? __ldg(ids + r) : -1;
    const bool valid = in && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid) {
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int p = off[e] + my[e] + rank;
      sorted_route[p] = r;
      sorted_w[p] = __ldg(wts + r);
      if (route_pos) route_pos[r] = p;
    } else if (in && route_pos) {
      route_pos[r] = -1;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
  }

  // pads inside each segment, block -> expert map, segment starts
  for (int e = tid; e < E; e += kSortThreads) {
    const int lo = off[e], hi = off[e + 1];
    for (int p = lo + tot[e]; p < hi; ++p) {
      sorted_route[p] = R;
      sorted_w[p] = 0.f;
    }
    for (int b = lo / bm; b < hi / bm; ++b) block_expert[b] = e;
    expert_off[e] = lo;
  }
  if (tid == 0) {
    expert_off[E] = P;
    num_padded[0] = P;
  }
  // tail beyond P
  for (int64_t p = P + tid; p < p_max; p += kSortThreads) {
    sorted_route[p] = R;
    sorted_w[p] = 0.f;
  }
  for (int64_t b = P / bm + tid; b < p_max / bm; b += kSortThreads) block_expert[b] = -1;
}

size_t sort_smem_bytes(int E) { return sizeof(int32_t) * (size_t)(kSortWarps * E + 2 * E + 1); }

cudaError_t launch_sort(const int32_t* ids, const float* wts, int R, int E, int bm, int64_t p_max,
                        int32_t* sorted_route, float* sorted_w, int32_t* block_expert,
                        int32_t* expert_off, int32_t* num_padded, int32_t* route_pos,
                        int32_t* status, cudaStream_t s) {
  const size_t smem = sort_smem_bytes(E);
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(&sort_routes_kernel),
                                     static_cast<int>(sort_smem_bytes(kMaxExperts)));
  if (err != cudaSuccess) return err;
  sort_routes_kernel<<<1, kSortThreads, smem, s>>>(ids, wts, R, E, bm, p_max, sorted_route,
                                                   sorted_w, block_expert, expert_off,
                                                   num_padded, route_pos, status);
  return cudaGetLastError();
}

}  // namespace moe

// Route sort of the fused MoE layer: a stable counting sort of the
// token-expert routes by expert id, each expert's segment padded to a
// multiple of block_m ("the sorter" of AITER #5609 "Add DeepSeek V4.1 Flash
// TP4 gfx950 MoE tuning", Performance on the measured runtime; its block size
// must equal the GEMM block, Commands run).
//
// Every CTA has 32 warps; each warp owns a contiguous slice of the routes
// and keeps its ids and weights in registers (kItems per lane), so the whole
// input is fetched with one round of independent loads. Stability falls out
// of (CTA order, warp order, order inside the warp):
//   count   per-warp expert histogram: a ballot per id bit groups the lanes
//           holding the same expert; the group leader adds the group size;
//   scan    per expert, exclusive prefix over warps (and over earlier CTAs),
//           then an exclusive scan of the padded totals gives segment starts;
//   scatter the same walk again; a route's position is its expert's start +
//           the prefix of everything before its warp + its rank among equal
//           lanes below it.
// Up to kRoutesPerCta routes every CTA of a small grid computes the whole
// layout (the counting is cheap) and writes only its share of the scattered
// stores, which dominate the cost. Beyond that a count kernel writes each
// CTA's expert histogram to a small scratch array and a scatter kernel (same
// grid) combines them. Launch shapes depend only on the route count.
#include <cstdint>
#include "common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"
#include "timeline.cuh"

MOE_TL_DEFINE(moe_tl_dump_sort)

namespace moe {
namespace {

constexpr int kWarps = 32;
constexpr int kThreads = kWarps * 32;
constexpr int kItems = 8;                                  // routes per lane
constexpr int kRoutesPerCta = kThreads * kItems;           // 8192

struct SortArgs {
  const int32_t* ids;
  const float* wts;
  int R, E, bm, bm_shift;
  int64_t p_max;
  int32_t* sorted_route;
  float* sorted_w;
  int32_t* block_expert;
  int32_t* expert_off;
  int32_t* num_padded;
  int32_t* route_pos;
  int32_t* status;
  int32_t* hist;   // [num_ctas][E] (multi-CTA only)
};

// Load this lane's routes of the CTA's slice: warp w owns routes
// [cta_base + w*chunk, cta_base + (w+1)*chunk), chunk a multiple of 32.
__device__ __forceinline__ void load_routes(const SortArgs& a, int cta_base, int cta_count,
                                            int chunk, int w, int lane, int (&e)[kItems],
                                            float (&wt)[kItems], bool load_w) {
  const int wb = cta_base + w * chunk;
  const int we = min(cta_base + cta_count, wb + chunk);
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int r = wb + it * 32 + lane;
    const bool in = r < we;
    const int v = in ? __ldg(a.ids + r) : -1;
    e[it] = (in && v >= 0 && v < a.E) ? v : -1;
    if (load_w) wt[it] = in ? __ldg(a.wts + r) : 0.f;
  }
}

// Lanes of the warp holding the same expert id as this lane (ids < 512, or
// -1 for "no route": those match only each other). Built from one ballot per
// id bit, which keeps the work on the ALU pipes (cheaper here than
// __match_any_sync).
__device__ __forceinline__ unsigned same_expert_lanes(int e) {
  const unsigned valid = __ballot_sync(0xffffffffu, e >= 0);
  unsigned m = e >= 0 ? valid : ~valid;
#pragma unroll
  for (int b = 0; b < 9; ++b) {
    const unsigned bit = __ballot_sync(0xffffffffu, (e >> b) & 1);
    m &= ((e >> b) & 1) ? bit : ~bit;
  }
  return m;
}

// Per-warp histogram of the lane-held routes into my[] (this warp's row).
// n_it = number of 32-route slots this warp actually holds (warp-uniform).
__device__ __forceinline__ void warp_count(const int (&e)[kItems], int32_t* my, int lane,
                                           int n_it) {
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    if (it >= n_it) break;
    const unsigned peers = same_expert_lanes(e[it]);
    if (e[it] >= 0 && lane == __ffs(peers) - 1) my[e[it]] += __popc(peers);
  }
}

// 32-route slots of [wb, we) (0 if the range is empty).
__device__ __forceinline__ int slots_held(int wb, int we) { return we > wb ? (we - wb + 31) >> 5 : 0; }

// Exclusive scan of padded totals over experts by warp 0 -> off[0..E].
__device__ __forceinline__ void scan_offsets(const int32_t* tot, int32_t* off, int E, int bm,
                                             int lane) {
  int running = 0;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    const int v = e < E ? (tot[e] + bm - 1) & ~(bm - 1) : 0;   // bm: power of two
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

// Writes the sorted position of this warp's routes. Every CTA walks every
// iteration (the running counts in my[] must advance), but iteration `it` of
// warp w is written only by CTA (w * kItems + it) % n_share == share, which
// spreads the scattered stores over the grid.
__device__ __forceinline__ void scatter(const SortArgs& a, const int (&e)[kItems],
                                        const float (&wt)[kItems], int cta_base, int cta_count,
                                        int chunk, int w, int lane, int32_t* my,
                                        const int32_t* off, int share, int n_share) {
  const int wb = cta_base + w * chunk;
  const int we = min(cta_base + cta_count, wb + chunk);   // end of this warp's slice
  const int n_it = slots_held(wb, we);
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    if (it >= n_it) break;
    const int r = wb + it * 32 + lane;
    const unsigned peers = same_expert_lanes(e[it]);
    if (((w * kItems + it) & (n_share - 1)) == share) {   // n_share is a power of two
      if (e[it] >= 0) {
        const int p = off[e[it]] + my[e[it]] + __popc(peers & ((1u << lane) - 1u));
        a.sorted_route[p] = r;
        a.sorted_w[p] = wt[it];
        if (a.route_pos) a.route_pos[r] = p;
      } else if (r < we && a.route_pos) {
        a.route_pos[r] = -1;                              // dropped route of this warp
      }
    }
    __syncwarp();
    if (e[it] >= 0 && lane == __ffs(peers) - 1) my[e[it]] += __popc(peers);
    __syncwarp();
  }
}

// Pads inside each segment, block -> expert map, segment starts and the
// tail, for the experts and positions owned by this CTA (expert e by CTA
// e % n_share). One warp per expert so that lanes write consecutive entries.
__device__ __forceinline__ void finish_layout(const SortArgs& a, const int32_t* off,
                                              const int32_t* tot, int share, int n_share) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int e = share + w * n_share; e < a.E; e += n_share * kWarps) {
    const int lo = off[e], hi = off[e + 1];
    for (int p = lo + tot[e] + lane; p < hi; p += 32) {
      a.sorted_route[p] = a.R;
      a.sorted_w[p] = 0.f;
    }
    for (int b = (lo >> a.bm_shift) + lane; b < (hi >> a.bm_shift); b += 32) a.block_expert[b] = e;
    if (lane == 0) a.expert_off[e] = lo;
  }
  const int P = off[a.E];
  if (share == 0 && tid == 0) {
    a.expert_off[a.E] = P;
    a.num_padded[0] = P;
  }
  const int64_t stride = static_cast<int64_t>(n_share) * kThreads;
  for (int64_t p = P + static_cast<int64_t>(share) * kThreads + tid; p < a.p_max; p += stride) {
    a.sorted_route[p] = a.R;
    a.sorted_w[p] = 0.f;
  }
  for (int64_t b = (P >> a.bm_shift) + static_cast<int64_t>(share) * kThreads + tid;
       b < (a.p_max >> a.bm_shift); b += stride)
    a.block_expert[b] = -1;
}

__device__ __forceinline__ int warp_chunk(int count) {
  return ((count + kWarps - 1) / kWarps + 31) / 32 * 32;
}

// R <= kRoutesPerCta: every CTA of the (small) grid computes the whole
// layout from all routes and writes only its share of it.
__global__ void __launch_bounds__(kThreads, 1) sort_small_kernel(const SortArgs a) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                      // [kWarps][E]
  int32_t* off = sm + kWarps * a.E;       // [E + 1]
  int32_t* tot = off + a.E + 1;           // [E]
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  pdl_launch_dependents();   // the next kernel waits for this one to finish anyway
  if (tid == 0) MOE_TL(0, 0);
  if (blockIdx.x == 0 && tid == 0 && a.status) a.status[0] = 0;
  const int chunk = warp_chunk(a.R);
  int e[kItems];
  float wt[kItems];
  load_routes(a, 0, a.R, chunk, w, lane, e, wt, true);
  for (int i = tid; i < kWarps * a.E; i += kThreads) cnt[i] = 0;
  __syncthreads();
  warp_count(e, cnt + w * a.E, lane, slots_held(w * chunk, min(a.R, (w + 1) * chunk)));
  __syncthreads();
  for (int x = tid; x < a.E; x += kThreads) {
    int s = 0;
    for (int ww = 0; ww < kWarps; ++ww) {
      const int c = cnt[ww * a.E + x];
      cnt[ww * a.E + x] = s;
      s += c;
    }
    tot[x] = s;
  }
  __syncthreads();
  if (w == 0) scan_offsets(tot, off, a.E, a.bm, lane);
  __syncthreads();
  scatter(a, e, wt, 0, a.R, chunk, w, lane, cnt + w * a.E, off, blockIdx.x, gridDim.x);
  finish_layout(a, off, tot, blockIdx.x, gridDim.x);
  if (tid == 0) MOE_TL(0, 7);
}

// Multi-CTA, pass 1: CTA c writes the expert histogram of its slice to hist[c].
__global__ void __launch_bounds__(kThreads, 1) sort_count_kernel(const SortArgs a) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                      // [kWarps][E]
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) MOE_TL(1, 0);
  const int base = blockIdx.x * kRoutesPerCta;
  const int count = min(kRoutesPerCta, a.R - base);
  const int chunk = warp_chunk(count);
  int e[kItems];
  float wt[kItems];
  load_routes(a, base, count, chunk, w, lane, e, wt, false);
  for (int i = tid; i < kWarps * a.E; i += kThreads) cnt[i] = 0;
  __syncthreads();
  warp_count(e, cnt + w * a.E, lane,
             slots_held(base + w * chunk, min(base + count, base + (w + 1) * chunk)));
  __syncthreads();
  for (int x = tid; x < a.E; x += kThreads) {
    int s = 0;
    for (int ww = 0; ww < kWarps; ++ww) s += cnt[ww * a.E + x];
    a.hist[static_cast<int64_t>(blockIdx.x) * a.E + x] = s;
  }
  if (tid == 0) MOE_TL(1, 7);
}

// Multi-CTA, pass 2: combine the histograms, then scatter; CTA 0 also writes
// the pads, the block map, the offsets and the tail.
__global__ void __launch_bounds__(kThreads, 1) sort_scatter_kernel(const SortArgs a) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                      // [kWarps][E]
  int32_t* off = sm + kWarps * a.E;       // [E + 1]
  int32_t* tot = off + a.E + 1;           // [E]
  int32_t* pre = tot + a.E;               // [E] routes of this expert in earlier CTAs
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  pdl_launch_dependents();
  if (tid == 0) MOE_TL(2, 0);
  if (blockIdx.x == 0 && tid == 0 && a.status) a.status[0] = 0;
  const int base = blockIdx.x * kRoutesPerCta;
  const int count = min(kRoutesPerCta, a.R - base);
  const int chunk = warp_chunk(count);
  int e[kItems];
  float wt[kItems];
  load_routes(a, base, count, chunk, w, lane, e, wt, true);
  for (int i = tid; i < kWarps * a.E; i += kThreads) cnt[i] = 0;
  for (int x = tid; x < a.E; x += kThreads) {
    int before = 0, all = 0;
    for (int c = 0; c < static_cast<int>(gridDim.x); ++c) {
      const int h = a.hist[static_cast<int64_t>(c) * a.E + x];
      if (c < static_cast<int>(blockIdx.x)) before += h;
      all += h;
    }
    pre[x] = before;
    tot[x] = all;
  }
  __syncthreads();
  warp_count(e, cnt + w * a.E, lane,
             slots_held(base + w * chunk, min(base + count, base + (w + 1) * chunk)));
  __syncthreads();
  for (int x = tid; x < a.E; x += kThreads) {
    int s = pre[x];
    for (int ww = 0; ww < kWarps; ++ww) {
      const int c = cnt[ww * a.E + x];
      cnt[ww * a.E + x] = s;
      s += c;
    }
  }
  if (w == 0) scan_offsets(tot, off, a.E, a.bm, lane);
  __syncthreads();
  scatter(a, e, wt, base, count, chunk, w, lane, cnt + w * a.E, off, 0, 1);
  finish_layout(a, off, tot, blockIdx.x, gridDim.x);
  if (tid == 0) MOE_TL(2, 7);
}

size_t smem_bytes(int E) { return sizeof(int32_t) * (static_cast<size_t>(kWarps) * E + 3 * E + 1); }

}  // namespace

int sort_num_ctas(int R) { return R <= kRoutesPerCta ? 1 : (R + kRoutesPerCta - 1) / kRoutesPerCta; }

size_t sort_scratch_bytes(int R, int E) {
  const int n = sort_num_ctas(R);
  return n > 1 ? sizeof(int32_t) * static_cast<size_t>(n) * E : 0;
}

cudaError_t launch_sort(const int32_t* ids, const float* wts, int R, int E, int bm, int64_t p_max,
                        int32_t* sorted_route, float* sorted_w, int32_t* block_expert,
                        int32_t* expert_off, int32_t* num_padded, int32_t* route_pos,
                        int32_t* status, int32_t* scratch, cudaStream_t s) {
  int bm_shift = 0;
  while ((1 << bm_shift) < bm) ++bm_shift;
  SortArgs a{ids, wts, R, E, bm, bm_shift, p_max, sorted_route, sorted_w, block_expert,
             expert_off, num_padded, route_pos, status, scratch};
  const size_t smem = smem_bytes(E);
  const int n = sort_num_ctas(R);
  if (n == 1) {
    cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(&sort_small_kernel),
                                       static_cast<int>(smem_bytes(kMaxExperts)));
    if (err != cudaSuccess) return err;
    // one CTA per ~256 routes shares the scattered stores (a power of two, at most 16)
    int grid = 1;
    while (grid < 16 && grid * 256 < R) grid <<= 1;
    sort_small_kernel<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
  }
  if (!scratch) return cudaErrorInvalidValue;
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(&sort_count_kernel),
                                     static_cast<int>(smem_bytes(kMaxExperts)));
  if (err != cudaSuccess) return err;
  err = ensure_smem_attr(reinterpret_cast<const void*>(&sort_scatter_kernel),
                         static_cast<int>(smem_bytes(kMaxExperts)));
  if (err != cudaSuccess) return err;
  sort_count_kernel<<<n, kThreads, smem, s>>>(a);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  sort_scatter_kernel<<<n, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

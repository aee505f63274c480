// Gating in front of the route sort: per token, the topk largest router
// logits (equal logits taken in ascending expert order, listed by descending
// logit) and their routing weights, the softmax over the selected logits;
// optionally a shared expert appended with weight 1 (AITER #5609 "Add
// DeepSeek V4.1 Flash TP4 gfx950 MoE tuning", Performance on the measured
// runtime, times the call including gating; the 385-expert top-7 layout with
// an always-selected shared expert is AITER #6286 "Retune gfx942 a16w4
// DSv4.1 tiles for Triton 3.8", first table).
//
// One warp per token: lane l holds logits l, l+32, ... in registers (one
// coalesced 128-byte load per 32 experts) as order-preserving integer keys,
// so each of the topk rounds picks the next expert with two warp
// reductions (largest key, then lowest expert holding it); lane j keeps
// pick j, and lanes 0..topk-1 form the softmax with one warp sum. The
// kernel reads each logit once: HBM-bound for large M, latency-bound for
// decode sizes.
#include <cmath>
#include <cstdint>
#include "common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kRouterWarps = 8;                    // tokens per CTA

// Order-preserving 32-bit key of a finite float (larger float, larger key);
// both zeros map to the key of +0 so that they tie, and key 0 is below every
// finite value (it marks absent and already picked experts).
__device__ __forceinline__ uint32_t logit_key(float f) {
  const uint32_t u = f == 0.f ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// SLOTS: logits per lane (32 * SLOTS >= E)
template <int SLOTS>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_topk_kernel(const float* __restrict__ logits, int M, int E, int ld, int topk,
                       int shared_id, int kout, int32_t* __restrict__ ids,
                       float* __restrict__ weights) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
  if (t >= M) return;
  const float* row = logits + static_cast<int64_t>(t) * ld;
  uint32_t v[SLOTS];   // keys of experts lane, lane + 32, ...
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int e = i * 32 + lane;
    v[i] = e < E ? logit_key(__ldg(row + e)) : 0u;
  }
  uint32_t mine = 0;   // lane j: key of pick j
  int mine_e = 0;
  for (int j = 0; j < topk; ++j) {
    // this lane's best remaining expert (slots in ascending e: ties keep the lower)
    uint32_t bk = 0;
    int be = 0;
#pragma unroll
    for (int i = 0; i < SLOTS; ++i)
      if (v[i] > bk) { bk = v[i]; be = i * 32 + lane; }
    // warp arg-max in two reductions: the largest key, then the lowest
    // expert among the lanes that hold it
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const int win = static_cast<int>(
        __reduce_min_sync(0xffffffffu, bk == kmax ? static_cast<uint32_t>(be) : 0xffffffffu));
    if (lane == j) { mine = kmax; mine_e = win; }
    if ((win & 31) == lane) {
#pragma unroll
      for (int i = 0; i < SLOTS; ++i)
        if (i == (win >> 5)) v[i] = 0u;
    }
  }
  // softmax over the picks, shifted by the largest (pick 0)
  const float top = key_logit(__shfl_sync(0xffffffffu, mine, 0));
  const float ex = lane < topk ? expf(key_logit(mine) - top) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const int64_t base = static_cast<int64_t>(t) * kout;
  if (lane < topk) {
    ids[base + lane] = mine_e;
    weights[base + lane] = ex / sum;
  } else if (lane == topk && shared_id >= 0) {
    ids[base + lane] = shared_id;
    weights[base + lane] = 1.f;
  }
}

}  // namespace

cudaError_t launch_router_topk(const float* logits, int M, int E, int ld, int topk,
                               int shared_id, int32_t* ids, float* weights, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  const int kout = topk + (shared_id >= 0 ? 1 : 0);
  const int grid = (M + kRouterWarps - 1) / kRouterWarps;
  const dim3 block(kRouterWarps * 32);
  if (E <= 128)
    router_topk_kernel<4><<<grid, block, 0, s>>>(logits, M, E, ld, topk, shared_id, kout, ids,
                                                 weights);
  else if (E <= 256)
    router_topk_kernel<8><<<grid, block, 0, s>>>(logits, M, E, ld, topk, shared_id, kout, ids,
                                                 weights);
  else if (E <= 384)
    router_topk_kernel<12><<<grid, block, 0, s>>>(logits, M, E, ld, topk, shared_id, kout, ids,
                                                  weights);
  else
    router_topk_kernel<kMaxExperts / 32><<<grid, block, 0, s>>>(logits, M, E, ld, topk, shared_id,
                                                                kout, ids, weights);
  return cudaGetLastError();
}

}  // namespace moe

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
#include "router_warp.cuh"

namespace moe {
namespace {

constexpr int kRouterWarps = 8;                    // tokens per CTA

// One warp per token (measured: as fast as persistent warps that load the
// next token's logits ahead, and faster than a 64-bit shuffle arg-max; the
// selection's instruction count, not the loads, bounds the kernel at large M).
template <int SLOTS>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_topk_kernel(const float* __restrict__ logits, int M, int E, int ld, int topk,
                       int shared_id, int n_shared, int kout, int32_t* __restrict__ ids,
                       float* __restrict__ weights) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
  if (t >= M) return;
  uint32_t v[SLOTS];
  router_load<SLOTS>(logits + static_cast<int64_t>(t) * ld, E, lane, v);
  int e;
  float w;
  router_select<SLOTS>(v, topk, lane, &e, &w);
  const int64_t base = static_cast<int64_t>(t) * kout;
  if (lane < topk) {
    ids[base + lane] = e;
    weights[base + lane] = w;
  } else if (lane < topk + n_shared) {   // the shared expert's columns
    ids[base + lane] = shared_id + lane - topk;
    weights[base + lane] = 1.f;
  }
}

}  // namespace

cudaError_t launch_router_topk(const float* logits, int M, int E, int ld, int topk,
                               int shared_id, int n_shared, int32_t* ids, float* weights,
                               cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (shared_id < 0) n_shared = 0;
  const int kout = topk + n_shared;
  const int grid = (M + kRouterWarps - 1) / kRouterWarps;
  const dim3 block(kRouterWarps * 32);
  switch (router_slots(E)) {
    case 4:
      router_topk_kernel<4><<<grid, block, 0, s>>>(logits, M, E, ld, topk, shared_id, n_shared, kout, ids,
                                                   weights);
      break;
    case 8:
      router_topk_kernel<8><<<grid, block, 0, s>>>(logits, M, E, ld, topk, shared_id, n_shared, kout, ids,
                                                   weights);
      break;
    case 12:
      router_topk_kernel<12><<<grid, block, 0, s>>>(logits, M, E, ld, topk, shared_id, n_shared, kout, ids,
                                                    weights);
      break;
    default:
      router_topk_kernel<16><<<grid, block, 0, s>>>(logits, M, E, ld, topk, shared_id, n_shared, kout, ids,
                                                     weights);
  }
  return cudaGetLastError();
}

}  // namespace moe

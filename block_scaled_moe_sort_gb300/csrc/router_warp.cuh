// Gating of one token by one warp: the topk largest router logits (equal
// logits taken in ascending expert order, listed by descending logit) and
// their routing weights, the softmax over the selected logits (AITER #5609
// "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning", Performance on the
// measured runtime, times the call including gating; the weights are the
// softmax over the picks, as in the pages' synthetic routing).
//
// Lane l holds logits l, l+32, ... as order-preserving integer keys and
// keeps its three largest; each of the topk rounds picks the largest head
// key of the warp (the lowest expert among equal keys); lane j keeps pick j.
// Used by the standalone gating kernel and by the decode front kernel of the
// gated call.
#pragma once
#include <cstdint>

namespace moe {

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

// Keys of row `row` (E logits) for this lane: experts lane, lane + 32, ...
template <int SLOTS>
__device__ __forceinline__ void router_load(const float* row, int E, int lane,
                                            uint32_t (&v)[SLOTS]) {
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int e = i * 32 + lane;
    v[i] = e < E ? logit_key(__ldg(row + e)) : 0u;
  }
}

// This lane's kCache largest keys in (key descending, slot ascending) order,
// among the keys that come after (lk, ls) in that order (all keys for
// lk = ~0u, ls = -1); empty entries have key 0.
constexpr int kRouterCache = 3;
template <int SLOTS>
__device__ __forceinline__ void router_lane_top(const uint32_t (&v)[SLOTS], uint32_t lk, int ls,
                                                uint32_t (&hk)[kRouterCache],
                                                int (&hs)[kRouterCache]) {
#pragma unroll
  for (int c = 0; c < kRouterCache; ++c) { hk[c] = 0u; hs[c] = 0; }
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const uint32_t k = v[i];
    if (!(k < lk || (k == lk && i > ls))) continue;
    // insertion after the entries >= k (an equal key of a lower slot stays first)
    if (k > hk[kRouterCache - 1]) {
#pragma unroll
      for (int c = kRouterCache - 1; c > 0; --c) {
        if (k > hk[c - 1]) { hk[c] = hk[c - 1]; hs[c] = hs[c - 1]; }
        else if (k > hk[c]) { hk[c] = k; hs[c] = i; }
      }
      if (k > hk[0]) { hk[0] = k; hs[0] = i; }
    }
  }
}

// Selects the topk experts of the keys in v. Lane j < topk gets pick j: its
// expert in *expert and its routing weight in *weight.
// Each lane first keeps its three largest keys; every round takes the warp's
// largest head key (one reduction; a second one, over expert ids, only when
// several lanes hold that key) and the winning lane moves to its next key,
// rescanning its slots after the keys it has given (rare: a lane holding
// more than three of the picks).
template <int SLOTS>
__device__ __forceinline__ void router_select(const uint32_t (&v)[SLOTS], int topk, int lane,
                                              int* expert, float* weight) {
  uint32_t hk[kRouterCache];
  int hs[kRouterCache];
  router_lane_top<SLOTS>(v, ~0u, -1, hk, hs);
  int left = kRouterCache;     // cached entries of this lane not yet given
  uint32_t mine = 0;           // lane j: key of pick j
  int mine_e = 0;
  for (int j = 0; j < topk; ++j) {
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, hk[0]);
    const uint32_t holders = __ballot_sync(0xffffffffu, hk[0] == kmax);
    int win;
    if (__popc(holders) == 1) {
      const int wl = __ffs(holders) - 1;
      win = __shfl_sync(0xffffffffu, hs[0], wl) * 32 + wl;
    } else {
      // equal largest keys in several lanes: the lowest expert
      win = static_cast<int>(__reduce_min_sync(
          0xffffffffu, hk[0] == kmax ? static_cast<uint32_t>(hs[0] * 32 + lane) : 0xffffffffu));
    }
    if (lane == j) { mine = kmax; mine_e = win; }
    if ((win & 31) == lane) {
      const uint32_t lk = hk[0];
      const int ls = hs[0];
#pragma unroll
      for (int c = 0; c + 1 < kRouterCache; ++c) { hk[c] = hk[c + 1]; hs[c] = hs[c + 1]; }
      hk[kRouterCache - 1] = 0u;
      if (--left == 0) {
        router_lane_top<SLOTS>(v, lk, ls, hk, hs);
        left = kRouterCache;
      }
    }
  }
  // softmax over the picks, shifted by the largest (pick 0)
  const float top = key_logit(__shfl_sync(0xffffffffu, mine, 0));
  const float ex = lane < topk ? expf(key_logit(mine) - top) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  *expert = mine_e;
  *weight = ex / sum;
}

// Logits per lane for E experts (32 * slots >= E): 4, 8, 12 or 16.
__host__ __device__ constexpr int router_slots(int E) {
  return E <= 128 ? 4 : E <= 256 ? 8 : E <= 384 ? 12 : 16;
}

}  // namespace moe

// Gating of one token by one warp: the topk largest router logits (equal
// logits taken in ascending expert order, listed by descending logit) and
// their routing weights, the softmax over the selected logits (AITER #5609
// "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning", Performance on the
// measured runtime, times the call including gating; the weights are the
// softmax over the picks, as in the pages' synthetic routing).
//
// Lane l holds logits l, l+32, ... as order-preserving integer keys; each
// of the topk rounds picks the largest remaining key of the warp (the lowest
// expert among equal keys); lane j keeps pick j. Two forms with the same
// result: router_select keeps each lane's two largest keys (the standalone
// gating kernel, many tokens per launch), router_select_rounds scans the
// lane's keys once per pick (the gated decode front kernel and the GEMMs'
// local layout, a few tokens per CTA: measured 12 us faster per call at
// M=6 there, equal at M=12-24).
#pragma once
#include <cstdint>

namespace moe {

// Order-preserving 32-bit key of a finite float (larger float, larger key);
// both zeros map to the key of +0 so that they tie, and key 0 is below every
// finite value (it marks absent and already picked experts).
__device__ __forceinline__ uint32_t logit_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);                    // -0 + +0 = +0
  const uint32_t neg = static_cast<uint32_t>(static_cast<int32_t>(u) >> 31);
  return u ^ (neg | 0x80000000u);   // negative: all bits flipped; else the sign bit set
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

// Keeps (h0, s0) >= (h1, s1), the two largest (key, slot) seen in (key
// descending, slot ascending) order: slots come in ascending order, so an
// equal key never displaces an earlier one.
__device__ __forceinline__ void router_insert2(uint32_t k, int i, uint32_t& h0, int& s0,
                                               uint32_t& h1, int& s1) {
  const bool c0 = k > h0, c1 = k > h1;
  h1 = c0 ? h0 : (c1 ? k : h1);
  s1 = c0 ? s0 : (c1 ? i : s1);
  h0 = c0 ? k : h0;
  s0 = c0 ? i : s0;
}

// Selects the topk experts of the keys in v. Lane j < topk gets pick j: its
// expert in *expert and its routing weight in *weight.
// Each lane first keeps its two largest keys; every round takes the warp's
// largest head key (one reduction; a second one, over expert ids, only when
// several lanes hold that key) and the winning lane moves to its second key,
// or, having given both, rescans its slots for the two that follow the last
// one it gave.
template <int SLOTS>
__device__ __forceinline__ void router_select(const uint32_t (&v)[SLOTS], int topk, int lane,
                                              int* expert, float* weight) {
  uint32_t h0 = 0u, h1 = 0u;
  int s0 = 0, s1 = 0;
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) router_insert2(v[i], i, h0, s0, h1, s1);
  bool second = false;         // this lane has given one of its two cached keys
  uint32_t mine = 0;           // lane j: key of pick j
  int mine_e = 0;
  for (int j = 0; j < topk; ++j) {
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, h0);
    const uint32_t holders = __ballot_sync(0xffffffffu, h0 == kmax);
    int win;
    if (__popc(holders) == 1) {
      const int wl = __ffs(holders) - 1;
      win = __shfl_sync(0xffffffffu, s0, wl) * 32 + wl;
    } else {
      // equal largest keys in several lanes: the lowest expert
      win = static_cast<int>(__reduce_min_sync(
          0xffffffffu, h0 == kmax ? static_cast<uint32_t>(s0 * 32 + lane) : 0xffffffffu));
    }
    if (lane == j) { mine = kmax; mine_e = win; }
    if ((win & 31) == lane) {
      if (!second) {
        h0 = h1; s0 = s1;
        second = true;
      } else {
        // both cached keys given: the two that follow (h0, s0) in the order
        const uint32_t lk = h0;
        const int ls = s0;
        h0 = h1 = 0u;
        s0 = s1 = 0;
#pragma unroll
        for (int i = 0; i < SLOTS; ++i)
          if (v[i] < lk || (v[i] == lk && i > ls)) router_insert2(v[i], i, h0, s0, h1, s1);
        second = false;
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

// The same selection with one scan of the lane's keys per pick (two warp
// reductions per pick, no cached heads).
template <int SLOTS>
__device__ __forceinline__ void router_select_rounds(const uint32_t (&keys)[SLOTS], int topk,
                                                     int lane, int* expert, float* weight) {
  uint32_t v[SLOTS];
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) v[i] = keys[i];
  uint32_t mine = 0;   // lane j: key of pick j
  int mine_e = 0;
  for (int j = 0; j < topk; ++j) {
    // this lane's best remaining expert (slots in ascending e: ties keep the lower)
    uint32_t bk = 0;
    int be = 0;
#pragma unroll
    for (int i = 0; i < SLOTS; ++i)
      if (v[i] > bk) { bk = v[i]; be = i * 32 + lane; }
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

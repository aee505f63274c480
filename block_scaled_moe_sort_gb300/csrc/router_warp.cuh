// Gating of one token by one warp: the topk largest router logits (equal
// logits taken in ascending expert order, listed by descending logit) and
// their routing weights, the softmax over the selected logits (AITER #5609
// "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning", Performance on the
// measured runtime, times the call including gating; the weights are the
// softmax over the picks, as in the pages' synthetic routing).
//
// Lane l holds logits l, l+32, ... as order-preserving integer keys, so each
// of the topk rounds picks the next expert with two warp reductions (largest
// key, then lowest expert holding it); lane j keeps pick j. Used by the
// standalone gating kernel and by the decode front kernel of the gated call.
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

// Selects the topk experts of the keys in v (consumed). Lane j < topk gets
// pick j: its expert in *expert and its routing weight in *weight.
template <int SLOTS>
__device__ __forceinline__ void router_select(uint32_t (&v)[SLOTS], int topk, int lane,
                                              int* expert, float* weight) {
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
  *expert = mine_e;
  *weight = ex / sum;
}

// Logits per lane for E experts (32 * slots >= E): 4, 8, 12 or 16.
__host__ __device__ constexpr int router_slots(int E) {
  return E <= 128 ? 4 : E <= 256 ? 8 : E <= 384 ? 12 : 16;
}

}  // namespace moe

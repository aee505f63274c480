// Internal launch interface between the C-ABI front end (moe_mx.cu) and the
// kernel translation units. Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Gating input of a GEMM's local route layout (gated calls): router logits
// [M, ld] of E_route experts, topk_sel picks plus n_shared shared columns.
struct LocalGate {
  const float* logits;
  int ld, E_route, topk_sel, shared_id, n_shared;
};

// Sets the dynamic shared-memory limit of `func` once per device.
cudaError_t ensure_smem_attr(const void* func, int bytes);

int sort_num_ctas(int R);
size_t sort_scratch_bytes(int R, int E);
cudaError_t launch_sort(const int32_t* ids, const float* wts, int R, int E, int bm, int64_t p_max,
                        int32_t* sorted_route, float* sorted_w, int32_t* block_expert,
                        int32_t* expert_off, int32_t* num_padded, int32_t* route_pos,
                        int32_t* status, int32_t* scratch, cudaStream_t s);

cudaError_t launch_quant_act(const void* x, int M, int K, int ldx, uint8_t* q, uint8_t* scale,
                             cudaStream_t s);

cudaError_t launch_wait_selftest(int32_t* status, uint64_t timeout_ns, cudaStream_t s);

cudaError_t launch_router_topk(const float* logits, int M, int E, int ld, int topk,
                               int shared_id, int n_shared, int32_t* ids, float* weights,
                               cudaStream_t s);

cudaError_t launch_prepack_weights(const uint8_t* w, int E, int N, int K, uint8_t* out,
                                   bool a16, cudaStream_t s);
cudaError_t launch_dequant_a16w4(const uint8_t* w, const uint8_t* sf, int E, int N, int K,
                                 void* out, cudaStream_t s);
cudaError_t launch_prepack_scales(const uint8_t* scale, int E, int N, int K, uint8_t* out,
                                  cudaStream_t s);

// Gating inside the decode front kernel (the gated calls): router logits
// [M, ld] of E_route experts; topk_sel picks per token plus, with
// shared_id >= 0, n_shared shared-expert columns (ids shared_id,
// shared_id + 1, ..., weight 1); the ids and weights are written to
// ids_out / w_out [M, topk] as well.
struct FrontGating {
  const float* logits;
  int ld, E_route, topk_sel, shared_id, n_shared;
  int32_t* ids_out;
  float* w_out;
};

// Few routes (M * topk <= kFrontMaxRoutes): the sort and the gather in one
// launch; writes everything launch_sort and launch_gather_act write. With
// gate, the routes come from the router logits instead of ids / wts.
cudaError_t launch_front_tiny(bool a16, const void* x, const int32_t* ids, const float* wts, int M,
                              int H, int topk, int E, int bm, int64_t p_max,
                              int32_t* sorted_route, float* sorted_w, int32_t* block_expert,
                              int32_t* expert_off, int32_t* num_padded, int32_t* route_pos,
                              int32_t* status, void* act, uint8_t* act_sf, float* acc,
                              void* zero2, int64_t zero2_bytes, const FrontGating* gate,
                              cudaStream_t s);

// Writes each token's activation row to the sorted position of each of its
// routes (quantised to FP8 with scale atoms for a8w4, as BF16 for a16w4) and
// zeroes the FP32 accumulator [M, H] and zero2_bytes (a multiple of 16) at zero2.
cudaError_t launch_gather_act(bool a16, const void* x, int M, int H, int topk, int bm,
                              const int32_t* route_pos, void* act, uint8_t* act_sf, float* acc,
                              void* zero2, int64_t zero2_bytes, cudaStream_t s);

cudaError_t launch_finalize(const float* acc, int64_t n, void* out, cudaStream_t s);

struct GemmArgs {
  bool a16;
  int M, H, Ip, E, topk, bm;
  int prefetch1, prefetch2;  // weight L2 prefetch lead per stage in k-blocks (0 = default)
  int split;                 // split walk (a8w4): 0 = by the route bound, 1 = always, 2 = never
  int64_t p_max;
  const int32_t* topk_ids;   // the call's routing input (local layout at decode sizes)
  LocalGate gate;            // gated calls: router logits instead (topk_ids is then null)
  const int32_t* sorted_route;
  const float* sorted_w;
  const int32_t* block_expert;
  const int32_t* num_padded;
  const uint8_t* w1;
  const uint8_t* w1s;   // prepacked atoms
  const uint8_t* w2;
  const uint8_t* w2s;
  const void* act;      // gathered activations [p_max, H]
  const uint8_t* act_sf;
  void* inter;          // [p_max, Ip]
  uint8_t* inter_sf;
  float* acc;           // [M, H]
  float* split_part;    // split walk, stage 1: [kSplitSlots][block_m][128] FP32, zeroed per call
  int32_t* split_cnt;   // [kSplitSlots], zeroed per call
  int32_t* status;
};

// A grouped-GEMM launch with all host-side work (tensor-map encoding,
// attribute setup) done by prepare_*; launch_gemm only enqueues the kernel.
struct GemmPlan {
  alignas(64) unsigned char tmap_a[128];   // CUtensorMap of the weights
  alignas(64) unsigned char tmap_b[128];   // CUtensorMap of the route rows
  unsigned char args[256];                 // kernel argument block
  const void* kernel;
  int grid, threads, smem;
};
// tcgen05 block-scaled grouped GEMM, a8w4, stage 1 or 2.
cudaError_t prepare_gemm_mx(int stage, const GemmArgs& a, GemmPlan* plan);
// tcgen05 BF16 x (MXFP4 dequantised into TMEM) grouped GEMM, a16w4.
cudaError_t prepare_gemm_bf16w4(int stage, const GemmArgs& a, GemmPlan* plan);
cudaError_t launch_gemm(const GemmPlan& plan, cudaStream_t s);


}  // namespace moe

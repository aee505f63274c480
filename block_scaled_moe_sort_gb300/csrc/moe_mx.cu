// C-ABI front end of the fused MoE library: argument checks, workspace
// carving, block_m choice and the launch sequence of one layer call.
// Declarations and the full contract are in include/moe_mx.h.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <cuda_runtime.h>
#include "moe_mx.h"
#include "common.cuh"
#include "moe_internal.h"
#include "sm100_ptx.cuh"

namespace moe {

cudaError_t ensure_smem_attr(const void* func, int bytes) {
  // One flag per (device, function); the set of functions is small and fixed.
  struct Entry { const void* f; int dev; int bytes; };
  static Entry done[256];
  static int n_done = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].f == func && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
  err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err != cudaSuccess) return err;
  if (n_done < 256) done[n_done++] = Entry{func, dev, bytes};
  return cudaSuccess;
}

namespace {

constexpr int64_t kAlign = 256;

int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) % kAlign) == 0; }

bool valid_bm(int bm) { return bm == 16 || bm == 32 || bm == 64 || bm == 128 || bm == 256; }

// Upper bound of the padded sorted length: every valid route plus at most
// block_m - 1 pads for each expert that can be non-empty.
int64_t max_padded(int64_t R, int E, int bm) {
  const int64_t nonempty = R < E ? R : E;
  return align_up(R + nonempty * (bm - 1), bm);
}

// Route block of both GEMMs, from the mean routes per expert.
int choose_block_m(int M, int topk, int E) {
  const int64_t per_expert = (static_cast<int64_t>(M) * topk + E - 1) / E;
  if (per_expert <= 16) return 16;
  if (per_expert <= 32) return 32;
  if (per_expert <= 64) return 64;
  return 128;
}

moe_status_t check_shape(int M, int H, int Ip, int E, int topk) {
  if (M < 0 || H <= 0 || Ip <= 0 || E <= 0 || topk <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 128 != 0 || Ip % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (E > kMaxExperts || topk > kMaxTopk) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(M) * topk > (int64_t(1) << 24)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// bm_req: the route block asked for (0 = choose_block_m)
void build_layout(int M, int H, int Ip, int E, int topk, bool a16, int bm_req,
                  moe_ws_layout_t* L) {
  std::memset(L, 0, sizeof(*L));
  const int bm = bm_req > 0 ? bm_req : choose_block_m(M, topk, E);
  const int64_t R = static_cast<int64_t>(M) * topk;
  const int64_t pm = max_padded(R, E, bm);
  const int64_t nblk = pm / bm;
  const int64_t atoms = (bm + 127) / 128;
  int64_t o = 0;
  auto take = [&](int64_t bytes) {
    const int64_t at = o;
    o = align_up(o + (bytes > 0 ? bytes : 0), kAlign);
    return at;
  };
  L->block_m = bm;
  L->p_max = pm;
  L->status_off = take(16);
  L->expert_off_off = take(4 * (E + 1));
  L->sorted_route_off = take(4 * pm);
  L->sorted_w_off = take(4 * pm);
  L->block_expert_off = take(4 * nblk);
  L->route_pos_off = take(4 * R);
  L->sort_scratch_off = take(static_cast<int64_t>(sort_scratch_bytes(static_cast<int>(R), E)));
  L->act_off = take(pm * H * (a16 ? 2 : 1));
  L->act_sf_off = take(a16 ? 0 : nblk * (H / 128) * atoms * 512);
  L->inter_off = take(pm * Ip * (a16 ? 2 : 1));
  L->inter_sf_off = take(a16 ? 0 : nblk * (Ip / 128) * atoms * 512);
  L->acc_off = take(static_cast<int64_t>(M) * H * 4);
  // split-walk slots of stage 1 (decode block sizes)
  const bool split = bm <= 32;
  L->split_part_off = take(split ? static_cast<int64_t>(kSplitSlots) * bm * 128 * 4 : 0);
  L->split_cnt_off = take(split ? kSplitSlots * 4 : 0);
  L->total_bytes = o;
}

moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ---------------------------------------------------------------- timing
constexpr int kProfSlots = MOE_PROFILE_SLOTS;
constexpr int kProfMaxCalls = 1024;
struct Profiler {
  bool enabled = false;
  int pending = 0;
  int dropped = 0;
  cudaEvent_t ev[kProfMaxCalls][2 * kProfSlots] = {};
  bool created[kProfMaxCalls] = {};
};
Profiler g_prof;

// Records the begin (before=true) or end event of `slot` for the current call.
void prof_mark(int slot, bool before, cudaStream_t s) {
  if (!g_prof.enabled || g_prof.pending >= kProfMaxCalls) return;
  const int c = g_prof.pending;
  if (!g_prof.created[c]) {
    for (int i = 0; i < 2 * kProfSlots; ++i) cudaEventCreate(&g_prof.ev[c][i]);
    g_prof.created[c] = true;
  }
  cudaEventRecord(g_prof.ev[c][2 * slot + (before ? 0 : 1)], s);
}
void prof_end_call() {
  if (!g_prof.enabled) return;
  if (g_prof.pending < kProfMaxCalls) ++g_prof.pending;
  else ++g_prof.dropped;
}

// gate: the gated calls (routing from router logits, written to gate->ids_out /
// w_out, which then stand for ids / wts); nullptr for the plain calls.
moe_status_t fused_moe_impl(bool a16, const void* x, const int32_t* ids, const float* wts, int M,
                            int H, int topk, const uint8_t* w1, const uint8_t* w1s,
                            const uint8_t* w2, const uint8_t* w2s, int E, int Ip, void* out,
                            void* ws, size_t ws_bytes, int bm_req, cudaStream_t s,
                            const FrontGating* gate = nullptr, int pf1 = 0, int pf2 = 0,
                            int split_walk = 0) {
  moe_status_t st = check_shape(M, H, Ip, E, topk);
  if (st != MOE_OK) return st;
  if (bm_req != 0 && !valid_bm(bm_req)) return MOE_ERR_UNSUPPORTED;
  if (pf1 < 0 || pf1 > kMaxPrefetch || pf2 < 0 || pf2 > kMaxPrefetch) return MOE_ERR_UNSUPPORTED;
  if (split_walk < 0 || split_walk > 2) return MOE_ERR_UNSUPPORTED;
  if (!ws || !w1 || !w1s || !w2 || !w2s) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!x || !ids || !wts || !out)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, ids, wts, w1, w1s, w2, w2s, out, ws};
  for (const void* p : ptrs)
    if (p && !aligned(p)) return MOE_ERR_ALIGNMENT;
  moe_ws_layout_t L;
  build_layout(M, H, Ip, E, topk, a16, bm_req, &L);
  if (ws_bytes < static_cast<size_t>(L.total_bytes)) return MOE_ERR_WORKSPACE;
  if (M == 0) return MOE_OK;

  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(base + L.status_off);
  int32_t* num_padded = status + 1;
  int32_t* expert_off = reinterpret_cast<int32_t*>(base + L.expert_off_off);
  int32_t* sorted_route = reinterpret_cast<int32_t*>(base + L.sorted_route_off);
  float* sorted_w = reinterpret_cast<float*>(base + L.sorted_w_off);
  int32_t* block_expert = reinterpret_cast<int32_t*>(base + L.block_expert_off);
  int32_t* route_pos = reinterpret_cast<int32_t*>(base + L.route_pos_off);
  void* act = base + L.act_off;
  uint8_t* act_sf = base + L.act_sf_off;
  void* inter = base + L.inter_off;
  uint8_t* inter_sf = base + L.inter_sf_off;
  float* acc = reinterpret_cast<float*>(base + L.acc_off);
  const int R = M * topk;
  const bool split = L.split_cnt_off > L.split_part_off;
  float* split_part = split ? reinterpret_cast<float*>(base + L.split_part_off) : nullptr;
  int32_t* split_cnt = split ? reinterpret_cast<int32_t*>(base + L.split_cnt_off) : nullptr;
  // the split buffers are zeroed with the accumulator (one contiguous region)
  const int64_t split_bytes = split ? L.split_cnt_off + kSplitSlots * 4 - L.split_part_off : 0;

  cudaError_t e;
  if (R <= kFrontMaxRoutes) {
    // decode: gating (gated calls), sort and gather in one launch (profiled
    // as the sort slot)
    prof_mark(0, true, s);
    e = launch_front_tiny(a16, x, ids, wts, M, H, topk, E, L.block_m, L.p_max, sorted_route,
                          sorted_w, block_expert, expert_off, num_padded, route_pos, status, act,
                          act_sf, acc, split_part, split_bytes, gate, s);
    if (e != cudaSuccess) return from_cuda(e);
    prof_mark(0, false, s);
    prof_mark(1, true, s);
    prof_mark(1, false, s);
  } else {
    prof_mark(0, true, s);
    if (gate) {
      e = launch_router_topk(gate->logits, M, gate->E_route, gate->ld, gate->topk_sel,
                             gate->shared_id, gate->n_shared, gate->ids_out, gate->w_out, s);
      if (e != cudaSuccess) return from_cuda(e);
    }
    int32_t* sort_scratch = reinterpret_cast<int32_t*>(base + L.sort_scratch_off);
    e = launch_sort(ids, wts, R, E, L.block_m, L.p_max, sorted_route, sorted_w, block_expert,
                    expert_off, num_padded, route_pos, status, sort_scratch, s);
    if (e != cudaSuccess) return from_cuda(e);
    prof_mark(0, false, s);
    prof_mark(1, true, s);
    e = launch_gather_act(a16, x, M, H, topk, L.block_m, route_pos, act, act_sf, acc, split_part,
                          split_bytes, s);
    if (e != cudaSuccess) return from_cuda(e);
    prof_mark(1, false, s);
  }
  GemmArgs g{};
  g.a16 = a16;
  g.M = M; g.H = H; g.Ip = Ip; g.E = E; g.topk = topk; g.bm = L.block_m;
  g.prefetch1 = pf1; g.prefetch2 = pf2;
  g.split = split_walk;
  g.p_max = L.p_max;
  // the GEMMs may read topk_ids before their dependency wait only when it is
  // an input of the call (not when the gating kernel writes it)
  g.topk_ids = gate ? nullptr : ids;
  g.gate = gate ? LocalGate{gate->logits, gate->ld, gate->E_route, gate->topk_sel,
                            gate->shared_id, gate->n_shared}
                : LocalGate{nullptr, 0, 0, 0, -1, 0};
  g.sorted_route = sorted_route; g.sorted_w = sorted_w; g.block_expert = block_expert;
  g.num_padded = num_padded;
  g.w1 = w1; g.w1s = w1s; g.w2 = w2; g.w2s = w2s;
  g.act = act; g.act_sf = act_sf; g.inter = inter; g.inter_sf = inter_sf; g.acc = acc;
  g.split_part = split_part;
  g.split_cnt = split_cnt;
  g.status = status;
  GemmPlan plan1, plan2;
  e = a16 ? prepare_gemm_bf16w4(1, g, &plan1) : prepare_gemm_mx(1, g, &plan1);
  if (e != cudaSuccess) return from_cuda(e);
  e = a16 ? prepare_gemm_bf16w4(2, g, &plan2) : prepare_gemm_mx(2, g, &plan2);
  if (e != cudaSuccess) return from_cuda(e);
  prof_mark(2, true, s);
  e = launch_gemm(plan1, s);
  if (e != cudaSuccess) return from_cuda(e);
  prof_mark(2, false, s);
  prof_mark(3, true, s);
  e = launch_gemm(plan2, s);
  if (e != cudaSuccess) return from_cuda(e);
  prof_mark(3, false, s);
  prof_mark(4, true, s);
  e = launch_finalize(acc, static_cast<int64_t>(M) * H, out, s);
  if (e != cudaSuccess) return from_cuda(e);
  prof_mark(4, false, s);
  prof_end_call();
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_ALIGNMENT: return "pointer not 256-byte aligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side check failed (expert id out of range)";
  }
  return "unknown status";
}

int64_t moe_sort_max_padded(int M, int topk, int E, int block_m) {
  if (M < 0 || topk <= 0 || E <= 0 || !valid_bm(block_m)) return -1;
  return max_padded(static_cast<int64_t>(M) * topk, E, block_m);
}

size_t moe_sort_workspace_bytes(int M, int topk, int E, int block_m) {
  if (M < 0 || topk <= 0 || E <= 0 || !valid_bm(block_m)) return 0;
  return sort_scratch_bytes(M * topk, E);
}

moe_status_t moe_sort(const int32_t* topk_ids, const float* topk_weights, int M, int topk, int E,
                      int block_m, int32_t* sorted_route, float* sorted_w, int32_t* block_expert,
                      int32_t* expert_off, int32_t* num_padded, int32_t* route_pos, void* ws,
                      size_t ws_bytes, moe_stream_t stream) {
  if (M < 0 || topk <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (!valid_bm(block_m) || E > kMaxExperts || topk > kMaxTopk) return MOE_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(M) * topk > (int64_t(1) << 24)) return MOE_ERR_UNSUPPORTED;
  const int64_t pm = max_padded(static_cast<int64_t>(M) * topk, E, block_m);
  if (!expert_off || !num_padded) return MOE_ERR_INVALID_ARG;
  if (pm > 0 && (!sorted_route || !sorted_w || !block_expert)) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!topk_ids || !topk_weights)) return MOE_ERR_INVALID_ARG;
  const size_t need = sort_scratch_bytes(M * topk, E);
  if (need > 0 && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  if (ws && !aligned(ws)) return MOE_ERR_ALIGNMENT;
  return from_cuda(launch_sort(topk_ids, topk_weights, M * topk, E, block_m, pm, sorted_route,
                               sorted_w, block_expert, expert_off, num_padded, route_pos, nullptr,
                               static_cast<int32_t*>(ws), reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_quant_act_mx(const void* x_bf16, int M, int K, int ldx, uint8_t* q,
                              uint8_t* scale, moe_stream_t stream) {
  if (M < 0 || K <= 0 || ldx < K) return MOE_ERR_INVALID_ARG;
  if (K % 32 != 0 || ldx % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (M > 0 && (!x_bf16 || !q || !scale)) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!aligned(x_bf16) || !aligned(q) || !aligned(scale))) return MOE_ERR_ALIGNMENT;
  return from_cuda(launch_quant_act(x_bf16, M, K, ldx, q, scale,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_router_topk(const float* logits, int M, int E, int ld, int topk, int shared_id,
                             int n_shared, int32_t* topk_ids, float* topk_weights,
                             moe_stream_t stream) {
  if (M < 0 || E <= 0 || ld < E || topk < 1 || topk > E) return MOE_ERR_INVALID_ARG;
  // a shared expert is an extra expert after the routed ones: an id among
  // them would double-count a pick, one beyond the sort's range would be
  // dropped silently
  if (shared_id >= 0 && (shared_id < E || n_shared < 1 || shared_id + n_shared > kMaxExperts))
    return MOE_ERR_INVALID_ARG;
  if (shared_id < 0) n_shared = 0;
  if (E > kMaxExperts || topk + n_shared > kMaxTopk) return MOE_ERR_UNSUPPORTED;
  if (M > 0 && (!logits || !topk_ids || !topk_weights)) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!aligned(logits) || !aligned(topk_ids) || !aligned(topk_weights)))
    return MOE_ERR_ALIGNMENT;
  return from_cuda(launch_router_topk(logits, M, E, ld, topk, shared_id, n_shared, topk_ids,
                                      topk_weights,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_prepacked_weight_bytes(int E, int N, int K) {
  if (E <= 0 || N <= 0 || K <= 0 || N % 128 || K % 128) return 0;
  return static_cast<size_t>(E) * N * (K / 2);
}

moe_status_t moe_prepack_weights_mx(const uint8_t* w, int E, int N, int K, uint8_t* out,
                                    moe_stream_t stream) {
  if (E <= 0 || N <= 0 || K <= 0 || !w || !out || w == out) return MOE_ERR_INVALID_ARG;
  if (N % 128 || K % 128) return MOE_ERR_UNSUPPORTED;
  if (!aligned(w) || !aligned(out)) return MOE_ERR_ALIGNMENT;
  return from_cuda(launch_prepack_weights(w, E, N, K, out, false,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_prepack_weights_a16w4(const uint8_t* w, int E, int N, int K, uint8_t* out,
                                       moe_stream_t stream) {
  if (E <= 0 || N <= 0 || K <= 0 || !w || !out || w == out) return MOE_ERR_INVALID_ARG;
  if (N % 128 || K % 128) return MOE_ERR_UNSUPPORTED;
  if (!aligned(w) || !aligned(out)) return MOE_ERR_ALIGNMENT;
  return from_cuda(launch_prepack_weights(w, E, N, K, out, true,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_dequant_a16w4(const uint8_t* w_packed, const uint8_t* scale_packed, int E, int N,
                               int K, void* out_bf16, moe_stream_t stream) {
  if (E <= 0 || N <= 0 || K <= 0 || !w_packed || !scale_packed || !out_bf16)
    return MOE_ERR_INVALID_ARG;
  if (N % 128 || K % 128) return MOE_ERR_UNSUPPORTED;
  if (!aligned(w_packed) || !aligned(scale_packed) || !aligned(out_bf16))
    return MOE_ERR_ALIGNMENT;
  return from_cuda(launch_dequant_a16w4(w_packed, scale_packed, E, N, K, out_bf16,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_prepacked_scale_bytes(int E, int N, int K) {
  if (E <= 0 || N <= 0 || K <= 0 || N % 128 || K % 128) return 0;
  return static_cast<size_t>(E) * N * (K / 32);
}

moe_status_t moe_prepack_scales_mx(const uint8_t* scale, int E, int N, int K, uint8_t* out,
                                   moe_stream_t stream) {
  if (E <= 0 || N <= 0 || K <= 0 || !scale || !out) return MOE_ERR_INVALID_ARG;
  if (N % 128 || K % 128) return MOE_ERR_UNSUPPORTED;
  if (!aligned(scale) || !aligned(out)) return MOE_ERR_ALIGNMENT;
  return from_cuda(launch_prepack_scales(scale, E, N, K, out,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

size_t fused_moe_workspace_bytes_bm(int M, int H, int Ip, int E, int topk, int a16, int block_m) {
  if (check_shape(M, H, Ip, E, topk) != MOE_OK) return 0;
  if (block_m != 0 && !valid_bm(block_m)) return 0;
  moe_ws_layout_t L;
  build_layout(M, H, Ip, E, topk, a16 != 0, block_m, &L);
  return static_cast<size_t>(L.total_bytes);
}

size_t fused_moe_workspace_bytes(int M, int H, int Ip, int E, int topk, int a16) {
  return fused_moe_workspace_bytes_bm(M, H, Ip, E, topk, a16, 0);
}

moe_status_t fused_moe_workspace_layout_bm(int M, int H, int Ip, int E, int topk, int a16,
                                           int block_m, moe_ws_layout_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_shape(M, H, Ip, E, topk);
  if (st != MOE_OK) return st;
  if (block_m != 0 && !valid_bm(block_m)) return MOE_ERR_UNSUPPORTED;
  build_layout(M, H, Ip, E, topk, a16 != 0, block_m, out);
  return MOE_OK;
}

moe_status_t fused_moe_workspace_layout(int M, int H, int Ip, int E, int topk, int a16,
                                        moe_ws_layout_t* out) {
  return fused_moe_workspace_layout_bm(M, H, Ip, E, topk, a16, 0, out);
}

moe_status_t fused_moe_a8w4_bm(const void* x, const int32_t* topk_ids, const float* topk_weights,
                               int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                               const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip,
                               void* out, void* ws, size_t ws_bytes, int block_m,
                               moe_stream_t stream) {
  return fused_moe_impl(false, x, topk_ids, topk_weights, M, H, topk, w1, w1_scale, w2, w2_scale,
                        E, Ip, out, ws, ws_bytes, block_m, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t fused_moe_a16w4_bm(const void* x, const int32_t* topk_ids, const float* topk_weights,
                                int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                                const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip,
                                void* out, void* ws, size_t ws_bytes, int block_m,
                                moe_stream_t stream) {
  return fused_moe_impl(true, x, topk_ids, topk_weights, M, H, topk, w1, w1_scale, w2, w2_scale,
                        E, Ip, out, ws, ws_bytes, block_m, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t fused_moe_a8w4_cfg(const void* x, const int32_t* topk_ids, const float* topk_weights,
                                int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                                const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip,
                                void* out, void* ws, size_t ws_bytes, const moe_call_config_t* cfg,
                                moe_stream_t stream) {
  return fused_moe_impl(false, x, topk_ids, topk_weights, M, H, topk, w1, w1_scale, w2, w2_scale,
                        E, Ip, out, ws, ws_bytes, cfg ? cfg->block_m : 0,
                        reinterpret_cast<cudaStream_t>(stream), nullptr,
                        cfg ? cfg->prefetch1 : 0, cfg ? cfg->prefetch2 : 0,
                        cfg ? cfg->split : 0);
}

moe_status_t fused_moe_a16w4_cfg(const void* x, const int32_t* topk_ids, const float* topk_weights,
                                 int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                                 const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip,
                                 void* out, void* ws, size_t ws_bytes, const moe_call_config_t* cfg,
                                 moe_stream_t stream) {
  return fused_moe_impl(true, x, topk_ids, topk_weights, M, H, topk, w1, w1_scale, w2, w2_scale,
                        E, Ip, out, ws, ws_bytes, cfg ? cfg->block_m : 0,
                        reinterpret_cast<cudaStream_t>(stream), nullptr,
                        cfg ? cfg->prefetch1 : 0, cfg ? cfg->prefetch2 : 0,
                        cfg ? cfg->split : 0);
}

moe_status_t fused_moe_a8w4(const void* x, const int32_t* topk_ids, const float* topk_weights,
                            int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                            const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip, void* out,
                            void* ws, size_t ws_bytes, moe_stream_t stream) {
  return fused_moe_a8w4_bm(x, topk_ids, topk_weights, M, H, topk, w1, w1_scale, w2, w2_scale, E,
                           Ip, out, ws, ws_bytes, 0, stream);
}

moe_status_t fused_moe_a16w4(const void* x, const int32_t* topk_ids, const float* topk_weights,
                             int M, int H, int topk, const uint8_t* w1, const uint8_t* w1_scale,
                             const uint8_t* w2, const uint8_t* w2_scale, int E, int Ip, void* out,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  return fused_moe_a16w4_bm(x, topk_ids, topk_weights, M, H, topk, w1, w1_scale, w2, w2_scale, E,
                            Ip, out, ws, ws_bytes, 0, stream);
}

namespace {
moe_status_t gated_call(bool a16, const void* x, const float* logits, int ld, int E_route,
                        int topk, int shared_id, int n_shared, int M, int H, const uint8_t* w1,
                        const uint8_t* w1_scale, const uint8_t* w2, const uint8_t* w2_scale,
                        int E, int Ip, void* out, int32_t* topk_ids, float* topk_weights,
                        void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (M < 0 || E_route <= 0 || ld < E_route || topk < 1 || topk > E_route)
    return MOE_ERR_INVALID_ARG;
  if (shared_id >= 0 && (shared_id < E_route || n_shared < 1 || shared_id + n_shared > kMaxExperts))
    return MOE_ERR_INVALID_ARG;
  if (shared_id < 0) n_shared = 0;
  if (E_route > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  const int kout = topk + n_shared;
  if (kout > kMaxTopk) return MOE_ERR_UNSUPPORTED;
  if (M > 0 && (!logits || !topk_ids || !topk_weights)) return MOE_ERR_INVALID_ARG;
  if (M > 0 && (!aligned(logits) || !aligned(topk_ids) || !aligned(topk_weights)))
    return MOE_ERR_ALIGNMENT;
  FrontGating gate{logits, ld, E_route, topk, shared_id, n_shared, topk_ids, topk_weights};
  return fused_moe_impl(a16, x, topk_ids, topk_weights, M, H, kout, w1, w1_scale, w2, w2_scale,
                        E, Ip, out, ws, ws_bytes, 0, reinterpret_cast<cudaStream_t>(stream),
                        &gate);
}
}  // namespace

moe_status_t fused_moe_a8w4_gated(const void* x, const float* router_logits, int ld, int E_route,
                                  int topk, int shared_id, int n_shared, int M, int H,
                                  const uint8_t* w1, const uint8_t* w1_scale, const uint8_t* w2,
                                  const uint8_t* w2_scale, int E, int Ip, void* out,
                                  int32_t* topk_ids, float* topk_weights, void* ws,
                                  size_t ws_bytes, moe_stream_t stream) {
  return gated_call(false, x, router_logits, ld, E_route, topk, shared_id, n_shared, M, H, w1,
                    w1_scale, w2, w2_scale, E, Ip, out, topk_ids, topk_weights, ws, ws_bytes,
                    stream);
}

moe_status_t fused_moe_a16w4_gated(const void* x, const float* router_logits, int ld,
                                   int E_route, int topk, int shared_id, int n_shared, int M,
                                   int H, const uint8_t* w1, const uint8_t* w1_scale,
                                   const uint8_t* w2,
                                   const uint8_t* w2_scale, int E, int Ip, void* out,
                                   int32_t* topk_ids, float* topk_weights, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  return gated_call(true, x, router_logits, ld, E_route, topk, shared_id, n_shared, M, H, w1,
                    w1_scale, w2, w2_scale, E, Ip, out, topk_ids, topk_weights, ws, ws_bytes,
                    stream);
}

moe_status_t moe_profile_enable(int enable) {
  g_prof.enabled = enable != 0;
  return MOE_OK;
}

moe_status_t moe_profile_collect(double* kernel_ms, int32_t* n_calls) {
  if (!kernel_ms || !n_calls) return MOE_ERR_INVALID_ARG;
  for (int c = 0; c < g_prof.pending; ++c) {
    if (cudaEventSynchronize(g_prof.ev[c][2 * kProfSlots - 1]) != cudaSuccess) return MOE_ERR_CUDA;
    for (int k = 0; k < kProfSlots; ++k) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, g_prof.ev[c][2 * k], g_prof.ev[c][2 * k + 1]) != cudaSuccess)
        return MOE_ERR_CUDA;
      kernel_ms[k] += ms;
    }
  }
  *n_calls = g_prof.pending;
  g_prof.pending = 0;
  g_prof.dropped = 0;
  return MOE_OK;
}

moe_status_t moe_debug_wait_selftest(int32_t* status, int timeout_us, moe_stream_t stream) {
  if (!status || timeout_us < 1 || timeout_us > 1000000) return MOE_ERR_INVALID_ARG;
  if (!aligned(status)) return MOE_ERR_ALIGNMENT;
  return from_cuda(launch_wait_selftest(status, static_cast<uint64_t>(timeout_us) * 1000u,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_decode_device_status(int32_t status_word) {
  if (status_word & kDevTimeout) return MOE_ERR_TIMEOUT;
  if (status_word & kDevBadExpert) return MOE_ERR_DEVICE_CHECK;
  return MOE_OK;
}

}  // extern "C"

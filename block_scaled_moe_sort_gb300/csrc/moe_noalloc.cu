// fused_moe_a8w4_noalloc: the a8w4 fused MoE call for callers that cannot
// give this library a workspace buffer.
//
// Who needs it: code that must not (or cannot) obtain device memory at the
// point where it runs the layer - for example a plugin inside an inference
// engine that owns every device allocation and offers its plugins no way to
// request scratch, or a real-time path that is not allowed to call into a
// device allocator at all. Such a caller still passes its inputs, weights
// and output, but the layer's scratch (sorted route lists, gathered
// activation rows, the intermediate and the FP32 accumulator) must come from
// somewhere else.
//
// Here that scratch is one file-scope __device__ array of
// MOE_NOALLOC_WORKSPACE_BYTES. Every GPU that loads this library reserves
// it (in each process) until the process exits. In host code the array's
// name is only a stand-in, never a device address, so the first call on each
// device looks the real address up with cudaGetSymbolAddress (with that
// device current) and caches it; later calls reuse the cached pointer.
// The call itself is the ordinary fused_moe_a8w4 with that pointer as its
// workspace: nothing else changes.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>
#include "moe_mx.h"

namespace moe {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_ws[MOE_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_ws on the current device (looked up once).
cudaError_t noalloc_ws_current_device(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (err != cudaSuccess) return err;
    if (!p) return cudaErrorInvalidSymbol;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t fused_moe_a8w4_noalloc(const void* x, const int32_t* topk_ids,
                                               const float* topk_weights, int M, int H,
                                               int topk, const uint8_t* w1,
                                               const uint8_t* w1_scale, const uint8_t* w2,
                                               const uint8_t* w2_scale, int E, int Ip,
                                               void* out, moe_stream_t stream) {
  // Shape errors are reported by fused_moe_a8w4 itself (size 0 = bad shape).
  const size_t need = fused_moe_workspace_bytes(M, H, Ip, E, topk, 0);
  if (need > MOE_NOALLOC_WORKSPACE_BYTES) return MOE_ERR_WORKSPACE;
  void* ws = nullptr;
  if (moe::noalloc_ws_current_device(&ws) != cudaSuccess) return MOE_ERR_CUDA;
  // Nothing in the workspace has to start at zero: every call's kernels
  // write what they read (the front kernel or the sort resets the status
  // word and writes the route lists, the stage-1 GEMM zeroes the
  // accumulator, the front kernel or the gather zeroes the split buffers).
  return fused_moe_a8w4(x, topk_ids, topk_weights, M, H, topk, w1, w1_scale, w2, w2_scale, E,
                        Ip, out, ws, MOE_NOALLOC_WORKSPACE_BYTES, stream);
}

extern "C" moe_status_t moe_noalloc_status(int32_t* status_out, moe_stream_t stream) {
  if (!status_out) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(status_out) % 16 != 0) return MOE_ERR_ALIGNMENT;
  void* ws = nullptr;
  if (moe::noalloc_ws_current_device(&ws) != cudaSuccess) return MOE_ERR_CUDA;
  moe_ws_layout_t L;
  // the status words sit at the same offset for every shape (the first
  // region of the layout); any valid shape gives it
  if (fused_moe_workspace_layout(1, 128, 128, 1, 1, 0, &L) != MOE_OK) return MOE_ERR_CUDA;
  const cudaError_t e = cudaMemcpyAsync(status_out, static_cast<uint8_t*>(ws) + L.status_off,
                                        4 * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                        reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

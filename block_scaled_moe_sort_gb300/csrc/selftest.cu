// Self-test of the bounded waits every kernel of the layer uses: one CTA
// waits on an mbarrier that nothing ever completes, with a short limit. The
// wait gives up, sets the timeout bit of the status word and the kernel
// returns, so a stalled pipeline is reported to the host as MOE_ERR_TIMEOUT
// (moe_decode_device_status) without a hung or faulted GPU, and the context
// stays usable for the next call.
#include <cstdint>
#include "moe_internal.h"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

__global__ void wait_selftest_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // one arrival expected; none ever comes
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool completed = mbar_wait(&bar, 0, status, timeout_ns);
    status[1] = completed ? 2 : 1;   // 1: the wait gave up and returned
  }
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* status, uint64_t timeout_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace moe

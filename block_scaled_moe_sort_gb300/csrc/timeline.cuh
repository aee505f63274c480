// Per-CTA global-timer stamps for experiment builds (-DMOE_TIMELINE): every
// kernel of the fused call records when each CTA reaches a few fixed points
// (entry, dependency wait returned, first load, first MMA, last MMA, last
// epilogue, exit), so that a graph replay can be laid out as a timeline.
// Off by default: the macros expand to nothing and no symbol is emitted.
//
// Kernel ids: 0 sort (single launch), 1 sort count, 2 sort scatter,
// 3 gather/quant, 4 stage-1 GEMM, 5 stage-2 GEMM, 6 finalize.
// Points:     0 entry, 1 wait returned, 2 first load issued, 3 first k-block
//             ready, 4 last MMA committed, 5 last epilogue done, 7 exit
//             (gather: 2 zeroing done, 3 route positions in, 4 first block
//             quantised, 5 stores issued).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#ifdef MOE_TIMELINE
#define MOE_TL_DEFINE(dump_name)                                                         \
  static __device__ unsigned long long g_moe_tl[8][1024][8];                            \
  extern "C" void dump_name(unsigned long long* out, int reset) {                       \
    cudaMemcpyFromSymbol(out, g_moe_tl, sizeof(g_moe_tl));                              \
    if (reset) {                                                                        \
      static unsigned long long zeros[8][1024][8] = {};                                 \
      cudaMemcpyToSymbol(g_moe_tl, zeros, sizeof(zeros));                               \
    }                                                                                   \
  }
// Stamp after `value` has been computed (orders the timer read behind it).
#define MOE_TL_AFTER(kernel, point, value)                                               \
  do {                                                                                  \
    asm volatile("" ::"r"(static_cast<uint32_t>(value)));                               \
    MOE_TL(kernel, point);                                                              \
  } while (0)
#define MOE_TL(kernel, point)                                                            \
  do {                                                                                  \
    unsigned long long t_;                                                              \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                              \
    g_moe_tl[(kernel) & 7][blockIdx.x & 1023][(point) & 7] = t_;                         \
  } while (0)
#else
#define MOE_TL_DEFINE(dump_name)
#define MOE_TL(kernel, point) ((void)0)
#define MOE_TL_AFTER(kernel, point, value) ((void)0)
#endif

// CUDA-core grouped GEMMs of the fused MoE layer (both stages, a8w4 and
// a16w4). Straightforward tiles: each CTA takes one block_m block of sorted
// routes (one expert) and 64 weight rows, stages dequantised FP32 operands in
// shared memory 128 K-elements at a time and accumulates in FP32.
//
// Stage 1 (AITER #5609 "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning",
// Configuration): 64 interleaved w1 rows = 32 gate/up pairs, so one CTA
// yields one 32-column block of the intermediate: SiLU(gate)*up, then
// per-1x32 FP8 requantisation (a8w4) or BF16 rounding (a16w4).
// Stage 2: 64 output features; the routing weight multiplies each route's
// result, which is added into the FP32 token accumulator.
#include <cstdint>
#include "common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kRC = 32;    // routes per sub-chunk
constexpr int kKC = 64;    // K per staged chunk
constexpr int kNT = 64;    // weight rows per CTA

__device__ __forceinline__ int64_t atom_index(int64_t blk, int nslab, int slab, int atoms, int rr) {
  return (blk * nslab + slab) * atoms + rr / 128;
}

// Dequantise 64 weight rows x 128 K of one expert into smem (FP32).
__device__ __forceinline__ void load_w_tile(float (*Ws)[kKC + 1], const uint8_t* __restrict__ w,
                                            const uint8_t* __restrict__ ws, int e, int N, int K,
                                            int n0, int k0) {
  const int nb_n = N / 128, nb_k = K / 128;
  for (int i = threadIdx.x; i < kNT * (kKC / 2); i += blockDim.x) {
    const int row = i / (kKC / 2), byte = i % (kKC / 2);
    const int n = n0 + row;
    const uint8_t b = __ldg(w + (static_cast<int64_t>(e) * N + n) * (K / 2) + k0 / 2 + byte);
    const int kk = 2 * byte;  // element index within the chunk
    const int ka = k0 + kk;   // absolute K
    const int64_t atom = (static_cast<int64_t>(e) * nb_n + n / 128) * nb_k + ka / 128;
    const float s = e8m0_to_float(__ldg(ws + atom * 512 + sf_atom_off(n % 128, (ka / 32) % 4)));
    Ws[row][kk] = e2m1_to_float(b & 15) * s;
    Ws[row][kk + 1] = e2m1_to_float(b >> 4) * s;
  }
}

template <bool A16>
__device__ __forceinline__ void load_x_tile(float (*Xs)[kKC + 1], const void* __restrict__ act,
                                            const uint8_t* __restrict__ act_sf, int64_t p0, int rc,
                                            int K, int bm, int k0) {
  const int atoms = (bm + 127) / 128;
  for (int i = threadIdx.x; i < rc * kKC; i += blockDim.x) {
    const int row = i / kKC, kk = i % kKC;
    const int64_t p = p0 + row;
    float v;
    if (A16) {
      const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(act);
      v = __bfloat162float(xb[p * K + k0 + kk]);
    } else {
      const uint8_t* xq = static_cast<const uint8_t*>(act);
      const int64_t blk = p / bm;
      const int rr = static_cast<int>(p % bm);
      const int ka = k0 + kk;
      const int64_t atom = atom_index(blk, K / 128, ka / 128, atoms, rr);
      const float s = e8m0_to_float(act_sf[atom * 512 + sf_atom_off(rr % 128, (ka / 32) % 4)]);
      v = e4m3_to_float(xq[p * K + k0 + kk]) * s;
    }
    Xs[row][kk] = v;
  }
}

template <bool A16, int STAGE>
__global__ void __launch_bounds__(256) grouped_gemm_simt_kernel(GemmArgs a) {
  __shared__ float Xs[kRC][kKC + 1];
  __shared__ float Ws[kNT][kKC + 1];
  __shared__ float Hs[kRC][kNT + 1];
  const int blk = blockIdx.x;
  const int P = *a.num_padded;
  if (static_cast<int64_t>(blk) * a.bm >= P) return;
  const int e = a.block_expert[blk];
  if (e < 0 || e >= a.E) return;
  const int n0 = blockIdx.y * kNT;
  const int K = STAGE == 1 ? a.H : a.Ip;
  const int N = STAGE == 1 ? 2 * a.Ip : a.H;
  const uint8_t* w = STAGE == 1 ? a.w1 : a.w2;
  const uint8_t* ws = STAGE == 1 ? a.w1s : a.w2s;
  const void* act = STAGE == 1 ? a.act : static_cast<const void*>(a.inter);
  const uint8_t* act_sf = STAGE == 1 ? a.act_sf : a.inter_sf;
  const int R = a.M * a.topk;
  const int tn = threadIdx.x % kNT, tr = threadIdx.x / kNT;  // 64 x 4

  for (int sub = 0; sub < a.bm; sub += kRC) {
    const int rc = min(kRC, a.bm - sub);
    const int64_t p0 = static_cast<int64_t>(blk) * a.bm + sub;
    float accv[kRC / 4];
#pragma unroll
    for (int i = 0; i < kRC / 4; ++i) accv[i] = 0.f;
    for (int k0 = 0; k0 < K; k0 += kKC) {
      __syncthreads();
      load_w_tile(Ws, w, ws, e, N, K, n0, k0);
      load_x_tile<A16>(Xs, act, act_sf, p0, rc, K, a.bm, k0);
      __syncthreads();
#pragma unroll
      for (int i = 0; i < kRC / 4; ++i) {
        const int row = tr + 4 * i;
        if (row < rc) {
          float s = 0.f;
          for (int kk = 0; kk < kKC; ++kk) s = fmaf(Xs[row][kk], Ws[tn][kk], s);
          accv[i] += s;
        }
      }
    }
    if (STAGE == 1) {
      __syncthreads();
#pragma unroll
      for (int i = 0; i < kRC / 4; ++i) {
        const int row = tr + 4 * i;
        if (row < rc) Hs[row][tn] = accv[i];
      }
      __syncthreads();
      if (threadIdx.x < rc) {
        const int row = threadIdx.x;
        const int64_t p = p0 + row;
        const bool pad = a.sorted_route[p] >= R;
        const int j0 = n0 / 2;  // first intermediate column of this CTA
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = pad ? 0.f : silu_mul(Hs[row][2 * j], Hs[row][2 * j + 1]);
        if (A16) {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.inter) + p * a.Ip + j0;
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[j] = __float2bfloat16_rn(v[j]);
        } else {
          uint32_t c[8];
          const uint8_t sb = quant_block32(v, c);
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.inter) + p * a.Ip + j0);
          dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
          dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
          const int atoms = (a.bm + 127) / 128;
          const int rr = static_cast<int>(p % a.bm);
          const int64_t atom = atom_index(blk, a.Ip / 128, j0 / 128, atoms, rr);
          a.inter_sf[atom * 512 + sf_atom_off(rr % 128, (j0 / 32) % 4)] = sb;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < kRC / 4; ++i) {
        const int row = tr + 4 * i;
        if (row < rc) {
          const int64_t p = p0 + row;
          const int r = a.sorted_route[p];
          if (r < R) {
            const int t = r / a.topk;
            atomicAdd(a.acc + static_cast<int64_t>(t) * a.H + n0 + tn, a.sorted_w[p] * accv[i]);
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_stage1_simt(const GemmArgs& a, cudaStream_t s) {
  const int64_t nblk = a.p_max / a.bm;
  if (nblk == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(nblk), (2 * a.Ip) / kNT);
  if (a.a16) grouped_gemm_simt_kernel<true, 1><<<grid, 256, 0, s>>>(a);
  else grouped_gemm_simt_kernel<false, 1><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_stage2_simt(const GemmArgs& a, cudaStream_t s) {
  const int64_t nblk = a.p_max / a.bm;
  if (nblk == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(nblk), a.H / kNT);
  if (a.a16) grouped_gemm_simt_kernel<true, 2><<<grid, 256, 0, s>>>(a);
  else grouped_gemm_simt_kernel<false, 2><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

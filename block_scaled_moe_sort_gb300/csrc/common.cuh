// Shared device helpers of the MoE kernels: FP8/E8M0 block quantisation and
// the 512-byte scale-factor atom layout the tcgen05 block-scaled MMA reads.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace moe {

constexpr int kMaxExperts = 512;   // expert ids fit 9 bits (route sort)
constexpr int kMaxTopk = 16;
constexpr int kMaxPrefetch = 64;   // weight L2 prefetch lead per call, k-blocks
// Stage-1 slots of the split walk (>= the GEMM grid: SMs x 2; a split tile
// takes the slot of the first CTA whose share it starts in).
constexpr int kSplitSlots = 320;
// Up to this many routes the call's front (sort + gather) is one launch.
constexpr int kFrontMaxRoutes = 256;
// Upper bound of the static shared memory of a GEMM CTA (mbarriers, flags
// and the local route layout of kMaxExperts + 1 ints).
constexpr int kStaticSmem = 512 + 4 * (kMaxExperts + 1);

// Stage-2 tile walk: feature tiles per group (route-block major inside a
// group). While the intermediate fits comfortably in L2 (decode sizes) the
// walk is route-block major (-1: all feature tiles of a route block in a
// row; measured 0.5-2.4 % faster there than feature-tile major). Once it no
// longer fits, every feature stripe of a feature-major walk re-reads all of
// it from HBM; a group of G stripes reads it once while the G stripes' FP32
// accumulator columns (M x G x 512 bytes) stay resident. Returns log2(G).
inline int stage2_n_group_log2(int64_t M, int64_t inter_bytes, int n_tiles) {
  if (inter_bytes <= (int64_t(32) << 20)) return -1;
  int lg = 0;
  while (lg < 3 && n_tiles % (2 << lg) == 0 && M * 512 * (2 << lg) <= (int64_t(32) << 20)) ++lg;
  return lg;
}

// Byte offset of (row r, 32-block i) inside a 128-row x 4-block scale atom:
// rows are split into four 32-row groups that sit side by side in each
// 16-byte line, so a 32-lane x 128-bit TMEM copy places row r's four block
// scales in lane r % 32, column r / 32.
__host__ __device__ __forceinline__ int sf_atom_off(int r, int i) {
  return (r & 31) * 16 + ((r >> 5) & 3) * 4 + (i & 3);
}

// Per-1x32 FP8 quantisation of 32 FP32 values held by one thread.
// Scale byte = max(biased_exp(amax) - 8, 0), i.e. e = floor(log2 amax) - 8
// clamped to >= -127; amax == 0 gives byte 0 and zero codes. Codes are
// round-to-nearest-even E4M3 of v * 2^-e, saturating at +-448. The scaling
// is by a power of two, so it is exact and the code is a single rounding.
__device__ __forceinline__ uint8_t quant_block32(const float* v, uint32_t* codes /*8 words*/) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  if (amax == 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i] = 0u;
    return 0;
  }
  int sb = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 8;
  sb = sb < 0 ? 0 : sb;
  const float inv = __uint_as_float(static_cast<uint32_t>(254 - sb) << 23);  // 2^(127 - sb)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(v[4 * i] * inv, v[4 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
    __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(v[4 * i + 2] * inv, v[4 * i + 3] * inv), __NV_SATFINITE, __NV_E4M3);
    codes[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return static_cast<uint8_t>(sb);
}

__device__ __forceinline__ float e8m0_to_float(uint32_t b) {
  // 2^(b-127); b = 0 gives 2^-127, a float32 subnormal
  return b == 0 ? 5.877471754111438e-39f : __uint_as_float(b << 23);
}

__device__ __forceinline__ float e2m1_to_float(uint32_t code) {
  const uint32_t mag = code & 7;
  // 0, 0.5, 1, 1.5, 2, 3, 4, 6
  const float v = mag < 2 ? 0.5f * mag : (mag < 4 ? 1.0f + 0.5f * (mag - 2) : (mag < 6 ? 2.0f + (mag - 4) : 4.0f + 2.0f * (mag - 6)));
  return (code & 8) ? -v : v;
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3);
  return __half2float(__half(hr));
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

}  // namespace moe

// MXFP4 -> BF16 for the a16w4 GEMMs without a lookup table.
//
// An MXFP4 weight is an E2M1 code times the E8M0 scale 2^(s - 127) of its
// 32-element block (OCP Microscaling Formats v1.0, the MXFP4 element and
// scale types), and every such product is a BF16 number, so the MMA can see
// the exact weights in BF16. The a16w4 weight prepack stores each 32-bit
// word of eight codes with its bits moved so that the BF16 pair of codes
// (2k, 2k+1) comes out of one or two rotations and a mask:
//
//   pair 0 = w & P,  pair 1 = rotr(w, 6) & P,  pair 2 = rotr(w, 12) & P,
//   pair 3 = (rotr(w, 2) & PA) | (rotr(w, 10) & PB),      P = PA | PB.
//
// P places a code's mantissa bit at BF16 bit 6, its two exponent bits at 7-8
// and its sign at 15 (plus 16 for the odd code of the pair). Read as BF16,
// such a half is the E2M1 value times 2^-126: the BF16 exponent field equals
// the code's exponent field e, so a normal code 2^(e-1) (1 + m/2) becomes
// 2^(e-127) (1 + m/2), and the subnormal code m/2 becomes the BF16 subnormal
// (m/2) 2^-126. One BF16 multiplication by 2^(s - 1) then applies the block
// scale exactly (s <= 128; for a larger exponent a second multiplication
// follows, a path the warp takes only when one of its rows needs it).
// Canonical order: code j of a word in bits 4j..4j+3, bit 3 the sign, bits
// 2-1 the exponent, bit 0 the mantissa (byte b holds codes 2b and 2b+1).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace moe {

constexpr uint32_t kA16P = 0x81C081C0u;
constexpr uint32_t kA16PA = 0x81808180u;
constexpr uint32_t kA16PB = 0x00400040u;

// Bit of the a16w4 word that holds canonical bit b.
__host__ __device__ constexpr int a16_dst_bit(int b) {
  const int j = b >> 2, c = b & 3, k = j >> 1;
  const int p = ((j & 1) ? 16 : 0) + (c == 3 ? 15 : 6 + c);   // its BF16 bit
  const int r = k == 0 ? 0 : k == 1 ? 6 : k == 2 ? 12 : ((p & 15) == 6 ? 10 : 2);
  return (p + r) & 31;
}

__host__ __device__ inline uint32_t a16_permute_word(uint32_t w) {
  uint32_t o = 0;
  for (int b = 0; b < 32; ++b) o |= ((w >> b) & 1u) << a16_dst_bit(b);
  return o;
}

__device__ __forceinline__ uint32_t a16_bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 z = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&z);
}

// The 16 tiny BF16 pairs (E2M1 value times 2^-126, K order) of one
// 32-element block from its four a16w4 words.
__device__ __forceinline__ void a16_tiny_block(const uint4 v, uint32_t (&t)[16]) {
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w = words[i];
    t[4 * i + 0] = w & kA16P;
    t[4 * i + 1] = __funnelshift_r(w, w, 6) & kA16P;
    t[4 * i + 2] = __funnelshift_r(w, w, 12) & kA16P;
    t[4 * i + 3] = (__funnelshift_r(w, w, 2) & kA16PA) | (__funnelshift_r(w, w, 10) & kA16PB);
  }
}

// Nonzero iff one of the four E8M0 bytes of `sfw` exceeds 128 (2^(s-1) past
// the BF16 range): per byte, the top bit and a nonzero low part.
__host__ __device__ constexpr uint32_t a16_big_scales(uint32_t sfw) {
  return (sfw & 0x80808080u) & ((sfw & 0x7F7F7F7Fu) + 0x7F7F7F7Fu);
}

// BF16 pair 2^(s-1) of block c for scale bytes all <= 128: t = sfw +
// 0x7E7E7E7E holds s + 126 per byte (no carries), the BF16 exponent field.
__device__ __forceinline__ uint32_t a16_scale_pair(uint32_t t, int c) {
  const uint32_t b = (t >> (8 * c)) & 0xFFu;
  return b * 0x00800080u;
}

// For a scale byte above 128 the block is converted with the pair of 128
// (2^127: the tiny values times 2^127 stay at most 12) and then multiplied
// by this second pair, 2^(s - 128); s = 255, the NaN scale, gives
// infinities (NaN for the zero codes). For s <= 128 the pair is 1.
__device__ __forceinline__ uint32_t a16_big_pair(uint32_t s) {
  const uint32_t h = s == 255u ? 0x7F80u : ((s > 128u ? s : 128u) - 1u) << 7;
  return h * 0x00010001u;
}

// Pair of the first multiplication for any scale byte: 2^(min(s, 128) - 1).
__device__ __forceinline__ uint32_t a16_first_pair(uint32_t s) {
  return ((s < 128u ? s : 128u) + 126u) * 0x00800080u;
}

// The 16 BF16 pairs (K order) of one block from its four a16w4 words: the
// tiny values times the pair sc (a16_scale_pair, or a16_first_pair and then
// a16_big_pair for a scale byte above 128).
__device__ __forceinline__ void a16_dequant_block(const uint4 v, uint32_t sc, uint32_t (&out)[16]) {
  uint32_t t[16];
  a16_tiny_block(v, t);
#pragma unroll
  for (int i = 0; i < 16; ++i) out[i] = a16_bf16x2_mul(t[i], sc);
}

}  // namespace moe

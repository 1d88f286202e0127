// One new key or value row into the paged cache, by one warp: the rule of the KV append
// (the step before attention in every decode step writes each sequence's new rows into its
// cache, Step-3 page section 7 "Implementation and Results"), shared by the append kernel and
// the decode kernel's fused append.  Lane l holds elements 8 l .. 8 l + 7 of the 256-element
// bf16 row (x).  The cache formats:
//   bf16  : the bits, unchanged;
//   e4m3  : one fp32 scale s = absmax / 448 (1 for an all-zero row), codes e4m3(x / s) rounded
//           to nearest even and saturated to +-448 (section 5 "Model-System Co-design": 8-bit KV);
//   MXFP4 : per block of 32 elements one E8M0 scale 2^(floor(log2 amax) - 2) and E2M1 codes of
//           x over it, rounded to nearest even and saturated to 6 (the 4-bit reading of the
//           page's further KV quantisation, section 5 "Quantization and MTP").
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "mfa.h"

namespace mfa {

constexpr int kRowElems = 256;        // elements of a cache row (MFA head width)
constexpr float kE4m3Max = 448.0f;    // largest finite e4m3 value

// Two fp32 values to two e4m3 codes (round to nearest even, saturate to +-448): lo in the
// low byte.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight non-negative fp32 values to eight E2M1 codes (round to nearest even, saturate to 6),
// element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t e2m1x8_rn_sat(const float (&a)[8]) {
  uint32_t r;
  // (the first source of each pair goes to the high nibble)
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(a[0]), "f"(a[1]), "f"(a[2]), "f"(a[3]), "f"(a[4]), "f"(a[5]), "f"(a[6]), "f"(a[7]));
  return r;
}

__device__ __forceinline__ float bf16_bits_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_bits_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Row `row` (= page * 64 + slot) of `cache` (and `scale`: fp32 per row for e4m3, 8 E8M0 bytes
// per row for MXFP4, unused for bf16) in format kv.  All 32 lanes call it with their x.
__device__ __forceinline__ void append_row_warp(int kv, uint4 x, int lane, void* cache, void* scale, size_t row) {
  if (kv == MFA_KV_MXFP4) {
    // lanes 4j .. 4j + 3 hold block j (elements 32 j .. 32 j + 31)
    float f[8] = {bf16_bits_lo(x.x), bf16_bits_hi(x.x), bf16_bits_lo(x.y), bf16_bits_hi(x.y),
                  bf16_bits_lo(x.z), bf16_bits_hi(x.z), bf16_bits_lo(x.w), bf16_bits_hi(x.w)};
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    // scale 2^e, e = floor(log2 amax) - 2 = E - 129 for amax's biased exponent E, clamped to
    // -127 (E < 2, zero and subnormal blocks included): the byte e + 127 = max(E - 2, 0)
    const uint32_t E = (__float_as_uint(am) >> 23) & 0xFFu;
    const uint32_t sb = E > 2u ? E - 2u : 0u;
    const float inv = __uint_as_float((254u - sb) << 23);   // 2^-e, a normal number (sb <= 252)
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = fabsf(f[i]) * inv;   // exact, or tiny enough to round to 0
    uint32_t sign = 0;   // bit 3 of each nibble: the sign of its element (-0 included)
#pragma unroll
    for (int i = 0; i < 8; ++i) sign |= (__float_as_uint(f[i]) >> 31) << (4 * i + 3);
    reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(cache) + row * (kRowElems / 2))[lane] = e2m1x8_rn_sat(a) | sign;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      lo |= __shfl_sync(0xffffffffu, sb, 4 * j) << (8 * j);
      hi |= __shfl_sync(0xffffffffu, sb, 16 + 4 * j) << (8 * j);
    }
    if (lane == 0)
      reinterpret_cast<uint2*>(static_cast<uint8_t*>(scale))[row] = make_uint2(lo, hi);
    return;
  }
  if (kv == MFA_KV_BF16) {
    uint4* dst = static_cast<uint4*>(cache) + row * (kRowElems / 8) + lane;
    *dst = x;
    return;
  }
  float f[8] = {bf16_bits_lo(x.x), bf16_bits_hi(x.x), bf16_bits_lo(x.y), bf16_bits_hi(x.y),
                bf16_bits_lo(x.z), bf16_bits_hi(x.z), bf16_bits_lo(x.w), bf16_bits_hi(x.w)};
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  const float s = (am > 0.f) ? __fdiv_rn(am, kE4m3Max) : 1.f;
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = e4m3x2_rn_sat(__fdiv_rn(f[2 * i], s), __fdiv_rn(f[2 * i + 1], s));
  uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + row * kRowElems) + lane;
  *dst = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  if (lane == 0) static_cast<float*>(scale)[row] = s;
}

}  // namespace mfa

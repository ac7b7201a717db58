// Device codecs of the CSA2 KV formats ("DeepSeek V4.1: model architecture and
// system design, a close reading" section 2.3; "DeepSeek-V4.1-Flash: Pushing
// the Limits of KV Cache Compression" section 3.6):
//   MXFP4 = E2M1 codes with one E4M3 scale per 16 channels, no global scale;
//   FP8   = E4M3 without scale (sliding-window KV).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace csa2 {

// fp32 -> E4M3, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint8_t e4m3_from_f32(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
  return static_cast<uint16_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Two E4M3 bytes -> f16x2 (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t b) {
  const uint32_t h2 = e4m3x2_to_f16x2(b);
  return __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFFu)));
}

// Two E2M1 codes in one byte (low nibble -> low half) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(byte));
  return r;
}

// One 16-channel MXFP4 block: scale byte and 8 code bytes (channel 2i in the
// low nibble of byte i). The E2M1 magnitude code of |v| / scale is the nearest
// grid value {0, .5, 1, 1.5, 2, 3, 4, 6} with ties to the even code and
// saturation at 6. It is found by comparing |v| with the midpoints times the
// scale; those products are exact in fp32, so no division by the scale is
// rounded.
__device__ __forceinline__ void mxfp4_block(const float (&v)[16], uint8_t& scale,
                                            uint32_t& codes_lo, uint32_t& codes_hi) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  scale = e4m3_from_f32(__fdiv_rn(amax, 6.0f));
  const float sf = e4m3_to_f32(scale);
  const float t0 = 0.25f * sf, t1 = 0.75f * sf, t2 = 1.25f * sf, t3 = 1.75f * sf,
              t4 = 2.5f * sf, t5 = 3.5f * sf, t6 = 5.0f * sf;
  uint32_t c[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float a = fabsf(v[i]);
    uint32_t k = (a > t0) + (a >= t1) + (a > t2) + (a >= t3) + (a > t4) + (a >= t5) + (a > t6);
    if (sf == 0.f) k = 0;
    if (k != 0 && v[i] < 0.f) k |= 8u;
    c[i] = k;
  }
  codes_lo = 0;
  codes_hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) codes_lo |= (c[2 * i] | (c[2 * i + 1] << 4)) << (8 * i);
#pragma unroll
  for (int i = 0; i < 4; ++i) codes_hi |= (c[8 + 2 * i] | (c[8 + 2 * i + 1] << 4)) << (8 * i);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Dequantises 16 bytes of E2M1 codes (32 channels) with the two scales of
// their blocks into 32 f16 values (exact: an E2M1 value times an E4M3 scale
// has at most 6 significant bits and lies within f16's normal range).
__device__ __forceinline__ void dequant32_f16(const uint4 codes, uint16_t scales2, uint4 (&out)[4]) {
  const uint32_t s2 = e4m3x2_to_f16x2(scales2);
  const __half2 sc0 = __low2half2(*reinterpret_cast<const __half2*>(&s2));
  const __half2 sc1 = __high2half2(*reinterpret_cast<const __half2*>(&s2));
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
  uint32_t o[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 sc = (i < 2) ? sc0 : sc1;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t h = e2m1x2_to_f16x2((w[i] >> (8 * b)) & 0xFFu);
      __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h), sc);
      o[4 * i + b] = *reinterpret_cast<uint32_t*>(&v);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) out[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
}

}  // namespace csa2

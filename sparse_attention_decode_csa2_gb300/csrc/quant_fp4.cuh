// One FP4 main-KV row from 512 fp32 latent channels, by one warp
// (DeepSeek-V4.1-Flash paper walkthrough, 1.(5).4 "FP4 Main KV Cache": E2M1
// codes, one E4M3 scale per 16 channels, no global scale).
//
// Lane l holds channels 4l..4l+3 (+128 i), so each 16-channel block sits in
// 4 consecutive lanes and its absmax is two shuffles away.  The row is
// assembled in a 288-byte shared-memory buffer of the warp and written out as
// 18 16-byte vectors.
//
// Rounding is bit-exact with respect to the exact quotients:
//  * scale: fp32 absmax/6 is rounded once by IEEE division, then converted to
//    E4M3 with round-to-nearest-even.  The fp32 quotient can equal an E4M3
//    rounding midpoint only when the exact quotient does (an fp32 dividend
//    next to 6 x midpoint lies at least 4 fp32 ulps of the midpoint away), so
//    the double rounding never changes the result.
//  * codes: instead of rounding the inexact fp32 |x|/s, |x| is compared with
//    the seven E2M1 midpoints times s.  Each product t*s (t has <= 3
//    significant bits, s <= 4) is exact in fp32.  Strict / non-strict
//    comparisons encode ties-to-even: 0.25, 1.25, 2.5 and 5 round down,
//    0.75, 1.75 and 3.5 round up.
#pragma once
#include "csa2_internal.cuh"

namespace csa2 {

__device__ __forceinline__ uint32_t e2m1_code(float x, float s) {
  uint32_t sign = __float_as_uint(x) >> 31;
  float m = fabsf(x);
  uint32_t c = 0;
  if (s > 0.0f) {
    c = (m > 0.25f * s) + (m >= 0.75f * s) + (m > 1.25f * s) + (m >= 1.75f * s) +
        (m > 2.5f * s) + (m >= 3.5f * s) + (m > 5.0f * s);
  }
  return (sign << 3) | c;
}

// x: the row's 512 channels (16-byte aligned, read-only); dst: the row's 288
// bytes (16-byte aligned); buf: this warp's 288-byte shared buffer.
__device__ __forceinline__ void quantize_fp4_row_warp(const float* __restrict__ x,
                                                      uint8_t* __restrict__ dst, uint8_t* buf,
                                                      int lane) {
  const float4* xr = reinterpret_cast<const float4*>(x);
  float4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __ldg(xr + lane + 32 * i);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a = fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w)));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    uint32_t sbyte = f32_to_e4m3_satfinite(a / 6.0f);
    float s = half2_bits_to_float2(e4m3x2_to_f16x2((uint16_t)sbyte)).x;
    uint32_t c0 = e2m1_code(v[i].x, s), c1 = e2m1_code(v[i].y, s);
    uint32_t c2 = e2m1_code(v[i].z, s), c3 = e2m1_code(v[i].w, s);
    uint16_t packed = (uint16_t)((c0 | (c1 << 4)) | ((c2 | (c3 << 4)) << 8));
    // channels 4*lane + 128*i .. +3 -> code bytes 2*lane + 64*i, +1
    *reinterpret_cast<uint16_t*>(buf + 2 * lane + 64 * i) = packed;
    if ((lane & 3) == 0) buf[kCodeBytes + (lane >> 2) + 8 * i] = (uint8_t)sbyte;
  }
  __syncwarp();
  if (lane < kRowBytes / 16)
    *reinterpret_cast<uint4*>(dst + 16 * lane) = *reinterpret_cast<const uint4*>(buf + 16 * lane);
  __syncwarp();
}

}  // namespace csa2

// MXFP8 quantisation of bf16 rows held eight values per lane (the ring
// producers' and the activation gradient's form) or sixteen (the
// dispatch's), and the non-coherent 16-byte load they read rows with.
#pragma once
#include <cuda_fp8.h>

#include "common.cuh"

namespace mok {

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Smallest e with amax <= 448 * 2^e for a finite amax >= 0: with
// amax = 1.f * 2^E, 448 = 1.75 * 2^8, e = E - 8 if 1.f <= 1.75 else E - 7.
// Zero and subnormal amax give the E8M0 minimum, -127.
__device__ __forceinline__ int mx_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int eb = static_cast<int>((b >> 23) & 0xFFu);
  if (eb == 0) return -127;
  const int e = eb - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// E4M3 codes of 8 values held by one lane when 4 consecutive lanes hold one
// 32-value block: the block's amax by two xor shuffles (warp-wide call),
// scale 2^e with e = mx_exponent(amax), codes packed little-endian.
__device__ __forceinline__ uint2 mx_codes8(const float (&f)[8], int& e) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  e = mx_exponent(amax);
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
  uint32_t packed[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * j] * inv, f[4 * j + 1] * inv),
                                                             __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * j + 2] * inv, f[4 * j + 3] * inv),
                                                             __NV_SATFINITE, __NV_E4M3);
    packed[j] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint2(packed[0], packed[1]);
}

// The scale word of the 128 columns held by lanes 16h .. 16h + 15 (8 values
// each): byte b from lane 16h + 4b (warp-wide call).
__device__ __forceinline__ uint32_t mx_word16(int e, int lane) {
  const uint32_t byte = static_cast<uint32_t>(e + 127);
  const int base = lane & 16;
  return __shfl_sync(0xffffffffu, byte, base) | (__shfl_sync(0xffffffffu, byte, base + 4) << 8) |
         (__shfl_sync(0xffffffffu, byte, base + 8) << 16) | (__shfl_sync(0xffffffffu, byte, base + 12) << 24);
}

// E4M3 codes of 16 values held by one lane when 2 consecutive lanes hold
// one 32-value block: the block's amax by one xor shuffle (warp-wide call),
// then the same scale and conversions as mx_codes8, codes packed
// little-endian.
__device__ __forceinline__ uint4 mx_codes16(const float (&f)[16], int& e) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  e = mx_exponent(amax);
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
  uint32_t packed[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * j] * inv, f[4 * j + 1] * inv),
                                                             __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * j + 2] * inv, f[4 * j + 3] * inv),
                                                             __NV_SATFINITE, __NV_E4M3);
    packed[j] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

// The scale word of the 128 columns held by lanes 8h .. 8h + 7 (16 values
// each): byte b from lane 8h + 2b (warp-wide call).
__device__ __forceinline__ uint32_t mx_word8(int e, int lane) {
  const uint32_t byte = static_cast<uint32_t>(e + 127);
  const int base = lane & 24;
  return __shfl_sync(0xffffffffu, byte, base) | (__shfl_sync(0xffffffffu, byte, base + 2) << 8) |
         (__shfl_sync(0xffffffffu, byte, base + 4) << 16) | (__shfl_sync(0xffffffffu, byte, base + 6) << 24);
}

}  // namespace mok

// Device helpers shared by the MXFP8 quantisers (OCP MX v1.0, E4M3 elements,
// emax = 8): the block scale exponent and the scaled E4M3 encoding.
#pragma once
#include <cstdint>
#include <cuda_fp8.h>

namespace moe {

// floor(log2(amax)) - 8 clamped to [-127, 127] (-127 for an all-zero block),
// read from amax's exponent bits (leading-bit position for a subnormal).
__device__ __forceinline__ int mx_scale_exponent(float amax) {
  if (!(amax > 0.0f)) return -127;
  const uint32_t b = __float_as_uint(amax);
  const int ex = static_cast<int>(b >> 23);
  const int fl = ex ? ex - 127 : -149 + (31 - __clz(static_cast<int>(b)));
  return max(-127, min(127, fl - 8));
}

// 2^-e for a block exponent e in [-127, 119] (every finite bf16 amax).
__device__ __forceinline__ float mx_inv_scale(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

// Codes of f[0..7] * inv: E4M3, round to nearest even, saturating at +-448.
__device__ __forceinline__ uint2 mx_encode8(const float (&f)[8], float inv) {
  uint32_t w[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(f[4 * i] * inv, f[4 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(f[4 * i + 2] * inv, f[4 * i + 3] * inv), __NV_SATFINITE, __NV_E4M3);
    w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint2(w[0], w[1]);
}

// One 32-element block of bf16 (four 16-byte words, in order): its E8M0
// scale byte (exponent + 127) and its 32 E4M3 codes (c0: elements 0..15,
// c1: 16..31), element i encoded as x_i * 2^-e.
__device__ __forceinline__ uint8_t mx_quant_block32(const uint4 (&v)[4], uint4& c0, uint4& c1) {
  float f[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t ws[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[8 * i + 2 * j] = __uint_as_float(ws[j] << 16);
      f[8 * i + 2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u);
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  const int e = mx_scale_exponent(amax);
  const float inv = mx_inv_scale(e);
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(f[4 * i] * inv, f[4 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(f[4 * i + 2] * inv, f[4 * i + 3] * inv), __NV_SATFINITE, __NV_E4M3);
    out[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  c0 = make_uint4(out[0], out[1], out[2], out[3]);
  c1 = make_uint4(out[4], out[5], out[6], out[7]);
  return static_cast<uint8_t>(e + 127);
}

}  // namespace moe

// Shared device helpers of the decode-step kernels: row codecs, paging, warp reductions.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/dsv4.h"

namespace dsv4 {

constexpr int D = DSV4_LATENT_DIM;      // 576
constexpr int DV = DSV4_VALUE_DIM;      // 512
constexpr int D_NOPE = 512;
constexpr int D_ROPE = DSV4_ROPE_DIM;   // 64
constexpr int FP8_REC = DSV4_FP8_DS_MLA_BYTES;  // 656
constexpr int FP8_ROPE_OFF = 512;
constexpr int FP8_SCALE_OFF = 640;

// range-check flag bits (see dsv4_read_device_flags)
constexpr uint32_t FLAG_PAGE = 1u;
constexpr uint32_t FLAG_TOPK = 2u;

__host__ __device__ inline int64_t row_bytes(int dtype, int width) {
  switch (dtype) {
    case DSV4_F32: return 4LL * width;
    case DSV4_BF16: return 2LL * width;
    case DSV4_FP8_DS_MLA: return FP8_REC;
    case DSV4_I8_ROWSCALE: return width + 4;
    case DSV4_MXFP4: return width / 2 + width / 32;
  }
  return 0;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// Two e4m3fn codes (low byte first) -> two floats, exact (e4m3 -> f16 is exact).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)codes, __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// UE8M0 block exponent: the smallest integer e with 448 * 2^e >= amax, from the bits of amax.
// 448 = 1.75 * 2^8: with amax = f * 2^E (f in [1,2)), e = E - 8 when f <= 1.75, else E - 7.
__device__ __forceinline__ int ue8m0_exponent(float amax) {
  uint32_t bits = __float_as_uint(amax);
  if (amax == 0.0f) return 0;
  int E = (int)((bits >> 23) & 0xFF) - 127;
  uint32_t mant = bits & 0x7FFFFF;
  if (E == -127) return -127;  // subnormal block max: the smallest scale covers it
  int e = (mant <= 0x600000u) ? E - 8 : E - 7;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as an exact float for e in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float exp2_neg_int(int e) {
  int b = 127 - e;
  return b >= 1 ? __uint_as_float((uint32_t)b << 23) : __uint_as_float(0x00400000u);
}

// Scale of a UE8M0 byte: 2^(byte - 127), exact.
__device__ __forceinline__ float ue8m0_scale(uint8_t byte) {
  return byte >= 1 ? __uint_as_float((uint32_t)byte << 23) : __uint_as_float(0x00400000u);
}

// E2M1 code (low 4 bits: sign, 2 exponent bits with bias 1, 1 mantissa bit) -> float, exact.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t ee = (c >> 1) & 3u, m = c & 1u;
  const float mag = ee == 0u ? 0.5f * (float)m : __uint_as_float(((ee + 126u) << 23) | (m << 22));
  return (c & 8u) ? -mag : mag;
}

// E2M1 code of x (round to nearest, ties to the even code, saturating to +-6; the sign of x, zero
// included, kept): the magnitude code counts the grid midpoints 0.25, 0.75, ..., 5 below |x|, with a
// tie going to the even code.
__device__ __forceinline__ uint32_t e2m1_code(float x) {
  const float a = fabsf(x);
  const uint32_t c = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) + (uint32_t)(a >= 1.75f) +
                     (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
  return c | (signbit(x) ? 8u : 0u);
}

// MXFP4 block exponent: the smallest integer e with 6 * 2^e >= amax, from the bits of amax (with
// amax = f * 2^E, f in [1, 2): e = E - 2 when f <= 1.5, else E - 1), clamped to [-127, 127]; 0 for 0.
__device__ __forceinline__ int mxfp4_exponent(float amax) {
  if (amax == 0.0f) return 0;
  const uint32_t bits = __float_as_uint(amax);
  const int E = (int)((bits >> 23) & 0xFF) - 127;
  if (E == -127) return -127;
  const int e = ((bits & 0x7FFFFFu) <= 0x400000u) ? E - 2 : E - 1;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

__device__ __forceinline__ uint16_t float2_to_e4m3x2(float a, float b) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ uint32_t float2_to_bf16x2_bits(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Encodes one 576-dim row held as 288 pairs, pair i = dims (2i, 2i+1) owned by thread i of a
// 288-thread group (9 warps).  Warp w < 8 owns no-pe block w (64 dims) and computes its UE8M0
// exponent with a warp max; warp 8 owns the rope dims.
__device__ __forceinline__ void encode_pair_store(int dtype, uint8_t* row, int i, float x0, float x1) {
  if (dtype == DSV4_F32) {
    reinterpret_cast<float2*>(row)[i] = make_float2(x0, x1);
  } else if (dtype == DSV4_BF16) {
    reinterpret_cast<uint32_t*>(row)[i] = float2_to_bf16x2_bits(x0, x1);
  } else {  // DSV4_FP8_DS_MLA
    const int w = i >> 5, lane = i & 31;
    if (w < 8) {
      float amax = warp_max(fmaxf(fabsf(x0), fabsf(x1)));
      int e = ue8m0_exponent(amax);
      float s = exp2_neg_int(e);
      reinterpret_cast<uint16_t*>(row)[i] = float2_to_e4m3x2(x0 * s, x1 * s);
      if (lane == 0) row[FP8_SCALE_OFF + w] = (uint8_t)(e + 127);
    } else {
      reinterpret_cast<uint32_t*>(row + FP8_ROPE_OFF)[lane] = float2_to_bf16x2_bits(x0, x1);
      if (lane == 0) *reinterpret_cast<uint2*>(row + 648) = make_uint2(0u, 0u);
    }
  }
}

// Decodes dims (2i, 2i+1) of a stored 576-dim row.
__device__ __forceinline__ float2 decode_pair(int dtype, const uint8_t* row, int i) {
  if (dtype == DSV4_F32) return reinterpret_cast<const float2*>(row)[i];
  if (dtype == DSV4_BF16) {
    uint32_t v = reinterpret_cast<const uint32_t*>(row)[i];
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
  }
  if (i < 256) {
    float2 f = e4m3x2_to_float2(reinterpret_cast<const uint16_t*>(row)[i]);
    float s = ue8m0_scale(row[FP8_SCALE_OFF + (i >> 5)]);
    return make_float2(f.x * s, f.y * s);
  }
  uint32_t v = reinterpret_cast<const uint32_t*>(row + FP8_ROPE_OFF)[i - 256];
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

}  // namespace dsv4

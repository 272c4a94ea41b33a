// e4m3 helpers of the FP8 tensor-core paths: packing, and the split of an
// fp32 value into two e4m3 terms (hi = e4m3(x), lo = e4m3(x - hi)) whose sum
// carries about 7 significant bits more than hi alone.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "va_split.cuh"

namespace va {

__device__ __forceinline__ uint32_t pack_fp8x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float2 unpack_fp8x2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  return __half22float2(__half2(h));
}

// p (two fp32 values, a first) -> e4m3 hi and lo bytes, via f16x2.
__device__ __forceinline__ void split_p(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const __nv_fp8x2_storage_t h8 = __nv_cvt_halfraw2_to_fp8x2(__half2_raw(h), __NV_SATFINITE, __NV_E4M3);
  const __half2 hh = __half2(__nv_cvt_fp8x2_to_halfraw2(h8, __NV_E4M3));
  const __half2 r = __hsub2(h, hh);
  const __nv_fp8x2_storage_t l8 = __nv_cvt_halfraw2_to_fp8x2(__half2_raw(r), __NV_SATFINITE, __NV_E4M3);
  hi = (uint32_t)h8;
  lo = (uint32_t)l8;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)float_to_bf16_bits(lo) | ((uint32_t)float_to_bf16_bits(hi) << 16);
}

}  // namespace va

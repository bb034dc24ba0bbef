// Element access of the output C in its storage type: fp32, or fp16 / bf16
// (the extra rounding stage of a 16-bit output: the fp32 result
// alpha*acc + beta*C is rounded once, to nearest even, when stored).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace mpg {

enum : int { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };

__device__ __forceinline__ float out_load(const void* base, int64_t idx, int dt) {
  if (dt == kOutF16) return __half2float(reinterpret_cast<const __half*>(base)[idx]);
  if (dt == kOutBF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}

__device__ __forceinline__ void out_store(void* base, int64_t idx, float v, int dt) {
  if (dt == kOutF16) reinterpret_cast<__half*>(base)[idx] = __float2half_rn(v);
  else if (dt == kOutBF16) reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
  else reinterpret_cast<float*>(base)[idx] = v;
}

// Four consecutive elements starting at idx (idx * element size aligned to
// the 4-element vector: 16 bytes for fp32, 8 bytes for 16-bit types).
__device__ __forceinline__ float4 out_load4(const void* base, int64_t idx, int dt) {
  if (dt == kOutF32) return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx);
  const uint2 w = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(base) + idx);
  float4 v;
  if (dt == kOutF16) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
    v = make_float4(a.x, a.y, b.x, b.y);
  } else {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    v = make_float4(a.x, a.y, b.x, b.y);
  }
  return v;
}

__device__ __forceinline__ void out_store4(void* base, int64_t idx, float4 v, int dt) {
  if (dt == kOutF32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx) = v;
    return;
  }
  uint2 w;
  if (dt == kOutF16) {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    w = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    w = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
  *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(base) + idx) = w;
}

}  // namespace mpg

// nvfp4.cuh -- NVFP4 (E2M1 values, E4M3 block scales) rounding helpers of the
// QAT path ("NVFP4 Attention QAT Backward" page, Overview): a block of 16 values
// gets the local scale s = E4M3(amax / 6); each value becomes E2M1(x / s) * s.
// Both divisions are correctly rounded fp32 divisions; the E4M3 and E2M1
// roundings are the hardware conversions (nearest, ties to even, saturating).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace sdpa {

// Two fp32 values rounded to E4M3 / E2M1 and widened back to fp32; `a` -> .x.
// (The packing conversions put their first source in the upper half, and the
// half2 -> float2 widening reads .x from the lower half, so `b` goes first.)
__device__ __forceinline__ float2 round_e4m3x2(float a, float b) {
  uint16_t e;
  uint32_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(e) : "f"(b), "f"(a));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(e));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}
__device__ __forceinline__ float2 round_e2m1x2(float a, float b) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h) : "f"(b), "f"(a));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Local scales of two blocks with maxima amax0, amax1.
__device__ __forceinline__ float2 nvfp4_scales(float amax0, float amax1) {
  return round_e4m3x2(__fdiv_rn(amax0, 6.0f), __fdiv_rn(amax1, 6.0f));
}

// Fake NVFP4 of two values x0, x1 whose blocks have the local scales s0, s1
// (a zero scale gives 0), as a bf16 pair (exact: E2M1 times E4M3 fits in bf16).
__device__ __forceinline__ uint32_t fake_nvfp4_pair_bf16(float x0, float x1, float s0, float s1) {
  const float y0 = s0 > 0.f ? __fdiv_rn(x0, s0) : 0.f;
  const float y1 = s1 > 0.f ? __fdiv_rn(x1, s1) : 0.f;
  const float2 q = round_e2m1x2(y0, y1);
  return pack_bf16x2(q.x * s0, q.y * s1);
}

}  // namespace sdpa

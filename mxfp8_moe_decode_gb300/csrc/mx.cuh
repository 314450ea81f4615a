// MXFP8 device arithmetic: the E8M0 code of a 32-group, its quant
// multiplier, and E4M3 conversion.
//
// "vllm.models.deepseek_v41.amd.mono.attention.device", mx_code: the code is
// clamp(ceil(log2(amax / 448)) + 127, 0, 254) with amax floored at FLT_MIN;
// div_rn: the quotient is the IEEE single division; ceil_exp: the biased
// exponent of the smallest power of two >= q, read from the bits of q.
// mx_mul: the quant multiplier 2^(127 - code) built from its bit pattern.
// "vllm.models.deepseek_v41.amd.mono.layer", store_x8: clamp to the E4M3 range,
// then round to nearest even (fp8_pack4).
//
// ceil_exp is stated for a normal q; for a subnormal q (amax < 448 * 2^-126)
// the formula itself is used: ceil(log2 q) + 127 is 1 for q in
// (2^-127, 2^-126) and <= 0 below, clamped to 0. This keeps the code exact
// for every finite amax. (Requires IEEE division without flush-to-zero,
// which is nvcc's default without --use_fast_math.)
#pragma once

#include <cuda_fp8.h>

#include <cfloat>
#include <cstdint>

namespace moe {

__device__ __forceinline__ int mx_code(float amax) {
  const float a = fmaxf(amax, FLT_MIN);
  const float q = __fdiv_rn(a, 448.0f);
  const uint32_t b = __float_as_uint(q);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  int code;
  if (e == 0) {
    code = (q > 0x1p-127f) ? 1 : 0;
  } else {
    code = e + ((b & 0x7FFFFFu) != 0u ? 1 : 0);
  }
  return min(max(code, 0), 254);
}

// 2^(127 - code) for code in [0, 253] (bit construction, exact).
__device__ __forceinline__ float mx_mul(int code) {
  return __uint_as_float(static_cast<uint32_t>(254 - code) << 23);
}

__device__ __forceinline__ float clamp_e4m3(float v) {
  return fminf(fmaxf(v, -448.0f), 448.0f);
}

// Two floats -> two E4M3 bytes (lo in the low byte), round to nearest even.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint8_t e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

}  // namespace moe

// The store of one 16-byte chunk of a new K/V row into the pool, and the FP8
// quantisation it uses (device code shared by the append kernel and the
// split-KV kernel's append CTAs of the fused call).
#pragma once
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace pkv {

// The fp32 quotient x / scale, correctly rounded.  For a scale that is a
// power of two with a normal reciprocal, x times that reciprocal rounds the
// same real number and is the same float (overflow and subnormal results
// included), without a division; any other scale divides.  The test is the
// same for every thread (one scale per pool).
__device__ __forceinline__ float quant_div(float x, float scale) {
  const uint32_t sb = __float_as_uint(scale);   // scale > 0
  const uint32_t e = sb >> 23;
  if ((sb & 0x7fffffu) == 0 && e >= 1u && e <= 253u) return x * __uint_as_float((254u - e) << 23);
  return __fdiv_rn(x, scale);
}

// Four bf16 (two packed words, lowest element in the low half) -> four e4m3
// codes, lowest element in the lowest byte: the code nearest (ties to even)
// to the fp32 quotient x / scale, finite values beyond 448 saturating (the
// conversion's satfinite mode).
__device__ __forceinline__ uint32_t quant_e4m3x4(uint32_t w0, uint32_t w1, float scale) {
  const float x0 = __uint_as_float(w0 << 16), x1 = __uint_as_float(w0 & 0xffff0000u);
  const float x2 = __uint_as_float(w1 << 16), x3 = __uint_as_float(w1 & 0xffff0000u);
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(quant_div(x0, scale), quant_div(x1, scale)), __NV_SATFINITE,
                                               __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(quant_div(x2, scale), quant_div(x3, scale)), __NV_SATFINITE,
                                               __NV_E4M3);
  return lo | (hi << 16);
}

// Two bf16 (one packed word) -> two e4m3 codes (lowest element in the low byte).
__device__ __forceinline__ uint32_t quant_e4m3x2(uint32_t w, float scale) {
  const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xffff0000u);
  return __nv_cvt_float2_to_fp8x2(make_float2(quant_div(x0, scale), quant_div(x1, scale)), __NV_SATFINITE,
                                  __NV_E4M3);
}

// Stores one chunk (8 bf16 of K and of V) at chunk index dst of the pool.
// F8: quantised to 8 codes each.
template <bool F8>
__device__ __forceinline__ void append_store(void* __restrict__ kp, void* __restrict__ vp, int64_t dst, uint4 kx,
                                             uint4 vx, float k_scale, float v_scale) {
  if constexpr (F8) {
    static_cast<uint2*>(kp)[dst] = make_uint2(quant_e4m3x4(kx.x, kx.y, k_scale), quant_e4m3x4(kx.z, kx.w, k_scale));
    static_cast<uint2*>(vp)[dst] = make_uint2(quant_e4m3x4(vx.x, vx.y, v_scale), quant_e4m3x4(vx.z, vx.w, v_scale));
  } else {
    static_cast<uint4*>(kp)[dst] = kx;
    static_cast<uint4*>(vp)[dst] = vx;
  }
}

}  // namespace pkv

// spa_kvwrite_quant.cuh - e4m3 codes of x / scale for the paged KV write (FreeToken clone PR 3,
// "Perf/kv fp8 read path": one fp32 scale per token and kv_head row, scale = max|x| / 448).
//
// The code of an element is the e4m3 rounding (nearest even, saturating) of its binary32 quotient
// x / scale.  One IEEE division per element costs more issue slots than the row's memory traffic,
// so the quotient is taken by Markstein's method (a correctly rounded reciprocal, then one
// correction step with the exact residual; P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", 1990):
//   r = RN(1 / scale),  q0 = RN(x r),  e = x - q0 scale  (exact, one fma),  q = RN(q0 + e r).
// A zero quotient takes the sign of x (the correction would turn -0 into +0).  The residual is exact
// while it stays in the normal range, about |x| >= 2^-100.  An element's code can differ from zero
// only if |x / scale| >= 2^-11 (half of e4m3's smallest step is 2^-10), so rows with scale >= 2^-88
// take this path (kvq_fast_scale): there every element whose code matters has |x| >= 2^-99, and
// the others give a zero of x's sign on both paths.  Rows with a smaller scale divide.  Every
// input the write can see was checked: for every positive finite bf16 row
// maximum and every bf16 x up to it, both signs, the code equals that of the IEEE quotient
// (tests/kvwrite_quant_check.cu).
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

namespace spa {

__device__ __forceinline__ float kvq_bf16_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint32_t kvq_e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// True when the row's scale allows the reciprocal path.
__device__ __forceinline__ bool kvq_fast_scale(float scale) {
  return scale >= 0x1p-88f && scale <= 0x1p126f;
}

// x / scale by one correction step from r = RN(1 / scale).
__device__ __forceinline__ float kvq_div(float x, float scale, float r) {
  const float q0 = x * r;
  const float e = fmaf(-q0, scale, x);
  return copysignf(fmaf(e, r, q0), x);
}

// Eight bf16 values (a 16-byte chunk) -> eight e4m3 codes of x / scale, first value in the lowest
// byte.  r = RN(1 / scale); fast = kvq_fast_scale(scale), else IEEE divisions.
__device__ __forceinline__ uint2 kvq_chunk(const uint4& u, float scale, float r, bool fast) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t c[4];
  if (fast) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c[i] = kvq_e4m3x2(kvq_div(kvq_bf16_to_f32(w[i] & 0xFFFFu), scale, r),
                        kvq_div(kvq_bf16_to_f32(w[i] >> 16), scale, r));
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c[i] = kvq_e4m3x2(__fdiv_rn(kvq_bf16_to_f32(w[i] & 0xFFFFu), scale),
                        __fdiv_rn(kvq_bf16_to_f32(w[i] >> 16), scale));
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

}  // namespace spa

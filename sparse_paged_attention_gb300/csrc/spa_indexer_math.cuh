// spa_indexer_math.cuh - the element arithmetic of the indexer kernels, callable on the host too
// so that the very code the kernels run can be checked on a CPU against the oracle.
//
//   e2m1_to_bf16_bits / e8m0_to_f32: the fp4_e8m0_b32 key-row decoding (OCP MX E2M1 codes, E8M0
//   scales), every product exact in bf16 (FreeToken PR 634, "Correctness and tests");
//   e2m1x2_to_bf16x2_bits: the same for a pair of codes, on the device.
//   topk_order_key: the 64-bit key whose order is the top-k output order.
#pragma once

#include <cstdint>
#include <cstring>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>

namespace spa {

__host__ __device__ __forceinline__ float f32_from_bits(uint32_t u) {
#ifdef __CUDA_ARCH__
  return __uint_as_float(u);
#else
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
#endif
}

__host__ __device__ __forceinline__ uint32_t f32_bits(float f) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(f);
#else
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return u;
#endif
}

// e2m1 code (4 bits) times a scale -> bf16 bits.  The magnitude is built from the code's fields
// ((1 + m/2) 2^(e-1), or m/2 for e = 0), the product with a power of two is exact in fp32 (down to
// fp32 subnormals; past the fp32 range it is inf), and the bf16 conversion of an exact value with
// two significant bits is exact.  Bit 3 is the sign.
__host__ __device__ __forceinline__ uint32_t e2m1_to_bf16_bits(uint32_t c, float scale) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const uint32_t mag = e ? (((e + 126u) << 23) | (m << 22)) : (m ? 0x3F000000u : 0u);
  const float v = f32_from_bits(mag) * scale;
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v)) | ((c & 8u) << 12);
}

#ifdef __CUDACC__
// Two e2m1 codes (the byte's low nibble first) times a scale -> bf16x2 bits, the first code's
// value in the low half: the same bits as e2m1_to_bf16_bits for each code (the code's value is
// exact in f16 and in fp32, its product with the scale is the same fp32 product, rounded to bf16
// the same way; the sign is the code's, carried through the product), for every scale but the NaN
// one, where both give a NaN and only its sign bit may differ.  The pair conversion is one
// instruction where e2m1_to_bf16_bits builds each magnitude, and the kernel's unrolled decoding
// loop stays small (it is instruction-cache bound: keeping the per-code path beside this one, for
// NaN scales, cost a fifth of the full-prefill speed).
__device__ __forceinline__ uint32_t e2m1x2_to_bf16x2_bits(uint32_t byte, float scale) {
  const __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)byte, __NV_E2M1);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
  return *reinterpret_cast<const uint32_t*>(&b);
}
#endif

// ue8m0 scale byte -> fp32: 2^(s - 127); 0 is the fp32 subnormal 2^-127; 0xFF is NaN.
__host__ __device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  if (s == 0u) return f32_from_bits(0x00400000u);
  if (s == 255u) return f32_from_bits(0x7FC00000u);
  return f32_from_bits(s << 23);
}

// Top-k order bits of a logit: the top 32 bits of its order key, the logit's order-preserving
// bits (-0 folded into +0), or 0 when the logit is not scored (-inf; +inf and NaN are not scored
// either).  A scored logit's bits are never 0: the most negative finite logit gives 0x00800000.
__host__ __device__ __forceinline__ uint32_t topk_order_bits(float x) {
  if (!(x > -INFINITY && x < INFINITY)) return 0u;  // also 0 for NaN
  if (x == 0.f) x = 0.f;
  const uint32_t u = f32_bits(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k order key of a scored logit: its order bits above the complement of the entry index, so
// that a larger key is a larger logit, or the same logit and a smaller index.
__host__ __device__ __forceinline__ unsigned long long topk_key(uint32_t order_bits, uint32_t id) {
  return ((unsigned long long)order_bits << 32) | (unsigned long long)(0xFFFFFFFFu - id);
}

__host__ __device__ __forceinline__ bool topk_order_key(float x, uint32_t id,
                                                        unsigned long long& key) {
  const uint32_t ord = topk_order_bits(x);
  if (ord == 0u) return false;
  key = topk_key(ord, id);
  return true;
}

}  // namespace spa

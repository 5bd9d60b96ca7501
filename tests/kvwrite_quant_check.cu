// Exhaustive check of the paged KV write's e4m3 codes (spa_kvwrite_quant.cuh) against the IEEE
// binary32 division.  A row's elements are bf16 values x with |x| <= m, m = max|x| of the row, and
// scale = m / 448: for every positive finite bf16 m and every bf16 x with |x| <= m, both signs,
// the code the write takes equals the e4m3 code (nearest even, saturating) of x / scale.
// Prints: pairs checked, pairs whose code differs, pairs on the reciprocal path, pairs whose
// quotient differs from the IEEE one (informative: only the codes must agree).
#include <cstdio>

#include "spa_kvwrite_quant.cuh"

using namespace spa;

__device__ unsigned long long g_pairs, g_bad, g_fast, g_qdiff;

__global__ void check_all() {
  const uint32_t mb = blockIdx.x + 1;  // bf16 bits of the row maximum, 0x0001 .. 0x7F7F
  const float m = kvq_bf16_to_f32(mb);
  const float scale = __fdiv_rn(m, 448.f);
  const float r = __frcp_rn(scale);
  const bool fast = kvq_fast_scale(scale);
  unsigned long long pairs = 0, bad = 0, qdiff = 0;
  for (uint32_t xb = threadIdx.x; xb <= mb; xb += blockDim.x) {
    const float x = kvq_bf16_to_f32(xb);
    // one chunk: x, -x in the first pair, the rest zeros of both signs
    const uint4 u = make_uint4(xb | ((xb | 0x8000u) << 16), 0x80000000u, 0u, 0x8000u);
    const uint2 got = kvq_chunk(u, scale, r, fast);
    const uint32_t want0 = kvq_e4m3x2(__fdiv_rn(x, scale), __fdiv_rn(-x, scale));
    const uint32_t want1 = kvq_e4m3x2(__fdiv_rn(0.f, scale), __fdiv_rn(-0.f, scale));
    const uint32_t want2 = kvq_e4m3x2(__fdiv_rn(0.f, scale), __fdiv_rn(0.f, scale));
    const uint32_t want3 = kvq_e4m3x2(__fdiv_rn(-0.f, scale), __fdiv_rn(0.f, scale));
    const uint2 want = make_uint2(want0 | (want1 << 16), want2 | (want3 << 16));
    pairs += 2;
    for (int b = 0; b < 2; ++b) bad += ((got.x ^ want.x) >> (8 * b)) & 0xFFu ? 1 : 0;
    bad += (got.x >> 16) != (want.x >> 16) || got.y != want.y;   // the zeros
    if (fast) {
      qdiff += __float_as_uint(kvq_div(x, scale, r)) != __float_as_uint(__fdiv_rn(x, scale));
      qdiff += __float_as_uint(kvq_div(-x, scale, r)) != __float_as_uint(__fdiv_rn(-x, scale));
    }
  }
  atomicAdd(&g_pairs, pairs);
  atomicAdd(&g_bad, bad);
  if (fast) atomicAdd(&g_fast, pairs);
  atomicAdd(&g_qdiff, qdiff);
}

int main() {
  check_all<<<0x7F7F, 256>>>();
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  unsigned long long pairs = 0, bad = 0, fast = 0, qdiff = 0;
  cudaMemcpyFromSymbol(&pairs, g_pairs, sizeof pairs);
  cudaMemcpyFromSymbol(&bad, g_bad, sizeof bad);
  cudaMemcpyFromSymbol(&fast, g_fast, sizeof fast);
  cudaMemcpyFromSymbol(&qdiff, g_qdiff, sizeof qdiff);
  printf("%llu %llu %llu %llu\n", pairs, bad, fast, qdiff);
  return 0;
}

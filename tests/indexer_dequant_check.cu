// Exhaustive check of the indexer's paired key decoding (spa_indexer_math.cuh): for every byte of
// two e2m1 codes and every ue8m0 scale byte but the NaN one, e2m1x2_to_bf16x2_bits gives the bits
// of e2m1_to_bf16_bits for the low-nibble code in the low half and for the high-nibble code in
// the high half.  Prints: pairs checked, pairs that differ.
#include <cstdio>

#include "spa_indexer_math.cuh"

using namespace spa;

__device__ unsigned int g_pairs, g_bad;

__global__ void check_all() {
  const uint32_t byte = threadIdx.x;   // 0 .. 255
  const uint32_t s = blockIdx.x;       // 0 .. 254
  const float sc = e8m0_to_f32(s);
  const uint32_t want = e2m1_to_bf16_bits(byte & 0xFu, sc) | (e2m1_to_bf16_bits(byte >> 4, sc) << 16);
  const uint32_t got = e2m1x2_to_bf16x2_bits(byte, sc);
  atomicAdd(&g_pairs, 1u);
  if (got != want) atomicAdd(&g_bad, 1u);
}

int main() {
  check_all<<<255, 256>>>();
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  unsigned int pairs = 0, bad = 0;
  cudaMemcpyFromSymbol(&pairs, g_pairs, sizeof pairs);
  cudaMemcpyFromSymbol(&bad, g_bad, sizeof bad);
  printf("%u %u\n", pairs, bad);
  return 0;
}

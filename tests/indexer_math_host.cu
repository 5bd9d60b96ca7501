// Host program for tests/test_indexer_math_host.py: runs the indexer kernels' element arithmetic
// (spa_indexer_math.cuh, the code the kernels call) on the CPU.
//   indexer_math_host decode          -> 16 x 256 lines "code scale bf16bits" (hex)
//   indexer_math_host keys < pairs    -> for each stdin line "f32bits id" (hex, decimal): the
//                                        top-k order key in hex, or "-" when not scored
#include <cstdio>
#include <cstring>

#include "spa_indexer_math.cuh"

int main(int argc, char** argv) {
  if (argc > 1 && std::strcmp(argv[1], "decode") == 0) {
    for (unsigned c = 0; c < 16; ++c)
      for (unsigned s = 0; s < 256; ++s)
        std::printf("%x %x %04x\n", c, s, spa::e2m1_to_bf16_bits(c, spa::e8m0_to_f32(s)));
    return 0;
  }
  if (argc > 1 && std::strcmp(argv[1], "keys") == 0) {
    unsigned bits, id;
    while (std::scanf("%x %u", &bits, &id) == 2) {
      unsigned long long key;
      if (spa::topk_order_key(spa::f32_from_bits(bits), id, key))
        std::printf("%016llx\n", key);
      else
        std::printf("-\n");
    }
    return 0;
  }
  return 2;
}

// Host program for tests/test_plan_host.py: the chunk schedule of the prefill from host buffers
// (spa_plan.h, the code the library calls) on the CPU.
//   host_chunks < cases   -> for each stdin line "T tc": the chunk sizes, in order
#include <cstdio>

#include "spa_plan.h"

int main() {
  long long T, tc;
  while (std::scanf("%lld %lld", &T, &tc) == 2) {
    for (long long c0 = 0, n = 0; c0 < T; c0 += n) {
      n = spa::host_chunk_tokens(T, tc, c0);
      if (n < 1) {   // would never end
        std::printf("bad\n");
        return 1;
      }
      std::printf("%lld ", n);
    }
    std::printf("\n");
  }
  return 0;
}

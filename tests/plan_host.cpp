// Host program for tests/test_plan_host.py: runs the split arithmetic of the decode path whose
// partials live in global memory (spa_plan.h, the code the library calls) on the CPU.
//   plan_host < cases   -> for each stdin line "C T H D sms max_splits cap": "splits cols bytes"
#include <cstdio>

#include "spa_plan.h"

int main() {
  int C, H, D, sms, max_splits;
  long long T;
  unsigned long long cap;
  while (std::scanf("%d %lld %d %d %d %d %llu", &C, &T, &H, &D, &sms, &max_splits, &cap) == 7) {
    int splits = 0, cols = 0;
    spa::plan_partials(C, T, H, D, sms, max_splits, (size_t)cap, &splits, &cols);
    std::printf("%d %d %zu\n", splits, cols, spa::partials_bytes(T, H, D, splits));
  }
  return 0;
}

// spa_plan.h - host-side split arithmetic of the decode path that keeps its split-K partials in
// global memory (a caller workspace, or the library's built-in scratch array), the bytes those
// partials take, and the chunk schedule of the prefill from host buffers.  Plain C++ with no CUDA
// dependency, so that it can be compiled and checked on a machine without a GPU.
#pragma once

#include <cstddef>
#include <cstdint>

namespace spa {

inline size_t plan_align256(size_t x) { return (x + 255) & ~size_t(255); }

// Partials of `splits` splits per query: fp32 O [T][S][H][D], then base-2 log-sum-exps [T][S][H],
// each block 256-byte aligned.
inline size_t partials_bytes(long long T, int H, int D, int splits) {
  const size_t tsh = (size_t)T * (size_t)splits * (size_t)H;
  return plan_align256(tsh * (size_t)D * sizeof(float)) + plan_align256(tsh * sizeof(float));
}

// Split plan of the partials path for T queries of C columns, H heads of head_dim D on `sms` SMs:
// enough splits that every SM gets about one (query, 64-head group, split) item, at least 32
// columns per split (a multiple of 32), at most `max_splits` splits (what the merge kernel reads
// per head), and partials of at most `cap_bytes` (fewer, longer splits until they fit; one split
// is always allowed, and the caller rejects it if even that does not fit).
inline void plan_partials(int C, long long T, int H, int D, int sms, int max_splits,
                          size_t cap_bytes, int* splits, int* cols) {
  if (C < 1) C = 1;
  const long long groups = (H + 63) / 64;
  const long long base = T * groups;
  long long want = base > 0 ? sms / base : 1;
  if (want < 1) want = 1;
  int c = (int)((C + want - 1) / want);
  c = ((c + 31) / 32) * 32;
  if (c > C) c = C;
  int n = (C + c - 1) / c;
  if (n > max_splits) {
    c = (C + max_splits - 1) / max_splits;
    n = (C + c - 1) / c;
  }
  // fewer splits while the partials do not fit (n strictly decreases: c >= C / w gives n <= w)
  while (n > 1 && partials_bytes(T, H, D, n) > cap_bytes) {
    const int w = n - 1;
    c = (C + w - 1) / w;
    c = ((c + 31) / 32) * 32;
    if (c > C) c = C;
    n = (C + c - 1) / c;
  }
  *cols = c;
  *splits = n;
}

// Chunk schedule of the prefill from host buffers: the tokens of the chunk that starts at token c0
// of T, with chunks of at most tc tokens (1 <= tc <= T).  A quarter chunk first and last, so that
// the copy pipeline fills and drains sooner, full chunks between; a tail shorter than two quarters
// is one chunk.  Every size is in [1, tc] and the chunks cover [0, T) in order.
inline long long host_chunk_tokens(long long T, long long tc, long long c0) {
  const long long quarter = tc / 4 > 0 ? tc / 4 : 1;
  const long long rest = T - c0;
  if (c0 == 0) return quarter < rest ? quarter : rest;
  if (rest > tc + quarter) return tc;
  return rest >= 2 * quarter ? rest - quarter : rest;   // (both at most tc)
}

}  // namespace spa

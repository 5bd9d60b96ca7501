// spa_topk.cu - the top-k selection after the indexer logits: for each query, the k scored entries
// (finite logit) with the largest logits, in decreasing order of logit, ties going to the smaller
// entry index, -1 filling the list when fewer than k were scored.  The result is the attention's
// top-k list.
//
// One CTA per query.  Every scored entry gets a 64-bit key, the logit's order-preserving 32 bits
// above the complement of its entry index, so that keys are distinct (up to repeated candidates,
// which are the same entry) and "larger key" is exactly the output order.  An MSB-first radix
// select (8 bits a pass, 256-bin shared histograms) finds the k-th largest key, stopping as soon
// as the bucket it lands in holds exactly the entries still needed; one more pass collects the
// keys above that bucket and the needed ones inside it, and a bitonic sort in shared memory puts
// the k keys in order.  Each pass re-reads the logits row (from L2 for the sizes the indexer
// writes); no pass waits on anything but __syncthreads.
#include "spa_indexer.h"
#include "spa_indexer_math.cuh"

namespace spa {

namespace {

constexpr int kThreads = 512;

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a) {
  __shared__ unsigned int s_hist[256];
  __shared__ unsigned long long s_keys[kIdxTopkMax];
  __shared__ unsigned int s_count, s_eq_taken, s_sel, s_need, s_done;
  const int tid = threadIdx.x;
  const long long t = blockIdx.x;
  const float* row = a.logits + t * a.ncols;
  const int32_t* ids = a.cand ? a.cand + t * a.ncols : nullptr;
  const auto entry_of = [&](int c) -> uint32_t { return ids ? (uint32_t)__ldg(ids + c) : (uint32_t)c; };

  // how many entries are scored
  if (tid == 0) s_count = 0;
  __syncthreads();
  unsigned int mine = 0;
  for (int c = tid; c < a.ncols; c += kThreads) {
    unsigned long long key;
    mine += topk_order_key(__ldg(row + c), entry_of(c), key) ? 1u : 0u;
  }
  atomicAdd(&s_count, mine);
  __syncthreads();
  const unsigned int scored = s_count;
  const unsigned int take = scored < (unsigned int)a.k ? scored : (unsigned int)a.k;

  // radix select of the take-th largest key: after the loop, keys whose top (64 - shift) bits
  // exceed `prefix` are all selected, and `need` of those equal to it
  unsigned long long prefix = 0ull;
  int shift = 64;
  unsigned int need = take;
  if (take < scored) {
    for (int pass = 0; pass < 8; ++pass) {
      const int sh = 56 - 8 * pass;
      for (int i = tid; i < 256; i += kThreads) s_hist[i] = 0u;
      __syncthreads();
      for (int c = tid; c < a.ncols; c += kThreads) {
        unsigned long long key;
        if (!topk_order_key(__ldg(row + c), entry_of(c), key)) continue;
        if (shift < 64 && (key >> shift) != (prefix >> shift)) continue;
        atomicAdd(&s_hist[(key >> sh) & 0xFFu], 1u);
      }
      __syncthreads();
      if (tid < 32) {  // warp 0: lane l sums bins 255-8l .. 248-8l, scans from the top
        unsigned int part = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) part += s_hist[255 - 8 * tid - b];
        unsigned int incl = part;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += v;
        }
        const unsigned int excl = incl - part;
        if (excl < need && incl >= need) {  // exactly one lane: the bucket is among its 8 bins
          unsigned int cum = excl;
          for (int b = 0; b < 8; ++b) {
            const int bin = 255 - 8 * tid - b;
            const unsigned int h = s_hist[bin];
            if (cum + h >= need) {
              s_sel = (unsigned int)bin;
              s_need = need - cum;
              s_done = (h == need - cum) ? 1u : 0u;
              break;
            }
            cum += h;
          }
        }
      }
      __syncthreads();
      prefix |= (unsigned long long)s_sel << sh;
      need = s_need;
      shift = sh;
      const bool done = s_done != 0u;
      __syncthreads();  // s_sel / s_need / s_done are rewritten by the next pass
      if (done) break;
    }
  }

  // collect the selected keys (every thread has read s_count: the radix passes may not have run)
  __syncthreads();
  if (tid == 0) {
    s_count = 0;
    s_eq_taken = 0;
  }
  __syncthreads();
  for (int c = tid; c < a.ncols; c += kThreads) {
    unsigned long long key;
    if (!topk_order_key(__ldg(row + c), entry_of(c), key)) continue;
    bool keep = true;
    if (shift < 64) {
      const unsigned long long kt = key >> shift, pt = prefix >> shift;
      if (kt < pt) keep = false;
      else if (kt == pt) keep = atomicAdd(&s_eq_taken, 1u) < need;
    }
    if (keep) {
      const unsigned int slot = atomicAdd(&s_count, 1u);
      if (slot < (unsigned int)kIdxTopkMax) s_keys[slot] = key;
    }
  }
  __syncthreads();

  // bitonic sort (descending) of the take keys, padded with zeros to a power of two
  int n = 1;
  while (n < (int)take) n <<= 1;
  for (int i = (int)take + tid; i < n; i += kThreads) s_keys[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < n; i += kThreads) {
        const int partner = i ^ stride;
        if (partner > i) {
          const bool desc = (i & size) == 0;
          const unsigned long long x = s_keys[i], y = s_keys[partner];
          if (desc ? (x < y) : (x > y)) {
            s_keys[i] = y;
            s_keys[partner] = x;
          }
        }
      }
      __syncthreads();
    }
  }

  int32_t* out = a.topk + t * a.k;
  for (int i = tid; i < a.k; i += kThreads)
    out[i] = i < (int)take ? (int32_t)(0xFFFFFFFFu - (uint32_t)(s_keys[i] & 0xFFFFFFFFull)) : -1;
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.T == 0 || a.k == 0) return cudaSuccess;
  topk_kernel<<<(unsigned)a.T, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace spa

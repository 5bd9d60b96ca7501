// spa_topk.cu - the top-k selection after the indexer logits: for each query, the k scored entries
// (finite logit) with the largest logits, in decreasing order of logit, ties going to the smaller
// entry index, -1 filling the list when fewer than k were scored.  The result is the attention's
// top-k list.
//
// One CTA per query.  Every scored entry gets a 64-bit key, the logit's order-preserving 32 bits
// above the complement of its entry index, so that keys are distinct (up to repeated candidates,
// which are the same entry) and "larger key" is exactly the output order.  The row is read twice:
//   1. count the scored entries and histogram the keys' top 12 bits (4096 bins in shared memory);
//      a scan of the bins from the top finds the bucket B holding the take-th largest key;
//   2. keys above B are selected outright, keys in B are copied to a shared-memory buffer.
// An MSB-first radix select (8 bits a pass, 256 bins) over the bucket's keys then finds the
// threshold, stopping as soon as the bucket it lands in holds exactly the keys still needed; the
// keys above it and the needed ones equal to it are selected.  When B holds more keys than the
// buffer (many equal logits), the select reads them from the row instead, filtered to B.  A
// bitonic sort in shared memory puts the k keys in order.  No pass waits on anything but
// __syncthreads.
#include "spa_indexer.h"
#include "spa_indexer_math.cuh"

namespace spa {

namespace {

constexpr int kBins = 4096;        // first-pass histogram: the keys' top 12 bits
constexpr int kBinShift = 52;      // of the 64-bit key
constexpr int kBinShift32 = 20;    // of its top 32 bits (the order bits)
constexpr int kCandMax = 4096;     // keys of bucket B kept in shared memory
// dynamic shared memory: histogram, selected keys, bucket keys
constexpr int kSmemBytes = kBins * 4 + kIdxTopkMax * 8 + kCandMax * 8;

// kThreads threads, each loading kUnroll columns before it looks at any of them: 1024 x 16 when
// there are fewer rows than SMs (a row's two passes are then one SM's latency-bound loop), 512 x 8
// otherwise (more CTAs per SM).
template <int kThreads, int kUnroll>
__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a) {
  constexpr int kBinsPerThread = kBins / kThreads;   // bins a thread sums in the bucket scan
  static_assert(kBins % kThreads == 0 && kBinsPerThread <= 32, "bucket scan");
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned int* s_hist = reinterpret_cast<unsigned int*>(smem);
  unsigned long long* s_keys = reinterpret_cast<unsigned long long*>(smem + kBins * 4);
  unsigned long long* s_cand = s_keys + kIdxTopkMax;
  __shared__ unsigned int s_count, s_ncand, s_eq_taken, s_sel, s_need, s_done;
  __shared__ unsigned int s_scan[kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long t = blockIdx.x;
  const float* row = a.logits + t * a.ncols;
  const int32_t* ids = a.cand ? a.cand + t * a.ncols : nullptr;
  const auto entry_of = [&](int c) -> uint32_t { return ids ? (uint32_t)__ldg(ids + c) : (uint32_t)c; };
  // A chunk of kThreads * kUnroll columns from c0: the order bits (topk_order_bits: 0 = not scored
  // or past the row) of a thread's kUnroll columns, all loads issued before any is looked at.  Rows
  // that start 16-byte aligned with a multiple of 4 columns are read as float4 (thread t takes
  // columns 4t .. 4t+3 of each kThreads * 4 block), the others one float a thread per kThreads.
  // The passes need only these bits; the 64-bit key, and a candidate's entry id, are formed for the
  // few columns that are kept.
  const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15u) == 0u) && (a.ncols & 3) == 0;
  const auto col_of = [&](int c0, int u) -> int {
    return vec ? c0 + 4 * ((u >> 2) * kThreads + tid) + (u & 3) : c0 + u * kThreads + tid;
  };
  const auto row_ords = [&](int c0, uint32_t (&o)[kUnroll]) {
    if (vec) {
      float4 f[kUnroll / 4];
#pragma unroll
      for (int v = 0; v < kUnroll / 4; ++v) {
        const int c = c0 + 4 * (v * kThreads + tid);   // the row's length is a multiple of 4
        f[v] = c < a.ncols ? __ldg(reinterpret_cast<const float4*>(row + c))
                           : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int v = 0; v < kUnroll / 4; ++v) {
        o[4 * v + 0] = topk_order_bits(f[v].x);
        o[4 * v + 1] = topk_order_bits(f[v].y);
        o[4 * v + 2] = topk_order_bits(f[v].z);
        o[4 * v + 3] = topk_order_bits(f[v].w);
      }
    } else {
      float x[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * kThreads + tid;
        x[u] = c < a.ncols ? __ldg(row + c) : -INFINITY;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) o[u] = topk_order_bits(x[u]);
    }
  };

  // ---- pass 1: scored count, histogram of the top 12 bits ----
  for (int i = tid; i < kBins; i += kThreads) s_hist[i] = 0u;
  if (tid == 0) s_count = 0;
  __syncthreads();
  unsigned int mine = 0;
  for (int c0 = 0; c0 < a.ncols; c0 += kThreads * kUnroll) {
    uint32_t o[kUnroll];
    row_ords(c0, o);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (o[u] == 0u) continue;
      ++mine;
      atomicAdd(&s_hist[o[u] >> kBinShift32], 1u);
    }
  }
  atomicAdd(&s_count, mine);
  __syncthreads();
  const unsigned int scored = s_count;
  const unsigned int take = scored < (unsigned int)a.k ? scored : (unsigned int)a.k;
  const bool all = take == scored;   // every scored key is selected

  // ---- bucket B of the take-th largest key: thread i holds kBinsPerThread bins, from the top ----
  if (!all) {
    unsigned int part = 0;
#pragma unroll
    for (int b = 0; b < kBinsPerThread; ++b) part += s_hist[kBins - 1 - kBinsPerThread * tid - b];
    unsigned int incl = part;   // inclusive scan in thread order (= descending bins)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_scan[warp] = incl;
    __syncthreads();
    unsigned int before = 0;
    for (int w = 0; w < warp; ++w) before += s_scan[w];
    incl += before;
    const unsigned int excl = incl - part;
    if (excl < take && incl >= take) {   // exactly one thread: B is among its bins
      unsigned int cum = excl;
      for (int b = 0; b < kBinsPerThread; ++b) {
        const int bin = kBins - 1 - kBinsPerThread * tid - b;
        const unsigned int h = s_hist[bin];
        if (cum + h >= take) {
          s_sel = (unsigned int)bin;
          s_need = take - cum;
          break;
        }
        cum += h;
      }
    }
  }
  if (tid == 0) {
    s_count = 0;
    s_ncand = 0;
    s_eq_taken = 0;
  }
  __syncthreads();
  const uint32_t bucket = all ? 0u : s_sel;
  unsigned int need = all ? 0u : s_need;

  // ---- pass 2: keys above B are selected, keys in B go to the bucket buffer ----
  for (int c0 = 0; c0 < a.ncols; c0 += kThreads * kUnroll) {
    uint32_t o[kUnroll];
    row_ords(c0, o);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (o[u] == 0u) continue;
      const uint32_t top = o[u] >> kBinShift32;
      if (all || top > bucket) {
        s_keys[atomicAdd(&s_count, 1u)] = topk_key(o[u], entry_of(col_of(c0, u)));  // < take
      } else if (top == bucket) {
        const unsigned int slot = atomicAdd(&s_ncand, 1u);
        if (slot < (unsigned int)kCandMax) s_cand[slot] = topk_key(o[u], entry_of(col_of(c0, u)));
      }
    }
  }
  __syncthreads();

  if (!all) {
    // the keys of bucket B: from the buffer, or from the row when they did not all fit
    const unsigned int ncand = s_ncand;
    const bool in_smem = ncand <= (unsigned int)kCandMax;
    // f(key) for every key of bucket B
    const auto for_bucket = [&](auto f) {
      if (in_smem) {
        for (int i = tid; i < (int)ncand; i += kThreads) f(s_cand[i]);
        return;
      }
      for (int c0 = 0; c0 < a.ncols; c0 += kThreads * kUnroll) {
        uint32_t o[kUnroll];
        row_ords(c0, o);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (o[u] != 0u && (o[u] >> kBinShift32) == bucket) f(topk_key(o[u], entry_of(col_of(c0, u))));
      }
    };
    // radix select below the top 12 bits: keys whose top (64 - shift) bits exceed `prefix` are
    // all selected, and `need` of those equal to it
    unsigned long long prefix = (unsigned long long)bucket << kBinShift;
    int shift = kBinShift;
    while (shift > 0) {
      const int sh = shift > 8 ? shift - 8 : 0;
      const unsigned int width_mask = (1u << (shift - sh)) - 1u;
      for (int i = tid; i < 256; i += kThreads) s_hist[i] = 0u;
      __syncthreads();
      for_bucket([&](unsigned long long key) {
        if ((key >> shift) == (prefix >> shift)) atomicAdd(&s_hist[(key >> sh) & width_mask], 1u);
      });
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
    // collect: bucket keys above the threshold, and `need` of those equal to it
    for_bucket([&](unsigned long long key) {
      const unsigned long long kt = key >> shift, pt = prefix >> shift;
      bool keep = kt > pt;
      if (kt == pt) keep = atomicAdd(&s_eq_taken, 1u) < need;
      if (keep) {
        const unsigned int slot = atomicAdd(&s_count, 1u);
        if (slot < (unsigned int)kIdxTopkMax) s_keys[slot] = key;
      }
    });
    __syncthreads();
  }

  // bitonic sort (descending) of the take keys, padded with zeros to a power of two.  Stages of
  // stride 32 and more exchange through shared memory, one barrier each; for every size the stages
  // of stride below 32 pair elements of one warp (n is a multiple of the warp's 32 elements, or
  // one warp holds it all) and run together in registers, with shuffles, behind one barrier.
  int n = 1;
  while (n < (int)take) n <<= 1;
  for (int i = (int)take + tid; i < n; i += kThreads) s_keys[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= n; size <<= 1) {
    int stride = size >> 1;
    for (; stride >= 32; stride >>= 1) {
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
    for (int i0 = warp * 32; i0 < n; i0 += kThreads) {   // warp-uniform bounds
      const int i = i0 + lane;
      unsigned long long x = i < n ? s_keys[i] : 0ull;
      const bool desc = (i & size) == 0;
      for (int st = stride; st > 0; st >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, st);
        const bool lower = (lane & st) == 0;         // element i is the pair's first
        x = (lower == desc) ? (x > y ? x : y) : (x < y ? x : y);
      }
      if (i < n) s_keys[i] = x;
    }
    __syncthreads();
  }

  int32_t* out = a.topk + t * a.k;
  for (int i = tid; i < a.k; i += kThreads)
    out[i] = i < (int)take ? (int32_t)(0xFFFFFFFFu - (uint32_t)(s_keys[i] & 0xFFFFFFFFull)) : -1;
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.T == 0 || a.k == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const bool few = a.T < sms;
  const auto kern = few ? topk_kernel<1024, 16> : topk_kernel<512, 8>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)a.T, few ? 1024 : 512, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace spa

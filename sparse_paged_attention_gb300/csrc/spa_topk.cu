// spa_topk.cu - the top-k selection after the indexer logits: for each query, the k scored entries
// (finite logit) with the largest logits, in decreasing order of logit, ties going to the smaller
// entry index, -1 filling the list when fewer than k were scored.  The result is the attention's
// top-k list.
//
// One CTA (or one cluster of CTAs) per query.  Every scored entry gets a 64-bit key, the logit's
// order-preserving 32 bits above the complement of its entry index, so that keys are distinct (up
// to repeated candidates, which are the same entry) and "larger key" is exactly the output order.
// The row is read twice:
//   1. count the scored entries and histogram the keys' top 12 bits (4096 bins in shared memory);
//      a scan of the bins from the top finds the bucket B holding the take-th largest key;
//   2. keys above B are selected outright, keys in B are copied to a shared-memory buffer.
// An MSB-first radix select (8 bits a pass, 256 bins) over the bucket's keys then finds the
// threshold, stopping as soon as the bucket it lands in holds exactly the keys still needed; the
// keys above it and the needed ones equal to it are selected.  When B holds more keys than the
// buffer (many equal logits), the select reads them from the row instead, filtered to B.  A
// bitonic sort in shared memory puts the k keys in order (a cluster of CTAs that shares a row
// ranks them instead, below).  No pass waits on anything but __syncthreads and, in a cluster,
// cluster barriers that every thread passes.
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

// Distributed shared memory between the CTAs of a cluster (one row per cluster).
__device__ __forceinline__ unsigned int ld_cluster_u32(uint32_t addr) {
  unsigned int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_cluster_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned int atom_add_cluster(uint32_t addr, unsigned int v) {
  unsigned int old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v)
               : "memory");
  return old;
}
// Every thread of every CTA of the cluster; shared-memory writes before it are seen after it.
__device__ __forceinline__ void cluster_sync_all() {
  cluster_arrive();
  cluster_wait();
}

// kThreads threads, each loading kUnroll columns before it looks at any of them: 1024 x 16 when
// there are fewer rows than SMs (a row's two passes are then one SM's latency-bound loop), 512 x 8
// otherwise (more CTAs per SM).  kCluster > 1: a cluster of kCluster CTAs per row (for a few rows),
// each taking one chunk of the row through both passes:
//   - after pass 1 (cluster barrier 1) CTA r sums bins [r, r + 1) * kBins / kCluster of every
//     CTA's histogram, and the row's scored count;
//   - after cluster barrier 2 every CTA copies the summed histogram and finds the same bucket B;
//   - pass 2 appends each CTA's kept keys and bucket keys to CTA 0's buffers (remote atomics);
//   - after cluster barrier 3 CTA 0 selects as a single CTA would;
//   - after cluster barrier 4 every CTA copies the selected keys and writes the output positions
//     of its share of them (a key's rank: the number of keys above it), in place of a sort;
//   - a last split barrier keeps CTA 0 resident until every copy from it is done.
// Every thread of every CTA passes every barrier, whatever the row holds.
// (three 512-thread CTAs an SM for many rows, whose 64 KB of shared memory allows three; two for
// a cluster's CTAs, so that the clusters of up to 19 rows are all resident together)
template <int kThreads, int kUnroll, int kCluster>
__global__ void __launch_bounds__(kThreads, kCluster > 1 ? 2 : (kThreads == 512 ? 3 : 1))
    topk_kernel(const TopkArgs a) {
  constexpr int kBinsPerThread = kBins / kThreads;   // bins a thread sums in the bucket scan
  static_assert(kBins % kThreads == 0 && kBinsPerThread <= 32, "bucket scan");
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned int* s_hist = reinterpret_cast<unsigned int*>(smem);
  unsigned long long* s_keys = reinterpret_cast<unsigned long long*>(smem + kBins * 4);
  unsigned long long* s_cand = s_keys + kIdxTopkMax;
  __shared__ unsigned int s_count, s_kcnt, s_ncand, s_eq_taken, s_sel, s_need, s_done, s_total;
  __shared__ unsigned int s_scan[kThreads / 32];
  __shared__ unsigned int s_red[kCluster > 1 ? kBins / kCluster : 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long t = blockIdx.x / kCluster;
  const int rank = kCluster > 1 ? (int)cluster_ctarank() : 0;
  // this CTA's columns: the whole row, or its chunk (a multiple of 4 columns: float4 alignment)
  const int chunk = kCluster > 1 ? (((a.ncols + kCluster - 1) / kCluster + 3) & ~3) : a.ncols;
  const int cbeg = min(a.ncols, rank * chunk), cend = min(a.ncols, cbeg + chunk);
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
  const auto row_ords = [&](int c0, uint32_t (&o)[kUnroll], int cend_) {
    if (vec) {
      float4 f[kUnroll / 4];
#pragma unroll
      for (int v = 0; v < kUnroll / 4; ++v) {
        const int c = c0 + 4 * (v * kThreads + tid);   // the row's length is a multiple of 4
        f[v] = c < cend_ ? __ldg(reinterpret_cast<const float4*>(row + c))
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
        x[u] = c < cend_ ? __ldg(row + c) : -INFINITY;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) o[u] = topk_order_bits(x[u]);
    }
  };

  pdl_launch_dependents();
  // ---- pass 1: scored count, histogram of the top 12 bits ----
  for (int i = tid; i < kBins; i += kThreads) s_hist[i] = 0u;
  if (tid == 0) {
    s_count = 0;
    s_kcnt = 0;
    s_ncand = 0;
    s_eq_taken = 0;
  }
  __syncthreads();
  pdl_wait();   // nothing global before the grid before this one is done
  unsigned int mine = 0;
  for (int c0 = cbeg; c0 < cend; c0 += kThreads * kUnroll) {
    uint32_t o[kUnroll];
    row_ords(c0, o, cend);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (o[u] == 0u) continue;
      ++mine;
      atomicAdd(&s_hist[o[u] >> kBinShift32], 1u);
    }
  }
  atomicAdd(&s_count, mine);
  __syncthreads();
  if constexpr (kCluster > 1) {
    constexpr int kSlice = kBins / kCluster;
    cluster_sync_all();   // 1: every CTA's histogram and count are complete
    for (int i = tid; i < kSlice; i += kThreads) {
      const uint32_t bin = smem_u32(&s_hist[rank * kSlice + i]);
      unsigned int v[kCluster];   // all loads in flight before the sum
#pragma unroll
      for (int k = 0; k < kCluster; ++k) v[k] = ld_cluster_u32(mapa_cluster(bin, (uint32_t)k));
      unsigned int sum = 0;
#pragma unroll
      for (int k = 0; k < kCluster; ++k) sum += v[k];
      s_red[i] = sum;
    }
    if (tid == 0) {
      unsigned int v[kCluster];
#pragma unroll
      for (int k = 0; k < kCluster; ++k)
        v[k] = ld_cluster_u32(mapa_cluster(smem_u32(&s_count), (uint32_t)k));
      unsigned int tot = 0;
#pragma unroll
      for (int k = 0; k < kCluster; ++k) tot += v[k];
      s_total = tot;
    }
    cluster_sync_all();   // 2: every slice is summed; no CTA reads another's histogram any more
    {
      constexpr int kPer = kBins / kThreads;
      unsigned int v[kPer];   // all loads in flight before the stores
#pragma unroll
      for (int m = 0; m < kPer; ++m) {
        const int i = tid + m * kThreads;
        v[m] = ld_cluster_u32(mapa_cluster(smem_u32(&s_red[i % kSlice]), (uint32_t)(i / kSlice)));
      }
#pragma unroll
      for (int m = 0; m < kPer; ++m) s_hist[tid + m * kThreads] = v[m];
    }
    __syncthreads();
  }
  const unsigned int scored = kCluster > 1 ? s_total : s_count;
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
  __syncthreads();
  const uint32_t bucket = all ? 0u : s_sel;
  unsigned int need = all ? 0u : s_need;

  // ---- pass 2: keys above B are selected, keys in B go to the bucket buffer ----
  // (a cluster: to CTA 0's buffers)
  const auto keep_key = [&](unsigned long long key) {   // fewer than take of them
    if constexpr (kCluster > 1) {
      const unsigned int slot = atom_add_cluster(mapa_cluster(smem_u32(&s_kcnt), 0u), 1u);
      st_cluster_u64(mapa_cluster(smem_u32(&s_keys[slot]), 0u), key);
    } else {
      s_keys[atomicAdd(&s_kcnt, 1u)] = key;
    }
  };
  const auto bucket_keep = [&](unsigned long long key) {
    if constexpr (kCluster > 1) {
      const unsigned int slot = atom_add_cluster(mapa_cluster(smem_u32(&s_ncand), 0u), 1u);
      if (slot < (unsigned int)kCandMax)
        st_cluster_u64(mapa_cluster(smem_u32(&s_cand[slot]), 0u), key);
    } else {
      const unsigned int slot = atomicAdd(&s_ncand, 1u);
      if (slot < (unsigned int)kCandMax) s_cand[slot] = key;
    }
  };
  for (int c0 = cbeg; c0 < cend; c0 += kThreads * kUnroll) {
    uint32_t o[kUnroll];
    row_ords(c0, o, cend);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (o[u] == 0u) continue;
      const uint32_t top = o[u] >> kBinShift32;
      if (all || top > bucket) keep_key(topk_key(o[u], entry_of(col_of(c0, u))));
      else if (top == bucket) bucket_keep(topk_key(o[u], entry_of(col_of(c0, u))));
    }
  }
  __syncthreads();
  if constexpr (kCluster > 1) cluster_sync_all();   // 3: every CTA's keys are in CTA 0

  if (!all && rank == 0) {
    // the keys of bucket B: from the buffer, or from the row when they did not all fit
    const unsigned int ncand = s_ncand;
    const bool in_smem = ncand <= (unsigned int)kCandMax;
    // f(key) for every key of bucket B
    const auto for_bucket = [&](auto f) {
      if (in_smem) {
        for (int i = tid; i < (int)ncand; i += kThreads) f(s_cand[i]);
        return;
      }
      for (int c0 = 0; c0 < a.ncols; c0 += kThreads * kUnroll) {   // the whole row
        uint32_t o[kUnroll];
        row_ords(c0, o, a.ncols);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (o[u] != 0u && (o[u] >> kBinShift32) == bucket)
            f(topk_key(o[u], entry_of(col_of(c0, u))));
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
        const unsigned int slot = atomicAdd(&s_kcnt, 1u);
        if (slot < (unsigned int)kIdxTopkMax) s_keys[slot] = key;
      }
    });
    __syncthreads();
  }

  int32_t* out = a.topk + t * a.k;
  if constexpr (kCluster > 1) {
    // The take keys sit unordered in CTA 0's s_keys.  Each CTA copies them, then ranks its share
    // [lo, hi): a key's output position is the number of keys above it (keys of one entry, which
    // are equal, in their order in the buffer).  G threads (a power of two, aligned lanes of a
    // warp) count one key's rank over every G-th key, and their sum places it.
    cluster_sync_all();   // 4: CTA 0's s_keys[0, take) are the selected keys
    const uint32_t src = mapa_cluster(smem_u32(s_keys), 0u);
    {
      constexpr int kPer = kIdxTopkMax / kThreads;
      unsigned long long v[kPer];   // all loads in flight before the stores
#pragma unroll
      for (int m = 0; m < kPer; ++m) {
        const int i = tid + m * kThreads;
        v[m] = i < (int)take ? ld_cluster_u64(src + 8u * (uint32_t)i) : 0ull;
      }
#pragma unroll
      for (int m = 0; m < kPer; ++m)
        if (tid + m * kThreads < (int)take) s_cand[tid + m * kThreads] = v[m];
    }
    cluster_arrive();   // 5 (arrival): this CTA no longer reads CTA 0's memory
    __syncthreads();
    const int per = ((int)take + kCluster - 1) / kCluster;
    const int lo = min((int)take, rank * per), hi = min((int)take, lo + per);
    int G = 1;
    while (G < 32 && 2 * G * per <= kThreads) G <<= 1;
    const int mine = lo + tid / G;   // the key this thread helps rank
    const int gl = tid & (G - 1);
    unsigned int above = 0;
    if (mine < hi) {
      const unsigned long long key = s_cand[mine];
      for (int j = gl; j < (int)take; j += G) {
        const unsigned long long o = s_cand[j];
        above += (o > key || (o == key && j < mine)) ? 1u : 0u;
      }
    }
    for (int o = 1; o < G; o <<= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
    if (mine < hi && gl == 0)
      out[above] = (int32_t)(0xFFFFFFFFu - (uint32_t)(s_cand[mine] & 0xFFFFFFFFull));
    for (int i = (int)take + rank * kThreads + tid; i < a.k; i += kThreads * kCluster) out[i] = -1;
    cluster_wait();   // 5: no CTA reads this CTA's memory any more
    return;
  }

  // bitonic sort (descending) of the take keys, padded with zeros to a power of two.  Stages of
  // stride 32 and more exchange through shared memory, one barrier each; the stages of stride
  // below 32 pair elements of one warp and run together in registers, with shuffles, behind one
  // barrier: all of sizes 2 .. 32 in one pass, then those of each larger size.
  int n = 1;
  while (n < (int)take) n <<= 1;
  // sizes 2 .. min(n, 32): every stage of these pairs elements of one warp, so they all run in
  // registers in one pass (the padding past take enters as zero keys)
  const int n_reg = n < 32 ? n : 32;
  for (int i0 = warp * 32; i0 < n; i0 += kThreads) {   // warp-uniform bounds
    const int i = i0 + lane;
    unsigned long long x = i < (int)take ? s_keys[i] : 0ull;
    for (int size = 2; size <= n_reg; size <<= 1) {
      const bool desc = (i & size) == 0;
      for (int st = size >> 1; st > 0; st >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, st);
        const bool lower = (lane & st) == 0;         // element i is the pair's first
        x = (lower == desc) ? (x > y ? x : y) : (x < y ? x : y);
      }
    }
    if (i < n) s_keys[i] = x;
  }
  __syncthreads();
  for (int size = 64; size <= n; size <<= 1) {
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

  for (int i = tid; i < a.k; i += kThreads)
    out[i] = i < (int)take ? (int32_t)(0xFFFFFFFFu - (uint32_t)(s_keys[i] & 0xFFFFFFFFull)) : -1;
}

// One row per cluster of kCluster CTAs.
template <int kThreads, int kUnroll, int kCluster>
cudaError_t launch_topk_cluster(const TopkArgs& a, cudaStream_t stream, bool query_only,
                                int* max_clusters, int sms) {
  const auto kern = topk_kernel<kThreads, kUnroll, kCluster>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess && kCluster > 8)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t c = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1] = pdl_attribute();
  c.gridDim = dim3((unsigned)(a.T * kCluster));
  c.blockDim = dim3(kThreads);
  c.dynamicSmemBytes = kSmemBytes;
  c.stream = stream;
  c.attrs = at;
  c.numAttrs = (query_only || 2LL * a.T * kCluster > sms) ? 1 : 2;
  if (query_only) return cudaOccupancyMaxActiveClusters(max_clusters, kern, &c);
  return cudaLaunchKernelEx(&c, kern, a);
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  if (a.T == 0 || a.k == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // A few rows: a cluster of CTAs per row, 16 (a non-portable size, if this device can place one)
  // or 8.  16 CTAs of 4096 columns take one row of 65,536 in 18.4 us, 8 of 8192 in 20.5 us, one
  // CTA in 30.7 us (GB300, L2 flushed).
  static int c16_fits[64];   // per device: 0 unknown, 1 yes, 2 no
  if ((long long)a.T * 16 <= sms && dev < 64) {
    if (c16_fits[dev] == 0) {
      int n = 0;
      e = launch_topk_cluster<512, 8, 16>(a, stream, true, &n, sms);
      if (e != cudaSuccess) (void)cudaGetLastError();
      c16_fits[dev] = (e == cudaSuccess && n >= 1) ? 1 : 2;
    }
    if (c16_fits[dev] == 1)
      return launch_topk_cluster<512, 8, 16>(a, stream, false, nullptr, sms);
  }
  if ((long long)a.T * 8 <= sms)
    return launch_topk_cluster<512, 16, 8>(a, stream, false, nullptr, sms);
  const bool few = a.T < sms;
  const auto kern = few ? topk_kernel<1024, 16, 1> : topk_kernel<512, 8, 1>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const bool pdl = 2LL * a.T <= sms;
  return launch_with_pdl(kern, dim3((unsigned)a.T), dim3(few ? 1024 : 512), (size_t)kSmemBytes,
                         stream, pdl, a);
}

}  // namespace spa

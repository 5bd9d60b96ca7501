// spa_kvwrite.cu - paged KV write: the rows of new tokens go to their pool slots, copied (bf16
// pools) or quantised to e4m3 with one scale per token and kv_head (FreeToken clone PR 3, "Perf/kv
// fp8 read path": the per-(token, kv_head) K and V scales its read path folds back in).
//
// The kernel is bound by HBM: per token it reads 4·D bytes and writes 4·D (bf16) or 2·D (e4m3)
// bytes plus the scales.  To keep enough bytes in flight it is a pipeline through shared memory.
// A producer thread bulk-copies the K rows and the V rows of a group of eight consecutive tokens
// (each contiguous in k and v) into a stage of a four-stage ring.  Eight consumer warps take one
// token of the group each, read its rows from shared memory, and store them to the token's slot:
// 16-byte chunks for bf16 pools; for e4m3 pools max|x| by shuffles, then 8 codes per 16-byte chunk
// (the codes of the IEEE fp32 quotients x / scale, spa_kvwrite_quant.cuh) and the row's scale.
// Each lane resolves the slot of its warp's token 32 groups ahead, so the dependent loads of a slot
// (position, sequence, block table) overlap the copies.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "spa_kvwrite_quant.cuh"
#include "spa_launch.h"

namespace spa {

namespace {

// |x| of the eight bf16 values of a 16-byte chunk, maximum
__device__ __forceinline__ float chunk_absmax(const uint4& u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(kvq_bf16_to_f32(w[i] & 0xFFFFu)));
    m = fmaxf(m, fabsf(kvq_bf16_to_f32(w[i] >> 16)));
  }
  return m;
}

constexpr int kKvwGroup = 8;                          // tokens per stage, one per consumer warp
constexpr int kKvwStages = 4;                         // stages of the shared-memory ring
constexpr int kKvwThreads = 32 * (kKvwGroup + 1);     // consumer warps + the producer warp
constexpr int kKvwCtasPerSm = 3;

// Shared memory of a CTA: the ring (per stage the K rows, then the V rows of kKvwGroup tokens),
// the stages' full and empty barriers, the abort flag.
int kvw_smem_bytes(int D) { return kKvwStages * 2 * kKvwGroup * 2 * D + 2 * kKvwStages * 8 + 16; }

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// A wait with the same outcome on every lane of the warp.
__device__ __forceinline__ bool kvw_warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// A wait that ends even when the CTA is aborting (the copies in flight must land before exit).
__device__ __forceinline__ void kvw_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; !mbar_try_wait(bar, parity); ++it) {
    if (it >= kWaitLimitPolls && globaltimer() - t0 > kWaitLimitNs) {
      flag_error(SPA_ERR_TIMEOUT);
      return;
    }
  }
}

// Slot row of token t: block_table[b][x / ps] * ps + x % ps, or -1 if it cannot be resolved.
__device__ __forceinline__ long long kvw_slot(const KvWriteArgs& a, long long t) {
  const int x = __ldg(a.positions + t);
  const int b = a.seq_of_token ? __ldg(a.seq_of_token + t) : 0;
  if (x < 0 || b < 0 || b >= a.B) return -1;
  const int page = x / a.ps;
  if (page >= a.bt_stride) return -1;
  const int blk = __ldg(a.bt + (size_t)b * a.bt_stride + page);
  if (blk < 0 || (long long)blk >= a.num_blocks) return -1;
  return (long long)blk * a.ps + x % a.ps;
}

template <bool kFp8>
__global__ void __launch_bounds__(kKvwThreads, kKvwCtasPerSm) kv_write_kernel(const KvWriteArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int row_bytes = 2 * a.D;                       // one bf16 input row
  const int blk_bytes = kKvwGroup * row_bytes;         // a stage's K (or V) rows
  const int ring_bytes = kKvwStages * 2 * blk_bytes;
  const uint32_t ring = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + ring_bytes + 2 * kKvwStages * 8);
#define FULL(s) (ring + (uint32_t)ring_bytes + 8u * (uint32_t)(s))
#define EMPTY(s) (ring + (uint32_t)ring_bytes + 8u * (uint32_t)(kKvwStages + (s)))
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long n_groups = ((long long)a.T + kKvwGroup - 1) / kKvwGroup;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kKvwStages; ++s) {
      mbar_init(FULL(s), 1);                 // the producer's armed arrival
      mbar_init(EMPTY(s), kKvwGroup);        // lane 0 of every consumer warp
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();   // nothing global before the grid before this one is done

  if (warp == kKvwGroup) {
    // ---- producer: group g's K rows and V rows into stage (local group index) % kKvwStages ----
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      for (long long g = blockIdx.x; g < n_groups; g += gridDim.x) {
        if (!mbar_wait(EMPTY(s), ph ^ 1u, abort_flag)) break;
        const long long t0 = g * kKvwGroup;
        const long long nt = a.T - t0 < kKvwGroup ? a.T - t0 : kKvwGroup;
        const uint32_t bytes = (uint32_t)(nt * row_bytes);
        const uint32_t dst = ring + (uint32_t)(s * 2 * blk_bytes);
        mbar_arrive_expect_tx(FULL(s), 2 * bytes);
        bulk_load(dst, a.k + t0 * row_bytes, bytes, FULL(s));
        bulk_load(dst + (uint32_t)blk_bytes, a.v + t0 * row_bytes, bytes, FULL(s));
        ++issued;
        if (++s == kKvwStages) { s = 0; ph ^= 1u; }
      }
      // Every copy must have landed before the CTA ends: at once after a normal run (the consumers
      // waited for them all), after the wait limit if the run was aborted.  Fill f went to stage
      // f % kKvwStages, barrier phase f / kKvwStages.
      for (long long f = issued - 1; f >= 0 && f >= issued - kKvwStages; --f)
        kvw_wait_drain(FULL(f % kKvwStages), (uint32_t)((f / kKvwStages) & 1));
    }
    return;
  }

  // ---- consumers: warp w takes token w of every group of this CTA ----
  int s = 0;
  uint32_t ph = 0;
  long long slot_ahead = -1;    // lane L: slot of this warp's token in group (it & ~31) + L
  int it = 0;
  for (long long g = blockIdx.x; g < n_groups; g += gridDim.x, ++it) {
    if ((it & 31) == 0) {
      const long long gl = g + (long long)lane * gridDim.x;
      const long long tl = gl * kKvwGroup + warp;
      slot_ahead = (gl < n_groups && tl < a.T) ? kvw_slot(a, tl) : -1;
    }
    const long long row = __shfl_sync(0xffffffffu, slot_ahead, it & 31);
    const long long t = g * kKvwGroup + warp;
    if (!kvw_warp_wait(FULL(s), ph, abort_flag)) break;
    if (t < a.T && row < 0) {
      if (lane == 0) flag_error(SPA_ERR_INDEX);
    } else if (t < a.T) {
      const uint8_t* sk = smem + s * 2 * blk_bytes + warp * row_bytes;   // the token's K row
      const uint8_t* sv = sk + blk_bytes;                                 // and V row
      const int nch = a.D >> 3;   // 16-byte chunks of eight bf16 values in a row (<= 64)
      if (!kFp8) {
        // slot row [2][D] bf16: K then V, 2 * nch chunks (<= 128, four per lane)
        uint4* dst = reinterpret_cast<uint4*>(a.kv + (size_t)row * 2 * row_bytes);
        uint4 u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = lane + 32 * i;
          if (c < 2 * nch)
            u[i] = *reinterpret_cast<const uint4*>(c < nch ? sk + 16 * c : sv + 16 * (c - nch));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = lane + 32 * i;
          if (c < 2 * nch) dst[c] = u[i];
        }
      } else {
        uint4 u[2], w[2];
        float amax = 0.f, vmax = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = lane + 32 * i;
          u[i] = c < nch ? *reinterpret_cast<const uint4*>(sk + 16 * c) : make_uint4(0, 0, 0, 0);
          w[i] = c < nch ? *reinterpret_cast<const uint4*>(sv + 16 * c) : make_uint4(0, 0, 0, 0);
          amax = fmaxf(amax, chunk_absmax(u[i]));
          vmax = fmaxf(vmax, chunk_absmax(w[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
        }
        const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        const float vscale = vmax > 0.f ? __fdiv_rn(vmax, 448.f) : 1.f;
        const float r = __frcp_rn(scale), vr = __frcp_rn(vscale);
        const bool fast = kvq_fast_scale(scale), vfast = kvq_fast_scale(vscale);
        uint2* dst = reinterpret_cast<uint2*>(a.kv + (size_t)row * 2 * a.D);
        uint2* dstv = reinterpret_cast<uint2*>(a.kv + ((size_t)row * 2 + 1) * a.D);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = lane + 32 * i;
          if (c < nch) {
            dst[c] = kvq_chunk(u[i], scale, r, fast);
            dstv[c] = kvq_chunk(w[i], vscale, vr, vfast);
          }
        }
        if (lane == 0) {
          a.k_scale[row] = scale;
          a.v_scale[row] = vscale;
        }
      }
    }
    // the stage's rows of this warp have been read into registers: hand the stage back
    __syncwarp();
    if (lane == 0) mbar_arrive(EMPTY(s));
    if (++s == kKvwStages) { s = 0; ph ^= 1u; }
  }
#undef FULL
#undef EMPTY
}

}  // namespace

// This translation unit's copy of the device error word (see spa_device.cuh).
cudaError_t read_and_clear_kv_write_error_word(int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_spa_error, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_spa_error, &zero, sizeof(int));
}

cudaError_t launch_kv_write(const KvWriteArgs& a, bool fp8, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int smem = kvw_smem_bytes(a.D);
  const auto kern = fp8 ? kv_write_kernel<true> : kv_write_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long groups = ((long long)a.T + kKvwGroup - 1) / kKvwGroup;
  const long long cap = (long long)sms * kKvwCtasPerSm;
  const unsigned blocks = (unsigned)(groups < cap ? groups : cap);
  return launch_with_pdl(kern, dim3(blocks), dim3(kKvwThreads), (size_t)smem, stream,
                         2LL * blocks <= sms, a);
}

}  // namespace spa

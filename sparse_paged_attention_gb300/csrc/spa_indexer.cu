// spa_indexer.cu - indexer logits over packed fp4 key rows (FreeToken PR 634, "Changes": key rows
// of 17 int32 words, 16 of e2m1 codes and one of ue8m0 scales, one scale per 32 elements, index
// head_dim 128; "Kernel time": 32 index heads; Full and candidate modes).
//
//   logit[t][c] = sum_h w[t][h] * max(0, q[t][h][:] . k[j][:]),   j = c (full) or cand[t][c]
//
// and -inf where entry j does not exist for query t (-1, non-causal: r*j + r - 1 > pos, or an
// invalid page, which also raises SPA_ERR_INDEX).
//
// The contraction runs on the tensor cores: a tile of 128 key rows is the MMA's M side, a group
// of up to eight queries' 32 heads its N side (N = 32 per query, up to 256) and the 128 dims its
// K, as tcgen05 kind::f16 with both operands bf16 in 128-byte-swizzled shared memory and the
// scores fp32 in TMEM.  The key rows are dequantised on the way into shared memory: every e2m1
// code times its ue8m0 scale is exactly a bf16 value (two significant bits times a power of two),
// so the keys enter the MMA unrounded.  The epilogue reads one key row's scores per thread
// (TMEM lane = key row), applies the ReLU and the head weights, and writes one logit per query.
//
// A CTA of four warps runs its units (query group, key tile) one after the other: load and
// dequantise, MMA, epilogue.  Units of one query group are contiguous in a CTA's range, so its
// queries stay in shared memory across tiles; full-mode tiles past every query's causal limit are
// written as -inf without an MMA.
#include <cuda_bf16.h>

#include "spa_indexer.h"
#include "spa_indexer_math.cuh"

namespace spa {

namespace {

constexpr int kTile = kIdxTile;            // key rows per unit (MMA M)
constexpr int kAAtom = kTile * 128;        // bytes of one 64-dim column of the key tile
constexpr int kAOff = 0;
constexpr int kBOff = 2 * kAAtom;          // 32 KB: the query tile follows the key tile
constexpr int kIdxCtasPerSm = 4;           // register budget: 128 threads x 128 registers each

// Shared memory and TMEM of a CTA, sized by its group's N = nq * 32 (queries x heads), so that
// groups of one query (candidate mode, several sequences, decode) leave room for many CTAs per SM
// where groups of eight fit two:
//   key tile [2 atoms][128 rows][128 B] | query tile [2 atoms][N rows][128 B] | weights [nq][32]
//   | positions [8], sequences [8] | mbarrier, TMEM base, abort flag
struct IdxLayout {
  int b_atom;          // bytes of one 64-dim column of the query tile (N rows x 128 B)
  int w_off, pos_off, bar_off, used;
  uint32_t tmem_cols;  // a power of two >= 32 covering N accumulator columns
};
__host__ __device__ inline IdxLayout idx_layout(int nq) {
  IdxLayout L;
  const int N = nq * kIdxHeads;
  L.b_atom = N * 128;                         // multiple of 1024 (N is a multiple of 32)
  L.w_off = kBOff + 2 * L.b_atom;
  L.pos_off = L.w_off + nq * kIdxHeads * 4;
  L.bar_off = L.pos_off + 2 * kIdxMaxQ * 4;
  L.used = L.bar_off + 64;
  L.tmem_cols = N <= 32 ? 32u : N <= 64 ? 64u : N <= 128 ? 128u : 256u;
  return L;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

template <bool kCand>
__global__ void __launch_bounds__(kIdxThreads, kIdxCtasPerSm) indexer_kernel(const IndexerArgs p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const IdxLayout L = idx_layout(p.nq);
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5;
  float* s_w = reinterpret_cast<float*>(sm + L.w_off);
  int* s_pos = reinterpret_cast<int*>(sm + L.pos_off);
  int* s_seq = s_pos + kIdxMaxQ;
  const uint32_t bar = sb + L.bar_off;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L.bar_off + 16);

  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();  // lane 0 of warp 0 took the branch above; the allocation is warp-collective
  if (warp == 0) tmem_alloc(sb + L.bar_off + 8, L.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();
  pdl_wait();   // nothing global before the grid before this one is done
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + L.bar_off + 8);
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);

  const int nq = p.nq, N = nq * kIdxHeads;
  const uint32_t idesc = idesc_bf16(kTile, N, 0, 0);
  const long long u0 = (long long)blockIdx.x * p.nunits / gridDim.x;
  const long long u1 = (long long)(blockIdx.x + 1) * p.nunits / gridDim.x;
  long long cur_group = -1;
  uint32_t phase = 0;

  for (long long u = u0; u < u1; ++u) {
    const long long g = u / p.ntiles;
    const int tile = (int)(u % p.ntiles);
    const int q0 = (int)(g * nq);
    const int nqg = min(nq, p.T - q0);

    if (g != cur_group) {  // the previous unit's MMA has completed: the query tile is free
      const int chunks = N * 16;  // 16-byte chunks of the N query rows (8 dims each)
      for (int idx = tid; idx < chunks; idx += kIdxThreads) {
        const int n = idx >> 4, k = idx & 15;
        const int ql = n / kIdxHeads, h = n % kIdxHeads;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ql < nqg)
          v = __ldg(reinterpret_cast<const uint4*>(
              p.q + ((size_t)(q0 + ql) * kIdxHeads + h) * kIdxDim + k * 8));
        st_shared_v4(sb + kBOff + (k >> 3) * L.b_atom + n * 128 + (((k & 7) ^ (n & 7)) << 4), v.x,
                     v.y, v.z, v.w);
      }
      for (int idx = tid; idx < nq * kIdxHeads; idx += kIdxThreads) {
        const int ql = idx / kIdxHeads;
        s_w[idx] = ql < nqg ? __ldg(p.w + (size_t)q0 * kIdxHeads + idx) : 0.f;
      }
      if (tid < kIdxMaxQ) {
        const bool live = tid < nqg;
        s_pos[tid] = live ? __ldg(p.positions + q0 + tid) : -1;
        s_seq[tid] = live ? (p.seq_of_token ? __ldg(p.seq_of_token + q0 + tid) : 0) : 0;
      }
      cur_group = g;
    }
    __syncthreads();

    int max_pos = -1;
    for (int ql = 0; ql < nqg; ++ql) max_pos = max(max_pos, s_pos[ql]);
    const long long causal_entries = max_pos < 0 ? 0 : ((long long)max_pos + 1) / p.ratio;
    const int c = tile * kTile + tid;

    if (!kCand && (long long)tile * kTile >= causal_entries) {
      // no query of the group reaches this tile: all -inf, no MMA (uniform over the CTA)
      if (c < p.ncols)
        for (int ql = 0; ql < nqg; ++ql)
          p.logits[(size_t)(q0 + ql) * p.ncols + c] = -INFINITY;
      __syncthreads();
      continue;
    }

    // this thread's key row: entry j, resolved through the sequence's block table
    long long j = -1, row = -1;
    if (c < p.ncols) j = kCand ? (long long)__ldg(p.cand + (size_t)q0 * p.ncols + c) : c;
    if (j >= 0 && j < causal_entries) {
      const int b = s_seq[0];
      const long long page = j / p.ps;
      bool ok = b >= 0 && b < p.B && page < p.bt_stride;
      if (ok) {
        const int blk = __ldg(p.bt + (size_t)b * p.bt_stride + page);
        ok = blk >= 0 && (long long)blk < p.num_blocks;
        if (ok) row = (long long)blk * p.ps + j % p.ps;
      }
      if (!ok) flag_error(SPA_ERR_INDEX);
    }
    {
      uint32_t words[kIdxRowWords];
      if (row >= 0) {
        const int32_t* src = p.keys + row * kIdxRowWords;
#pragma unroll
        for (int w = 0; w < kIdxRowWords; ++w) words[w] = (uint32_t)__ldg(src + w);
      } else {
#pragma unroll
        for (int w = 0; w < kIdxRowWords; ++w) words[w] = 0u;
        words[kIdxRowWords - 1] = 0x7F7F7F7Fu;  // scale 1: the row's scores are 0, then masked
      }
      float scale[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) scale[s] = e8m0_to_f32((words[16] >> (8 * s)) & 0xFFu);
      // a NaN scale (byte 0xFF) keeps the per-code path, whose NaN carries the code's sign
#pragma unroll
      for (int w = 0; w < 16; ++w) {  // word w: dims 8w .. 8w+7, one 16-byte chunk of the row
        const float sc = scale[w >> 2];
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t byte = (words[w] >> (8 * e)) & 0xFFu;
          pk[e] = e2m1x2_to_bf16x2_bits(byte, sc);
        }
        st_shared_v4(sb + kAOff + (w >> 3) * kAAtom + tid * 128 + (((w & 7) ^ (tid & 7)) << 4),
                     pk[0], pk[1], pk[2], pk[3]);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    if (tid == 0) {
      fence_proxy_async_smem();
      tc_fence_after();
#pragma unroll
      for (int s = 0; s < 8; ++s) {  // K = 128 in steps of 16: two 64-dim columns of 4 steps
        const uint64_t da = sdesc(sb + kAOff + (s >> 2) * kAAtom + (s & 3) * 32, 16, 1024);
        const uint64_t db = sdesc(sb + kBOff + (s >> 2) * L.b_atom + (s & 3) * 32, 16, 1024);
        mma_bf16(tmem, da, db, idesc, s > 0 ? 1u : 0u);
      }
      mma_commit(bar);
    }
    const bool done = mbar_wait(bar, phase, abort_flag);
    phase ^= 1u;
    if (!__syncthreads_and(done)) break;  // a wait gave up: SPA_ERR_TIMEOUT is set
    tc_fence_after();

    // tcgen05.ld and tcgen05.wait::ld are warp-collective (.sync.aligned): every lane of every
    // warp runs them, converged, whatever its column; only the store depends on the column
    __syncwarp();
    for (int ql = 0; ql < nqg; ++ql) {
      float v[32];
      tmem_ld32(lane_base + ql * kIdxHeads, v);
      tmem_wait_ld();
      float acc = 0.f;
#pragma unroll
      for (int h = 0; h < 32; ++h) acc = fmaf(s_w[ql * kIdxHeads + h], fmaxf(v[h], 0.f), acc);
      const bool causal = row >= 0 && (long long)p.ratio * j + p.ratio - 1 <= s_pos[ql];
      if (c < p.ncols) p.logits[(size_t)(q0 + ql) * p.ncols + c] = causal ? acc : -INFINITY;
    }
    tc_fence_before();
    __syncthreads();  // scores read and key tile consumed before the next unit overwrites them
  }

  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L.tmem_cols);
  }
}

}  // namespace

// This translation unit's copy of the device error word (see spa_device.cuh).
cudaError_t read_and_clear_indexer_error_word(int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_spa_error, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_spa_error, &zero, sizeof(int));
}

int indexer_smem_bytes(int nq) { return idx_layout(nq).used + 1024; }

cudaError_t launch_indexer(const IndexerArgs& a, bool cand, int num_sms, cudaStream_t stream) {
  if (a.nunits == 0) return cudaSuccess;
  const IdxLayout L = idx_layout(a.nq);
  const int smem = indexer_smem_bytes(a.nq);
  const void* fn = cand ? reinterpret_cast<const void*>(indexer_kernel<true>)
                        : reinterpret_cast<const void*>(indexer_kernel<false>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       indexer_smem_bytes(kIdxMaxQ));
  if (e != cudaSuccess) return e;
  // CTAs per SM: what shared memory (228 KB an SM, 1 KB of it reserved per CTA), registers (the
  // 4 CTAs of the launch bounds) and TMEM (512 columns: a CTA past that would wait in its
  // allocation for another CTA to end) allow together
  int per_sm = (228 * 1024) / (smem + 1024);
  if (per_sm > kIdxCtasPerSm) per_sm = kIdxCtasPerSm;
  const int tmem_fit = (int)(512u / L.tmem_cols);
  if (per_sm > tmem_fit) per_sm = tmem_fit;
  if (per_sm < 1) per_sm = 1;
  const long long cap = (long long)per_sm * num_sms;
  const long long grid = a.nunits < cap ? a.nunits : cap;
  const bool pdl = 2 * grid <= num_sms;
  if (cand)
    return launch_with_pdl(indexer_kernel<true>, dim3((unsigned)grid), dim3(kIdxThreads),
                           (size_t)smem, stream, pdl, a);
  return launch_with_pdl(indexer_kernel<false>, dim3((unsigned)grid), dim3(kIdxThreads),
                         (size_t)smem, stream, pdl, a);
}

}  // namespace spa

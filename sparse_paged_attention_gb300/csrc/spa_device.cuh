// spa_device.cuh - device helpers for the sm_103a sparse paged attention kernels:
// inline-PTX wrappers (mbarrier, cp.async, tcgen05), UMMA descriptors and the per-column
// page-table resolution shared by the attention kernels and the column dump.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "sparse_attn_paged.h"

namespace spa {

// ----------------------------------------------------------------------------------------
// Problem parameters as the kernels see them.
// ----------------------------------------------------------------------------------------
struct PoolDev {
  const uint8_t* kv;       // [num_blocks][page_size][2][D] elements
  const float* k_scale;    // fp8 only
  const float* v_scale;
  const int32_t* bt;       // [num_seqs][bt_stride]
  long long num_blocks;
  int ps;
  int ps_shift;            // log2(ps) when ps is a power of two, else -1
  int bt_stride;
};

struct ResolveArgs {
  PoolDev win, cmp;
  const int32_t* positions;
  const int32_t* seq_of_token;
  const int32_t* topk;
  int T, B, W, K, r;
};

constexpr int kColPoolShift = 30;

// Device error word: OR of SPA_ERR_INDEX / SPA_ERR_TIMEOUT.  Every translation unit that
// includes this header has its own copy on every device that loads the library; the host reads
// and clears the copies of the units whose kernels set it (spa_attention.cu, spa_kvwrite.cu) in
// sparse_attn_paged_check_errors.
static __device__ int g_spa_error;

__device__ __forceinline__ void flag_error(int code) { atomicOr(&g_spa_error, code); }

// Column c of query t (sequence b, position pos): the physical row in the dump encoding, or -1.
// Window column c < W holds token pos - W + 1 + c; top-k column holds entry topk[t][c - W],
// present iff >= 0, r > 0 and r*j + r - 1 <= pos.  Out-of-table pages and out-of-pool blocks
// are input errors: the column is dropped and SPA_ERR_INDEX is raised.
//
// Two steps, so that a caller resolving many columns can have all the loads of one step in
// flight at once: column_page finds the pool, the page of the block table and the slot in the
// page (it reads the top-k list), column_row reads the block table.
struct ColumnPage {
  int pool;   // 0 window, 1 compressed, -1 no column
  int page;   // index into the sequence's block table (-1: beyond the table, an input error)
  int slot;   // row within the page
};

// x = page * ps + slot for 0 <= x < 2^31 (a shift and a mask for the usual power-of-two pages)
__device__ __forceinline__ void split_page(int x, const PoolDev& pl, int& page, int& slot) {
  if (pl.ps_shift >= 0) {
    page = x >> pl.ps_shift;
    slot = x & (pl.ps - 1);
  } else {
    page = x / pl.ps;
    slot = x - page * pl.ps;
  }
}

// The top-k entry of column c of query t, or -1 for a window column (or no compressed pool): the
// one read of a column that does not depend on the query's sequence or position, so a caller can
// have it in flight together with those.
__device__ __forceinline__ int column_topk(const ResolveArgs& a, int t, int c) {
  return (c >= a.W && a.r > 0) ? __ldg(a.topk + (long long)t * a.K + (c - a.W)) : -1;
}

// column_page given the column's top-k entry j (column_topk).
__device__ __forceinline__ ColumnPage column_page_j(const ResolveArgs& a, int pos, int c, int j) {
  ColumnPage cp{-1, 0, 0};
  if (c < a.W) {
    const long long x = (long long)pos - a.W + 1 + c;
    if (x < 0) return cp;
    cp.pool = 0;
    if (x <= 0x7fffffffLL) {
      int lp;
      split_page((int)x, a.win, lp, cp.slot);
      cp.page = lp < a.win.bt_stride ? lp : -1;
    } else {
      const long long lp = x / a.win.ps;
      cp.page = lp < a.win.bt_stride ? (int)lp : -1;
      cp.slot = (int)(x % a.win.ps);
    }
    return cp;
  }
  if (a.r <= 0) return cp;
  if (j < 0) return cp;
  if ((long long)a.r * j + a.r - 1 > pos) return cp;
  int lp;
  split_page(j, a.cmp, lp, cp.slot);
  cp.pool = 1;
  cp.page = lp < a.cmp.bt_stride ? lp : -1;
  return cp;
}

__device__ __forceinline__ ColumnPage column_page(const ResolveArgs& a, int t, int pos, int c) {
  return column_page_j(a, pos, c, column_topk(a, t, c));
}

__device__ __forceinline__ int32_t column_row(const ResolveArgs& a, int b, const ColumnPage& cp) {
  if (cp.pool < 0) return -1;
  const PoolDev& pl = cp.pool ? a.cmp : a.win;
  if (cp.page < 0) { flag_error(SPA_ERR_INDEX); return -1; }
  const int blk = __ldg(pl.bt + (long long)b * pl.bt_stride + cp.page);
  if (blk < 0 || blk >= pl.num_blocks) { flag_error(SPA_ERR_INDEX); return -1; }
  const uint32_t row = (uint32_t)((long long)blk * pl.ps + cp.slot);
  return (int32_t)(cp.pool ? ((1u << kColPoolShift) | row) : row);
}

__device__ __forceinline__ int32_t resolve_column(const ResolveArgs& a, int t, int b, int pos,
                                                  int c) {
  return column_row(a, b, column_page(a, t, pos, c));
}

// Sequence of token t, checked against the table height.
__device__ __forceinline__ int seq_of(const ResolveArgs& a, int t, bool* ok) {
  const int b = a.seq_of_token ? __ldg(a.seq_of_token + t) : 0;
  *ok = (b >= 0 && b < a.B);
  if (!*ok) flag_error(SPA_ERR_INDEX);
  return b;
}

// ----------------------------------------------------------------------------------------
// PTX wrappers
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Programmatic dependent launch (griddepcontrol, sm_90 and later).  A grid launched with
// programmatic stream serialization may start while the grid before it in the stream still runs:
// pdl_launch_dependents() lets the next grid start (once every CTA of this one has run it or
// exited), and pdl_wait() returns once the grid before has completed and its memory operations
// are visible (at once when the launch had no such predecessor).  A kernel runs pdl_wait() in
// every thread before its first global memory access, so it reads and writes nothing that the
// grid before it may still touch.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// The launch attribute that allows it.
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a = {};
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}
// A launch with that attribute when `pdl`.  The launchers set it when a grid has at most half as
// many CTAs as there are SMs, so that the next grid can set up on idle SMs while this one runs.
// A larger grid would instead have its CTAs placed where the grid before it leaves room, beside
// its CTAs or in the order they finish (measured slower: the indexer's 128-CTA decode grid, the
// attention's prefill grid).
template <typename Kern, typename... Args>
inline cudaError_t launch_with_pdl(Kern kern, dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t stream, bool pdl, const Args&... args) {
  cudaLaunchConfig_t c = {};
  c.gridDim = grid;
  c.blockDim = block;
  c.dynamicSmemBytes = smem;
  c.stream = stream;
  cudaLaunchAttribute at[1] = {pdl_attribute()};
  c.attrs = at;
  c.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&c, kern, args...);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Limits of one pipeline wait.  A wait gives up only after at least kWaitLimitPolls polls AND
// kWaitLimitNs of wall-clock time: the poll count keeps a pause of the whole GPU (a debugger or
// profiler stopping the kernel) from being mistaken for a stuck pipeline, the clock keeps fast
// polls from giving up early.  Giving up raises SPA_ERR_TIMEOUT and sets the CTA's abort flag,
// after which every role leaves its loop and the kernel ends cleanly.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitLimitPolls = 1u << 24;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort_flag) return false;
      if (it >= kWaitLimitPolls && globaltimer() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        flag_error(SPA_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ---- thread-block clusters: distributed shared memory between the CTAs of one cluster ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The same shared-memory offset in CTA `rank` of this cluster (a shared::cluster address).
__device__ __forceinline__ uint32_t mapa_cluster(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr)
               : "memory");
  return v;
}
// Arrive on an mbarrier of any CTA of the cluster.  Release at cluster scope: this thread's
// earlier shared-memory writes (local or remote) are visible to whoever acquires the phase.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded wait for a phase completed by arrivals from other CTAs of the cluster (same limits
// as mbar_wait; gives up early when this CTA is aborting).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag) {
  if (mbar_try_wait_acq_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort_flag) return false;
      if (it >= kWaitLimitPolls && globaltimer() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        flag_error(SPA_ERR_TIMEOUT);
        return false;
      }
    }
  }
}
// Arm a barrier phase with an expected transaction byte count (counts as this thread's arrival).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Bulk copy from this CTA's shared memory to the shared memory of a CTA of the cluster; the
// bytes complete the transaction count of the destination CTA's barrier `cluster_bar`.
// Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_cluster(uint32_t cluster_dst, uint32_t src, uint32_t bytes,
                                                  uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(cluster_dst), "r"(src), "r"(bytes), "r"(cluster_bar)
      : "memory");
}
// Cluster-wide barrier of all threads of all CTAs (every thread arrives once per phase).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// Named barrier over `count` threads (whole warps).  bar.sync is the warp-aligned form: a warp
// must reach it converged, or it may be counted more than once and the barrier's later phases
// pair up the wrong warps.  The warp is reconverged first, whatever divergent code (a lane-0
// store, a per-lane poll loop) came before.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// 16-byte global -> shared copy; src_bytes == 0 writes zeros without reading.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed (no pending-count
// increment: the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Tensor-map row copies into shared memory (the map's box is 128 bytes of one row, 128-byte
// swizzle; the swizzle follows the destination address, so a row may land at any 128-byte line of
// a 1024-byte-aligned atom).  Completion: `bytes` of the barrier's transaction count.
//   tma_gather4: four rows (any row indices of the map) to four consecutive 128-byte lines.
//   tma_row:     one row.
// x is the byte offset within the row (a multiple of 128 here).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0,
                                            int r1, int r2, int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_row(uint32_t dst, const CUtensorMap* map, int x, int r,
                                        uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4 (here e4m3 x e4m3, fp32 accumulate).
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` when every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 bits, 32 consecutive TMEM columns: thread i of the warp gets lane (base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// 32 lanes x 32 bits, 16 consecutive TMEM columns: thread i of the warp writes lane (base + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x on the SFU (PTX ex2.approx; ftz: subnormal results flush to zero, which only drops
// probabilities below 2^-126 of the running maximum).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ----------------------------------------------------------------------------------------
// UMMA descriptors (tcgen05 shared-memory matrix descriptor, 128-byte swizzle).
//
// Every operand tile here is built from 128-byte rows grouped by 8 into 1024-byte swizzle
// atoms; inside an atom the 16-byte chunk k of row r sits at chunk position (k ^ (r & 7)).
//   K-major operand (rows = M or N, 64 bf16 / 128 e4m3 of K per row): SBO = 1024 (next group
//     of 8 rows); LBO unused.  Advancing K inside the atom adds the byte offset to the start.
//   MN-major operand (rows = K, 128 bytes of M or N per row): LBO = byte distance to the next
//     128-byte block along M/N, SBO = 1024 (next group of 8 K rows).
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn_major << 15) |
         ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with e4m3 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)a_mn_major << 15) |
         ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace spa

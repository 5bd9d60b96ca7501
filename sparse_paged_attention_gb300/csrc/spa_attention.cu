// spa_attention.cu - sm_103a sparse paged attention: tcgen05 kernel, split-K merge, column dump.
//
// One CTA per SM runs a persistent loop over work items (query token, group of 64 heads, split
// of the column list).  For each item it resolves and compacts the query's column set, then
// streams it in tiles of 128 columns:
//
//   gather warps (5..)   resolve columns through the block tables (FreeToken PR 633, "Changes":
//                        per-column choice of window or compressed pool), then copy every K and V
//                        row into shared memory, already in the 128-byte-swizzled operand layout,
//                        through a 4-slot ring: by tensor-map gathers (four rows of 128 bytes per
//                        copy, six warps issuing in pairs) when CTAs take several items, by
//                        16-byte cp.async (four warps) in CTAs of a single item (decode).
//   MMA warp (4)         S^T[c][h] = K[c][:] . Q[h][:]    tcgen05, M = 128 columns, N = heads
//                        O^T[d][h] += V[c][d] * P^T[c][h] tcgen05, M = 128 of head_dim, N = 64
//                        both accumulate in TMEM (S^T double-buffered, O^T resident).
//   softmax warps (0..3) one thread per column: read S^T from TMEM, mask, online max and sum
//                        across columns (warp shuffles plus a 4-warp exchange), write P^T to
//                        shared memory; at the end divide O by the denominators and store.
//
// Heads sit in the N dimension, columns (and head_dim) in M = 128: an M = 128 tcgen05 tile runs
// the tensor core at its full per-SM rate and keeps one TMEM lane per row, which a 64-row tile of
// heads would not.
//
// e4m3 pools (FreeToken clone PR 3, "Perf/kv fp8 read path", part 1): K and V codes reach the
// MMA unwidened (kind::f8f6f4, both operands e4m3).  q is split into q_hi + q_lo, two e4m3 terms
// (times a power of two per token) that the S MMA reads as N = 128 rows, so the sum of the two
// accumulator halves carries q to about bf16 precision.  The per-row K scale multiplies the scores
// in fp32.  The probabilities are scaled by the per-row V scale (and a power of two per item),
// split the same way into two e4m3 terms, and both accumulate into the same O; the softmax
// denominator sums the unscaled fp32 probabilities.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "spa_launch.h"

namespace spa {

namespace cfg {
constexpr int kStages = 4;            // K/V ring slots
constexpr int kSlotBytes = 32768;     // 128 rows x 256 bytes (two 128-byte swizzle atoms)
constexpr int kAtomBytes = 16384;     // 128 rows x 128 bytes
constexpr int kTi = 4;                // tile-info ring entries
constexpr int kTmemCols = 512;

struct TileInfo {                     // one entry of the tile-info ring
  int item, n, flags, pad;
  float q_scale, p_scale, pad1, pad2; // e4m3 only: 2^k applied to q and to the probabilities
  float k_scale[128];                 // e4m3 only: per-column K and V scales of this tile
  float v_scale[128];
};

constexpr int kRingOff = 0;
constexpr int kQOff = kRingOff + kStages * kSlotBytes;      // 131072 (64 KB)
constexpr int kPOff = kQOff + 65536;                        // 196608 (16 KB)
constexpr int kListOff = kPOff + 16384;                     // 212992  int32 [2][kMaxColumns]
constexpr int kRedOff = kListOff + 2 * kMaxColumns * 4;     // 221184  float [2][4][64]
constexpr int kMrowOff = kRedOff + 2 * 4 * 64 * 4;          // 219136  float [4][64]
constexpr int kArowOff = kMrowOff + 4 * 64 * 4;             // 220160  float [4][64]
constexpr int kTiOff = kArowOff + 4 * 64 * 4;               // 221184  TileInfo [kTi]
constexpr int kCntOff = kTiOff + kTi * (int)sizeof(TileInfo);
constexpr int kInfoOff = kCntOff + 128;                     // ItemInfo [2]
constexpr int kBarOff = kInfoOff + 32;

struct ItemInfo {                     // one resolved item, handed from the resolver to the gather
  int item;                           // -1: no more items
  int n;                              // compacted columns in the item's list
  float p_scale;                      // e4m3 only: 2^k applied to the probabilities
  int pad;
};

enum {
  B_FULL = 0, B_EMPTY = 4, B_QFULL = 8, B_QEMPTY = 9, B_SFULL = 10, B_SEMPTY = 12,
  B_PFULL = 14, B_PVDONE = 15, B_OFREE = 16, B_TIFULL = 17, B_TIEMPTY = 21, B_RED = 25,
  B_DRAIN = 27, B_READY = 28, B_RECV = 29, B_RECVML = 30, B_LFULL = 31, B_LEMPTY = 33,
  B_COUNT = 35
};
constexpr int kMiscOff = kBarOff + B_COUNT * 8;             // TMEM base, abort flag
constexpr int kSmemBytes = kMiscOff + 16 + 1024;            // + slack to align the base to 1 KB
static_assert(sizeof(TileInfo) % 16 == 0, "tile info alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr int kFirst = 1, kLast = 2;
constexpr int kTmaFillWarps = 2;      // gather warps that issue one ring fill together
}  // namespace cfg

template <bool kFp8, bool kTmaRows>
struct Mode {
  static constexpr int kElt = kFp8 ? 1 : 2;        // bytes per K/V element
  static constexpr int kSCols = kFp8 ? 128 : 64;   // N of the S MMA (q, or q_hi | q_lo)
  static constexpr int kOCol = 2 * kSCols;         // first TMEM column of O^T
  static constexpr int kQAtom = kSCols * 128;      // bytes of one 128-byte-wide Q atom
  static constexpr float kTau = kFp8 ? 4.0f : 8.0f;  // lazy rescale threshold (log2 units)
  static constexpr bool kTma = kTmaRows;           // rows by tensor-map gathers (else cp.async)
  static constexpr int kNG = attn_gather_warps(kTmaRows);  // gather warps
  static constexpr int kNGT = 32 * kNG;
};

int attn_smem_bytes() { return cfg::kSmemBytes; }

// Butterfly "transpose-reduce" of 32 per-thread values across the 32 lanes of a warp: after five
// halving steps (16 + 8 + 4 + 2 + 1 shuffles) lane L holds the reduction over the warp of value L.
template <bool kMax>
__device__ __forceinline__ float xreduce32(const float (&v)[32], int lane) {
  float a[16], b[8], c[4], d[2];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float send = up ? v[k] : v[k + 16];
      const float keep = up ? v[k + 16] : v[k];
      const float o = __shfl_xor_sync(0xffffffffu, send, 16);
      a[k] = kMax ? fmaxf(keep, o) : keep + o;
    }
  }
  {
    const bool up = lane & 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float send = up ? a[k] : a[k + 8];
      const float keep = up ? a[k + 8] : a[k];
      const float o = __shfl_xor_sync(0xffffffffu, send, 8);
      b[k] = kMax ? fmaxf(keep, o) : keep + o;
    }
  }
  {
    const bool up = lane & 4;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float send = up ? b[k] : b[k + 4];
      const float keep = up ? b[k + 4] : b[k];
      const float o = __shfl_xor_sync(0xffffffffu, send, 4);
      c[k] = kMax ? fmaxf(keep, o) : keep + o;
    }
  }
  {
    const bool up = lane & 2;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float send = up ? c[k] : c[k + 2];
      const float keep = up ? c[k + 2] : c[k];
      const float o = __shfl_xor_sync(0xffffffffu, send, 2);
      d[k] = kMax ? fmaxf(keep, o) : keep + o;
    }
  }
  const bool up = lane & 1;
  const float send = up ? d[0] : d[1];
  const float keep = up ? d[1] : d[0];
  const float o = __shfl_xor_sync(0xffffffffu, send, 1);
  return kMax ? fmaxf(keep, o) : keep + o;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// A wait whose outcome is the same on every lane of the warp (the softmax warps shuffle right
// after their waits, so a lane must never leave the loop alone).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// The same for phases completed by arrivals from the CTAs of the cluster (parity 0: one use).
__device__ __forceinline__ bool warp_wait_cl(uint32_t bar, volatile int* abort_flag) {
  const bool ok = mbar_wait_cluster(bar, 0, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// A wait that must end even when the CTA is aborting (drain before releasing TMEM).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; !mbar_try_wait(bar, parity); ++it) {
    if (it >= kWaitLimitPolls && globaltimer() - t0 > kWaitLimitNs) {
      flag_error(SPA_ERR_TIMEOUT);
      return;
    }
  }
}

// Storage position of compacted column i in a column list.  Tensor-map gathers take four
// consecutive columns, so their lists are in column order (natural).  For cp.async, within each
// block of 128 columns, column 16b + c is stored at 8c + b, so the eight columns a gather thread
// copies in one tile (c fixed, b = 0..7) are eight consecutive words: two 16-byte loads.
__device__ __forceinline__ int list_pos(int i, bool natural) {
  return natural ? i : ((i & ~127) | ((i & 15) << 3) | ((i >> 4) & 7));
}

// 2^floor(log2 x) for finite x > 0 (clears the mantissa; x is kept within the normal range).
__device__ __forceinline__ float pow2_floor(float x) {
  x = fminf(fmaxf(x, 1.17549435e-38f), 1.0e38f);
  return __int_as_float(__float_as_int(x) & 0x7F800000);
}

// Two fp32 values -> two e4m3 codes (round to nearest even, saturating), first value low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}
// (a, b) -> hi = e4m3(a, b), lo = e4m3(a - hi_a, b - hi_b): hi + lo carries about 8 bits.  The
// pair is rounded to f16 first (11 bits, far finer than the split's 8; the values are at most 448
// here) so that the codes, their values and the residual are all packed half arithmetic.
__device__ __forceinline__ void split_e4m3x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 ah = __floats2half2_rn(a, b);
  hi = (uint32_t)__nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&ah),
                                            __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)hi, __NV_E4M3);
  const __half2 res = __hsub2(ah, *reinterpret_cast<const __half2*>(&hr));
  lo = (uint32_t)__nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&res),
                                            __NV_SATFINITE, __NV_E4M3);
}

// Two fp32 values -> packed bf16x2 (round to nearest even), first value in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// tcgen05 shared-memory descriptor, 64-byte swizzle (used for the e4m3 P^T operand).
__device__ __forceinline__ uint64_t sdesc64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;  // 64-byte swizzle
  return d;
}

// A descriptor moved by `bytes` within shared memory: the start address is bits [0, 14) in 16-byte
// units, and every address of the CTA's shared memory fits them, so the sum never carries into the
// next field.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// kRes: a resolver warp (the last) walks the page tables of a CTA's next item while the gather
// warps copy the current one; launched only when CTAs have more than one item.
// kTma: K/V rows move by tensor-map gathers (CTAs with many items: throughput); otherwise by
// cp.async, whose lower issue latency suits CTAs of a single item (decode), and which also takes
// e4m3 rows of a head_dim that is not a multiple of 128.
template <bool kFp8, bool kRes, bool kTma>
__global__ void __launch_bounds__(attn_threads(kTma, kRes), 1)
    attn_kernel(const __grid_constant__ AttnParams p) {
  using namespace cfg;
  using M = Mode<kFp8, kTma>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kMiscOff + 4);
  TileInfo* ti = reinterpret_cast<TileInfo*>(sm + kTiOff);
#define BAR(i) (sb + (uint32_t)kBarOff + 8u * (uint32_t)(i))

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      // tensor maps: the armed arrivals of the pair of gather warps that fills the slot;
      // cp.async: the noinc arrivals of the first 128 gather threads
      mbar_init(BAR(B_FULL + i), M::kTma ? kTmaFillWarps : 128);
      mbar_init(BAR(B_EMPTY + i), 1);
    }
    mbar_init(BAR(B_QFULL), 128);
    mbar_init(BAR(B_QEMPTY), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(B_SFULL + i), 1);
      mbar_init(BAR(B_SEMPTY + i), 128);
      mbar_init(BAR(B_RED + i), 4);
    }
    mbar_init(BAR(B_PFULL), 128);
    mbar_init(BAR(B_PVDONE), 1);
    mbar_init(BAR(B_OFREE), 128);
    for (int i = 0; i < kTi; ++i) {
      mbar_init(BAR(B_TIFULL + i), 1);
      mbar_init(BAR(B_TIEMPTY + i), 5);
    }
    mbar_init(BAR(B_DRAIN), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(B_LFULL + i), 1);    // the resolver's lane 0
      mbar_init(BAR(B_LEMPTY + i), M::kNG);   // lane 0 of every gather warp
    }
    // cluster merge: one "ring idle" arrival from every CTA; the bulk copies of every CTA's
    // slice and (m, l) complete the receive barrier's transaction count, armed here
    mbar_init(BAR(B_READY), p.cluster > 1 ? p.cluster : 1);
    mbar_init(BAR(B_RECV), 1);
    mbar_init(BAR(B_RECVML), 1);
    if (p.cluster > 1) {
      mbar_arrive_expect_tx(BAR(B_RECV), (uint32_t)(p.D * p.gh * 2));
      mbar_arrive_expect_tx(BAR(B_RECVML), (uint32_t)(p.cluster * p.gh * 8));
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) tmem_alloc(sb + kMiscOff, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + kMiscOff);
  // The set-up above touches no global memory.  Under programmatic dependent launch the next grid
  // may now start setting up, and nothing below runs before the grid before this one is done.
  if (p.pdl) {
    pdl_launch_dependents();
    pdl_wait();
  }
  // A cluster's CTAs touch one another's shared memory only after all of them have started and
  // initialised their barriers: every thread arrives here and waits before its first remote access.
  const bool clustered = p.cluster > 1;
  bool cl_started = !clustered;
  bool recv_ok = false;  // thread 0: the cluster merge's receive barrier was seen complete
  if (clustered) cluster_arrive();

  const int D = p.D;
  const int P16 = D * M::kElt / 16;       // 16-byte pieces per K (or V) row
  const int n_atoms = (P16 + 7) >> 3;     // 128-byte swizzle atoms per row
  const int n_chunks = (n_atoms + 1) >> 1;  // ring slots per K tile (and per V tile)
  const int n_ks = P16 >> 1;              // 32-byte K steps of the S MMA
  const int n_mt = (D + 127) >> 7;        // 128-wide head_dim tiles of O^T
  const int C = p.rs.W + p.rs.K;
  constexpr bool tma = M::kTma;

  if (warp >= 4) {
    if (kRes && warp == 5 + M::kNG) {
      // ==================================== resolve =====================================
      // One warp walks the page tables of the next item while the gather warps copy the rows of
      // the current one: two column lists, handed over through B_LFULL / B_LEMPTY.
      // The CTA's first item is resolved by the gather warps themselves (nothing to overlap it
      // with); this warp takes the u-th item, u >= 1, into list u & 1.
      int32_t* lists = reinterpret_cast<int32_t*>(sm + kListOff);
      ItemInfo* info = reinterpret_cast<ItemInfo*>(sm + kInfoOff);
      for (int u = 1;; ++u) {
        const long long item_ll = (long long)blockIdx.x + (long long)u * gridDim.x;
        const int lb = u & 1;
        if ((long long)blockIdx.x + (long long)u * gridDim.x >= p.n_items) break;
        // the list is free once the gather warps are done with item u - 2
        if (u >= 2 && !warp_wait(BAR(B_LEMPTY + lb), ((u - 2) >> 1) & 1, abort_flag)) break;
        const int item = (int)item_ll;
        const int s = item % p.n_splits;
        const int tg = item / p.n_splits;
        const int t = tg / p.n_groups;
        const int c_lo = s * p.cols_per_split;
        const int c_hi = min(C, c_lo + p.cols_per_split);
        bool seq_ok;
        const int b = seq_of(p.rs, t, &seq_ok);
        const int pos = __ldg(p.rs.positions + t);
        int32_t* list = lists + lb * kMaxColumns;
        int n = 0;
        float vmax = 0.f;  // largest V scale of the item's columns (e4m3)
        // 256 columns per round, eight per lane: the eight top-k reads, then the eight block-table
        // reads, are each in flight together
        for (int c0 = c_lo; c0 < c_hi; c0 += 256) {
          ColumnPage cp[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int c = c0 + k * 32 + lane;
            cp[k] = (seq_ok && c < c_hi) ? column_page(p.rs, t, pos, c) : ColumnPage{-1, 0, 0};
          }
          int32_t code[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) code[k] = column_row(p.rs, b, cp[k]);
          if (kFp8) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (code[k] >= 0) {
                const float* vs = (code[k] >> kColPoolShift) ? p.rs.cmp.v_scale : p.rs.win.v_scale;
                vmax = fmaxf(vmax, fabsf(__ldg(vs + (code[k] & ((1 << kColPoolShift) - 1)))));
              }
            }
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const unsigned m = __ballot_sync(0xffffffffu, code[k] >= 0);
            if (code[k] >= 0) list[list_pos(n + __popc(m & ((1u << lane) - 1u)), tma)] = code[k];
            n += __popc(m);
          }
        }
        float p_scale = 1.f;
        if (kFp8 && n > 0) {
          vmax = warp_max(vmax);
          // probabilities are <= 2^tau, so P * v_scale * p_scale stays <= 448
          p_scale = vmax > 0.f ? pow2_floor(448.f / (exp2f(M::kTau) * vmax)) : 1.f;
        }
        if (lane == 0) info[lb] = ItemInfo{item, n, p_scale, 0};
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_LFULL + lb));
      }
    } else if (warp >= 5 && warp < 5 + M::kNG) {
      // ===================================== gather ======================================
      constexpr int NG = M::kNG, NGT = M::kNGT;
      static_assert(!M::kTma || NG % kTmaFillWarps == 0, "tensor-map gathers run in warp groups");
      const int ptid = threadIdx.x - 160;
      const int pw = warp - 5;
      volatile int* cnt = reinterpret_cast<volatile int*>(sm + kCntOff);            // [16]
      volatile int* abort_copy = cnt + 16;
      volatile float* fred = reinterpret_cast<volatile float*>(sm + kCntOff + 80);  // [8]
      const int jj = ptid & 7, r0 = ptid >> 3;
      // cp.async: this thread copies chunk jj of rows r0, r0 + 16, ...: (r & 7) == (r0 & 7) for all
      const uint32_t dst_thread = (uint32_t)(r0 * 128 + ((jj ^ (r0 & 7)) << 4));
      const size_t row_bytes = (size_t)2 * D * M::kElt;  // K row then V row
      int ring = 0, tik = 0;
      uint32_t ring_ph = 0, ti_ph = 0, q_ph = 0;
      int fills = 0;  // ring slots this thread has filled
      // threads that write a tile-info entry: thread 0, and for e4m3 the first 128 (per-column
      // K and V scales)
      const bool ti_writer = kFp8 ? ptid < 128 : ptid == 0;
      int32_t* lists = reinterpret_cast<int32_t*>(sm + kListOff);
      const ItemInfo* info = reinterpret_cast<const ItemInfo*>(sm + kInfoOff);
      for (int u = 0;; ++u) {
        const int lb = kRes ? (u & 1) : 0;
        if ((long long)blockIdx.x + (long long)u * gridDim.x >= p.n_items) break;
        // item u's column list: resolved right here for the first item (and for every item
        // without a resolver warp), handed over by the resolver warp for the later ones
        const bool handed = kRes && u > 0;
        if (handed) mbar_wait(BAR(B_LFULL + lb), ((u - 1) >> 1) & 1, abort_flag);
        // uniform abort check (one thread samples the flag, everyone reads the copy); it also
        // catches a list wait that gave up
        named_bar_sync(2, NGT);
        if (ptid == 0) *abort_copy = *abort_flag;
        named_bar_sync(2, NGT);
        if (*abort_copy) break;
        int item, n;
        float p_scale = 1.f;
        int32_t* list = lists + lb * kMaxColumns;
        if (handed) {
          const ItemInfo ii = info[lb];
          item = ii.item;
          n = ii.n;
          p_scale = ii.p_scale;
        } else {
          item = (int)((long long)blockIdx.x + (long long)u * gridDim.x);
          const int s0 = item % p.n_splits;
          const int t0 = item / p.n_splits / p.n_groups;
          const int c_lo = s0 * p.cols_per_split;
          const int c_hi = min(C, c_lo + p.cols_per_split);
          // the first round's top-k entries are read together with the sequence and position
          const int j0 = c_lo + ptid < c_hi ? column_topk(p.rs, t0, c_lo + ptid) : -1;
          bool seq_ok;
          const int b = seq_of(p.rs, t0, &seq_ok);
          const int pos = __ldg(p.rs.positions + t0);
          n = 0;
          float vmax = 0.f;  // largest V scale of the item's columns (e4m3)
          for (int c0 = c_lo; c0 < c_hi; c0 += NGT) {
            const int c = c0 + ptid;
            const int j = c0 == c_lo ? j0 : (c < c_hi ? column_topk(p.rs, t0, c) : -1);
            const int32_t code =
                (seq_ok && c < c_hi) ? column_row(p.rs, b, column_page_j(p.rs, pos, c, j)) : -1;
            if (kFp8 && code >= 0) {
              const float* vs = (code >> kColPoolShift) ? p.rs.cmp.v_scale : p.rs.win.v_scale;
              vmax = fmaxf(vmax, fabsf(__ldg(vs + (code & ((1 << kColPoolShift) - 1)))));
            }
            const unsigned m = __ballot_sync(0xffffffffu, code >= 0);
            if (lane == 0) cnt[pw] = __popc(m);
            named_bar_sync(2, NGT);
            int off = n, tot = 0;
#pragma unroll
            for (int w = 0; w < NG; ++w) {
              const int cw = cnt[w];
              off += (w < pw) ? cw : 0;
              tot += cw;
            }
            if (code >= 0) list[list_pos(off + __popc(m & ((1u << lane) - 1u)), tma)] = code;
            n += tot;
            named_bar_sync(2, NGT);
          }
          if (kFp8 && n > 0) {
            vmax = warp_max(vmax);
            if (lane == 0) fred[pw] = vmax;
            named_bar_sync(2, NGT);
            vmax = 0.f;
#pragma unroll
            for (int w = 0; w < NG; ++w) vmax = fmaxf(vmax, fred[w]);
            named_bar_sync(2, NGT);
            // probabilities are <= 2^tau, so P * v_scale * p_scale stays <= 448
            p_scale = vmax > 0.f ? pow2_floor(448.f / (exp2f(M::kTau) * vmax)) : 1.f;
          }
        }
        const int s = item % p.n_splits;
        const int tg = item / p.n_splits;
        const int g = tg % p.n_groups;
        const int t = tg / p.n_groups;
        (void)s;
        float q_scale = 1.f;
        const int n_tiles = (n + 127) >> 7;
        // Q of this token and head group, loaded by the first 128 gather threads.  Every item takes
        // one turn of the buffer, also one without columns.  The first item's bf16 q is loaded by
        // the softmax warps at kernel start, while the resolver walks the first page tables.
        if (!kFp8 && item == (int)blockIdx.x) {
          q_ph ^= 1;
        } else if (ptid < 128) {
          mbar_wait(BAR(B_QEMPTY), q_ph ^ 1, abort_flag);
          q_ph ^= 1;
          if (n == 0) {
            mbar_arrive(BAR(B_QFULL));
          } else if (!kFp8) {
            const uint32_t qs = sb + kQOff;
            // bf16: [atom][64 heads][128 B], heads beyond H zero-filled
            for (int it = 0; it < 4 * n_atoms; ++it) {
              const int h = (it & 3) * 16 + r0;
              const int a = it >> 2;
              const int hg = g * p.gh + h;
              const bool ok = h < p.gh && hg < p.H;
              const uint8_t* src = p.q + (((size_t)t * p.H + (ok ? hg : 0)) * D) * 2 + a * 128 + jj * 16;
              cp_async_16(qs + a * M::kQAtom + h * 128 + ((jj ^ (h & 7)) << 4), src, ok ? 16u : 0u);
            }
            cp_async_arrive_noinc(BAR(B_QFULL));
          } else {
            // e4m3: rows 0..63 hold q_hi, rows 64..127 q_lo, both times a power of two per token
            float qm = 0.f;
            for (int pass = 0; pass < 2; ++pass) {
              if (pass == 1) {
                qm = warp_max(qm);
                if (lane == 0) fred[pw] = qm;
                named_bar_sync(3, 128);   // (barrier 3: the first 128 gather threads)
                qm = fmaxf(fmaxf(fred[0], fred[1]), fmaxf(fred[2], fred[3]));
                named_bar_sync(3, 128);
                q_scale = qm > 0.f ? pow2_floor(448.f / qm) : 1.f;
              }
              // four pieces per round, their eight 16-byte loads in flight together
              for (int it0 = 0; it0 < 4 * n_atoms; it0 += 4) {
                uint4 u[4][2];
#pragma unroll
                for (int b4 = 0; b4 < 4; ++b4) {
                  const int it = it0 + b4;
                  const int h = (it & 3) * 16 + r0;
                  const int piece = (it >> 2) * 8 + jj;   // 16 head_dim values
                  const int hg = g * p.gh + h;
                  const bool ok = h < p.gh && hg < p.H && piece < P16;
                  u[b4][0] = u[b4][1] = make_uint4(0, 0, 0, 0);
                  if (ok) {
                    const uint4* src = reinterpret_cast<const uint4*>(
                        p.q + (((size_t)t * p.H + hg) * D + piece * 16) * 2);
                    u[b4][0] = __ldg(src);
                    u[b4][1] = __ldg(src + 1);
                  }
                }
#pragma unroll
                for (int b4 = 0; b4 < 4; ++b4) {
                  const int it = it0 + b4;
                  const int h = (it & 3) * 16 + r0;
                  const int a = it >> 2;
                  const uint32_t w[8] = {u[b4][0].x, u[b4][0].y, u[b4][0].z, u[b4][0].w,
                                         u[b4][1].x, u[b4][1].y, u[b4][1].z, u[b4][1].w};
                  if (pass == 0) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                      qm = fmaxf(qm, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
                  } else {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                      uint32_t h0, l0, h1, l1;
                      split_e4m3x2(bf16_lo(w[2 * k]) * q_scale, bf16_hi(w[2 * k]) * q_scale, h0, l0);
                      split_e4m3x2(bf16_lo(w[2 * k + 1]) * q_scale, bf16_hi(w[2 * k + 1]) * q_scale, h1, l1);
                      hi[k] = h0 | (h1 << 16);
                      lo[k] = l0 | (l1 << 16);
                    }
                    uint8_t* qrow = sm + kQOff + a * M::kQAtom;
                    *reinterpret_cast<uint4*>(qrow + h * 128 + ((jj ^ (h & 7)) << 4)) =
                        make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(qrow + (64 + h) * 128 + ((jj ^ (h & 7)) << 4)) =
                        make_uint4(lo[0], lo[1], lo[2], lo[3]);
                  }
                }
              }
            }
            fence_proxy_async_smem();
            mbar_arrive(BAR(B_QFULL));
          }
        }
        // Fill order of the ring: K0, K1, V0, K2, V1, ..., K(m-1), V(m-2), V(m-1): the MMA computes
        // S(j+1) before PV(j), so the next tile's K is copied while the softmax works on this one.
        // A single tile of at most 64 columns is packed: K in rows 0..63 and V in rows 64..127 of
        // the same slots (the S MMA's rows past 63 are masked columns).
        const bool packed = n_tiles == 1 && n <= 64;
        const int n_steps = n == 0 ? 0 : (packed ? 1 : 2 * n_tiles);
        const uint8_t* sc[8];   // rows of the newest tile whose K was copied
        const uint8_t* sv[8];   // rows of the tile before it
        int nj_c = 0, nj_v = 0;
        if (n == 0) {
          // no column: one tile-info entry tells the consumers
          if (ti_writer) mbar_wait(BAR(B_TIEMPTY + tik), ti_ph ^ 1, abort_flag);
          if (kFp8 && ptid < 128) {
            ti[tik].k_scale[ptid] = 0.f;
            ti[tik].v_scale[ptid] = 0.f;
            named_bar_sync(3, 128);
          }
          if (ptid == 0) {
            TileInfo& e = ti[tik];
            e.item = item;
            e.n = 0;
            e.flags = kFirst | kLast;
            e.q_scale = q_scale;
            e.p_scale = p_scale;
            mbar_arrive(BAR(B_TIFULL + tik));
          }
          if (++tik == kTi) { tik = 0; ti_ph ^= 1; }
        }
        for (int st = 0; st < n_steps; ++st) {
          // step -> (tile, K or V)
          int j, half;
          if (st == 0) { j = 0; half = 0; }
          else if (st == n_steps - 1) { j = n_tiles - 1; half = 1; }
          else if (st & 1) { j = (st + 1) >> 1; half = 0; }
          else { j = (st >> 1) - 1; half = 1; }
          if (half == 0) {
            // publish tile j to the MMA and softmax warps.  Only threads that write the entry
            // wait for it to be free, and all of them have seen it free before it is published:
            // a thread that waited without taking part could look only after the consumers had
            // freed the entry's next use too, and then wait on a parity that never comes back.
            if (ti_writer) mbar_wait(BAR(B_TIEMPTY + tik), ti_ph ^ 1, abort_flag);
            if (kFp8 && ptid < 128) {
              const int idx = j * 128 + ptid;
              const int32_t code = idx < n ? list[list_pos(idx, tma)] : -1;
              float ks = 0.f, vs = 0.f;
              if (code >= 0) {
                const bool cmp = code >> kColPoolShift;
                const int row = code & ((1 << kColPoolShift) - 1);
                ks = __ldg((cmp ? p.rs.cmp.k_scale : p.rs.win.k_scale) + row);
                vs = __ldg((cmp ? p.rs.cmp.v_scale : p.rs.win.v_scale) + row);
              }
              ti[tik].k_scale[ptid] = ks;
              ti[tik].v_scale[ptid] = vs;
              named_bar_sync(3, 128);
            }
            if (ptid == 0) {
              TileInfo& e = ti[tik];
              e.item = item;
              e.n = min(128, n - j * 128);
              e.flags = (j == 0 ? kFirst : 0) | (j == n_tiles - 1 ? kLast : 0);
              e.q_scale = q_scale;
              e.p_scale = p_scale;
              mbar_arrive(BAR(B_TIFULL + tik));
            }
            if (++tik == kTi) { tik = 0; ti_ph ^= 1; }
            if (!tma && ptid < 128) {
              // the 8 rows of tile j that this thread copies (columns j*128 + 16k + r0, stored
              // consecutively)
              const int4 lw0 = *reinterpret_cast<const int4*>(list + j * 128 + r0 * 8);
              const int4 lw1 = *reinterpret_cast<const int4*>(list + j * 128 + r0 * 8 + 4);
              const int32_t lc[8] = {lw0.x, lw0.y, lw0.z, lw0.w, lw1.x, lw1.y, lw1.z, lw1.w};
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                sv[k] = sc[k];
                const int idx = j * 128 + k * 16 + r0;
                const int32_t code = idx < n ? lc[k] : -1;
                if (code < 0) {
                  sc[k] = nullptr;
                } else {
                  const uint8_t* base = (code >> kColPoolShift) ? p.rs.cmp.kv : p.rs.win.kv;
                  sc[k] = base + (size_t)(code & ((1 << kColPoolShift) - 1)) * row_bytes;
                }
              }
            }
            nj_v = nj_c;
            nj_c = min(128, n - j * 128);
          }
          // V of the newest tile only at the very last step; otherwise V of the tile before it
          const bool cur = half == 0 || st == n_steps - 1;
          const int nj = cur ? nj_c : nj_v;
          // Rows the MMAs read: the S MMA masks columns >= nj in the softmax, so K rows past nj
          // may hold anything; the PV MMA reads V rows up to its K-step multiple, which must be
          // finite past nj (zero probability times a stale NaN would still be NaN).
          const int pv_step = kFp8 ? 32 : 16;
          const int v_rows = (nj + pv_step - 1) / pv_step * pv_step;
          if (tma) {
            // Four rows per copy: K row groups over [0, nj) (the last one may repeat its first
            // row), V row groups over [0, v_rows) (rows past nj repeat a row of the tile: finite
            // values that meet zero probabilities).  A packed tile takes both, V at row 64.
            // The gather warps work in pairs, fill f to pair f % (NG / 2), each of the two warps
            // issuing up to 32 copies (one instruction) and arming the slot's barrier with their
            // bytes: copies spread thinly over all warps issue far slower than full-warp batches.
            const int32_t* tl = list + j * 128;
            const int gk = half == 0 ? (nj + 3) >> 2 : 0;
            const int gv = (half == 1 || packed) ? v_rows >> 2 : 0;
            const int vrow0 = packed ? 64 : 0;
            constexpr int rmask = (1 << kColPoolShift) - 1;
            constexpr int kFillWarps = kTmaFillWarps;
            for (int kc = 0; kc < n_chunks; ++kc) {
              if (pw / kFillWarps == fills % (NG / kFillWarps)) {
                const int na = min(2, n_atoms - 2 * kc);
                const int ops = (gk + gv) * na;
                const int per = (ops + kFillWarps - 1) / kFillWarps;
                const int o0 = (pw % kFillWarps) * per;
                const int mine = max(0, min(per, ops - o0));
                bool okw = true;
                if (lane == 0) okw = mbar_wait(BAR(B_EMPTY + ring), ring_ph ^ 1, abort_flag);
                okw = __shfl_sync(0xffffffffu, okw, 0);
                const uint32_t full = BAR(B_FULL + ring);
                if (lane == 0) mbar_arrive_expect_tx(full, okw ? (uint32_t)mine * 512u : 0u);
                __syncwarp();
                if (okw && lane < mine) {
                  const int o = o0 + lane;
                  const int gi = o / na, aa = o - gi * na;
                  const bool isv = gi >= gk;
                  const int r = 4 * (isv ? gi - gk : gi);   // first tile row of the group
                  const int4 c4 = *reinterpret_cast<const int4*>(tl + r);
                  int32_t code[4] = {c4.x, c4.y, c4.z, c4.w};
                  const int32_t fill = r < nj ? code[0] : tl[0];
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    if (r + i >= nj) code[i] = fill;
                  const int pool = code[0] >> kColPoolShift;
                  bool same = true;
#pragma unroll
                  for (int i = 1; i < 4; ++i) same = same && (code[i] >> kColPoolShift) == pool;
                  const uint32_t dst = sb + kRingOff + ring * kSlotBytes + aa * kAtomBytes +
                                       (uint32_t)((isv ? vrow0 : 0) + r) * 128u;
                  const int x = (2 * kc + aa) * 128;
                  const int mv = isv ? 1 : 0;
                  if (same) {
                    tma_gather4(dst, &p.kv_map[2 * pool + mv], x, code[0] & rmask, code[1] & rmask,
                                code[2] & rmask, code[3] & rmask, full);
                  } else {  // the group where the window rows end and the compressed rows begin
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                      tma_row(dst + 128u * i, &p.kv_map[2 * (code[i] >> kColPoolShift) + mv], x,
                              code[i] & rmask, full);
                  }
                }
              }
              if (++ring == kStages) { ring = 0; ring_ph ^= 1; }
              ++fills;
            }
            continue;
          }
          // Row groups of 16 past the rows the MMAs read are skipped with a warp-uniform test;
          // V rows past nj are zero-filled.
          const int kmax = ((half == 0 ? nj : v_rows) + 15) >> 4;
          const int kmax_v = packed ? (v_rows + 15) >> 4 : 0;
          const uint8_t* sr[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) sr[k] = cur ? sc[k] : sv[k];
          for (int kc = 0; kc < n_chunks; ++kc) {
            if (ptid < 128) {   // cp.async copies: the first 128 gather threads
              mbar_wait(BAR(B_EMPTY + ring), ring_ph ^ 1, abort_flag);
              const uint32_t d0 = sb + kRingOff + ring * kSlotBytes + dst_thread;
              const bool a0 = (2 * kc) * 8 + jj < P16, a1 = (2 * kc + 1) * 8 + jj < P16;
              const size_t so = (size_t)half * D * M::kElt + (size_t)(2 * kc) * 128 + jj * 16;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (k < kmax) {
                  const uint8_t* sp = sr[k] ? sr[k] + so : p.q;
                  const uint32_t sz = sr[k] ? 16u : 0u;
                  if (a0) cp_async_16(d0 + k * 2048, sp, sz);
                  if (a1) cp_async_16(d0 + kAtomBytes + k * 2048, sp + 128, sz);
                }
              }
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                if (k < kmax_v) {
                  const uint8_t* sp = sr[k] ? sr[k] + so + D * M::kElt : p.q;
                  const uint32_t sz = sr[k] ? 16u : 0u;
                  if (a0) cp_async_16(d0 + (4 + k) * 2048, sp, sz);
                  if (a1) cp_async_16(d0 + kAtomBytes + (4 + k) * 2048, sp + 128, sz);
                }
              }
              cp_async_arrive_noinc(BAR(B_FULL + ring));
            }
            if (++ring == kStages) { ring = 0; ring_ph ^= 1; }
            ++fills;
          }
        }
        // this warp is done with the item's list
        if (kRes) {
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_LEMPTY + lb));
        }
      }
      // end-of-work marker for the consumers
      if (!*abort_flag && ptid == 0) {
        mbar_wait(BAR(B_TIEMPTY + tik), ti_ph ^ 1, abort_flag);
        ti[tik].item = -1;
        ti[tik].n = 0;
        ti[tik].flags = kFirst | kLast;
        mbar_arrive(BAR(B_TIFULL + tik));
      }
      cp_async_wait_all();
      if (tma && lane == 0) {
        // Tensor-map copies land asynchronously: before this CTA can end, the last fill of every
        // slot must have completed (at once after a normal run, whose MMAs consumed them all; an
        // aborted run may wait out the drain limit).  Fill f went to slot f % 4, barrier phase f / 4.
        for (int sl = 0; sl < kStages && sl < fills; ++sl) {
          const int f = fills - 1 - ((fills - 1 - sl) % kStages);
          mbar_wait_drain(BAR(B_FULL + sl), (uint32_t)((f / kStages) & 1));
        }
      }
    } else if (warp == 4) {
      // ====================================== MMA ========================================
      if (lane == 0) {
        // S: A = K rows (K-major), B = q rows (K-major).  O: A = V^T (MN-major), B = P^T (MN-major)
        const uint32_t idS = kFp8 ? idesc_e4m3(128, 128, 0, 0) : idesc_bf16(128, 64, 0, 0);
        const uint32_t idO = kFp8 ? idesc_e4m3(128, 64, 1, 1) : idesc_bf16(128, 64, 1, 1);
        const uint32_t qbase = sb + kQOff, pbase = sb + kPOff;
        int ring = 0, tik = 0, sbuf = 0;
        uint32_t ring_ph = 0, ti_ph = 0, q_ph = 0, s_ph = 0, p_ph = 0, o_ph = 0;
        // S of a tile: A = K rows from the ring (K-major), B = q (K-major), into S buffer sbuf.
        // Releases the K slots unless the tile is packed (V still to be read from them).
        auto issue_s = [&](bool packed) -> bool {
          if (!mbar_wait(BAR(B_SEMPTY + sbuf), ((s_ph >> sbuf) & 1u) ^ 1u, abort_flag)) return false;
          s_ph ^= 1u << sbuf;
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t dS = tmem + sbuf * M::kSCols;
          const uint64_t dq0 = sdesc(qbase, 16, 1024);
          for (int kc = 0; kc < n_chunks; ++kc) {
            if (!mbar_wait(BAR(B_FULL + ring), ring_ph, abort_flag)) return false;
            fence_proxy_async_smem();
            tc_fence_after();
            const uint64_t dk0 = sdesc(sb + kRingOff + ring * kSlotBytes, 16, 1024);
            for (int aa = 0; aa < 2; ++aa) {
              const int atom = 2 * kc + aa;
              if (atom >= n_atoms) break;
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                if (atom * 4 + ks >= n_ks) break;
                const uint64_t da = desc_add(dk0, aa * kAtomBytes + ks * 32);
                const uint64_t db = desc_add(dq0, atom * M::kQAtom + ks * 32);
                if (kFp8)
                  mma_f8(dS, da, db, idS, (kc | aa | ks) != 0);
                else
                  mma_bf16(dS, da, db, idS, (kc | aa | ks) != 0);
              }
            }
            if (!packed) mma_commit(BAR(B_EMPTY + ring));
            if (++ring == kStages) { ring = 0; ring_ph ^= 1; }
          }
          mma_commit(BAR(B_SFULL + sbuf));
          sbuf ^= 1;
          return true;
        };
        // PV of a tile of n columns: A = V^T from the ring (MN-major), B = P^T (MN-major).
        auto issue_pv = [&](int n, bool first, bool packed) -> bool {
          if (!mbar_wait(BAR(B_PFULL), p_ph, abort_flag)) return false;
          p_ph ^= 1;
          if (first) {
            if (!mbar_wait(BAR(B_OFREE), o_ph ^ 1, abort_flag)) return false;
            o_ph ^= 1;
          }
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t v_off = packed ? 64u * 128u : 0u;
          if (!kFp8 && packed) {
            // A packed tile's slots were waited for by its S just before: issue the MMAs of all
            // head_dim tiles back to back (interleaved, no per-slot wait), then release the slots.
            const int nk = (n + 15) >> 4;
            const uint64_t dp0 = sdesc(pbase, kAtomBytes, 1024);
            const uint64_t dv0 = sdesc(sb + kRingOff + v_off, kAtomBytes, 1024);
            for (int kk = 0; kk < nk; ++kk) {
              const uint64_t db = desc_add(dp0, kk * 2048);
              int r = ring;
              for (int vc = 0; vc < n_chunks; ++vc) {
                const uint64_t da = desc_add(dv0, r * kSlotBytes + kk * 2048);
                mma_bf16(tmem + M::kOCol + vc * 64, da, db, idO, (first && kk == 0) ? 0u : 1u);
                if (++r == kStages) r = 0;
              }
            }
            for (int vc = 0; vc < n_chunks; ++vc) {
              mma_commit(BAR(B_EMPTY + ring));
              if (++ring == kStages) { ring = 0; ring_ph ^= 1; }
            }
            mma_commit(BAR(B_PVDONE));
            return true;
          }
          for (int vc = 0; vc < n_chunks; ++vc) {
            if (!mbar_wait(BAR(B_FULL + ring), ring_ph, abort_flag)) return false;
            fence_proxy_async_smem();
            tc_fence_after();
            const uint32_t slot = sb + kRingOff + ring * kSlotBytes;
            if (!kFp8) {
              // one 128-wide head_dim tile per slot (two 64-wide atoms, LBO apart); K = 16 columns
              const uint32_t dO = tmem + M::kOCol + vc * 64;
              const int nk = (n + 15) >> 4;
              const uint64_t dv0 = sdesc(slot + v_off, kAtomBytes, 1024);
              const uint64_t dp0 = sdesc(pbase, kAtomBytes, 1024);
              for (int kk = 0; kk < nk; ++kk) {
                const uint64_t da = desc_add(dv0, kk * 2048);
                const uint64_t db = desc_add(dp0, kk * 2048);
                mma_bf16(dO, da, db, idO, (first && kk == 0) ? 0u : 1u);
              }
            } else {
              // two 128-wide head_dim tiles per slot (one atom each); K = 32 columns; P^T is
              // p_hi (64-byte rows, 64-byte swizzle) followed by p_lo, both into the same O
              const int nk = (n + 31) >> 5;
              const uint64_t dv0 = sdesc(slot + v_off, kAtomBytes, 1024);
              const uint64_t dp0 = sdesc64(pbase, 8192, 512);
              for (int aa = 0; aa < 2; ++aa) {
                const int mt = 2 * vc + aa;
                if (mt >= n_mt) break;
                const uint32_t dO = tmem + M::kOCol + mt * 64;
                for (int kk = 0; kk < nk; ++kk) {
                  const uint64_t da = desc_add(dv0, aa * kAtomBytes + kk * 4096);
                  const uint64_t dh = desc_add(dp0, kk * 2048);
                  const uint64_t dl = desc_add(dp0, 8192 + kk * 2048);
                  mma_f8(dO, da, dh, idO, (first && kk == 0) ? 0u : 1u);
                  mma_f8(dO, da, dl, idO, 1u);
                }
              }
            }
            mma_commit(BAR(B_EMPTY + ring));
            if (++ring == kStages) { ring = 0; ring_ph ^= 1; }
          }
          mma_commit(BAR(B_PVDONE));
          return true;
        };
        // Per item: S(0); then for every tile j: S(j + 1) (if any), PV(j).  The tile-info entry of
        // the next tile is read before PV of the current one.
        bool ok = true;
        for (;;) {
          if (!mbar_wait(BAR(B_TIFULL + tik), ti_ph, abort_flag)) break;
          int n = ti[tik].n;
          const int item = ti[tik].item;
          int flags = ti[tik].flags;
          mbar_arrive(BAR(B_TIEMPTY + tik));
          if (++tik == kTi) { tik = 0; ti_ph ^= 1; }
          if (item < 0) break;
          if (!mbar_wait(BAR(B_QFULL), q_ph, abort_flag)) break;   // (every item begins a tile 0)
          q_ph ^= 1;
          if (n == 0) {  // an item without columns: hand the Q buffer back untouched
            mma_commit(BAR(B_QEMPTY));
            continue;
          }
          const bool packed = (flags & kLast) && n <= 64;   // a single packed tile
          const int ring0 = ring;
          const uint32_t ring_ph0 = ring_ph;
          if (!(ok = issue_s(packed))) break;
          if (flags & kLast) mma_commit(BAR(B_QEMPTY));
          bool first = true;
          for (;;) {
            const bool last = flags & kLast;
            int n_next = 0, flags_next = 0;
            if (!last) {
              if (!(ok = mbar_wait(BAR(B_TIFULL + tik), ti_ph, abort_flag))) break;
              n_next = ti[tik].n;
              flags_next = ti[tik].flags;
              mbar_arrive(BAR(B_TIEMPTY + tik));
              if (++tik == kTi) { tik = 0; ti_ph ^= 1; }
              if (!(ok = issue_s(false))) break;
              if (flags_next & kLast) mma_commit(BAR(B_QEMPTY));
            }
            if (packed) {  // PV reads the slots S just read
              ring = ring0;
              ring_ph = ring_ph0;
            }
            if (!(ok = issue_pv(n, first, packed))) break;
            first = false;
            if (last) break;
            n = n_next;
            flags = flags_next;
          }
          if (!ok) break;
        }
        // nothing may still write TMEM when it is released
        mma_commit(BAR(B_DRAIN));
        mbar_wait_drain(BAR(B_DRAIN), 0);
      }
      __syncwarp();
    }
  } else {
    // ================================ softmax / epilogue ================================
    const int tid = threadIdx.x;  // column of the tile == TMEM lane
    float* red = reinterpret_cast<float*>(sm + kRedOff);
    float* mrow = reinterpret_cast<float*>(sm + kMrowOff) + warp * 64;
    float* arow = reinterpret_cast<float*>(sm + kArowOff) + warp * 64;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    int tik = 0, sbuf = 0, rb = 0;
    uint32_t ti_ph = 0, s_ph = 0, pv_ph = 0, red_ph = 0;
    // running max (base-2 units) and this warp's partial denominator of heads lane, 32 + lane
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float p_scale = 1.f;
    int t = 0, g = 0, s = 0;
    bool had = false;
    if (!kFp8) {
      // q of this CTA's first item (bf16: [atom][64 heads][128 B], heads beyond H zero-filled),
      // loaded here while the gather warps walk the page tables; the buffer starts out free
      const int tg0 = (int)blockIdx.x / p.n_splits;
      const int g0 = tg0 % p.n_groups, t0 = tg0 / p.n_groups;
      const int jq = tid & 7, rq = tid >> 3;
      const uint32_t qs = sb + kQOff;
      for (int it = 0; it < 4 * n_atoms; ++it) {
        const int h = (it & 3) * 16 + rq;
        const int a = it >> 2;
        const int hg = g0 * p.gh + h;
        const bool okq = h < p.gh && hg < p.H;
        const uint8_t* src = p.q + (((size_t)t0 * p.H + (okq ? hg : 0)) * D) * 2 + a * 128 + jq * 16;
        cp_async_16(qs + a * M::kQAtom + h * 128 + ((jq ^ (h & 7)) << 4), src, okq ? 16u : 0u);
      }
      cp_async_arrive_noinc(BAR(B_QFULL));
    }
    for (;;) {
      if (!warp_wait(BAR(B_TIFULL + tik), ti_ph, abort_flag)) break;
      const int item = ti[tik].item;
      const int n = ti[tik].n;
      const int flags = ti[tik].flags;
      float col_scale = sl2, v_fold = 0.f;
      if (kFp8) {
        col_scale = sl2 * ti[tik].k_scale[tid] / ti[tik].q_scale;
        p_scale = ti[tik].p_scale;
        v_fold = ti[tik].v_scale[tid] * p_scale;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_TIEMPTY + tik));
      if (++tik == kTi) { tik = 0; ti_ph ^= 1; }
      if (item < 0) break;
      const bool first = flags & kFirst, last = flags & kLast;
      if (first) {
        s = item % p.n_splits;
        const int tg = item / p.n_splits;
        g = tg % p.n_groups;
        t = tg / p.n_groups;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
        had = false;
      }
      if (n > 0) {
        had = true;
        if (!warp_wait(BAR(B_SFULL + sbuf), (s_ph >> sbuf) & 1u, abort_flag)) break;
        s_ph ^= 1u << sbuf;
        tc_fence_after();
        const bool valid = tid < n;
        const uint32_t s_addr = lane_base + sbuf * M::kSCols;
        float* rr = red + rb * 256;
        // pass 1: tile maximum of every head (lane L ends up with heads L and 32 + L)
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          float x[32];
          tmem_ld32(s_addr + hf * 32, x);
          if (kFp8) {
            float y[32];
            tmem_ld32(s_addr + 64 + hf * 32, y);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) x[k] += y[k];
          } else {
            tmem_wait_ld();
          }
#pragma unroll
          for (int k = 0; k < 32; ++k) x[k] = valid ? x[k] * col_scale : -INFINITY;
          rr[warp * 64 + hf * 32 + lane] = xreduce32<true>(x, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_RED + rb));
        if (!warp_wait(BAR(B_RED + rb), (red_ph >> rb) & 1u, abort_flag)) break;
        red_ph ^= 1u << rb;
        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          M0 = fmaxf(M0, rr[w * 64 + lane]);
          M1 = fmaxf(M1, rr[w * 64 + 32 + lane]);
        }
        rb ^= 1;
        const float n0 = (M0 > m0 + M::kTau) ? M0 : m0;
        const float n1 = (M1 > m1 + M::kTau) ? M1 : m1;
        const float a0 = fast_exp2(m0 - n0), a1 = fast_exp2(m1 - n1);
        const bool grow = __any_sync(0xffffffffu, (n0 != m0) || (n1 != m1));
        m0 = n0;
        m1 = n1;
        mrow[lane] = n0;
        mrow[32 + lane] = n1;
        arow[lane] = a0;
        arow[32 + lane] = a1;
        __syncwarp();
        l0 *= a0;
        l1 *= a1;
        // pass 2: this column's probabilities and this warp's denominators.  P^T of the column
        // (bf16: 64 heads x 2 B; e4m3: the hi then the lo codes of 2 x 16 heads per head half) is
        // parked as 32 words in the TMEM columns of this S buffer that the thread has just read
        // (half 0 reads columns 0..31 and parks in 0..15, half 1 reads 32..63 and parks in
        // 16..31; e4m3's lo half of S, 64..127, is read before either).  So the work of pass 2
        // overlaps PV of the tile before, which still reads the one P buffer in shared memory.
        // (Parking the first tile of an item too, which has no PV to wait for, measured faster
        // than storing it straight away.)
        // (Chunk k of the P^T row: bf16 heads 8k .. 8k+7 at position k ^ (column & 7); e4m3 heads
        // 16k .. 16k+15 of p_hi, and of p_lo 8 KB on, at position k ^ ((column >> 1) & 3).)
        uint8_t* const prow = sm + kPOff + tid * (kFp8 ? 64 : 128);
        const auto store_chunk = [&](int k, const uint32_t* w) {
          if (!kFp8) {
            *reinterpret_cast<uint4*>(prow + ((k ^ (tid & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          } else {
            const int off = (k ^ ((tid >> 1) & 3)) << 4;
            *reinterpret_cast<uint4*>(prow + off) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(prow + 8192 + off) = make_uint4(w[8], w[9], w[10], w[11]);
          }
        };
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          float x[32];
          tmem_ld32(s_addr + hf * 32, x);
          if (kFp8) {
            float y[32];
            tmem_ld32(s_addr + 64 + hf * 32, y);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) x[k] += y[k];
          } else {
            tmem_wait_ld();
          }
#pragma unroll
          for (int k = 0; k < 32; ++k)
            x[k] = valid ? fast_exp2(x[k] * col_scale - mrow[hf * 32 + k]) : 0.f;
          uint32_t pw[16];
          if (!kFp8) {
#pragma unroll
            for (int k = 0; k < 16; ++k) pw[k] = pack_bf16x2(x[2 * k], x[2 * k + 1]);
          } else {
            // P * v_scale * p_scale as p_hi + p_lo (e4m3): words 0..7 hi, 8..15 lo
#pragma unroll
            for (int w = 0; w < 8; ++w) {
              uint32_t h0, l0v, h1, l1v;
              split_e4m3x2(x[4 * w + 0] * v_fold, x[4 * w + 1] * v_fold, h0, l0v);
              split_e4m3x2(x[4 * w + 2] * v_fold, x[4 * w + 3] * v_fold, h1, l1v);
              pw[w] = h0 | (h1 << 16);
              pw[8 + w] = l0v | (l1v << 16);
            }
          }
          tmem_st16(s_addr + hf * 16, pw);
          const float ts = xreduce32<false>(x, lane);
          if (hf == 0) l0 += ts; else l1 += ts;
        }
        tmem_wait_st();
        if (!first) {
          // wait for PV of the tile before (the MMA warp issues S of a tile before PV of the
          // one before it): then O can be rescaled and the P buffer reused
          if (!warp_wait(BAR(B_PVDONE), pv_ph, abort_flag)) break;
          pv_ph ^= 1;
          tc_fence_after();
        }
        if (grow && !first) {
          // the running max moved: rescale O
          for (int i = 0; i < n_mt; ++i) {
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
              float o[32];
              const uint32_t ta = lane_base + M::kOCol + i * 64 + hf * 32;
              tmem_ld32(ta, o);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] *= arow[hf * 32 + k];
              tmem_st32(ta, o);
            }
          }
          tmem_wait_st();
        }
        {
          // the parked P^T row into the P buffer
          float pf[32];
          tmem_ld32(s_addr, pf);
          tmem_wait_ld();
          uint32_t pw[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) pw[k] = __float_as_uint(pf[k]);
          if (!kFp8) {
#pragma unroll
            for (int k = 0; k < 8; ++k) store_chunk(k, pw + 4 * k);
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) store_chunk(k, pw + (k >> 1) * 16 + (k & 1) * 4);
          }
        }
        tc_fence_before();
        mbar_arrive(BAR(B_SEMPTY + sbuf));
        sbuf ^= 1;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(BAR(B_PFULL));
      }
      if (last && clustered) {
        // ---- split-K merge inside the cluster (one item per CTA; rank == split index) ----
        // Every CTA sends CTA k its (m, l) per head and the rows [k*dpo, (k+1)*dpo) of its
        // unnormalised O^T in bf16; CTA k weights split s by 2^(m_s - M) / sum_j 2^(m_j - M) l_j
        // and stores the sum.  Transfers are bulk copies between the shared memories of the
        // cluster; the (m, l) copies go first so the weights are ready when the rows land.
        // No early exit until the last named barrier: all four softmax warps must reach each of
        // them; a failed wait (which sets the abort flag) only skips work.
        const int S = p.cluster;
        const int dpo = D / S;
        float L0 = 0.f, L1 = 0.f;
        bool ok = true;
        if (had) {
          ok = warp_wait(BAR(B_PVDONE), pv_ph, abort_flag);
          pv_ph ^= 1;
          tc_fence_after();
          float* rr = red + rb * 256;
          rr[warp * 64 + lane] = l0;
          rr[warp * 64 + 32 + lane] = l1;
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_RED + rb));
          ok = ok && warp_wait(BAR(B_RED + rb), (red_ph >> rb) & 1u, abort_flag);
          red_ph ^= 1u << rb;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            L0 += rr[w * 64 + lane];
            L1 += rr[w * 64 + 32 + lane];
          }
          rb ^= 1;
        }
        cluster_wait();
        cl_started = true;
        const uint32_t rank = cluster_ctarank();
        // this CTA's ring is idle from here on: tell every CTA of the cluster
        if (ok && tid < S) mbar_arrive_cluster(mapa_cluster(BAR(B_READY), (uint32_t)tid));
        // (m - log2 p, l * p) per head: O carries the probability scale p (e4m3; 1 for bf16)
        // and l does not, so 2^(m' - M') = 2^(m - M') / p while 2^(m' - M') l' is unchanged
        const int gh = p.gh;
        const int rb_bytes = gh * 2;          // one staged O^T row: gh bf16 heads
        const int cpr = gh >> 3;              // 16-byte chunks per row
        const int ml_bytes = gh * 8;
        if (warp == 0) {
          const float lp = __log2f(p_scale);
          float2* mlo = reinterpret_cast<float2*>(sm + kPOff);
          if (lane < gh) mlo[lane] = make_float2(had ? m0 - lp : -INFINITY, L0 * p_scale);
          if (32 + lane < gh) mlo[32 + lane] = make_float2(had ? m1 - lp : -INFINITY, L1 * p_scale);
        }
        // stage O^T as bf16 [D rows][gh heads] in the Q buffer (zeros for a split without
        // columns, whose TMEM was never written), chunk c of row d at position c ^ (d & (cpr-1))
#pragma unroll 1
        for (int i = 0; i < n_mt; ++i) {
          const int d = i * 128 + tid;
#pragma unroll 1
          for (int hf = 0; hf < (gh >> 5); ++hf) {
            float o[32];
            if (had) {
              tmem_ld32(lane_base + M::kOCol + i * 64 + hf * 32, o);
              tmem_wait_ld();
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = 0.f;
            }
            if (d < D) {
              uint8_t* row = sm + kQOff + (size_t)d * rb_bytes;
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                uint4 u;
                u.x = pack_bf16x2(o[8 * q4 + 0], o[8 * q4 + 1]);
                u.y = pack_bf16x2(o[8 * q4 + 2], o[8 * q4 + 3]);
                u.z = pack_bf16x2(o[8 * q4 + 4], o[8 * q4 + 5]);
                u.w = pack_bf16x2(o[8 * q4 + 6], o[8 * q4 + 7]);
                *reinterpret_cast<uint4*>(row + (((hf * 4 + q4) ^ (d & (cpr - 1))) << 4)) = u;
              }
            }
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        // lane l of warp w sends to CTA k = 4l + w: first its (m, l) block, then its row slice,
        // so the small copies are not queued behind the large ones.  A warp's copies issue one
        // after the other, so the sends are spread over the four warps.
        const uint32_t recv_ml = sb + kRingOff + (uint32_t)(D * rb_bytes);
        const bool send = ok && __shfl_sync(0xffffffffu, *abort_flag == 0 ? 1 : 0, 0) != 0;
        const int k_to = 4 * lane + warp;
        const int senders = warp < S ? (S - warp + 3) >> 2 : 0;   // lanes of this warp that send
        if (k_to < S && send) {   // (the same lanes on both sides of the warp sync)
          const uint32_t k = (uint32_t)k_to;
          const bool go = mbar_wait_cluster(BAR(B_READY), 0, abort_flag);
          if (go)
            bulk_copy_cluster(mapa_cluster(recv_ml + rank * ml_bytes, k), sb + kPOff, ml_bytes,
                              mapa_cluster(BAR(B_RECVML), k));
          __syncwarp((1u << senders) - 1u);
          if (go)
            bulk_copy_cluster(mapa_cluster(sb + kRingOff + rank * dpo * rb_bytes, k),
                              sb + kQOff + (uint32_t)(k * dpo * rb_bytes), dpo * rb_bytes,
                              mapa_cluster(BAR(B_RECV), k));
        }
        // merge weights per (split, head), computed while the rows are in flight
        ok = ok && warp_wait(BAR(B_RECVML), 0, abort_flag);
        const float2* mlr = reinterpret_cast<const float2*>(sm + kRingOff + D * rb_bytes);
        float* wk = reinterpret_cast<float*>(sm + kPOff + 1024);
        if (ok && tid < gh) {
          float m[16], l[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 v = k < S ? mlr[k * gh + tid] : make_float2(-INFINITY, 0.f);
            m[k] = v.x;
            l[k] = v.y;
          }
          float Mh = -INFINITY;
#pragma unroll
          for (int k = 0; k < 16; ++k) Mh = fmaxf(Mh, m[k]);
          float tot = 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            m[k] = (m[k] != -INFINITY) ? fast_exp2(m[k] - Mh) : 0.f;
            tot += m[k] * l[k];
          }
          const float it = tot > 0.f ? 1.f / tot : 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (k < S) wk[k * 64 + tid] = m[k] * it;
        }
        ok = ok && warp_wait(BAR(B_RECV), 0, abort_flag);
        if (ok && tid == 0) recv_ok = true;
        named_bar_sync(1, 128);
        if (!ok || *abort_flag) break;
        {
          // out rows [rank*dpo, (rank+1)*dpo) of every head: sum_s w[s][h] * O_s[row][h]
          // (a split without columns sent zeros with weight 0)
          const int Hg = min(gh, p.H - g * gh);
          const uint8_t* rv = sm + kRingOff;
          __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(p.out) +
                              ((size_t)t * p.H + g * gh) * D + rank * dpo;
#pragma unroll 1
          for (int idx = tid; idx < dpo * cpr; idx += 128) {
            const int dl = idx % dpo, c = idx / dpo;   // row, chunk of 8 heads
            const int pos = (c ^ ((rank * dpo + dl) & (cpr - 1))) << 4;
            const uint8_t* src = rv + (size_t)dl * rb_bytes + pos;
            const float* wc = wk + 8 * c;
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 4
            for (int k = 0; k < S; ++k) {
              const uint4 u = *reinterpret_cast<const uint4*>(src + (size_t)k * dpo * rb_bytes);
              const float4 wa = *reinterpret_cast<const float4*>(wc + k * 64);
              const float4 wb = *reinterpret_cast<const float4*>(wc + k * 64 + 4);
              acc[0] = fmaf(wa.x, bf16_lo(u.x), acc[0]);
              acc[1] = fmaf(wa.y, bf16_hi(u.x), acc[1]);
              acc[2] = fmaf(wa.z, bf16_lo(u.y), acc[2]);
              acc[3] = fmaf(wa.w, bf16_hi(u.y), acc[3]);
              acc[4] = fmaf(wb.x, bf16_lo(u.z), acc[4]);
              acc[5] = fmaf(wb.y, bf16_hi(u.z), acc[5]);
              acc[6] = fmaf(wb.z, bf16_lo(u.w), acc[6]);
              acc[7] = fmaf(wb.w, bf16_hi(u.w), acc[7]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (8 * c + e < Hg) ob[(size_t)(8 * c + e) * D + dl] = __float2bfloat16_rn(acc[e]);
          }
        }
        continue;
      }
      if (last) {
        const int Hg = min(p.gh, p.H - g * p.gh);
        if (!had) {
          // no column at all: out = 0 (prefill) or an empty partial (decode)
          if (p.decode) {
            const size_t pb = ((size_t)t * p.n_splits + s) * p.H + g * p.gh;
            for (int i = tid; i < Hg * D; i += 128) p.ws_o[pb * D + i] = 0.f;
            if (tid < Hg) p.ws_lse[pb + tid] = -INFINITY;
          } else {
            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + ((size_t)t * p.H + g * p.gh) * D;
            for (int i = tid; i < Hg * D; i += 128) o[i] = __float2bfloat16_rn(0.f);
          }
          continue;
        }
        if (!warp_wait(BAR(B_PVDONE), pv_ph, abort_flag)) break;
        pv_ph ^= 1;
        tc_fence_after();
        // softmax denominators per head
        float* rr = red + rb * 256;
        rr[warp * 64 + lane] = l0;
        rr[warp * 64 + 32 + lane] = l1;
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_RED + rb));
        if (!warp_wait(BAR(B_RED + rb), (red_ph >> rb) & 1u, abort_flag)) break;
        red_ph ^= 1u << rb;
        float L0 = 0.f, L1 = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          L0 += rr[w * 64 + lane];
          L1 += rr[w * 64 + 32 + lane];
        }
        rb ^= 1;
        arow[lane] = 1.f / (L0 * p_scale);
        arow[32 + lane] = 1.f / (L1 * p_scale);
        __syncwarp();
        if (p.decode && warp == 0) {
          const size_t pb = ((size_t)t * p.n_splits + s) * p.H + g * p.gh;
          if (lane < Hg) p.ws_lse[pb + lane] = m0 + __log2f(L0);
          if (32 + lane < Hg) p.ws_lse[pb + 32 + lane] = m1 + __log2f(L1);
        }
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          const float* inv = arow + hf * 32;   // 1 / denominator of each head of this half
          const size_t row0 = (size_t)t * p.H + g * p.gh + hf * 32;  // first head of this half
          const int nh = min(32, Hg - hf * 32);                     // heads of this half present
#pragma unroll 1
          for (int i = 0; i < n_mt; ++i) {
            const int d = i * 128 + tid;
            float o[32];
            tmem_ld32(lane_base + M::kOCol + i * 64 + hf * 32, o);
            tmem_wait_ld();
            if (d < D) {
              if (p.decode) {
                float* wo = p.ws_o + (((size_t)t * p.n_splits + s) * p.H + g * p.gh + hf * 32) * D + d;
#pragma unroll
                for (int k = 0; k < 32; ++k)
                  if (k < nh) wo[(uint32_t)(k * D)] = o[k] * inv[k];
              } else {
                // lanes 2m and 2m+1 swap halves so each stores two adjacent head_dim values
                const bool odd = lane & 1;
                __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(p.out) + row0 * D + (d & ~1);
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                  const float v0 = o[k] * inv[k], v1 = o[k + 1] * inv[k + 1];
                  const float recv = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
                  const __nv_bfloat162 pr = odd ? __floats2bfloat162_rn(recv, v1)
                                                : __floats2bfloat162_rn(v0, recv);
                  const int hh = k + (odd ? 1 : 0);
                  if (hh < nh) *reinterpret_cast<__nv_bfloat162*>(ob + (uint32_t)(hh * D)) = pr;
                }
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(BAR(B_OFREE));
      }
    }
  }
  if (clustered) {
    // no CTA leaves while a peer may still read or write its shared memory
    // (a relaxed arrival: this barrier orders no data, every copy between the CTAs was waited for)
    if (!cl_started) cluster_wait();
    cluster_arrive_relaxed();
    cluster_wait();
    // after a failed merge, copies from peers may still be landing here: let them finish
    if (threadIdx.x == 0 && !recv_ok) {
      mbar_wait_drain(BAR(B_RECVML), 0);
      mbar_wait_drain(BAR(B_RECV), 0);
    }
  }
#undef BAR
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Log-sum-exp merge of the split partials (base-2 LSE): out = sum_s 2^(lse_s - L) O_s / sum_s
// 2^(lse_s - L), L = max_s lse_s.  One block per (token, head); all partial loads of a thread are
// issued before any is used.
constexpr int kMergeMaxSplits = 32;

__global__ void __launch_bounds__(128) merge_kernel(const float* __restrict__ ws_o,
                                                    const float* __restrict__ ws_lse,
                                                    __nv_bfloat16* __restrict__ out, int S, int H,
                                                    int D) {
  __shared__ float w_s[kMergeMaxSplits];
  __shared__ float inv_sum;
  const int t = blockIdx.x / H, h = blockIdx.x % H;
  const float* lse = ws_lse + (size_t)t * S * H + h;
  if (threadIdx.x < 32) {
    const float l = threadIdx.x < S ? lse[(size_t)threadIdx.x * H] : -INFINITY;
    const float L = warp_max(l);
    const float w = (l == -INFINITY) ? 0.f : exp2f(l - L);
    float sum = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (threadIdx.x < S) w_s[threadIdx.x] = w;
    if (threadIdx.x == 0) inv_sum = sum > 0.f ? 1.f / sum : 0.f;
  }
  __syncthreads();
  const float inv = inv_sum;
  for (int d = threadIdx.x * 4; d < D; d += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 8) {     // eight partial loads in flight at a time
      float4 o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (s0 + k < S)
          o[k] = __ldg(reinterpret_cast<const float4*>(ws_o + (((size_t)t * S + s0 + k) * H + h) * D + d));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (s0 + k < S) {
          const float w = w_s[s0 + k];
          if (w != 0.f) {
            acc.x += w * o[k].x;
            acc.y += w * o[k].y;
            acc.z += w * o[k].z;
            acc.w += w * o[k].w;
          }
        }
      }
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + ((size_t)t * H + h) * D + d) = u;
  }
}

__global__ void resolve_dump_kernel(const ResolveArgs a, int32_t* __restrict__ cols) {
  const int C = a.W + a.K;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)a.T * C) return;
  const int t = (int)(i / C), c = (int)(i % C);
  bool ok;
  const int b = seq_of(a, t, &ok);
  cols[i] = ok ? resolve_column(a, t, b, __ldg(a.positions + t), c) : -1;
}

namespace {
// the kernel variants: rows by cp.async (one item per CTA, or e4m3 rows of a head_dim that is
// not a multiple of 128) or by tensor-map gathers, with or without the resolver warp
constexpr int kVariants = 7;
const void* attn_kernel_ptr(int v) {
  switch (v) {
    case 0: return reinterpret_cast<const void*>(attn_kernel<true, false, false>);
    case 1: return reinterpret_cast<const void*>(attn_kernel<true, true, false>);
    case 2: return reinterpret_cast<const void*>(attn_kernel<false, false, false>);
    case 3: return reinterpret_cast<const void*>(attn_kernel<false, false, true>);
    case 4: return reinterpret_cast<const void*>(attn_kernel<false, true, true>);
    case 5: return reinterpret_cast<const void*>(attn_kernel<true, false, true>);
    default: return reinterpret_cast<const void*>(attn_kernel<true, true, true>);
  }
}
int attn_variant(bool fp8, bool res, bool tma) {
  if (fp8) return tma ? (res ? 6 : 5) : (res ? 1 : 0);
  if (!tma) return 2;   // (bf16 by cp.async only for one item per CTA: no resolver)
  return res ? 4 : 3;
}
}  // namespace

cudaError_t prepare_attn_kernels() {
  for (int f = 0; f < kVariants; ++f) {
    const void* k = attn_kernel_ptr(f);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    // clusters of up to 16 CTAs (the split-K merge through distributed shared memory)
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {
// attr: room for two attributes (the cluster shape, programmatic dependent launch)
cudaLaunchConfig_t attn_config(int grid, int cluster, cudaStream_t stream,
                               cudaLaunchAttribute* attr, bool tma, bool res, bool pdl) {
  cudaLaunchConfig_t c = {};
  c.gridDim = dim3((unsigned)grid, 1, 1);
  c.blockDim = dim3((unsigned)attn_threads(tma, res), 1, 1);
  c.dynamicSmemBytes = cfg::kSmemBytes;
  c.stream = stream;
  unsigned n = 0;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) attr[n++] = pdl_attribute();
  c.attrs = attr;
  c.numAttrs = n;
  return c;
}
}  // namespace

int attn_max_active_clusters(int cluster, bool fp8) {
  // cluster launches give every CTA one item: the cp.async kernel without the resolver warp
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t c = attn_config(cluster, cluster, nullptr, attr, false, false, false);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attn_kernel_ptr(attn_variant(fp8, false, false)), &c) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_attn(const AttnParams& p_in, int grid, bool fp8, cudaStream_t stream) {
  AttnParams p = p_in;
  cudaLaunchAttribute attr[2];
  // a resolver warp pays off when CTAs have more than one item and the column sets are long
  // enough that walking the page tables is a real share of an item (a single window tile is not)
  const bool res = grid < p.n_items && p.rs.W + p.rs.K >= 256;
  const bool tma = attn_uses_tma(grid, p.n_items, fp8, p.D);
  // Programmatic dependent launch for grids of at most a quarter of the SMs (one CTA an SM): the
  // next grid then sets up on idle SMs while this one runs (decode B1, 32 CTAs: 13.9 -> 13.3 us a
  // call in a CUDA graph).  At 64 CTAs (decode B8) it measured 0.1-0.25 us slower; a grid that
  // fills the GPU would be placed SM by SM in the order the one before it finishes (prefill S2048
  // in a graph: 299 -> 320 us).
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  p.pdl = 4 * grid <= sms ? 1 : 0;
  cudaLaunchConfig_t c = attn_config(grid, p.cluster, stream, attr, tma, res, p.pdl != 0);
  switch (attn_variant(fp8, res, tma)) {
    case 0: return cudaLaunchKernelEx(&c, attn_kernel<true, false, false>, p);
    case 1: return cudaLaunchKernelEx(&c, attn_kernel<true, true, false>, p);
    case 2: return cudaLaunchKernelEx(&c, attn_kernel<false, false, false>, p);
    case 3: return cudaLaunchKernelEx(&c, attn_kernel<false, false, true>, p);
    case 4: return cudaLaunchKernelEx(&c, attn_kernel<false, true, true>, p);
    case 5: return cudaLaunchKernelEx(&c, attn_kernel<true, false, true>, p);
    default: return cudaLaunchKernelEx(&c, attn_kernel<true, true, true>, p);
  }
}

int merge_max_splits() { return kMergeMaxSplits; }

cudaError_t launch_merge(const AttnParams& p, cudaStream_t stream) {
  merge_kernel<<<p.rs.T * p.H, 128, 0, stream>>>(p.ws_o, p.ws_lse,
                                                 reinterpret_cast<__nv_bfloat16*>(p.out),
                                                 p.n_splits, p.H, p.D);
  return cudaGetLastError();
}

cudaError_t launch_resolve_dump(const ResolveArgs& a, int32_t* cols, cudaStream_t stream) {
  const long long total = (long long)a.T * (a.W + a.K);
  if (total == 0) return cudaSuccess;
  const int blocks = (int)((total + 255) / 256);
  resolve_dump_kernel<<<blocks, 256, 0, stream>>>(a, cols);
  return cudaGetLastError();
}

cudaError_t read_and_clear_error_word(int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_spa_error, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_spa_error, &zero, sizeof(int));
}

}  // namespace spa

// spa_launch.h - parameters and launchers shared by the kernel file and the C ABI file.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "spa_device.cuh"

namespace spa {

struct AttnParams {
  // Tensor maps of the pools' rows: K rows of the window pool, its V rows, then the same for the
  // compressed pool.  Each is a 2D byte tensor, one row per token (D elements, the row stride
  // twice that: K and V interleave), 128-byte boxes one row high, 128-byte swizzle.  Set only
  // for launches that gather rows by tensor maps.
  CUtensorMap kv_map[4];
  ResolveArgs rs;
  const uint8_t* q;     // bf16 [T][H][D]
  uint8_t* out;         // bf16 [T][H][D] (prefill)
  float* ws_o;          // decode partials [T][S][H][D], each normalised by its own denominator
  float* ws_lse;        // decode partial log-sum-exp, base 2, [T][S][H]
  int H, D;
  int gh;               // heads per group: 64, or 32 when a decode needs more CTAs per query
  int n_groups;         // ceil(H / gh): the MMAs always see 64 head rows, the ones past gh zero
  int n_splits;         // S: split-K parts per (token, head group); 1 for prefill
  int cols_per_split;   // raw columns per split
  int n_items;          // T * n_groups * n_splits
  float scale_log2;     // softmax scale * log2(e)
  int decode;           // 1: write split partials to ws_o / ws_lse for the merge kernel
  int cluster;          // > 1: the n_splits CTAs of one (token, head group) form a thread-block
                        // cluster and merge their partials through distributed shared memory
  int pdl;              // 1: launched with programmatic dependent launch (set by the launcher)
};

// Kernel launch configuration: 4 softmax warps, 1 MMA warp, the gather warps and 1 resolver
// warp when CTAs have more than one item.  6 gather warps when rows move by tensor-map gathers
// (their issue rate grows with the warps issuing them; 12 warps in all keep 168 registers a
// thread), 4 when they move by cp.async.
__host__ __device__ constexpr int attn_gather_warps(bool tma) { return tma ? 6 : 4; }
__host__ __device__ constexpr int attn_threads(bool tma, bool res) {
  return 32 * (5 + attn_gather_warps(tma) + (res ? 1 : 0));
}
// Rows move by tensor-map gathers when CTAs take more than one item (throughput) and a row is a
// whole number of 128-byte boxes; otherwise by cp.async.
inline bool attn_uses_tma(long long grid, long long n_items, bool fp8, int head_dim) {
  return grid < n_items && (head_dim * (fp8 ? 1 : 2)) % 128 == 0;
}
int attn_smem_bytes();
constexpr int kMaxColumns = 1024;     // window + top-k columns per query

cudaError_t launch_attn(const AttnParams& p, int grid, bool fp8, cudaStream_t stream);
// Largest number of `cluster`-CTA clusters of the attention kernel that can run at once
// (0 when clusters of that size cannot be launched on this device).
int attn_max_active_clusters(int cluster, bool fp8);
int merge_max_splits();
cudaError_t launch_merge(const AttnParams& p, cudaStream_t stream);
cudaError_t launch_resolve_dump(const ResolveArgs& a, int32_t* cols, cudaStream_t stream);

// Paged KV write (the step that fills the pools).
struct KvWriteArgs {
  const uint8_t* k;           // bf16 [T][D]
  const uint8_t* v;           // bf16 [T][D]
  uint8_t* kv;                // pool [num_blocks][page_size][2][D] (bf16 or e4m3)
  float* k_scale;             // e4m3 pools: [num_blocks * page_size]
  float* v_scale;
  const int32_t* bt;          // [B][bt_stride]
  const int32_t* positions;   // [T]
  const int32_t* seq_of_token;  // [T] or NULL
  long long num_blocks;
  int T, D, B, ps, bt_stride;
};
cudaError_t launch_kv_write(const KvWriteArgs& a, bool fp8, cudaStream_t stream);
cudaError_t read_and_clear_kv_write_error_word(int* value);
// Gated pool of the KV compressor (R rows -> one entry per channel).
constexpr int kGatedPoolMaxWarps = 16;
struct GatedPoolArgs {
  const float* kv;             // [B][R][D] fp32, element strides kv_sb, kv_sr, 1
  const float* gate;           // [B][R][D] fp32, element strides gate_sb, gate_sr, 1
  void* out;                   // [B][D] fp32 or bf16, element stride out_sb, 1
  long long kv_sb, kv_sr, gate_sb, gate_sr, out_sb;
  int B, R, D;
  int out_bf16;
};
// 4 when every row of kv and gate starts 16-byte aligned (float4 loads possible), else 1
inline int gated_pool_vector_width(const GatedPoolArgs& g) {
  const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool rows4 = (g.R <= 1 || (g.kv_sr % 4 == 0 && g.gate_sr % 4 == 0)) &&
                     (g.B <= 1 || (g.kv_sb % 4 == 0 && g.gate_sb % 4 == 0));
  return (g.D % 4 == 0 && a16(g.kv) && a16(g.gate) && rows4) ? 4 : 1;
}
cudaError_t launch_gated_pool(const GatedPoolArgs& g, int num_sms, cudaStream_t stream);
cudaError_t prepare_attn_kernels();   // per-device one-time attributes (dynamic shared memory)
cudaError_t read_and_clear_error_word(int* value);

// Decode through split-K partials in a caller-given buffer and the merge kernel, whatever the
// usual plan would be (the path of the no-alloc entry point), and the bytes its partials take when
// the buffer holds cap_bytes (the split count shrinks until they fit; with one split they may
// still not fit, which the caller checks).
size_t decode_partials_bytes(const spa_problem_t* prob, size_t cap_bytes);
int decode_with_partials(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                         const spa_problem_t* prob, void* out, void* ws, size_t ws_bytes,
                         void* stream);

}  // namespace spa

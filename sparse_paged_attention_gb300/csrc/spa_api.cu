// spa_api.cu - the C ABI: host-side validation, work planning and launches.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "sparse_attn_paged.h"
#include "spa_indexer.h"
#include "spa_launch.h"
#include "spa_plan.h"

namespace {

thread_local char g_cuda_msg[512] = "no CUDA error recorded";

int cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(g_cuda_msg, sizeof g_cuda_msg, "%s: %s (%s)", what, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return SPA_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];
bool g_prepared[kMaxDevices];
// clusters of 2, 4, 8, 16 attention CTAs that can be resident at once (both kernel variants)
int g_clusters[kMaxDevices][5];

// SM count of the current device; sets the kernels' shared-memory attribute once per device.
int current_device(int* dev, int* sms) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return SPA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_prepared[*dev]) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = spa::prepare_attn_kernels();
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    g_sms[*dev] = n;
    for (int i = 1; i <= 4; ++i) {
      const int a = spa::attn_max_active_clusters(1 << i, false);
      const int b = spa::attn_max_active_clusters(1 << i, true);
      g_clusters[*dev][i] = a < b ? a : b;
    }
    g_prepared[*dev] = true;
  }
  *sms = g_sms[*dev];
  return SPA_OK;
}

int max_active_clusters(int dev, int size) {
  int i = 0;
  while ((1 << i) < size) ++i;
  if (i < 1 || i > 4) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  return g_clusters[dev][i];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_pool(const spa_pool_t* pl, bool fp8, int head_dim) {
  if (!pl || !pl->kv || !pl->block_table) return SPA_ERR_NULL;
  if (pl->num_blocks < 1 || pl->page_size < 1 || pl->bt_stride < 1) return SPA_ERR_SHAPE;
  if ((long double)pl->num_blocks * pl->page_size > (long double)(1ll << 30)) return SPA_ERR_UNSUPPORTED;
  if (!aligned16(pl->kv)) return SPA_ERR_ALIGN;
  if (fp8 && (!pl->k_scale || !pl->v_scale)) return SPA_ERR_NULL;
  (void)head_dim;
  return SPA_OK;
}

bool uses_cmp(const spa_problem_t* pr) { return pr->ratio > 0 && pr->topk > 0; }

// ---- tensor maps of the bf16 pools (the kernel gathers their rows with tensor-map copies) ----
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return (EncodeTiledFn) nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// K rows (v = 0) or V rows (v = 1) of a pool [num_blocks][page_size][2][D] (elt bytes each) as a
// 2D byte tensor: row i = token row i of the pool (D*elt bytes), row stride 2*D*elt bytes.  Boxes
// are 128 bytes of one row; the 128-byte swizzle puts them straight into the MMA operand layout.
bool encode_pool_rows(CUtensorMap* m, const spa_pool_t* pl, int D, int elt, int v) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t row_bytes = (cuuint64_t)D * elt;
  const cuuint64_t rows = (cuuint64_t)pl->num_blocks * (cuuint64_t)pl->page_size;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {2 * row_bytes};
  const cuuint32_t box[2] = {128, 1};
  const cuuint32_t elem[2] = {1, 1};
  void* base = const_cast<uint8_t*>(static_cast<const uint8_t*>(pl->kv) + v * row_bytes);
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The maps of the last pools each host thread used, kept for the next call on the same pools.
struct PoolMaps {
  const void* kv = nullptr;
  long long num_blocks = 0;
  int page_size = 0, D = 0, elt = 0;
  CUtensorMap map[2];
};
thread_local PoolMaps g_maps[2];

bool pool_maps(CUtensorMap* out, const spa_pool_t* pl, int D, int elt, int which) {
  PoolMaps& c = g_maps[which];
  if (c.kv != pl->kv || c.num_blocks != pl->num_blocks || c.page_size != pl->page_size ||
      c.D != D || c.elt != elt) {
    c.kv = nullptr;
    if (!encode_pool_rows(&c.map[0], pl, D, elt, 0) ||
        !encode_pool_rows(&c.map[1], pl, D, elt, 1))
      return false;
    c.kv = pl->kv;
    c.num_blocks = pl->num_blocks;
    c.page_size = pl->page_size;
    c.D = D;
    c.elt = elt;
  }
  out[0] = c.map[0];
  out[1] = c.map[1];
  return true;
}

int validate(const void* q, const spa_pool_t* win, const spa_pool_t* cmp, const spa_problem_t* pr,
             const void* out, bool fp8) {
  if (!pr) return SPA_ERR_NULL;
  if (pr->num_tokens < 0 || pr->num_seqs < 1 || pr->num_heads < 1 || pr->window < 0 ||
      pr->topk < 0 || pr->ratio < 0 || pr->head_dim < 1)
    return SPA_ERR_SHAPE;
  if (!std::isfinite(pr->scale)) return SPA_ERR_SHAPE;
  if (pr->head_dim % 64 != 0 || pr->head_dim > 512) return SPA_ERR_UNSUPPORTED;
  // (the sum in 64 bits: two large int32 sizes must not wrap past the limit)
  if ((long long)pr->window + (long long)pr->topk > spa::kMaxColumns) return SPA_ERR_UNSUPPORTED;
  if (pr->num_tokens == 0) return SPA_OK;
  if (!q || !out || !pr->positions) return SPA_ERR_NULL;
  if (pr->topk > 0 && !pr->topk_idx) return SPA_ERR_NULL;
  if (!aligned16(q) || !aligned16(out)) return SPA_ERR_ALIGN;
  int st = check_pool(win, fp8, pr->head_dim);
  if (st) return st;
  if (uses_cmp(pr)) {
    st = check_pool(cmp, fp8, pr->head_dim);
    if (st) return st;
  }
  return SPA_OK;
}

void fill_pool(spa::PoolDev& d, const spa_pool_t* s) {
  d.kv = static_cast<const uint8_t*>(s->kv);
  d.k_scale = s->k_scale;
  d.v_scale = s->v_scale;
  d.bt = s->block_table;
  d.num_blocks = s->num_blocks;
  d.ps = s->page_size;
  d.ps_shift = -1;
  for (int k = 0; k < 31; ++k)
    if (s->page_size == (1 << k)) d.ps_shift = k;
  d.bt_stride = s->bt_stride;
}

void fill_resolve(spa::ResolveArgs& a, const spa_pool_t* win, const spa_pool_t* cmp,
                  const spa_problem_t* pr) {
  std::memset(&a, 0, sizeof a);
  fill_pool(a.win, win);
  if (uses_cmp(pr)) {
    fill_pool(a.cmp, cmp);
  } else {
    fill_pool(a.cmp, win);  // never dereferenced: ratio 0 or topk 0 yields no compressed column
  }
  a.positions = pr->positions;
  a.seq_of_token = pr->seq_of_token;
  a.topk = pr->topk_idx;
  a.T = pr->num_tokens;
  a.B = pr->num_seqs;
  a.W = pr->window;
  a.K = pr->topk;
  a.r = uses_cmp(pr) ? pr->ratio : 0;
}

// Decode plan.  With T*G (token, head group) pairs and C columns per query:
//  * T*G >= SMs/2: no split; each CTA attends over whole queries and writes the output directly.
//  * otherwise the columns are split S ways (S a power of two <= 16, at least 16 columns per
//    split, S*T*G CTAs at most one per SM) and the S CTAs of a pair form a thread-block cluster
//    that merges the partial results through distributed shared memory: no workspace, no
//    second kernel.  S shrinks until all T*G clusters fit on the device at once.
//  * if no cluster size fits, the split-K partials go through the workspace and the merge
//    kernel (decode_plan_ws).
struct DecodePlan {
  int splits, cols, cluster;  // cluster == 0 with splits > 1: workspace + merge kernel
  int gh;                     // heads per group (64, or 32 to give one query more CTAs)
};

void decode_plan_ws(const spa_problem_t* pr, int sms, int* splits, int* cols,
                    size_t cap_bytes = SIZE_MAX);

DecodePlan decode_plan(const spa_problem_t* pr, int dev, int sms) {
  const int C = pr->window + pr->topk > 0 ? pr->window + pr->topk : 1;
  const long long T = pr->num_tokens;
  DecodePlan pl{1, C, 0, 64};
  // groups of 32 heads halve what each CTA merges; worth it when 16-way splits still fit
  if (pr->num_heads <= 32 || T * ((pr->num_heads + 31) / 32) * 16 <= sms) pl.gh = 32;
  const long long groups = (pr->num_heads + pl.gh - 1) / pl.gh;
  const long long base = T * groups;
  if (base <= 0 || 2 * base >= sms) {
    pl.gh = 64;
    return pl;
  }
  int S = 16;
  while (S > 1 && ((long long)S * base > sms || (C + S - 1) / S < 16)) S >>= 1;
  while (S > 1 && max_active_clusters(dev, S) < base) S >>= 1;
  if (S > 1) {
    pl.splits = S;
    pl.cols = (C + S - 1) / S;
    pl.cluster = S;
    return pl;
  }
  pl.gh = 64;
  if (max_active_clusters(dev, 2) >= 1) return pl;  // clusters work; one split is the best fit
  decode_plan_ws(pr, sms, &pl.splits, &pl.cols);
  return pl;
}

// Split plan of the workspace path (spa_plan.h): enough splits to give every SM one item, at least
// 32 columns per split, partials of at most cap_bytes.
void decode_plan_ws(const spa_problem_t* pr, int sms, int* splits, int* cols, size_t cap_bytes) {
  spa::plan_partials(pr->window + pr->topk, pr->num_tokens, pr->num_heads, pr->head_dim, sms,
                     spa::merge_max_splits(), cap_bytes, splits, cols);
}

size_t workspace_bytes(const spa_problem_t* pr, int splits) {
  return spa::partials_bytes(pr->num_tokens, pr->num_heads, pr->head_dim, splits);
}

int run(const void* q, const spa_pool_t* win, const spa_pool_t* cmp, const spa_problem_t* pr,
        void* out, void* ws, size_t ws_bytes, void* stream, bool decode, bool fp8,
        bool force_partials = false) {
  int st = validate(q, win, cmp, pr, out, fp8);
  if (st) return st;
  if (pr->num_tokens == 0) return SPA_OK;
  int dev = 0, sms = 0;
  st = current_device(&dev, &sms);
  if (st) return st;

  spa::AttnParams p;
  std::memset(&p, 0, sizeof p);
  fill_resolve(p.rs, win, cmp, pr);
  p.q = static_cast<const uint8_t*>(q);
  p.out = static_cast<uint8_t*>(out);
  p.H = pr->num_heads;
  p.D = pr->head_dim;
  p.gh = 64;
  p.n_groups = (pr->num_heads + 63) / 64;
  p.scale_log2 = pr->scale * 1.4426950408889634f;
  const int C = pr->window + pr->topk;
  bool merge = false;
  if (decode) {
    DecodePlan pl = decode_plan(pr, dev, sms);
    if (force_partials) {   // partials in the caller's buffer, as many splits as fit in it
      pl.cluster = 0;
      pl.gh = 64;
      decode_plan_ws(pr, sms, &pl.splits, &pl.cols, ws_bytes);
    }
    p.gh = pl.gh;
    p.n_groups = (pr->num_heads + pl.gh - 1) / pl.gh;
    p.n_splits = pl.splits;
    p.cols_per_split = pl.cols;
    p.cluster = pl.cluster;
    if (pl.cluster == 0 && (pl.splits > 1 || force_partials)) {
      const size_t need = workspace_bytes(pr, pl.splits);
      if (!ws) return SPA_ERR_NULL;
      if (!aligned16(ws)) return SPA_ERR_ALIGN;
      if (ws_bytes < need) return SPA_ERR_WORKSPACE;
      const size_t tsh = (size_t)pr->num_tokens * pl.splits * pr->num_heads;
      p.ws_o = static_cast<float*>(ws);
      p.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                          spa::plan_align256(tsh * pr->head_dim * sizeof(float)));
      p.decode = 1;
      merge = true;
    }
  } else {
    p.n_splits = 1;
    p.cols_per_split = C > 0 ? C : 1;
    p.decode = 0;
  }
  const long long items = (long long)pr->num_tokens * p.n_groups * p.n_splits;
  if (items > 0x7fffffffLL) return SPA_ERR_UNSUPPORTED;
  p.n_items = (int)items;
  // clustered: one item per CTA; otherwise a persistent grid of at most one CTA per SM
  const int grid = p.cluster > 1 ? (int)items : (int)(items < sms ? items : sms);
  if (spa::attn_uses_tma(grid, items, fp8, pr->head_dim)) {
    const int elt = fp8 ? 1 : 2;
    if (!pool_maps(&p.kv_map[0], win, pr->head_dim, elt, 0)) return SPA_ERR_CUDA;
    if (!pool_maps(&p.kv_map[2], uses_cmp(pr) ? cmp : win, pr->head_dim, elt, 1))
      return SPA_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = spa::launch_attn(p, grid, fp8, s);
  if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
  if (merge) {
    e = spa::launch_merge(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  }
  return SPA_OK;
}

}  // namespace

namespace spa {
size_t decode_partials_bytes(const spa_problem_t* prob, size_t cap_bytes) {
  if (!prob || prob->num_tokens < 0 || prob->num_heads < 1 || prob->head_dim < 1) return 0;
  int dev = 0, sms = 0;
  if (current_device(&dev, &sms) != SPA_OK) return 0;
  int splits = 1, cols = 1;
  decode_plan_ws(prob, sms, &splits, &cols, cap_bytes);
  return workspace_bytes(prob, splits);
}

int decode_with_partials(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                         const spa_problem_t* prob, void* out, void* ws, size_t ws_bytes,
                         void* stream) {
  return run(q, win, cmp, prob, out, ws, ws_bytes, stream, true, false, true);
}
}  // namespace spa

namespace {
int kv_write(const void* k, const void* v, int32_t T, int32_t D, const int32_t* positions,
             const int32_t* seq_of_token, int32_t B, const spa_pool_t* pool, void* stream,
             bool fp8) {
  if (T < 0 || B < 1 || D < 1) return SPA_ERR_SHAPE;
  if (D % 64 != 0 || D > 512) return SPA_ERR_UNSUPPORTED;
  if (T == 0) return SPA_OK;
  if (!k || !v || !positions) return SPA_ERR_NULL;
  if (!aligned16(k) || !aligned16(v)) return SPA_ERR_ALIGN;
  const int st = check_pool(pool, fp8, D);
  if (st) return st;
  int dev = 0, sms = 0;
  const int ds = current_device(&dev, &sms);
  if (ds) return ds;
  spa::KvWriteArgs a;
  std::memset(&a, 0, sizeof a);
  a.k = static_cast<const uint8_t*>(k);
  a.v = static_cast<const uint8_t*>(v);
  a.kv = static_cast<uint8_t*>(const_cast<void*>(pool->kv));       // written by these calls
  a.k_scale = const_cast<float*>(pool->k_scale);
  a.v_scale = const_cast<float*>(pool->v_scale);
  a.bt = pool->block_table;
  a.positions = positions;
  a.seq_of_token = seq_of_token;
  a.num_blocks = pool->num_blocks;
  a.T = T;
  a.D = D;
  a.B = B;
  a.ps = pool->page_size;
  a.bt_stride = pool->bt_stride;
  const cudaError_t e = spa::launch_kv_write(a, fp8, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv write kernel launch");
  return SPA_OK;
}
}  // namespace

namespace {
// ---- prefill from host buffers: chunks through a device staging area of kHostSlots slots ----
constexpr int kHostSlots = 2;   // (three measured the same)
// Per device: a stream each for the copies in, the kernels and the copies out, and the events
// that order them; made on the first call, kept for the process.
struct HostPipe {
  bool ready;
  cudaStream_t in, comp, out;
  cudaEvent_t entry, exit, in_done[kHostSlots], comp_done[kHostSlots], out_done[kHostSlots];
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte offsets of one staging slot (a chunk of tc tokens): q, out, top-k lists, positions,
// sequence ids, each 256-byte aligned.
struct HostSlot {
  size_t q, out, topk, pos, seq, bytes;
};
HostSlot host_slot(const spa_problem_t* pr, long long tc) {
  const size_t rows = (size_t)tc * (size_t)pr->num_heads * (size_t)pr->head_dim * 2;
  HostSlot s;
  s.q = 0;
  s.out = round256(rows);
  s.topk = s.out + round256(rows);
  s.pos = s.topk + round256((size_t)tc * (size_t)pr->topk * 4);
  s.seq = s.pos + round256((size_t)tc * 4);
  s.bytes = s.seq + round256((size_t)tc * 4);
  return s;
}

int host_pipe(int dev, HostPipe** out) {
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    cudaError_t e = cudaSuccess;
    for (cudaStream_t* st : {&hp.in, &hp.comp, &hp.out})
      if (e == cudaSuccess) e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&hp.entry, &hp.exit})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    for (int i = 0; i < kHostSlots; ++i)
      for (cudaEvent_t* ev : {&hp.in_done[i], &hp.comp_done[i], &hp.out_done[i]})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "host prefill streams");
    hp.ready = true;
  }
  *out = &hp;
  return SPA_OK;
}

int prefill_host(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                 const spa_problem_t* pr, void* out, int32_t chunk, void* staging,
                 size_t staging_bytes, void* stream, bool fp8) {
  int st = validate(q, win, cmp, pr, out, fp8);
  if (st) return st;
  if (chunk < 1) return SPA_ERR_SHAPE;
  if (pr->num_tokens == 0) return SPA_OK;
  if (!staging) return SPA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(staging) % 256 != 0) return SPA_ERR_ALIGN;
  const long long T = pr->num_tokens;
  const long long tc = chunk < T ? chunk : T;
  const HostSlot sl = host_slot(pr, tc);
  if (staging_bytes < kHostSlots * sl.bytes) return SPA_ERR_WORKSPACE;
  int dev = 0, sms = 0;
  st = current_device(&dev, &sms);
  if (st) return st;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* hp = nullptr;
  st = host_pipe(dev, &hp);
  if (st) return st;
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  const size_t qrow = (size_t)pr->num_heads * (size_t)pr->head_dim * 2;   // bytes of one token
  const int K = pr->topk;
  const auto H2D = cudaMemcpyHostToDevice;
  cudaError_t e = cudaEventRecord(hp->entry, user);
  for (cudaStream_t s : {hp->in, hp->comp, hp->out})
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->entry, 0);
  // chunk sizes (spa_plan.h): a quarter chunk first and last, so that the pipeline fills and
  // drains sooner (nothing overlaps the first chunk's copy in, nor the last chunk's kernel and
  // copy out), full chunks between
  int c = 0;
  for (long long c0 = 0, n = 0; c0 < T && e == cudaSuccess && st == SPA_OK; c0 += n, ++c) {
    n = spa::host_chunk_tokens(T, tc, c0);
    const int slot = c % kHostSlots;
    uint8_t* base = static_cast<uint8_t*>(staging) + (size_t)slot * sl.bytes;
    // copies in, once the kernel of the chunk kHostSlots back has read this slot
    if (c >= kHostSlots) e = cudaStreamWaitEvent(hp->in, hp->comp_done[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(base + sl.q, static_cast<const uint8_t*>(q) + (size_t)c0 * qrow,
                          (size_t)n * qrow, H2D, hp->in);
    if (e == cudaSuccess && K > 0)
      e = cudaMemcpyAsync(base + sl.topk, pr->topk_idx + (size_t)c0 * K, (size_t)n * K * 4, H2D,
                          hp->in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(base + sl.pos, pr->positions + c0, (size_t)n * 4, H2D, hp->in);
    if (e == cudaSuccess && pr->seq_of_token)
      e = cudaMemcpyAsync(base + sl.seq, pr->seq_of_token + c0, (size_t)n * 4, H2D, hp->in);
    if (e == cudaSuccess) e = cudaEventRecord(hp->in_done[slot], hp->in);
    // the chunk's attention, once its inputs are in and the slot's previous copy out is done
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->comp, hp->in_done[slot], 0);
    if (e == cudaSuccess && c >= kHostSlots)
      e = cudaStreamWaitEvent(hp->comp, hp->out_done[slot], 0);
    if (e != cudaSuccess) break;
    spa_problem_t cp = *pr;
    cp.num_tokens = (int32_t)n;
    cp.positions = reinterpret_cast<const int32_t*>(base + sl.pos);
    cp.topk_idx = K > 0 ? reinterpret_cast<const int32_t*>(base + sl.topk) : nullptr;
    cp.seq_of_token = pr->seq_of_token ? reinterpret_cast<const int32_t*>(base + sl.seq) : nullptr;
    st = run(base + sl.q, win, cmp, &cp, base + sl.out, nullptr, 0, hp->comp, false, fp8);
    if (st != SPA_OK) break;
    e = cudaEventRecord(hp->comp_done[slot], hp->comp);
    // copy out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->comp_done[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<uint8_t*>(out) + (size_t)c0 * qrow, base + sl.out,
                          (size_t)n * qrow, cudaMemcpyDeviceToHost, hp->out);
    if (e == cudaSuccess) e = cudaEventRecord(hp->out_done[slot], hp->out);
  }
  // the caller's stream resumes after everything enqueued here, also after a failure part way
  for (cudaStream_t s : {hp->in, hp->comp, hp->out}) {
    cudaError_t e2 = cudaEventRecord(hp->exit, s);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(user, hp->exit, 0);
    if (e == cudaSuccess) e = e2;
  }
  if (st != SPA_OK) return st;
  if (e != cudaSuccess) return cuda_fail(e, "host prefill copies");
  return SPA_OK;
}
}  // namespace

extern "C" {

size_t sparse_attn_paged_prefill_host_staging_size(const spa_problem_t* prob,
                                                   int32_t chunk_tokens) {
  if (!prob || prob->num_tokens < 0 || prob->num_heads < 1 || prob->head_dim < 1 ||
      prob->topk < 0 || chunk_tokens < 1)
    return 0;
  const long long tc = chunk_tokens < prob->num_tokens ? chunk_tokens : prob->num_tokens;
  return kHostSlots * host_slot(prob, tc > 0 ? tc : 1).bytes;
}

int sparse_attn_paged_prefill_host(const void* q_host, const spa_pool_t* win,
                                   const spa_pool_t* cmp, const spa_problem_t* prob,
                                   void* out_host, int32_t chunk_tokens, void* staging,
                                   size_t staging_bytes, void* stream) {
  return prefill_host(q_host, win, cmp, prob, out_host, chunk_tokens, staging, staging_bytes,
                      stream, false);
}

int sparse_attn_paged_prefill_host_fp8(const void* q_host, const spa_pool_t* win,
                                       const spa_pool_t* cmp, const spa_problem_t* prob,
                                       void* out_host, int32_t chunk_tokens, void* staging,
                                       size_t staging_bytes, void* stream) {
  return prefill_host(q_host, win, cmp, prob, out_host, chunk_tokens, staging, staging_bytes,
                      stream, true);
}

int sparse_attn_paged_prefill(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                              const spa_problem_t* prob, void* out, void* stream) {
  return run(q, win, cmp, prob, out, nullptr, 0, stream, false, false);
}

int sparse_attn_paged_prefill_fp8(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                                  const spa_problem_t* prob, void* out, void* stream) {
  return run(q, win, cmp, prob, out, nullptr, 0, stream, false, true);
}

size_t sparse_attn_paged_decode_workspace_size(const spa_problem_t* prob) {
  if (!prob || prob->num_tokens < 0 || prob->num_heads < 1 || prob->head_dim < 1) return 0;
  int dev = 0, sms = 0;
  if (current_device(&dev, &sms) != SPA_OK) return 0;
  const DecodePlan pl = decode_plan(prob, dev, sms);
  return (pl.cluster > 1 || pl.splits == 1) ? 0 : workspace_bytes(prob, pl.splits);
}

int sparse_attn_paged_decode(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                             const spa_problem_t* prob, void* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return run(q, win, cmp, prob, out, workspace, workspace_bytes, stream, true, false);
}

int sparse_attn_paged_decode_fp8(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                                 const spa_problem_t* prob, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return run(q, win, cmp, prob, out, workspace, workspace_bytes, stream, true, true);
}

int sparse_attn_paged_resolve_columns(const spa_pool_t* win, const spa_pool_t* cmp,
                                      const spa_problem_t* prob, int32_t* cols, void* stream) {
  if (!prob) return SPA_ERR_NULL;
  if (prob->num_tokens < 0 || prob->num_seqs < 1 || prob->window < 0 || prob->topk < 0 ||
      prob->ratio < 0)
    return SPA_ERR_SHAPE;
  // (the column count in 64 bits: window + topk must not wrap)
  if ((long long)prob->window + (long long)prob->topk > 0x7fffffffLL) return SPA_ERR_UNSUPPORTED;
  if (prob->num_tokens == 0 || prob->window + prob->topk == 0) return SPA_OK;
  if (!cols || !prob->positions) return SPA_ERR_NULL;
  if (prob->topk > 0 && !prob->topk_idx) return SPA_ERR_NULL;
  int st = check_pool(win, false, prob->head_dim);
  if (st) return st;
  if (uses_cmp(prob)) {
    st = check_pool(cmp, false, prob->head_dim);
    if (st) return st;
  }
  spa::ResolveArgs a;
  fill_resolve(a, win, cmp, prob);
  cudaError_t e = spa::launch_resolve_dump(a, cols, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "resolve kernel launch");
  return SPA_OK;
}

int sparse_attn_gated_pool(const float* kv, const float* gate, int32_t batch, int32_t rows,
                           int32_t dim, int64_t kv_stride_b, int64_t kv_stride_r,
                           int64_t gate_stride_b, int64_t gate_stride_r, void* out,
                           int32_t out_dtype, int64_t out_stride_b, void* stream) {
  if (batch < 0 || rows < 0 || dim < 0 || kv_stride_b < 0 || kv_stride_r < 0 ||
      gate_stride_b < 0 || gate_stride_r < 0 || out_stride_b < 0)
    return SPA_ERR_SHAPE;
  if (out_dtype != SPA_DTYPE_F32 && out_dtype != SPA_DTYPE_BF16) return SPA_ERR_UNSUPPORTED;
  if (batch == 0 || dim == 0) return SPA_OK;
  if (!out || (rows > 0 && (!kv || !gate))) return SPA_ERR_NULL;
  const uintptr_t out_align = out_dtype == SPA_DTYPE_BF16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(kv) & 3u) || (reinterpret_cast<uintptr_t>(gate) & 3u) ||
      (reinterpret_cast<uintptr_t>(out) & (out_align - 1)))
    return SPA_ERR_ALIGN;
  int dev = 0, sms = 0;
  const int ds = current_device(&dev, &sms);
  if (ds) return ds;
  spa::GatedPoolArgs g;
  std::memset(&g, 0, sizeof g);
  g.kv = kv;
  g.gate = gate;
  g.out = out;
  g.kv_sb = kv_stride_b;
  g.kv_sr = kv_stride_r;
  g.gate_sb = gate_stride_b;
  g.gate_sr = gate_stride_r;
  g.out_sb = out_stride_b;
  g.B = batch;
  g.R = rows;
  g.D = dim;
  g.out_bf16 = out_dtype == SPA_DTYPE_BF16;
  const cudaError_t e = spa::launch_gated_pool(g, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gated pool kernel launch");
  return SPA_OK;
}

int sparse_attn_indexer_logits(const void* q, const float* weights, int32_t num_tokens,
                               int32_t num_heads, const spa_pool_t* keys,
                               const int32_t* positions, const int32_t* seq_of_token,
                               int32_t num_seqs, int32_t ratio, const int32_t* cand,
                               int32_t num_cols, float* logits, void* stream) {
  if (num_tokens < 0 || num_cols < 0 || num_seqs < 1 || ratio < 1 || num_heads < 1)
    return SPA_ERR_SHAPE;
  if (num_heads != spa::kIdxHeads) return SPA_ERR_UNSUPPORTED;
  if (num_tokens == 0 || num_cols == 0) return SPA_OK;
  if (!q || !weights || !keys || !keys->kv || !keys->block_table || !positions || !logits)
    return SPA_ERR_NULL;
  if (keys->num_blocks < 1 || keys->page_size < 1 || keys->bt_stride < 1) return SPA_ERR_SHAPE;
  const auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!aligned16(q) || !a4(weights) || !a4(keys->kv) || !a4(logits)) return SPA_ERR_ALIGN;
  int dev = 0, sms = 0;
  const int ds = current_device(&dev, &sms);
  if (ds) return ds;
  spa::IndexerArgs a;
  std::memset(&a, 0, sizeof a);
  a.q = static_cast<const uint16_t*>(q);
  a.w = weights;
  a.keys = static_cast<const int32_t*>(keys->kv);
  a.bt = keys->block_table;
  a.positions = positions;
  a.seq_of_token = seq_of_token;
  a.cand = cand;
  a.logits = logits;
  a.num_blocks = keys->num_blocks;
  a.T = num_tokens;
  a.B = num_seqs;
  a.ps = keys->page_size;
  a.bt_stride = keys->bt_stride;
  a.ratio = ratio;
  a.ncols = num_cols;
  // queries share a key tile only when they share a sequence: with no sequence ids every query
  // is in sequence 0 and groups of eight share each tile; otherwise (and in candidate mode, where
  // every query has its own entries) one query per group
  a.nq = (cand || seq_of_token) ? 1 : (num_tokens < spa::kIdxMaxQ ? num_tokens : spa::kIdxMaxQ);
  a.ntiles = (num_cols + spa::kIdxTile - 1) / spa::kIdxTile;
  a.nunits = (long long)((num_tokens + a.nq - 1) / a.nq) * a.ntiles;
  const cudaError_t e = spa::launch_indexer(a, cand != nullptr, sms,
                                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "indexer kernel launch");
  return SPA_OK;
}

int sparse_attn_indexer_topk(const float* logits, int32_t num_tokens, int32_t num_cols,
                             const int32_t* cand, int32_t k, int32_t* topk_idx, void* stream) {
  if (num_tokens < 0 || num_cols < 0 || k < 0) return SPA_ERR_SHAPE;
  if (k > spa::kIdxTopkMax) return SPA_ERR_UNSUPPORTED;
  if (num_tokens == 0 || k == 0) return SPA_OK;
  if (!topk_idx || (num_cols > 0 && !logits)) return SPA_ERR_NULL;
  const auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!a4(logits) || !a4(cand) || !a4(topk_idx)) return SPA_ERR_ALIGN;
  int dev = 0, sms = 0;
  const int ds = current_device(&dev, &sms);
  if (ds) return ds;
  spa::TopkArgs a;
  std::memset(&a, 0, sizeof a);
  a.logits = logits;
  a.cand = cand;
  a.topk = topk_idx;
  a.T = num_tokens;
  a.ncols = num_cols;
  a.k = k;
  const cudaError_t e = spa::launch_topk(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "top-k kernel launch");
  return SPA_OK;
}

int sparse_attn_paged_kv_write(const void* k, const void* v, int32_t num_tokens, int32_t head_dim,
                               const int32_t* positions, const int32_t* seq_of_token,
                               int32_t num_seqs, const spa_pool_t* pool, void* stream) {
  return kv_write(k, v, num_tokens, head_dim, positions, seq_of_token, num_seqs, pool, stream,
                  false);
}

int sparse_attn_paged_kv_write_fp8(const void* k, const void* v, int32_t num_tokens,
                                   int32_t head_dim, const int32_t* positions,
                                   const int32_t* seq_of_token, int32_t num_seqs,
                                   const spa_pool_t* pool, void* stream) {
  return kv_write(k, v, num_tokens, head_dim, positions, seq_of_token, num_seqs, pool, stream,
                  true);
}

int sparse_attn_paged_check_errors(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = spa::read_and_clear_error_word(&v);
  if (e != cudaSuccess) return cuda_fail(e, "device error word");
  int w = 0;
  e = spa::read_and_clear_kv_write_error_word(&w);
  if (e != cudaSuccess) return cuda_fail(e, "device error word");
  int x = 0;
  e = spa::read_and_clear_indexer_error_word(&x);
  if (e != cudaSuccess) return cuda_fail(e, "device error word");
  return v | w | x;
}

const char* sparse_attn_paged_strerror(int status) {
  switch (status) {
    case SPA_OK: return "SPA_OK";
    case SPA_ERR_NULL: return "SPA_ERR_NULL: a required pointer is NULL";
    case SPA_ERR_ALIGN: return "SPA_ERR_ALIGN: a buffer is not 16-byte aligned";
    case SPA_ERR_SHAPE: return "SPA_ERR_SHAPE: negative or inconsistent sizes";
    case SPA_ERR_UNSUPPORTED: return "SPA_ERR_UNSUPPORTED: shape outside the supported range";
    case SPA_ERR_WORKSPACE: return "SPA_ERR_WORKSPACE: decode workspace too small";
    case SPA_ERR_CUDA: return "SPA_ERR_CUDA: CUDA runtime error";
    case SPA_ERR_INDEX: return "SPA_ERR_INDEX: a column referenced a page or block outside its table or pool";
    case SPA_ERR_TIMEOUT: return "SPA_ERR_TIMEOUT: a pipeline wait gave up";
    case SPA_ERR_INDEX | SPA_ERR_TIMEOUT: return "SPA_ERR_INDEX | SPA_ERR_TIMEOUT";
    default: return "unknown status";
  }
}

const char* sparse_attn_paged_last_cuda_error(void) { return g_cuda_msg; }

const char* sparse_attn_paged_version(void) { return "sparse_paged_attention_gb300 0.1 (sm_103a)"; }

}  // extern "C"

/*
 * sparse_attn_paged.h - C ABI of the GB300 (sm_103a) sparse paged attention library.
 *
 * What is computed (FreeToken PR 633, "perf(kernel): keep 16-byte kv loads in dsv4 sparse
 * attention and unroll gated pool": call paths and "Changes"; the workloads of its "Kernel time"
 * table): every query token t, at absolute position p = positions[t] in sequence
 * b = seq_of_token[t], attends with ONE softmax over a gathered column set:
 *
 *   window columns   c = 0 .. window-1  : token  x = p - window + 1 + c, present iff x >= 0,
 *                                         row = win.block_table[b][x / ps] * ps + x % ps
 *   top-k columns    c = window .. +topk: entry  j = topk_idx[t][c - window], present iff
 *                                         j >= 0, ratio > 0 and ratio*j + ratio - 1 <= p,
 *                                         row = cmp.block_table[b][j / ps] * ps + j % ps
 *
 *   s_c   = scale * sum_d q[t][h][d] * K[row_c][d]
 *   out[t][h][:] = sum_c softmax(s)_c * V[row_c][:]          (bf16, round to nearest even)
 *
 * K/V rows have one kv_head shared by all query heads.  With fp8 pools the K and V values are
 * e4m3 codes times a per-(token, kv_head) fp32 scale (FreeToken clone PR 3, "Perf/kv fp8 read
 * path", part 1): the K scale multiplies the scores, the V scale multiplies the probabilities
 * before the PV product, and the softmax denominator accumulates the unscaled probabilities.
 *
 * Stream order: every call is asynchronous on its stream and ordered after the work enqueued
 * before it.  Calls whose grids take at most half the SMs launch with programmatic dependent
 * launch: their CTAs may be resident and set up while the kernel before them in the stream still
 * runs, but they read and write no global memory until that kernel has completed.
 *
 * Memory layout (all device pointers are owned by the caller; the library never allocates,
 * frees or keeps a pointer after a call returns, and never synchronises the stream except in
 * sparse_attn_paged_check_errors):
 *   q          bf16  [num_tokens][num_heads][head_dim], 16-byte aligned
 *   out        bf16  [num_tokens][num_heads][head_dim], 16-byte aligned
 *   pool.kv    [num_blocks][page_size][2][head_dim]: index 0 is K, index 1 is V; bf16, or e4m3
 *              codes (one byte each) for the _fp8 entry points; 16-byte aligned (the pool may be
 *              a view that starts at any row of a larger allocation)
 *   pool.k_scale, pool.v_scale   fp32 [num_blocks * page_size] (fp8 only, else NULL)
 *   pool.block_table             int32 [num_seqs][bt_stride]; -1 marks an unmapped page
 *   positions  int32 [num_tokens];  seq_of_token int32 [num_tokens] or NULL (all in seq 0)
 *   topk_idx   int32 [num_tokens][topk], -1 padded anywhere; NULL allowed when topk == 0
 *
 * Errors: every entry point returns an spa_status_t.  Host-side checks (NULL pointers,
 * alignment, unsupported shapes, workspace size) return before anything is launched.  Input
 * errors found on the device (a referenced page beyond its block table, a block id outside the
 * pool, a sequence id outside [0, num_seqs)) drop the column and set SPA_ERR_INDEX in a device
 * error word; a pipeline wait that exceeds its time limit sets SPA_ERR_TIMEOUT and ends the
 * kernel early.  sparse_attn_paged_check_errors() reads and clears that word.
 *
 * Supported shapes: head_dim in {64, 128, ..., 512} (multiple of 64), num_heads >= 1 (heads
 * are processed in groups of 64), window + topk <= 1024, num_blocks * page_size <= 2^30.
 *
 * Per-device state: on its first call on a device the library sets its kernels' launch attributes
 * and caches the SM count, cluster occupancy and the device address of its scratch array, for the
 * rest of the process.  cudaDeviceReset() discards the attributes and the array but not the
 * cache, so the library must not be used on a device after that device was reset.
 */
#ifndef SPARSE_ATTN_PAGED_H
#define SPARSE_ATTN_PAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum spa_status {
  SPA_OK = 0,
  SPA_ERR_NULL = 1,         /* a required pointer is NULL                                      */
  SPA_ERR_ALIGN = 2,        /* q, out, a pool or the workspace is not 16-byte aligned           */
  SPA_ERR_SHAPE = 3,        /* negative or inconsistent sizes                                   */
  SPA_ERR_UNSUPPORTED = 4,  /* head_dim, window + topk or pool size outside the supported range */
  SPA_ERR_WORKSPACE = 5,    /* decode workspace smaller than sparse_attn_paged_decode_workspace_size */
  SPA_ERR_CUDA = 6,         /* a CUDA runtime call failed: see sparse_attn_paged_last_cuda_error */
  SPA_ERR_INDEX = 8,        /* device: a column referenced a page or block outside its table/pool */
  SPA_ERR_TIMEOUT = 16      /* device: a pipeline wait gave up; outputs of that call are invalid */
} spa_status_t;

/* One paged pool: the window pool or the compressed pool. */
typedef struct spa_pool {
  const void* kv;               /* device, see layout above                                  */
  const float* k_scale;         /* device, fp8 pools only                                    */
  const float* v_scale;         /* device, fp8 pools only                                    */
  const int32_t* block_table;   /* device, [num_seqs][bt_stride]                             */
  int64_t num_blocks;           /* physical pages in the pool                                */
  int32_t page_size;            /* rows per page (> 0)                                       */
  int32_t bt_stride;            /* int32 entries per block-table row (> 0)                   */
} spa_pool_t;

/* Problem description shared by every entry point. */
typedef struct spa_problem {
  int32_t num_tokens;           /* T: query tokens (decode: one per sequence)                */
  int32_t num_seqs;             /* B: rows of the block tables                               */
  int32_t num_heads;            /* H: query heads sharing the single kv_head                 */
  int32_t head_dim;             /* D                                                         */
  int32_t window;               /* W: sliding-window columns                                 */
  int32_t topk;                 /* K: top-k columns per query                                */
  int32_t ratio;                /* r: compress ratio; 0 = no compressed columns (window only) */
  float scale;                  /* softmax scale applied to q.k (e.g. 1/sqrt(head_dim))      */
  const int32_t* positions;     /* device [T]                                                */
  const int32_t* seq_of_token;  /* device [T] or NULL                                        */
  const int32_t* topk_idx;      /* device [T][K] or NULL if K == 0                           */
} spa_problem_t;

/*
 * Prefill: one pass over every column of each query (FreeToken PR 633, call paths:
 * sparse_attn_paged -> prefill kernel).  cmp may be NULL iff ratio == 0 (the ratio-0 alias of
 * the page's "Correctness and tests").  Asynchronous on `stream` (a cudaStream_t, NULL = legacy
 * default stream).  Writes out[T][H][D].
 */
int sparse_attn_paged_prefill(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                              const spa_problem_t* prob, void* out, void* stream);

/* Same with e4m3 pools (FreeToken clone PR 3, part 1: the scale is folded into the scores and
 * into the probabilities before PV, never into the K/V tiles). */
int sparse_attn_paged_prefill_fp8(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                                  const spa_problem_t* prob, void* out, void* stream);

/*
 * Prefill from host buffers: the same result as sparse_attn_paged_prefill[_fp8], bit for bit,
 * for a caller whose queries and output live in host memory (the pages' prefill is one attention
 * call per chunk of tokens, FreeToken PR 633 "Call paths").
 *   q_host, out_host          host [T][H][D] bf16, 16-byte aligned;
 *   prob->positions, ->topk_idx, ->seq_of_token   host arrays (the other fields as above);
 *   win, cmp                  device pools and block tables (the resident KV cache);
 *   chunk_tokens              tokens per chunk (>= 1);
 *   staging                   device memory, 256-byte aligned, of at least
 *                             sparse_attn_paged_prefill_host_staging_size(prob, chunk_tokens) bytes
 *                             (two slots of one chunk's q, out, top-k lists, positions and
 *                             sequence ids).
 * The tokens go through the staging memory a chunk at a time (a quarter of chunk_tokens first and
 * last, chunk_tokens between): each chunk's q, top-k lists and positions are copied in, attended
 * and its output copied out, with the copies in, the kernels and the copies out of consecutive
 * chunks overlapping on streams of the library's own (made on the first call on a device, kept
 * for the process).  Every query's output depends only on
 * its own inputs, hence the bit-for-bit equality.  Host memory should be page-locked
 * (cudaHostAlloc / cudaHostRegister) for the copies to run asynchronously and overlap.
 * Stream order: the work starts after what was enqueued on `stream` before the call, and what
 * is enqueued on `stream` after it waits for all of it (out_host is complete once `stream` has
 * reached that point).  Calls from several host threads are serialised.  Errors: those of
 * sparse_attn_paged_prefill, SPA_ERR_SHAPE (chunk_tokens < 1), SPA_ERR_NULL / SPA_ERR_ALIGN /
 * SPA_ERR_WORKSPACE for the staging memory.
 */
size_t sparse_attn_paged_prefill_host_staging_size(const spa_problem_t* prob,
                                                   int32_t chunk_tokens);
int sparse_attn_paged_prefill_host(const void* q_host, const spa_pool_t* win,
                                   const spa_pool_t* cmp, const spa_problem_t* prob,
                                   void* out_host, int32_t chunk_tokens, void* staging,
                                   size_t staging_bytes, void* stream);
int sparse_attn_paged_prefill_host_fp8(const void* q_host, const spa_pool_t* win,
                                       const spa_pool_t* cmp, const spa_problem_t* prob,
                                       void* out_host, int32_t chunk_tokens, void* staging,
                                       size_t staging_bytes, void* stream);

/*
 * Decode: split-K over the column set (FreeToken PR 633, call paths: the split-K decode kernel),
 * then a log-sum-exp merge of the per-split partials into out.  When the queries leave SMs idle,
 * the column set of each query is split over up to 16 CTAs that form one thread-block cluster and
 * merge their partials through distributed shared memory, in the same kernel; when the queries
 * alone fill the GPU there is no split.  Both plans need no workspace and
 * sparse_attn_paged_decode_workspace_size returns 0 (workspace may then be NULL).  Only where
 * clusters cannot be launched do the partials go through a device workspace of at least
 * sparse_attn_paged_decode_workspace_size(prob) bytes (16-byte aligned, contents scratch; two
 * concurrent calls need different workspaces) and a second, merge kernel.
 */
size_t sparse_attn_paged_decode_workspace_size(const spa_problem_t* prob);
int sparse_attn_paged_decode(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                             const spa_problem_t* prob, void* out, void* workspace,
                             size_t workspace_bytes, void* stream);
int sparse_attn_paged_decode_fp8(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                                 const spa_problem_t* prob, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Decode that allocates nothing (the pages have no counterpart: this is a convenience of this
 * library).  For callers that cannot call cudaMalloc where they decode - a host runtime whose
 * device allocator belongs to someone else, or one with no allocator hooks at that point.  Same
 * computation and result as sparse_attn_paged_decode, with the
 * caller still passing q, the pools and out.  This entry point always takes the split-K path with
 * global partials and the merge kernel, and its partials go to a scratch array built into the
 * library (SPA_NOALLOC_SCRATCH_BYTES bytes on every device that loads it, held until the process
 * exits) instead of a caller workspace.
 *   - The first call on a device, with that device current, looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture on that device.
 *   - The partials take fp32 [T][S][H][D] plus [T][S][H] log-sum-exps for S splits per query.  S
 *     follows the SM count (about one split item per SM), and is lowered, down to 1, until the
 *     partials fit in SPA_NOALLOC_SCRATCH_BYTES.  Only a problem whose single-split partials do not
 *     fit (more than 127 tokens of 64 heads x head_dim 512) is rejected with SPA_ERR_WORKSPACE.
 *   - Every call on a device shares the one array and leaves its partials there: two calls that
 *     can overlap on the GPU (different streams without ordering between them) race and give
 *     wrong results.  Calls ordered on one stream are safe.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 */
#define SPA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int sparse_attn_paged_decode_noalloc(const void* q, const spa_pool_t* win, const spa_pool_t* cmp,
                                     const spa_problem_t* prob, void* out, void* stream);

/*
 * Column dump (the integer half of the method, exposed for exact checks): cols[T][W + K] gets
 * the physical row of every column, window columns as the row itself, top-k columns as
 * (1 << 30) | row, and -1 where the column does not exist.  Uses the same device resolution
 * code as the attention kernels.
 */
int sparse_attn_paged_resolve_columns(const spa_pool_t* win, const spa_pool_t* cmp,
                                      const spa_problem_t* prob, int32_t* cols, void* stream);

/*
 * Paged KV write: the step that fills the pools the attention reads.  Token t's K row k[t][:] and
 * V row v[t][:] (bf16, one kv_head, head_dim D each; [T][D] row-major, 16-byte aligned) go to the
 * pool slot of its position: row = block_table[b][x / page_size] * page_size + x % page_size
 * with x = positions[t] and b = seq_of_token[t] (NULL: every token in sequence 0).  Slot row of
 * pool.kv is [2][D]: K then V (the layout of the FreeToken PR 633 pools).  Rows of other slots are
 * untouched.
 *   - sparse_attn_paged_kv_write: bf16 pools, the rows are copied.
 *   - sparse_attn_paged_kv_write_fp8: e4m3 pools (FreeToken clone PR 3, "Perf/kv fp8 read path":
 *     one scale per token and kv_head, separately for K and V).  For each row x (fp32 values of the
 *     bf16 inputs): scale = max|x| / 448 (IEEE fp32 division; 1 if the row is all zero), codes =
 *     e4m3(x_i / scale), fp32 division then round to nearest even (the largest magnitude, 448,
 *     cannot be exceeded by more than rounding and saturates there).  Scales go to
 *     pool.k_scale / pool.v_scale [row].
 * A token whose position is negative, whose page is past the block table's stride, whose block id
 * is outside [0, num_blocks) or whose sequence id is outside [0, num_seqs) is skipped and sets
 * SPA_ERR_INDEX in the device error word.  Two tokens writing one slot: the later write is not
 * defined.  head_dim: a multiple of 64, at most 512.  Asynchronous on `stream`.
 */
int sparse_attn_paged_kv_write(const void* k, const void* v, int32_t num_tokens, int32_t head_dim,
                               const int32_t* positions, const int32_t* seq_of_token,
                               int32_t num_seqs, const spa_pool_t* pool, void* stream);
int sparse_attn_paged_kv_write_fp8(const void* k, const void* v, int32_t num_tokens,
                                   int32_t head_dim, const int32_t* positions,
                                   const int32_t* seq_of_token, int32_t num_seqs,
                                   const spa_pool_t* pool, void* stream);

/*
 * Gated pool of the KV compressor (FreeToken PR 633, call paths: the DeepSeek-V4 compressor's
 * decode step folds R buffered rows into one compressed entry; "Changes": a maximum over R, then a
 * weighted pass).  For every entry b and channel d, a softmax of the gates over the R rows weighs
 * the kv rows:
 *     out[b][d] = sum_r exp(gate[b][r][d] - M) * kv[b][r][d] / sum_r exp(gate[b][r][d] - M),
 *     M = max_r gate[b][r][d].
 * (The page prints no formula; this per-channel softmax is the reading taken.)
 *   kv, gate:  fp32 device arrays [batch][rows][dim], innermost stride 1, other strides in
 *              elements (>= 0; strided views allowed); 4-byte aligned.  Rows that start 16-byte
 *              aligned (base and strides multiples of 4 elements, dim % 4 == 0) are read with
 *              16-byte loads, others with 4-byte loads: same result.
 *   out:       device array [batch][dim] of out_dtype (SPA_DTYPE_F32 or SPA_DTYPE_BF16, rounded to
 *              nearest even), innermost stride 1, batch stride out_stride_b elements; aligned to
 *              its element size.  Must not overlap kv or gate.
 *   rows == 0 writes zeros.  batch == 0 or dim == 0 does nothing.  Arithmetic is fp32 with one
 *   online maximum per channel (the rows are read once).  Gates of +-inf or NaN give what the
 *   formula gives in IEEE arithmetic (NaN where it is undefined).
 * Returns SPA_ERR_SHAPE for negative sizes or strides, SPA_ERR_NULL, SPA_ERR_ALIGN,
 * SPA_ERR_UNSUPPORTED for an unknown out_dtype, SPA_ERR_CUDA if the launch fails.  Asynchronous on
 * `stream`; allocates nothing.
 */
#define SPA_DTYPE_F32 0
#define SPA_DTYPE_BF16 1
int sparse_attn_gated_pool(const float* kv, const float* gate, int32_t batch, int32_t rows,
                           int32_t dim, int64_t kv_stride_b, int64_t kv_stride_r,
                           int64_t gate_stride_b, int64_t gate_stride_r, void* out,
                           int32_t out_dtype, int64_t out_stride_b, void* stream);

/*
 * Indexer logits over packed fp4 key rows (FreeToken PR 634, "read dsv41 indexer key rows as
 * int32 words": call path Indexer -> indexer_logits_packed; Full mode and candidate mode).
 *   q:        device bf16 [num_tokens][num_heads][128], 16-byte aligned; num_heads must be 32.
 *   weights:  device fp32 [num_tokens][num_heads], 4-byte aligned (per-head weights).
 *   keys:     the index-key pool as an spa_pool_t: kv = packed rows, int32
 *             [num_blocks][page_size][17], 4-byte aligned; k_scale, v_scale unused (NULL).  Row
 *             format fp4_e8m0_b32: words 0..15 hold 128 OCP E2M1 codes (little-endian; byte i
 *             holds element 2i in its low nibble, 2i + 1 in its high nibble), word 16 four OCP
 *             E8M0 scale bytes, byte g scaling elements 32g .. 32g + 31.  Entry j of sequence b is
 *             row block_table[b][j / page_size] * page_size + j % page_size.
 *   positions, seq_of_token (NULL: every query in sequence 0), num_seqs: as for the attention.
 *   ratio:    r >= 1; entry j is causal for a query at position p iff r*j + r - 1 <= p.
 *   cand:     NULL for Full mode (column c scores entry c), else device int32
 *             [num_tokens][num_cols] candidate entries (-1: none).
 *   logits:   device fp32 [num_tokens][num_cols], 4-byte aligned:
 *             logits[t][c] = sum_h w[t][h] * max(0, q[t][h][:] . k[j][:]), or -inf where the
 *             entry is -1, not causal, or its page/block is invalid (which also sets SPA_ERR_INDEX
 *             in the device error word).
 * The logit formula is the reading this library takes (the page gives the key format and the
 * head counts, not the formula).  The keys enter the contraction exactly (every code times its
 * scale is a bf16 value, up to scale bytes of 252; larger products overflow to inf); q . k
 * accumulates in fp32 on the tensor cores, the head sum in fp32.  Returns SPA_ERR_NULL,
 * SPA_ERR_ALIGN, SPA_ERR_SHAPE (negative sizes, ratio < 1, bad pool geometry),
 * SPA_ERR_UNSUPPORTED (num_heads != 32), SPA_ERR_CUDA.  Asynchronous on `stream`; allocates
 * nothing.
 */
int sparse_attn_indexer_logits(const void* q, const float* weights, int32_t num_tokens,
                               int32_t num_heads, const spa_pool_t* keys,
                               const int32_t* positions, const int32_t* seq_of_token,
                               int32_t num_seqs, int32_t ratio, const int32_t* cand,
                               int32_t num_cols, float* logits, void* stream);

/*
 * Top-k selection over indexer logits (the step after sparse_attn_indexer_logits; FreeToken PR 634
 * lists a top-k test beside the logits kernel).  For each query t: the k entries with the largest
 * finite logits[t][c], in decreasing order of logit, ties going to the smaller entry index; -1
 * fills the row when fewer than k logits are finite (infinities and NaN are "not scored").
 * Column c is entry c, or cand[t][c] when cand is given (as for the logits).  -0 and +0 are
 * equal logits.
 *   logits:   device fp32 [num_tokens][num_cols]; cand: device int32 [num_tokens][num_cols] or
 *             NULL; topk_idx: device int32 [num_tokens][k], the attention's top-k list.
 *   k:        0 .. 2048 (SPA_ERR_UNSUPPORTED above).
 * The selection is exact (integer comparisons of the logits' bits and the entry indices).  Returns
 * SPA_ERR_SHAPE for negative sizes, SPA_ERR_NULL, SPA_ERR_ALIGN (4-byte alignment), SPA_ERR_CUDA.
 * Asynchronous on `stream`; allocates nothing.
 */
int sparse_attn_indexer_topk(const float* logits, int32_t num_tokens, int32_t num_cols,
                             const int32_t* cand, int32_t k, int32_t* topk_idx, void* stream);

/* Synchronises `stream`, returns the device error word (an OR of SPA_ERR_INDEX and
 * SPA_ERR_TIMEOUT, 0 if clean) accumulated since the last check on the current device, and
 * clears it.  Returns SPA_ERR_CUDA if the synchronisation itself fails. */
int sparse_attn_paged_check_errors(void* stream);

/* Human-readable name of a status code (static storage). */
const char* sparse_attn_paged_strerror(int status);

/* Message of the last CUDA runtime error seen by this thread (static per-thread storage). */
const char* sparse_attn_paged_last_cuda_error(void);

/* Library version string. */
const char* sparse_attn_paged_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SPARSE_ATTN_PAGED_H */

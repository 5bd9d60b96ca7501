// spa_indexer.h - launch interface of the indexer-logits kernel (spa_indexer.cu), kept apart from
// the attention kernel's headers.
#pragma once

#include "spa_launch.h"

namespace spa {

// Indexer logits over packed fp4_e8m0_b32 key rows (32 heads, head_dim 128).
constexpr int kIdxHeads = 32;
constexpr int kIdxDim = 128;
constexpr int kIdxRowWords = 17;
constexpr int kIdxTile = 128;          // key rows per MMA (M)
constexpr int kIdxMaxQ = 8;            // queries per group (N = 32 per query)
constexpr int kIdxMaxN = kIdxMaxQ * kIdxHeads;
constexpr int kIdxThreads = 128;
struct IndexerArgs {
  const uint16_t* q;            // bf16 [T][32][128]
  const float* w;               // [T][32]
  const int32_t* keys;          // [num_blocks * ps][17]
  const int32_t* bt;            // [B][bt_stride]
  const int32_t* positions;     // [T]
  const int32_t* seq_of_token;  // [T] or NULL (every query in sequence 0)
  const int32_t* cand;          // [T][ncols] (candidate mode) or NULL
  float* logits;                // [T][ncols]
  long long num_blocks;
  long long nunits;             // query groups x key tiles
  int T, B, ps, bt_stride, ratio, ncols;
  int nq;                       // queries per group (1 .. 8)
  int ntiles;                   // key tiles per query group
};
int indexer_smem_bytes(int nq);   // dynamic shared memory of a CTA whose groups hold nq queries
cudaError_t launch_indexer(const IndexerArgs& a, bool cand, int num_sms, cudaStream_t stream);
cudaError_t read_and_clear_indexer_error_word(int* value);

// Top-k selection over the logits rows.
constexpr int kIdxTopkMax = 2048;
struct TopkArgs {
  const float* logits;   // [T][ncols], -inf where no entry was scored
  const int32_t* cand;   // [T][ncols] entry ids of the columns, or NULL (column c is entry c)
  int32_t* topk;         // [T][k]
  long long T;
  int ncols, k;
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream);

}  // namespace spa

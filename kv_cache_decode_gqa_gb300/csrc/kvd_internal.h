// Internal interface between the C ABI layer (api.cu) and the kernel
// translation units: plain parameter structs and launcher functions.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kvd {

// Device error bits (mirrors of the KVD_DEVERR_* values in kvd.h).
enum : int {
  DEVERR_BLOCK = 1,
  DEVERR_POS = 2,
  DEVERR_TIMEOUT = 4,
  DEVERR_INDEX = 8,
  DEVERR_LEN = 16
};

enum : int { DT_BF16 = 0, DT_FP8 = 1, DT_MXFP4 = 2 };

// Bytes of one cached row of d channels.
__host__ __device__ constexpr int row_bytes(int d, int dtype) {
  return dtype == DT_BF16 ? 2 * d : dtype == DT_FP8 ? d : d / 2 + d / 16;
}
// kvd_seqs flags (mirrors of KVD_SEQS_STABLE and KVD_SEQS_PREFIX_READY in
// kvd.h).
enum : int { FLAG_SEQS_STABLE = 1, FLAG_PREFIX_READY = 2 };

struct AppendParams {
  uint8_t *k_cache;  // [num_blocks][n_kv][block_size][head_dim]
  uint8_t *v_cache;  // may be null (K-only)
  const float *k_inv_scale;
  const float *v_inv_scale;
  const int32_t *block_table;
  const int32_t *pos;
  const uint16_t *k_new;  // bf16 [batch][n_kv][head_dim]
  const uint16_t *v_new;
  int32_t num_blocks, block_size, n_kv, head_dim, dtype;
  int32_t max_blocks, batch;
  int *err;
};

// One decode launch over a paged cache (dense, MLA or gathered positions).
struct DecodeParams {
  const uint8_t *k;  // cache base pointers
  const uint8_t *v;  // == k for a latent cache (values are the first dv dims)
  const float *k_scale;
  const float *v_scale;
  const int32_t *block_table;
  const int32_t *seq_lens;
  const int32_t *indices;  // gathered positions (sparse), else null
  const uint16_t *q;       // bf16 [batch][n_h][dk]
  uint16_t *out;           // bf16 [batch][n_h][dv]
  float *lse;              // [batch][n_h] or null
  float *ws_o;             // partials [batch][n_h][n_splits][dv]
  float *ws_lse;           // partials [batch][n_h][n_splits]
  int32_t n_groups;        // head groups (tiles) per sequence
  int32_t batch, n_h, n_kv, dk, dv, block_size, num_blocks, max_blocks;
  int32_t dtype;        // DT_BF16, DT_FP8 or DT_MXFP4
  int32_t max_seq_len;  // clamp for device lengths
  int32_t n_idx;        // entries per row of `indices`
  int32_t split_len;    // tokens (or index entries) per split
  int32_t n_splits;
  // dense GQA only: 1 when CTA c takes unit c (sequence c / units per
  // sequence, head group c % units) whole instead of an equal share of all
  // chunks: no partials and no merge launch (units all short, see the plan)
  int32_t whole_units;
  // CUDA-core dense GQA only: > 1 when the units of a single sequence run
  // as clusters of this many CTAs, each an equal part of its unit, whose
  // partials merge in distributed shared memory (no merge launch)
  int32_t cluster;
  int32_t hp;           // kv heads per work unit (CUDA-core GQA kernel)
  int32_t flags;        // kvd_seqs flags (FLAG_SEQS_STABLE, FLAG_PREFIX_READY)
  // sliding window (dense GQA only): sequence b attends to positions
  // [max(win_start[b], len_b - window), len_b); window 0 and no starts:
  // every visible position
  int32_t window;
  const int32_t *win_start;
  // fused append (kvd_gqa_append_decode), else pos == nullptr: the new key
  // and value rows, bf16 [batch][n_kv][dk], written at slot pos[b]
  const int32_t *pos;
  const uint16_t *k_new;
  const uint16_t *v_new;
  const float *k_inv_scale;
  const float *v_inv_scale;
  float scale_log2;  // softmax scale * log2(e)
  int *err;
};

struct IndexerParams {
  const uint8_t *cache;  // indexer key cache [num_blocks][1][block_size][64]
  const int32_t *block_table;
  const int32_t *seq_lens;
  const uint16_t *q;  // bf16 [batch][n_heads][64]
  const float *w;     // [batch][n_heads]
  float *scores;      // [batch][score_stride]
  int32_t *indices;   // [batch][k]
  int32_t batch, n_heads, block_size, num_blocks, max_blocks, max_seq_len;
  int32_t score_stride, topk;
  // pool mode (a Reindex layer of the hierarchical indexer), else null: the
  // scored entries are the positions of the pool's 8-position blocks,
  // entry e = position 8 pool[b][e / 8] + e % 8, scores and top-k indexed
  // by entry, the selection mapped back to positions
  const int32_t *pool;    // [batch][kPoolBlocks] ascending block ids
  const int32_t *pool_n;  // [batch] blocks in the pool
  int32_t max_entries;    // launch sizing: max_seq_len, or 8 * kPoolBlocks
  int32_t flags;          // kvd_seqs flags (scores: honoured without a pool)
  int *err;
};

// The hierarchical indexer's pool: at most 2,048 blocks of 8 positions.
constexpr int kPoolBlocks = 2048;
constexpr int kPoolBlock = 8;

struct PoolParams {
  const int32_t *indices;  // [batch][k] a Full layer's selection
  const int32_t *seq_lens;
  int32_t *pool;    // [batch][kPoolBlocks]
  int32_t *pool_n;  // [batch]
  int32_t batch, k, max_seq_len;
  int *err;
};

// Count one kernel launch of the library (kvd_launch_count, api.cu).
void note_launch();

// Launchers. Each returns the launch error (cudaSuccess if queued).
cudaError_t launch_append(const AppendParams &p, cudaStream_t s);
// The pool of a Full layer's selection (one CTA per sequence).
cudaError_t launch_indexer_pool(const PoolParams &p, cudaStream_t s);
// Dense GQA/MHA, CUDA cores (group size <= 4).
cudaError_t launch_decode_simt(const DecodeParams &p, cudaStream_t s);
// kv heads the CUDA-core kernel takes per work unit for these shapes (its
// plan and its launch must agree).
// CTAs per unit (2..8) of a cluster-merged CUDA-core decode of one sequence
// (query groups of 1) whose `units` clusters are all resident at once on
// `sms` SMs; 0 when no size fits.
int simt_cluster_size(int head_dim, int dtype, int hp, int units, int sms);
int simt_heads_per_stage(int n_kv, int g, int head_dim, int dtype,
                         int block_size);
// Dense GQA on the tensor cores (group size 8 or 16, head_dim 128).
cudaError_t launch_decode_mma(const DecodeParams &p, int dtype,
                              cudaStream_t s);
// kv heads the tensor-core kernel takes per work unit (its plan and its
// launch must agree).
int mma_heads_per_unit(int n_kv, int block_size, int dtype);
// MLA latent decode (dk 576, dv 512, n_h multiple of 64), CUDA-core MMAs.
cudaError_t launch_decode_mla(const DecodeParams &p, cudaStream_t s);
// The same on tcgen05 tensor cores (n_h multiple of 128, block_size a
// multiple of 64): 64-position chunks, n_h / 32 CTAs per lane of
// n_splits / (n_h / 64).
constexpr int kLatentTcRows = 64;
// value parts of the tcgen05 latent decode: CTAs of a lane per 128-head tile
constexpr int kLatentTcParts = 2;
bool latent_tc_supported(int n_h, int block_size, long num_blocks);
cudaError_t launch_decode_mla_tc(const DecodeParams &p, cudaStream_t s);
// Log-sum-exp merge of the latent decode's split units (chunks of `rows`
// positions: 32 for the CUDA-core kernel, 64 for the tensor-core one).
cudaError_t launch_merge_mla(const DecodeParams &p, int rows, cudaStream_t s);
// Gathered-position decode (dk = dv = 512, n_kv 1, n_h multiple of 64) on
// tcgen05: n_splits = CTAs per (sequence, 64-head tile), as
// gather_tc_splits plans them (`forced` > 0: that many CTAs in all).
constexpr int kGatherMaxSplits = 32;
int gather_tc_splits(int units, int k, int sms, int forced);
cudaError_t launch_decode_sparse_tc(const DecodeParams &p, cudaStream_t s);
cudaError_t launch_indexer_scores(const IndexerParams &p, cudaStream_t s);
cudaError_t launch_topk(const IndexerParams &p, cudaStream_t s);

}  // namespace kvd

#include "kvd.h"

namespace kvd {
// Workspace bytes of a gqa_decode call, its arguments validated (api.cu).
kvd_status gqa_workspace_bytes(const kvd_cache *cache, const kvd_seqs *seqs,
                               int32_t n_h, size_t *total);

// Record `msg` as this host thread's last error and return `st` (api.cu).
kvd_status set_error(kvd_status st, const char *msg);
// The current device's error word (KVD_DEVERR_* bits), for kernels that
// flag bad inputs.
kvd_status device_error_word(int **err);

// Split plans (shared by workspace sizing and the calls).
constexpr int kStageRows = 64;  // tokens per pipeline stage (dense paths)

}  // namespace kvd

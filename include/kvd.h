/*
 * kvd.h -- C ABI of libkvd.so: one decode step of attention over a paged KV
 * cache on one GB300 (sm_103a) GPU.
 *
 * What is computed (pages cited by title and section):
 *   "KV cache" (this.guide), "A cache you keep because attention looks
 *   backwards": at decode step t the new token's query attends over the keys
 *   and values of every position up to and including t,
 *       o_t = softmax(q_t K^T * scale) V,   scale = 1/sqrt(d_h) by default,
 *   and the keys and values of earlier positions are read from a cache
 *   instead of being recomputed. "Two tensors per layer": per sequence and
 *   layer the cache is K and V, each [n_kv, L, d_h].
 *
 * Conventions shared by every call:
 *   - Every pointer argument that names tensor data is DEVICE memory owned by
 *     the caller. The library allocates no device memory, frees none and
 *     never synchronises the device (kvd_device_error is the one exception).
 *     The copy-on-write block pool (kvd_block_pool_*) is the one host object:
 *     it owns host memory for its counts and takes HOST arrays.
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream). Outputs are valid once the stream reaches
 *     that point.
 *   - Arguments are validated on the host before anything is launched; a
 *     call that returns anything but KVD_OK launched nothing (except
 *     KVD_ERR_CUDA, which reports a failed launch). kvd_last_error() then
 *     describes the problem in words (per host thread).
 *   - Device-resident values (block table entries, positions, lengths,
 *     top-k indices) cannot be checked on the host. Kernels check them and,
 *     instead of touching memory out of bounds, skip the access and set a
 *     bit in the library's device error word (KVD_DEVERR_*), which
 *     kvd_device_error() reads.
 *   - No exception crosses this boundary.
 *
 * Workspace: the decode calls split each sequence into runs of positions
 * processed by separate CTAs and merge the partial results (log-sum-exp
 * merge). The caller passes the scratch for the partials: at least
 * kvd_workspace_size() bytes, 256-byte aligned; nothing in it needs to
 * start at zero. Every partial result a call keeps there is written before
 * the call reads it, so a workspace can be reused by later calls on the
 * same stream without clearing; two calls that may run at the same time
 * need two workspaces. A GQA decode whose (sequence, head group) units are
 * all short -- a window (kvd_seqs.window) of at most 192 positions, or a
 * longest visible length of at most 256 -- and no more numerous than the
 * device's SMs runs each unit whole on one CTA and needs no workspace
 * (kvd_workspace_size returns 0; NULL is then accepted). Neither does a
 * single sequence with one query head per kv head (MHA) whose units run as
 * thread-block clusters merging their parts in distributed shared memory
 * (units of at most two heads, when the clusters fill most of the SMs).
 *
 * Paged layout ("KV cache", "The allocator, not the algorithm"; the paging
 * of the My Weird Prompts 640482 transcript): a cache is a pool of fixed-size
 * blocks, each holding `block_size` consecutive positions of one sequence,
 *     element (block, kv_head, slot, i) at
 *     ((block * n_kv + kv_head) * block_size + slot) * head_dim + i,
 * and a per-sequence block table maps logical block j (positions
 * [j*block_size, (j+1)*block_size)) to a physical block. Block tables may
 * alias physical blocks (shared prefixes are read-only here).
 */
#ifndef KVD_H
#define KVD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVD_VERSION 1

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st *kvd_stream;

typedef enum kvd_status {
  KVD_OK = 0,
  KVD_ERR_NULL = 1,        /* a required pointer is NULL                     */
  KVD_ERR_SHAPE = 2,       /* inconsistent sizes, or a pointer misaligned    */
  KVD_ERR_UNSUPPORTED = 3, /* head size / group size / dtype not compiled in */
  KVD_ERR_CAPACITY = 4,    /* a host-visible length exceeds the block table  */
  KVD_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than required        */
  KVD_ERR_CUDA = 6         /* a CUDA runtime call or launch failed           */
} kvd_status;

/* Bits of the device error word. */
#define KVD_DEVERR_BLOCK 1   /* a block table entry outside [0, num_blocks)   */
#define KVD_DEVERR_POS 2     /* an append position outside the block table    */
#define KVD_DEVERR_TIMEOUT 4 /* a bounded wait on a copy gave up               */
#define KVD_DEVERR_INDEX 8   /* a top-k index >= that sequence's length        */
#define KVD_DEVERR_LEN 16    /* a sequence length above the block table, or
                                above the max_seq_len the call was given      */

typedef enum kvd_dtype {
  KVD_BF16 = 0,     /* 2-byte bfloat16 elements                              */
  KVD_FP8_E4M3 = 1, /* 1-byte OCP E4M3 codes; value = code * per-head scale  */
  KVD_MXFP4 = 2     /* rows of E2M1 codes + one E4M3 scale per 16 channels   */
} kvd_dtype;

/*
 * One layer's cache. Layout [num_blocks][n_kv][block_size][head_dim] for K
 * and for V. `v` is NULL for a K-only cache (the MLA latent cache and the
 * indexer key cache). Both base pointers must be 16-byte aligned.
 *
 * fp8 ("KV cache", "Fewer bits per number": halving the element size
 * halves the cache and doubles arithmetic intensity): one fp32 scale per
 * (layer, kv head) for K and one for V. A stored code c means c * scale;
 * kvd_kv_append stores E4M3(x * inv_scale) rounded to nearest even and
 * saturated to +-448. Scale arrays are device memory, [n_kv] each; unused
 * (may be NULL) for bf16 caches.
 */
/*
 * mxfp4 ("890 bytes a token ...", section 6: E2M1 with one E4M3 scale per
 * 16 channels, NVFP4's layout without the second-level global scale, so
 * the largest value is 448 x 6 = 2688). A row of head_dim channels is
 * head_dim/2 bytes of E2M1 codes (OCP MX FP4: 1 sign, 2 exponent, 1
 * mantissa bit; channel 2j in the low nibble of byte j, 2j+1 in the high
 * one) followed by head_dim/16 E4M3 scale codes (scale g covers channels
 * 16g..16g+15): 72 bytes for head_dim 128, where K and V are laid out
 * [num_blocks][n_kv][block_size][72] bytes. Value = code value * scale
 * value. kvd_kv_append (and kvd_gqa_append_decode) encode each group of a
 * new bf16 row as: amax = max |x| (fp32), scale = E4M3(amax / 6), code =
 * E2M1(x / scale), both divisions in fp32 and both conversions round to
 * nearest even and saturate; a group whose scale rounds to 0 stores zero
 * codes. Quantise after RoPE: the library stores what it is given. The
 * scale pointers are unused. Supported: head_dim 128, an even block_size,
 * kv_append and GQA decode with n_h / n_kv of 1, 2 or 4 (dequantised in the
 * CUDA-core decode kernel; there is no fp4 MMA).
 */
typedef struct kvd_cache {
  void *k;
  void *v;
  int32_t num_blocks;
  int32_t block_size;
  int32_t n_kv;
  int32_t head_dim;
  int32_t dtype; /* kvd_dtype */
  int32_t reserved;
  const float *k_scale;
  const float *v_scale;
  const float *k_inv_scale;
  const float *v_inv_scale;
} kvd_cache;

/*
 * The batch of sequences being decoded.
 *   block_table   device [batch][max_blocks_per_seq] int32 physical block ids
 *   seq_lens      device [batch] int32: positions visible to this step's
 *                 query, i.e. the cached length AFTER this step's append
 *   max_seq_len   host: an upper bound on every seq_lens[b]; sizes the split
 *                 plan and the workspace. Must be <= max_blocks_per_seq *
 *                 block_size (else KVD_ERR_CAPACITY). A device length above
 *                 it is clamped to it and flagged KVD_DEVERR_LEN.
 *   flags         0, KVD_SEQS_STABLE, or KVD_SEQS_STABLE |
 *                 KVD_SEQS_PREFIX_READY (other bits: KVD_ERR_SHAPE)
 *   window        0 (every visible position), or W > 0: sliding-window
 *                 decode ("890 bytes a token", section 7, SWA bounded
 *                 replay, n_win = 128; "KV cache" on local-attention
 *                 layers): the query of sequence b, at position
 *                 seq_lens[b] - 1, attends to the positions
 *                 [max(s_b, seq_lens[b] - W), seq_lens[b]) only
 *   window_start  device int32 [batch] replay starts s_b, or NULL (s_b = 0);
 *                 read like seq_lens (KVD_SEQS_STABLE covers it too)
 * window and window_start are honoured by kvd_gqa_decode,
 * kvd_gqa_append_decode and kvd_gqa_decode_noalloc; the other calls need
 * window == 0 and window_start == NULL (else KVD_ERR_UNSUPPORTED).
 *
 * Kernels of this library may start while the kernel before them on the
 * stream is still running (programmatic dependent launch); they read their
 * inputs only after that kernel has completed. KVD_SEQS_STABLE declares that
 * block_table and seq_lens (and, for kvd_gqa_append_decode, pos) already
 * hold their final values when the kernel launched just before this call
 * starts, and that no kernel still running writes them (for example: they
 * are set by host copies at the start of a decode step and read by every
 * layer). kvd_gqa_decode, kvd_gqa_append_decode and kvd_indexer_topk then
 * read them, and plan their work, while that kernel finishes. Other calls
 * ignore the flag.
 *
 * KVD_SEQS_PREFIX_READY (only with KVD_SEQS_STABLE) declares as well that
 * every cache row the call reads at a position below seq_lens[b] - 1
 * already holds its final value when the kernel launched just before this
 * call starts, and that no kernel still running writes it: only the newest
 * position, seq_lens[b] - 1, may be written by that kernel (a kv_append of
 * this step), or by kvd_gqa_append_decode itself. That holds in a decode
 * step, where older rows were appended by earlier steps; it does not hold
 * right after kvd_copy_blocks, which writes older rows. kvd_gqa_decode,
 * kvd_gqa_append_decode and kvd_indexer_topk may then start copying those
 * rows while that kernel finishes (the query rows, and everything written,
 * still wait for it); the CUDA-core decode kernel (query groups of 1, 2 or
 * 4) and the indexer's scores do. Other calls ignore the flag.
 */
#define KVD_SEQS_STABLE 1
#define KVD_SEQS_PREFIX_READY 2
typedef struct kvd_seqs {
  const int32_t *block_table;
  const int32_t *seq_lens;
  int32_t batch;
  int32_t max_blocks_per_seq;
  int32_t max_seq_len;
  int32_t flags;
  int32_t window;
  const int32_t *window_start;
} kvd_seqs;

typedef enum kvd_op {
  KVD_OP_GQA_DECODE = 0,
  KVD_OP_MLA_DECODE = 1,
  KVD_OP_INDEXER_TOPK = 2,
  KVD_OP_SPARSE_DECODE = 3,
  KVD_OP_INDEXER_TOPK_POOL = 4
} kvd_op;

/*
 * kvd_kv_append -- write this step's new key (and value) of every sequence
 * into the cache. The My Weird Prompts 640482 transcript, on decode: each
 * new token computes its own query, key and value, and its key and value
 * are appended, so the cache grows by one entry per layer per token.
 *
 *   cache          the layer's cache (K-only when cache->v is NULL)
 *   block_table    device [batch][max_blocks_per_seq]
 *   pos            device [batch]: the slot (logical position) to write,
 *                  normally the cached length before this step
 *   k_new, v_new   device bf16 [batch][n_kv][head_dim]; v_new is ignored
 *                  (may be NULL) for a K-only cache and required otherwise
 * bf16 caches receive the bytes unchanged; fp8 caches receive
 * E4M3_rne_satfinite(float(x) * inv_scale[kv_head]); MXFP4 caches receive
 * each 16-channel group encoded as described at kvd_cache.
 * Errors: KVD_ERR_NULL, KVD_ERR_SHAPE (batch < 0, head_dim not a multiple of
 * 8, misaligned pointer), KVD_ERR_UNSUPPORTED (dtype). A position or block id
 * out of range on the device skips that row and sets KVD_DEVERR_POS /
 * KVD_DEVERR_BLOCK.
 */
kvd_status kvd_kv_append(const kvd_cache *cache, const int32_t *block_table,
                         int32_t max_blocks_per_seq, const int32_t *pos,
                         int32_t batch, const void *k_new, const void *v_new,
                         kvd_stream stream);

/*
 * kvd_gqa_decode -- grouped-query attention for one decode step ("KV cache",
 * "Fewer KV heads, held at the same quality": n_h query heads in n_kv groups,
 * one KV head per group; MHA is n_kv == n_h and MQA is n_kv == 1). Query
 * head h reads KV head h / (n_h / n_kv).
 *
 *   q         device bf16 [batch][n_h][head_dim]
 *   scale     softmax scale; <= 0 selects 1/sqrt(head_dim)
 *   out       device bf16 [batch][n_h][head_dim]
 *   lse       device fp32 [batch][n_h], natural-log log-sum-exp of the
 *             scaled scores (-inf for an empty sequence); may be NULL
 *   workspace device scratch of at least kvd_workspace_size(KVD_OP_GQA_DECODE)
 *             bytes, 256-byte aligned (see "Workspace" above)
 * Supported: bf16 or fp8 cache, head_dim 64 or 128, n_h / n_kv in
 * {1, 2, 4, 8, 16} (8 and 16 need head_dim 128 and a block_size that is a
 * multiple of 64 or one of 16, 32); an MXFP4 cache with head_dim 128 and
 * n_h / n_kv of 1, 2 or 4; at most 1024 sequences per call. An empty
 * sequence gives out = 0 and lse = -inf.
 */
kvd_status kvd_gqa_decode(const kvd_cache *cache, const kvd_seqs *seqs,
                          const void *q, int32_t n_h, float scale, void *out,
                          float *lse, void *workspace, size_t workspace_bytes,
                          kvd_stream stream);

/*
 * kvd_gqa_append_decode -- kvd_kv_append(cache, seqs->block_table,
 * seqs->max_blocks_per_seq, pos, seqs->batch, k_new, v_new) followed by
 * kvd_gqa_decode(cache, seqs, q, ...), done in the decode's own pass over
 * the cache: the CTA that copies the chunk holding pos[b] writes sequence
 * b's new key and value rows just before it copies that chunk, and rows no
 * chunk reads (pos[b] at or past the visible length) are written by one
 * CTA. The My Weird Prompts 640482 transcript: the new token's key and value
 * join the cache, and its query attends to the cache including them.
 *
 *   pos, k_new, v_new   as for kvd_kv_append (v_new required)
 *   other arguments     as for kvd_gqa_decode; the same workspace size
 * Cache contents, out and lse equal those of the two separate calls. The
 * slot written for sequence b must not be visible to another sequence of
 * the call (no two sequences share the block that receives a new row).
 * Errors: those of both calls (KVD_ERR_NULL when pos is NULL and batch > 0);
 * a position or block id out of range on the device is skipped and flagged
 * as kvd_kv_append does.
 */
kvd_status kvd_gqa_append_decode(const kvd_cache *cache, const kvd_seqs *seqs,
                                 const int32_t *pos, const void *k_new,
                                 const void *v_new, const void *q, int32_t n_h,
                                 float scale, void *out, float *lse,
                                 void *workspace, size_t workspace_bytes,
                                 kvd_stream stream);

/*
 * kvd_gqa_decode_noalloc -- kvd_gqa_decode for callers that cannot allocate
 * device memory. (The pages have no counterpart of this call; it exists for
 * how the library is embedded, not for what it computes.)
 *
 * kvd_gqa_decode needs scratch memory for its split-K partial results, which
 * its caller normally allocates and passes as `workspace`. Some callers
 * cannot do that: a plug-in loaded into a host program that owns every
 * device allocation and gives it no allocator, or a latency-critical path
 * that must not call cudaMalloc (an allocation can synchronise the device).
 * This variant takes only inputs and outputs and uses a scratch array
 * compiled into the library: KVD_NOALLOC_SCRATCH_BYTES (16 MiB) of device
 * memory that every GPU which loads the library holds until the process
 * exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   Arguments, results and supported shapes are those of kvd_gqa_decode.
 *   Shapes whose workspace (kvd_workspace_size) exceeds the array return
 *   KVD_ERR_WORKSPACE and launch nothing.
 *   The first call on each device looks up the array's device address with
 *   that device current; make that first call before any stream capture.
 *   Every call uses the same array, and it keeps the last call's contents
 *   (nothing in it needs to start at zero: each call writes every partial
 *   result before reading it).
 *   Calls whose work can overlap on the GPU -- on different streams or from
 *   different host threads -- race on the array and give wrong results;
 *   serialise them, or use kvd_gqa_decode with separate workspaces.
 */
#define KVD_NOALLOC_SCRATCH_BYTES (16u << 20)
kvd_status kvd_gqa_decode_noalloc(const kvd_cache *cache,
                                  const kvd_seqs *seqs, const void *q,
                                  int32_t n_h, float scale, void *out,
                                  float *lse, kvd_stream stream);

/*
 * kvd_mla_decode -- decode against a latent cache ("KV cache", "Caching a
 * compressed latent instead of the keys", and the MLA footnote of "Where the
 * memory actually goes": one latent c of d_c dims plus one shared positional
 * key of head_dim - d_c dims per token and layer). The key up-projection is
 * folded into the query ahead of time, so scores run directly against the
 * cached rows, and the output stays in latent space:
 *     s_t = scale * (q_lat . c_t + q_rope . k_rope_t),  out = softmax(s) . c
 *
 *   latent    K-only bf16 cache with n_kv = 1, head_dim = d_c + d_rope
 *   q         device bf16 [batch][n_h][head_dim] = [q_lat | q_rope]
 *   out       device bf16 [batch][n_h][d_c]
 *   lse       device fp32 [batch][n_h] or NULL
 *   workspace at least kvd_workspace_size(KVD_OP_MLA_DECODE) bytes (see
 *             "Workspace" above)
 * Supported: d_c = 512, head_dim = 576, n_h a multiple of 64, at most 256
 * sequences per call.
 */
kvd_status kvd_mla_decode(const kvd_cache *latent, int32_t d_c,
                          const kvd_seqs *seqs, const void *q, int32_t n_h,
                          float scale, void *out, float *lse, void *workspace,
                          size_t workspace_bytes, kvd_stream stream);

/*
 * kvd_indexer_topk -- score every visible cached position with the indexer
 * and select the top k (the My Weird Prompts 640482 transcript on DeepSeek
 * Sparse Attention: a lightning indexer scores the prefix and a top-k subset,
 * k = 2048, is read; "890 bytes a token", section 3: Full and Reindex layers
 * score with their own indexer query over a shared indexer key cache):
 *     s_t = sum_j w[j] * max(0, q_idx[j] . k_t),   t < seq_lens[b]
 *
 *   index_cache  K-only bf16 cache, n_kv = 1, head_dim = d_idx (64)
 *   q_idx        device bf16 [batch][n_idx_heads][d_idx]
 *   w            device fp32 [batch][n_idx_heads]
 *   indices      device int32 [batch][k]: the k positions with the largest
 *                scores (computed in fp32), equal scores going to the lower
 *                position, in ascending position order; -1 pads when fewer
 *                than k positions are visible
 *   scores       device fp32 [batch][max_seq_len] or NULL: if given, the
 *                scores the selection used (entries >= seq_lens[b] are
 *                unspecified)
 *   workspace    when scores is NULL: at least
 *                kvd_workspace_size(KVD_OP_INDEXER_TOPK) bytes (the scores)
 * Supported: d_idx = 64, n_idx_heads <= 8, 1 <= k <= 16384.
 */
kvd_status kvd_indexer_topk(const kvd_cache *index_cache, const kvd_seqs *seqs,
                            const void *q_idx, int32_t n_idx_heads,
                            const float *w, int32_t k, int32_t *indices,
                            float *scores, void *workspace,
                            size_t workspace_bytes, kvd_stream stream);

/*
 * The hierarchical indexer ("890 bytes a token", section 4; the My Weird
 * Prompts 640482 transcript on CSA2): the first Full layer publishes the
 * blocks its selection came from as a candidate pool of at most 2,048
 * blocks of 8 positions (16,384 candidates), and later Reindex layers
 * select only from that pool, so their cost is bounded by the pool, not by
 * the context length.
 */
#define KVD_POOL_BLOCKS 2048 /* blocks a pool holds                         */
#define KVD_POOL_BLOCK 8     /* positions per pool block                    */

/*
 * kvd_indexer_pool -- the pool of a selection.
 *   indices  device int32 [batch][k]: positions in any order; entries < 0
 *            are skipped, and so are entries >= seq_lens[b] (flagged
 *            KVD_DEVERR_INDEX)
 *   pool     device int32 [batch][KVD_POOL_BLOCKS], written: the ascending
 *            ids (position / 8) of the blocks holding a selected position,
 *            the lowest KVD_POOL_BLOCKS when there are more; entries past
 *            pool_n[b] are unspecified
 *   pool_n   device int32 [batch], written: the blocks in each pool
 * Reads seqs->seq_lens only (not the block table). Supported: k >= 1,
 * max_seq_len <= 50,331,648.
 */
kvd_status kvd_indexer_pool(const kvd_seqs *seqs, const int32_t *indices,
                            int32_t k, int32_t *pool, int32_t *pool_n,
                            kvd_stream stream);

/*
 * kvd_indexer_topk_pool -- a Reindex layer over a pool: the indexer scores
 * of the pool's candidates only (positions 8 * pool[b][i] + j, j < 8, that
 * are below seq_lens[b]), and the top k of them, selected as
 * kvd_indexer_topk selects (fp32 scores, equal scores to the lower
 * position, ascending positions, -1 padding).
 *   pool, pool_n  device, as kvd_indexer_pool writes them
 *   scores        device fp32 [batch][KVD_POOL_BLOCKS * 8] or NULL: if
 *                 given, the candidate scores by pool entry (entry e is
 *                 position 8 * pool[b][e / 8] + e % 8; entries at or past
 *                 seq_lens[b] are -inf, entries past 8 * pool_n[b]
 *                 unspecified)
 *   workspace     when scores is NULL: at least
 *                 kvd_workspace_size(KVD_OP_INDEXER_TOPK_POOL) bytes
 * Other arguments as for kvd_indexer_topk, and block_size a multiple of 8.
 */
kvd_status kvd_indexer_topk_pool(const kvd_cache *index_cache,
                                 const kvd_seqs *seqs, const void *q_idx,
                                 int32_t n_idx_heads, const float *w,
                                 const int32_t *pool, const int32_t *pool_n,
                                 int32_t k, int32_t *indices, float *scores,
                                 void *workspace, size_t workspace_bytes,
                                 kvd_stream stream);

/*
 * kvd_sparse_decode -- GQA decode restricted to given positions ("890 bytes
 * a token", section 3: a Reuse layer attends to the selection an earlier
 * layer computed; the transcript: sparse attention changes which stored
 * positions are read).
 *
 *   indices  device int32 [batch][k] positions; entries < 0 are skipped, and
 *            so are entries >= seq_lens[b] (flagged KVD_DEVERR_INDEX)
 *   q, out, lse, scale as for kvd_gqa_decode
 *   workspace at least kvd_workspace_size(KVD_OP_SPARSE_DECODE, ..., k)
 *            bytes (see "Workspace" above)
 * Supported: bf16 cache with n_kv = 1, head_dim = 512, n_h a multiple of 64,
 * at most 256 sequences per call.
 */
kvd_status kvd_sparse_decode(const kvd_cache *cache, const kvd_seqs *seqs,
                             const int32_t *indices, int32_t k, const void *q,
                             int32_t n_h, float scale, void *out, float *lse,
                             void *workspace, size_t workspace_bytes,
                             kvd_stream stream);

/*
 * Copy-on-write block pool ("KV cache", "The allocator, not the
 * algorithm": block tables of sequences with a common prefix point at the
 * same physical blocks, copied when they diverge; each sequence wastes at
 * most block_size - 1 slots of its last block). A host object: reference
 * counts of num_blocks physical block ids and their free list (the lowest
 * free id is handed out first). Thread-safe; block tables and id arrays
 * passed to it are HOST memory. Errors: KVD_ERR_NULL, KVD_ERR_SHAPE (bad
 * ids, over-release), KVD_ERR_CAPACITY (pool exhausted); a failing call
 * changes nothing.
 */
typedef struct kvd_block_pool kvd_block_pool;

kvd_status kvd_block_pool_create(int32_t num_blocks, kvd_block_pool **out);
void kvd_block_pool_destroy(kvd_block_pool *pool);
/* free blocks, or -1 for a NULL pool */
int32_t kvd_block_pool_free_count(kvd_block_pool *pool);
/* references held on a block (0 = free), or -1 for a bad id */
int32_t kvd_block_pool_refcount(kvd_block_pool *pool, int32_t block);
/* n fresh blocks (reference count 1) into blocks[0..n) */
kvd_status kvd_block_pool_alloc(kvd_block_pool *pool, int32_t n,
                                int32_t *blocks);
/* one more reference on each held block (a fork sharing a prefix); ids < 0
 * are skipped */
kvd_status kvd_block_pool_share(kvd_block_pool *pool, const int32_t *blocks,
                                int32_t n);
/* one reference fewer on each block; a block reaching 0 is free again */
kvd_status kvd_block_pool_release(kvd_block_pool *pool, const int32_t *blocks,
                                  int32_t n);
/*
 * Before appending at slot pos[b] of each sequence: a table entry that is
 * -1 gets a fresh block; one that names a block with other references gets
 * a fresh block too, and the pair (old, fresh) goes to src / dst
 * [*n_copies] so that kvd_copy_blocks can copy the shared rows first (the
 * table drops its reference on the old block). block_table is HOST int32
 * [batch][max_blocks], updated in place; src and dst hold up to batch ids.
 */
kvd_status kvd_block_pool_prepare_append(kvd_block_pool *pool,
                                         int32_t *block_table, int32_t batch,
                                         int32_t max_blocks,
                                         const int32_t *pos,
                                         int32_t block_size, int32_t *src,
                                         int32_t *dst, int32_t *n_copies);
/* device: whole blocks dst[i] := src[i] of K and V (every kv head's rows),
 * src / dst DEVICE int32 [n]. The copies run in parallel: the dst ids must be
 * distinct and none may be a src of the same call (kvd_block_pool_prepare_
 * append's pairs meet this, every dst being a fresh block). An id outside
 * [0, num_blocks) skips that copy and sets KVD_DEVERR_BLOCK. Host errors,
 * before any launch: KVD_ERR_NULL (no cache, or src / dst NULL with n > 0),
 * KVD_ERR_SHAPE (n < 0, n > 65535, or a block not a multiple of 16 bytes);
 * KVD_ERR_CUDA if a launch fails. n = 0 does nothing. */
kvd_status kvd_copy_blocks(const kvd_cache *cache, const int32_t *src,
                           const int32_t *dst, int32_t n, kvd_stream stream);

/*
 * kvd_workspace_size -- bytes of workspace the call `op` needs for these
 * shapes on the current device (the split plan depends on its SM count,
 * and for a GQA decode on `seqs`->window as well, so pass the window the
 * call will use).
 * `n_h` is the query head count (indexer heads for KVD_OP_INDEXER_TOPK) and
 * `k` the top-k size (0 where unused). Queries the device; KVD_ERR_CUDA if
 * there is none.
 */
kvd_status kvd_workspace_size(kvd_op op, const kvd_cache *cache,
                              const kvd_seqs *seqs, int32_t n_h, int32_t k,
                              size_t *bytes);

/*
 * kvd_bytes_per_token -- cache bytes per token ("KV cache", "The size
 * formula"): 2 tensors x n_l layers x n_kv heads x d_h x elem_bytes.
 */
uint64_t kvd_bytes_per_token(int32_t n_l, int32_t n_kv, int32_t d_h,
                             int32_t elem_bytes);

/* Text for a status code, and the last error of this host thread. */
const char *kvd_status_string(kvd_status status);
const char *kvd_last_error(void);

/*
 * kvd_device_error -- synchronise the current device, then read and clear
 * the device error word (KVD_DEVERR_* bits; 0 means no error).
 */
kvd_status kvd_device_error(int32_t *code);

int32_t kvd_version(void);

/*
 * kvd_set_tuning -- process-wide overrides of the library's launch choices,
 * for tests and experiments (the pages have no counterpart).
 *   decode_ctas     > 0: every decode launch uses this many CTAs (the split
 *                   plan and kvd_workspace_size follow it); 0: the default,
 *                   one per SM
 *   mla_cuda_cores  != 0: kvd_mla_decode runs its CUDA-core kernel even
 *                   where the tcgen05 kernel applies; 0: the default
 * Their starting values come from the environment variables
 * KVD_DECODE_CTAS and KVD_MLA_CUDA_CORES, read once when the library is
 * loaded. A workspace sized before a change may be too small after it.
 * Errors: KVD_ERR_SHAPE (decode_ctas < 0).
 */
kvd_status kvd_set_tuning(int32_t decode_ctas, int32_t mla_cuda_cores);

/*
 * kvd_launch_count -- kernels this library has launched in this process so
 * far (every device and host thread). A launch recorded into a CUDA graph
 * under stream capture counts once, when it is recorded, so the count
 * across a capture is the kernels one replay runs. A diagnostic for
 * counting a step's kernels; the pages have no counterpart.
 */
uint64_t kvd_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* KVD_H */

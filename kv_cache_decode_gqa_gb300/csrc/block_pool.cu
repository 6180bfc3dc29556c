// Copy-on-write block pool for prefix sharing ("KV cache", section "The
// allocator, not the algorithm": blocks are indirected, so sequences with a
// common prefix point their block tables at the same physical blocks, with
// copy-on-write when they diverge; parallel sampling, beam search and shared
// system prompts stop duplicating memory).
//
// Host side: a pool of num_blocks physical blocks with a reference count
// each and a free list (lowest ids first, so a fresh pool hands out
// 0, 1, 2, ...). Device side: one launch copies whole blocks (every kv head's
// rows, K and V) for the copies an append step needs.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "kvd.h"
#include "kvd_common.cuh"

struct kvd_block_pool {
  std::mutex mu;
  std::vector<int32_t> refs;   // reference count per block
  std::vector<int32_t> free_;  // free block ids, largest last-popped first
};

namespace {

// free_ is kept sorted descending so that back() is the lowest free id
void push_free(kvd_block_pool *p, int32_t b) {
  auto it = std::lower_bound(p->free_.begin(), p->free_.end(), b,
                             [](int32_t a, int32_t v) { return a > v; });
  p->free_.insert(it, b);
}

bool valid_block(const kvd_block_pool *p, int32_t b) {
  return b >= 0 && b < (int32_t)p->refs.size();
}

// Whole blocks of one tensor: block dst[i] := block src[i], 16 bytes per
// thread, grid (pieces of a block, copies).
__global__ void copy_blocks_kernel(uint8_t *base, long block_bytes,
                                   const int32_t *src, const int32_t *dst,
                                   int num_blocks, int *err) {
  kvd::pdl_trigger();
  kvd::pdl_wait();
  const int i = blockIdx.y;
  const int s = src[i], d = dst[i];
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
      kvd::report(err, kvd::DEVERR_BLOCK);
    return;
  }
  const long n16 = block_bytes / 16;
  const uint4 *from = reinterpret_cast<const uint4 *>(base + s * block_bytes);
  uint4 *to = reinterpret_cast<uint4 *>(base + d * block_bytes);
  for (long j = (long)blockIdx.x * blockDim.x + threadIdx.x; j < n16;
       j += (long)gridDim.x * blockDim.x)
    to[j] = from[j];
}

}  // namespace

extern "C" {

kvd_status kvd_block_pool_create(int32_t num_blocks, kvd_block_pool **out) {
  if (!out) return kvd::set_error(KVD_ERR_NULL, "block_pool_create: out is NULL");
  *out = nullptr;
  if (num_blocks < 1)
    return kvd::set_error(KVD_ERR_SHAPE, "block_pool_create: num_blocks >= 1");
  auto *p = new kvd_block_pool;
  p->refs.assign(num_blocks, 0);
  p->free_.resize(num_blocks);
  for (int32_t i = 0; i < num_blocks; ++i) p->free_[i] = num_blocks - 1 - i;
  *out = p;
  return KVD_OK;
}

void kvd_block_pool_destroy(kvd_block_pool *pool) { delete pool; }

int32_t kvd_block_pool_free_count(kvd_block_pool *pool) {
  if (!pool) return -1;
  std::lock_guard<std::mutex> g(pool->mu);
  return (int32_t)pool->free_.size();
}

int32_t kvd_block_pool_refcount(kvd_block_pool *pool, int32_t block) {
  if (!pool) return -1;
  std::lock_guard<std::mutex> g(pool->mu);
  return valid_block(pool, block) ? pool->refs[block] : -1;
}

kvd_status kvd_block_pool_alloc(kvd_block_pool *pool, int32_t n,
                                int32_t *blocks) {
  if (!pool || (n > 0 && !blocks))
    return kvd::set_error(KVD_ERR_NULL, "block_pool_alloc: NULL argument");
  if (n < 0) return kvd::set_error(KVD_ERR_SHAPE, "block_pool_alloc: n < 0");
  std::lock_guard<std::mutex> g(pool->mu);
  if ((size_t)n > pool->free_.size())
    return kvd::set_error(KVD_ERR_CAPACITY, "block_pool_alloc: pool exhausted");
  for (int32_t i = 0; i < n; ++i) {
    blocks[i] = pool->free_.back();
    pool->free_.pop_back();
    pool->refs[blocks[i]] = 1;
  }
  return KVD_OK;
}

kvd_status kvd_block_pool_share(kvd_block_pool *pool, const int32_t *blocks,
                                int32_t n) {
  if (!pool || (n > 0 && !blocks))
    return kvd::set_error(KVD_ERR_NULL, "block_pool_share: NULL argument");
  std::lock_guard<std::mutex> g(pool->mu);
  for (int32_t i = 0; i < n; ++i)  // validate first: all or nothing
    if (blocks[i] >= 0 &&
        (!valid_block(pool, blocks[i]) || pool->refs[blocks[i]] == 0))
      return kvd::set_error(KVD_ERR_SHAPE,
                            "block_pool_share: a block that is not held");
  for (int32_t i = 0; i < n; ++i)
    if (blocks[i] >= 0) ++pool->refs[blocks[i]];
  return KVD_OK;
}

kvd_status kvd_block_pool_release(kvd_block_pool *pool, const int32_t *blocks,
                                  int32_t n) {
  if (!pool || (n > 0 && !blocks))
    return kvd::set_error(KVD_ERR_NULL, "block_pool_release: NULL argument");
  std::lock_guard<std::mutex> g(pool->mu);
  std::vector<int32_t> drop(pool->refs.size(), 0);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = blocks[i];
    if (b < 0) continue;
    if (!valid_block(pool, b) || ++drop[b] > pool->refs[b])
      return kvd::set_error(KVD_ERR_SHAPE,
                            "block_pool_release: more releases than holds");
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = blocks[i];
    if (b >= 0 && --pool->refs[b] == 0) push_free(pool, b);
  }
  return KVD_OK;
}

kvd_status kvd_block_pool_prepare_append(kvd_block_pool *pool,
                                         int32_t *block_table, int32_t batch,
                                         int32_t max_blocks,
                                         const int32_t *pos,
                                         int32_t block_size, int32_t *src,
                                         int32_t *dst, int32_t *n_copies) {
  if (!pool || !n_copies || (batch > 0 && (!block_table || !pos || !src ||
                                           !dst)))
    return kvd::set_error(KVD_ERR_NULL, "block_pool_prepare_append: NULL "
                          "argument");
  if (batch < 0 || max_blocks < 1 || block_size < 1)
    return kvd::set_error(KVD_ERR_SHAPE, "block_pool_prepare_append: batch >= "
                          "0, max_blocks >= 1, block_size >= 1");
  std::lock_guard<std::mutex> g(pool->mu);
  // plan first (all or nothing): which sequences need a fresh block (two
  // tables appending into one shared block both count, though only the
  // first copies: the second then holds the block alone)
  int32_t need = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t lb = pos[b] / block_size;
    if (pos[b] < 0 || lb >= max_blocks)
      return kvd::set_error(KVD_ERR_SHAPE, "block_pool_prepare_append: a "
                            "position outside the block table");
    const int32_t blk = block_table[(long)b * max_blocks + lb];
    if (blk >= 0 && (!valid_block(pool, blk) || pool->refs[blk] == 0))
      return kvd::set_error(KVD_ERR_SHAPE, "block_pool_prepare_append: a "
                            "table names a block the pool does not hold");
    if (blk < 0 || pool->refs[blk] > 1) ++need;
  }
  if ((size_t)need > pool->free_.size())
    return kvd::set_error(KVD_ERR_CAPACITY,
                          "block_pool_prepare_append: pool exhausted");
  int32_t nc = 0;
  for (int32_t b = 0; b < batch; ++b) {
    int32_t &slot = block_table[(long)b * max_blocks + pos[b] / block_size];
    if (slot >= 0 && pool->refs[slot] == 1) continue;  // already private
    const int32_t fresh = pool->free_.back();
    pool->free_.pop_back();
    pool->refs[fresh] = 1;
    if (slot >= 0) {  // shared: copy its rows, drop this table's hold
      src[nc] = slot;
      dst[nc] = fresh;
      ++nc;
      --pool->refs[slot];
    }
    slot = fresh;
  }
  *n_copies = nc;
  return KVD_OK;
}

kvd_status kvd_copy_blocks(const kvd_cache *cache, const int32_t *src,
                           const int32_t *dst, int32_t n, kvd_stream stream) {
  if (!cache || !cache->k)
    return kvd::set_error(KVD_ERR_NULL, "copy_blocks: cache required");
  if (n < 0) return kvd::set_error(KVD_ERR_SHAPE, "copy_blocks: n < 0");
  if (n == 0) return KVD_OK;
  if (!src || !dst)
    return kvd::set_error(KVD_ERR_NULL, "copy_blocks: src and dst required");
  const long row = cache->dtype == KVD_BF16    ? 2L * cache->head_dim
                   : cache->dtype == KVD_MXFP4 ? cache->head_dim / 2 +
                                                     cache->head_dim / 16
                                               : (long)cache->head_dim;
  const long block_bytes = row * cache->n_kv * cache->block_size;
  if (block_bytes % 16 != 0)
    return kvd::set_error(KVD_ERR_SHAPE, "copy_blocks: a block must be a "
                          "multiple of 16 bytes");
  if (n > 65535)
    return kvd::set_error(KVD_ERR_SHAPE, "copy_blocks: at most 65535 copies "
                          "per call");
  int *dev_err = nullptr;
  const kvd_status st = kvd::device_error_word(&dev_err);
  if (st != KVD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long n16 = block_bytes / 16;
  const dim3 grid((unsigned)std::min<long>((n16 + 255) / 256, 64), n);
  void *tensors[2] = {cache->k, cache->v};
  for (void *t : tensors) {
    if (!t) continue;
    const cudaError_t e =
        kvd::launch_pdl(copy_blocks_kernel, grid, dim3(256), 0, s, 1,
                        static_cast<uint8_t *>(t), block_bytes, src, dst,
                        cache->num_blocks, dev_err);
    if (e != cudaSuccess)
      return kvd::set_error(KVD_ERR_CUDA, "copy_blocks: launch failed");
  }
  return KVD_OK;
}

}  // extern "C"

// kv_append: write the new token's key and value rows into the paged cache.
//
// One thread moves 8 elements (16 bytes of bf16 input). bf16 caches get the
// bytes unchanged; fp8 caches get E4M3(x * inv_scale[kv_head]) with the
// product rounded once to fp32 and the conversion done by the hardware's
// round-to-nearest-even, saturating cvt. MXFP4 caches: one thread encodes
// one 16-channel group (store_mxfp4_group).
#include <cuda_fp16.h>

#include "kvd_common.cuh"

namespace kvd {

__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  pdl_trigger();
  pdl_wait();
  const bool fp4 = p.dtype == DT_MXFP4;
  const int chunks = p.head_dim / (fp4 ? 16 : 8);
  const long per_tensor = (long)p.batch * p.n_kv * chunks;
  const long total = p.v_cache ? 2 * per_tensor : per_tensor;
  const long gid = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= total) return;
  const bool is_v = gid >= per_tensor;
  long r = is_v ? gid - per_tensor : gid;
  const int c = (int)(r % chunks);
  r /= chunks;
  const int h = (int)(r % p.n_kv);
  const int b = (int)(r / p.n_kv);

  const int pos = p.pos[b];
  if (pos < 0 || pos >= p.max_blocks * p.block_size) {
    if (c == 0 && h == 0 && !is_v) report(p.err, DEVERR_POS);
    return;
  }
  const int blk = p.block_table[(long)b * p.max_blocks + pos / p.block_size];
  if (blk < 0 || blk >= p.num_blocks) {
    if (c == 0 && h == 0 && !is_v) report(p.err, DEVERR_BLOCK);
    return;
  }
  const long row = ((long)blk * p.n_kv + h) * p.block_size + pos % p.block_size;
  uint8_t *cache = is_v ? p.v_cache : p.k_cache;
  if (fp4) {
    const uint16_t *src = (is_v ? p.v_new : p.k_new) +
                          ((long)b * p.n_kv + h) * p.head_dim + c * 16;
    uint8_t *rowp = cache + row * row_bytes(p.head_dim, DT_MXFP4);
    store_mxfp4_group(rowp + c * 8, rowp + p.head_dim / 2 + c, src);
    return;
  }
  const uint16_t *src = (is_v ? p.v_new : p.k_new) +
                        ((long)b * p.n_kv + h) * p.head_dim + c * 8;
  const int es = p.dtype == DT_BF16 ? 2 : 1;
  const float inv =
      p.dtype == DT_BF16 ? 1.0f : (is_v ? p.v_inv_scale : p.k_inv_scale)[h];
  store_new8(cache + (row * p.head_dim + c * 8) * es, src, p.dtype, inv);
}

cudaError_t launch_append(const AppendParams &p, cudaStream_t s) {
  const long per_tensor = (long)p.batch * p.n_kv *
                          (p.head_dim / (p.dtype == DT_MXFP4 ? 16 : 8));
  const long total = p.v_cache ? 2 * per_tensor : per_tensor;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long blocks = (total + threads - 1) / threads;
  return launch_pdl(append_kernel, dim3((unsigned)blocks), dim3(threads), 0, s,
                    1, p);
}

}  // namespace kvd

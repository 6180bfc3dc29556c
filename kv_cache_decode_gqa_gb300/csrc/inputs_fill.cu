// libkvd_inputs.so: fills device buffers with seeded synthetic inputs, byte
// for byte the values the host generator (kv_cache_decode_gqa_gb300/inputs.py)
// produces. Element i of a fill gets table[draw(key, offset + i) >> (64 - bits)]
// where draw is SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): the output
// for counter n is mix(key + (n + 1) * 0x9E3779B97F4A7C15). Not part of the
// decode library.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t splitmix_draw(uint64_t key, uint64_t n) {
  uint64_t z = key + (n + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

template <typename T>
__global__ void fill_kernel(T *dst, uint64_t n, uint64_t key, uint64_t offset,
                            const T *table, int bits) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    dst[i] = table[splitmix_draw(key, offset + i) >> (64 - bits)];
  }
}

}  // namespace

extern "C" int kvdi_fill_table(void *dst, uint64_t n, int elem_bytes,
                               uint64_t key, uint64_t offset,
                               const void *table, int bits, void *stream) {
  if (n == 0) return 0;
  if (!dst || !table || bits < 1 || bits > 32) return 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const uint64_t want = (n + 255) / 256;
  const unsigned blocks = (unsigned)(want < (uint64_t)sms * 32 ? want
                                                                : (uint64_t)sms * 32);
  if (elem_bytes == 2)
    fill_kernel<uint16_t><<<blocks, 256, 0, s>>>(
        static_cast<uint16_t *>(dst), n, key, offset,
        static_cast<const uint16_t *>(table), bits);
  else if (elem_bytes == 1)
    fill_kernel<uint8_t><<<blocks, 256, 0, s>>>(
        static_cast<uint8_t *>(dst), n, key, offset,
        static_cast<const uint8_t *>(table), bits);
  else
    return 1;
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

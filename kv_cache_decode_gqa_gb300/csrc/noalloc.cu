// kvd_gqa_decode_noalloc: kvd_gqa_decode for callers that cannot allocate
// device memory.
//
// kvd_gqa_decode needs scratch memory for its split-K partial results, and
// its caller normally provides it. Some callers have no way to: a plug-in
// running inside a host program that owns every device allocation and
// offers it no allocator, or a latency-critical path that must never call
// cudaMalloc (which can synchronise the device). This entry point uses a
// scratch array compiled into the library instead, so the caller passes
// only inputs and outputs.
//
// The scratch is a file-scope __device__ array of KVD_NOALLOC_SCRATCH_BYTES
// bytes: every GPU that loads the library holds it until the process exits.
// In host code its name is only a stand-in for the device object, so the
// device address is looked up once per device with cudaGetSymbolAddress (on
// that device's first call, with it current) and passed to the kernels.
// Every call shares the one array: calls whose work can overlap on the GPU
// (different streams, or different host threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "kvd.h"
#include "kvd_internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[KVD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once).
kvd_status scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return kvd::set_error(KVD_ERR_CUDA, "gqa_decode_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return kvd::set_error(KVD_ERR_CUDA, "gqa_decode_noalloc: device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return kvd::set_error(KVD_ERR_CUDA,
                            "gqa_decode_noalloc: cudaGetSymbolAddress failed");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KVD_OK;
}

}  // namespace

extern "C" kvd_status kvd_gqa_decode_noalloc(const kvd_cache *cache,
                                             const kvd_seqs *seqs,
                                             const void *q, int32_t n_h,
                                             float scale, void *out,
                                             float *lse, kvd_stream stream) {
  size_t total = 0;
  kvd_status st = kvd::gqa_workspace_bytes(cache, seqs, n_h, &total);
  if (st != KVD_OK) return st;
  if (total > (size_t)KVD_NOALLOC_SCRATCH_BYTES)
    return kvd::set_error(
        KVD_ERR_WORKSPACE,
        "gqa_decode_noalloc: these shapes need more scratch than the library's "
        "static array holds (KVD_NOALLOC_SCRATCH_BYTES); use kvd_gqa_decode "
        "with a caller-provided workspace");
  void *scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != KVD_OK) return st;
  // the GQA decode's scratch holds only partial results, each written
  // before it is read within the call: nothing needs clearing
  return kvd_gqa_decode(cache, seqs, q, n_h, scale, out, lse, scratch,
                        (size_t)KVD_NOALLOC_SCRATCH_BYTES, stream);
}

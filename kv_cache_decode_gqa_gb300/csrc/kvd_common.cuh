// Device helpers shared by the libkvd kernels: inline PTX for mbarriers,
// bulk asynchronous copies (the TMA engine's untiled form), warp MMA, and
// exact bf16 / fp8 unpacking. Only documented PTX instructions are used.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvd_internal.h"

namespace kvd {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void report(int *err, int bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialisation (launch_pdl): it may be scheduled while the kernel before it
// on the stream is still running, so its launch overlaps that kernel's last
// CTAs instead of following their completion. pdl_trigger lets this grid's
// successor be scheduled (the successor still cannot pass its pdl_wait
// before this grid completes); pdl_wait blocks until this grid's
// predecessor has completed and its writes are visible, and every kernel
// calls it before it touches global memory the predecessor may write.
// Decode kernels trigger only after their wait, so the merge launch that
// follows a decode launch never overlaps the decode's predecessor. Without
// a programmatic predecessor both are no-ops.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch `kern` on `s` with programmatic stream serialisation allowed, plus
// an optional cluster shape (cluster_x > 1).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block,
                              size_t smem, cudaStream_t s, int cluster_x,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e == cudaSuccess) note_launch();
  return e;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of phase `parity` of `bar` (true once it completed).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar`. Each try_wait may suspend the
// thread for a short hardware-defined time; 2^22 tries bound the wait to well
// under a few seconds. Returns false (and the caller reports
// KVD_DEVERR_TIMEOUT) if the phase never completed.
// A non-blocking test comes first: a phase that has already completed then
// costs a test instead of a try_wait, which took a few hundred cycles even
// then.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < (1u << 22); ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// ---------------------------------------------------------------------------
// bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0),
// completion counted in bytes on `bar`.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src,
                                         uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (used for data read exactly once).
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src,
                                              uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes."
      "L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// tiled TMA copy of a 2-D box (coordinates: innermost first), completion
// counted in bytes on `bar`. `tmap` is the address of a CUtensorMap held in
// kernel-parameter (grid-constant) space.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x,
                                            int y, uint64_t *bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
          smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (copy engine) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------------------
// warp-level matrix multiply-accumulate (m16n8k16, fp32 accumulators) and
// shared-memory matrix loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, "
      "[%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4],
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte permute: result byte i = byte sel_i of {b:a} (a = bytes 0-3)
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b,
                                         uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// ---------------------------------------------------------------------------
// thread-block clusters (distributed shared memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; orders shared-memory writes
// before the barrier against the other CTAs' reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of cluster_sync, for work between them: a thread that has
// arrived must wait before it arrives again.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Generic address of `local`'s counterpart in the shared memory of CTA
// `rank` of this cluster. Plain loads through it are ordered by the
// compiler against the cluster barriers and can be issued together.
template <typename T>
__device__ __forceinline__ const T *cluster_ptr(const T *local,
                                                uint32_t rank) {
  const T *r;
  asm("mapa.u64 %0, %1, %2;" : "=l"(r) : "l"(local), "r"(rank));
  return r;
}

// Shared-memory window address (shared::cluster) of `local`'s counterpart in
// CTA `rank` of this cluster, and a 16-byte load through it.
__device__ __forceinline__ uint32_t cluster_saddr(const void *local,
                                                  uint32_t rank) {
  uint32_t r;
  asm("mapa.shared::cluster.u32 %0, %1, %2;"
      : "=r"(r)
      : "r"(smem_u32(local)), "r"(rank));
  return r;
}
// Stores into distributed shared memory (an address from cluster_saddr).
__device__ __forceinline__ void st_dsmem_f4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v)
               : "memory");
}
// One arrival on the mbarrier at `addr` in another CTA of the cluster, with
// release semantics at cluster scope (this thread's earlier writes, remote
// ones included, are visible to a thread that then observes the phase).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
  asm volatile(
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
          addr)
      : "memory");
}
// Bounded wait for phase `parity` of this CTA's `bar` with acquire
// semantics at cluster scope (for arrivals of other CTAs of the cluster).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar,
                                                  uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], "
        "%2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// 16-byte asynchronous copies global -> shared through the load path
// (cp.async): `src_bytes` 0 fills the 16 bytes with zeros and reads nothing.
// Completion is per thread, by commit groups.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void *dst, const void *src,
                                           uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's most recent groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// named barriers (a subset of the CTA's warps)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Arrive at named barrier `id` (of `count` threads) without waiting.
__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// numbers
// ---------------------------------------------------------------------------
// 2^x with the hardware approximation (relative error ~2^-22).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 pair (low element in the low half) -> two exact floats.
__device__ __forceinline__ float bf16lo(uint32_t u) {
  return __uint_as_float(u << 16);
}
__device__ __forceinline__ float bf16hi(uint32_t u) {
  return __uint_as_float(u & 0xffff0000u);
}

// float -> bf16 bits, round to nearest even (hardware conversion).
__device__ __forceinline__ uint16_t f2bf(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

// two floats -> packed bf16x2 (a in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// two floats -> packed f16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// two E4M3 codes (low byte = first element) -> packed f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}

// f16 halves of a packed pair -> float, exact.
__device__ __forceinline__ float f16_to_f32(uint16_t h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}
__device__ __forceinline__ float f16lo(uint32_t u) {
  return f16_to_f32(static_cast<uint16_t>(u & 0xffffu));
}
__device__ __forceinline__ float f16hi(uint32_t u) {
  return f16_to_f32(static_cast<uint16_t>(u >> 16));
}

// Two floats -> two E4M3 codes (first in the low byte), round to nearest
// even, saturating to +-448 (the hardware's satfinite conversion).
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float first, float second) {
  uint16_t r;
  // cvt puts its first source operand in the upper byte.
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
      : "=h"(r)
      : "f"(second), "f"(first));
  return r;
}

// One 8-element piece of a new key or value row into the cache: the 16
// bytes of bf16 unchanged, or (fp8) E4M3(x * inv) with the product rounded
// once to fp32. `src` holds 8 bf16 elements; `dst` is 16 (bf16) or 8 (fp8)
// bytes of the cached row.
__device__ __forceinline__ void store_new8(uint8_t *dst, const uint16_t *src,
                                           int dtype, float inv) {
  const uint4 x = *reinterpret_cast<const uint4 *>(src);
  if (dtype == DT_BF16) {
    *reinterpret_cast<uint4 *>(dst) = x;
  } else {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t packed[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint16_t a = e4m3x2_from_f32(__fmul_rn(bf16lo(w[2 * j]), inv),
                                         __fmul_rn(bf16hi(w[2 * j]), inv));
      const uint16_t b = e4m3x2_from_f32(__fmul_rn(bf16lo(w[2 * j + 1]), inv),
                                         __fmul_rn(bf16hi(w[2 * j + 1]), inv));
      packed[j] = (uint32_t)a | ((uint32_t)b << 16);
    }
    *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
  }
}

// ---------------------------------------------------------------------------
// MXFP4 rows: E2M1 codes with one E4M3 scale per 16 channels
// ---------------------------------------------------------------------------
// E2M1 code of q: round to nearest with ties to the code whose mantissa bit
// is 0, saturating at +-6 (comparisons against the midpoints of the grid
// 0, 0.5, 1, 1.5, 2, 3, 4, 6; NaN saturates), sign in bit 3.
__device__ __forceinline__ uint32_t e2m1_code(float q) {
  const float a = fabsf(q);
  const uint32_t c = a <= 0.25f   ? 0u
                     : a < 0.75f  ? 1u
                     : a <= 1.25f ? 2u
                     : a < 1.75f  ? 3u
                     : a <= 2.5f  ? 4u
                     : a < 3.5f   ? 5u
                     : a <= 5.f   ? 6u
                                  : 7u;
  return c | ((__float_as_uint(q) >> 31) << 3);
}

// Two E2M1 codes (the low byte of `b`: the first code in its low nibble) to
// their f16 values, first in the low half (exact: every E2M1 value is an
// f16).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t b) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(b & 0xffu));
  return r;
}

// One 16-channel group of a new bf16 row into an MXFP4 row: 8 bytes of
// codes (channel 2j low nibble) at `codes`, the E4M3 scale byte at
// `scale`. amax and both divisions in fp32, conversions round to nearest
// even and saturate; a scale that rounds to 0 gives zero codes.
__device__ __forceinline__ void store_mxfp4_group(uint8_t *codes,
                                                  uint8_t *scale,
                                                  const uint16_t *src) {
  const uint4 u0 = *reinterpret_cast<const uint4 *>(src);
  const uint4 u1 = *reinterpret_cast<const uint4 *>(src + 8);
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  float x[16];
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    x[2 * j] = bf16lo(w[j]);
    x[2 * j + 1] = bf16hi(w[j]);
    amax = fmaxf(amax, fmaxf(fabsf(x[2 * j]), fabsf(x[2 * j + 1])));
  }
  const uint32_t sc =
      e4m3x2_from_f32(__fdiv_rn(amax, 6.0f), 0.f) & 0xffu;  // low byte
  const float s = f16lo(e4m3x2_to_f16x2((uint16_t)sc));
  uint32_t packed[2] = {0u, 0u};
  if (s > 0.f) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      packed[j >> 3] |= e2m1_code(__fdiv_rn(x[j], s)) << (4 * (j & 7));
  }
  *reinterpret_cast<uint2 *>(codes) = make_uint2(packed[0], packed[1]);
  *scale = (uint8_t)sc;
}

// Orders this thread's generic-proxy global-memory writes before later
// async-proxy (copy engine) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Opt a kernel into `bytes` of dynamic shared memory, once per device (the
// attribute call stays out of stream capture after the first launch). Each
// kernel passes its own `done` table (one flag per device ordinal).
template <typename K>
inline cudaError_t set_smem_once(K kern, int bytes, bool (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

}  // namespace kvd

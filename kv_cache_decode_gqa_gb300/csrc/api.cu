// The C ABI of libkvd.so (declared in include/kvd.h): host-side argument
// validation, split planning and kernel dispatch. Nothing here allocates
// device memory or synchronises, except kvd_device_error().
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "kvd.h"
#include "kvd_internal.h"

namespace {

// The library's device error word (one per device that loads the module).
__device__ int g_kvd_device_error;

thread_local char g_msg[512] = "";

kvd_status fail(kvd_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

kvd_status ok() {
  g_msg[0] = 0;
  return KVD_OK;
}

kvd_status cuda_fail(cudaError_t e, const char *what) {
  return fail(KVD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int *err = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

// Per-device facts, looked up once per device with that device current.
kvd_status device_info(const DeviceInfo **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(KVD_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_devices_mu);
  DeviceInfo &d = g_devices[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err),
                             g_kvd_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    d.ready = true;
  }
  *out = &d;
  return KVD_OK;
}

bool aligned(const void *p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

int env_int(const char *name, int dflt) {
  const char *s = std::getenv(name);
  if (!s || !*s) return dflt;
  return std::atoi(s);
}

// Tuning overrides (kvd_set_tuning): read from the environment once, when
// the library is loaded, and changed only by kvd_set_tuning.
std::atomic<int> g_decode_ctas{env_int("KVD_DECODE_CTAS", 0)};
std::atomic<int> g_mla_cuda_cores{env_int("KVD_MLA_CUDA_CORES", 0)};

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
kvd_status check_cache(const kvd_cache *c, bool need_v, const char *what) {
  if (!c) return fail(KVD_ERR_NULL, "%s: cache is NULL", what);
  if (!c->k) return fail(KVD_ERR_NULL, "%s: cache->k is NULL", what);
  if (need_v && !c->v)
    return fail(KVD_ERR_NULL, "%s: cache->v is NULL (K and V required)", what);
  if (c->num_blocks < 1 || c->block_size < 1 || c->n_kv < 1 ||
      c->head_dim < 1)
    return fail(KVD_ERR_SHAPE,
                "%s: num_blocks, block_size, n_kv and head_dim must be >= 1",
                what);
  if (c->dtype != KVD_BF16 && c->dtype != KVD_FP8_E4M3 &&
      c->dtype != KVD_MXFP4)
    return fail(KVD_ERR_UNSUPPORTED, "%s: unknown dtype %d", what, c->dtype);
  if (!aligned(c->k, 16) || (c->v && !aligned(c->v, 16)))
    return fail(KVD_ERR_SHAPE, "%s: cache base pointers must be 16-byte aligned",
                what);
  if (c->dtype == KVD_MXFP4) {
    // 72-byte rows, copied two at a time: whole (block, head) runs stay
    // 16-byte multiples when the block size is even
    if (c->head_dim != 128)
      return fail(KVD_ERR_UNSUPPORTED, "%s: mxfp4 caches need head_dim 128",
                  what);
    if (c->block_size % 2 != 0)
      return fail(KVD_ERR_SHAPE, "%s: mxfp4 caches need an even block_size",
                  what);
    return KVD_OK;
  }
  const long row_bytes =
      (long)c->head_dim * (c->dtype == KVD_BF16 ? 2 : 1);
  if (row_bytes % 16 != 0)
    return fail(KVD_ERR_SHAPE, "%s: a cache row (%ld bytes) must be a multiple "
                "of 16 bytes", what, row_bytes);
  return KVD_OK;
}

// Calls other than the dense GQA decode attend to every position they are
// given: a sliding window there is refused.
kvd_status no_window(const kvd_seqs *s, const char *what) {
  if (s && (s->window != 0 || s->window_start))
    return fail(KVD_ERR_UNSUPPORTED, "%s: no sliding window (window and "
                "window_start are for the GQA decode calls)", what);
  return KVD_OK;
}

kvd_status check_seqs(const kvd_seqs *s, const kvd_cache *c, const char *what) {
  if (!s) return fail(KVD_ERR_NULL, "%s: seqs is NULL", what);
  if (s->batch < 0 || s->max_blocks_per_seq < 1 || s->max_seq_len < 0)
    return fail(KVD_ERR_SHAPE,
                "%s: batch >= 0, max_blocks_per_seq >= 1, max_seq_len >= 0 "
                "required", what);
  if (s->batch > 65535)
    return fail(KVD_ERR_SHAPE, "%s: batch %d above 65535", what, s->batch);
  if (s->flags & ~(KVD_SEQS_STABLE | KVD_SEQS_PREFIX_READY))
    return fail(KVD_ERR_SHAPE, "%s: unknown seqs flags 0x%x", what,
                (unsigned)s->flags);
  if ((s->flags & KVD_SEQS_PREFIX_READY) && !(s->flags & KVD_SEQS_STABLE))
    return fail(KVD_ERR_SHAPE, "%s: KVD_SEQS_PREFIX_READY needs "
                "KVD_SEQS_STABLE", what);
  if (s->batch > 0 && (!s->block_table || !s->seq_lens))
    return fail(KVD_ERR_NULL, "%s: block_table and seq_lens are required", what);
  if (s->window < 0)
    return fail(KVD_ERR_SHAPE, "%s: window must be >= 0", what);
  if ((long)s->max_seq_len > (long)s->max_blocks_per_seq * c->block_size)
    return fail(KVD_ERR_CAPACITY,
                "%s: max_seq_len %d exceeds the block table's capacity %ld",
                what, s->max_seq_len,
                (long)s->max_blocks_per_seq * c->block_size);
  return KVD_OK;
}

// ---------------------------------------------------------------------------
// split plans
// ---------------------------------------------------------------------------
struct Plan {
  int split_len = kvd::kStageRows;
  int n_splits = 1;
  int n_groups = 1;        // head groups (tiles) per sequence
  size_t ws_o_bytes = 0;   // partial outputs
  size_t ws_lse_bytes = 0; // partial log-sum-exps
  size_t ws_bytes = 0;     // total
  int hp = 1;              // kv heads per work unit (CUDA-core GQA kernel)
  int whole_units = 0;     // dense GQA: one CTA per unit, no merge
  int cluster = 0;         // dense GQA: CTAs per unit of a cluster merge
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

enum class DenseKernel { Simt, Mma };

kvd_status gqa_shape(const kvd_cache *c, int n_h, DenseKernel *kind) {
  if (n_h < 1 || n_h % c->n_kv != 0)
    return fail(KVD_ERR_SHAPE, "gqa_decode: n_h (%d) must be a positive "
                "multiple of n_kv (%d)", n_h, c->n_kv);
  const int g = n_h / c->n_kv;
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(KVD_ERR_UNSUPPORTED, "gqa_decode: head_dim %d (64 or 128)",
                c->head_dim);
  if (c->dtype == KVD_MXFP4 && g != 1 && g != 2 && g != 4)
    return fail(KVD_ERR_UNSUPPORTED, "gqa_decode: mxfp4 caches are decoded "
                "on the CUDA-core kernel: group size 1, 2 or 4 (got %d)", g);
  if (g == 1 || g == 2 || g == 4) {
    *kind = DenseKernel::Simt;
  } else if ((g == 8 || g == 16) && c->head_dim == 128) {
    *kind = DenseKernel::Mma;
  } else {
    return fail(KVD_ERR_UNSUPPORTED,
                "gqa_decode: group size %d with head_dim %d", g, c->head_dim);
  }
  return KVD_OK;
}

// Units (sequence, head group) of at most this many 64-token chunks run one
// per CTA when they fit in one wave: the merge launch and its two grid
// dependencies (about 3 us) then cost more than the imbalance of whole
// units (at most this many chunks against the average share).
constexpr int kWholeUnitChunks = 4;

// Persistent stream-K plan of the dense GQA kernels: `ctas_per_sm` CTAs per
// SM (never more CTAs than 64-token chunks), each leaving at most two
// partials of G heads x head_dim, which the merge launch combines. Short
// units instead run whole, one CTA each (no partials, no merge): every unit
// holds at most kWholeUnitChunks chunks (the window bounds it, or the
// longest visible length does) and there are no more units than CTAs.
Plan plan_stream_k(int sms, int ctas_per_sm, int batch, int n_kv, int g,
                   int d, int max_seq_len, int window = 0) {
  Plan pl;
  const int R = kvd::kStageRows;
  const long unit_chunks =
      window > 0 ? std::min<long>((window + R - 1) / R + 1,
                                  (max_seq_len + R - 1) / R)
                 : (max_seq_len + R - 1) / R;
  const long chunks = (long)batch * n_kv * ((max_seq_len + R - 1) / R);
  long ctas = (long)sms * ctas_per_sm;
  const int forced = g_decode_ctas.load(std::memory_order_relaxed);
  const long units = (long)batch * n_kv;
  if (forced <= 0 && units >= 1 && units <= ctas &&
      unit_chunks <= kWholeUnitChunks) {
    pl.whole_units = 1;
    pl.n_splits = (int)units;
    pl.n_groups = n_kv;
    return pl;  // no workspace
  }
  if (forced > 0) ctas = forced;
  ctas = std::max(1L, std::min(ctas, std::max(chunks, 1L)));
  pl.n_splits = (int)ctas;
  pl.n_groups = n_kv;
  pl.ws_o_bytes = round_up((size_t)ctas * 2 * g * d * 4, 256);
  pl.ws_lse_bytes = round_up((size_t)ctas * 2 * g * 4, 256);
  pl.ws_bytes = pl.ws_o_bytes + pl.ws_lse_bytes;
  return pl;
}

Plan gqa_plan(const kvd_cache *c, const kvd_seqs *s, int n_h, int sms,
              DenseKernel kind) {
  const int g = n_h / c->n_kv;
  const int hp = kind == DenseKernel::Simt
                     ? kvd::simt_heads_per_stage(c->n_kv, g, c->head_dim,
                                                 c->dtype, c->block_size)
                     : kvd::mma_heads_per_unit(c->n_kv, c->block_size,
                                               c->dtype);
  Plan pl = plan_stream_k(sms, 1, s->batch, c->n_kv / hp, g * hp,
                          c->head_dim, s->max_seq_len, s->window);
  pl.hp = hp;
  // One sequence (every unit as long as the others) on the CUDA-core
  // kernel with query groups of 1: its units run as clusters of CTAs that
  // merge their parts in distributed shared memory, when all the clusters
  // fit at once -- no workspace and no merge launch.
  if (kind == DenseKernel::Simt && !pl.whole_units && s->batch == 1 &&
      g == 1 && g_decode_ctas.load(std::memory_order_relaxed) <= 0) {
    const int units = c->n_kv / hp;
    const int cs =
        kvd::simt_cluster_size(c->head_dim, c->dtype, hp, units, sms);
    if (cs >= 2) {
      Plan cl;
      cl.cluster = cs;
      cl.n_splits = units * cs;
      cl.n_groups = units;
      cl.hp = hp;
      return cl;
    }
  }
  return pl;
}

// Persistent stream-K plan of the latent decode kernels: 32-position (or
// 64-position) chunks of `rows` positions per sequence and head tile;
// partials of 64 heads x dv per CTA side, merged by a second launch.
// `per_lane` CTAs of the launch share a lane's chunk range (one per head
// tile, or per head tile and value part for the tensor-core latent
// kernel); n_splits counts 64-head tiles per lane whatever the kernel.
Plan plan_wide(int sms, int batch, int n_h, int rows, int dv,
               int per_lane = 0, int chunk_rows = 32) {
  Plan pl;
  const int tiles = n_h / 64;
  if (per_lane <= 0) per_lane = tiles;
  const long chunks = (long)batch * ((rows + chunk_rows - 1) / chunk_rows);
  long ctas = sms;
  const int forced = g_decode_ctas.load(std::memory_order_relaxed);
  if (forced > 0) ctas = forced;
  const long lanes =
      std::max(1L, std::min(ctas / per_lane, std::max(chunks, 1L)));
  ctas = lanes * tiles;
  pl.n_splits = (int)ctas;
  pl.n_groups = tiles;
  pl.ws_o_bytes = round_up((size_t)ctas * 2 * 64 * dv * 4, 256);
  pl.ws_lse_bytes = round_up((size_t)ctas * 2 * 64 * 4, 256);
  pl.ws_bytes = pl.ws_o_bytes + pl.ws_lse_bytes;
  return pl;
}

// The latent decode runs on the tcgen05 kernel where its shape allows
// (kvd_set_tuning can select the CUDA-core kernel everywhere).
bool mla_on_tensor_memory(const kvd_cache *c, int n_h) {
  return g_mla_cuda_cores.load(std::memory_order_relaxed) == 0 &&
         kvd::latent_tc_supported(n_h, c->block_size, c->num_blocks);
}

Plan mla_plan(const kvd_seqs *s, int n_h, int dv, int sms, bool tc) {
  return tc ? plan_wide(sms, s->batch, n_h, s->max_seq_len, dv,
                       n_h / 128 * kvd::kLatentTcParts,
                       kvd::kLatentTcRows)
            : plan_wide(sms, s->batch, n_h, s->max_seq_len, dv);
}

// The tcgen05 gather kernel: S CTAs per (sequence, 64-head tile), one
// wave. With S > 1 each CTA leaves its part (64 heads x 512 values fp32 +
// 64 lse) for the merge launch.
Plan sparse_plan(const kvd_seqs *s, int n_h, int k, int dv, int sms) {
  Plan pl;
  const int units = std::max(s->batch * (n_h / 64), 1);
  const int S = kvd::gather_tc_splits(
      units, std::max(k, 1), sms, g_decode_ctas.load(std::memory_order_relaxed));
  pl.n_splits = S;
  pl.n_groups = 1;
  const size_t slots = (size_t)units * S;
  pl.ws_o_bytes = S > 1 ? round_up(slots * 64 * dv * 4, 256) : 0;
  pl.ws_lse_bytes = S > 1 ? round_up(slots * 64 * 4, 256) : 0;
  pl.ws_bytes = pl.ws_o_bytes + pl.ws_lse_bytes;
  return pl;
}

size_t topk_ws_bytes(const kvd_seqs *s) {
  return round_up((size_t)s->batch * std::max(s->max_seq_len, 1) * 4, 256);
}

kvd_status check_ws(const Plan &pl, void *ws, size_t bytes, const char *what) {
  if (pl.ws_bytes == 0) return KVD_OK;
  if (!ws)
    return fail(KVD_ERR_WORKSPACE, "%s: workspace of %zu bytes required", what,
                pl.ws_bytes);
  if (!aligned(ws, 256))
    return fail(KVD_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned",
                what);
  if (bytes < pl.ws_bytes)
    return fail(KVD_ERR_WORKSPACE, "%s: workspace %zu < required %zu bytes",
                what, bytes, pl.ws_bytes);
  return KVD_OK;
}

float log2_scale(float scale, int dk) {
  const float s = scale > 0.f ? scale : 1.0f / std::sqrt((float)dk);
  return s * 1.4426950408889634f;
}

kvd_status launched(cudaError_t e, const char *what) {
  if (e == cudaErrorNotSupported)
    return fail(KVD_ERR_UNSUPPORTED, "%s: kernel not available", what);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return ok();
}

}  // namespace

namespace kvd {
namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Workspace bytes of a gqa_decode call with these arguments on the current
// device (validating them as the call does). Used by the no-allocation entry
// point.
kvd_status gqa_workspace_bytes(const kvd_cache *cache, const kvd_seqs *seqs,
                               int32_t n_h, size_t *total) {
  kvd_status st = check_cache(cache, true, "gqa_decode");
  if (st != KVD_OK) return st;
  st = check_seqs(seqs, cache, "gqa_decode");
  if (st != KVD_OK) return st;
  DenseKernel kind;
  st = gqa_shape(cache, n_h, &kind);
  if (st != KVD_OK) return st;
  const DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != KVD_OK) return st;
  *total = gqa_plan(cache, seqs, n_h, d->sms, kind).ws_bytes;
  return KVD_OK;
}

kvd_status device_error_word(int **err) {
  const DeviceInfo *d = nullptr;
  const kvd_status st = device_info(&d);
  if (st != KVD_OK) return st;
  *err = d->err;
  return KVD_OK;
}

kvd_status set_error(kvd_status st, const char *msg) {
  return fail(st, "%s", msg);
}
}  // namespace kvd

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

int32_t kvd_version(void) { return KVD_VERSION; }

kvd_status kvd_set_tuning(int32_t decode_ctas, int32_t mla_cuda_cores) {
  if (decode_ctas < 0)
    return fail(KVD_ERR_SHAPE, "set_tuning: decode_ctas must be >= 0");
  g_decode_ctas.store(decode_ctas, std::memory_order_relaxed);
  g_mla_cuda_cores.store(mla_cuda_cores != 0, std::memory_order_relaxed);
  return ok();
}

uint64_t kvd_launch_count(void) {
  return kvd::g_launches.load(std::memory_order_relaxed);
}

const char *kvd_last_error(void) { return g_msg; }

const char *kvd_status_string(kvd_status st) {
  switch (st) {
    case KVD_OK: return "KVD_OK";
    case KVD_ERR_NULL: return "KVD_ERR_NULL";
    case KVD_ERR_SHAPE: return "KVD_ERR_SHAPE";
    case KVD_ERR_UNSUPPORTED: return "KVD_ERR_UNSUPPORTED";
    case KVD_ERR_CAPACITY: return "KVD_ERR_CAPACITY";
    case KVD_ERR_WORKSPACE: return "KVD_ERR_WORKSPACE";
    case KVD_ERR_CUDA: return "KVD_ERR_CUDA";
  }
  return "KVD_ERR_UNKNOWN";
}

uint64_t kvd_bytes_per_token(int32_t n_l, int32_t n_kv, int32_t d_h,
                             int32_t elem_bytes) {
  if (n_l < 0 || n_kv < 0 || d_h < 0 || elem_bytes < 0) return 0;
  return 2ull * (uint64_t)n_l * (uint64_t)n_kv * (uint64_t)d_h *
         (uint64_t)elem_bytes;
}

kvd_status kvd_device_error(int32_t *code) {
  if (!code) return fail(KVD_ERR_NULL, "device_error: code is NULL");
  const DeviceInfo *d = nullptr;
  kvd_status st = device_info(&d);
  if (st != KVD_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, d->err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  const int zero = 0;
  e = cudaMemcpy(d->err, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
  *code = v;
  return ok();
}

kvd_status kvd_kv_append(const kvd_cache *cache, const int32_t *block_table,
                         int32_t max_blocks_per_seq, const int32_t *pos,
                         int32_t batch, const void *k_new, const void *v_new,
                         kvd_stream stream) {
  kvd_status st = check_cache(cache, false, "kv_append");
  if (st != KVD_OK) return st;
  if (batch < 0 || batch > 65535 || max_blocks_per_seq < 1)
    return fail(KVD_ERR_SHAPE, "kv_append: 0 <= batch <= 65535 and "
                "max_blocks_per_seq >= 1 required");
  if (cache->head_dim % 8 != 0)
    return fail(KVD_ERR_SHAPE, "kv_append: head_dim must be a multiple of 8");
  if (batch == 0) return ok();
  if (!block_table || !pos || !k_new)
    return fail(KVD_ERR_NULL, "kv_append: block_table, pos and k_new required");
  if (cache->v && !v_new)
    return fail(KVD_ERR_NULL, "kv_append: v_new required for a K/V cache");
  if (!aligned(k_new, 16) || (cache->v && !aligned(v_new, 16)))
    return fail(KVD_ERR_SHAPE, "kv_append: k_new / v_new must be 16-byte "
                "aligned");
  if (cache->dtype == KVD_FP8_E4M3 &&
      (!cache->k_inv_scale || (cache->v && !cache->v_inv_scale)))
    return fail(KVD_ERR_NULL, "kv_append: fp8 cache needs inverse scales");
  const DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != KVD_OK) return st;
  kvd::AppendParams p{};
  p.k_cache = static_cast<uint8_t *>(cache->k);
  p.v_cache = static_cast<uint8_t *>(cache->v);
  p.k_inv_scale = cache->k_inv_scale;
  p.v_inv_scale = cache->v_inv_scale;
  p.block_table = block_table;
  p.pos = pos;
  p.k_new = static_cast<const uint16_t *>(k_new);
  p.v_new = static_cast<const uint16_t *>(v_new);
  p.num_blocks = cache->num_blocks;
  p.block_size = cache->block_size;
  p.n_kv = cache->n_kv;
  p.head_dim = cache->head_dim;
  p.dtype = cache->dtype;
  p.max_blocks = max_blocks_per_seq;
  p.batch = batch;
  p.err = d->err;
  return launched(kvd::launch_append(p, reinterpret_cast<cudaStream_t>(stream)),
                  "kv_append");
}

kvd_status kvd_workspace_size(kvd_op op, const kvd_cache *cache,
                              const kvd_seqs *seqs, int32_t n_h, int32_t k,
                              size_t *bytes) {
  if (!bytes) return fail(KVD_ERR_NULL, "workspace_size: bytes is NULL");
  kvd_status st = check_cache(cache, false, "workspace_size");
  if (st != KVD_OK) return st;
  st = check_seqs(seqs, cache, "workspace_size");
  if (st != KVD_OK) return st;
  const DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != KVD_OK) return st;
  switch (op) {
    case KVD_OP_GQA_DECODE: {
      DenseKernel kind;
      st = gqa_shape(cache, n_h, &kind);
      if (st != KVD_OK) return st;
      *bytes = gqa_plan(cache, seqs, n_h, d->sms, kind).ws_bytes;
      return ok();
    }
    case KVD_OP_MLA_DECODE:
      if (n_h < 64 || n_h % 64 != 0)
        return fail(KVD_ERR_UNSUPPORTED, "mla: n_h must be a multiple of 64");
      *bytes = mla_plan(seqs, n_h, 512, d->sms,
                        mla_on_tensor_memory(cache, n_h)).ws_bytes;
      return ok();
    case KVD_OP_SPARSE_DECODE:
      if (n_h < 64 || n_h % 64 != 0 || k < 1)
        return fail(KVD_ERR_UNSUPPORTED,
                    "sparse: n_h must be a multiple of 64 and k >= 1");
      *bytes = sparse_plan(seqs, n_h, k, cache->head_dim, d->sms).ws_bytes;
      return ok();
    case KVD_OP_INDEXER_TOPK:
      *bytes = topk_ws_bytes(seqs);
      return ok();
    case KVD_OP_INDEXER_TOPK_POOL:
      *bytes = round_up((size_t)seqs->batch * kvd::kPoolBlocks *
                            kvd::kPoolBlock * 4, 256);
      return ok();
  }
  return fail(KVD_ERR_UNSUPPORTED, "workspace_size: unknown op %d", (int)op);
}

}  // extern "C"

namespace {
// kvd_gqa_decode, and kvd_gqa_append_decode when pos != nullptr.
kvd_status gqa_decode_impl(const kvd_cache *cache, const kvd_seqs *seqs,
                           const int32_t *pos, const void *k_new,
                           const void *v_new, const void *q, int32_t n_h,
                           float scale, void *out, float *lse,
                           void *workspace, size_t workspace_bytes,
                           kvd_stream stream) {
  kvd_status st = check_cache(cache, true, "gqa_decode");
  if (st != KVD_OK) return st;
  st = check_seqs(seqs, cache, "gqa_decode");
  if (st != KVD_OK) return st;
  DenseKernel kind;
  st = gqa_shape(cache, n_h, &kind);
  if (st != KVD_OK) return st;
  if (seqs->batch > 1024)
    return fail(KVD_ERR_UNSUPPORTED, "gqa_decode: at most 1024 sequences "
                "per call (got %d)", seqs->batch);
  if (cache->dtype == KVD_FP8_E4M3 && (!cache->k_scale || !cache->v_scale))
    return fail(KVD_ERR_NULL, "gqa_decode: fp8 cache needs k_scale, v_scale");
  if (seqs->batch == 0) return ok();
  if (!q || !out) return fail(KVD_ERR_NULL, "gqa_decode: q and out required");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(KVD_ERR_SHAPE, "gqa_decode: q and out must be 16-byte aligned");
  if (pos) {
    if (!k_new || !v_new)
      return fail(KVD_ERR_NULL, "gqa_append_decode: k_new and v_new required");
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
      return fail(KVD_ERR_SHAPE, "gqa_append_decode: k_new / v_new must be "
                  "16-byte aligned");
    if (cache->dtype == KVD_FP8_E4M3 &&
        (!cache->k_inv_scale || !cache->v_inv_scale))
      return fail(KVD_ERR_NULL,
                  "gqa_append_decode: fp8 cache needs inverse scales");
  }
  const DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != KVD_OK) return st;
  const Plan pl = gqa_plan(cache, seqs, n_h, d->sms, kind);
  st = check_ws(pl, workspace, workspace_bytes, "gqa_decode");
  if (st != KVD_OK) return st;

  kvd::DecodeParams p{};
  p.k = static_cast<const uint8_t *>(cache->k);
  p.v = static_cast<const uint8_t *>(cache->v);
  p.k_scale = cache->k_scale;
  p.v_scale = cache->v_scale;
  p.block_table = seqs->block_table;
  p.seq_lens = seqs->seq_lens;
  p.q = static_cast<const uint16_t *>(q);
  p.out = static_cast<uint16_t *>(out);
  p.lse = lse;
  p.ws_o = static_cast<float *>(workspace);
  p.ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                       pl.ws_o_bytes);
  p.n_groups = pl.n_groups;
  p.batch = seqs->batch;
  p.n_h = n_h;
  p.n_kv = cache->n_kv;
  p.dk = p.dv = cache->head_dim;
  p.dtype = cache->dtype;
  p.block_size = cache->block_size;
  p.num_blocks = cache->num_blocks;
  p.max_blocks = seqs->max_blocks_per_seq;
  p.max_seq_len = seqs->max_seq_len;
  p.split_len = pl.split_len;
  p.n_splits = pl.n_splits;
  p.whole_units = pl.whole_units;
  p.cluster = pl.cluster;
  p.hp = pl.hp;
  p.flags = seqs->flags;
  p.window = seqs->window;
  p.win_start = seqs->window_start;
  p.pos = pos;
  p.k_new = static_cast<const uint16_t *>(k_new);
  p.v_new = static_cast<const uint16_t *>(v_new);
  p.k_inv_scale = cache->k_inv_scale;
  p.v_inv_scale = cache->v_inv_scale;
  p.scale_log2 = log2_scale(scale, cache->head_dim);
  p.err = d->err;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = kind == DenseKernel::Simt
                      ? kvd::launch_decode_simt(p, s)
                      : kvd::launch_decode_mma(p, cache->dtype, s);
  return launched(e, "gqa_decode");
}
}  // namespace


extern "C" {

kvd_status kvd_gqa_decode(const kvd_cache *cache, const kvd_seqs *seqs,
                          const void *q, int32_t n_h, float scale, void *out,
                          float *lse, void *workspace, size_t workspace_bytes,
                          kvd_stream stream) {
  return gqa_decode_impl(cache, seqs, nullptr, nullptr, nullptr, q, n_h, scale,
                         out, lse, workspace, workspace_bytes, stream);
}

kvd_status kvd_gqa_append_decode(const kvd_cache *cache, const kvd_seqs *seqs,
                                 const int32_t *pos, const void *k_new,
                                 const void *v_new, const void *q, int32_t n_h,
                                 float scale, void *out, float *lse,
                                 void *workspace, size_t workspace_bytes,
                                 kvd_stream stream) {
  if (!pos && seqs && seqs->batch > 0)
    return fail(KVD_ERR_NULL, "gqa_append_decode: pos required");
  return gqa_decode_impl(cache, seqs, pos, k_new, v_new, q, n_h, scale, out,
                         lse, workspace, workspace_bytes, stream);
}

kvd_status kvd_mla_decode(const kvd_cache *latent, int32_t d_c,
                          const kvd_seqs *seqs, const void *q, int32_t n_h,
                          float scale, void *out, float *lse, void *workspace,
                          size_t workspace_bytes, kvd_stream stream) {
  kvd_status st = check_cache(latent, false, "mla_decode");
  if (st != KVD_OK) return st;
  st = check_seqs(seqs, latent, "mla_decode");
  if (st != KVD_OK) return st;
  st = no_window(seqs, "mla_decode");
  if (st != KVD_OK) return st;
  if (latent->dtype != KVD_BF16 || latent->n_kv != 1 || d_c != 512 ||
      latent->head_dim != 576)
    return fail(KVD_ERR_UNSUPPORTED, "mla_decode: bf16 latent cache with "
                "n_kv = 1, d_c = 512, head_dim = 576 required");
  if (n_h < 64 || n_h % 64 != 0)
    return fail(KVD_ERR_UNSUPPORTED, "mla_decode: n_h must be a multiple of 64");
  if (seqs->batch > 256)
    return fail(KVD_ERR_UNSUPPORTED, "mla_decode: at most 256 sequences");
  if (seqs->batch == 0) return ok();
  if (!q || !out) return fail(KVD_ERR_NULL, "mla_decode: q and out required");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(KVD_ERR_SHAPE, "mla_decode: q and out must be 16-byte aligned");
  const DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != KVD_OK) return st;
  const bool tc = mla_on_tensor_memory(latent, n_h);
  const Plan pl = mla_plan(seqs, n_h, d_c, d->sms, tc);
  st = check_ws(pl, workspace, workspace_bytes, "mla_decode");
  if (st != KVD_OK) return st;
  kvd::DecodeParams p{};
  p.k = p.v = static_cast<const uint8_t *>(latent->k);
  p.block_table = seqs->block_table;
  p.seq_lens = seqs->seq_lens;
  p.q = static_cast<const uint16_t *>(q);
  p.out = static_cast<uint16_t *>(out);
  p.lse = lse;
  p.ws_o = static_cast<float *>(workspace);
  p.ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                       pl.ws_o_bytes);
  p.n_groups = pl.n_groups;
  p.batch = seqs->batch;
  p.n_h = n_h;
  p.n_kv = 1;
  p.dk = latent->head_dim;
  p.dv = d_c;
  p.block_size = latent->block_size;
  p.num_blocks = latent->num_blocks;
  p.max_blocks = seqs->max_blocks_per_seq;
  p.max_seq_len = seqs->max_seq_len;
  p.split_len = pl.split_len;
  p.n_splits = pl.n_splits;
  p.scale_log2 = log2_scale(scale, latent->head_dim);
  p.err = d->err;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return launched(tc ? kvd::launch_decode_mla_tc(p, s)
                     : kvd::launch_decode_mla(p, s),
                  "mla_decode");
}

kvd_status kvd_sparse_decode(const kvd_cache *cache, const kvd_seqs *seqs,
                             const int32_t *indices, int32_t k, const void *q,
                             int32_t n_h, float scale, void *out, float *lse,
                             void *workspace, size_t workspace_bytes,
                             kvd_stream stream) {
  kvd_status st = check_cache(cache, true, "sparse_decode");
  if (st != KVD_OK) return st;
  st = check_seqs(seqs, cache, "sparse_decode");
  if (st != KVD_OK) return st;
  st = no_window(seqs, "sparse_decode");
  if (st != KVD_OK) return st;
  if (cache->dtype != KVD_BF16 || cache->n_kv != 1 || cache->head_dim != 512)
    return fail(KVD_ERR_UNSUPPORTED, "sparse_decode: bf16 cache with n_kv = 1 "
                "and head_dim = 512 required");
  if (n_h < 64 || n_h % 64 != 0)
    return fail(KVD_ERR_UNSUPPORTED,
                "sparse_decode: n_h must be a multiple of 64");
  if (k < 1) return fail(KVD_ERR_SHAPE, "sparse_decode: k must be >= 1");
  if (seqs->batch > 256)
    return fail(KVD_ERR_UNSUPPORTED, "sparse_decode: at most 256 sequences");
  if (seqs->batch == 0) return ok();
  if (!indices || !q || !out)
    return fail(KVD_ERR_NULL, "sparse_decode: indices, q and out required");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(KVD_ERR_SHAPE, "sparse_decode: q and out must be 16-byte "
                "aligned");
  const DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != KVD_OK) return st;
  const Plan pl = sparse_plan(seqs, n_h, k, cache->head_dim, d->sms);
  st = check_ws(pl, workspace, workspace_bytes, "sparse_decode");
  if (st != KVD_OK) return st;
  kvd::DecodeParams p{};
  p.k = static_cast<const uint8_t *>(cache->k);
  p.v = static_cast<const uint8_t *>(cache->v);
  p.block_table = seqs->block_table;
  p.seq_lens = seqs->seq_lens;
  p.indices = indices;
  p.q = static_cast<const uint16_t *>(q);
  p.out = static_cast<uint16_t *>(out);
  p.lse = lse;
  p.ws_o = static_cast<float *>(workspace);
  p.ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                       pl.ws_o_bytes);
  p.n_groups = pl.n_groups;
  p.batch = seqs->batch;
  p.n_h = n_h;
  p.n_kv = 1;
  p.dk = p.dv = cache->head_dim;
  p.block_size = cache->block_size;
  p.num_blocks = cache->num_blocks;
  p.max_blocks = seqs->max_blocks_per_seq;
  p.max_seq_len = seqs->max_seq_len;
  p.n_idx = k;
  p.split_len = pl.split_len;
  p.n_splits = pl.n_splits;
  p.scale_log2 = log2_scale(scale, cache->head_dim);
  p.err = d->err;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return launched(kvd::launch_decode_sparse_tc(p, s), "sparse_decode");
}

}  // extern "C"

namespace {

// kvd_indexer_topk and (pool != NULL) kvd_indexer_topk_pool.
kvd_status indexer_topk_impl(const kvd_cache *index_cache,
                             const kvd_seqs *seqs, const void *q_idx,
                             int32_t n_idx_heads, const float *w,
                             const int32_t *pool, const int32_t *pool_n,
                             int32_t k, int32_t *indices, float *scores,
                             void *workspace, size_t workspace_bytes,
                             kvd_stream stream) {
  kvd_status st = check_cache(index_cache, false, "indexer_topk");
  if (st != KVD_OK) return st;
  st = check_seqs(seqs, index_cache, "indexer_topk");
  if (st != KVD_OK) return st;
  st = no_window(seqs, "indexer_topk");
  if (st != KVD_OK) return st;
  if (index_cache->dtype != KVD_BF16 || index_cache->n_kv != 1 ||
      index_cache->head_dim != 64)
    return fail(KVD_ERR_UNSUPPORTED, "indexer_topk: bf16 K-only cache with "
                "n_kv = 1 and head_dim = 64 required");
  if (n_idx_heads < 1 || n_idx_heads > 8)
    return fail(KVD_ERR_UNSUPPORTED, "indexer_topk: 1..8 indexer heads");
  if (k < 1 || k > 16384)
    return fail(KVD_ERR_UNSUPPORTED, "indexer_topk: k must be in [1, 16384]");
  if (pool && index_cache->block_size % kvd::kPoolBlock != 0)
    return fail(KVD_ERR_UNSUPPORTED, "indexer_topk_pool: block_size must be "
                "a multiple of 8");
  if (seqs->batch == 0) return ok();
  if (!q_idx || !w || !indices)
    return fail(KVD_ERR_NULL, "indexer_topk: q_idx, w and indices required");
  if (pool && !pool_n)
    return fail(KVD_ERR_NULL, "indexer_topk_pool: pool and pool_n required");
  if (!aligned(q_idx, 16))
    return fail(KVD_ERR_SHAPE, "indexer_topk: q_idx must be 16-byte aligned");
  const DeviceInfo *d = nullptr;
  st = device_info(&d);
  if (st != KVD_OK) return st;
  const int entries = pool ? kvd::kPoolBlocks * kvd::kPoolBlock
                           : seqs->max_seq_len;
  float *sc = scores;
  if (!sc) {
    const size_t need =
        pool ? round_up((size_t)seqs->batch * entries * 4, 256)
             : topk_ws_bytes(seqs);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
      return fail(KVD_ERR_WORKSPACE, "indexer_topk: workspace of %zu bytes "
                  "(256-byte aligned) required when scores is NULL", need);
    sc = static_cast<float *>(workspace);
  }
  kvd::IndexerParams p{};
  p.cache = static_cast<const uint8_t *>(index_cache->k);
  p.block_table = seqs->block_table;
  p.seq_lens = seqs->seq_lens;
  p.q = static_cast<const uint16_t *>(q_idx);
  p.w = w;
  p.scores = sc;
  p.indices = indices;
  p.batch = seqs->batch;
  p.n_heads = n_idx_heads;
  p.block_size = index_cache->block_size;
  p.num_blocks = index_cache->num_blocks;
  p.max_blocks = seqs->max_blocks_per_seq;
  p.max_seq_len = seqs->max_seq_len;
  p.score_stride = std::max(entries, 1);
  p.topk = k;
  p.pool = pool;
  p.pool_n = pool_n;
  p.max_entries = entries;
  p.flags = seqs->flags;
  p.err = d->err;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = launched(kvd::launch_indexer_scores(p, s), "indexer_topk (scores)");
  if (st != KVD_OK) return st;
  return launched(kvd::launch_topk(p, s), "indexer_topk (select)");
}

}  // namespace

extern "C" {

kvd_status kvd_indexer_topk(const kvd_cache *index_cache, const kvd_seqs *seqs,
                            const void *q_idx, int32_t n_idx_heads,
                            const float *w, int32_t k, int32_t *indices,
                            float *scores, void *workspace,
                            size_t workspace_bytes, kvd_stream stream) {
  return indexer_topk_impl(index_cache, seqs, q_idx, n_idx_heads, w, nullptr,
                           nullptr, k, indices, scores, workspace,
                           workspace_bytes, stream);
}

kvd_status kvd_indexer_topk_pool(const kvd_cache *index_cache,
                                 const kvd_seqs *seqs, const void *q_idx,
                                 int32_t n_idx_heads, const float *w,
                                 const int32_t *pool, const int32_t *pool_n,
                                 int32_t k, int32_t *indices, float *scores,
                                 void *workspace, size_t workspace_bytes,
                                 kvd_stream stream) {
  if (!pool)
    return fail(KVD_ERR_NULL, "indexer_topk_pool: pool required");
  return indexer_topk_impl(index_cache, seqs, q_idx, n_idx_heads, w, pool,
                           pool_n, k, indices, scores, workspace,
                           workspace_bytes, stream);
}

kvd_status kvd_indexer_pool(const kvd_seqs *seqs, const int32_t *indices,
                            int32_t k, int32_t *pool, int32_t *pool_n,
                            kvd_stream stream) {
  if (!seqs) return fail(KVD_ERR_NULL, "indexer_pool: seqs is NULL");
  if (seqs->batch < 0 || seqs->batch > 65535 || seqs->max_seq_len < 0)
    return fail(KVD_ERR_SHAPE, "indexer_pool: 0 <= batch <= 65535 and "
                "max_seq_len >= 0 required");
  if (k < 1) return fail(KVD_ERR_SHAPE, "indexer_pool: k must be >= 1");
  kvd_status wst = no_window(seqs, "indexer_pool");
  if (wst != KVD_OK) return wst;
  if ((long)seqs->max_seq_len > 50331648L)
    return fail(KVD_ERR_UNSUPPORTED, "indexer_pool: max_seq_len above "
                "50,331,648");
  if (seqs->batch == 0) return ok();
  if (!seqs->seq_lens || !indices || !pool || !pool_n)
    return fail(KVD_ERR_NULL, "indexer_pool: seq_lens, indices, pool and "
                "pool_n required");
  const DeviceInfo *d = nullptr;
  kvd_status st = device_info(&d);
  if (st != KVD_OK) return st;
  kvd::PoolParams p{};
  p.indices = indices;
  p.seq_lens = seqs->seq_lens;
  p.pool = pool;
  p.pool_n = pool_n;
  p.batch = seqs->batch;
  p.k = k;
  p.max_seq_len = seqs->max_seq_len;
  p.err = d->err;
  return launched(kvd::launch_indexer_pool(
                      p, reinterpret_cast<cudaStream_t>(stream)),
                  "indexer_pool");
}

}  // extern "C"

// Indexer scores and top-k selection (the My Weird Prompts 640482
// transcript on DeepSeek Sparse Attention: a lightning indexer scores the
// cached prefix and a top-k subset of positions, k = 2048, is read; "890
// bytes a token ...", section 3: Full and Reindex layers score with their
// own indexer query over a shared indexer key cache).
//
// Scores: s_t = sum_j w_j * max(0, q_j . k_t) for every visible position t,
// with the 64-wide indexer keys read from the paged K-only cache. Eight
// lanes cover one key row (16 bytes each, one coalesced 128-byte read per
// row); the lane's slice of every indexer query is held in registers, each
// dot product finishes with three xor-shuffles, and the sum is formed in
// fp32.
//
// Selection: the k largest scores of a sequence, equal scores taken in
// ascending position order, returned as ascending positions (-1 padding
// when fewer than k positions are visible). A cluster of eight CTAs per
// sequence runs an exact radix select on order-preserving 32-bit keys of
// the fp32 scores (negative zero counted as zero): three histogram passes
// (12, 12 and 8 bits), summed across the cluster in distributed shared
// memory, find the k-th largest key K* and how many keys exceed it; a final
// pass in position order keeps every key above K* and the lowest-indexed
// keys equal to K*, placing each kept position with block-wide prefix sums
// after the selections of the lower-ranked CTAs. The result is exactly the
// selection the scores define.
#include <cmath>

#include "kvd_common.cuh"

namespace kvd {
namespace {

// ---------------------------------------------------------------------------
// scores
// ---------------------------------------------------------------------------
constexpr int kIdxDim = 64;
constexpr int kScoreThreads = 256;
constexpr int kTokPerCta = 1024;

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <int H>
__global__ void __launch_bounds__(kScoreThreads)
    indexer_score_kernel(const IndexerParams p) {
  const int b = blockIdx.y;
  int T = p.seq_lens[b];
  T = max(0, min(T, p.max_seq_len));
  const int t0 = blockIdx.x * kTokPerCta;
  if (t0 >= T) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane >> 3, sub = lane & 7;
  // this lane's 8 dims of every indexer query, and the head weights
  float qf[H][8], w[H];
#pragma unroll
  for (int j = 0; j < H; ++j) {
    if (j < p.n_heads) {
      const uint4 u = *reinterpret_cast<const uint4 *>(
          p.q + ((long)b * p.n_heads + j) * kIdxDim + sub * 8);
      const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qf[j][2 * e] = bf16lo(v[e]);
        qf[j][2 * e + 1] = bf16hi(v[e]);
      }
      w[j] = p.w[(long)b * p.n_heads + j];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[j][e] = 0.f;
      w[j] = 0.f;
    }
  }
  const int32_t *bt = p.block_table + (long)b * p.max_blocks;
  float *out = p.scores + (long)b * p.score_stride;
  constexpr int kUnroll = 8;
  // warp w, lane group g: tokens t0 + 32 * it + 4 * w + g
  for (int it0 = 0; it0 < kTokPerCta / 32; it0 += kUnroll) {
    uint4 kv[kUnroll];
    int tok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      tok[u] = t0 + 32 * (it0 + u) + 4 * warp + grp;
      kv[u] = make_uint4(0, 0, 0, 0);
      if (tok[u] < T) {
        int blk = bt[tok[u] / p.block_size];
        if (blk < 0 || blk >= p.num_blocks) {
          report(p.err, DEVERR_BLOCK);
          blk = 0;  // read a valid block; the result is flagged as wrong
        }
        const long row = (long)blk * p.block_size + tok[u] % p.block_size;
        kv[u] = ld_stream(p.cache + (row * kIdxDim + sub * 8) * 2);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t v[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
      float kf[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kf[2 * e] = bf16lo(v[e]);
        kf[2 * e + 1] = bf16hi(v[e]);
      }
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < H; ++j) {
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) d = fmaf(qf[j][e], kf[e], d);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        s = fmaf(w[j], fmaxf(d, 0.f), s);
      }
      if (sub == 0 && tok[u] < T) out[tok[u]] = s;
    }
  }
}

// ---------------------------------------------------------------------------
// top-k
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 1024;
constexpr int kBins = 4096;

// Order-preserving key of an fp32 score; -0 counts as +0.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix sum of `v` (1024 threads); *total = sum.
__device__ __forceinline__ int block_excl_scan(int v, int *tmp, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = tmp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    tmp[lane] = t;  // inclusive warp totals
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? tmp[warp - 1] : 0);
  *total = tmp[31];
  __syncthreads();
  return excl;
}

// ---- thread-block cluster helpers (distributed shared memory) ----
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Load an int from the shared memory of CTA `rank` of this cluster, at the
// address `local` has in the calling CTA.
__device__ __forceinline__ int ld_cluster(const int *local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(smem_u32(local)), "r"(rank));
  int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote)
               : "memory");
  return v;
}

constexpr int kCluster = 8;  // CTAs per sequence

// One cluster per sequence; CTA r of the cluster owns positions
// [r T / 8, (r + 1) T / 8). Histograms are summed across the cluster
// through distributed shared memory (each CTA reads the 8 copies of the
// bins it scans); all CTAs reach the same digits. The compaction places
// each CTA's selections after those of the lower-ranked CTAs.
__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const IndexerParams p) {
  __shared__ int hist[2][kBins];  // double-buffered across passes
  __shared__ int tmp[32];
  __shared__ int s_digit, s_above;
  __shared__ int s_counts[2];  // this CTA's keys above / equal to K*
  const uint32_t rank = cluster_rank();
  const int b = blockIdx.x / kCluster;
  const int tid = threadIdx.x;
  int T = p.seq_lens[b];
  T = max(0, min(T, p.max_seq_len));
  const int k = p.topk;
  const float *sc = p.scores + (long)b * p.score_stride;
  int32_t *out = p.indices + (long)b * k;
  if (T <= k) {  // every position, then -1 padding (uniform per cluster)
    if (rank == 0)
      for (int i = tid; i < k; i += kTopkThreads) out[i] = i < T ? i : -1;
    return;
  }
  const int r0 = (int)((long)T * rank / kCluster);
  const int r1 = (int)((long)T * (rank + 1) / kCluster);
  // ---- radix select of the k-th largest key ----
  uint32_t prefix = 0;  // digits chosen so far
  int remaining = k;    // keys still to take at or below the prefix
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
  for (int pass = 0; pass < 3; ++pass) {
    int *h = hist[pass & 1];
    const int shift = shifts[pass], bits = widths[pass];
    const int nb = 1 << bits;
    const int hi_shift = shift + bits;  // bits above this digit
    for (int i = tid; i < kBins; i += kTopkThreads) h[i] = 0;
    __syncthreads();
    constexpr int kU = 16;  // independent loads in flight per thread
    for (int base = r0; base < r1; base += kU * kTopkThreads) {
      float v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * kTopkThreads + tid;
        v[u] = i < r1 ? sc[i] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * kTopkThreads + tid;
        const uint32_t key = score_key(v[u]);
        const bool match =
            i < r1 && (hi_shift >= 32 || (key >> hi_shift) == prefix);
        const int digit = match ? (int)((key >> shift) & (nb - 1)) : -1;
        // warp-aggregated increments: one atomic per distinct digit
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        if (match && (__ffs(peers) - 1) == (tid & 31))
          atomicAdd(&h[digit], __popc(peers));
      }
    }
    cluster_sync();  // every CTA's histogram of this pass is complete
    // suffix sums over thread ranges of bins (high digits first), summing
    // the cluster's copies of each bin
    const int per = (nb + kTopkThreads - 1) / kTopkThreads;
    const int r = kTopkThreads - 1 - tid;  // reversed: thread 0 owns the top
    int cnt[4] = {0, 0, 0, 0};
    int local = 0;
    for (int j = 0; j < per; ++j) {
      const int d = r * per + j;
      if (d < nb) {
        int c = 0;
        for (uint32_t q = 0; q < kCluster; ++q) c += ld_cluster(&h[d], q);
        cnt[j] = c;
        local += c;
      }
    }
    int tot;
    const int before = block_excl_scan(local, tmp, &tot);  // bins above range
    if (before < remaining && before + local >= remaining) {
      int acc = before;
      for (int j = per - 1; j >= 0; --j) {
        const int d = r * per + j;
        if (d >= nb) continue;
        if (acc + cnt[j] >= remaining) {
          s_digit = d;
          s_above = acc;
          break;
        }
        acc += cnt[j];
      }
    }
    __syncthreads();
    prefix = (prefix << bits) | (uint32_t)s_digit;
    remaining -= s_above;
    __syncthreads();
  }
  const uint32_t kstar = prefix;
  const int need_eq = remaining;  // keys equal to K* to take (>= 1)
  // ---- counts of this CTA's keys above / equal to K* ----
  constexpr int kPer = 16;  // consecutive positions per thread
  int my_gt = 0, my_eq = 0;
  for (int base = r0; base < r1; base += kPer * kTopkThreads) {
    const int i0 = base + kPer * tid;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (i0 + j < r1) {
        const uint32_t key = score_key(sc[i0 + j]);
        my_gt += key > kstar;
        my_eq += key == kstar;
      }
    }
  }
  int tot_gt, tot_eq0;
  block_excl_scan(my_gt, tmp, &tot_gt);
  block_excl_scan(my_eq, tmp, &tot_eq0);
  if (tid == 0) {
    s_counts[0] = tot_gt;
    s_counts[1] = tot_eq0;
  }
  cluster_sync();
  // selections and equal keys of the lower-ranked CTAs
  int run_sel = 0, run_eq = 0;
  for (uint32_t q = 0; q < rank; ++q) {
    const int g = ld_cluster(&s_counts[0], q);
    const int e = ld_cluster(&s_counts[1], q);
    run_sel += g + max(0, min(e, need_eq - run_eq));
    run_eq += e;
  }
  // ---- compaction of this CTA's range in position order ----
  for (int base = r0; base < r1; base += kPer * kTopkThreads) {
    const int i0 = base + kPer * tid;
    float v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) v[j] = i0 + j < r1 ? sc[i0 + j] : 0.f;
    unsigned gt = 0, eq = 0;  // bit j: position i0 + j above / at K*
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint32_t key = score_key(v[j]);
      if (i0 + j < r1) {
        gt |= (key > kstar ? 1u : 0u) << j;
        eq |= (key == kstar ? 1u : 0u) << j;
      }
    }
    int tot_eq;
    const int eq_before = run_eq + block_excl_scan(__popc(eq), tmp, &tot_eq);
    unsigned sel = gt;
    int e = eq_before;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if ((eq >> j) & 1) {
        if (e < need_eq) sel |= 1u << j;
        ++e;
      }
    }
    int tot_sel;
    int pos = run_sel + block_excl_scan(__popc(sel), tmp, &tot_sel);
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (((sel >> j) & 1) && pos < k) out[pos++] = i0 + j;
    run_eq += tot_eq;
    run_sel += tot_sel;
  }
  cluster_sync();  // no CTA leaves while another may read its shared memory
}

}  // namespace

cudaError_t launch_indexer_scores(const IndexerParams &p, cudaStream_t s) {
  if (p.batch == 0 || p.max_seq_len == 0) return cudaSuccess;
  dim3 grid((p.max_seq_len + kTokPerCta - 1) / kTokPerCta, p.batch);
  if (p.n_heads <= 1)
    indexer_score_kernel<1><<<grid, kScoreThreads, 0, s>>>(p);
  else if (p.n_heads <= 2)
    indexer_score_kernel<2><<<grid, kScoreThreads, 0, s>>>(p);
  else if (p.n_heads <= 4)
    indexer_score_kernel<4><<<grid, kScoreThreads, 0, s>>>(p);
  else if (p.n_heads <= 8)
    indexer_score_kernel<8><<<grid, kScoreThreads, 0, s>>>(p);
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

cudaError_t launch_topk(const IndexerParams &p, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.batch * kCluster);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel, p);
}

}  // namespace kvd

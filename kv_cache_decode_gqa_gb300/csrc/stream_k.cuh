// Stream-K work partition for the dense decode kernels.
//
// The work of one decode launch is every 64-token chunk of every unit
// u = (sequence b, kv head h): n_b = ceil(T_b / 64) chunks per unit, laid
// out in order (b, h, chunk). The P CTAs of a persistent launch take equal
// contiguous ranges [lo(c), hi(c)) of that list, so the copy engine of every
// SM streams the same number of bytes whatever the sequence lengths are.
// A unit lying wholly inside one CTA's range is finished by that CTA; a
// unit cut between CTAs leaves one partial result per covering CTA (at most
// two per CTA: the unit its range starts in and the unit it ends in), which
// the last covering CTA to finish merges (log-sum-exp merge).
#pragma once

#include "kvd_common.cuh"

namespace kvd {

constexpr int kMaxDecodeBatch = 1024;

// Chunk list of one launch: `units` units per sequence (kv heads, or query
// head tiles) of nch[b] chunks each.
template <int NB>
struct WorkPartitionT {
  int total;        // chunks in the launch
  int units;        // units per sequence
  int pre[NB + 1];  // first chunk of sequence b's first unit
  int nch[NB];      // chunks per unit of sequence b
  int len[NB];      // visible length of sequence b (clamped)
};
using WorkPartition = WorkPartitionT<kMaxDecodeBatch>;

// Fill `wp` (shared memory) from the device sequence lengths. Sequence b
// has `units` units of ceil(rows_b / chunk) chunks, rows_b = its visible
// length, or `fixed_rows` (a position list's length) when that is > 0 and
// the sequence is not empty. Every thread of the block calls it (blockDim.x
// a multiple of 32); it ends with a barrier.
template <int NB>
__device__ __forceinline__ void build_partition(WorkPartitionT<NB> &wp,
                                                const DecodeParams &p,
                                                int *len_error,
                                                int chunk = kStageRows,
                                                int units = -1,
                                                int fixed_rows = 0) {
  const int nthreads = blockDim.x;
  const int tid = threadIdx.x;
  if (units < 0) units = p.n_kv;
  for (int b = tid; b < p.batch; b += nthreads) {
    int T = p.seq_lens[b];
    if (T > p.max_seq_len) {
      *len_error = 1;
      T = p.max_seq_len;
    }
    T = max(T, 0);
    wp.len[b] = T;
    const int rows = (fixed_rows > 0 && T > 0) ? fixed_rows : T;
    wp.nch[b] = (rows + chunk - 1) / chunk;
  }
  if (tid == 0) wp.units = units;
  __syncthreads();
  // exclusive scan over b of the chunks of sequence b's n_kv units: each
  // thread sums a run of consecutive sequences, then warp and block scans
  __shared__ int warp_tot[32];
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  const int per = (p.batch + nthreads - 1) / nthreads;
  const int b0 = tid * per;
  int local = 0;
  for (int j = 0; j < per; ++j)
    if (b0 + j < p.batch) local += wp.nch[b0 + j] * units;
  int x = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    if (lane < nwarps) warp_tot[lane] = t;
  }
  __syncthreads();
  int excl = x - local + (warp > 0 ? warp_tot[warp - 1] : 0);
  for (int j = 0; j < per; ++j) {
    if (b0 + j < p.batch) {
      wp.pre[b0 + j] = excl;
      excl += wp.nch[b0 + j] * units;
    }
  }
  if (tid == 0) {
    wp.total = warp_tot[nwarps - 1];
    wp.pre[p.batch] = wp.total;
  }
  __syncthreads();
}

// Sequence owning global chunk x (0 <= x < total): the largest b with
// pre[b] <= x (sequences without chunks share the next one's prefix).
template <int NB>
__device__ __forceinline__ int find_seq(const WorkPartitionT<NB> &wp,
                                        int batch, int x) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (wp.pre[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int range_lo(int c, int total, int P) {
  return (int)(((long long)c * total) / P);
}

// The CTA whose range holds chunk x (P <= total, so no range is empty).
__device__ __forceinline__ int cta_of(int x, int total, int P) {
  return (int)((((long long)x + 1) * P - 1) / total);
}

struct ChunkCursor {
  int b, h, k;  // sequence, kv head, chunk within the unit
};

template <int NB>
__device__ __forceinline__ ChunkCursor cursor_at(const WorkPartitionT<NB> &wp,
                                                 int batch, int x) {
  ChunkCursor cur;
  cur.b = find_seq(wp, batch, x);
  const int off = x - wp.pre[cur.b];
  cur.h = off / wp.nch[cur.b];
  cur.k = off % wp.nch[cur.b];
  return cur;
}

template <int NB>
__device__ __forceinline__ void cursor_next(const WorkPartitionT<NB> &wp,
                                            int batch, int n_kv,
                                            ChunkCursor &cur) {
  if (++cur.k < wp.nch[cur.b]) return;
  cur.k = 0;
  if (++cur.h < n_kv) return;
  cur.h = 0;
  do {
    ++cur.b;
  } while (cur.b < batch && wp.nch[cur.b] == 0);
}

// Slot of a CTA's partial result for a unit starting at chunk `ustart`:
// side 0 for the unit its range starts inside, 1 for the unit it ends in.
__device__ __forceinline__ int partial_side(int ustart, int lo) {
  return ustart < lo ? 0 : 1;
}

// Arrival counter increment with release semantics: the partial results
// this CTA wrote (ordered before this call by a barrier) become visible
// before the increment does. Returns the previous count.
__device__ __forceinline__ int arrive_release(int *ctr) {
  int prev;
  asm volatile("atom.release.gpu.global.add.s32 %0, [%1], 1;"
               : "=r"(prev)
               : "l"(ctr)
               : "memory");
  return prev;
}

// Merge the partials of every unit in `merge` (unit start chunks, -1 for
// none): out = sum_s w_s o_s with w_s = e^(lse_s - M) / sum_s e^(lse_s - M),
// M = max_s lse_s, and lse = M + ln sum_s e^(lse_s - M). Thread `t` of `nt`
// cooperating threads (named barrier `bar`). `scratch` (cap floats) first
// holds the parts' lse values, then their weights e^(lse_s - M); the partial
// outputs are then summed part by part with batches of independent 16-byte
// loads, so a part costs about one L2 round trip. Part i is the partial of
// CTA c_first + i: side 1 of the first covering CTA, side 0 of the others.
template <int D, int G, int NB>
__device__ __forceinline__ void merge_owed(const DecodeParams &p,
                                           const WorkPartitionT<NB> &wp,
                                           const int *merge, float *scratch,
                                           int cap, int total, int P, int t,
                                           int nt, int bar) {
  static_assert(D % 4 == 0, "vector loads");
  float *mg = scratch + cap - 2 * G;  // per-head M and 1 / W
  for (int j = 0; j < 2; ++j) {
    const int ustart = merge[j];
    if (ustart < 0) continue;
    const int b = find_seq(wp, p.batch, ustart);
    const int h = (ustart - wp.pre[b]) / wp.nch[b];
    const int uend = ustart + wp.nch[b];
    const int c_first = cta_of(ustart, total, P);
    const int parts = cta_of(uend - 1, total, P) - c_first + 1;
    const long bh0 = (long)b * p.n_h + (long)h * G;  // first head of the unit
    const bool staged = parts * G <= cap - 2 * G;
    auto slot = [&](int i) { return (c_first + i) * 2 + (i == 0 ? 1 : 0); };
    __threadfence();
    if (staged)
      for (int i = t; i < parts * G; i += nt)
        scratch[i] = __ldcg(p.ws_lse + (long)slot(i / G) * G + i % G);
    named_sync(bar, nt);
    for (int g = t; g < G; g += nt) {
      float M = -INFINITY;
      for (int i = 0; i < parts; ++i)
        M = fmaxf(M, staged ? scratch[i * G + g]
                            : __ldcg(p.ws_lse + (long)slot(i) * G + g));
      float W = 0.f;
      for (int i = 0; i < parts; ++i) {
        const float l = staged ? scratch[i * G + g]
                               : __ldcg(p.ws_lse + (long)slot(i) * G + g);
        const float w = M == -INFINITY ? 0.f : expf(l - M);
        if (staged) scratch[i * G + g] = w;
        W += w;
      }
      mg[g] = M;
      mg[G + g] = W > 0.f ? 1.f / W : 0.f;
      if (p.lse) p.lse[bh0 + g] = W > 0.f ? M + logf(W) : -INFINITY;
    }
    named_sync(bar, nt);
    constexpr int kBatch = 8;  // float4 loads in flight per thread
    const int n4 = G * D / 4;
    for (int e0 = t; e0 < n4; e0 += nt * kBatch) {
      float4 acc[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i < parts; ++i) {
        const float4 *src =
            reinterpret_cast<const float4 *>(p.ws_o + (long)slot(i) * G * D);
        float4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int e = e0 + u * nt;
          v[u] = e < n4 ? __ldcg(src + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int e = e0 + u * nt;
          if (e >= n4) continue;
          const int g = (4 * e) / D;
          float w;
          if (staged) {
            w = scratch[i * G + g];
          } else {
            const float M = mg[g];
            w = M == -INFINITY
                    ? 0.f
                    : expf(__ldcg(p.ws_lse + (long)slot(i) * G + g) - M);
          }
          acc[u].x = fmaf(w, v[u].x, acc[u].x);
          acc[u].y = fmaf(w, v[u].y, acc[u].y);
          acc[u].z = fmaf(w, v[u].z, acc[u].z);
          acc[u].w = fmaf(w, v[u].w, acc[u].w);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * nt;
        if (e >= n4) continue;
        const int g = (4 * e) / D;
        const float iw = mg[G + g];
        uint2 packed;
        packed.x = pack_bf16x2(acc[u].x * iw, acc[u].y * iw);
        packed.y = pack_bf16x2(acc[u].z * iw, acc[u].w * iw);
        *reinterpret_cast<uint2 *>(p.out + bh0 * D + 4 * e) = packed;
      }
    }
    named_sync(bar, nt);
  }
}

}  // namespace kvd

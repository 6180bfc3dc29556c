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
// none): out = sum_s w_s o_s, w_s = e^(lse_s - M) / sum e^(lse_s - M),
// lse = M + ln sum e^(lse_s - M). Thread `t` of `nt` cooperating threads (named barrier `bar`);
// `scratch` holds the weights (one float per part). Every load of a pass is
// independent, so a pass costs about one L2 round trip.
template <int D, int G, int NB>
__device__ __forceinline__ void merge_owed(const DecodeParams &p,
                                           const WorkPartitionT<NB> &wp,
                                           const int *merge, float *scratch,
                                           int cap, int total, int P, int t,
                                           int nt, int bar) {
  for (int j = 0; j < 2; ++j) {
    const int ustart = merge[j];
    if (ustart < 0) continue;
    const int b = find_seq(wp, p.batch, ustart);
    const int h = (ustart - wp.pre[b]) / wp.nch[b];
    const int uend = ustart + wp.nch[b];
    const int c_first = cta_of(ustart, total, P);
    const int parts = cta_of(uend - 1, total, P) - c_first + 1;
    const long bh0 = (long)b * p.n_h + (long)h * G;  // first head of the unit
    __threadfence();
    // pass 1: lse of every part (part i of CTA c_first + i; the first CTA's
    // partial for this unit is its side-1 slot, the others' their side 0),
    // kept in shared memory when they fit
    const bool staged = parts * G <= cap;
    for (int i = t; staged && i < parts * G; i += nt) {
      const int part = i / G, g = i % G;
      const int ws = (c_first + part) * 2 + (part == 0 ? 1 : 0);
      scratch[i] = __ldcg(p.ws_lse + (long)ws * G + g);
    }
    named_sync(bar, nt);
    for (int idx = t; idx < G * D; idx += nt) {
      const int g = idx / D, d = idx % D;
      auto lse_of = [&](int i) {
        const int ws = (c_first + i) * 2 + (i == 0 ? 1 : 0);
        return staged ? scratch[i * G + g] : __ldcg(p.ws_lse + (long)ws * G + g);
      };
      float M = -INFINITY;
      for (int i = 0; i < parts; ++i) M = fmaxf(M, lse_of(i));
      float W = 0.f, acc = 0.f;
      // pass 2: the partial outputs
      for (int i = 0; i < parts; ++i) {
        const int ws = (c_first + i) * 2 + (i == 0 ? 1 : 0);
        const float w = expf(lse_of(i) - M);
        W += w;
        acc = fmaf(w, __ldcg(p.ws_o + ((long)ws * G + g) * D + d), acc);
      }
      const long bh = bh0 + g;
      p.out[bh * D + d] = f2bf(acc / W);
      if (d == 0 && p.lse) p.lse[bh] = M + logf(W);
    }
    named_sync(bar, nt);
  }
}

}  // namespace kvd

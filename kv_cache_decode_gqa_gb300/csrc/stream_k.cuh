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
// a short second launch merges (log-sum-exp merge).
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

// First position sequence b attends to (its visible length is T): the
// sliding window's and the replay start's lower bound, 0 without them.
__device__ __forceinline__ int seq_lo(const DecodeParams &p, int b, int T) {
  int lo = p.win_start ? p.win_start[b] : 0;
  if (p.window > 0) lo = max(lo, T - p.window);
  return min(max(lo, 0), T);
}

// Position of the first row of sequence b's first chunk: its first
// attended position rounded down to the chunk size (rows below `lo` in
// that chunk are copied and masked).
__device__ __forceinline__ int seq_first(const DecodeParams &p, int b, int T,
                                         int chunk) {
  const int lo = seq_lo(p, b, T);
  return lo - lo % chunk;
}

// Whether any sequence of the call has a lower bound (window or start).
__device__ __forceinline__ bool has_window(const DecodeParams &p) {
  return p.window > 0 || p.win_start != nullptr;
}

// Fill `wp` (shared memory) from the device sequence lengths. Sequence b
// has `units` units of ceil(rows_b / chunk) chunks, rows_b = its visible
// length from its first chunk's start (seq_first; 0 when nothing is
// attended). Every thread of the block calls it (blockDim.x a multiple of
// 32); it ends with a barrier.
template <int NB>
__device__ __forceinline__ void build_partition(WorkPartitionT<NB> &wp,
                                                const DecodeParams &p,
                                                int *len_error,
                                                int chunk = kStageRows,
                                                int units = -1) {
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
    const int lo = seq_lo(p, b, T);
    const int rows = lo < T ? T - (lo - lo % chunk) : 0;
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

// First chunk of unit u, units in (sequence, head group) order; u = batch x
// n_units gives the end of the last (the range of CTA c of a whole-unit
// launch is [unit_lo(c), unit_lo(c + 1))).
template <int NB>
__device__ __forceinline__ int unit_lo(const WorkPartitionT<NB> &wp,
                                      int batch, int n_units, int u) {
  const int b = u / n_units;
  if (b >= batch) return wp.total;
  return wp.pre[b] + (u % n_units) * wp.nch[b];
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

// ---------------------------------------------------------------------------
// fused append (kvd_gqa_append_decode)
// ---------------------------------------------------------------------------
// The calling warp writes the new key and value rows of kv heads
// [h0, h0 + nh) of sequence b into slot P of physical block pb (checked by
// the caller), lane-parallel over 8-element pieces (16-channel groups for
// an MXFP4 cache), and each lane orders its writes before later
// copy-engine reads of the same rows.
__device__ __forceinline__ void append_rows(const DecodeParams &p, int b,
                                            int h0, int nh, int P, int pb,
                                            int lane) {
  const int D = p.dk, es = p.dtype == DT_BF16 ? 2 : 1;
  if (p.dtype == DT_MXFP4) {
    const int groups = D / 16, rb = row_bytes(D, DT_MXFP4);
    for (int e = lane; e < 2 * nh * groups; e += 32) {
      const bool is_v = e >= nh * groups;
      const int r = is_v ? e - nh * groups : e;
      const int h = h0 + r / groups, g = r % groups;
      const uint16_t *src =
          (is_v ? p.v_new : p.k_new) + ((long)b * p.n_kv + h) * D + g * 16;
      const long row =
          ((long)pb * p.n_kv + h) * p.block_size + P % p.block_size;
      uint8_t *rowp = const_cast<uint8_t *>(is_v ? p.v : p.k) + row * rb;
      store_mxfp4_group(rowp + g * 8, rowp + D / 2 + g, src);
    }
    fence_proxy_async_global();
    __syncwarp();
    return;
  }
  const int pieces = D / 8;
  for (int e = lane; e < 2 * nh * pieces; e += 32) {
    const bool is_v = e >= nh * pieces;
    const int r = is_v ? e - nh * pieces : e;
    const int h = h0 + r / pieces, c8 = r % pieces;
    const uint16_t *src =
        (is_v ? p.v_new : p.k_new) + ((long)b * p.n_kv + h) * D + c8 * 8;
    const long row =
        ((long)pb * p.n_kv + h) * p.block_size + P % p.block_size;
    uint8_t *dst = const_cast<uint8_t *>(is_v ? p.v : p.k) +
                   (row * D + c8 * 8) * es;
    const float inv = p.dtype == DT_BF16
                          ? 1.0f
                          : (is_v ? p.v_inv_scale : p.k_inv_scale)[h];
    store_new8(dst, src, p.dtype, inv);
  }
  fence_proxy_async_global();
  __syncwarp();
}

// The fused-append rows that this CTA's chunk range [lo, hi) will read:
// for every unit (b, h) the range touches whose sequence's new slot pos[b]
// is visible and lies in one of the range's chunks, the calling warp writes
// the unit's `nh` kv heads' rows (a block id out of range is left to the
// copy of that chunk to flag). Units are taken 32 at a time: a walk of the
// partition gives lane j the j-th unit, the lanes load their slots and
// block ids together, then the warp writes the rows unit by unit. With
// `wait_first` (stable metadata) the loads of the first 32 units run before
// the grid dependency wait and the writes after it. Run by a warp that
// issues no copies, before the producer copies the first such chunk.
template <int NB>
__device__ __forceinline__ void append_range_rows(
    const DecodeParams &p, const WorkPartitionT<NB> &wp, int nh, int lo,
    int hi, int lane, bool wait_first) {
  int x = lo;
  bool waited = !wait_first;
  do {
    int mb = -1, mh = 0, mstart = 0;
    for (int j = 0; j < 32 && x < hi; ++j) {  // warp-uniform, shared memory
      const ChunkCursor u = cursor_at(wp, p.batch, x);
      const int ustart = wp.pre[u.b] + u.h * wp.nch[u.b];
      if (lane == j) mb = u.b, mh = u.h, mstart = ustart;
      x = min(ustart + wp.nch[u.b], hi);
    }
    int P = -1, pb = -1;
    if (mb >= 0) {
      P = p.pos[mb];
      const int first = seq_first(p, mb, wp.len[mb], kStageRows);
      const int xp = mstart + (P - first) / kStageRows;  // chunk holding P
      if (P >= first && P < wp.len[mb] && wp.nch[mb] > 0 && xp >= lo &&
          xp < hi)
        pb = p.block_table[(long)mb * p.max_blocks + P / p.block_size];
    }
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    unsigned todo = __ballot_sync(0xffffffffu, pb >= 0 && pb < p.num_blocks);
    while (todo) {
      const int j = __ffs(todo) - 1;
      todo &= todo - 1;
      append_rows(p, __shfl_sync(0xffffffffu, mb, j),
                  __shfl_sync(0xffffffffu, mh, j) * nh, nh,
                  __shfl_sync(0xffffffffu, P, j),
                  __shfl_sync(0xffffffffu, pb, j), lane);
    }
  } while (x < hi);
}

// Rows of the fused append that no chunk of this launch reads (a slot at or
// past the visible length, an empty sequence) or that are out of range: one
// warp of CTA 0 writes the former and flags the latter, as kv_append does.
// Visible rows are written by the producer that copies their chunk.
template <int NB>
__device__ __forceinline__ void append_unread_rows(
    const DecodeParams &p, const WorkPartitionT<NB> &wp, int lane) {
  for (int b0 = 0; b0 < p.batch; b0 += 32) {
    const int b = b0 + lane;
    int P = 0, need = 0;
    if (b < p.batch) {
      P = p.pos[b];
      const int first = seq_first(p, b, wp.len[b], kStageRows);
      need = !(P >= first && P < wp.len[b] && wp.nch[b] > 0);
    }
    unsigned todo = __ballot_sync(0xffffffffu, need);
    while (todo) {
      const int j = __ffs(todo) - 1;
      todo &= todo - 1;
      const int bj = b0 + j;
      const int Pj = __shfl_sync(0xffffffffu, P, j);
      if (Pj < 0 || Pj >= p.max_blocks * p.block_size) {
        if (lane == 0) report(p.err, DEVERR_POS);
        continue;
      }
      const int pb = p.block_table[(long)bj * p.max_blocks + Pj / p.block_size];
      if (pb < 0 || pb >= p.num_blocks) {
        if (lane == 0) report(p.err, DEVERR_BLOCK);
        continue;
      }
      append_rows(p, bj, 0, p.n_kv, Pj, pb, lane);
    }
  }
}

// Online log-sum-exp merge of the partials of one float4 of outputs, its
// parts split over an aligned group of LANES (1 or 4) lanes: lane q takes
// parts q, q + LANES, ... with up to 8 of its loads in flight at once (so
// 8 LANES parts take one round), then the group's states are combined with
// xor-shuffles. `slot(i)` is part i's partial slot; `lse` / `o` point at
// the partials' log-sum-exps and outputs, `g` / `e` index the head and the
// float4 within a slot of `gu` heads x `d` values. Every lane of the warp
// calls it (inactive ones with parts = 0). On return the quad's lanes hold
// M = max lse, W = sum e^(lse - M), acc = sum e^(lse - M) o.
template <int LANES, class SlotF>
__device__ __forceinline__ void quad_merge(const float *lse, const float *o,
                                           int gu, int d, int g, int e,
                                           int parts, SlotF slot, float &M,
                                           float &W, float4 &acc) {
  const int q = threadIdx.x & (LANES - 1);
  M = -INFINITY;
  W = 0.f;
  acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = q; i0 < parts; i0 += 8 * LANES) {
    float4 v[8];
    float l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + LANES * j;
      if (i < parts) {
        const long sl = slot(i);
        l[j] = __ldcg(lse + sl * gu + g);
        v[j] = __ldcg(reinterpret_cast<const float4 *>(o + sl * gu * d) + e);
      } else {
        l[j] = -INFINITY;
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (l[j] == -INFINITY) continue;  // an empty part adds nothing
      const float Mn = fmaxf(M, l[j]);
      const float a = M == -INFINITY ? 0.f : expf(M - Mn);
      const float w = expf(l[j] - Mn);
      W = W * a + w;
      acc.x = acc.x * a + w * v[j].x;
      acc.y = acc.y * a + w * v[j].y;
      acc.z = acc.z * a + w * v[j].z;
      acc.w = acc.w * a + w * v[j].w;
      M = Mn;
    }
  }
#pragma unroll
  for (int off = 1; off < LANES; off <<= 1) {
    const float M2 = __shfl_xor_sync(0xffffffffu, M, off);
    const float W2 = __shfl_xor_sync(0xffffffffu, W, off);
    float4 a2;
    a2.x = __shfl_xor_sync(0xffffffffu, acc.x, off);
    a2.y = __shfl_xor_sync(0xffffffffu, acc.y, off);
    a2.z = __shfl_xor_sync(0xffffffffu, acc.z, off);
    a2.w = __shfl_xor_sync(0xffffffffu, acc.w, off);
    const float Mn = fmaxf(M, M2);
    const float a = M == -INFINITY ? 0.f : expf(M - Mn);
    const float b = M2 == -INFINITY ? 0.f : expf(M2 - Mn);
    W = W * a + W2 * b;
    acc.x = acc.x * a + a2.x * b;
    acc.y = acc.y * a + a2.y * b;
    acc.z = acc.z * a + a2.z * b;
    acc.w = acc.w * a + a2.w * b;
    M = Mn;
  }
}

// Log-sum-exp merge of the units a dense decode launch cut between CTAs,
// run as a second launch right after it (programmatic dependent launch, so
// its CTAs are resident and waiting when the decode grid completes). Each
// CTA rebuilds the partition from the sequence lengths and takes units
// u = blockIdx.x, + gridDim.x, ...; for a unit covered by more than one
// CTA it merges, per float4 of outputs (4 values of one head), the parts'
// partial results with an online log-sum-exp merge (quad_merge: 4 lanes
// per float4, all of a lane's loads in flight at once):
//   out = sum_s w_s o_s,  w_s = e^(lse_s - M) / sum_s e^(lse_s - M),
//   M = max_s lse_s,  lse = M + ln sum_s e^(lse_s - M).
// Part i is the partial of CTA c_first + i: side 1 of the first covering
// CTA, side 0 of the others. Units inside one CTA were written whole.
constexpr int kMergeThreads = 256;
// Partition capacity of the merge launch for batches up to 64: its CTAs then
// hold under 1 KB of shared memory, so that one fits beside a decode CTA of
// the next call (which holds up to ~215 KB) instead of delaying its start.
constexpr int kMergeSmallBatch = 64;

template <int D, int GU, int NB>
__global__ void __launch_bounds__(kMergeThreads)
    merge_dense_kernel(const DecodeParams p, int n_units) {
  __shared__ WorkPartitionT<NB> wp;
  __shared__ int s_len_err;
  pdl_trigger();
  // The lengths may be read before the decode launch completes: that launch
  // (this launch's only possible predecessor still running, since it lets
  // its dependants start only after its own predecessor has completed)
  // does not write them. The partials are read after pdl_wait.
  build_partition(wp, p, &s_len_err, kStageRows, n_units);
  pdl_wait();
  const int total = wp.total;
  if (total == 0) return;
  const int P = min(p.n_splits, total);
  constexpr int N4 = GU * D / 4;
  for (int u = blockIdx.x; u < p.batch * n_units; u += gridDim.x) {
    const int b = u / n_units, h = u % n_units;
    if (wp.nch[b] == 0) continue;
    const int ustart = wp.pre[b] + h * wp.nch[b];
    const int uend = ustart + wp.nch[b];
    const int c_first = cta_of(ustart, total, P);
    const int parts = cta_of(uend - 1, total, P) - c_first + 1;
    if (parts == 1) continue;
    const long bh0 = (long)b * p.n_h + (long)h * GU;
    auto slot = [&](int i) {
      return (long)(c_first + i) * 2 + (i == 0 ? 1 : 0);
    };
    auto store = [&](int e, float M, float W, const float4 &acc) {
      const int g = (4 * e) / D;  // head within the unit
      const float iw = W > 0.f ? 1.f / W : 0.f;
      uint2 packed;
      packed.x = pack_bf16x2(acc.x * iw, acc.y * iw);
      packed.y = pack_bf16x2(acc.z * iw, acc.w * iw);
      *reinterpret_cast<uint2 *>(p.out + bh0 * D + 4 * e) = packed;
      if ((4 * e) % D == 0 && p.lse)
        p.lse[bh0 + g] = W > 0.f ? M + logf(W) : -INFINITY;
    };
    float M, W;
    float4 acc;
    if (parts <= 8) {
      // one lane per float4: its loads take one round
      for (int e = threadIdx.x; e < N4; e += kMergeThreads) {
        quad_merge<1>(p.ws_lse, p.ws_o, GU, D, (4 * e) / D, e, parts, slot,
                      M, W, acc);
        store(e, M, W, acc);
      }
    } else {
      // a quad of lanes per float4; the bound is whole warps, so that every
      // lane reaches the quad's shuffles
      for (int e4 = threadIdx.x; e4 < (4 * N4 + 31) / 32 * 32;
           e4 += kMergeThreads) {
        const int e = e4 >> 2;
        const bool active = e < N4;
        quad_merge<4>(p.ws_lse, p.ws_o, GU, D, active ? (4 * e) / D : 0,
                      active ? e : 0, active ? parts : 0, slot, M, W, acc);
        if (active && (e4 & 3) == 0) store(e, M, W, acc);
      }
    }
  }
}

// Queue the merge launch of a dense decode launch that used more than one
// CTA (`n_units` work units per sequence of GU query heads each).
template <int D, int GU>
inline cudaError_t launch_merge_dense(const DecodeParams &p, int n_units,
                                      cudaStream_t s) {
  if (p.n_splits <= 1 || p.whole_units || p.cluster > 1 || p.batch == 0)
    return cudaSuccess;
  const long nu = (long)p.batch * n_units;
  const int grid = (int)(nu < 1024 ? nu : 1024);
  if (p.batch <= kMergeSmallBatch)
    return launch_pdl(merge_dense_kernel<D, GU, kMergeSmallBatch>, dim3(grid),
                      dim3(kMergeThreads), 0, s, 1, p, n_units);
  return launch_pdl(merge_dense_kernel<D, GU, kMaxDecodeBatch>, dim3(grid),
                    dim3(kMergeThreads), 0, s, 1, p, n_units);
}

}  // namespace kvd

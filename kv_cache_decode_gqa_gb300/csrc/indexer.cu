// Indexer scores and top-k selection (the My Weird Prompts 640482
// transcript on DeepSeek Sparse Attention: a lightning indexer scores the
// cached prefix and a top-k subset of positions, k = 2048, is read; "890
// bytes a token ...", section 3: Full and Reindex layers score with their
// own indexer query over a shared indexer key cache).
//
// Scores: s_t = sum_j w_j * max(0, q_j . k_t) for every visible position t,
// with the 64-wide indexer keys read from the paged K-only cache and
// staged in shared memory by bulk copies. Four lanes cover one key row (32
// bytes each); the lane's slice of every indexer query is held in
// registers as fp32 pairs, so the products are formed two at a time
// (packed fp32 fused multiply-adds), each dot product finishes with two
// xor-shuffles, and every sum is formed in fp32.
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
constexpr int kTokPerCta = 512;  // 8 warps x 64 positions

// Packed fp32 pair: two independent fused multiply-adds in one instruction.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b,
                                          uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t pack_f32x2(uint32_t lo, uint32_t hi) {
  return ((uint64_t)hi << 32) | lo;
}
// The two bf16 of a 32-bit word as an fp32 pair (exact).
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
  return pack_f32x2(w << 16, w & 0xffff0000u);
}
__device__ __forceinline__ float sum_f32x2(uint64_t v) {
  return __uint_as_float((uint32_t)v) + __uint_as_float((uint32_t)(v >> 32));
}

// Warp w of a CTA owns the 64 positions t0 + 64 w .. + 63. It stages their
// key rows in shared memory with bulk asynchronous copies (one per paged
// block the slice touches, completing on the warp's own mbarrier), then
// scores them eight rows per step: lane group g = lane / 4 takes row
// 8 i + g, its 4 lanes 16 dims each. Products are summed in fp32 pairs,
// then across the 4 lanes with two xor-shuffles. Several CTAs per SM keep
// enough copies in flight to stream the cache at HBM speed.
constexpr int kSlice = 64;  // positions per warp
template <int H>
__global__ void __launch_bounds__(kScoreThreads, 2)
    indexer_score_kernel(const IndexerParams p) {
  extern __shared__ __align__(128) uint8_t srows[];  // [kTokPerCta][128 B]
  __shared__ uint64_t bars[kScoreThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  int T = p.seq_lens[b];
  T = max(0, min(T, p.max_seq_len));
  // entries: the visible positions, or (pool mode) the pool's positions
  const int32_t *pool = p.pool ? p.pool + (long)b * kPoolBlocks : nullptr;
  const int E = pool ? kPoolBlock * max(0, min(p.pool_n[b], kPoolBlocks)) : T;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tw = blockIdx.x * kTokPerCta + warp * kSlice;  // warp's first
  if (tw >= E) return;
  const int rows = min(kSlice, E - tw);
  uint8_t *mine = srows + warp * kSlice * kIdxDim * 2;
  uint64_t *bar = &bars[warp];
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, rows * kIdxDim * 2);
  }
  __syncwarp();
  // one copy per block piece of the slice; lane j takes pieces j, j + 32..
  const int32_t *bt = p.block_table + (long)b * p.max_blocks;
  const int bs = p.block_size;
  if (pool) {
    // one copy per pool block (8 rows, inside one cache block); a block past
    // the visible length reads block 0 (its scores are set to -inf below)
    if (lane < rows / kPoolBlock) {
      const int pos0 = kPoolBlock * pool[tw / kPoolBlock + lane];
      int blk = 0, slot = 0;
      if (pos0 >= 0 && pos0 < T) {
        blk = bt[pos0 / bs];
        slot = pos0 % bs;
        if (blk < 0 || blk >= p.num_blocks) {
          report(p.err, DEVERR_BLOCK);
          blk = 0;  // read a valid block; the result is flagged as wrong
        }
      } else {
        report(p.err, DEVERR_INDEX);
      }
      bulk_g2s(mine + lane * kPoolBlock * kIdxDim * 2,
               p.cache + ((long)blk * bs + slot) * kIdxDim * 2,
               kPoolBlock * kIdxDim * 2, bar);
    }
  }
  const int lb0 = tw / bs, lb1 = (tw + rows - 1) / bs;
  for (int lb = lb0 + lane; !pool && lb <= lb1; lb += 32) {
    int blk = bt[lb];
    if (blk < 0 || blk >= p.num_blocks) {
      report(p.err, DEVERR_BLOCK);
      blk = 0;  // read a valid block; the result is flagged as wrong
    }
    const int first = max(tw, lb * bs), last = min(tw + rows, (lb + 1) * bs);
    bulk_g2s(mine + (first - tw) * kIdxDim * 2,
             p.cache + ((long)blk * bs + (first - lb * bs)) * kIdxDim * 2,
             (last - first) * kIdxDim * 2, bar);
  }
  // this lane's 16 dims of every indexer query (fp32 pairs), head weights
  const int grp = lane >> 2, sub = lane & 3;
  uint64_t q2[H][8];
  float w[H];
#pragma unroll
  for (int j = 0; j < H; ++j) {
    if (j < p.n_heads) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          p.q + ((long)b * p.n_heads + j) * kIdxDim + sub * 16);
      const uint4 u0 = src[0], u1 = src[1];
      const uint32_t v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) q2[j][e] = bf16x2_to_f32x2(v[e]);
      w[j] = p.w[(long)b * p.n_heads + j];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) q2[j][e] = 0;
      w[j] = 0.f;
    }
  }
  if (!mbar_wait(bar, 0)) {
    // a copy that never lands: flag it, give the copies one more bounded
    // wait, and leave without scoring
    if (lane == 0) report(p.err, DEVERR_TIMEOUT);
    mbar_wait(bar, 0);
    return;
  }
  float *out = p.scores + (long)b * p.score_stride + tw;
#pragma unroll 2
  for (int i = 0; i < kSlice / 8; ++i) {
    const int r = 8 * i + grp;
    const uint4 *src =
        reinterpret_cast<const uint4 *>(mine + r * kIdxDim * 2 + sub * 32);
    const uint4 u0 = src[0], u1 = src[1];
    const uint32_t v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint64_t k2[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) k2[e] = bf16x2_to_f32x2(v[e]);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < H; ++j) {
      uint64_t acc = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = ffma2(q2[j][e], k2[e], acc);
      float d = sum_f32x2(acc);
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      d += __shfl_xor_sync(0xffffffffu, d, 2);
      s = fmaf(w[j], fmaxf(d, 0.f), s);
    }
    if (sub == 0 && r < rows) {
      if (pool) {
        const int pos = kPoolBlock * pool[(tw + r) / kPoolBlock] +
                        (tw + r) % kPoolBlock;
        if (pos < 0 || pos >= T) s = -INFINITY;
      }
      out[r] = s;
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

// Exclusive prefix sum over the 32 warps of the block of a warp-uniform
// value `v` (each warp passes its own); *total = sum over all warps.
__device__ __forceinline__ int warp_excl_scan(int v, int *wsum, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) wsum[warp] = v;
  __syncthreads();
  int x = wsum[lane];
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  const int excl = __shfl_sync(0xffffffffu, x, warp) - v;
  *total = __shfl_sync(0xffffffffu, x, 31);
  __syncthreads();  // wsum may be rewritten by the next call
  return excl;
}

__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
  uint32_t r;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
  return r;
}

constexpr int kCluster = 8;            // CTAs per sequence
constexpr int kCacheKeys = 40 * 1024;  // keys a CTA keeps in shared memory

// One cluster per sequence; CTA r of the cluster owns positions
// [r T / 8, (r + 1) T / 8). When its range fits (T <= 8 * 40960) the CTA
// reads its scores once, converts them to keys in shared memory and runs
// every pass from there; otherwise each pass reads the scores again.
// Histograms are summed across the cluster through distributed shared
// memory in two steps of 16-byte remote loads: CTA r sums the 8 copies of
// its eighth of the bins, then every thread reads the totals of its bins
// from their owners; all CTAs reach the same digits. The compaction places each CTA's selections after those of
// the lower-ranked CTAs.
__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const IndexerParams p) {
  __shared__ __align__(16) int hist[2][kBins];  // double-buffered per pass
  __shared__ __align__(16) int tot[kBins];      // cluster totals, own eighth
  __shared__ int tmp[32];
  __shared__ int s_digit, s_above;
  __shared__ int s_counts[2];  // this CTA's keys above / equal to K*
  extern __shared__ uint32_t s_keys[];
  pdl_trigger();
  pdl_wait();
  const uint32_t rank = cluster_rank();
  const int b = blockIdx.x / kCluster;
  const int tid = threadIdx.x;
  int T = p.seq_lens[b];
  T = max(0, min(T, p.max_seq_len));
  const int k = p.topk;
  const float *sc = p.scores + (long)b * p.score_stride;
  int32_t *out = p.indices + (long)b * k;
  // pool mode: entries are the pool's positions (ascending), selected by
  // entry and written as positions (-1 for one past the visible length,
  // which are the last entries)
  const int32_t *pool = p.pool ? p.pool + (long)b * kPoolBlocks : nullptr;
  const int Tv = T;
  if (pool) T = kPoolBlock * max(0, min(p.pool_n[b], kPoolBlocks));
  auto position = [&](int e) -> int32_t {
    if (!pool) return e;
    const int pos = kPoolBlock * pool[e / kPoolBlock] + e % kPoolBlock;
    return pos >= 0 && pos < Tv ? pos : -1;
  };
  if (T <= k) {  // every position, then -1 padding (uniform per cluster)
    if (rank == 0)
      for (int i = tid; i < k; i += kTopkThreads)
        out[i] = i < T ? position(i) : -1;
    return;
  }
  const int r0 = (int)((long)T * rank / kCluster);
  const int r1 = (int)((long)T * (rank + 1) / kCluster);
  const int n = r1 - r0;
  const bool cached = (uint32_t)n * 4u <= dynamic_smem_bytes();
  if (cached) {
    for (int i = tid; i < n; i += kTopkThreads) s_keys[i] = score_key(sc[r0 + i]);
    __syncthreads();
  }
  auto key_at = [&](int i) {  // i relative to r0, 0 <= i < n
    return cached ? s_keys[i] : score_key(sc[r0 + i]);
  };
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
    constexpr int kU = 16;  // keys per thread per round
    for (int base = 0; base < n; base += kU * kTopkThreads) {
      uint32_t key[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * kTopkThreads + tid;
        key[u] = i < n ? key_at(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * kTopkThreads + tid;
        const bool match =
            i < n && (hi_shift >= 32 || (key[u] >> hi_shift) == prefix);
        // plain shared-memory atomics: lanes of a warp that meet on one
        // bin are serialised by the hardware, which costs less than
        // grouping the lanes by digit when many distinct digits occur
        if (match) atomicAdd(&h[(key[u] >> shift) & (nb - 1)], 1);
      }
    }
    cluster_sync();  // every CTA's histogram of this pass is complete
    // totals of this CTA's eighth of the bins, four bins per thread
    const int own = nb / kCluster;  // bins per owner (512 or 32)
    for (int d = rank * own + 4 * tid; d < (int)(rank + 1) * own;
         d += 4 * kTopkThreads) {
      int4 part[kCluster];
#pragma unroll
      for (int q = 0; q < kCluster; ++q)
        part[q] = *reinterpret_cast<const int4 *>(cluster_ptr(&h[d], q));
      int4 s = make_int4(0, 0, 0, 0);
#pragma unroll
      for (int q = 0; q < kCluster; ++q) {
        s.x += part[q].x;
        s.y += part[q].y;
        s.z += part[q].z;
        s.w += part[q].w;
      }
      *reinterpret_cast<int4 *>(&tot[d]) = s;
    }
    cluster_sync();  // every owner's totals are complete
    // suffix sums over thread ranges of bins (high digits first)
    const int per = (nb + kTopkThreads - 1) / kTopkThreads;  // 4 or 1
    const int r = kTopkThreads - 1 - tid;  // reversed: thread 0 owns the top
    int cnt[4] = {0, 0, 0, 0};
    int local = 0;
    if (r * per < nb) {
      const int d0 = r * per;
      const int *src = cluster_ptr(&tot[d0], (uint32_t)(d0 / own));
      if (per == 4) {
        const int4 v = *reinterpret_cast<const int4 *>(src);
        cnt[0] = v.x, cnt[1] = v.y, cnt[2] = v.z, cnt[3] = v.w;
      } else {
        cnt[0] = *src;
      }
      local = cnt[0] + cnt[1] + cnt[2] + cnt[3];
    }
    int all;
    const int before = block_excl_scan(local, tmp, &all);  // bins above range
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
  int my_gt = 0, my_eq = 0;
  for (int i = tid; i < n; i += kTopkThreads) {
    const uint32_t key = key_at(i);
    my_gt += key > kstar;
    my_eq += key == kstar;
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
    const int g = *cluster_ptr(&s_counts[0], q);
    const int e = *cluster_ptr(&s_counts[1], q);
    run_sel += g + max(0, min(e, need_eq - run_eq));
    run_eq += e;
  }
  // ---- compaction of this CTA's range in position order ----
  // Warp w owns the runs of kRun positions [base + w kRun, + kRun); lane l
  // takes positions run + 32 j + l, so position order within a run is
  // (j, l) and one ballot per j ranks the lanes. A first sweep counts each
  // warp's keys equal to K*, a second decides every selection, a third
  // writes the positions; block scans over the 32 warp totals place the
  // warps after each other.
  constexpr int kRun = 512;  // positions per warp and round
  const int lane = tid & 31, wid = tid >> 5;
  const unsigned lt = (1u << lane) - 1;
  __shared__ int s_wsum[32];
  for (int base = 0; base < n; base += kRun * 32) {
    const int run = base + wid * kRun;
    unsigned gtb[kRun / 32], eqb[kRun / 32];
    int weq = 0;
#pragma unroll
    for (int j = 0; j < kRun / 32; ++j) {
      const int i = run + 32 * j + lane;
      const uint32_t key = i < n ? key_at(i) : 0u;
      gtb[j] = __ballot_sync(0xffffffffu, i < n && key > kstar);
      eqb[j] = __ballot_sync(0xffffffffu, i < n && key == kstar);
      weq += __popc(eqb[j]);
    }
    int tot_eq;
    const int eq_base = run_eq + warp_excl_scan(weq, s_wsum, &tot_eq);
    // selections: every key above K*, and the first need_eq keys equal
    int e = eq_base, wsel = 0;
    unsigned selb[kRun / 32];
#pragma unroll
    for (int j = 0; j < kRun / 32; ++j) {
      const int rank_eq = e + __popc(eqb[j] & lt);
      const bool mine_eq = (eqb[j] >> lane) & 1;
      selb[j] = gtb[j] | __ballot_sync(0xffffffffu, mine_eq && rank_eq < need_eq);
      e += __popc(eqb[j]);
      wsel += __popc(selb[j]);
    }
    int tot_sel;
    int pos = run_sel + warp_excl_scan(wsel, s_wsum, &tot_sel);
#pragma unroll
    for (int j = 0; j < kRun / 32; ++j) {
      const int at = pos + __popc(selb[j] & lt);
      if (((selb[j] >> lane) & 1) && at < k)
        out[at] = position(r0 + run + 32 * j + lane);
      pos += __popc(selb[j]);
    }
    run_eq += tot_eq;
    run_sel += tot_sel;
  }
  cluster_sync();  // no CTA leaves while another may read its shared memory
}

}  // namespace

// ---------------------------------------------------------------------------
// hierarchical indexer pool
// ---------------------------------------------------------------------------
// One CTA per sequence: a bitmap of the 8-position blocks holding the
// selection's visible positions (one bit per block, shared memory), then an
// ordered compaction: thread t counts the set bits of its run of words, a
// block scan places the runs, and each thread writes its block ids in
// ascending order while their rank is below the cap (the lowest blocks
// kept).
constexpr int kPoolThreads = 1024;
constexpr int kPoolSmemMax = 192 * 1024;  // bitmap of up to 50M positions

__global__ void __launch_bounds__(kPoolThreads) pool_kernel(const PoolParams p) {
  extern __shared__ uint32_t bm[];  // (max_seq_len + 255) / 256 words
  __shared__ int s_wsum[32];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  int T = p.seq_lens[b];
  T = max(0, min(T, p.max_seq_len));
  const int words = (T + 255) >> 8;
  for (int i = tid; i < words; i += kPoolThreads) bm[i] = 0u;
  __syncthreads();
  const int32_t *idx = p.indices + (long)b * p.k;
  for (int i = tid; i < p.k; i += kPoolThreads) {
    const int t = idx[i];
    if (t >= T) report(p.err, DEVERR_INDEX);
    if (t >= 0 && t < T) atomicOr(&bm[t >> 8], 1u << ((t >> 3) & 31));
  }
  __syncthreads();
  const int per = (words + kPoolThreads - 1) / kPoolThreads;
  const int w0 = min(tid * per, words), w1 = min(w0 + per, words);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(bm[w]);
  // exclusive scan of cnt over the CTA: within the warp, then the warps
  int x = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  int total;
  const int wexcl =
      warp_excl_scan(__shfl_sync(0xffffffffu, x, 31), s_wsum, &total);
  int rank = wexcl + x - cnt;
  int32_t *pool = p.pool + (long)b * kPoolBlocks;
  for (int w = w0; w < w1 && rank < kPoolBlocks; ++w) {
    uint32_t bits = bm[w];
    while (bits && rank < kPoolBlocks) {
      pool[rank++] = w * 32 + __ffs(bits) - 1;
      bits &= bits - 1;
    }
  }
  if (tid == 0) p.pool_n[b] = min(total, kPoolBlocks);
}

template <int H>
cudaError_t launch_scores_h(const IndexerParams &p, cudaStream_t s) {
  constexpr int kSmem = kTokPerCta * kIdxDim * 2;
  static bool done[64] = {};
  cudaError_t e = set_smem_once(indexer_score_kernel<H>, kSmem, done);
  if (e != cudaSuccess) return e;
  dim3 grid((p.max_entries + kTokPerCta - 1) / kTokPerCta, p.batch);
  return launch_pdl(indexer_score_kernel<H>, grid, dim3(kScoreThreads), kSmem,
                    s, 1, p);
}

cudaError_t launch_indexer_scores(const IndexerParams &p, cudaStream_t s) {
  if (p.batch == 0 || p.max_seq_len == 0 || p.max_entries == 0)
    return cudaSuccess;
  if (p.n_heads <= 1) return launch_scores_h<1>(p, s);
  if (p.n_heads <= 2) return launch_scores_h<2>(p, s);
  if (p.n_heads <= 4) return launch_scores_h<4>(p, s);
  if (p.n_heads <= 8) return launch_scores_h<8>(p, s);
  return cudaErrorNotSupported;
}

cudaError_t launch_topk(const IndexerParams &p, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  static bool done[64] = {};
  cudaError_t e = set_smem_once(topk_kernel, kCacheKeys * 4, done);
  if (e != cudaSuccess) return e;
  // the largest range a CTA owns; cached in shared memory when it fits
  const long range = ((long)p.max_entries + kCluster - 1) / kCluster;
  return launch_pdl(topk_kernel, dim3(p.batch * kCluster), dim3(kTopkThreads),
                    range <= kCacheKeys ? (size_t)range * 4 : 0, s, kCluster,
                    p);
}

cudaError_t launch_indexer_pool(const PoolParams &p, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  const int smem = ((p.max_seq_len + 255) / 256) * 4;
  if (smem > kPoolSmemMax) return cudaErrorNotSupported;
  static bool done[64] = {};
  cudaError_t e = set_smem_once(pool_kernel, kPoolSmemMax, done);
  if (e != cudaSuccess) return e;
  return launch_pdl(pool_kernel, dim3(p.batch), dim3(kPoolThreads),
                    (size_t)smem, s, 1, p);
}

}  // namespace kvd

// Indexer scores and top-k selection (the My Weird Prompts 640482
// transcript on DeepSeek Sparse Attention: a lightning indexer scores the
// cached prefix and a top-k subset of positions, k = 2048, is read; "890
// bytes a token ...", section 3: Full and Reindex layers score with their
// own indexer query over a shared indexer key cache).
//
// Scores: s_t = sum_j w_j * max(0, q_j . k_t) for every visible position t,
// with the 64-wide indexer keys read from the paged K-only cache into shared
// memory by 16-byte asynchronous copies. The dot products are bf16 tensor-
// core products with fp32 accumulation (the bf16 products are exact); the
// ReLU, the weights and the sum over heads are fp32.
//
// Selection: the k largest scores of a sequence, equal scores taken in
// ascending position order, returned as ascending positions (-1 padding
// when fewer than k positions are visible). A cluster of eight CTAs per
// sequence runs an exact radix select on order-preserving 32-bit keys of
// the fp32 scores (negative zero counted as zero): a histogram of the top
// 12 bits summed across the cluster in distributed shared memory finds the
// bin of the k-th largest key; the keys in that bin (the candidates) are
// gathered into every CTA, which finishes the select on them alone (bits
// 19..8, then 7..0) and finds the k-th largest key K* and how many keys
// exceed it. A final pass in position order keeps every key above K* and
// the lowest-indexed keys equal to K*, placing each kept position after the
// selections of the lower-ranked CTAs. The result is exactly the selection
// the scores define.
#include <cmath>

#include "kvd_common.cuh"

namespace kvd {
namespace {

// ---------------------------------------------------------------------------
// scores
// ---------------------------------------------------------------------------
constexpr int kIdxDim = 64;

// A persistent launch over the batch's 64-entry slices: slice s of sequence
// b covers entries 64 s .. 64 s + 63 (the visible positions, or the pool's
// entries). The J slices, sequence-major, are dealt to the G CTAs in
// contiguous runs [c J / G, (c + 1) J / G), so every CTA gets the same
// number whatever the lengths. A CTA walks its run in windows of up to 256
// slices (32 sequences at most), and warp w takes the slices at offsets w,
// w + 8, ... of each window, resolved lane-parallel a window ahead: their
// sequences by a warp scan of the slice counts, their block ids by
// independent loads. A warp streams its slices' key rows into three 8 KB
// slots of its own with 16-byte asynchronous copies, two slices in flight
// while it scores the third (192 KB a CTA); 16-byte chunk c of row r goes
// to chunk c ^ (r mod 8) of the row, so that the matrix loads below meet no
// bank conflicts. (Bulk copies would keep fewer bytes in flight: a thread
// that issues one waits until the copy engine has taken it, about one copy
// latency for 8 KB.)
//
// The dot products q_j . k_t of a slice's 64 rows with the (up to 8)
// indexer queries form one 64 x 64 by 64 x 8 bf16 product with fp32
// accumulation: 16 warp-level tensor-core MMAs (m16n8k16). The ReLU, the
// head weights and the sum over heads run on the accumulators and end in
// two xor-shuffles across the 4 lanes that hold a row.
constexpr int kSlice = 64;                         // entries per slice
constexpr int kSliceBytes = kSlice * kIdxDim * 2;  // 8 KB
constexpr int kScoreWarps = 8;
constexpr int kScoreThreads = 32 * kScoreWarps;
constexpr int kDepth = 3;      // slots a warp
constexpr int kPieceRegs = 8;  // block pieces a lane resolves ahead
constexpr int kScoreSmem = kScoreWarps * kDepth * kSliceBytes;  // 192 KB

// A resolved slice: its sequence and geometry, and the cache rows of its
// first kPieceRegs block pieces (a piece: the rows of the slice in one
// paged block, or one 8-entry pool block).
struct SliceJob {
  int b, tw, rows, T, np;
  uint32_t row[kPieceRegs];  // cache row of piece q's first row
  int pos0[kPieceRegs];      // pool mode: the pool block's first position,
                             // or -1
};

__device__ __forceinline__ int clamp_len(int v, int hi) {
  return max(0, min(v, hi));
}

__global__ void __launch_bounds__(kScoreThreads, 1)
    indexer_score_kernel(const IndexerParams p) {
  // [warp][slot][64 rows][128 B], 16-byte chunks swizzled by row
  extern __shared__ __align__(1024) uint8_t ring[];
  __shared__ SliceJob s_job[kScoreWarps][32];      // the window's slices
  __shared__ uint32_t s_row[kScoreWarps][kSlice];  // cache row of each row
  __shared__ int s_scan[32];
  __shared__ int s_start[3];  // first sequence, its first slice, slices
  pdl_trigger();
  // With stable lengths and block tables (no pool), the plan is made while
  // the kernel before finishes; with a ready prefix, the copies of slices
  // without a sequence's newest row go out then too. Queries, weights, the
  // newest rows and every write wait for it.
  const bool early = (p.flags & FLAG_SEQS_STABLE) && !p.pool;
  const bool prefix = early && (p.flags & FLAG_PREFIX_READY);
  bool waited = !early;
  if (waited) pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.batch, bs = p.block_size;
  const bool pow2 = (bs & (bs - 1)) == 0;
  const int bs_shift = __ffs(bs) - 1;
  auto div_bs = [&](int t) { return pow2 ? t >> bs_shift : t / bs; };
  auto entries = [&](int b, int T) {
    return p.pool ? kPoolBlock * clamp_len(p.pool_n[b], kPoolBlocks) : T;
  };
  // ---- this CTA's run of slices: thread t counts the slices of its
  // contiguous chunk of sequences, a block scan places the chunks ----
  {
    const int per = (B + kScoreThreads - 1) / kScoreThreads;
    const int c0 = min(B, tid * per), c1 = min(B, c0 + per);
    int mine = 0;
    for (int b = c0; b < c1; ++b) {
      const int T = clamp_len(p.seq_lens[b], p.max_seq_len);
      mine += (entries(b, T) + kSlice - 1) / kSlice;
    }
    int x = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_scan[warp] = x;
    __syncthreads();
    int before = 0, J = 0;
    for (int w = 0; w < kScoreWarps; ++w) {
      const int v = s_scan[w];
      before += w < warp ? v : 0;
      J += v;
    }
    const int excl = before + x - mine;
    const long j0 = (long)blockIdx.x * J / gridDim.x;
    const long j1 = (long)(blockIdx.x + 1) * J / gridDim.x;
    if (tid == 0) s_start[2] = (int)(j1 - j0);
    if (j0 < j1 && excl <= j0 && j0 < excl + mine) {
      int acc = excl;
      for (int b = c0; b < c1; ++b) {
        const int T = clamp_len(p.seq_lens[b], p.max_seq_len);
        const int n = (entries(b, T) + kSlice - 1) / kSlice;
        if (j0 < acc + n) {
          s_start[0] = b;
          s_start[1] = (int)(j0 - acc);
          break;
        }
        acc += n;
      }
    }
    __syncthreads();
  }
  const int nj = s_start[2];
  if (nj == 0) return;

  int cb = s_start[0], cs = s_start[1];  // next slice to resolve
  int k0 = 0;                            // its index in the CTA's run
  const int g = lane >> 2, t4 = lane & 3;
  // B fragments (head g, dims 16 kt + 2 t4 and + 8) and the weights of
  // heads 2 t4, 2 t4 + 1 of the sequence qb; the next sequence's are loaded
  // when its first slice's copies go out
  uint32_t qf[4][2], qn[4][2];
  float w0 = 0.f, w1 = 0.f, wn0 = 0.f, wn1 = 0.f;
  int qb = -1, qbn = -1;
  auto load_query = [&](int b, uint32_t (&f)[4][2], float &x0, float &x1) {
    const uint32_t *q32 = reinterpret_cast<const uint32_t *>(
        p.q + ((long)b * p.n_heads + min(g, p.n_heads - 1)) * kIdxDim);
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      f[kt][0] = g < p.n_heads ? q32[8 * kt + t4] : 0u;
      f[kt][1] = g < p.n_heads ? q32[8 * kt + 4 + t4] : 0u;
    }
    const float *wb = p.w + (long)b * p.n_heads;
    x0 = 2 * t4 < p.n_heads ? wb[2 * t4] : 0.f;
    x1 = 2 * t4 + 1 < p.n_heads ? wb[2 * t4 + 1] : 0.f;
  };
  const bool two_lanes = p.n_heads <= 4;  // heads on lanes t4 = 0, 1 only
  uint8_t *wring = ring + warp * kDepth * kSliceBytes;
  for (;;) {
    // ---- resolve the next window of up to 256 slices of the run (the same
    // windows in every warp); lane m takes slice 8 m + warp of it ----
    if (k0 >= nj || cb >= B) break;
    const int bl = cb + lane;
    int Tl = 0, nl = 0;
    if (bl < B) {
      Tl = clamp_len(p.seq_lens[bl], p.max_seq_len);
      nl = (entries(bl, Tl) + kSlice - 1) / kSlice;
    }
    int inc = max(0, nl - (lane == 0 ? cs : 0));
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    const int total = __shfl_sync(0xffffffffu, inc, 31);
    if (total == 0) {  // 32 sequences without slices left
      cb += 32;
      cs = 0;
      continue;
    }
    const int win = min(32 * kScoreWarps, min(total, nj - k0));
    const int idx = kScoreWarps * lane + warp;  // this lane's slice
    // the sequence (relative to cb) of this lane's slice: the first lane l
    // with inc_l > idx (inc is non-decreasing), by binary search
    int j = 0;
#pragma unroll
    for (int step = 16; step > 0; step >>= 1)
      if (__shfl_sync(0xffffffffu, inc, j + step - 1) <= idx) j += step;
    if (__shfl_sync(0xffffffffu, inc, j) <= idx) ++j;  // idx >= inc_31: 32
    const int jj = min(j, 31);
    const int before = __shfl_sync(0xffffffffu, inc, max(jj - 1, 0));
    const int sl = (jj == 0 ? cs + idx : idx - before);
    const int bc = min(cb + jj, B - 1);
    SliceJob job;
    job.b = bc;
    job.T = __shfl_sync(0xffffffffu, Tl, jj);
    const int E = p.pool ? kPoolBlock * clamp_len(p.pool_n[bc], kPoolBlocks)
                         : job.T;
    job.tw = sl * kSlice;
    job.rows = idx < win ? max(0, min(kSlice, E - job.tw)) : 0;
    // the next window starts after this one's last slice
    const int jl = __popc(__ballot_sync(0xffffffffu, inc <= win - 1));
    const int jl_before = __shfl_sync(0xffffffffu, inc, max(jl - 1, 0));
    cs = (jl == 0 ? cs + win : win - jl_before);
    cb += jl;
    k0 += win;
    // block ids of the first kPieceRegs pieces (independent loads), then
    // checked and turned into cache rows
    const int32_t *bt = p.block_table + (long)bc * p.max_blocks;
    int blk[kPieceRegs];
    if (p.pool) {
      job.np = job.rows / kPoolBlock;
      const int32_t *pool = p.pool + (long)bc * kPoolBlocks;
#pragma unroll
      for (int q = 0; q < kPieceRegs; ++q)
        job.pos0[q] =
            q < job.np ? kPoolBlock * pool[job.tw / kPoolBlock + q] : -1;
#pragma unroll
      for (int q = 0; q < kPieceRegs; ++q) {
        const int pos = job.pos0[q];
        blk[q] = (q < job.np && pos >= 0 && pos < job.T) ? bt[div_bs(pos)] : 0;
      }
    } else {
      job.np = job.rows > 0
                   ? div_bs(job.tw + job.rows - 1) - div_bs(job.tw) + 1 : 0;
      const int lb0 = div_bs(job.tw);
#pragma unroll
      for (int q = 0; q < kPieceRegs; ++q) {
        blk[q] = q < job.np ? bt[lb0 + q] : 0;
        job.pos0[q] = -1;
      }
    }
#pragma unroll
    for (int q = 0; q < kPieceRegs; ++q) {
      int bq = blk[q], slot = 0;
      if (q >= job.np) {
        job.row[q] = 0;
        continue;
      }
      if (p.pool) {
        const int pos = job.pos0[q];
        if (pos >= 0 && pos < job.T) {
          slot = pos - div_bs(pos) * bs;
        } else {
          report(p.err, DEVERR_INDEX);
          bq = 0;
          job.pos0[q] = -1;
        }
      } else {
        const int lb = div_bs(job.tw) + q;
        slot = max(job.tw, lb * bs) - lb * bs;
      }
      if (bq < 0 || bq >= p.num_blocks) {
        report(p.err, DEVERR_BLOCK);
        bq = 0;  // read a valid block; the result is flagged as wrong
      }
      job.row[q] = (uint32_t)bq * (uint32_t)bs + (uint32_t)slot;
    }
    __syncwarp();  // the previous window's table has been read
    s_job[warp][lane] = job;
    __syncwarp();
    const int bn = win > warp ? (win - warp + kScoreWarps - 1) / kScoreWarps : 0;

    // ---- this warp's slices of the window: three slots, the copies of
    // slice m + 3 go out into slice m's slot as soon as its MMAs have
    // read it (three slices in flight during the epilogue) ----
    const int col = lane & 7;
    for (int m = -3; m < bn; ++m) {
      float c[4][4];
      int rows = 0, T = 0;
      float *out = nullptr;
      const SliceJob *Jp = nullptr;
      if (m >= 0) {
        if (!waited) {
          pdl_wait();
          waited = true;
        }
        cp_async_wait<2>();  // slice m has landed (this lane's copies)
        __syncwarp();        // ... and every lane's
        Jp = &s_job[warp][m];
        const int b = Jp->b, tw = Jp->tw;
        rows = Jp->rows;
        T = Jp->T;
        if (b != qb) {
          if (b == qbn) {
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
              qf[kt][0] = qn[kt][0];
              qf[kt][1] = qn[kt][1];
            }
            w0 = wn0;
            w1 = wn1;
          } else {  // a sequence of fewer than three slices came between
            load_query(b, qf, w0, w1);
          }
          qb = b;
        }
        const uint32_t sbase = smem_u32(wring + (m % kDepth) * kSliceBytes);
        out = p.scores + (long)b * p.score_stride + tw;
        // the matrix loads of k-step kt + 1 go out before the MMAs of step
        // kt, which are independent across the four row tiles
        uint32_t a[2][4][4];
#pragma unroll
        for (int rt = 0; rt < 4; ++rt) {
          c[rt][0] = c[rt][1] = c[rt][2] = c[rt][3] = 0.f;
        }
        auto load_a = [&](int kt, uint32_t (&dst)[4][4]) {
#pragma unroll
          for (int rt = 0; rt < 4; ++rt) {
            const int lr = 16 * rt + (lane & 15);  // this lane's ldmatrix row
            const int chunk = 2 * kt + (lane >> 4);
            ldsm_x4(dst[rt], sbase + lr * 128 + ((chunk ^ (lr & 7)) << 4));
          }
        };
        load_a(0, a[0]);
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          if (kt < 3) load_a(kt + 1, a[(kt + 1) & 1]);
#pragma unroll
          for (int rt = 0; rt < 4; ++rt)
            mma_bf16(c[rt], a[kt & 1][rt], qf[kt][0], qf[kt][1]);
        }
        __syncwarp();  // every lane has read the slot before it is refilled
      }
      const int mi = m + 3;  // the slice whose copies go out now
      if (mi < bn) {
        const SliceJob &J = s_job[warp][mi];
        const int irows = J.rows, np = J.np;
        uint8_t *dst = wring + (mi % kDepth) * kSliceBytes;
        if (!waited && !(prefix && J.tw + irows < J.T)) {
          pdl_wait();
          waited = true;
        }
        if (waited && J.b != qbn && J.b != qb) {  // its query travels with it
          qbn = J.b;
          load_query(qbn, qn, wn0, wn1);
        }
        if (p.pool) {
          // rows 8 q .. 8 q + 7 are pool block q: row r of chunk j is in
          // block j / 2
#pragma unroll
          for (int jc = 0; jc < kSlice / 4; ++jc) {
            const int r = (lane >> 3) + 4 * jc;
            if (r < irows)
              cp_async16(dst + r * 128 + ((col ^ (r & 7)) << 4),
                         p.cache + ((size_t)J.row[jc >> 1] + (r & 7)) * 128 +
                             col * 16, 16);
          }
        } else if (np == 1) {  // one block piece: consecutive cache rows
          const size_t r0 = J.row[0];
#pragma unroll
          for (int jc = 0; jc < kSlice / 4; ++jc) {
            const int r = (lane >> 3) + 4 * jc;
            if (r < irows)
              cp_async16(dst + r * 128 + ((col ^ (r & 7)) << 4),
                         p.cache + (r0 + r) * 128 + col * 16, 16);
          }
        } else {
          // several pieces: the cache row of each row first
          const int tw = J.tw, lb0 = div_bs(tw);
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            const int r = lane + 32 * h;
            const int t = tw + r;
            const int q = div_bs(t) - lb0;
            const int first = max(tw, (lb0 + q) * bs);
            uint32_t pr = 0;
            if (r < irows) {
              if (q < kPieceRegs) {
                pr = J.row[q];
              } else {  // pieces past the resolved ones
                int bq = p.block_table[(long)J.b * p.max_blocks + lb0 + q];
                if (bq < 0 || bq >= p.num_blocks) {
                  report(p.err, DEVERR_BLOCK);
                  bq = 0;
                }
                pr = (uint32_t)bq * (uint32_t)bs +
                     (uint32_t)(first - (lb0 + q) * bs);
              }
            }
            s_row[warp][r] = pr + (uint32_t)(t - first);
          }
          __syncwarp();
#pragma unroll 4
          for (int jc = 0; jc < kSlice / 4; ++jc) {
            const int r = (lane >> 3) + 4 * jc;
            if (r < irows)
              cp_async16(dst + r * 128 + ((col ^ (r & 7)) << 4),
                         p.cache + (size_t)s_row[warp][r] * 128 + col * 16,
                         16);
          }
          __syncwarp();  // s_row is rewritten by the next slice
        }
      }
      cp_async_commit();  // one group a step (empty past the last slice)
      if (m < 0) continue;
      // rows 16 rt + g (s[rt][0]) and 16 rt + g + 8 (s[rt][1]): heads 2 t4
      // and 2 t4 + 1 here, summed over the lanes t4
      float sv[4][2];
#pragma unroll
      for (int rt = 0; rt < 4; ++rt) {
        sv[rt][0] = fmaf(w1, fmaxf(c[rt][1], 0.f), w0 * fmaxf(c[rt][0], 0.f));
        sv[rt][1] = fmaf(w1, fmaxf(c[rt][3], 0.f), w0 * fmaxf(c[rt][2], 0.f));
      }
#pragma unroll
      for (int rt = 0; rt < 4; ++rt) {
        sv[rt][0] += __shfl_xor_sync(0xffffffffu, sv[rt][0], 1);
        sv[rt][1] += __shfl_xor_sync(0xffffffffu, sv[rt][1], 1);
      }
      if (!two_lanes) {
#pragma unroll
        for (int rt = 0; rt < 4; ++rt) {
          sv[rt][0] += __shfl_xor_sync(0xffffffffu, sv[rt][0], 2);
          sv[rt][1] += __shfl_xor_sync(0xffffffffu, sv[rt][1], 2);
        }
      }
      if (t4 == 0) {
#pragma unroll
        for (int rt = 0; rt < 4; ++rt) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r = 16 * rt + g + 8 * hh;
            float sc = sv[rt][hh];
            if (r < rows) {
              if (p.pool) {  // a position past the visible length: -inf
                const int pos0 = Jp->pos0[r / kPoolBlock];
                if (pos0 < 0 || pos0 + r % kPoolBlock >= T) sc = -INFINITY;
              }
              out[r] = sc;
            }
          }
        }
      }
    }
  }
  cp_async_wait<0>();
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
constexpr int kCacheKeys = 20 * 1024;  // keys a CTA keeps in shared memory
constexpr int kHiCap = 4096;           // high keys a CTA lists
constexpr int kGatherCap = 12288;      // high keys of the whole cluster

// The digit (high digits first) whose bin holds the remaining-th largest
// key, and the count of keys in the bins above it, into *s_digit and
// *s_above. Thread t holds the bins of range 1023 - t (4 bins of 4096, or 1
// of 256), read by load(first bin, bins, counts); a block scan over the
// ranges finds the one that holds it.
template <class Load>
__device__ __forceinline__ void find_digit(int nb, int remaining, Load load,
                                           int *tmp, int *s_digit,
                                           int *s_above) {
  const int per = (nb + kTopkThreads - 1) / kTopkThreads;  // 4 or 1
  const int r = kTopkThreads - 1 - threadIdx.x;  // thread 0 owns the top
  int cnt[4] = {0, 0, 0, 0};
  int local = 0;
  if (r * per < nb) {
    load(r * per, per, cnt);
    local = cnt[0] + cnt[1] + cnt[2] + cnt[3];
  }
  int all;
  const int before = block_excl_scan(local, tmp, &all);  // bins above range
  if (before < remaining && before + local >= remaining) {
    int acc = before;
    for (int j = per - 1; j >= 0; --j) {
      if (acc + cnt[j] >= remaining) {
        *s_digit = r * per + j;
        *s_above = acc;
        break;
      }
      acc += cnt[j];
    }
  }
  __syncthreads();
}

// One cluster per sequence; CTA r of the cluster owns positions
// [r T / 8, (r + 1) T / 8). When its range fits (T <= 8 * 20480) the CTA
// reads its scores once, converts them to keys in shared memory and works
// from there; otherwise each sweep reads the scores again.
//  1. The histogram of the first digit (key bits 31..20) is summed across
//     the cluster through distributed shared memory in two steps of
//     16-byte remote loads (CTA r sums the 8 copies of its eighth of the
//     bins, then every thread reads the totals of its bins from their
//     owners), giving every CTA the digit d1 of the k-th largest key.
//  2. Each CTA lists its high keys (first digit >= d1: every selection is
//     one of them), with their positions, in position order: about k / 8
//     plus a share of d1's bin. Every CTA copies the cluster's high keys
//     into its own shared memory and finishes the select on those in d1's
//     bin alone: two local passes on bits 19..8 and 7..0 give the k-th
//     largest key K* and how many keys equal to K* to take; the high keys
//     of each source CTA above / equal to K* place every CTA's selections
//     after those of the lower-ranked CTAs, and a pass over its own list
//     writes them.
//  3. If the high keys do not fit (4,096 a CTA, 12,288 a cluster: a large
//     k, or many equal or near-equal scores), the cluster instead runs the
//     second and third digits as cluster-wide passes over every key, as in
//     step 1, and a sweep over every key in position order writes the
//     selections.
__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const IndexerParams p) {
  __shared__ __align__(16) int hist[2][kBins];
  __shared__ __align__(16) int tot[kBins];  // cluster totals, own eighth
  __shared__ int tmp[32];
  __shared__ int s_digit, s_above;
  __shared__ uint32_t s_kstar;         // K* when its last bin holds one key
  __shared__ int s_nhi;                // this CTA's high keys
  __shared__ int s_off[kCluster + 1];  // high keys of the lower ranks
  __shared__ int s_src[2][kCluster];   // high keys above / equal to K*
  __shared__ int s_run[3];  // lower ranks' selections and K*s, own K*s
  __shared__ int s_counts[2];  // this CTA's keys above / equal to K*
  __shared__ int s_wsum[32];
  // [kHiCap] high keys, [kHiCap] their indices, [kGatherCap] the
  // cluster's high keys, [n] keys
  extern __shared__ uint32_t dsm[];
  uint32_t *s_hik = dsm;
  int *s_hii = reinterpret_cast<int *>(dsm + kHiCap);
  uint32_t *s_gath = dsm + 2 * kHiCap;
  uint32_t *s_keys = dsm + 2 * kHiCap + kGatherCap;
  pdl_trigger();
  pdl_wait();
  const uint32_t rank = cluster_rank();
  const int b = blockIdx.x / kCluster;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const unsigned lt = (1u << lane) - 1;
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
  const bool cached = (uint32_t)(2 * kHiCap + kGatherCap + n) * 4u <=
                      dynamic_smem_bytes();
  auto key_at = [&](int i) {  // i relative to r0, 0 <= i < n
    return cached ? s_keys[i] : score_key(sc[r0 + i]);
  };
  for (int i = tid; i < kBins; i += kTopkThreads) hist[0][i] = 0;
  if (tid < 2 * kCluster) s_src[tid / kCluster][tid % kCluster] = 0;
  __syncthreads();
  // ---- 1. keys, and the cluster's histogram of the first digit ----
  {
    constexpr int kU = 8;  // independent loads a thread keeps in flight
    for (int base = 0; base < n; base += kU * kTopkThreads) {
      float v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * kTopkThreads + tid;
        v[u] = i < n ? sc[r0 + i] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * kTopkThreads + tid;
        if (i < n) {
          const uint32_t key = score_key(v[u]);
          if (cached) s_keys[i] = key;
          // plain shared-memory atomics: lanes of a warp that meet on one
          // bin are serialised by the hardware, which costs less than
          // grouping the lanes by digit when many distinct digits occur
          atomicAdd(&hist[0][key >> 20], 1);
        }
      }
    }
  }
  // Sum of the cluster's histograms `h` (nb bins) into the totals of this
  // CTA's eighth, then the digit search over the totals of their owners.
  auto cluster_digit = [&](const int *h, int nb, int remaining) {
    cluster_sync();  // every CTA's histogram of this pass is complete
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
    find_digit(nb, remaining,
               [&](int d0, int per, int (&cnt)[4]) {
                 const int *src = cluster_ptr(&tot[d0], (uint32_t)(d0 / own));
                 if (per == 4) {
                   const int4 v = *reinterpret_cast<const int4 *>(src);
                   cnt[0] = v.x, cnt[1] = v.y, cnt[2] = v.z, cnt[3] = v.w;
                 } else {
                   cnt[0] = *src;
                 }
               },
               tmp, &s_digit, &s_above);
  };
  cluster_digit(hist[0], kBins, k);
  const uint32_t d1 = (uint32_t)s_digit;
  int remaining = k - s_above;  // keys still to take at or below d1's bin
  // ---- 2. this CTA's high keys in position order ----
  // Warp w owns the runs of kRun positions [base + w kRun, + kRun); lane l
  // takes positions run + 32 j + l, so position order within a run is
  // (j, l) and one ballot per j ranks the lanes; a scan over the 32 warp
  // totals places the warps after each other. The list's runs are long
  // enough that a cached range takes one round.
  constexpr int kRun = 512;  // positions per warp and round (final sweep)
  constexpr int kHiRun = kCacheKeys / kTopkThreads * 32;  // list: 640
  {
    int nhi = 0;  // high keys of the earlier rounds
    for (int base = 0; base < n; base += kHiRun * 32) {
      const int run = base + wid * kHiRun;
      uint32_t key[kHiRun / 32];
      unsigned hib[kHiRun / 32];
      int whi = 0;
#pragma unroll
      for (int j = 0; j < kHiRun / 32; ++j) {
        const int i = run + 32 * j + lane;
        key[j] = i < n ? key_at(i) : 0u;
        hib[j] = __ballot_sync(0xffffffffu, i < n && (key[j] >> 20) >= d1);
        whi += __popc(hib[j]);
      }
      int tot_hi;
      int at = nhi + warp_excl_scan(whi, s_wsum, &tot_hi);
#pragma unroll
      for (int j = 0; j < kHiRun / 32; ++j) {
        if (hib[j] == 0u) continue;  // most groups hold no high key
        const int idx = at + __popc(hib[j] & lt);
        if (((hib[j] >> lane) & 1) && idx < kHiCap) {
          s_hik[idx] = key[j];
          s_hii[idx] = run + 32 * j + lane;
        }
        at += __popc(hib[j]);
      }
      nhi += tot_hi;
    }
    if (tid == 0) s_nhi = nhi;
  }
  cluster_sync();  // every CTA's high keys are listed
  if (wid == 0) {
    int c = lane < kCluster ? *cluster_ptr(&s_nhi, (uint32_t)lane) : 0;
    const bool over = __any_sync(0xffffffffu, c > kHiCap);
    int inc = c;
#pragma unroll
    for (int o = 1; o < kCluster; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 0) s_off[0] = 0;
    if (lane < kCluster) s_off[lane + 1] = over ? kGatherCap + 1 : inc;
  }
  __syncthreads();
  const int C = s_off[kCluster];
  const bool fits = C <= kGatherCap;  // the same decision in every CTA
  const int nhi = s_nhi;
  auto source = [&](int i) {  // the CTA gathered key i came from
    int q = 0;
#pragma unroll
    for (int j = 1; j < kCluster; ++j) q += i >= s_off[j];
    return q;
  };
  uint32_t kstar;
  int need_eq, run_sel, run_eq;
  if (fits) {
    for (int i = tid; i < C; i += kTopkThreads) {
      const int q = source(i);
      s_gath[i] = *cluster_ptr(&s_hik[i - s_off[q]], (uint32_t)q);
    }
    // done with the other CTAs' shared memory; the matching wait comes
    // before this CTA leaves
    cluster_arrive();
    for (int i = tid; i < kBins; i += kTopkThreads) hist[1][i] = 0;
    __syncthreads();
    for (int i = tid; i < C; i += kTopkThreads) {
      const uint32_t key = s_gath[i];
      if ((key >> 20) == d1) atomicAdd(&hist[1][(key >> 8) & 0xfff], 1);
    }
    __syncthreads();
    find_digit(kBins, remaining,
               [&](int d0, int, int (&cnt)[4]) {
                 const int4 v = *reinterpret_cast<const int4 *>(&hist[1][d0]);
                 cnt[0] = v.x, cnt[1] = v.y, cnt[2] = v.z, cnt[3] = v.w;
               },
               tmp, &s_digit, &s_above);
    const uint32_t p2 = (d1 << 12) | (uint32_t)s_digit;  // bits 31..8
    remaining -= s_above;
    if (hist[1][s_digit] == 1) {
      // the usual case for spread scores: the bin holds one key, K*
      for (int i = tid; i < C; i += kTopkThreads) {
        const uint32_t key = s_gath[i];
        if ((key >> 8) == p2) s_kstar = key;
      }
      __syncthreads();
      kstar = s_kstar;
      need_eq = 1;
    } else {
      for (int i = tid; i < 256; i += kTopkThreads) hist[0][i] = 0;
      __syncthreads();
      for (int i = tid; i < C; i += kTopkThreads) {
        const uint32_t key = s_gath[i];
        if ((key >> 8) == p2) atomicAdd(&hist[0][key & 0xff], 1);
      }
      __syncthreads();
      find_digit(256, remaining,
                 [&](int d0, int, int (&cnt)[4]) { cnt[0] = hist[0][d0]; },
                 tmp, &s_digit, &s_above);
      kstar = (p2 << 8) | (uint32_t)s_digit;
      need_eq = remaining - s_above;
    }
    // keys above / equal to K* of each source CTA: warp q counts the
    // gathered list of CTA q (a contiguous segment)
    if (wid < kCluster) {
      int gt = 0, eq = 0;
      for (int i = s_off[wid] + lane; i < s_off[wid + 1]; i += 32) {
        const uint32_t key = s_gath[i];
        gt += key > kstar;
        eq += key == kstar;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        gt += __shfl_xor_sync(0xffffffffu, gt, o);
        eq += __shfl_xor_sync(0xffffffffu, eq, o);
      }
      if (lane == 0) {
        s_src[0][wid] = gt;
        s_src[1][wid] = eq;
      }
    }
    __syncthreads();
    if (tid == 0) {
      int sel = 0, eq = 0;
      for (uint32_t q = 0; q < rank; ++q) {
        const int e = s_src[1][q];
        sel += s_src[0][q] + max(0, min(e, need_eq - eq));
        eq += e;
      }
      s_run[0] = sel;
      s_run[1] = eq;
    }
    __syncthreads();
    run_sel = s_run[0];
    run_eq = s_run[1];
    // ---- the selections: this CTA's high keys in position order ----
    for (int base = 0; base < nhi; base += kTopkThreads) {
      const int e = base + tid;
      const uint32_t key = e < nhi ? s_hik[e] : 0u;
      const bool eq = e < nhi && key == kstar;
      const unsigned eqb = __ballot_sync(0xffffffffu, eq);
      int tot_eq;
      const int rank_eq = run_eq +
                          warp_excl_scan(__popc(eqb), s_wsum, &tot_eq) +
                          __popc(eqb & lt);
      const bool sel = (e < nhi && key > kstar) || (eq && rank_eq < need_eq);
      const unsigned selb = __ballot_sync(0xffffffffu, sel);
      int tot_sel;
      const int at = run_sel + warp_excl_scan(__popc(selb), s_wsum, &tot_sel) +
                     __popc(selb & lt);
      if (sel && at < k) out[at] = position(r0 + s_hii[e]);
      run_eq += tot_eq;
      run_sel += tot_sel;
    }
    cluster_wait();  // no CTA leaves while another may read its list
    return;
  }
  // ---- 3. cluster-wide passes on bits 19..8 and 7..0 ----
  {
    uint32_t prefix = d1;
    const int shifts[2] = {8, 0};
    const int widths[2] = {12, 8};
    for (int pass = 0; pass < 2; ++pass) {
      int *h = hist[(pass + 1) & 1];
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
          if (i < n && (key[u] >> hi_shift) == prefix)
            atomicAdd(&h[(key[u] >> shift) & (nb - 1)], 1);
        }
      }
      cluster_digit(h, nb, remaining);
      prefix = (prefix << bits) | (uint32_t)s_digit;
      remaining -= s_above;
      __syncthreads();
    }
    kstar = prefix;
    need_eq = remaining;
  }
  // counts of this CTA's keys above / equal to K*, placed by rank
  {
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
    if (tid < kCluster) {
      s_src[0][tid] = *cluster_ptr(&s_counts[0], (uint32_t)tid);
      s_src[1][tid] = *cluster_ptr(&s_counts[1], (uint32_t)tid);
    }
    __syncthreads();
    run_sel = run_eq = 0;
    for (uint32_t q = 0; q < rank; ++q) {
      const int e = s_src[1][q];
      run_sel += s_src[0][q] + max(0, min(e, need_eq - run_eq));
      run_eq += e;
    }
  }
  // the selections: a sweep over every key in position order. A first
  // sweep counts each warp's keys equal to K*, a second decides every
  // selection, a third writes the positions.
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
  cluster_sync();  // no CTA leaves while another may read its counts
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

cudaError_t launch_indexer_scores(const IndexerParams &p, cudaStream_t s) {
  if (p.batch == 0 || p.max_seq_len == 0 || p.max_entries == 0)
    return cudaSuccess;
  if (p.n_heads < 1 || p.n_heads > 8) return cudaErrorNotSupported;
  static bool done[64] = {};
  cudaError_t e = set_smem_once(indexer_score_kernel, kScoreSmem, done);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // at most one CTA per slice of the longest sequence's entries
  const long slices =
      (long)p.batch * ((p.max_entries + kSlice - 1) / kSlice);
  const int grid = (int)(slices < sms ? slices : sms);
  return launch_pdl(indexer_score_kernel, dim3(grid), dim3(kScoreThreads),
                    kScoreSmem, s, 1, p);
}

cudaError_t launch_topk(const IndexerParams &p, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  constexpr int kCandBytes = (2 * kHiCap + kGatherCap) * 4;
  static bool done[64] = {};
  cudaError_t e =
      set_smem_once(topk_kernel, kCandBytes + kCacheKeys * 4, done);
  if (e != cudaSuccess) return e;
  // the largest range a CTA owns; its keys cached in shared memory when
  // they fit
  const long range = ((long)p.max_entries + kCluster - 1) / kCluster;
  const size_t smem =
      kCandBytes + (range <= kCacheKeys ? (size_t)range * 4 : 0);
  return launch_pdl(topk_kernel, dim3(p.batch * kCluster), dim3(kTopkThreads),
                    smem, s, kCluster, p);
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

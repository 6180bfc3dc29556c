// Top-k sparse decode on the 5th-generation tensor cores ("890 bytes a
// token ...", section 3: a Reuse layer attends to the selection an earlier
// layer made; the My Weird Prompts 640482 transcript on DeepSeek Sparse
// Attention: only the top-k positions of the cache are read). Each
// sequence's query heads (n_kv = 1) attend to the k cached rows an index
// list names; K and V rows are 512 wide and stored apart.
//
// The scores are computed transposed, S^T = K Q^T: the gathered positions
// are the MMA's M (128 per chunk, the shape whose tensor-memory layout is
// one row per lane) and a tile of 64 query heads its N, so no M row is
// padding. The output is transposed too, O^T = V^T P^T: 4 MMAs of M = 128
// value columns and N = 64 heads per 16 positions, accumulated in tensor
// memory (4 x 64 columns). Each gathered byte is copied into shared memory
// once and read by one MMA; the query tile is a 64 KB B operand loaded once.
//
// Rows are gathered with 16-byte cp.async pieces, placed in the MMA's
// 128-byte-swizzled layout by the address each piece is given (a row that
// is not attended -- an entry out of the CTA's share, a negative entry, one
// at or past the length, a bad block id -- is filled with zeros). Measured
// on this GPU: TMA tile::gather4 (four 128-byte rows per instruction)
// delivered about 13 GB/s per SM for these random rows, the cp.async
// pieces about twice that with two slices in flight per CTA and more with
// four; a bulk copy per row lands unswizzled, which the MMA cannot read.
//
// Work: a unit is (sequence, 64-head tile) with k index entries, split
// over S CTAs (one wave: S = SMs / units, at most 32, none with fewer than
// 32 entries), each taking an equal share of the entries in chunks of 128.
// With S = 1 a CTA writes the unit's outputs. Otherwise each writes its
// normalised partial outputs (64 heads x 512 values, fp32: one value per
// tensor-memory lane, so each store of a warp covers 32 consecutive values)
// and their log-sum-exps to the workspace, and a short second launch merges
// the S parts of every output (log-sum-exp merge). (A merge of four CTAs in
// distributed shared memory, tried first, took longer than the copies: its
// remote loads were latency-bound with the kernel's 192 threads.)
//
// Warp roles (192 threads; at most two warps per SM sub-partition, so a
// thread may hold up to 255 registers):
//   warp 0: the query tile, by tiled TMA (eight 64 x 64 boxes).
//   warp 1: tensor memory; the MMA loop (one elected lane issues): S^T of a
//     chunk as 32 k-steps (A = K slice, K-major; B = the query tile,
//     K-major), then O^T += V^T P^T as 4 value blocks x 8 k-steps (A = V
//     slice, MN-major; B = P, MN-major).
//   warps 2-5: workers. Per chunk each thread resolves one row (index
//     entry -> position -> block table -> cache row); worker w copies K
//     slice w (dims 128 w ..) into ring slot w, and V slice w (values
//     128 w ..) into the same slot once the scores have read it, so four
//     32 KB slices are in flight per CTA. Then the softmax, one thread per
//     position (tensor-memory lane): a thread reads its position's 64
//     scores; per-head maxima and sums over
//     the chunk's 128 positions are reduce-scatters across the warp (62
//     shuffles for 64 heads) and four warps in shared memory. Each thread
//     writes its position's row of P (bf16) into the swizzled P tile, and
//     rescales the tensor-memory O^T columns of heads whose maximum grew.
#include <cmath>

#include "kvd_common.cuh"
#include "stream_k.cuh"
#include "tcgen05.cuh"
#include "tmap.h"

namespace kvd {
namespace {

constexpr int kH = 64;            // query heads per unit (MMA N)
constexpr int kD = 512;           // key and value width
constexpr int kRows = 128;        // positions per chunk (MMA M of S^T)
constexpr int kSliceCols = 128;   // dims (K) or values (V) per ring slice
constexpr int kSlicesPerChunk = 2 * kD / kSliceCols;  // 8: 4 of K, 4 of V
constexpr int kCBBytes = kRows * 128;                 // a 64-column block
constexpr int kSlotBytes = kRows * kSliceCols * 2;    // 32 KB
constexpr int kNSlot = 4;
constexpr int kQCB = kH * 128;                        // Q: one column block
constexpr int kQBytes = kH * kD * 2;                  // 64 KB
constexpr int kPBytes = kRows * kH * 2;               // 16 KB
constexpr int kMaxS = kGatherMaxSplits;               // CTAs per unit
constexpr int kMmaWarp = 1;
constexpr int kSoft0 = 2;                             // first softmax warp
constexpr int kThreads = 6 * 32;
constexpr int kSoftBar = 1;                           // softmax warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S^T: 128 lanes (positions) x 64 heads
constexpr uint32_t kColO = 64;    // O^T: 4 blocks x (128 values x 64 heads)

// shared memory
constexpr int Q_OFF = 0;
constexpr int RING_OFF = Q_OFF + kQBytes;
constexpr int P_OFF = RING_OFF + kNSlot * kSlotBytes;
constexpr int F_OFF = P_OFF + kPBytes;  // floats: m, l, cr, mu [64] each,
                                        // red, red2 [4][64], inverse sums
                                        // and lse [64] each
constexpr int F_M = 0, F_L = 64, F_CR = 128, F_MU = 192, F_RED = 256,
              F_RED2 = 512, F_INV = 768, F_LSE = 832, F_END = 896;
constexpr int FLAG_OFF = F_OFF + F_END * 4;         // int [8]
constexpr int ROW_OFF = FLAG_OFF + 32;              // int [128]: chunk rows
constexpr int BAR_OFF = ROW_OFF + kRows * 4;
// full[4] empty[4] qfull sfull sfree pfull ofull done
constexpr int kBars = 2 * kNSlot + 6;
constexpr int SMEM = BAR_OFF + kBars * 8;
static_assert(SMEM <= 227 * 1024, "shared memory budget");

struct GatherParams {
  DecodeParams p;
  CUtensorMap tq;  // queries [batch * n_h][512] bf16, 64 x 64 boxes
};

// Address in a 128-byte-swizzled operand tile of 16-byte piece `c` of row
// `r`: rows of 128 bytes in 8-row atoms of 1 KB, piece c at c ^ (r % 8).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Reduce-scatter of 64 values across the 32 lanes of a warp: afterwards
// lane L holds the reduction over all lanes of values 2L and 2L + 1.
template <bool MAX>
__device__ __forceinline__ void reduce_scatter64(const float (&v)[64],
                                                 float &r0, float &r1) {
  const int lane = threadIdx.x & 31;
  float a[32];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float keep = hi ? v[i + 32] : v[i];
      const float send = hi ? v[i] : v[i + 32];
      const float got = __shfl_xor_sync(0xffffffffu, send, 16);
      a[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int w = 16, off = 8; off >= 1; w >>= 1, off >>= 1) {
    const bool hi = lane & off;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < w) {
        const float keep = hi ? a[i + w] : a[i];
        const float send = hi ? a[i] : a[i + w];
        const float got = __shfl_xor_sync(0xffffffffu, send, off);
        a[i] = MAX ? fmaxf(keep, got) : keep + got;
      }
    }
  }
  r0 = a[0];
  r1 = a[1];
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_gather_tc_kernel(const __grid_constant__ GatherParams gp) {
  const DecodeParams &p = gp.p;
  extern __shared__ __align__(1024) uint8_t smem[];
  float *fs = reinterpret_cast<float *>(smem + F_OFF);
  float *s_m = fs + F_M, *s_l = fs + F_L, *s_cr = fs + F_CR, *s_mu = fs + F_MU;
  float *s_red = fs + F_RED;    // per-warp maxima
  float *s_red2 = fs + F_RED2;  // per-warp sums
  float *s_inv = fs + F_INV, *s_lse = fs + F_LSE;
  int *flags = reinterpret_cast<int *>(smem + FLAG_OFF);
  volatile int *s_abort = flags;
  volatile int *s_issued = flags + 2;  // the query tile was requested
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(flags + 3);
  // cache row of each position of the current chunk, -1 for a zero row
  int *s_row = reinterpret_cast<int *>(smem + ROW_OFF);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + BAR_OFF);
  uint64_t *empty = full + kNSlot;
  uint64_t *qfull = empty + kNSlot;
  uint64_t *sfull = qfull + 1;
  uint64_t *sfree = sfull + 1;
  uint64_t *pfull = sfree + 1;
  uint64_t *ofull = pfull + 1;
  uint64_t *done = ofull + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int S = p.n_splits;  // CTAs per unit
  const int tiles = p.n_h / kH;
  const int u = (int)blockIdx.x / S, part = (int)blockIdx.x % S;
  const int b = u / tiles, ht = u % tiles;
  const int k = p.n_idx;
  const int e0 = (int)((long)k * part / S);
  const int e1 = (int)((long)k * (part + 1) / S);
  const int nch = (e1 - e0 + kRows - 1) / kRows;

  if (tid == 0) {
    for (int s = 0; s < kNSlot; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(qfull, 1);
    mbar_init(sfull, 1);
    mbar_init(sfree, 128);
    mbar_init(pfull, 128);
    mbar_init(ofull, 1);
    mbar_init(done, 1);
    *s_abort = 0;
    *s_issued = 0;
    fence_mbar_init();
  }
  if (tid < kH) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *s_tmem;
  // The setup above (barriers, tensor memory) touches nothing the kernel
  // before may write, so it overlaps that kernel's end; everything below
  // reads after its completion.
  pdl_wait();
  pdl_trigger();  // after the wait: dependants never overlap this grid's
                  // predecessor
  int T = p.seq_lens[b];
  if (T > p.max_seq_len) {
    if (tid == 0 && part == 0 && ht == 0) report(p.err, DEVERR_LEN);
    T = p.max_seq_len;
  }
  T = max(T, 0);
  // the swizzled operand tiles assume 1 KB atoms (every CTA sees the same
  // layout)
  const bool aligned = (smem_u32(smem) & 1023u) == 0;
  if (!aligned && tid == 0) {
    if (blockIdx.x == 0) report(p.err, DEVERR_TIMEOUT);
    *s_abort = 1;  // the outputs are then zeros (and flagged)
  }

  if (!aligned) {
    // nothing to do: every CTA takes this branch
  } else if (warp == 0) {
    // ======================= query tile (TMA) =============================
    if (nch > 0 && lane == 0) {
      // the unit's query tile: 64 heads x 512, eight 64-column boxes
      mbar_arrive_expect_tx(qfull, kQBytes);
      const int y = b * p.n_h + ht * kH;
      for (int cb = 0; cb < kD / 64; ++cb)
        tma_load_2d_plain(smem + Q_OFF + cb * kQCB, &gp.tq, 64 * cb, y,
                          qfull);
      *s_issued = 1;
    }
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer ===================================
    constexpr uint32_t idS = umma_idesc_bf16(kRows, kH, false);  // K, K
    // A MN-major (bit 15) and B MN-major (bit 16)
    constexpr uint32_t idO = umma_idesc_bf16(kRows, kH, true) | (1u << 15);
    const uint32_t q_addr = smem_u32(smem + Q_OFF);
    const uint32_t ring = smem_u32(smem + RING_OFF);
    const uint32_t p_addr = smem_u32(smem + P_OFF);
    bool ok = nch == 0 || __all_sync(0xffffffffu, mbar_wait(qfull, 0));
    for (int i = 0; ok && i < nch; ++i) {
      // ---- S^T = K Q^T over four 128-dim slices
      for (int j = 0; ok && j < kSlicesPerChunk / 2; ++j) {
        // slot j holds K_j, then V_j: phases 2i and 2i + 1 of each chunk
        const int slot = j;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], 0));
        // S^T of the chunk before was read by the softmax
        if (ok && j == 0 && i > 0)
          ok = __all_sync(0xffffffffu, mbar_wait(sfree, (i - 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const uint32_t a0 = ring + slot * kSlotBytes;
#pragma unroll
        for (int ks = 0; ks < kSliceCols / 16; ++ks) {
          // 16 dims: column block ks / 4 of the slice, 32-byte step
          const int cbk = ks >> 2, st = (ks & 3) * 32;
          const int qcb = j * (kSliceCols / 64) + cbk;  // Q column block
          const uint64_t a =
              umma_desc_sw128(a0 + cbk * kCBBytes + st, 16, 1024);
          const uint64_t bq = umma_desc_sw128(q_addr + qcb * kQCB + st, 16,
                                              1024);
          umma_ss_elect(tbase + kColS, a, bq, idS,
                        (j > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit_elect(&empty[slot]);
      }
      if (!ok) break;
      umma_commit_elect(sfull);
      // ---- O^T += V^T P^T over four 128-column value slices
      for (int j = 0; ok && j < kSlicesPerChunk / 2; ++j) {
        const int slot = j;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], 1));
        if (ok && j == 0)  // P of this chunk written, O^T rescaled
          ok = __all_sync(0xffffffffu, mbar_wait(pfull, i & 1));
        if (!ok) break;
        tc_fence_after();
        const uint32_t a0 = ring + slot * kSlotBytes;
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk) {
          // 16 positions = two 8-row groups of the slot and of P
          const uint64_t a = umma_desc_sw128(a0 + kk * 2048, kCBBytes, 1024);
          const uint64_t bp = umma_desc_sw128(p_addr + kk * 2048, kPBytes,
                                              1024);
          umma_ss_elect(tbase + kColO + j * kH, a, bp, idO,
                        (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit_elect(&empty[slot]);
      }
      if (!ok) break;
      umma_commit_elect(ofull);
    }
    if (!ok && lane == 0) {
      report(p.err, DEVERR_TIMEOUT);
      *s_abort = 1;
    }
    // every MMA issued has completed before the epilogue and the dealloc
    umma_commit_elect(done);
    mbar_wait(done, 0);
  } else {
    // ======================= workers: copies and softmax ==================
    // Worker warp w owns ring slot w: per chunk it copies K slice w (dims
    // 128 w ..) into it, hands it over, copies V slice w (values 128 w ..)
    // into it once the scores have read K slice w, runs the softmax while
    // that copy lands, then hands the V slice over. Lanes 0-15 copy one
    // row's 256-byte slice and lanes 16-31 the next, 16 bytes a lane, in
    // the MMA's 128-byte-swizzled layout; copies complete per thread
    // (commit groups), then a proxy fence orders them before the tensor
    // core's reads.
    const int sw = warp - kSoft0;              // 0..3: the slot it owns
    const int qw = warp & 3;                   // tensor-memory lane quarter
    const int r = qw * 32 + lane;              // chunk position (lane)
    const int st = tid - kSoft0 * 32;          // 0..127
    const uint32_t tl = tbase + ((uint32_t)(qw * 32) << 16);
    const float sl2 = p.scale_log2;
    uint8_t *myslot = smem + RING_OFF + sw * kSlotBytes;
    const int pc = lane & 15, cb = pc >> 3, c8 = pc & 7;
    // copy slice `col0` of every row of the chunk from `base` into my slot
    auto copy_slice = [&](const uint8_t *base, int col0) {
#pragma unroll 4
      for (int rr = 0; rr < kRows; rr += 2) {
        const int rw_i = rr + (lane >> 4);
        const int rw = s_row[rw_i];
        const uint8_t *src =
            base + ((long)max(rw, 0) * kD + col0) * 2 + pc * 16;
        cp_async16(myslot + cb * kCBBytes + sw128(rw_i, c8), src,
                   rw >= 0 ? 16 : 0);
      }
      cp_async_commit();
    };
    auto hand_over = [&]() {
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[sw]);
    };
    // After a bounded wait gives up, the loop still runs its course (every
    // worker warp meets the same named barriers) without copying or
    // waiting again.
    bool ok = true;
    for (int i = 0; i < nch; ++i) {
      // resolve row st of chunk i (a zero row: an entry out of the CTA's
      // range, a negative entry, one at or past the length, a bad block);
      // the barrier also means every worker has issued chunk i-1's copies
      {
        const int e = e0 + i * kRows + st;
        int row = -1;
        if (e < e1) {
          const int pos = p.indices[(long)b * p.n_idx + e];
          if (pos >= T) {
            report(p.err, DEVERR_INDEX);
          } else if (pos >= 0) {
            const int blk =
                p.block_table[(long)b * p.max_blocks + pos / p.block_size];
            if (blk < 0 || blk >= p.num_blocks)
              report(p.err, DEVERR_BLOCK);
            else
              row = blk * p.block_size + pos % p.block_size;
          }
        }
        named_sync(kSoftBar, 128);
        s_row[st] = row;
        named_sync(kSoftBar, 128);
      }
      const bool valid = s_row[r] >= 0;
      // K slice sw (its slot's V slice of the chunk before was consumed)
      if (ok && i > 0)
        ok = __all_sync(0xffffffffu, mbar_wait(&empty[sw], 1));
      if (ok) copy_slice(p.k, sw * kSliceCols);
      hand_over();
      // V slice sw once S^T has read K slice sw
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&empty[sw], 0));
      if (ok) copy_slice(p.v, sw * kSliceCols);
      ok = ok && __all_sync(0xffffffffu, mbar_wait(sfull, i & 1));
      tc_fence_after();
      float x[64];
      {
        uint32_t v[32];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          if (ok) {
            tmem_ld32(tl + kColS + h2 * 32, v);
            tmem_wait_ld(v);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j)
            x[h2 * 32 + j] =
                valid && ok ? __uint_as_float(v[j]) * sl2 : -INFINITY;
        }
      }
      tc_fence_before();
      mbar_arrive(sfree);
      // per-head maximum over the chunk's 128 positions
      float r0, r1;
      reduce_scatter64<true>(x, r0, r1);
      s_red[sw * 64 + 2 * lane] = r0;
      s_red[sw * 64 + 2 * lane + 1] = r1;
      named_sync(kSoftBar, 128);
      if (st < kH) {
        const float cmax = fmaxf(fmaxf(s_red[st], s_red[64 + st]),
                                 fmaxf(s_red[128 + st], s_red[192 + st]));
        const float mo = s_m[st];
        const float mn = fmaxf(mo, cmax);
        s_cr[st] = mo == -INFINITY ? 0.f : ex2(mo - mn);
        s_mu[st] = mn == -INFINITY ? 0.f : mn;
        s_m[st] = mn;
      }
      named_sync(kSoftBar, 128);
      // the probabilities replace the scores
#pragma unroll
      for (int h = 0; h < 64; ++h) x[h] = ex2(x[h] - s_mu[h]);
      if (i > 0) {
        // O^T of the chunk before is complete (and P is free again)
        ok = ok && __all_sync(0xffffffffu, mbar_wait(ofull, (i - 1) & 1));
        tc_fence_after();
        // rescale the O^T columns of heads whose maximum grew
        bool any = false;
#pragma unroll 8
        for (int h = 0; h < kH; ++h) any |= s_cr[h] != 1.f;
        if (any && ok) {
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t o[32];
              const uint32_t ta = tl + kColO + blk * kH + h2 * 32;
              tmem_ld32(ta, o);
              tmem_wait_ld(o);
#pragma unroll
              for (int j = 0; j < 32; ++j)
                o[j] = __float_as_uint(__uint_as_float(o[j]) *
                                       s_cr[h2 * 32 + j]);
              tmem_st32(ta, o);
            }
          }
          tmem_wait_st();
        }
      }
      // this position's row of P, bf16, swizzled (16-byte piece c holds
      // heads 8c .. 8c + 7)
      {
        uint8_t *prow = smem + P_OFF;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 w4;
          w4.x = pack_bf16x2(x[8 * c], x[8 * c + 1]);
          w4.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
          w4.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
          w4.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
          *reinterpret_cast<uint4 *>(prow + sw128(r, c)) = w4;
        }
      }
      // per-head sums over the chunk (in their own buffer: the maxima of
      // the next chunk may be written before these are read)
      reduce_scatter64<false>(x, r0, r1);
      s_red2[sw * 64 + 2 * lane] = r0;
      s_red2[sw * 64 + 2 * lane + 1] = r1;
      named_sync(kSoftBar, 128);
      if (st < kH)
        s_l[st] = s_l[st] * s_cr[st] + (s_red2[st] + s_red2[64 + st]) +
                  (s_red2[128 + st] + s_red2[192 + st]);
      fence_proxy_async_smem();  // P is read by the tensor core
      tc_fence_before();
      mbar_arrive(pfull);
      // the V slice, once landed
      hand_over();
    }
    if (ok && nch > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(ofull, (nch - 1) & 1));
      if (ok) tc_fence_after();
    }
    if (!ok && lane == 0) {
      report(p.err, DEVERR_TIMEOUT);
      *s_abort = 1;
    }
  }

  // ======================= teardown of the copies =========================
  // Every copy this CTA issued has landed before its ring is reused (the
  // workers waited for theirs; after an abort, the query tile's too).
  __syncthreads();
  if (tid == 0 && *s_abort && *s_issued) mbar_wait(qfull, 0);
  __syncthreads();

  // ======================= outputs ========================================
  // per head: 1 / sum and the log-sum-exp of this CTA's part
  if (tid < kH) {
    const float L = s_l[tid];
    const bool any = L > 0.f && !*s_abort && nch > 0;
    s_inv[tid] = any ? 1.f / L : 0.f;
    s_lse[tid] =
        any ? (s_m[tid] + log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const long bh0 = (long)b * p.n_h + (long)ht * kH;
  // S = 1: the outputs (bf16); else this CTA's part of the workspace,
  // [unit][part][64 heads][512 values] fp32 and [unit][part][64] lse
  const long slot = (long)u * S + part;
  if (warp >= kSoft0) {
    const int qw = warp & 3;
    const int r = qw * 32 + lane;
    const uint32_t tl = tbase + ((uint32_t)(qw * 32) << 16);
    const bool have = nch > 0 && !*s_abort;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      const int v = blk * 128 + r;  // this lane's value
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t o[32];
        if (have) {
          tmem_ld32(tl + kColO + blk * kH + h2 * 32, o);
          tmem_wait_ld(o);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int h = h2 * 32 + j;
          const float x = __uint_as_float(o[j]) * s_inv[h];
          if (S == 1)
            p.out[(bh0 + h) * kD + v] = f2bf(x);
          else
            p.ws_o[(slot * kH + h) * kD + v] = x;
        }
      }
    }
  }
  if (tid < kH) {
    if (S == 1) {
      if (p.lse) p.lse[bh0 + tid] = s_lse[tid];
    } else {
      p.ws_lse[slot * kH + tid] = s_lse[tid];
    }
  }
  tc_fence_before();
  __syncthreads();  // every read of tensor memory is done
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// The S CTAs of a unit leave their normalised partial outputs (64 heads x
// 512 values) and log-sum-exps in the workspace; this second launch merges
// the S parts of every output (log-sum-exp merge with a running maximum),
// one thread per float4, the loads of up to 20 parts in flight together
// (one round for the usual S <= 19; two blocks a SM). Grid: (units, 64 x
// 512 / 4 / 256).
constexpr int kGMergeThreads = 256;
constexpr int kMergeBatch = 20;
__global__ void __launch_bounds__(kGMergeThreads)
    gather_merge_kernel(const DecodeParams p) {
  pdl_trigger();
  pdl_wait();  // the parts of the decode launch
  const int S = p.n_splits;
  const int tiles = p.n_h / kH;
  const int u = blockIdx.x, b = u / tiles, ht = u % tiles;
  const int e = blockIdx.y * kGMergeThreads + threadIdx.x;  // float4 index
  if (e >= kH * kD / 4) return;
  const int h = e / (kD / 4), v = 4 * (e % (kD / 4));
  const float *lse = p.ws_lse + (long)u * S * kH + h;
  const float *o = p.ws_o + ((long)u * S * kH + h) * kD + v;
  float M = -INFINITY, W = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < S; s0 += kMergeBatch) {
    float l[kMergeBatch];
    float4 x[kMergeBatch];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      l[j] = -INFINITY;
      if (s0 + j < S) {
        l[j] = __ldcg(lse + (long)(s0 + j) * kH);
        x[j] = __ldcg(
            reinterpret_cast<const float4 *>(o + (long)(s0 + j) * kH * kD));
      }
    }
    float Mn = M;
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) Mn = fmaxf(Mn, l[j]);
    if (Mn == -INFINITY) continue;  // no part so far has any weight
    const float r = M == -INFINITY ? 0.f : expf(M - Mn);
    W *= r;
    a.x *= r;
    a.y *= r;
    a.z *= r;
    a.w *= r;
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      if (l[j] == -INFINITY) continue;  // an empty part adds nothing
      const float c = expf(l[j] - Mn);
      W += c;
      a.x = fmaf(c, x[j].x, a.x);
      a.y = fmaf(c, x[j].y, a.y);
      a.z = fmaf(c, x[j].z, a.z);
      a.w = fmaf(c, x[j].w, a.w);
    }
    M = Mn;
  }
  const long bh = (long)b * p.n_h + (long)ht * kH + h;
  const float iw = W > 0.f ? 1.f / W : 0.f;
  uint2 pk;
  pk.x = pack_bf16x2(a.x * iw, a.y * iw);
  pk.y = pack_bf16x2(a.z * iw, a.w * iw);
  *reinterpret_cast<uint2 *>(p.out + bh * kD + v) = pk;
  if (v == 0 && p.lse) p.lse[bh] = W > 0.f ? M + logf(W) : -INFINITY;
}

// 2-D tensor map of [rows][512] bf16 with 128-byte swizzle and boxes of 64
// columns x `box_rows` rows (rows out of range read as zeros).
cudaError_t make_rows_map(CUtensorMap *m, const void *base, long rows,
                          int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = tensor_map_encoder()(
      m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

// CTAs per unit: one wave (SMs / units), at most kGatherMaxSplits, none with
// fewer than 32 entries; when that gives every 128-entry chunk a CTA, the
// multiple of the chunk count below it if that keeps 3/4 of the CTAs, so
// that each CTA takes a whole chunk (or an equal fraction of one): for 8
// sequences and k = 2,048, 16 CTAs each
// instead of 19 (108 entries each, 20 of a chunk's rows zero-filled, and
// three more partials to merge) took the 8-layer step from 0.380 to
// 0.375 ms. `forced` > 0 asks for that many CTAs in all.
int gather_tc_splits(int units, int k, int sms, int forced) {
  int S = forced > 0 ? forced / units : sms / units;
  const int cap = (k + 31) / 32;
  if (forced <= 0) S = S < cap ? S : cap;
  S = S < kMaxS ? S : kMaxS;
  if (S < 1) return 1;
  const int chunks = (k + kRows - 1) / kRows;
  const int aligned = chunks * (S / chunks);
  if (forced <= 0 && S >= chunks && 4 * aligned >= 3 * S) S = aligned;
  return S;
}

cudaError_t launch_decode_sparse_tc(const DecodeParams &p, cudaStream_t s) {
  if (p.dk != kD || p.dv != kD || p.n_h % kH != 0 || p.n_kv != 1 ||
      p.n_splits < 1 || p.n_splits > kMaxS ||
      (long)p.num_blocks * p.block_size >= (1L << 31) - 1 ||
      (long)p.batch * p.n_h >= (1L << 31) || !tensor_map_encoder())
    return cudaErrorNotSupported;
  GatherParams gp;
  gp.p = p;
  cudaError_t e = make_rows_map(&gp.tq, p.q, (long)p.batch * p.n_h, kH);
  if (e != cudaSuccess) return e;
  auto kern = decode_gather_tc_kernel;
  static bool done[64] = {};
  e = set_smem_once(kern, SMEM, done);
  if (e != cudaSuccess) return e;
  const long ctas = (long)p.batch * (p.n_h / kH) * p.n_splits;
  if (ctas == 0) return cudaSuccess;
  e = launch_pdl(kern, dim3((unsigned)ctas), dim3(kThreads), SMEM, s, 1, gp);
  if (e != cudaSuccess || p.n_splits == 1) return e;
  const dim3 grid((unsigned)(p.batch * (p.n_h / kH)),
                  kH * kD / 4 / kGMergeThreads);
  return launch_pdl(gather_merge_kernel, grid, dim3(kGMergeThreads), 0, s, 1,
                    p);
}

}  // namespace kvd

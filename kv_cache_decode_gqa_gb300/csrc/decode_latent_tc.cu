// Latent-cache (MLA) decode on the 5th-generation tensor cores.
//
// DeepSeek-V2/V3 multi-head latent attention, absorbed form: every cached
// token is one 576-wide row (512-dim latent c, then the 64-dim shared rope
// key); a query head scores a token as q . row (q = absorbed latent query
// followed by its rope part) and its output is the softmax-weighted sum of
// the rows' latent parts. With 128 query heads on one row stream, the
// decode is a dense contraction: 128 x 1088 multiply-adds per 1152 cached
// bytes. This kernel runs it on tcgen05 MMAs with TMEM accumulators.
//
// Work: a persistent stream-K partition like the 64-head-tile latent
// kernel's, over 64-position chunks, with n_h / 128 x NP CTAs per lane:
// head tile ht (128 heads = the MMA's M) x value part vp (512 / NP of the
// output columns; NP = kLatentTcParts = 2). Each CTA of a lane computes the
// full scores S = Q K^T of its head tile (the softmax needs them) and
// O += P V for its value part. The parts read the same cache rows at about
// the same time, so all but one of the reads of a row hit L2.
//
// Tensor memory (512 columns x 128 lanes, lane = query head), NP = 2:
//   [0, 160)    Q: the first 320 of the tile's 576 query columns, bf16
//               (A operand of S)
//   [160, 224)  S: 128 x 64 fp32 scores of one chunk
//   [224, 256)  P: 128 x 64 bf16 probabilities (A operand of O)
//   [256, 512)  O: 128 x 256 fp32 output accumulator
// The query's other 256 columns are an A operand in shared memory (four
// 128-byte-swizzled boxes, 64 KB). With NP = 4 the whole query fits in
// tensor memory beside a 128-column O, but each tile's scores are then
// computed four times instead of twice: 1.15 against 0.90 ms for the
// 128-head, 64 x 32K-position call, whose tensor work the repeated scores
// dominate. The rest of shared memory holds two slots of each ring of cache
// chunks (64 rows x 1152 B, copied by TMA as nine 64-column boxes with
// 128-byte swizzle). An MMA of N = 64 positions streams its 128 x 16 A
// operand once per 64 positions; at N = 32 that stream, not the
// multiply-adds, set the MMA's duration.
//
// Warp roles (192 threads):
//   warp 0, one lane: TMA producer (per chunk: the block table lookup, the
//     score-only boxes into the score ring, this part's value boxes into
//     the value ring);
//   warp 1: TMEM allocation; the MMA loop (one elected lane issues each
//     MMA, the warp keeps the operands uniform): S(j) = 36 k-steps of
//     M=128 N=64 K=16 (A = Q, from TMEM for its first 320 columns and from
//     shared memory for the rest; B = K rows, K-major), and O += P(j) V(j)
//     as 4 k-steps of M=128 N=256 K=16 (A = P in TMEM, B = the chunk's
//     latent columns of this value part, MN-major);
//   warps 2..5 (one thread per head): online softmax. Thread r reads row r
//     of S(j) from TMEM, masks positions past the sequence end, and writes
//     P(j) = exp2(s * scale * log2 e - m) in bf16 back to TMEM, m the
//     running maximum of the head's scaled scores. When a chunk raises m the
//     thread rescales its row of O in TMEM and its running sum l. They also
//     store each unit's query tile into TMEM and shared memory and write the
//     results.
// Order of the MMA warp: S(j+1) as soon as the softmax has read S(j) (so it
// runs while the softmax of chunk j does), then O(j) once P(j) is written
// (the tensor core runs them in issue order); a chunk that starts a unit
// gets its S only after the previous unit's last O (its softmax threads
// first write that unit's results, then the new query tile). The softmax
// of chunk j+1 writes P and rescales O only after O(j) completed.
#include <cmath>

#include "kvd_common.cuh"
#include "stream_k.cuh"
#include "tcgen05.cuh"
#include "tmap.h"

namespace kvd {
namespace {

constexpr int kM = 128;             // query heads per CTA (MMA M)
constexpr int kDK = 576;            // row width (latent + rope)
constexpr int kDV = 512;            // latent width = output width
constexpr int kRows = kLatentTcRows;  // positions per chunk (MMA N of S)
constexpr int kBoxes = kDK / 64;    // 128-byte column boxes of a row
constexpr int kBoxBytes = kRows * 128;
constexpr int kQBox = kM * 128;     // one 64-column box of the query tile
constexpr int kNB = 256;            // largest batch of these calls
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
// The softmax offset m moves when a chunk's maximum exceeds it by more than
// this (log2 units). Any offset gives the same softmax, but the largest P is
// then up to 2^slack and its bf16 rounding is no longer exact: 0 keeps the
// running maximum exact, as the CUDA-core kernels do.
constexpr float kOffsetSlack = 0.f;

// The layout for NP value parts (CTAs of a lane per head tile).
template <int NP>
struct LCfg {
  static_assert(NP == 2 || NP == 4, "two or four value parts");
  static constexpr int VW = kDV / NP;     // output columns per CTA
  static constexpr int VB = VW / 64;      // value boxes of a chunk per CTA
  static constexpr int KB = kBoxes - VB;  // score-only boxes
  // tensor memory: the query's first QT boxes, S, P, O
  static constexpr uint32_t ColO = kTmemCols - VW;
  static constexpr uint32_t ColP = ColO - kRows / 2;
  static constexpr uint32_t ColS = ColP - kRows;
  static constexpr uint32_t ColQ = 0;
  static constexpr int QT = (int)ColS / 32;  // query boxes in tensor memory
  static constexpr int QS = kBoxes - QT;     // query boxes in shared memory
  // A chunk's boxes go to two rings: the score-only ones (freed as soon as
  // S has run) and this CTA's value boxes (read by S and by P V, freed
  // after P V), so a chunk's copy starts before the chunk ahead is done.
  static constexpr int KSlot = KB * kBoxBytes;
  static constexpr int VSlot = VB * kBoxBytes;
  static constexpr int QBYTES = QS * kQBox;
  static constexpr int FIXED =
      QBYTES + (int)sizeof(WorkPartitionT<kNB>) + 16 + (4 * 3 + 6) * 8 + 16;
  static constexpr int NS_FIT = (227 * 1024 - FIXED) / (KSlot + VSlot);
  static constexpr int NS = NS_FIT > 3 ? 3 : NS_FIT;  // slots of each ring
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + NS * KSlot;
  static constexpr int Q_OFF = V_OFF + NS * VSlot;  // 1 KB aligned
  static constexpr int WP_OFF = Q_OFF + QBYTES;
  static constexpr int BAR_OFF =
      (WP_OFF + (int)sizeof(WorkPartitionT<kNB>) + 15) / 16 * 16;
  // kfull[NS] kempty[NS] vfull[NS] vempty[NS] sfull sfree pfull ofull
  // qready done
  static constexpr int kBars = 4 * NS + 6;
  static constexpr int FLAG_OFF = BAR_OFF + kBars * 8;
  static constexpr int SMEM = FLAG_OFF + 16;
  static_assert(NS >= 2, "ring depth");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(ColO + VW == kTmemCols && ColS % 32 == 0,
                "tensor memory budget");
  static_assert(Q_OFF % 1024 == 0, "swizzle atoms");
};

struct LatentTcParams {
  DecodeParams p;
  CUtensorMap tmk;  // cache rows [rows][576], 64-column boxes
};

// Bounded wait for the producer: non-blocking tests only. A try_wait may
// suspend the thread, and the producer's wake-up after a slot is freed
// delays the copy that the tensor core waits for next (the producer warp
// has one active lane; the softmax warp on its scheduler has slack).
__device__ __forceinline__ bool spin_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 26); ++i)
    if (mbar_test_wait(bar, parity)) return true;
  return false;
}

template <int NP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_latent_tc_kernel(const __grid_constant__ LatentTcParams lp) {
  using C = LCfg<NP>;
  constexpr int kNS = C::NS;
  const DecodeParams &p = lp.p;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *sk = smem + C::K_OFF;
  uint8_t *sv = smem + C::V_OFF;
  uint8_t *sq = smem + C::Q_OFF;
  WorkPartitionT<kNB> &wp =
      *reinterpret_cast<WorkPartitionT<kNB> *>(smem + C::WP_OFF);
  uint64_t *kfull = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *kempty = kfull + kNS;
  uint64_t *vfull = kempty + kNS;
  uint64_t *vempty = vfull + kNS;
  uint64_t *sfull = vempty + kNS;
  uint64_t *sfree = sfull + 1;
  uint64_t *pfull = sfree + 1;
  uint64_t *ofull = pfull + 1;
  uint64_t *qready = ofull + 1;
  uint64_t *done = qready + 1;
  int *flags = reinterpret_cast<int *>(smem + C::FLAG_OFF);
  int *s_len_err = flags;
  volatile int *s_abort = flags + 1;
  volatile int *s_issued = flags + 2;
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(flags + 3);

  const int per_lane = p.n_h / kM * NP;  // CTAs sharing a chunk range
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_trigger();  // after the wait: see the merge launch

  if (tid == 0) {
    *s_len_err = 0;
    *s_abort = 0;
    *s_issued = 0;
  }
  __syncthreads();
  build_partition(wp, p, s_len_err, kRows, 1);
  if (tid == 0 && blockIdx.x == 0 && *s_len_err) report(p.err, DEVERR_LEN);
  const int total = wp.total;
  const int lanes = (int)gridDim.x / per_lane;
  const int P = min(lanes, max(total, 1));
  const int c = (int)blockIdx.x / per_lane;  // lane: a range of chunks
  const int ht = ((int)blockIdx.x % per_lane) / NP;  // head tile
  const int vp = (int)blockIdx.x % NP;                // value part

  if (blockIdx.x == 0) {  // sequences with nothing visible: out = 0, lse = -inf
    for (int b = 0; b < p.batch; ++b) {
      if (wp.nch[b] != 0) continue;
      for (int i = tid; i < p.n_h * kDV; i += kThreads)
        p.out[(long)b * p.n_h * kDV + i] = 0;
      if (p.lse)
        for (int i = tid; i < p.n_h; i += kThreads)
          p.lse[(long)b * p.n_h + i] = -INFINITY;
    }
  }
  if (c >= P || total == 0) return;  // (also CTAs beyond lanes * per_lane)
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layout needs 1 KB atoms
    if (tid == 0) report(p.err, DEVERR_TIMEOUT);
    return;
  }
  const int lo = range_lo(c, total, P);
  const int hi = range_lo(c + 1, total, P);
  const int n = hi - lo;

  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    mbar_init(sfull, 1);
    mbar_init(sfree, kM);
    mbar_init(pfull, kM);
    mbar_init(ofull, 1);
    mbar_init(qready, kM);
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *s_tmem;

  if (warp == 0) {
    // ======================= TMA producer ==================================
    if (lane == 0) {
      prefetch_tmap(&lp.tmk);
      ChunkCursor pc = cursor_at(wp, p.batch, lo);
      for (int i = 0; i < n; ++i) {
        const int s = i % kNS;
        const int t0 = pc.k * kRows;  // chunk start (inside one block)
        int blk = p.block_table[(long)pc.b * p.max_blocks + t0 / p.block_size];
        if (blk < 0 || blk >= p.num_blocks) {
          report(p.err, DEVERR_BLOCK);
          blk = 0;  // read a valid block; the result is flagged as wrong
        }
        const int row0 = blk * p.block_size + t0 % p.block_size;
        // the score-only boxes, once S(i - kNS) has run
        if (i >= kNS && !spin_wait(&kempty[s], (i / kNS - 1) & 1)) {
          report(p.err, DEVERR_TIMEOUT);
          *s_abort = 1;
        }
        if (*s_abort) break;
        mbar_arrive_expect_tx(&kfull[s], C::KSlot);
        for (int z = 0, j = 0; z < kBoxes; ++z) {
          if (z >= C::VB * vp && z < C::VB * (vp + 1)) continue;
          tma_load_2d_plain(sk + s * C::KSlot + j * kBoxBytes, &lp.tmk,
                            64 * z, row0, &kfull[s]);
          ++j;
        }
        *s_issued = 2 * i + 1;
        // the value part's boxes, once P V of chunk i - kNS has run
        if (i >= kNS && !spin_wait(&vempty[s], (i / kNS - 1) & 1)) {
          report(p.err, DEVERR_TIMEOUT);
          *s_abort = 1;
        }
        if (*s_abort) break;
        mbar_arrive_expect_tx(&vfull[s], C::VSlot);
        for (int z = 0; z < C::VB; ++z)
          tma_load_2d_plain(sv + s * C::VSlot + z * kBoxBytes, &lp.tmk,
                            64 * (C::VB * vp + z), row0, &vfull[s]);
        *s_issued = 2 * i + 2;
        cursor_next(wp, p.batch, 1, pc);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================= MMA issuer ====================================
    // The whole warp runs this loop (warp-uniform values); one elected lane
    // issues each MMA and commit.
    constexpr uint32_t idS = umma_idesc_bf16(kM, kRows, false);
    constexpr uint32_t idO = umma_idesc_bf16(kM, C::VW, true);
    const uint32_t k_addr = smem_u32(sk), v_addr = smem_u32(sv);
    // the query's boxes held in shared memory (K-major A operand)
    const uint64_t aq = umma_desc_sw128(smem_u32(sq), 16, 1024);
    ChunkCursor sc = cursor_at(wp, p.batch, lo);  // next S to issue
    ChunkCursor oc = sc;                          // next O to issue
    int s_prev_b = -1, o_prev_b = -1, units = 0;
    bool ok = true;
    auto wait_all = [&](uint64_t *bar, int parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };
    // S(j+1)'s commits (sfull, kempty) are issued after O(j)'s MMAs, not
    // between them: a commit in between delayed O(j) by a few hundred
    // cycles, and the tensor core idled after S(j+1) until it came; the
    // softmax and the score ring have that much slack.
    int pend_k = -1;  // score slot of an S whose commits are deferred
    auto issue_s = [&](int j, bool defer) -> bool {
      const int s = j % kNS;
      if (sc.b != s_prev_b) {  // the unit's query tile is in TMEM
        if (!wait_all(qready, units & 1)) return false;
        ++units;
        s_prev_b = sc.b;
      }
      if (!wait_all(&kfull[s], (j / kNS) & 1)) return false;
      if (!wait_all(&vfull[s], (j / kNS) & 1)) return false;
      // the softmax has read S(j-1)
      if (j >= 1 && !wait_all(sfree, (j - 1) & 1)) return false;
      tc_fence_after();
      // K-major B: box z = ks / 4 (in the value ring if it is one of this
      // part's, else in the score ring), 32-byte step ks % 4 inside the
      // 128-byte swizzled row (descriptor address in 16-byte units). A: the
      // query's box z, in tensor memory (z < QT) or in shared memory.
      const uint64_t bk = umma_desc_sw128(k_addr + s * C::KSlot, 16, 1024);
      const uint64_t bv = umma_desc_sw128(v_addr + s * C::VSlot, 16, 1024);
      const int v0 = C::VB * vp;
#pragma unroll
      for (int ks = 0; ks < kDK / 16; ++ks) {
        const int z = ks >> 2;
        const uint64_t b =
            (z >= v0 && z < v0 + C::VB)
                ? bv + (uint64_t)(((z - v0) * kBoxBytes) >> 4)
                : bk + (uint64_t)(((z < v0 ? z : z - C::VB) * kBoxBytes) >> 4);
        const uint64_t bs = b + (uint64_t)(((ks & 3) * 32) >> 4);
        if (z < C::QT)
          umma_ts_elect(tbase + C::ColS, tbase + C::ColQ + ks * 8, bs, idS,
                        ks > 0 ? 1u : 0u);
        else
          umma_ss_elect(tbase + C::ColS,
                        aq + (uint64_t)(((z - C::QT) * kQBox + (ks & 3) * 32) >>
                                        4),
                        bs, idS, ks > 0 ? 1u : 0u);
      }
      if (defer) {
        pend_k = s;
      } else {
        umma_commit_elect(sfull);
        umma_commit_elect(&kempty[s]);
      }
      cursor_next(wp, p.batch, 1, sc);
      return true;
    };
    auto issue_o = [&](int i) -> bool {
      const int s = i % kNS;
      if (!wait_all(pfull, i & 1)) return false;
      tc_fence_after();
      const bool first = oc.b != o_prev_b;
      o_prev_b = oc.b;
      // MN-major B: the part's 64-column boxes (LBO apart), 16 positions
      // (2 groups of 8 rows, SBO apart) per k-step
      const uint64_t b0 =
          umma_desc_sw128(v_addr + s * C::VSlot, kBoxBytes, 1024);
#pragma unroll
      for (int kk = 0; kk < kRows / 16; ++kk)
        umma_ts_elect(tbase + C::ColO, tbase + C::ColP + kk * 8,
                      b0 + (uint64_t)((kk * 16 * 128) >> 4), idO,
                      (!first || kk > 0) ? 1u : 0u);
      umma_commit_elect(&vempty[s]);
      umma_commit_elect(ofull);
      cursor_next(wp, p.batch, 1, oc);
      return true;
    };
    ok = n > 0 && issue_s(0, false);
    for (int i = 0; ok && i < n; ++i) {
      if (__any_sync(0xffffffffu, *s_abort)) break;
      // sc is chunk i+1's cursor here
      const bool next_starts = i + 1 < n && sc.b != s_prev_b;
      if (i + 1 < n && !next_starts) ok = issue_s(i + 1, true);
      ok = ok && issue_o(i);
      if (pend_k >= 0) {
        umma_commit_elect(sfull);
        umma_commit_elect(&kempty[pend_k]);
        pend_k = -1;
      }
      if (ok && next_starts) ok = issue_s(i + 1, false);
    }
    if (!ok && lane == 0) {
      report(p.err, DEVERR_TIMEOUT);
      *s_abort = 1;
    }
    // every MMA issued has completed before the TMEM is released
    umma_commit_elect(done);
    mbar_wait(done, 0);
    __syncwarp();
  } else {
    // ======================= softmax and epilogue ==========================
    const int qw = warp & 3;  // TMEM lane quarter of this warp
    const int r = qw * 32 + lane;  // head within the tile
    const uint32_t tl = tbase + ((uint32_t)(qw * 32) << 16);
    const float sl2 = p.scale_log2;
    ChunkCursor cc = cursor_at(wp, p.batch, lo);
    float m_ref = -INFINITY, l = 0.f;
    int cur_b = -1;
    bool ok = true;

    // results of unit b, whose last chunk was chunk `il` of the range
    auto flush = [&](int b, int il) -> bool {
      const bool w = mbar_wait(ofull, il & 1);
      if (!__all_sync(0xffffffffu, w)) return false;
      tc_fence_after();
      const int ustart = wp.pre[b];
      const int uend = ustart + wp.nch[b];
      const bool whole = ustart >= lo && uend <= hi;
      const long wslot = (long)c * 2 + partial_side(ustart, lo);
      const long head = (long)ht * kM + r;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int pc = 0; pc < C::VW / 32; ++pc) {
        uint32_t o[32];
        tmem_ld32(tl + C::ColO + pc * 32, o);
        tmem_wait_ld(o);
        const int col = vp * C::VW + pc * 32;
        if (whole) {
          uint4 *dst = reinterpret_cast<uint4 *>(
              p.out + ((long)b * p.n_h + head) * kDV + col);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * q4]) * inv,
                              __uint_as_float(o[8 * q4 + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv,
                              __uint_as_float(o[8 * q4 + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv,
                              __uint_as_float(o[8 * q4 + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv,
                              __uint_as_float(o[8 * q4 + 7]) * inv);
            dst[q4] = v;
          }
        } else {
          float4 *dst = reinterpret_cast<float4 *>(
              p.ws_o + (wslot * p.n_h + head) * kDV + col);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[q4] = make_float4(__uint_as_float(o[4 * q4]) * inv,
                                  __uint_as_float(o[4 * q4 + 1]) * inv,
                                  __uint_as_float(o[4 * q4 + 2]) * inv,
                                  __uint_as_float(o[4 * q4 + 3]) * inv);
        }
      }
      if (vp == 0) {
        const float lse =
            l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
        if (whole) {
          if (p.lse) p.lse[(long)b * p.n_h + head] = lse;
        } else {
          p.ws_lse[wslot * p.n_h + head] = lse;
        }
      }
      return true;
    };

    for (int i = 0; i < n; ++i) {
      if (__any_sync(0xffffffffu, *s_abort)) {
        ok = false;
        break;
      }
      const bool first = cc.b != cur_b;
      if (first) {
        if (cur_b >= 0 && !flush(cur_b, i - 1)) {
          ok = false;
          break;
        }
        cur_b = cc.b;
        m_ref = -INFINITY;
        l = 0.f;
        // the unit's query row of this head: its first QT boxes into TMEM
        // columns [0, 32 QT), the rest into shared memory (row r of each
        // box, 128-byte swizzled)
        const uint4 *qrow = reinterpret_cast<const uint4 *>(
            p.q + ((long)cc.b * p.n_h + (long)ht * kM + r) * kDK);
#pragma unroll 1
        for (int pc = 0; pc < C::QT; ++pc) {
          uint32_t v[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 u = __ldg(qrow + pc * 8 + j);
            v[4 * j] = u.x;
            v[4 * j + 1] = u.y;
            v[4 * j + 2] = u.z;
            v[4 * j + 3] = u.w;
          }
          tmem_st32(tl + C::ColQ + pc * 32, v);
        }
        if constexpr (C::QS > 0) {
#pragma unroll 1
          for (int pc = 0; pc < C::QS; ++pc) {
            uint8_t *row = sq + pc * kQBox + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4 *>(row + ((j ^ (r & 7)) << 4)) =
                  __ldg(qrow + (C::QT + pc) * 8 + j);
          }
          fence_proxy_async_smem();  // read by the tensor core
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(qready);
      }
      const bool w = mbar_wait(sfull, i & 1);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[kRows];
      {
        uint32_t v[32];
#pragma unroll
        for (int h2 = 0; h2 < kRows / 32; ++h2) {
          tmem_ld32(tl + C::ColS + h2 * 32, v);
          tmem_wait_ld(v);
#pragma unroll
          for (int j = 0; j < 32; ++j) x[h2 * 32 + j] = __uint_as_float(v[j]);
        }
      }
      tc_fence_before();
      mbar_arrive(sfree);

      const int nvalid = min(kRows, wp.len[cc.b] - cc.k * kRows);
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kRows; ++j) {
        x[j] = j < nvalid ? x[j] * sl2 : -INFINITY;
        mx = fmaxf(mx, x[j]);
      }
      bool need = false;
      if (first) {
        m_ref = mx;
      } else {
        need = mx > m_ref + kOffsetSlack;
      }
      if (i >= 1) {  // O(i-1) has read P and written O
        const bool w2 = mbar_wait(ofull, (i - 1) & 1);
        if (!__all_sync(0xffffffffu, w2)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, need)) {  // rescale this row of O
        const float cr = need ? ex2(m_ref - mx) : 1.f;
#pragma unroll 1
        for (int pc = 0; pc < C::VW / 32; ++pc) {
          uint32_t o[32];
          tmem_ld32(tl + C::ColO + pc * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            o[j] = __float_as_uint(__uint_as_float(o[j]) * cr);
          tmem_st32(tl + C::ColO + pc * 32, o);
        }
        if (need) {
          l *= cr;
          m_ref = mx;
        }
      }
      const float u = m_ref == -INFINITY ? 0.f : m_ref;
      float sum = 0.f;
#pragma unroll
      for (int h2 = 0; h2 < kRows / 32; ++h2) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float p0 = ex2(x[h2 * 32 + 2 * j] - u);
          const float p1 = ex2(x[h2 * 32 + 2 * j + 1] - u);
          sum += p0 + p1;
          pk[j] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tl + C::ColP + h2 * 16, pk);
      }
      l += sum;
      tmem_wait_st();
      if (nvalid < kRows) {
        // rows past the sequence end hold whatever the block held: zero this
        // part's value columns of them, so that P = 0 meets no NaN
        uint8_t *vb = sv + (i % kNS) * C::VSlot;
        const int cnt = (kRows - nvalid) * C::VB * 8;  // 16-byte pieces
        for (int e = r; e < cnt; e += kM) {
          const int row = nvalid + e / (C::VB * 8), box = (e / 8) % C::VB,
                    piece = e & 7;
          *reinterpret_cast<uint4 *>(vb + box * kBoxBytes + row * 128 +
                                     piece * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(pfull);
      cursor_next(wp, p.batch, 1, cc);
    }
    if (ok && cur_b >= 0 && !flush(cur_b, n - 1)) ok = false;
    if (!ok && lane == 0) {
      report(p.err, DEVERR_TIMEOUT);
      *s_abort = 1;
    }
  }

  // ======================= teardown ========================================
  if (tid == 0 && *s_abort) {
    // no copy may still land in this CTA's shared memory after it exits
    // loads issued: chunk i's score part when issued > 2i, its value part
    // when issued > 2i + 1; wait for the last one of each slot
    const int issued = *s_issued;
    const int nk = (issued + 1) >> 1, nv = issued >> 1;
    for (int s = 0; s < kNS; ++s) {
      int lk = -1, lv = -1;
      for (int i = s; i < nk; i += kNS) lk = i;
      for (int i = s; i < nv; i += kNS) lv = i;
      if (lk >= 0) mbar_wait(&kfull[s], (lk / kNS) & 1);
      if (lv >= 0) mbar_wait(&vfull[s], (lv / kNS) & 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// The cache as a 2-D tensor [rows][576] of bf16 rows (1152 bytes), copied
// in boxes of 64 columns (128 bytes) x one chunk of rows, 128-byte swizzle.
cudaError_t make_latent_map(CUtensorMap *m, const void *base, long rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)kDK, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kDK * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kRows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = tensor_map_encoder()(
      m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool latent_tc_supported(int n_h, int block_size, long num_blocks) {
  return n_h % kM == 0 && block_size % kRows == 0 &&
         num_blocks * block_size < (1L << 31) && tensor_map_encoder() != nullptr;
}

cudaError_t launch_decode_mla_tc(const DecodeParams &p, cudaStream_t s) {
  if (p.dk != kDK || p.dv != kDV || p.batch > kNB || p.n_kv != 1 ||
      !latent_tc_supported(p.n_h, p.block_size, p.num_blocks))
    return cudaErrorNotSupported;
  LatentTcParams lp;
  lp.p = p;
  cudaError_t e =
      make_latent_map(&lp.tmk, p.k, (long)p.num_blocks * p.block_size);
  if (e != cudaSuccess) return e;
  constexpr int NP = kLatentTcParts;
  auto kern = decode_latent_tc_kernel<NP>;
  static bool done[64] = {};
  e = set_smem_once(kern, LCfg<NP>::SMEM, done);
  if (e != cudaSuccess) return e;
  // n_splits counts 64-head tiles per lane (the partial layout and the
  // merge use it); this launch has n_h / 128 x NP CTAs per lane.
  const int lanes = p.n_splits / (p.n_h / 64);
  e = launch_pdl(kern, dim3(lanes * (p.n_h / kM) * NP), dim3(kThreads),
                 LCfg<NP>::SMEM, s, 1, lp);
  if (e != cudaSuccess || lanes <= 1) return e;
  return launch_merge_mla(p, kRows, s);
}

}  // namespace kvd

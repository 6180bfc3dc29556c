// Decode attention on the CUDA cores for small query groups (n_h / n_kv =
// G in {1, 2, 4}: MHA and narrow GQA). At these group sizes a decode step
// does 2G FLOPs per cached element ("KV cache", "Why decoding wastes almost
// all of your FLOPs": intensity 2 n_h / (n_kv b)), so the kernel is bound by
// HBM bandwidth and its job is to keep every SM's copy engine streaming.
//
// Persistent stream-K launch (stream_k.cuh): one CTA per SM, each taking an
// equal contiguous share of all (sequence, head group, 64-token chunk)
// work. A head group is HP consecutive kv heads: with 64-token blocks the
// HP heads' rows of one block are adjacent in the cache layout, so a whole
// chunk of a group moves as one bulk copy of HP x 64 rows for K and one for
// V. HP is chosen so that a copy is about 32 KB: the copy engine streams
// large copies much faster than small ones. A producer warp resolves 32
// chunks at a time (cursor and block ids, one chunk per lane, loaded in
// parallel), then streams each chunk into an NS-deep shared-memory ring
// with bulk asynchronous copies completing on "full" mbarriers; it refills
// a stage once the consumers release it on its "empty" mbarrier, so it runs
// up to NS chunks ahead across unit boundaries.
//
// The producer also copies the chunk's query rows into the stage, so a
// consumer starting a new unit reads its query from shared memory.
//
// Eight consumer warps process a chunk, 8 / HP warps per head of the group:
// lane group g = lane / 8 of local warp w owns the head's rows
// 8 HP w + 4 i + g (i < 2 HP); its 8 lanes each hold D/8 elements of
// the row, so a row is read from shared memory as one conflict-free sweep,
// and the dot product finishes with three xor-shuffles. Each lane group
// keeps its own online-softmax state (running max, sum, output slice) per
// head, in log2 units (the query is pre-multiplied by scale * log2 e). Each
// consumer warp walks the same deterministic chunk sequence as the
// producer, so all warps agree on unit changes. At a unit change a warp
// merges its four lane-group states and drops the result into one of two
// shared-memory flush slots, then goes on with the next unit at once. A
// finisher warp combines the warp states of each head of a flushed unit and
// writes the final output (a unit lying wholly in this CTA's range) or a
// partial, which the merge launch queued after this one combines with the
// other covering CTAs' partials (log-sum-exp merge). (A variant in which the
// last covering CTA to finish merged the unit itself, on arrival counters,
// was measured slower: its fence, atomic and merge sat at the end of every
// CTA, where the separate launch overlaps the next call's first copies.)
//
// With KVD_SEQS_PREFIX_READY the producer copies the ring's first chunks
// (not a unit's last chunk, which holds the newest position) before the
// grid dependency wait, so the cache streams while the previous kernel
// finishes; their query rows follow after the wait.
#include <cuda_fp16.h>

#include <cmath>

#include "kvd_common.cuh"
#include "stream_k.cuh"

namespace kvd {
namespace {

constexpr int kConsumers = 256;            // 8 consumer warps
constexpr int kWarps = kConsumers / 32;
constexpr int kProducer = kWarps;          // warp index of the producer
constexpr int kFinisher = kWarps + 1;      // warp index of the finisher
constexpr int kThreads = kConsumers + 64;
constexpr int kFinalBar = 1;               // the consumer warps, at the end
constexpr int kAppendBar = 2;              // finisher -> producer: rows written

template <int D, int G, int DT, int HP>
struct Cfg {
  static constexpr int ROW = row_bytes(D, DT);       // bytes per cached row
  static constexpr int HSTAGE = kStageRows * ROW;    // one head's K (or V)
  static constexpr int STAGE = HP * HSTAGE;          // K (or V) bytes / chunk
  static constexpr int E = D / 8;                    // elements per lane
  static constexpr int WPH = kWarps / HP;            // warps per head
  static constexpr int ITER = 2 * HP;                // 4-row steps per warp
  static constexpr int QB = HP * G * D * 2;          // query rows / stage
  static constexpr int SLOT = kWarps * G * (D + 2);   // floats per slot
  static constexpr int MERGE = 2 * SLOT * 4;
  // cluster merge (query groups of 1, units of at most 2 heads, whose
  // rings keep their depth with it): the partials of up to 8 CTAs of a unit
  // (GU heads x D outputs, then GU log-sum-exps, padded to 16 floats) in
  // the shared memory of the cluster's rank 0
  static constexpr int GU = HP * G;
  static constexpr int CL_RANKS = G == 1 && GU <= 2 ? 8 : 0;
  static constexpr int CPART = GU * D + 16;
  static constexpr int CBUF = CL_RANKS * CPART * 4;
  // ring depth: up to 160 KB (one head) or 192 KB (head groups) of K and V,
  // within what the flush slots, the partition and the barriers leave of
  // 227 KB (1 KB kept for the kernel's static shared variables)
  static constexpr int RING_BUDGET = HP == 1 ? 160 * 1024 : 192 * 1024;
  static constexpr int FIXED =
      MERGE + CBUF + (int)sizeof(WorkPartition) + 16 + 21 * 8 + 1024;
  static constexpr int NS_FIT = (227 * 1024 - FIXED) / (2 * STAGE + QB);
  static constexpr int NS_WANT = RING_BUDGET / (2 * STAGE);
  static constexpr int NS_MIN = NS_FIT < NS_WANT ? NS_FIT : NS_WANT;
  static constexpr int NS = NS_MIN > 8 ? 8 : NS_MIN;  // ring depth
  static constexpr int RING = 2 * NS * STAGE + NS * QB;
  static constexpr int CB_OFF = RING + MERGE;  // 16-byte aligned
  static constexpr int WP_OFF = CB_OFF + CBUF;
  static constexpr int BAR_OFF =
      (WP_OFF + (int)sizeof(WorkPartition) + 15) / 16 * 16;
  static constexpr int SMEM = BAR_OFF + (2 * NS + 5) * 8;
  static_assert(CB_OFF % 16 == 0 && GU <= 16, "cluster buffer layout");
};

// Element index (within a row of D) of the e-th value a lane holds.
template <int D, int DT>
__device__ __forceinline__ int elem_index(int sub, int e) {
  if constexpr (DT == DT_BF16) {
    return (e / 8) * 64 + sub * 8 + (e % 8);
  } else {
    return sub * (D / 8) + e;
  }
}

// The lane's D/8 elements of a shared-memory row, as floats. MXFP4 (D =
// 128): the lane's 16 channels are one scale group (8 code bytes at
// sub * 8): the code values, without the scale (row_scale gives it; the
// callers apply it once per row), each byte widened to an exact f16 pair
// by the hardware conversion.
template <int D, int DT>
__device__ __forceinline__ void load_row(const uint8_t *row, int sub,
                                         float (&x)[D / 8]) {
  if constexpr (DT == DT_MXFP4) {
    static_assert(D == 128, "one 16-channel scale group per lane");
    const uint2 u = *reinterpret_cast<const uint2 *>(row + sub * 8);
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int t = 0; t < 8; ++t) {  // byte t: channels 2t (low nibble), 2t+1
      const uint32_t h = e2m1x2_to_f16x2(w[t >> 2] >> (8 * (t & 3)));
      x[2 * t] = f16lo(h);
      x[2 * t + 1] = f16hi(h);
    }
  } else if constexpr (DT == DT_BF16) {
#pragma unroll
    for (int j = 0; j < D / 64; ++j) {
      const uint4 u =
          *reinterpret_cast<const uint4 *>(row + j * 128 + sub * 16);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        x[j * 8 + 2 * t] = bf16lo(w[t]);
        x[j * 8 + 2 * t + 1] = bf16hi(w[t]);
      }
    }
  } else {
    constexpr int WORDS = D / 32;  // 32-bit words of fp8 codes per lane
    uint32_t w[WORDS];
    if constexpr (WORDS == 4) {
      const uint4 u = *reinterpret_cast<const uint4 *>(row + sub * 16);
      w[0] = u.x, w[1] = u.y, w[2] = u.z, w[3] = u.w;
    } else {
      const uint2 u = *reinterpret_cast<const uint2 *>(row + sub * 8);
      w[0] = u.x, w[1] = u.y;
    }
#pragma unroll
    for (int t = 0; t < WORDS; ++t) {
      const uint32_t a = e4m3x2_to_f16x2((uint16_t)(w[t] & 0xffff));
      const uint32_t b = e4m3x2_to_f16x2((uint16_t)(w[t] >> 16));
      x[4 * t] = f16lo(a);
      x[4 * t + 1] = f16hi(a);
      x[4 * t + 2] = f16lo(b);
      x[4 * t + 3] = f16hi(b);
    }
  }
}

// The factor the lane's values of a row take: the lane's MXFP4 group scale
// (its E4M3 code at D/2 + sub), 1 for the other formats.
template <int D, int DT>
__device__ __forceinline__ float row_scale(const uint8_t *row, int sub) {
  if constexpr (DT == DT_MXFP4) {
    return f16lo(e4m3x2_to_f16x2((uint16_t)row[D / 2 + sub]));
  } else {
    return 1.0f;
  }
}

// 2^(x - M) for a state with running max x, 0 for an empty state.
__device__ __forceinline__ float weight(float x, float M) {
  return x == -INFINITY ? 0.f : ex2(x - M);
}

template <int D, int G, int DT, int HP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_simt_kernel(const DecodeParams p) {
  using C = Cfg<D, G, DT, HP>;
  constexpr int GU = HP * G;  // query heads per unit
  constexpr int E = C::E;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *sk = smem;
  uint8_t *sv = smem + C::NS * C::STAGE;
  uint8_t *sq = smem + 2 * C::NS * C::STAGE;
  float *slots = reinterpret_cast<float *>(smem + C::RING);
  WorkPartition &wp = *reinterpret_cast<WorkPartition *>(smem + C::WP_OFF);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *empty = full + C::NS;
  uint64_t *sfull = empty + C::NS;  // flush slot written (8 warp arrivals)
  uint64_t *sempty = sfull + 2;     // flush slot consumed (finisher)
  uint64_t *cbar = sempty + 2;      // cluster merge: the other ranks' parts
  float *cbuf = reinterpret_cast<float *>(smem + C::CB_OFF);
  __shared__ int s_len_err;
  __shared__ volatile int s_abort, s_issued, s_producer_done;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 3, sub = lane & 7;
  // With stable lengths and block table, the plan and the producer's first
  // block-id lookups run before the predecessor grid completes; every other
  // global access (cache, queries, scales, outputs) waits for it, except
  // the cache copies KVD_SEQS_PREFIX_READY allows. Dependants are let in only
  // after this grid's own wait (see the merge launch).
  const bool early = p.flags & FLAG_SEQS_STABLE;
  if (!early) {
    pdl_wait();
    pdl_trigger();
  }
  const bool prefetch = early && (p.flags & FLAG_PREFIX_READY);

  if (tid == 0) {
    s_len_err = 0;
    s_abort = 0;
    s_issued = 0;
    s_producer_done = 0;
  }
  __syncthreads();
  const int n_units = p.n_kv / HP;  // head groups per sequence
  build_partition(wp, p, &s_len_err, kStageRows, n_units);
  if (tid == 0 && blockIdx.x == 0 && s_len_err) report(p.err, DEVERR_LEN);
  const int total = wp.total;
  // Cluster merge: the cs CTAs of a cluster share one unit. Rank 0's
  // barrier counts the other ranks' consumer threads, each arriving after
  // its stores of the rank's partial into rank 0's buffer; the cluster
  // barrier here (every thread still present) makes the barrier's
  // initialisation visible before any arrival.
  const int cs = C::CL_RANKS >= 2 && p.cluster > 1 ? p.cluster : 1;
  const int crank = cs > 1 ? (int)cluster_rank() : 0;
  if (cs > 1) {
    if (crank == 0 && tid == 0) {
      mbar_init(cbar, (cs - 1) * kConsumers);
      fence_mbar_init();
    }
    cluster_sync();
  }
  const int P = p.whole_units || cs > 1 ? (int)gridDim.x
                                        : min((int)gridDim.x, max(total, 1));
  const int c = blockIdx.x;

  // sequences with nothing visible: out = 0, lse = -inf; fused-append rows
  // that no chunk reads
  if (c == 0) {
    if (early) pdl_wait();
    if (p.pos && warp == 0) append_unread_rows(p, wp, lane);
    for (int b = 0; b < p.batch; ++b) {
      if (wp.nch[b] != 0) continue;
      for (int i = tid; i < p.n_h * D; i += kThreads)
        p.out[(long)b * p.n_h * D + i] = 0;
      if (p.lse)
        for (int i = tid; i < p.n_h; i += kThreads)
          p.lse[(long)b * p.n_h + i] = -INFINITY;
    }
  }
  if (c >= P || total == 0) return;
  int lo, hi;
  if (cs > 1) {  // an equal part of unit c / cs
    const int u = c / cs, ub = u / n_units, uh = u % n_units;
    const int us = wp.pre[ub] + uh * wp.nch[ub], nc = wp.nch[ub];
    lo = us + (int)((long)nc * crank / cs);
    hi = us + (int)((long)nc * (crank + 1) / cs);
  } else {
    lo = p.whole_units ? unit_lo(wp, p.batch, n_units, c)
                       : range_lo(c, total, P);
    hi = p.whole_units ? unit_lo(wp, p.batch, n_units, c + 1)
                       : range_lo(c + 1, total, P);
  }
  const int n = hi - lo;
  // an empty unit of a whole-unit launch (a cluster's empty part still
  // hands rank 0 an empty partial)
  if (n == 0 && cs == 1) return;
  // this CTA's partial in rank 0's cluster buffer
  const uint32_t cpart =
      cs > 1 ? cluster_saddr(cbuf + crank * C::CPART, 0) : 0u;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sfull[s], kWarps);
      mbar_init(&sempty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // Combine the warp states of unit (b, h) held in flush slot sl and write
  // the unit's outputs (a unit inside this CTA's range) or its partial;
  // thread t of nt cooperating threads.
  auto write_unit = [&](int b, int h, int sl, int t, int nt) {
    const int ustart = wp.pre[b] + h * wp.nch[b];
    const int uend = ustart + wp.nch[b];
    const float *wm = slots + sl * C::SLOT;
    const float *wl = wm + kWarps * G;
    const float *wo = wl + kWarps * G;  // [warp][G][D]
    const bool whole = cs == 1 && ustart >= lo && uend <= hi;
    const int wslot = c * 2 + partial_side(ustart, lo);
    const long bh0 = (long)b * p.n_h + h * GU;
    const int ln = t & 31, wq = t >> 5, nw = nt >> 5;
    // lane jg (head (j, g) of the unit) of every warp: the weights c_w of
    // the head's warps, and its log-sum-exp
    float cw[C::WPH];
    {
      const int jg = ln < GU ? ln : 0;
      const int j = jg / G, g = jg % G, w0 = j * C::WPH;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::WPH; ++w) M = fmaxf(M, wm[(w0 + w) * G + g]);
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < C::WPH; ++w) {
        cw[w] = weight(wm[(w0 + w) * G + g], M);
        L = fmaf(wl[(w0 + w) * G + g], cw[w], L);
      }
      const float vs = DT == DT_FP8 ? p.v_scale[h * HP + j] : 1.0f;
      const float f = L > 0.f ? vs / L : 0.f;
#pragma unroll
      for (int w = 0; w < C::WPH; ++w) cw[w] *= f;
      const float lse_nat = (M + log2f(L)) * 0.69314718055994531f;
      if (wq == 0 && ln < GU) {
        if (cs > 1)
          st_dsmem_f32(cpart + (GU * D + jg) * 4, lse_nat);
        else if (!whole)
          p.ws_lse[(long)wslot * GU + jg] = lse_nat;
        else if (p.lse)
          p.lse[bh0 + jg] = lse_nat;
      }
    }
    // the output rows, four columns a lane (a warp step covers 32 / (D / 4)
    // rows)
    constexpr int LPR = D / 4;
    constexpr int RPI = 32 / LPR;
    const int col4 = ln % LPR;
    for (int r0 = wq * RPI; r0 < GU; r0 += nw * RPI) {
      const int jg = r0 + ln / LPR;
      const int jr = jg < GU ? jg : 0;
      const int w0 = (jr / G) * C::WPH, g = jr % G;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < C::WPH; ++w) {
        const float cf = __shfl_sync(0xffffffffu, cw[w], jr);
        const float4 v =
            reinterpret_cast<const float4 *>(wo + ((w0 + w) * G + g) * D)[col4];
        acc.x = fmaf(cf, v.x, acc.x);
        acc.y = fmaf(cf, v.y, acc.y);
        acc.z = fmaf(cf, v.z, acc.z);
        acc.w = fmaf(cf, v.w, acc.w);
      }
      if (jg >= GU) continue;
      if (whole) {
        uint2 packed;
        packed.x = pack_bf16x2(acc.x, acc.y);
        packed.y = pack_bf16x2(acc.z, acc.w);
        reinterpret_cast<uint2 *>(p.out + (bh0 + jg) * D)[col4] = packed;
      } else if (cs > 1) {
        st_dsmem_f4(cpart + (jg * D + 4 * col4) * 4, acc);
      } else {
        reinterpret_cast<float4 *>(p.ws_o + ((long)wslot * GU + jg) * D)[col4] =
            acc;
      }
    }
  };

  // ======================= producer warp ==================================
  if (warp == kProducer) {
    const uint64_t policy = policy_evict_first();
    constexpr int kPre = 4;  // block ids prefetched per chunk
    bool appended = false;   // fused append: the finisher's rows are written
    bool waited = !early;    // past the grid dependency wait
    int npre = 0;            // chunks copied before the wait (ring's first pass)
    int fb = 0, fh = 0, fk = 0;  // lane t < 32: chunk t's unit, for the wait
    // The wait, then the query rows of the chunks copied before it (chunk t
    // sits in stage t; a unit's first chunk, and chunk 0, carry its rows).
    auto wait_then_queries = [&]() {
      pdl_wait();
      pdl_trigger();
      waited = true;
      for (int t = 0; t < npre; ++t) {
        const int bt = __shfl_sync(0xffffffffu, fb, t);
        const int ht = __shfl_sync(0xffffffffu, fh, t);
        const int kt = __shfl_sync(0xffffffffu, fk, t);
        if (lane == 0 && (t == 0 || kt == 0))
          bulk_g2s(sq + t * C::QB, p.q + ((long)bt * p.n_h + ht * GU) * D,
                   C::QB, &full[t]);
      }
    };
    for (int base = 0; base < n; base += 32) {
      const int mine = base + lane;
      int mb = 0, mh = 0, mk = 0, mrows = 0, mtok = 0;
      int mblk[kPre] = {0, 0, 0, 0};
      int mpos = -1;  // fused append: the sequence's new slot
      if (mine < n) {
        const ChunkCursor cur = cursor_at(wp, p.batch, lo + mine);
        mb = cur.b, mh = cur.h, mk = cur.k;
        if (p.pos) mpos = p.pos[mb];
        const int tok =
            seq_first(p, mb, wp.len[mb], kStageRows) + mk * kStageRows;
        mtok = tok;
        mrows = min(kStageRows, wp.len[mb] - tok);
        const int lb0 = tok / p.block_size;
        const int lb1 = (tok + mrows - 1) / p.block_size;
        const int32_t *bt = p.block_table + (long)mb * p.max_blocks;
#pragma unroll
        for (int j = 0; j < kPre; ++j)
          if (lb0 + j <= lb1) mblk[j] = bt[lb0 + j];
      }
      const int cnt = min(32, n - base);
      if (base == 0) fb = mb, fh = mh, fk = mk;
      if (early && base == 0 && !prefetch) wait_then_queries();
      bool stop = false;
      for (int j = 0; j < cnt && !stop; ++j) {
        const int b = __shfl_sync(0xffffffffu, mb, j);
        const int h = __shfl_sync(0xffffffffu, mh, j);
        const int k = __shfl_sync(0xffffffffu, mk, j);
        const int rows = __shfl_sync(0xffffffffu, mrows, j);
        // position of the chunk's first row (looked up with its block ids)
        const int tok = __shfl_sync(0xffffffffu, mtok, j);
        int blk[kPre];
#pragma unroll
        for (int t = 0; t < kPre; ++t)
          blk[t] = __shfl_sync(0xffffffffu, mblk[t], j);
        if (!waited) {
          // before the wait: only the ring's first pass, and no chunk that
          // holds a unit's newest position or a row this call appends
          const int pn = p.pos ? __shfl_sync(0xffffffffu, mpos, j) : -1;
          if (base + j >= C::NS || k == wp.nch[b] - 1 ||
              (pn >= tok && pn < tok + rows))
            wait_then_queries();
        }
        if (p.pos && !appended) {
          // fused append: before the first chunk holding a new row is
          // copied, wait for the finisher to have written this CTA's rows
          const int P = __shfl_sync(0xffffffffu, mpos, j);
          if (P >= tok && P < tok + rows) {
            named_sync(kAppendBar, 64);
            appended = true;
          }
        }
        int go = 1;
        if (lane == 0) {
          const int i = base + j;
          const int s = i % C::NS;
          if (i >= C::NS && !mbar_wait(&empty[s], (i / C::NS - 1) & 1)) {
            report(p.err, DEVERR_TIMEOUT);
            go = 0;
          }
          if (s_abort) go = 0;
          if (go) {
            // the query rows travel only with a unit's first chunk here (the
            // consumers read them when the unit starts)
            const bool qrows = i == 0 || k == 0;
            // MXFP4 rows (72 bytes) are copied in pairs: a copy is a
            // multiple of 16 bytes. An odd tail takes the next row of its
            // block too (masked like any row past the end).
            const int crows =
                DT == DT_MXFP4 && rows < kStageRows ? (rows + 1) & ~1 : rows;
            mbar_arrive_expect_tx(&full[s], 2u * HP * crows * C::ROW +
                                                (qrows ? C::QB : 0u));
            // before the wait the query rows are left to wait_then_queries
            if (qrows && waited)
              bulk_g2s(sq + s * C::QB, p.q + ((long)b * p.n_h + h * GU) * D,
                       C::QB, &full[s]);
            const int32_t *bt = p.block_table + (long)b * p.max_blocks;
            const int lb0 = tok / p.block_size;
            if constexpr (HP > 1) {
              // 64-token blocks: the chunk is one block; its HP heads' rows
              // are adjacent, so a full chunk is one copy per tensor
              int pb = blk[0];
              if (pb < 0 || pb >= p.num_blocks) {
                report(p.err, DEVERR_BLOCK);
                pb = 0;  // read a valid block; the result is flagged as wrong
              }
              const size_t off =
                  ((size_t)pb * p.n_kv + (size_t)h * HP) * kStageRows * C::ROW;
              if (rows == kStageRows) {
                bulk_g2s_hint(sk + s * C::STAGE, p.k + off, C::STAGE,
                              &full[s], policy);
                bulk_g2s_hint(sv + s * C::STAGE, p.v + off, C::STAGE,
                              &full[s], policy);
              } else {
#pragma unroll
                for (int j = 0; j < HP; ++j) {
                  const size_t oj = off + (size_t)j * C::HSTAGE;
                  bulk_g2s_hint(sk + s * C::STAGE + j * C::HSTAGE, p.k + oj,
                                crows * C::ROW, &full[s], policy);
                  bulk_g2s_hint(sv + s * C::STAGE + j * C::HSTAGE, p.v + oj,
                                crows * C::ROW, &full[s], policy);
                }
              }
            }
            int done = HP > 1 ? crows : 0;
            while (done < crows) {
              const int t = tok + done;
              const int slot = t % p.block_size;
              const int piece = min(crows - done, p.block_size - slot);
              const int lb = t / p.block_size - lb0;
              int pb = lb == 0   ? blk[0]
                       : lb == 1 ? blk[1]
                       : lb == 2 ? blk[2]
                       : lb == 3 ? blk[3]
                                 : bt[lb0 + lb];
              if (pb < 0 || pb >= p.num_blocks) {
                report(p.err, DEVERR_BLOCK);
                pb = 0;  // read a valid block; the result is flagged as wrong
              }
              const size_t off =
                  (((size_t)pb * p.n_kv + h) * p.block_size + slot) * C::ROW;
              bulk_g2s_hint(sk + s * C::STAGE + done * C::ROW, p.k + off,
                            piece * C::ROW, &full[s], policy);
              bulk_g2s_hint(sv + s * C::STAGE + done * C::ROW, p.v + off,
                            piece * C::ROW, &full[s], policy);
              done += piece;
            }
            s_issued = i + 1;
          }
        }
        stop = __shfl_sync(0xffffffffu, go, 0) == 0;
        if (!waited && !stop) npre = base + j + 1;
      }
      if (stop) break;
    }
    if (!waited) wait_then_queries();
    if (p.pos && !appended) named_sync(kAppendBar, 64);
    if (lane == 0) s_producer_done = 1;
    return;
  }

  // ======================= finisher warp ==================================
  // Every unit of the range but the last: the consumer warps write the last
  // one themselves, all 256 threads at once, since nothing overlaps it.
  if (warp == kFinisher) {
    if (p.pos) {  // fused append: the new rows this CTA's chunks hold
      append_range_rows(p, wp, HP, lo, hi, lane, early);
      named_arrive(kAppendBar, 64);
    } else if (early) {
      pdl_wait();
    }
    // (an empty part of a cluster has no chunk to point at)
    ChunkCursor fc =
        n > 0 ? cursor_at(wp, p.batch, lo) : ChunkCursor{0, 0, 0};
    int x = lo;
    for (int e = 0; x < hi; ++e) {
      const int b = fc.b, h = fc.h;
      const int ustart = wp.pre[b] + h * wp.nch[b];
      const int uend = ustart + wp.nch[b];
      const int xend = min(uend, hi);
      if (xend >= hi) break;  // the last unit
      const int sl = e & 1;
      if (!mbar_wait(&sfull[sl], (e >> 1) & 1)) {
        if (lane == 0) report(p.err, DEVERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      write_unit(b, h, sl, lane, 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[sl]);  // the slot may be reused
      x = xend;
      if (x < hi) fc = cursor_at(wp, p.batch, x);
    }
    return;
  }

  // ======================= consumer warps =================================
  if (early) pdl_wait();
  int cur_b = -1, cur_h = -1, n_flush = 0;
  float qf[G][E], m[G], l[G], o[G][E];
  const int hj = warp / C::WPH;  // this warp's head within the group
  const int lw = warp % C::WPH;  // and its rank among that head's warps

  auto start_unit = [&](int s, int h) {
    const float qs =
        p.scale_log2 * (DT == DT_FP8 ? p.k_scale[h * HP + hj] : 1.0f);
    const uint16_t *qrows =
        reinterpret_cast<const uint16_t *>(sq + s * C::QB) + hj * G * D;
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int e = 0; e < E; e += 8) {
        const uint4 u = *reinterpret_cast<const uint4 *>(
            qrows + g * D + elem_index<D, DT>(sub, e));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          qf[g][e + 2 * t] = bf16lo(w[t]) * qs;
          qf[g][e + 2 * t + 1] = bf16hi(w[t]) * qs;
        }
      }
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) o[g][e] = 0.f;
    }
  };

  // Merge this warp's four lane-group states and hand them to the finisher
  // (or, for the last unit, leave them in the slot for the consumer warps).
  auto flush = [&](bool last) {
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m[g], off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l[g], off);
        const float M = fmaxf(m[g], m2);
        const float a = weight(m[g], M);
        const float a2 = weight(m2, M);
        l[g] = l[g] * a + l2 * a2;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float o2 = __shfl_xor_sync(0xffffffffu, o[g][e], off);
          o[g][e] = o[g][e] * a + o2 * a2;
        }
        m[g] = M;
      }
    }
    const int sl = n_flush & 1;
    if (n_flush >= 2) {
      bool ok = !s_abort && mbar_wait(&sempty[sl], ((n_flush >> 1) - 1) & 1);
      if (!__all_sync(0xffffffffu, ok) && lane == 0) {
        if (!s_abort) report(p.err, DEVERR_TIMEOUT);
        s_abort = 1;
      }
    }
    float *wm = slots + sl * C::SLOT;
    float *wl = wm + kWarps * G;
    float *wo = wl + kWarps * G;
    if (lane < 8) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (sub == 0) {
          wm[warp * G + g] = m[g];
          wl[warp * G + g] = l[g];
        }
#pragma unroll
        for (int e = 0; e < E; ++e)
          wo[(warp * G + g) * D + elem_index<D, DT>(sub, e)] = o[g][e];
      }
    }
    __syncwarp();
    if (lane == 0 && !last) mbar_arrive(&sfull[sl]);
    ++n_flush;
  };

  // (an empty part of a cluster has no chunk to point at)
  ChunkCursor cc =
      n > 0 ? cursor_at(wp, p.batch, lo) : ChunkCursor{0, 0, 0};
  for (int i = 0; i < n; ++i) {
    const int s = i % C::NS;
    // a copy that never completes (bounded wait) sets the abort flag; the
    // remaining chunks are then skipped and the results flagged wrong
    bool ok = !s_abort && mbar_wait(&full[s], (i / C::NS) & 1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) {
      if (!s_abort) report(p.err, DEVERR_TIMEOUT);
      s_abort = 1;
    }
    if (cc.b != cur_b || cc.h != cur_h) {
      if (cur_b >= 0) flush(false);
      cur_b = cc.b;
      cur_h = cc.h;
      start_unit(s, cur_h);
    }
    // rows [nlo, nvalid) of the chunk are attended: below nlo lie positions
    // before the sliding window (first chunk only), from nvalid on
    // positions past the visible length
    const bool win = has_window(p);
    const int ctok =
        (win ? seq_first(p, cc.b, wp.len[cc.b], kStageRows) : 0) +
        cc.k * kStageRows;
    const int nvalid = min(kStageRows, wp.len[cc.b] - ctok);
    const int nlo = win ? seq_lo(p, cc.b, wp.len[cc.b]) - ctok : 0;
    if (ok) {
      const uint8_t *kst = sk + s * C::STAGE + hj * C::HSTAGE;
      const uint8_t *vst = sv + s * C::STAGE + hj * C::HSTAGE;
      float sc[C::ITER][G];
#pragma unroll
      for (int i2 = 0; i2 < C::ITER; ++i2) {
        const int r = lw * 4 * C::ITER + i2 * 4 + grp;
        float kx[E];
        load_row<D, DT>(kst + r * C::ROW, sub, kx);
        const float ks = row_scale<D, DT>(kst + r * C::ROW, sub);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            a0 = fmaf(qf[g][e], kx[e], a0);
            a1 = fmaf(qf[g][e + 1], kx[e + 1], a1);
          }
          sc[i2][g] = (a0 + a1) * ks;
        }
      }
#pragma unroll
      for (int i2 = 0; i2 < C::ITER; ++i2) {
        const int r = lw * 4 * C::ITER + i2 * 4 + grp;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float v = sc[i2][g];
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          sc[i2][g] = r >= nlo && r < nvalid ? v : -INFINITY;
        }
      }
      float pr[C::ITER][G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mx = sc[0][g];
#pragma unroll
        for (int i2 = 1; i2 < C::ITER; ++i2) mx = fmaxf(mx, sc[i2][g]);
        const float m_new = fmaxf(m[g], mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float corr = ex2(m[g] - m_use);
        float lsum = 0.f;
#pragma unroll
        for (int i2 = 0; i2 < C::ITER; ++i2) {
          pr[i2][g] = ex2(sc[i2][g] - m_use);
          lsum += pr[i2][g];
        }
        l[g] = l[g] * corr + lsum;
        m[g] = m_new;
#pragma unroll
        for (int e = 0; e < E; ++e) o[g][e] *= corr;
      }
#pragma unroll
      for (int i2 = 0; i2 < C::ITER; ++i2) {
        const int r = lw * 4 * C::ITER + i2 * 4 + grp;
        if (r >= nlo && r < nvalid) {
          float vx[E];
          load_row<D, DT>(vst + r * C::ROW, sub, vx);
          const float vsr = row_scale<D, DT>(vst + r * C::ROW, sub);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float pv = pr[i2][g] * vsr;
#pragma unroll
            for (int e = 0; e < E; ++e) o[g][e] = fmaf(pv, vx[e], o[g][e]);
          }
        }
      }
    }
    // release the stage to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    cursor_next(wp, p.batch, n_units, cc);
  }
  if (cur_b >= 0) {
    flush(true);
    named_sync(kFinalBar, kConsumers);  // every warp's state is in the slot
    write_unit(cur_b, cur_h, (n_flush - 1) & 1, tid, kConsumers);
  }
  if (cs > 1) {
    // a part with no chunk is empty (its outputs are never read)
    if (cur_b < 0 && tid < GU)
      st_dsmem_f32(cpart + (GU * D + tid) * 4, -INFINITY);
    if (crank != 0) {
      mbar_arrive_remote(cluster_saddr(cbar, 0));
    } else {
      // rank 0: every part is in the buffer; log-sum-exp merge of the cs
      // parts of each output, one float4 a thread
      named_sync(kFinalBar, kConsumers);
      const bool got = mbar_wait_cluster(cbar, 0);
      if (!got && tid == 0) report(p.err, DEVERR_TIMEOUT);
      const int u = c / cs, ub = u / n_units, uh = u % n_units;
      const long bh0 = (long)ub * p.n_h + (long)uh * GU;
      for (int e = tid; got && e < GU * D / 4; e += kConsumers) {
        const int jg = (4 * e) / D;
        float M = -INFINITY;
        for (int r = 0; r < cs; ++r)
          M = fmaxf(M, cbuf[r * C::CPART + GU * D + jg]);
        float W = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < cs && M != -INFINITY; ++r) {
          const float lr = cbuf[r * C::CPART + GU * D + jg];
          if (lr == -INFINITY) continue;  // an empty part adds nothing
          const float w = expf(lr - M);
          const float4 v =
              reinterpret_cast<const float4 *>(cbuf + r * C::CPART)[e];
          W += w;
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z);
          acc.w = fmaf(w, v.w, acc.w);
        }
        const float iw = W > 0.f ? 1.f / W : 0.f;
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * iw, acc.y * iw);
        packed.y = pack_bf16x2(acc.z * iw, acc.w * iw);
        reinterpret_cast<uint2 *>(p.out + bh0 * D)[e] = packed;
        if ((4 * e) % D == 0 && p.lse)
          p.lse[bh0 + jg] = W > 0.f ? M + logf(W) : -INFINITY;
      }
    }
  }

  if (s_abort && tid == 0) {
    // let every copy the producer issued land before the CTA exits
    for (int t = 0; t < (1 << 20) && !s_producer_done; ++t) __nanosleep(1000);
    const int issued = s_issued;
    for (int st = 0; st < C::NS; ++st) {
      int last = -1;
      for (int c2 = st; c2 < issued; c2 += C::NS) last = c2;
      if (last >= 0) mbar_wait(&full[st], (last / C::NS) & 1);
    }
  }
}

template <int D, int G, int DT, int HP>
cudaError_t launch_t(const DecodeParams &p, cudaStream_t s) {
  using C = Cfg<D, G, DT, HP>;
  static_assert(C::SMEM <= 226 * 1024, "shared memory budget");
  static_assert(C::NS >= 2, "ring depth");
  auto kern = decode_simt_kernel<D, G, DT, HP>;
  if (p.cluster > 1 && (C::CL_RANKS < p.cluster || p.n_splits % p.cluster))
    return cudaErrorNotSupported;
  static bool done[64] = {};  // one table per instantiation
  cudaError_t e = set_smem_once(kern, C::SMEM, done);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(p.n_splits), dim3(kThreads), C::SMEM, s,
                 p.cluster > 1 ? p.cluster : 1, p);
  if (e != cudaSuccess) return e;
  return launch_merge_dense<D, G * HP>(p, p.n_kv / HP, s);
}

// Largest cluster (2..8 CTAs per unit, at most sms / units) whose `units`
// clusters are resident together and cover at least 60 % of the SMs (a
// one-sequence decode took the same time on 96 of 152 SMs as on all of
// them, and 11 % longer on 76; fewer CTAs would lose more than the merge
// launch costs), for the instantiation of query groups of 1; 0 when none is.
// Looked up once per device and unit count.
template <int D, int DT, int HP>
int cluster_fit(int units, int sms) {
  using C = Cfg<D, 1, DT, HP>;
  if (C::CL_RANKS < 2) return 0;
  static int memo[64][kMaxDecodeBatch + 1];
  static bool init = false;
  if (!init) {
    for (auto &row : memo)
      for (int &v : row) v = -1;
    init = true;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 ||
      units < 1 || units > kMaxDecodeBatch)
    return 0;
  if (memo[dev][units] >= 0) return memo[dev][units];
  auto kern = decode_simt_kernel<D, 1, DT, HP>;
  static bool done[64] = {};
  int best = 0;
  if (set_smem_once(kern, C::SMEM, done) == cudaSuccess) {
    for (int cs = sms / units < C::CL_RANKS ? sms / units : C::CL_RANKS;
         cs >= 2 && !best && 10 * cs * units >= 6 * sms; --cs) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(units * cs);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = C::SMEM;
      cudaLaunchAttribute a[1];
      a[0].id = cudaLaunchAttributeClusterDimension;
      a[0].val.clusterDim.x = cs;
      a[0].val.clusterDim.y = 1;
      a[0].val.clusterDim.z = 1;
      cfg.attrs = a;
      cfg.numAttrs = 1;
      int m = 0;
      if (cudaOccupancyMaxActiveClusters(&m, kern, &cfg) == cudaSuccess &&
          m >= units)
        best = cs;
    }
  }
  (void)cudaGetLastError();  // a refused query leaves no sticky error
  memo[dev][units] = best;
  return best;
}

// Head-group sizes built: 1 always; one larger size per row width (a 32 KB
// copy of 64-token rows), for groups of 1 or 2 query heads.
template <int D, int DT>
constexpr int kWideHP = row_bytes(D, DT) >= 256 ? 2 : 4;

template <int D, int DT>
cudaError_t launch_g(const DecodeParams &p, cudaStream_t s) {
  constexpr int W = kWideHP<D, DT>;
  const int g = p.n_h / p.n_kv;
  if (p.hp == 1) {
    switch (g) {
      case 1: return launch_t<D, 1, DT, 1>(p, s);
      case 2: return launch_t<D, 2, DT, 1>(p, s);
      case 4: return launch_t<D, 4, DT, 1>(p, s);
    }
  } else if (p.hp == W) {
    switch (g) {
      case 1: return launch_t<D, 1, DT, W>(p, s);
      case 2: return launch_t<D, 2, DT, W>(p, s);
    }
  }
  return cudaErrorNotSupported;
}

}  // namespace

int simt_cluster_size(int head_dim, int dtype, int hp, int units, int sms) {
  if (dtype == DT_MXFP4)
    return head_dim == 128 && hp == kWideHP<128, DT_MXFP4>
               ? cluster_fit<128, DT_MXFP4, kWideHP<128, DT_MXFP4>>(units, sms)
               : 0;
  if (head_dim == 128) {
    if (dtype == DT_BF16)
      return hp == 1 ? cluster_fit<128, DT_BF16, 1>(units, sms)
                     : cluster_fit<128, DT_BF16, kWideHP<128, DT_BF16>>(units,
                                                                        sms);
    return hp == 1 ? cluster_fit<128, DT_FP8, 1>(units, sms)
                   : cluster_fit<128, DT_FP8, kWideHP<128, DT_FP8>>(units, sms);
  }
  if (head_dim == 64) {
    if (dtype == DT_BF16)
      return hp == 1 ? cluster_fit<64, DT_BF16, 1>(units, sms)
                     : cluster_fit<64, DT_BF16, kWideHP<64, DT_BF16>>(units,
                                                                      sms);
    return hp == 1 ? cluster_fit<64, DT_FP8, 1>(units, sms)
                   : cluster_fit<64, DT_FP8, kWideHP<64, DT_FP8>>(units, sms);
  }
  return 0;
}

int simt_heads_per_stage(int n_kv, int g, int head_dim, int dtype,
                         int block_size) {
  if (block_size != kStageRows || g > 2) return 1;
  const int w = dtype == DT_MXFP4 ? kWideHP<128, DT_MXFP4>
                : head_dim == 128 ? (dtype == DT_BF16 ? kWideHP<128, DT_BF16>
                                                      : kWideHP<128, DT_FP8>)
                                  : (dtype == DT_BF16 ? kWideHP<64, DT_BF16>
                                                      : kWideHP<64, DT_FP8>);
  return n_kv % w == 0 ? w : 1;
}

cudaError_t launch_decode_simt(const DecodeParams &p, cudaStream_t s) {
  const bool fp8 = p.dtype == DT_FP8;
  if (p.batch > kMaxDecodeBatch) return cudaErrorNotSupported;
  if (p.dtype == DT_MXFP4)
    return p.dk == 128 ? launch_g<128, DT_MXFP4>(p, s) : cudaErrorNotSupported;
  if (p.dk == 128) return fp8 ? launch_g<128, DT_FP8>(p, s)
                              : launch_g<128, DT_BF16>(p, s);
  if (p.dk == 64) return fp8 ? launch_g<64, DT_FP8>(p, s)
                             : launch_g<64, DT_BF16>(p, s);
  return cudaErrorNotSupported;
}

}  // namespace kvd

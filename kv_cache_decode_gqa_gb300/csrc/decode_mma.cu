// Decode attention on the tensor cores for wide query groups (n_h / n_kv =
// G in {8, 16}, head_dim 128): the Llama-3.1-70B shape, bf16 or fp8 cache.
// A decode step does 2G FLOPs per cached element ("KV cache", "Why decoding
// wastes almost all of your FLOPs": intensity 2 n_h / (n_kv b)), 8 to 32
// FLOP/byte here: past what the CUDA cores sustain at HBM speed, while the
// work is still far below the tensor pipe's, so warp-level MMA
// (m16n8k16, fp32 accumulators) is enough to keep the kernel bound by HBM.
//
// Same persistent stream-K structure as the CUDA-core kernel (stream_k.cuh):
// one CTA per SM with an equal share of all (sequence, head group, 64-token
// chunk) work, a producer warp, a finisher warp (it writes every unit of the
// range but the last, which the consumer warps write together), and four
// consumer warps. (It ignores KVD_SEQS_PREFIX_READY: copying the first
// chunks before the grid dependency wait, as the CUDA-core kernel does,
// measured slower here -- 8.74 against 8.59 ms for the 80-layer
// Llama-3.1-70B step, 5.21 against 5.13 ms with the fp8 cache.)
// A head group is HP consecutive kv heads (HP = 2 for an fp8 cache with
// 64-token blocks, whose HP heads' rows are adjacent): the producer moves a
// chunk's K and V with tiled TMA copies of HP x 64 rows (boxes of 128-byte
// rows, 128-byte swizzle, so the ldmatrix reads of every 8x8 tile are free
// of bank conflicts) -- few large copies, which the copy engine streams
// much faster than many small ones -- and, with a unit's first chunk, the
// HP x G query rows. 4 / HP consumer warps take each head, 16 HP tokens of
// it per warp.
//
// Per chunk a consumer warp computes S = Q K^T for its 16 tokens (query
// heads on the MMA's M = 16 rows; G = 8 leaves rows 8..15 at zero), scales
// S in fp32 by softmax scale * log2 e (times the K scale for fp8), runs the
// online softmax per head row, and accumulates O += P V with P rounded to
// the MMA's 16-bit type. fp8 codes are widened exactly to f16 in registers
// (so the fp8 path runs f16 MMAs with the query in f16): for K the
// dimensions inside each 16-wide k-step are taken in a permuted order,
// matched in the query fragments (a dot product does not depend on the
// order of its terms); for V the output columns come out permuted and are
// put back in order when the state is flushed. The V scale multiplies the
// final output.
#include <cmath>

#include "kvd_common.cuh"
#include "stream_k.cuh"
#include "tmap.h"

namespace kvd {
namespace {

constexpr int kAppendBar = 1;  // finisher -> producer: fused-append rows written
constexpr int kFinalBar = 2;   // the consumer warps, at the end

constexpr int kD = 128;
constexpr int kWarps = 4;                 // consumer warps
constexpr int kConsumers = kWarps * 32;
constexpr int kProducer = kWarps;
constexpr int kFinisher = kWarps + 1;
constexpr int kThreads = kConsumers + 64;

struct MmaParams {
  DecodeParams p;
  CUtensorMap tmk;  // K cache as [rows][head_dim], 128-byte swizzled boxes
  CUtensorMap tmv;
};

template <int DT, int HP>
struct MCfg {
  static constexpr int ES = DT == DT_BF16 ? 2 : 1;
  static constexpr int ROW = kD * ES;        // bytes per cached row
  static constexpr int NBOX = ROW / 128;     // 128-byte column boxes per row
  static constexpr int BOX = HP * 64 * 128;  // one column box of a chunk
  static constexpr int STAGE = HP * 64 * ROW;  // K (or V) bytes per chunk
  static constexpr int QB = HP * 16 * kD * 2;  // query rows of a unit
  static constexpr int WPH = kWarps / HP;    // consumer warps per head
  static constexpr int TPW = 64 / WPH;       // tokens per warp and chunk
  static constexpr int NSUB = TPW / 16;      // 16-token tiles per warp
  static constexpr int SLOT = kWarps * 16 * (kD + 2);  // floats per slot
  // One flush slot: the finisher writes a unit in about the time of one or
  // two chunks, and units span tens of chunks at the long contexts this
  // kernel is sized for (a short-window unit of 2-3 chunks may wait for the
  // slot briefly). The rest of 226 KB is ring, as deep as fits: the bytes in
  // flight per SM are what keep HBM busy.
  static constexpr int NSLOT = 1;
  static constexpr int MERGE = NSLOT * SLOT * 4;
  static constexpr int FIXED =
      MERGE + (int)sizeof(WorkPartition) + 16 + 40 * 8 + 1024;
  static constexpr int NS_FIT = (226 * 1024 - FIXED) / (2 * STAGE + QB);
  static constexpr int NS = NS_FIT > 12 ? 12 : NS_FIT;
  static constexpr int RING = 2 * NS * STAGE + NS * QB;
  static constexpr int WP_OFF = RING + MERGE;
  static constexpr int BAR_OFF =
      (WP_OFF + (int)sizeof(WorkPartition) + 15) / 16 * 16;
  static constexpr int SMEM = BAR_OFF + (2 * NS + 2 * NSLOT) * 8;
};

// Shared-memory address of byte `cb` (0..127) of row `r` of a 128-byte
// swizzled box (16-byte chunk c of row r sits at chunk c ^ (r % 8)).
__device__ __forceinline__ uint32_t swz(uint32_t box, int r, int cb) {
  return box + r * 128 + ((((cb >> 4) ^ (r & 7)) << 4) | (cb & 15));
}

// Output column of accumulator element j (0..3) of n-tile nt for lane
// quad index c (fp8: the V tiles hold even / odd columns of 16-wide groups).
template <int DT>
__device__ __forceinline__ int out_col(int nt, int c, int j) {
  if constexpr (DT == DT_BF16) {
    return 8 * nt + 2 * c + (j & 1);
  } else {
    return 16 * (nt >> 1) + 4 * c + 2 * (j & 1) + (nt & 1);
  }
}

__device__ __forceinline__ uint32_t f16pair_from_bf16(uint32_t u) {
  return pack_f16x2(bf16lo(u), bf16hi(u));
}

template <int DT, int HP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_mma_kernel(const __grid_constant__ MmaParams mp) {
  using C = MCfg<DT, HP>;
  const DecodeParams &p = mp.p;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *sk = smem;
  uint8_t *sv = smem + C::NS * C::STAGE;
  uint8_t *sq = smem + 2 * C::NS * C::STAGE;
  float *slots = reinterpret_cast<float *>(smem + C::RING);
  WorkPartition &wp = *reinterpret_cast<WorkPartition *>(smem + C::WP_OFF);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *empty = full + C::NS;
  uint64_t *sfull = empty + C::NS;
  uint64_t *sempty = sfull + C::NSLOT;
  __shared__ int s_len_err;
  __shared__ volatile int s_abort, s_issued, s_producer_done;

  const int G = p.n_h / p.n_kv;  // 8 or 16 (checked by the launcher)
  const int GU = HP * G;         // query heads per unit
  const int n_units = p.n_kv / HP;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // With stable lengths and block table, the plan and the producer's first
  // block-id lookups run before the predecessor grid completes; every other
  // global access (cache, queries, scales, outputs) waits for it. Dependants
  // are let in only after this grid's own wait (see the merge launch).
  const bool early = p.flags & FLAG_SEQS_STABLE;
  if (!early) {
    pdl_wait();
    pdl_trigger();
  }
  const int qr = lane >> 2, qc = lane & 3;  // MMA fragment row / column quad

  if (tid == 0) {
    s_len_err = 0;
    s_abort = 0;
    s_issued = 0;
    s_producer_done = 0;
  }
  __syncthreads();
  build_partition(wp, p, &s_len_err, kStageRows, n_units);
  if (tid == 0 && blockIdx.x == 0 && s_len_err) report(p.err, DEVERR_LEN);
  const int total = wp.total;
  const int P = p.whole_units ? (int)gridDim.x
                              : min((int)gridDim.x, max(total, 1));
  const int c = blockIdx.x;

  if (c == 0) {
    if (early) pdl_wait();
    if (p.pos && warp == 0) append_unread_rows(p, wp, lane);
    for (int b = 0; b < p.batch; ++b) {
      if (wp.nch[b] != 0) continue;
      for (int i = tid; i < p.n_h * kD; i += kThreads)
        p.out[(long)b * p.n_h * kD + i] = 0;
      if (p.lse)
        for (int i = tid; i < p.n_h; i += kThreads)
          p.lse[(long)b * p.n_h + i] = -INFINITY;
    }
  }
  if (c >= P || total == 0) return;
  const int lo = p.whole_units ? unit_lo(wp, p.batch, n_units, c)
                               : range_lo(c, total, P);
  const int hi = p.whole_units ? unit_lo(wp, p.batch, n_units, c + 1)
                               : range_lo(c + 1, total, P);
  const int n = hi - lo;
  if (n == 0) return;  // an empty unit of a whole-unit launch

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&sfull[s], kWarps);
      mbar_init(&sempty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // Write flush slot `sl`, which holds every consumer warp's state of unit
  // (b, h), as the unit's output (a unit wholly in this CTA's range) or as
  // this CTA's partial of it, with threads t = 0 .. nt - 1 (whole warps).
  // Lane jg (a query head of the unit) of every warp combines the states of
  // its kv head's WPH warps once: M = max m_w, L = sum l_w 2^(m_w - M); the
  // output row is sum_w c_w o_w with c_w = 2^(m_w - M) vs / L, written by
  // warps in turn, four columns a lane.
  auto write_unit = [&](int b, int h, int sl, int t, int nt) {
    const int ustart = wp.pre[b] + h * wp.nch[b];
    const int uend = ustart + wp.nch[b];
    const float *wm = slots + sl * C::SLOT;  // [warp][16]
    const float *wl = wm + kWarps * 16;      // [warp][16]
    const float *wo = wl + kWarps * 16;      // [warp][16][D]
    const bool whole = ustart >= lo && uend <= hi;
    const int wslot = c * 2 + partial_side(ustart, lo);
    const long bh0 = (long)b * p.n_h + h * GU;
    const int ln = t & 31, wq = t >> 5, nw = nt >> 5;
    float cw[C::WPH];
    {
      const int jg = ln < GU ? ln : 0;
      const int j = jg / G, g = jg % G, w0 = j * C::WPH;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::WPH; ++w) M = fmaxf(M, wm[(w0 + w) * 16 + g]);
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < C::WPH; ++w) {
        const float mw = wm[(w0 + w) * 16 + g];
        cw[w] = mw == -INFINITY ? 0.f : ex2(mw - M);
        L = fmaf(wl[(w0 + w) * 16 + g], cw[w], L);
      }
      const float vs = DT == DT_FP8 ? p.v_scale[h * HP + j] : 1.0f;
      const float f = L > 0.f ? vs / L : 0.f;
#pragma unroll
      for (int w = 0; w < C::WPH; ++w) cw[w] *= f;
      const float lse_nat = (M + log2f(L)) * 0.69314718055994531f;
      if (wq == 0 && ln < GU) {
        if (!whole)
          p.ws_lse[(long)wslot * GU + jg] = lse_nat;
        else if (p.lse)
          p.lse[bh0 + jg] = lse_nat;
      }
    }
    for (int jg = wq; jg < GU; jg += nw) {
      const int w0 = (jg / G) * C::WPH, g = jg % G;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < C::WPH; ++w) {
        const float cf = __shfl_sync(0xffffffffu, cw[w], jg);
        const float4 v =
            reinterpret_cast<const float4 *>(wo + ((w0 + w) * 16 + g) * kD)[ln];
        acc.x = fmaf(cf, v.x, acc.x);
        acc.y = fmaf(cf, v.y, acc.y);
        acc.z = fmaf(cf, v.z, acc.z);
        acc.w = fmaf(cf, v.w, acc.w);
      }
      if (whole) {
        uint2 packed;
        packed.x = pack_bf16x2(acc.x, acc.y);
        packed.y = pack_bf16x2(acc.z, acc.w);
        reinterpret_cast<uint2 *>(p.out + (bh0 + jg) * kD)[ln] = packed;
      } else {
        reinterpret_cast<float4 *>(p.ws_o + ((long)wslot * GU + jg) * kD)[ln] =
            acc;
      }
    }
  };

  // ======================= producer warp ==================================
  if (warp == kProducer) {
    if (lane == 0) {
      prefetch_tmap(&mp.tmk);
      prefetch_tmap(&mp.tmv);
    }
    const uint64_t policy = policy_evict_first();
    // rows per box: one block piece (a head group needs 64-token blocks)
    const int br = HP > 1 ? 64 : min(64, p.block_size);
    bool appended = false;  // fused append: the finisher's rows are written
    const int npiece = 64 / br;            // <= 4 (block_size >= 16)
    for (int base = 0; base < n; base += 32) {
      const int mine = base + lane;
      int mb = 0, mh = 0, mk = 0, mrows = 0, mtok = 0, mblk[4] = {0, 0, 0, 0};
      int mpos = -1;  // fused append: the sequence's new slot
      if (mine < n) {
        const ChunkCursor cur = cursor_at(wp, p.batch, lo + mine);
        mb = cur.b, mh = cur.h, mk = cur.k;
        if (p.pos) mpos = p.pos[mb];
        const int tok =
            seq_first(p, mb, wp.len[mb], kStageRows) + mk * kStageRows;
        mtok = tok;
        mrows = min(kStageRows, wp.len[mb] - tok);
        const int32_t *bt = p.block_table + (long)mb * p.max_blocks;
        for (int j = 0; j < npiece; ++j) {
          const int t = tok + j * br;
          if (t < tok + mrows) mblk[j] = bt[t / p.block_size];
        }
      }
      const int cnt = min(32, n - base);
      if (early && base == 0) {
        pdl_wait();
        pdl_trigger();
      }
      bool stop = false;
      for (int j = 0; j < cnt && !stop; ++j) {
        const int b = __shfl_sync(0xffffffffu, mb, j);
        const int h = __shfl_sync(0xffffffffu, mh, j);
        const int k = __shfl_sync(0xffffffffu, mk, j);
        const int rows = __shfl_sync(0xffffffffu, mrows, j);
        // position of the chunk's first row (looked up with its block ids)
        const int tok = __shfl_sync(0xffffffffu, mtok, j);
        int blk[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) blk[t] = __shfl_sync(0xffffffffu, mblk[t], j);
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
            const int pieces = (rows + br - 1) / br;  // only visible blocks
            // the query rows travel only with a unit's first chunk here (the
            // consumers read them when the unit starts)
            const bool qrows = i == 0 || k == 0;
            mbar_arrive_expect_tx(
                &full[s], 2u * HP * pieces * br * C::ROW +
                              (qrows ? (uint32_t)GU * kD * 2 : 0u));
            if (qrows)
              bulk_g2s(sq + s * C::QB, p.q + ((long)b * p.n_h + h * GU) * kD,
                       GU * kD * 2, &full[s]);
            for (int pc = 0; pc < pieces; ++pc) {
              const int t = tok + pc * br;
              int pb = blk[pc];
              if (pb < 0 || pb >= p.num_blocks) {
                report(p.err, DEVERR_BLOCK);
                pb = 0;  // read a valid block; the result is flagged as wrong
              }
              const int row = (pb * p.n_kv + h * HP) * p.block_size +
                              t % p.block_size;
#pragma unroll
              for (int bx = 0; bx < C::NBOX; ++bx) {
                const int dst = bx * C::BOX + pc * br * 128;
                tma_load_2d(sk + s * C::STAGE + dst, &mp.tmk,
                            bx * (128 / C::ES), row, &full[s], policy);
                tma_load_2d(sv + s * C::STAGE + dst, &mp.tmv,
                            bx * (128 / C::ES), row, &full[s], policy);
              }
            }
            s_issued = i + 1;
          }
        }
        stop = __shfl_sync(0xffffffffu, go, 0) == 0;
      }
      if (stop) break;
    }
    if (p.pos && !appended) named_sync(kAppendBar, 64);
    if (lane == 0) s_producer_done = 1;
    return;
  }

  // ======================= finisher warp ==================================
  if (warp == kFinisher) {
    if (p.pos) {  // fused append: the new rows this CTA's chunks hold
      append_range_rows(p, wp, HP, lo, hi, lane, early);
      named_arrive(kAppendBar, 64);
    } else if (early) {
      pdl_wait();
    }
    ChunkCursor fc = cursor_at(wp, p.batch, lo);
    int x = lo;
    for (int e = 0; x < hi; ++e) {
      const int b = fc.b, h = fc.h;
      const int ustart = wp.pre[b] + h * wp.nch[b];
      const int uend = ustart + wp.nch[b];
      const int xend = min(uend, hi);
      if (xend >= hi) break;  // the last unit
      const int sl = e % C::NSLOT;
      if (!mbar_wait(&sfull[sl], (e / C::NSLOT) & 1)) {
        if (lane == 0) report(p.err, DEVERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      write_unit(b, h, sl, lane, 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[sl]);
      x = xend;
      if (x < hi) fc = cursor_at(wp, p.batch, x);
    }
    return;
  }

  // ======================= consumer warps =================================
  if (early) pdl_wait();
  // Per thread: rows qr and qr + 8 of the 16-row tiles, columns 2 qc, 2 qc+1
  // of every 8-wide n-tile. Warp w takes kv head hj = w / WPH of the unit
  // and tokens wt0 .. wt0 + TPW - 1 of it in every chunk (NSUB tiles of 16);
  // the head's rows sit at rows 64 hj .. of every column box of a stage.
  uint32_t qa[8][4];      // query A fragments, 8 k-steps of 16
  float o[16][4];         // O accumulators, 16 n-tiles of 8 columns
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  int cur_b = -1, cur_h = -1, n_flush = 0;
  float sl2 = 0.f;        // scale of S into log2 units
  const int hj = warp / C::WPH;
  const int wt0 = (warp % C::WPH) * C::TPW;  // this warp's first token
  const uint32_t sk0 = smem_u32(sk) + hj * 64 * 128;
  const uint32_t sv0 = smem_u32(sv) + hj * 64 * 128;

  auto start_unit = [&](int s, int h) {
    const uint32_t *q32 = reinterpret_cast<const uint32_t *>(
        sq + s * C::QB + hj * G * kD * 2);
    const bool r0 = qr < G, r1 = qr + 8 < G;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      if constexpr (DT == DT_BF16) {
        // A[r][16kk + 2qc .. +1], rows r, r+8; then columns + 8
        const int w0 = (16 * kk + 2 * qc) / 2;
        qa[kk][0] = r0 ? q32[qr * (kD / 2) + w0] : 0u;
        qa[kk][1] = r1 ? q32[(qr + 8) * (kD / 2) + w0] : 0u;
        qa[kk][2] = r0 ? q32[qr * (kD / 2) + w0 + 4] : 0u;
        qa[kk][3] = r1 ? q32[(qr + 8) * (kD / 2) + w0 + 4] : 0u;
      } else {
        // permuted k order: (2qc, 2qc+1) <- d 4qc, 4qc+1; (+8, +9) <- 4qc+2, +3
        const int w0 = (16 * kk + 4 * qc) / 2;
        qa[kk][0] = r0 ? f16pair_from_bf16(q32[qr * (kD / 2) + w0]) : 0u;
        qa[kk][1] = r1 ? f16pair_from_bf16(q32[(qr + 8) * (kD / 2) + w0]) : 0u;
        qa[kk][2] = r0 ? f16pair_from_bf16(q32[qr * (kD / 2) + w0 + 1]) : 0u;
        qa[kk][3] = r1 ? f16pair_from_bf16(q32[(qr + 8) * (kD / 2) + w0 + 1]) : 0u;
      }
    }
    sl2 = p.scale_log2 * (DT == DT_FP8 ? p.k_scale[h * HP + hj] : 1.0f);
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) o[nt][j] = 0.f;
  };

  auto flush = [&](bool last) {
    // full row sums across the quad
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const int sl = n_flush % C::NSLOT;
    if (n_flush >= C::NSLOT) {
      bool ok = !s_abort &&
                mbar_wait(&sempty[sl], (n_flush / C::NSLOT - 1) & 1);
      if (!__all_sync(0xffffffffu, ok) && lane == 0) {
        if (!s_abort) report(p.err, DEVERR_TIMEOUT);
        s_abort = 1;
      }
    }
    float *wm = slots + sl * C::SLOT;
    float *wl = wm + kWarps * 16;
    float *wo = wl + kWarps * 16;
    if (qc == 0) {
      wm[warp * 16 + qr] = m0;
      wm[warp * 16 + qr + 8] = m1;
      wl[warp * 16 + qr] = l0;
      wl[warp * 16 + qr + 8] = l1;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int row = qr + (j >= 2 ? 8 : 0);
        wo[(warp * 16 + row) * kD + out_col<DT>(nt, qc, j)] = o[nt][j];
      }
    }
    __syncwarp();
    if (lane == 0 && !last) mbar_arrive(&sfull[sl]);
    ++n_flush;
  };

  ChunkCursor cc = cursor_at(wp, p.batch, lo);
  for (int i = 0; i < n; ++i) {
    const int s = i % C::NS;
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
    // before the sliding window (first chunk only; cached rows, masked),
    // from nvalid on positions past the visible length
    const bool win = has_window(p);
    const int ctok =
        (win ? seq_first(p, cc.b, wp.len[cc.b], kStageRows) : 0) +
        cc.k * kStageRows;
    const int nvalid = min(kStageRows, wp.len[cc.b] - ctok);
    const int nlo = win ? seq_lo(p, cc.b, wp.len[cc.b]) - ctok : 0;
    if (ok) {
      const uint32_t kb = sk0 + s * C::STAGE;
      const uint32_t vb = sv0 + s * C::STAGE;
      if (nvalid < wt0 + C::TPW) {
        // rows past the sequence hold stale or unread data: zero this
        // warp's invalid V rows so that 0 * garbage cannot make a NaN
        for (int r = max(nvalid, wt0) + (lane >> 3); r < wt0 + C::TPW; r += 4)
          for (int bx = 0; bx < C::NBOX; ++bx)
            *reinterpret_cast<uint4 *>(sv + s * C::STAGE + bx * C::BOX +
                                       (hj * 64 + r) * 128 + (lane & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        __syncwarp();
      }
      // ---- S = Q K^T for tokens wt0 .. wt0 + TPW - 1 ----
      float sc[C::NSUB][2][4];
#pragma unroll
      for (int u = 0; u < C::NSUB; ++u)
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
          for (int j = 0; j < 4; ++j) sc[u][t2][j] = 0.f;
#pragma unroll
      for (int u = 0; u < C::NSUB; ++u) {
        const int ws = wt0 + 16 * u;
        const int mtx = lane >> 3, ri = lane & 7;
        if constexpr (DT == DT_BF16) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int tok = ws + (mtx >> 1) * 8 + ri;
            const int d = 16 * kk + (mtx & 1) * 8;
            uint32_t bk[4];
            ldsm_x4(bk, swz(kb + (d >> 6) * C::BOX, tok, (d & 63) * 2));
            mma_bf16(sc[u][0], qa[kk], bk[0], bk[1]);
            mma_bf16(sc[u][1], qa[kk], bk[2], bk[3]);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; kk += 2) {
            const int tok = ws + (mtx & 1) * 8 + ri;
            const int ks = kk + (mtx >> 1);
            uint32_t bk[4];
            ldsm_x4(bk, swz(kb, tok, ks * 16));
            // bk[m]: 4 codes of token row, dims 16 ks + 4 qc .. + 3
            mma_f16(sc[u][0], qa[kk], e4m3x2_to_f16x2(bk[0] & 0xffff),
                    e4m3x2_to_f16x2(bk[0] >> 16));
            mma_f16(sc[u][1], qa[kk], e4m3x2_to_f16x2(bk[1] & 0xffff),
                    e4m3x2_to_f16x2(bk[1] >> 16));
            mma_f16(sc[u][0], qa[kk + 1], e4m3x2_to_f16x2(bk[2] & 0xffff),
                    e4m3x2_to_f16x2(bk[2] >> 16));
            mma_f16(sc[u][1], qa[kk + 1], e4m3x2_to_f16x2(bk[3] & 0xffff),
                    e4m3x2_to_f16x2(bk[3] >> 16));
          }
        }
      }
      // ---- online softmax over the warp's tokens, rows qr and qr + 8 ----
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int u = 0; u < C::NSUB; ++u) {
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int col = wt0 + 16 * u + 8 * t2 + 2 * qc + (j & 1);
            sc[u][t2][j] =
                col >= nlo && col < nvalid ? sc[u][t2][j] * sl2 : -INFINITY;
          }
          mx0 = fmaxf(mx0, fmaxf(sc[u][t2][0], sc[u][t2][1]));
          mx1 = fmaxf(mx1, fmaxf(sc[u][t2][2], sc[u][t2][3]));
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float u0 = n0 == -INFINITY ? 0.f : n0;
      const float u1 = n1 == -INFINITY ? 0.f : n1;
      const float c0 = ex2(m0 - u0), c1 = ex2(m1 - u1);
      m0 = n0;
      m1 = n1;
      uint32_t pa[C::NSUB][4];
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int u = 0; u < C::NSUB; ++u) {
        float pp[2][4];
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          pp[t2][0] = ex2(sc[u][t2][0] - u0);
          pp[t2][1] = ex2(sc[u][t2][1] - u0);
          pp[t2][2] = ex2(sc[u][t2][2] - u1);
          pp[t2][3] = ex2(sc[u][t2][3] - u1);
          ls0 += pp[t2][0] + pp[t2][1];
          ls1 += pp[t2][2] + pp[t2][3];
        }
        if constexpr (DT == DT_BF16) {
          pa[u][0] = pack_bf16x2(pp[0][0], pp[0][1]);
          pa[u][1] = pack_bf16x2(pp[0][2], pp[0][3]);
          pa[u][2] = pack_bf16x2(pp[1][0], pp[1][1]);
          pa[u][3] = pack_bf16x2(pp[1][2], pp[1][3]);
        } else {
          pa[u][0] = pack_f16x2(pp[0][0], pp[0][1]);
          pa[u][1] = pack_f16x2(pp[0][2], pp[0][3]);
          pa[u][2] = pack_f16x2(pp[1][0], pp[1][1]);
          pa[u][3] = pack_f16x2(pp[1][2], pp[1][3]);
        }
      }
      l0 = l0 * c0 + ls0;
      l1 = l1 * c1 + ls1;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] *= c0;
        o[nt][1] *= c0;
        o[nt][2] *= c1;
        o[nt][3] *= c1;
      }
      // ---- O += P V ----
#pragma unroll
      for (int u = 0; u < C::NSUB; ++u) {
        const int mtx = lane >> 3, ri = lane & 7;
        const int tok = wt0 + 16 * u + (mtx & 1) * 8 + ri;
        if constexpr (DT == DT_BF16) {
#pragma unroll
          for (int np = 0; np < 8; ++np) {
            const int d = 8 * (2 * np + (mtx >> 1));
            uint32_t bv[4];
            ldsm_x4_t(bv, swz(vb + (d >> 6) * C::BOX, tok, (d & 63) * 2));
            mma_bf16(o[2 * np], pa[u], bv[0], bv[1]);
            mma_bf16(o[2 * np + 1], pa[u], bv[2], bv[3]);
          }
        } else {
#pragma unroll
          for (int dp = 0; dp < 4; ++dp) {
            const int g16 = 2 * dp + (mtx >> 1);  // 16-wide column group
            uint32_t bv[4];
            ldsm_x4_t(bv, swz(vb, tok, g16 * 16));
            // bv[m] bytes: (V[2qc][2qr], V[2qc][2qr+1], V[2qc+1][2qr],
            // V[2qc+1][2qr+1]) of the matrix's token half and column group
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const uint32_t lo_t = bv[2 * h2], hi_t = bv[2 * h2 + 1];
              const int gg = 2 * dp + h2;
              mma_f16(o[2 * gg], pa[u],
                      e4m3x2_to_f16x2((uint16_t)prmt(lo_t, 0, 0x0020)),
                      e4m3x2_to_f16x2((uint16_t)prmt(hi_t, 0, 0x0020)));
              mma_f16(o[2 * gg + 1], pa[u],
                      e4m3x2_to_f16x2((uint16_t)prmt(lo_t, 0, 0x0031)),
                      e4m3x2_to_f16x2((uint16_t)prmt(hi_t, 0, 0x0031)));
            }
          }
        }
      }
      if (nvalid < wt0 + C::TPW) fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    cursor_next(wp, p.batch, n_units, cc);
  }
  if (cur_b >= 0) {
    flush(true);
    named_sync(kFinalBar, kConsumers);  // every warp's state is in the slot
    write_unit(cur_b, cur_h, (n_flush - 1) % C::NSLOT, tid, kConsumers);
  }

  if (s_abort && tid == 0) {
    for (int t = 0; t < (1 << 20) && !s_producer_done; ++t) __nanosleep(1000);
    const int issued = s_issued;
    for (int st = 0; st < C::NS; ++st) {
      int last = -1;
      for (int c2 = st; c2 < issued; c2 += C::NS) last = c2;
      if (last >= 0) mbar_wait(&full[st], (last / C::NS) & 1);
    }
  }
}

// ---------------------------------------------------------------------------
// host side: tensor maps
// ---------------------------------------------------------------------------

// The cache as a 2-D tensor [num_blocks * n_kv * block_size][head_dim],
// copied in boxes of 128-byte rows x `box_rows` rows, 128-byte swizzle.
cudaError_t make_map(CUtensorMap *m, const void *base, long rows, bool fp8,
                     int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * (fp8 ? 1 : 2)};
  const cuuint32_t box[2] = {(cuuint32_t)(fp8 ? 128 : 64), (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = tensor_map_encoder()(
      m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
      2, const_cast<void *>(base), dims, strides, box, estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int DT, int HP>
cudaError_t launch_t(const MmaParams &mp, cudaStream_t s) {
  using C = MCfg<DT, HP>;
  static_assert(C::SMEM <= 226 * 1024, "shared memory budget");
  static_assert(C::NS >= 2, "ring depth");
  auto kern = decode_mma_kernel<DT, HP>;
  static bool done[64] = {};
  cudaError_t e = set_smem_once(kern, C::SMEM, done);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(mp.p.n_splits), dim3(kThreads), C::SMEM, s, 1, mp);
  if (e != cudaSuccess) return e;
  const int gu = HP * (mp.p.n_h / mp.p.n_kv);  // query heads per unit
  const int units = mp.p.n_kv / HP;
  return gu == 32   ? launch_merge_dense<kD, 32>(mp.p, units, s)
         : gu == 16 ? launch_merge_dense<kD, 16>(mp.p, units, s)
                    : launch_merge_dense<kD, 8>(mp.p, units, s);
}

}  // namespace

// Head groups of 2 for the fp8 cache (its 8 KB per head and block is too
// small a copy); a bf16 head's 16 KB copies stream well, and doubling them
// would leave room for only two ring stages.
int mma_heads_per_unit(int n_kv, int block_size, int dtype) {
  return dtype == DT_FP8 && block_size == 64 && n_kv % 2 == 0 ? 2 : 1;
}

cudaError_t launch_decode_mma(const DecodeParams &p, int dtype,
                              cudaStream_t s) {
  const int g = p.n_h / p.n_kv;
  if (p.dk != kD || (g != 8 && g != 16) || p.batch > kMaxDecodeBatch)
    return cudaErrorNotSupported;
  // a 64-token chunk must be whole blocks, or lie inside one block
  if (p.block_size < 16 ||
      (p.block_size % 64 != 0 && 64 % p.block_size != 0))
    return cudaErrorNotSupported;
  const long rows = (long)p.num_blocks * p.n_kv * p.block_size;
  if (rows >= (1L << 31)) return cudaErrorNotSupported;
  if (!tensor_map_encoder()) return cudaErrorNotSupported;
  cudaError_t e;
  MmaParams mp;
  mp.p = p;
  const bool fp8 = dtype == DT_FP8;
  if (p.hp != 1 && p.hp != mma_heads_per_unit(p.n_kv, p.block_size, dtype))
    return cudaErrorNotSupported;
  // a box is one block piece of one head, or the hp heads' rows of a block
  const int box_rows =
      p.hp > 1 ? p.hp * 64 : (p.block_size < 64 ? p.block_size : 64);
  e = make_map(&mp.tmk, p.k, rows, fp8, box_rows);
  if (e != cudaSuccess) return e;
  e = make_map(&mp.tmv, p.v, rows, fp8, box_rows);
  if (e != cudaSuccess) return e;
  if (p.hp == 2)
    return fp8 ? launch_t<DT_FP8, 2>(mp, s) : launch_t<DT_BF16, 2>(mp, s);
  return fp8 ? launch_t<DT_FP8, 1>(mp, s) : launch_t<DT_BF16, 1>(mp, s);
}

}  // namespace kvd

// Decode attention for 64-head query tiles against wide cached rows, on the
// tensor cores (warp-level m16n8k16 MMA, fp32 accumulators):
//
//  * latent (MLA) decode ("KV cache", "Caching a compressed latent instead
//    of the keys"): each cached row is [c (512) | k_rope (64)], scores are
//    q_lat . c + q_rope . k_rope over the whole 576-wide row, the values are
//    the row's first 512 elements, every position of the sequence is read;
//  * top-k sparse decode ("890 bytes a token ...", section 3; the
//    transcript on DeepSeek Sparse Attention): separate K and V rows of 512,
//    one kv head, only the positions an index list names are read.
//
// A unit is (sequence, 64-head tile); its work is cut into 32-position
// chunks and spread over a persistent launch by the stream-K partition of
// stream_k.cuh. A producer warp fetches a chunk with one bulk copy per row
// and lane (the positions of a chunk need not be contiguous: paged blocks,
// or index-selected positions) into rows padded by 16 bytes, which keeps
// every 8-row ldmatrix read free of bank conflicts. Sixteen consumer warps
// form 4 groups (16 query heads each) x 4 quarters of the value width: per
// chunk each warp of a group computes S = Q K^T for 8 of the 32 positions
// over the full key width, the group exchanges row maxima and the
// probabilities P (rounded to bf16) through shared memory, and each warp
// accumulates O += P V for its quarter of the value columns. So no product
// is computed twice. At a unit boundary the row sums are combined, and the
// unit is written out, or as a partial merged by the last covering CTA
// (log-sum-exp merge).
#include <cmath>

#include "kvd_common.cuh"
#include "stream_k.cuh"

namespace kvd {
namespace {

constexpr int kHeads = 64;                // query heads per unit
constexpr int kRows = 32;                 // positions per chunk
constexpr int kGroups = 4;                // 16-head row tiles
constexpr int kQuarters = 4;              // value-column quarters
constexpr int kCWarps = kGroups * kQuarters;
constexpr int kConsumers = kCWarps * 32;  // 512
constexpr int kThreads = kConsumers + 32; // + producer warp
constexpr int kAllBar = 1;                // all consumer warps
constexpr int kNB = 256;                  // largest batch of these calls

template <int DK, int DV, bool GATHER>
struct WCfg {
  static constexpr bool VFROMK = !GATHER;  // latent rows: V = K[:, :DV]
  static constexpr int KROW = DK * 2 + 16;  // padded bytes per K row
  static constexpr int VROW = DV * 2 + 16;
  static constexpr int KST = kRows * KROW;
  static constexpr int VST = VFROMK ? 0 : kRows * VROW;
  static constexpr int NS = VFROMK ? 3 : 2;
  static constexpr int QROW = DK * 2 + 16;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = kHeads * QROW;
  static constexpr int V_OFF = K_OFF + NS * KST;
  static constexpr int PROW = kRows * 2 + 16;  // padded P row (bf16)
  static constexpr int P_OFF = V_OFF + NS * VST;
  static constexpr int RED_OFF = P_OFF + kGroups * 16 * PROW;
  static constexpr int WP_OFF = RED_OFF + 2 * kCWarps * 16 * 4;
  static constexpr int BAR_OFF =
      (WP_OFF + (int)sizeof(WorkPartitionT<kNB>) + 15) / 16 * 16;
  static constexpr int SMEM = BAR_OFF + (2 * NS + 1) * 8;
  static constexpr int DVQ = DV / kQuarters;  // value columns per warp (128)
};

template <int DK, int DV, bool GATHER>
__global__ void __launch_bounds__(kThreads, 1)
    decode_wide_kernel(const DecodeParams p) {
  using C = WCfg<DK, DV, GATHER>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *sq = smem + C::Q_OFF;
  uint8_t *sk = smem + C::K_OFF;
  uint8_t *sv = smem + C::V_OFF;
  uint8_t *spv = smem + C::P_OFF;
  float *red = reinterpret_cast<float *>(smem + C::RED_OFF);  // row maxima
  float *lsum = red + kCWarps * 16;                            // row sums
  WorkPartitionT<kNB> &wp =
      *reinterpret_cast<WorkPartitionT<kNB> *>(smem + C::WP_OFF);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *empty = full + C::NS;
  uint64_t *qbar = empty + C::NS;
  __shared__ int s_len_err;
  __shared__ int s_merge[2];
  __shared__ volatile int s_abort, s_issued, s_producer_done;
  __shared__ unsigned s_valid[C::NS];  // rows of each stage that were fetched

  const int tiles = p.n_h / kHeads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qr = lane >> 2, qc = lane & 3;

  if (tid == 0) {
    s_len_err = 0;
    s_abort = 0;
    s_issued = 0;
    s_producer_done = 0;
    s_merge[0] = s_merge[1] = -1;
  }
  __syncthreads();
  build_partition(wp, p, &s_len_err, kRows, tiles, GATHER ? p.n_idx : 0);
  if (tid == 0 && blockIdx.x == 0 && s_len_err) report(p.err, DEVERR_LEN);
  const int total = wp.total;
  const int P = min((int)gridDim.x, max(total, 1));
  const int c = blockIdx.x;

  if (c == 0) {  // sequences with nothing visible: out = 0, lse = -inf
    for (int b = 0; b < p.batch; ++b) {
      if (wp.nch[b] != 0) continue;
      for (int i = tid; i < p.n_h * DV; i += kThreads)
        p.out[(long)b * p.n_h * DV + i] = 0;
      if (p.lse)
        for (int i = tid; i < p.n_h; i += kThreads)
          p.lse[(long)b * p.n_h + i] = -INFINITY;
    }
  }
  if (c >= P || total == 0) return;
  const int lo = range_lo(c, total, P);
  const int hi = range_lo(c + 1, total, P);
  const int n = hi - lo;

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCWarps);
    }
    mbar_init(qbar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ======================= producer warp ==================================
  // Lane r fetches row r of each chunk: its position (chunk start + r, or
  // the r-th entry of the chunk's slice of the index list), its block, and
  // one bulk copy per cached tensor.
  if (warp == kCWarps) {
    ChunkCursor pc = cursor_at(wp, p.batch, lo);
    for (int i = 0; i < n; ++i) {
      const int s = i % C::NS;
      int go = 1;
      if (i >= C::NS && !mbar_wait(&empty[s], (i / C::NS - 1) & 1)) go = 0;
      go = __shfl_sync(0xffffffffu, go, 0) && !s_abort;
      if (!go) {
        if (lane == 0) report(p.err, DEVERR_TIMEOUT);
        break;
      }
      const int T = wp.len[pc.b];
      const int e = pc.k * kRows + lane;  // entry of this lane's row
      int t;
      if constexpr (GATHER) {
        t = e < p.n_idx ? p.indices[(long)pc.b * p.n_idx + e] : -1;
        if (t >= T) {
          report(p.err, DEVERR_INDEX);
          t = -1;
        }
      } else {
        t = e < T ? e : -1;
      }
      int blk = -1;
      if (t >= 0) {
        blk = p.block_table[(long)pc.b * p.max_blocks + t / p.block_size];
        if (blk < 0 || blk >= p.num_blocks) {
          report(p.err, DEVERR_BLOCK);
          blk = 0;  // read a valid block; the result is flagged as wrong
        }
      }
      const unsigned valid = __ballot_sync(0xffffffffu, t >= 0);
      if (t < 0) {
        // a row that is not fetched keeps stale data: zero the value part,
        // so that its zero probability cannot meet a NaN in P V
        uint4 *vz = reinterpret_cast<uint4 *>(
            C::VFROMK ? sk + s * C::KST + lane * C::KROW
                      : sv + s * C::VST + lane * C::VROW);
        for (int j = 0; j < DV * 2 / 16; ++j) vz[j] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        s_valid[s] = valid;
        mbar_arrive_expect_tx(&full[s], __popc(valid) *
                                            (DK * 2 + (C::VFROMK ? 0 : DV * 2)));
      }
      __syncwarp();
      if (t >= 0) {
        const size_t row =
            ((size_t)blk * p.n_kv) * p.block_size + t % p.block_size;
        bulk_g2s(sk + s * C::KST + lane * C::KROW, p.k + row * DK * 2, DK * 2,
                 &full[s]);
        if constexpr (!C::VFROMK)
          bulk_g2s(sv + s * C::VST + lane * C::VROW, p.v + row * DV * 2,
                   DV * 2, &full[s]);
      }
      if (lane == 0) s_issued = i + 1;
      cursor_next(wp, p.batch, tiles, pc);
    }
    if (lane == 0) s_producer_done = 1;
    return;
  }

  // ======================= consumer warps =================================
  const int grp = warp >> 2;   // 16-head row tile
  const int qtr = warp & 3;    // value quarter / token slice of the group
  const uint32_t q0 = smem_u32(sq), k0 = smem_u32(sk), v0 = smem_u32(sv);
  const uint32_t p0 = smem_u32(spv) + grp * 16 * C::PROW;
  float o[C::DVQ / 8][4];      // O: 16 rows x DVQ columns
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  int cur_b = -1, cur_h = -1, n_units = 0;
  int pend_prev[2] = {-1, -1}, pend_start[2] = {0, 0}, n_pend = 0;

  auto start_unit = [&](int b, int h) {
    // the query tile of (b, head tile h): 64 rows, one bulk copy each
    named_sync(kAllBar, kConsumers);  // nobody still reads the old tile
    if (warp == 0) {
      if (lane == 0) mbar_arrive_expect_tx(qbar, kHeads * DK * 2);
      __syncwarp();
      for (int r = lane; r < kHeads; r += 32)
        bulk_g2s(sq + r * C::QROW,
                 p.q + ((long)b * p.n_h + (long)h * kHeads + r) * DK,
                 DK * 2, qbar);
    }
    if (!mbar_wait(qbar, n_units & 1) && lane == 0) {
      report(p.err, DEVERR_TIMEOUT);
      s_abort = 1;
    }
    ++n_units;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < C::DVQ / 8; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) o[nt][j] = 0.f;
  };

  auto flush = [&](int b, int h) {
    // row sums over the group's four token slices
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (qc == 0) {
      lsum[warp * 16 + qr] = l0;
      lsum[warp * 16 + qr + 8] = l1;
    }
    named_sync(kAllBar, kConsumers);
    float L0 = 0.f, L1 = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      L0 += lsum[(grp * 4 + w) * 16 + qr];
      L1 += lsum[(grp * 4 + w) * 16 + qr + 8];
    }
    const int ustart = wp.pre[b] + h * wp.nch[b];
    const int uend = ustart + wp.nch[b];
    const bool whole = ustart >= lo && uend <= hi;
    const int wslot = c * 2 + partial_side(ustart, lo);
    const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
    const int row0 = grp * 16 + qr, row1 = row0 + 8;  // head within the tile
    const float lse0 = L0 > 0.f ? (m0 + log2f(L0)) * 0.69314718055994531f
                                : -INFINITY;
    const float lse1 = L1 > 0.f ? (m1 + log2f(L1)) * 0.69314718055994531f
                                : -INFINITY;
    const long bh0 = (long)b * p.n_h + (long)h * kHeads;
#pragma unroll
    for (int nt = 0; nt < C::DVQ / 8; ++nt) {
      const int col = qtr * C::DVQ + nt * 8 + 2 * qc;
      if (whole) {
        *reinterpret_cast<uint32_t *>(p.out + (bh0 + row0) * DV + col) =
            pack_bf16x2(o[nt][0] * inv0, o[nt][1] * inv0);
        *reinterpret_cast<uint32_t *>(p.out + (bh0 + row1) * DV + col) =
            pack_bf16x2(o[nt][2] * inv1, o[nt][3] * inv1);
      } else {
        float *dst = p.ws_o + ((long)wslot * kHeads) * DV;
        *reinterpret_cast<float2 *>(dst + (long)row0 * DV + col) =
            make_float2(o[nt][0] * inv0, o[nt][1] * inv0);
        *reinterpret_cast<float2 *>(dst + (long)row1 * DV + col) =
            make_float2(o[nt][2] * inv1, o[nt][3] * inv1);
      }
    }
    if (qtr == 0 && qc == 0) {
      if (whole) {
        if (p.lse) {
          p.lse[bh0 + row0] = lse0;
          p.lse[bh0 + row1] = lse1;
        }
      } else {
        p.ws_lse[(long)wslot * kHeads + row0] = lse0;
        p.ws_lse[(long)wslot * kHeads + row1] = lse1;
      }
    }
    if (!whole) __threadfence();
    named_sync(kAllBar, kConsumers);  // partials written; lsum reusable
    if (!whole && tid == 0) {
      pend_prev[n_pend] = arrive_release(p.counters + (long)b * tiles + h);
      pend_start[n_pend] = ustart;
      ++n_pend;
    }
  };

  ChunkCursor cc = cursor_at(wp, p.batch, lo);
  const float sl2 = p.scale_log2;
  for (int i = 0; i < n; ++i) {
    const int s = i % C::NS;
    if (cc.b != cur_b || cc.h != cur_h) {
      if (cur_b >= 0) flush(cur_b, cur_h);
      cur_b = cc.b;
      cur_h = cc.h;
      start_unit(cur_b, cur_h);
    }
    bool ok = !s_abort && mbar_wait(&full[s], (i / C::NS) & 1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) {
      if (!s_abort) report(p.err, DEVERR_TIMEOUT);
      s_abort = 1;
    }
    // validity of this warp's S columns: rows qtr * 8 + 2 qc (+1)
    const unsigned vmask = s_valid[s];
    const bool val0 = (vmask >> (qtr * 8 + 2 * qc)) & 1;
    const bool val1 = (vmask >> (qtr * 8 + 2 * qc + 1)) & 1;
    const uint32_t kst = k0 + s * C::KST;
    const uint32_t vst = (C::VFROMK ? k0 + s * C::KST : v0 + s * C::VST);
    // ---- S = Q K^T: rows = this group's 16 heads, cols = 8 positions ----
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
      const int mtx = lane >> 3, ri = lane & 7;
      // A (query) rows grp*16 + (mtx & 1)*8 + ri, k half (mtx >> 1)
      const uint32_t qa_base =
          q0 + (grp * 16 + (mtx & 1) * 8 + ri) * C::QROW + (mtx >> 1) * 16;
      // B (keys): positions qtr*8 + ri, two k-steps per x4 (k halves)
      const uint32_t kb_base = kst + (qtr * 8 + ri) * C::KROW + mtx * 16;
#pragma unroll 4
      for (int ks = 0; ks < DK / 16; ks += 2) {
        uint32_t a0[4], a1[4], bk[4];
        ldsm_x4(a0, qa_base + ks * 32);
        ldsm_x4(a1, qa_base + (ks + 1) * 32);
        ldsm_x4(bk, kb_base + ks * 32);
        mma_bf16(sa, a0, bk[0], bk[1]);
        mma_bf16(sb, a1, bk[2], bk[3]);
      }
    }
    float sc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) sc[j] = (sa[j] + sb[j]) * sl2;
    if (!val0) sc[0] = sc[2] = -INFINITY;
    if (!val1) sc[1] = sc[3] = -INFINITY;
    // ---- row maxima across the group's four slices ----
    float mx0 = fmaxf(sc[0], sc[1]), mx1 = fmaxf(sc[2], sc[3]);
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    if (qc == 0) {
      red[warp * 16 + qr] = mx0;
      red[warp * 16 + qr + 8] = mx1;
    }
    named_sync(2 + grp, 128);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      mx0 = fmaxf(mx0, red[(grp * 4 + w) * 16 + qr]);
      mx1 = fmaxf(mx1, red[(grp * 4 + w) * 16 + qr + 8]);
    }
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float u0 = n0 == -INFINITY ? 0.f : n0;
    const float u1 = n1 == -INFINITY ? 0.f : n1;
    const float c0 = ex2(m0 - u0), c1 = ex2(m1 - u1);
    m0 = n0;
    m1 = n1;
    const float p00 = ex2(sc[0] - u0), p01 = ex2(sc[1] - u0);
    const float p10 = ex2(sc[2] - u1), p11 = ex2(sc[3] - u1);
    l0 = l0 * c0 + p00 + p01;
    l1 = l1 * c1 + p10 + p11;
    // P of this warp's 8 positions into the group's [16][32] tile
    {
      uint8_t *prow = spv + grp * 16 * C::PROW;
      *reinterpret_cast<uint32_t *>(prow + qr * C::PROW + (qtr * 8 + 2 * qc) * 2) =
          pack_bf16x2(p00, p01);
      *reinterpret_cast<uint32_t *>(prow + (qr + 8) * C::PROW +
                                    (qtr * 8 + 2 * qc) * 2) =
          pack_bf16x2(p10, p11);
    }
#pragma unroll
    for (int nt = 0; nt < C::DVQ / 8; ++nt) {
      o[nt][0] *= c0;
      o[nt][1] *= c0;
      o[nt][2] *= c1;
      o[nt][3] *= c1;
    }
    named_sync(2 + grp, 128);
    // ---- O += P V for this warp's value quarter ----
    if (ok) {
      const int mtx = lane >> 3, ri = lane & 7;
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {  // 16 positions per k-step
        uint32_t pa[4];
        ldsm_x4(pa, p0 + ((mtx & 1) * 8 + ri) * C::PROW + (kt * 16 + (mtx >> 1) * 8) * 2);
        // positions rows of V: kt*16 + (mtx & 1)*8 + ri; columns pairs
        const uint32_t vrow =
            vst + (kt * 16 + (mtx & 1) * 8 + ri) *
                      (C::VFROMK ? C::KROW : C::VROW) +
            qtr * C::DVQ * 2;
        // rows of unfetched positions were zeroed by the producer
#pragma unroll
        for (int np = 0; np < C::DVQ / 16; ++np) {
          uint32_t bv[4];
          ldsm_x4_t(bv, vrow + (2 * np + (mtx >> 1)) * 16);
          mma_bf16(o[2 * np], pa, bv[0], bv[1]);
          mma_bf16(o[2 * np + 1], pa, bv[2], bv[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    cursor_next(wp, p.batch, tiles, cc);
  }
  if (cur_b >= 0) flush(cur_b, cur_h);

  // ---- merges this CTA owes (it arrived last on the unit's counter) ----
  if (tid == 0) {
    for (int j = 0; j < n_pend; ++j) {
      const int ustart = pend_start[j];
      const int bb = find_seq(wp, p.batch, ustart);
      const int hh = (ustart - wp.pre[bb]) / wp.nch[bb];
      const int uend = ustart + wp.nch[bb];
      const int parts = cta_of(uend - 1, total, P) - cta_of(ustart, total, P) + 1;
      if (pend_prev[j] == parts - 1) {
        s_merge[j] = ustart;
        atomicExch(p.counters + (long)bb * tiles + hh, 0);
      }
    }
    __threadfence();
  }
  named_sync(kAllBar, kConsumers);
  merge_owed<DV, kHeads>(p, wp, s_merge,
                         reinterpret_cast<float *>(smem + C::K_OFF),
                         (C::NS * C::KST) / 4, total, P, tid, kConsumers,
                         kAllBar);

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

template <int DK, int DV, bool GATHER>
cudaError_t launch_t(const DecodeParams &p, cudaStream_t s) {
  using C = WCfg<DK, DV, GATHER>;
  static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
  auto kern = decode_wide_kernel<DK, DV, GATHER>;
  static bool done[64] = {};
  cudaError_t e = set_smem_once(kern, C::SMEM, done);
  if (e != cudaSuccess) return e;
  kern<<<p.n_splits, kThreads, C::SMEM, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_mla(const DecodeParams &p, cudaStream_t s) {
  if (p.dk != 576 || p.dv != 512 || p.n_h % kHeads != 0 || p.batch > kNB)
    return cudaErrorNotSupported;
  return launch_t<576, 512, false>(p, s);
}

cudaError_t launch_decode_sparse(const DecodeParams &p, cudaStream_t s) {
  if (p.dk != 512 || p.dv != 512 || p.n_h % kHeads != 0 || p.batch > kNB ||
      p.n_kv != 1)
    return cudaErrorNotSupported;
  return launch_t<512, 512, true>(p, s);
}

}  // namespace kvd

// Latent (MLA) decode for 64-head query tiles against wide cached rows, on
// the tensor cores (warp-level m16n8k16 MMA, fp32 accumulators), for the
// shapes the tcgen05 latent kernel does not take ("KV cache", "Caching a
// compressed latent instead of the keys"): each cached row is [c (512) |
// k_rope (64)], scores are q_lat . c + q_rope . k_rope over the whole
// 576-wide row, the values are the row's first 512 elements, every position
// of the sequence is read.
//
// A unit is (sequence, 64-head tile); its work is cut into 32-position
// chunks. The stream-K partition of stream_k.cuh spreads the chunks of all
// sequences over gridDim / tiles CTA "lanes", and the `tiles` neighbouring
// CTAs of a lane take the same chunk range, one head tile each: they stream
// the same rows at about the same time, so a row read for one tile is
// still in L2 for the others and HBM delivers it once. A producer warp fetches a chunk with one bulk copy per row
// and lane (the positions of a chunk need not be contiguous: paged blocks)
// into rows padded by 16 bytes, which keeps
// every 8-row ldmatrix read free of bank conflicts. Sixteen consumer warps
// share the products, with tiles as large as the registers allow (the
// kernel is bound by its ldmatrix traffic): for S = Q K^T a pair of warps
// takes a 16-head x 16-position tile, each warp half of the key width, the
// second handing its partial tile to the first; for O += P V a warp takes
// 32 heads x 64 value columns. Row maxima, P (rounded to bf16) and the
// per-head rescale factors go through shared memory. So no product is
// computed twice. At a unit boundary the row sums are combined, and the
// unit is written out, or as a partial. The partials of a unit cut between
// CTAs (64 heads x 512 values each, so a unit cut 19 ways holds 2.4 MB) are
// merged by a second, wide launch: one CTA per (unit, 1/32 of the unit's
// outputs), each running an online log-sum-exp merge over the parts with
// independent loads in flight, so no single SM reads a whole unit.
#include <cmath>

#include "kvd_common.cuh"
#include "stream_k.cuh"

namespace kvd {
namespace {

constexpr int kHeads = 64;                // query heads per unit
constexpr int kRows = 32;                 // positions per chunk
constexpr int kCWarps = 16;               // consumer warps
constexpr int kConsumers = kCWarps * 32;  // 512
// Four producer warps, each fetching 8 rows of every chunk: a warp issues
// its bulk copies one lane after another (about 50 ns a copy), so one warp
// copying 32 or 64 short rows per chunk was the kernel's limit.
constexpr int kPW = 4;                    // producer warps
constexpr int kPRows = kRows / kPW;       // rows per producer warp
constexpr int kThreads = kConsumers + 32 * kPW;
constexpr int kAllBar = 1;                // all consumer warps
constexpr int kNB = 256;                  // largest batch of these calls

// Latent rows: the values are the first DV columns of the K row.
template <int DK, int DV>
struct WCfg {
  static constexpr int KROW = DK * 2 + 16;  // padded bytes per K row
  static constexpr int KST = kRows * KROW;
  static constexpr int NS = 3;
  static constexpr int QROW = DK * 2 + 16;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = kHeads * QROW;
  static constexpr int PROW = kRows * 2 + 16;  // padded P row (bf16)
  static constexpr int P_OFF = K_OFF + NS * KST;   // P, two chunk buffers
  static constexpr int PBUF = kHeads * PROW;
  static constexpr int SP_OFF = P_OFF + 2 * PBUF;  // K-split partial S tiles
  static constexpr int RED_OFF = SP_OFF + 8 * 32 * 8 * 4;
  // row maxima [8 tiles][16]; rescale factors [2][64]; flush: row sums
  // [2][64] and maxima [64]
  static constexpr int WP_OFF = RED_OFF + (8 * 16 + 2 * 64 + 3 * 64) * 4;
  static constexpr int BAR_OFF =
      (WP_OFF + (int)sizeof(WorkPartitionT<kNB>) + 15) / 16 * 16;
  static constexpr int SMEM = BAR_OFF + (2 * NS + 1) * 8;
};

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    decode_wide_kernel(const DecodeParams p) {
  using C = WCfg<DK, DV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *sq = smem + C::Q_OFF;
  uint8_t *sk = smem + C::K_OFF;
  uint8_t *spv = smem + C::P_OFF;
  float *spart = reinterpret_cast<float *>(smem + C::SP_OFF);
  float *red = reinterpret_cast<float *>(smem + C::RED_OFF);  // row maxima
  float *hcor = red + 8 * 16;     // [2][64] per-head rescale of O
  float *lsum = hcor + 2 * 64;    // [2][64] row sums of the two halves
  float *mfin = lsum + 2 * 64;    // [64] running maxima at a flush
  WorkPartitionT<kNB> &wp =
      *reinterpret_cast<WorkPartitionT<kNB> *>(smem + C::WP_OFF);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
  uint64_t *empty = full + C::NS;
  uint64_t *qbar = empty + C::NS;
  __shared__ int s_len_err;
  __shared__ volatile int s_abort, s_issued, s_producer_done;
  // rows of each stage that were fetched, 8 bits per producer warp
  __shared__ __align__(4) uint8_t s_vpart[C::NS][kPW];

  const int tiles = p.n_h / kHeads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_trigger();  // after the wait: see the merge launch
  const int qr = lane >> 2, qc = lane & 3;

  if (tid == 0) {
    s_len_err = 0;
    s_abort = 0;
    s_issued = 0;
    s_producer_done = 0;
  }
  __syncthreads();
  build_partition(wp, p, &s_len_err, kRows, 1);
  if (tid == 0 && blockIdx.x == 0 && s_len_err) report(p.err, DEVERR_LEN);
  const int total = wp.total;
  const int lanes = (int)gridDim.x / tiles;
  const int P = min(lanes, max(total, 1));
  const int c = (int)blockIdx.x / tiles;     // lane: a range of chunks
  const int tile = (int)blockIdx.x % tiles;  // head tile of this CTA

  if (blockIdx.x == 0) {  // sequences with nothing visible: out = 0, lse = -inf
    for (int b = 0; b < p.batch; ++b) {
      if (wp.nch[b] != 0) continue;
      for (int i = tid; i < p.n_h * DV; i += kThreads)
        p.out[(long)b * p.n_h * DV + i] = 0;
      if (p.lse)
        for (int i = tid; i < p.n_h; i += kThreads)
          p.lse[(long)b * p.n_h + i] = -INFINITY;
    }
  }
  if (c >= P || total == 0) return;  // (also CTAs beyond lanes * tiles)
  const int lo = range_lo(c, total, P);
  const int hi = range_lo(c + 1, total, P);
  const int n = hi - lo;

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], kPW);  // each producer warp's arrive + bytes
      mbar_init(&empty[s], kCWarps);
    }
    mbar_init(qbar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ======================= producer warps =================================
  // Producer warp pw takes rows 8 pw .. 8 pw + 7 of every chunk: lane r < 8
  // looks up row 8 pw + r (its position: chunk start + r, or that entry of
  // the chunk's slice of the index list; then its block), lanes 0..7 copy
  // the rows' K and, for separate values, lanes 8..15 their V -- 8 or 16
  // bulk copies per warp and chunk, issued by the four warps side by side.
  if (warp >= kCWarps) {
    const int pw = warp - kCWarps;
    const int r8 = lane & 7;            // row of the warp's eight
    const int row_in_chunk = pw * kPRows + r8;
    ChunkCursor pc = cursor_at(wp, p.batch, lo);
    // position and block of row `row_in_chunk` of the chunk at `cc`
    auto lookup = [&](const ChunkCursor &cc, int &t, int &blk) {
      const int T = wp.len[cc.b];
      const int e = cc.k * kRows + row_in_chunk;  // position of the row
      t = e < T ? e : -1;
      blk = -1;
      if (t >= 0) {
        blk = p.block_table[(long)cc.b * p.max_blocks + t / p.block_size];
        if (blk < 0 || blk >= p.num_blocks) {
          if (lane < 8) report(p.err, DEVERR_BLOCK);
          blk = 0;  // read a valid block; the result is flagged as wrong
        }
      }
    };
    int t, blk;
    lookup(pc, t, blk);
    for (int i = 0; i < n; ++i) {
      const int s = i % C::NS;
      int go = 1;
      if (i >= C::NS && !mbar_wait(&empty[s], (i / C::NS - 1) & 1)) go = 0;
      go = __shfl_sync(0xffffffffu, go, 0) && !s_abort;
      if (!go) {
        if (lane == 0) report(p.err, DEVERR_TIMEOUT);
        break;
      }
      const unsigned valid =
          __ballot_sync(0xffffffffu, lane < 8 && t >= 0) & 0xffu;
      if (lane < 8 && t < 0) {
        // a row that is not fetched keeps stale data: zero the value part,
        // so that its zero probability cannot meet a NaN in P V
        uint4 *vz = reinterpret_cast<uint4 *>(sk + s * C::KST +
                                              row_in_chunk * C::KROW);
        for (int j = 0; j < DV * 2 / 16; ++j) vz[j] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        s_vpart[s][pw] = (uint8_t)valid;
        mbar_arrive_expect_tx(&full[s], __popc(valid) * (DK * 2));
      }
      __syncwarp();
      if (t >= 0) {
        const size_t row =
            ((size_t)blk * p.n_kv) * p.block_size + t % p.block_size;
        if (lane < 8)
          bulk_g2s(sk + s * C::KST + row_in_chunk * C::KROW,
                   p.k + row * DK * 2, DK * 2, &full[s]);
      }
      if (lane == 0 && pw == 0) s_issued = i + 1;
      // the next chunk's rows are looked up now, while the ring is full
      cursor_next(wp, p.batch, 1, pc);
      if (i + 1 < n) lookup(pc, t, blk);
    }
    if (lane == 0) atomicAdd(const_cast<int *>(&s_producer_done), 1);
    return;
  }

  // ======================= consumer warps =================================
  // S roles: tile st = warp / 2 = 16 heads (group hg = st / 2) x 16
  // positions (half ph = st % 2) of the chunk; the two warps of a tile take
  // halves of the key width (kh = warp % 2). The kh = 0 warps own the online
  // softmax state of their tile's head rows (maxima equal across the two
  // position halves of a group; row sums per half).
  // PV roles: warp (hh = warp / 8, cb = warp % 8): heads 32 hh .. + 31 (two
  // m-tiles) x value columns 64 cb .. + 63 (eight n-tiles).
  const int st = warp >> 1, hg = st >> 1, ph = st & 1, kh = warp & 1;
  const int hh = warp >> 3, cb = warp & 7;
  const uint32_t q0 = smem_u32(sq), k0 = smem_u32(sk);
  float o[2][8][4];            // O: 32 rows x 64 columns
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  int cur_b = -1, cur_h = -1, n_units = 0;
  const int gbar = 2 + hg;     // the 4 warps of head group hg

  auto start_unit = [&](int b, int h) {
    // the query tile of (b, head tile h): 64 rows, one bulk copy each,
    // issued by lanes 0..3 of every consumer warp (a warp issues its copies
    // one lane after another)
    named_sync(kAllBar, kConsumers);  // nobody still reads the old tile
    if (tid == 0) mbar_arrive_expect_tx(qbar, kHeads * DK * 2);
    named_sync(kAllBar, kConsumers);  // the bytes are expected before any lands
    if (lane < kHeads / kCWarps) {
      const int r = warp * (kHeads / kCWarps) + lane;
      bulk_g2s(sq + r * C::QROW,
               p.q + ((long)b * p.n_h + (long)h * kHeads + r) * DK, DK * 2,
               qbar);
    }
    if (!mbar_wait(qbar, n_units & 1) && lane == 0) {
      report(p.err, DEVERR_TIMEOUT);
      s_abort = 1;
    }
    ++n_units;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) o[mt][nt][j] = 0.f;
  };

  auto flush = [&](int b, int h) {
    // row sums of each position half (kh = 0 warps), then per head
    // L = sum of the two halves; the PV warps normalise and write
    if (kh == 0) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      if (qc == 0) {
        lsum[ph * 64 + 16 * hg + qr] = l0;
        lsum[ph * 64 + 16 * hg + qr + 8] = l1;
        if (ph == 0) {
          mfin[16 * hg + qr] = m0;
          mfin[16 * hg + qr + 8] = m1;
        }
      }
    }
    named_sync(kAllBar, kConsumers);
    const int ustart = wp.pre[b];
    const int uend = ustart + wp.nch[b];
    const bool whole = ustart >= lo && uend <= hi;
    const int wslot = (c * 2 + partial_side(ustart, lo)) * tiles + h;
    const long bh0 = (long)b * p.n_h + (long)h * kHeads;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int row = 32 * hh + 16 * mt + qr + 8 * half;  // head in tile
        const float L = lsum[row] + lsum[64 + row];
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int col = 64 * cb + 8 * nt + 2 * qc;
          const float x = o[mt][nt][2 * half] * inv;
          const float y = o[mt][nt][2 * half + 1] * inv;
          if (whole) {
            *reinterpret_cast<uint32_t *>(p.out + (bh0 + row) * DV + col) =
                pack_bf16x2(x, y);
          } else {
            *reinterpret_cast<float2 *>(p.ws_o + ((long)wslot * kHeads + row) *
                                                     DV + col) =
                make_float2(x, y);
          }
        }
        if (cb == 0 && qc == 0) {
          const float lse = L > 0.f
                                ? (mfin[row] + log2f(L)) * 0.69314718055994531f
                                : -INFINITY;
          if (whole) {
            if (p.lse) p.lse[bh0 + row] = lse;
          } else {
            p.ws_lse[(long)wslot * kHeads + row] = lse;
          }
        }
      }
    }
    named_sync(kAllBar, kConsumers);  // lsum / mfin reusable
  };

  ChunkCursor cc = cursor_at(wp, p.batch, lo);
  const float sl2 = p.scale_log2;
  for (int i = 0; i < n; ++i) {
    const int s = i % C::NS;
    const int pb = i & 1;  // P / rescale buffer of this chunk
    if (cc.b != cur_b) {
      if (cur_b >= 0) flush(cur_b, cur_h);
      cur_b = cc.b;
      cur_h = tile;
      start_unit(cur_b, cur_h);
    }
    bool ok = !s_abort && mbar_wait(&full[s], (i / C::NS) & 1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) {
      if (!s_abort) report(p.err, DEVERR_TIMEOUT);
      s_abort = 1;
    }
    const unsigned vmask = *reinterpret_cast<const volatile unsigned *>(
        &s_vpart[s][0]);
    const uint32_t kst = k0 + s * C::KST;
    const uint32_t vst = k0 + s * C::KST;  // values: K's first DV columns
    const int mtx = lane >> 3, ri = lane & 7;
    // ---- S tile: heads 16 hg .., positions 16 ph .., key half kh ----
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
      const uint32_t qa_base = q0 + (16 * hg + (mtx & 1) * 8 + ri) * C::QROW +
                               (mtx >> 1) * 16;
      const uint32_t kb_base = kst + (16 * ph + (mtx >> 1) * 8 + ri) * C::KROW +
                               (mtx & 1) * 16;
      constexpr int KS = DK / 32;  // k-steps of 16 in half the key width
#pragma unroll 6
      for (int ks = kh * KS; ks < (kh + 1) * KS; ++ks) {
        uint32_t a[4], bk[4];
        ldsm_x4(a, qa_base + ks * 32);
        ldsm_x4(bk, kb_base + ks * 32);
        mma_bf16(sa, a, bk[0], bk[1]);  // positions 0..7 of the half
        mma_bf16(sb, a, bk[2], bk[3]);  // positions 8..15
      }
    }
    // the kh = 1 warp's partial tile to its partner
    float *sp = spart + st * 256;
    if (kh == 1) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        sp[j * 32 + lane] = sa[j];
        sp[(4 + j) * 32 + lane] = sb[j];
      }
    }
    named_sync(gbar, 128);
    if (kh == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        sa[j] += sp[j * 32 + lane];
        sb[j] += sp[(4 + j) * 32 + lane];
      }
      // scale, mask, row maxima over this half's 16 positions
      const int c0p = 16 * ph + 2 * qc;  // position of sa[0]
      float sc[8];
      sc[0] = ((vmask >> c0p) & 1) ? sa[0] * sl2 : -INFINITY;
      sc[1] = ((vmask >> (c0p + 1)) & 1) ? sa[1] * sl2 : -INFINITY;
      sc[2] = ((vmask >> c0p) & 1) ? sa[2] * sl2 : -INFINITY;
      sc[3] = ((vmask >> (c0p + 1)) & 1) ? sa[3] * sl2 : -INFINITY;
      sc[4] = ((vmask >> (c0p + 8)) & 1) ? sb[0] * sl2 : -INFINITY;
      sc[5] = ((vmask >> (c0p + 9)) & 1) ? sb[1] * sl2 : -INFINITY;
      sc[6] = ((vmask >> (c0p + 8)) & 1) ? sb[2] * sl2 : -INFINITY;
      sc[7] = ((vmask >> (c0p + 9)) & 1) ? sb[3] * sl2 : -INFINITY;
      float mx0 = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[4], sc[5]));
      float mx1 = fmaxf(fmaxf(sc[2], sc[3]), fmaxf(sc[6], sc[7]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      if (qc == 0) {
        red[st * 16 + qr] = mx0;
        red[st * 16 + qr + 8] = mx1;
      }
      named_sync(gbar + 4, 64);  // the group's two kh = 0 warps
      const int other = (2 * hg + (ph ^ 1)) * 16;
      mx0 = fmaxf(mx0, red[other + qr]);
      mx1 = fmaxf(mx1, red[other + qr + 8]);
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float u0 = n0 == -INFINITY ? 0.f : n0;
      const float u1 = n1 == -INFINITY ? 0.f : n1;
      const float c0 = ex2(m0 - u0), c1 = ex2(m1 - u1);
      m0 = n0;
      m1 = n1;
      float pr[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) pr[j] = ex2(sc[j] - ((j & 2) ? u1 : u0));
      l0 = l0 * c0 + pr[0] + pr[1] + pr[4] + pr[5];
      l1 = l1 * c1 + pr[2] + pr[3] + pr[6] + pr[7];
      // P rows 16 hg + qr (+8), positions 16 ph + 2 qc (+1) and + 8
      uint8_t *prow = spv + pb * C::PBUF + (16 * hg + qr) * C::PROW +
                      (16 * ph + 2 * qc) * 2;
      *reinterpret_cast<uint32_t *>(prow) = pack_bf16x2(pr[0], pr[1]);
      *reinterpret_cast<uint32_t *>(prow + 8 * C::PROW) =
          pack_bf16x2(pr[2], pr[3]);
      *reinterpret_cast<uint32_t *>(prow + 16) = pack_bf16x2(pr[4], pr[5]);
      *reinterpret_cast<uint32_t *>(prow + 8 * C::PROW + 16) =
          pack_bf16x2(pr[6], pr[7]);
      if (ph == 0 && qc == 0) {
        hcor[pb * 64 + 16 * hg + qr] = c0;
        hcor[pb * 64 + 16 * hg + qr + 8] = c1;
      }
    }
    named_sync(kAllBar, kConsumers);  // P and the rescale factors are in
    // ---- O += P V: heads 32 hh .., columns 64 cb .. ----
    {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const float ca = hcor[pb * 64 + 32 * hh + 16 * mt + qr];
        const float cbf = hcor[pb * 64 + 32 * hh + 16 * mt + qr + 8];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          o[mt][nt][0] *= ca;
          o[mt][nt][1] *= ca;
          o[mt][nt][2] *= cbf;
          o[mt][nt][3] *= cbf;
        }
      }
      if (ok) {
        const uint32_t pbase = smem_u32(spv) + pb * C::PBUF;
        const int vrs = C::KROW;
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {  // 16 positions per k-step
          uint32_t pa[2][4];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
            ldsm_x4(pa[mt], pbase +
                                (32 * hh + 16 * mt + (mtx & 1) * 8 + ri) *
                                    C::PROW +
                                (kt * 16 + (mtx >> 1) * 8) * 2);
          // rows of unfetched positions were zeroed by the producer
          const uint32_t vrow = vst + (kt * 16 + (mtx & 1) * 8 + ri) * vrs +
                                64 * cb * 2;
#pragma unroll
          for (int jp = 0; jp < 4; ++jp) {
            uint32_t bv[4];
            ldsm_x4_t(bv, vrow + (2 * jp + (mtx >> 1)) * 16);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              mma_bf16(o[mt][2 * jp], pa[mt], bv[0], bv[1]);
              mma_bf16(o[mt][2 * jp + 1], pa[mt], bv[2], bv[3]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    cursor_next(wp, p.batch, 1, cc);
  }
  if (cur_b >= 0) flush(cur_b, cur_h);

  if (s_abort && tid == 0) {
    for (int t = 0; t < (1 << 20) && s_producer_done < kPW; ++t)
      __nanosleep(1000);
    const int issued = s_issued;
    for (int st = 0; st < C::NS; ++st) {
      int last = -1;
      for (int c2 = st; c2 < issued; c2 += C::NS) last = c2;
      if (last >= 0) mbar_wait(&full[st], (last / C::NS) & 1);
    }
  }
}

constexpr int kMergeSlices = 8;     // CTAs per split unit
constexpr int kMergeThreads = 256;
constexpr int kMergeBatch = 2;      // parts whose loads a thread issues together

// Log-sum-exp merge of the partials of every unit the decode launch cut
// between CTAs. Grid (units, kMergeSlices): CTA (u, j) rebuilds the launch's
// partition, returns if unit u lies inside one CTA's range, and otherwise
// merges the j-th 1/8 of the unit's outputs, four float4s (4 values of one
// head) a thread, the loads of all four for kMergeBatch parts in flight
// together (a unit has 2-3 parts at the usual shapes). The grid stays small
// enough to be resident beside the decode launch and pass its grid wait at
// once: one CTA per 1/128 of a unit (16,384 for 64 sequences x 2 tiles), each
// rebuilding the partition, took 108 us for the 64-sequence latent call.
// Part i is the partial of lane c_first + i: side 1 of the first covering
// lane, side 0 of the others.
template <int DV, int ROWS>
__global__ void __launch_bounds__(kMergeThreads)
    merge_wide_kernel(const DecodeParams p) {
  __shared__ WorkPartitionT<kNB> wp;
  __shared__ int s_len_err;
  pdl_trigger();
  const int tiles = p.n_h / kHeads;
  const int u = blockIdx.x, b = u / tiles, h = u % tiles;
  // The lengths may be read before the decode launch completes: that launch
  // (this launch's only possible predecessor still running, since it lets
  // its dependants start only after its own predecessor has completed)
  // does not write them. The partials are read after pdl_wait.
  build_partition(wp, p, &s_len_err, ROWS, 1);
  pdl_wait();
  const int total = wp.total;
  if (total == 0 || wp.nch[b] == 0) return;
  const int P = min(p.n_splits / tiles, total);
  const int ustart = wp.pre[b];
  const int uend = ustart + wp.nch[b];
  const int c_first = cta_of(ustart, total, P);
  const int parts = cta_of(uend - 1, total, P) - c_first + 1;
  if (parts == 1) return;  // written whole by the decode launch
  constexpr int N4 = kHeads * DV / 4;
  constexpr int PER = N4 / kMergeSlices;
  constexpr int IT = PER / kMergeThreads;  // float4s a thread
  static_assert(IT * kMergeThreads * kMergeSlices == N4, "merge tiling");
  const long bh0 = (long)b * p.n_h + (long)h * kHeads;
  auto slot = [&](int i) {  // partial of part i, in 64-head tiles
    return ((long)(c_first + i) * 2 + (i == 0 ? 1 : 0)) * tiles + h;
  };
  const float4 *o4 = reinterpret_cast<const float4 *>(p.ws_o);
  float M[IT], W[IT];
  float4 acc[IT];
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    M[it] = -INFINITY;
    W[it] = 0.f;
    acc[it] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int e0 = blockIdx.y * PER + threadIdx.x;
  for (int i0 = 0; i0 < parts; i0 += kMergeBatch) {
    float l[IT][kMergeBatch];
    float4 v[IT][kMergeBatch];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      const bool in = i0 + j < parts;
      const long sl = in ? slot(i0 + j) : 0;
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int e = e0 + it * kMergeThreads;
        const int g = (4 * e) / DV;  // head within the tile
        l[it][j] = in ? __ldcg(p.ws_lse + sl * kHeads + g) : -INFINITY;
        v[it][j] = in ? __ldcg(o4 + sl * (kHeads * DV / 4) + e)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int it = 0; it < IT; ++it) {
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        if (l[it][j] == -INFINITY) continue;  // an empty part adds nothing
        const float Mn = fmaxf(M[it], l[it][j]);
        const float a = M[it] == -INFINITY ? 0.f : expf(M[it] - Mn);
        const float w = expf(l[it][j] - Mn);
        W[it] = W[it] * a + w;
        acc[it].x = acc[it].x * a + w * v[it][j].x;
        acc[it].y = acc[it].y * a + w * v[it][j].y;
        acc[it].z = acc[it].z * a + w * v[it][j].z;
        acc[it].w = acc[it].w * a + w * v[it][j].w;
        M[it] = Mn;
      }
    }
  }
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int e = e0 + it * kMergeThreads;
    const int g = (4 * e) / DV;
    const float iw = W[it] > 0.f ? 1.f / W[it] : 0.f;
    uint2 packed;
    packed.x = pack_bf16x2(acc[it].x * iw, acc[it].y * iw);
    packed.y = pack_bf16x2(acc[it].z * iw, acc[it].w * iw);
    *reinterpret_cast<uint2 *>(p.out + bh0 * DV + 4 * e) = packed;
    if ((4 * e) % DV == 0 && p.lse)
      p.lse[bh0 + g] = W[it] > 0.f ? M[it] + logf(W[it]) : -INFINITY;
  }
}

// ROWS: positions per chunk of the decode launch whose partials are merged.
template <int DV, int ROWS = kRows>
cudaError_t launch_merge_wide(const DecodeParams &p, cudaStream_t s) {
  const dim3 grid(p.batch * (p.n_h / kHeads), kMergeSlices);
  return launch_pdl(merge_wide_kernel<DV, ROWS>, grid,
                    dim3(kMergeThreads), 0, s, 1, p);
}

template <int DK, int DV>
cudaError_t launch_t(const DecodeParams &p, cudaStream_t s) {
  using C = WCfg<DK, DV>;
  static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
  auto kern = decode_wide_kernel<DK, DV>;
  static bool done[64] = {};
  cudaError_t e = set_smem_once(kern, C::SMEM, done);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(p.n_splits), dim3(kThreads), C::SMEM, s, 1, p);
  if (e != cudaSuccess || p.n_splits <= 1) return e;
  return launch_merge_wide<DV>(p, s);
}

}  // namespace

cudaError_t launch_merge_mla(const DecodeParams &p, int rows,
                             cudaStream_t s) {
  if (rows == 64) return launch_merge_wide<512, 64>(p, s);
  if (rows == kRows) return launch_merge_wide<512, kRows>(p, s);
  return cudaErrorNotSupported;
}

cudaError_t launch_decode_mla(const DecodeParams &p, cudaStream_t s) {
  if (p.dk != 576 || p.dv != 512 || p.n_h % kHeads != 0 || p.batch > kNB)
    return cudaErrorNotSupported;
  return launch_t<576, 512>(p, s);
}


}  // namespace kvd

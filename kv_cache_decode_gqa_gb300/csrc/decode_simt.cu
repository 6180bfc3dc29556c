// Split-K decode attention on the CUDA cores, for small query groups
// (n_h / n_kv = G in {1, 2, 4}: MHA and narrow GQA). At these group sizes a
// decode step does 2G FLOPs per cached element ("KV cache", "Why decoding
// wastes almost all of your FLOPs": intensity 2 n_h / (n_kv b)), so the
// kernel is bound by HBM bandwidth and the work is to keep the copy engine
// streaming.
//
// One CTA handles (split, kv head, sequence): a run of whole 64-token stages.
// Thread 0 streams each stage's K and V rows (contiguous within a paged
// block) into a 4-deep shared-memory ring with bulk asynchronous copies
// completing on an mbarrier. Four warps consume a stage: lane group
// g = lane / 8 of warp w owns rows 16w + 4i + g (i = 0..3); its 8 lanes each
// hold D/8 elements of the row, so a row is read from shared memory as one
// conflict-free 128-byte (or 256-byte) sweep, and the dot product finishes
// with three xor-shuffles. Every lane group keeps its own online-softmax
// state (max, sum, output slice) per head; the 16 streams are merged in
// shared memory at the end. Scores are kept in log2 units (the query is
// pre-multiplied by scale * log2 e) so each exponential is one ex2.
#include <cuda_fp16.h>

#include <cmath>

#include "kvd_common.cuh"

namespace kvd {
namespace {

constexpr int kThreads = 128;
constexpr int kStages = 4;
constexpr int kStreams = 16;  // 4 warps x 4 lane groups

// Element index (within a row of D) of the e-th value a lane holds.
template <int D, int DT>
__device__ __forceinline__ int elem_index(int sub, int e) {
  if constexpr (DT == DT_BF16) {
    return (e / 8) * 64 + sub * 8 + (e % 8);
  } else {
    return sub * (D / 8) + e;
  }
}

// Load the lane's D/8 elements of a shared-memory row as floats.
template <int D, int DT>
__device__ __forceinline__ void load_row(const uint8_t *row, int sub,
                                         float (&x)[D / 8]) {
  if constexpr (DT == DT_BF16) {
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
  } else if constexpr (D == 128) {
    const uint4 u = *reinterpret_cast<const uint4 *>(row + sub * 16);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t a = e4m3x2_to_f16x2((uint16_t)(w[t] & 0xffff));
      const uint32_t b = e4m3x2_to_f16x2((uint16_t)(w[t] >> 16));
      x[4 * t] = f16lo(a);
      x[4 * t + 1] = f16hi(a);
      x[4 * t + 2] = f16lo(b);
      x[4 * t + 3] = f16hi(b);
    }
  } else {
    const uint2 u = *reinterpret_cast<const uint2 *>(row + sub * 8);
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint32_t a = e4m3x2_to_f16x2((uint16_t)(w[t] & 0xffff));
      const uint32_t b = e4m3x2_to_f16x2((uint16_t)(w[t] >> 16));
      x[4 * t] = f16lo(a);
      x[4 * t + 1] = f16hi(a);
      x[4 * t + 2] = f16lo(b);
      x[4 * t + 3] = f16hi(b);
    }
  }
}

template <int D, int G, int DT>
__global__ void __launch_bounds__(kThreads)
    decode_simt_kernel(const DecodeParams p) {
  constexpr int ES = DT == DT_BF16 ? 2 : 1;
  constexpr int ROW = D * ES;  // bytes per cached row
  constexpr int ROWS = kStageRows;
  constexpr int STAGE = ROWS * ROW;
  constexpr int E = D / 8;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *sk = smem;
  uint8_t *sv = smem + kStages * STAGE;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 2 * kStages * STAGE);

  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 3, sub = lane & 7;
  const int h0 = hkv * G;

  int T = p.seq_lens[b];
  if (T > p.max_seq_len) {
    if (tid == 0 && split == 0 && hkv == 0) report(p.err, DEVERR_LEN);
    T = p.max_seq_len;
  }
  T = max(T, 0);
  const int t0 = split * p.split_len;
  const int t1 = min(T, t0 + p.split_len);
  if (t0 >= t1) {
    // an empty sequence (T == 0) has no split to merge: split 0 writes
    // out = 0, lse = -inf
    if (split == 0) {
      for (int i = tid; i < G * D; i += kThreads)
        p.out[((long)b * p.n_h + h0 + i / D) * D + i % D] = 0;
      if (p.lse && tid < G) p.lse[(long)b * p.n_h + h0 + tid] = -INFINITY;
    }
    return;
  }
  const int nchunks = (t1 - t0 + ROWS - 1) / ROWS;
  const int32_t *bt = p.block_table + (long)b * p.max_blocks;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Producer (thread 0): copy the rows of chunk c into stage c % kStages.
  auto issue = [&](int c) {
    const int s = c % kStages;
    const int tok = t0 + c * ROWS;
    const int n = min(ROWS, t1 - tok);
    mbar_arrive_expect_tx(&bars[s], 2u * n * ROW);
    int done = 0;
    while (done < n) {
      const int t = tok + done;
      const int slot = t % p.block_size;
      const int piece = min(n - done, p.block_size - slot);
      int blk = bt[t / p.block_size];
      if (blk < 0 || blk >= p.num_blocks) {
        report(p.err, DEVERR_BLOCK);
        blk = 0;  // read a valid block; the result is flagged as wrong
      }
      const size_t off =
          (((size_t)blk * p.n_kv + hkv) * p.block_size + slot) * ROW;
      bulk_g2s(sk + s * STAGE + done * ROW, p.k + off, piece * ROW, &bars[s]);
      bulk_g2s(sv + s * STAGE + done * ROW, p.v + off, piece * ROW, &bars[s]);
      done += piece;
    }
  };
  if (tid == 0) {
    for (int c = 0; c < min(kStages, nchunks); ++c) issue(c);
  }

  // Query slice of this lane, in log2 units (fp8: times the K scale).
  float qf[G][E];
  {
    const float qs =
        p.scale_log2 * (DT == DT_FP8 ? p.k_scale[hkv] : 1.0f);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint16_t *qrow = p.q + ((long)b * p.n_h + h0 + h) * D;
#pragma unroll
      for (int e = 0; e < E; e += 8) {
        const uint4 u = *reinterpret_cast<const uint4 *>(
            qrow + elem_index<D, DT>(sub, e));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          qf[h][e + 2 * t] = bf16lo(w[t]) * qs;
          qf[h][e + 2 * t + 1] = bf16hi(w[t]) * qs;
        }
      }
    }
  }

  float m[G], l[G], o[G][E];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[h][e] = 0.f;
  }

  int fail_chunk = -1;
  for (int c = 0; c < nchunks; ++c) {
    const int s = c % kStages;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[s], (c / kStages) & 1));
    if (ok) {
      const int nvalid = min(ROWS, t1 - (t0 + c * ROWS));
      const uint8_t *kst = sk + s * STAGE;
      const uint8_t *vst = sv + s * STAGE;

      float sc[4][G];
  #pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = warp * 16 + i * 4 + grp;
        float kx[E];
        load_row<D, DT>(kst + r * ROW, sub, kx);
  #pragma unroll
        for (int h = 0; h < G; ++h) {
          float a0 = 0.f, a1 = 0.f;
  #pragma unroll
          for (int e = 0; e < E; e += 2) {
            a0 = fmaf(qf[h][e], kx[e], a0);
            a1 = fmaf(qf[h][e + 1], kx[e + 1], a1);
          }
          sc[i][h] = a0 + a1;
        }
      }
  #pragma unroll
      for (int i = 0; i < 4; ++i) {
  #pragma unroll
        for (int h = 0; h < G; ++h) {
          float v = sc[i][h];
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          const int r = warp * 16 + i * 4 + grp;
          sc[i][h] = r < nvalid ? v : -INFINITY;
        }
      }
      float pr[4][G];
  #pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = fmaxf(fmaxf(sc[0][h], sc[1][h]), fmaxf(sc[2][h], sc[3][h]));
        const float m_new = fmaxf(m[h], mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float corr = ex2(m[h] - m_use);
        float psum = 0.f;
  #pragma unroll
        for (int i = 0; i < 4; ++i) {
          pr[i][h] = ex2(sc[i][h] - m_use);
          psum += pr[i][h];
        }
        l[h] = l[h] * corr + psum;
        m[h] = m_new;
  #pragma unroll
        for (int e = 0; e < E; ++e) o[h][e] *= corr;
      }
  #pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = warp * 16 + i * 4 + grp;
        if (r < nvalid) {
          float vx[E];
          load_row<D, DT>(vst + r * ROW, sub, vx);
  #pragma unroll
          for (int h = 0; h < G; ++h) {
  #pragma unroll
            for (int e = 0; e < E; ++e) o[h][e] = fmaf(pr[i][h], vx[e], o[h][e]);
          }
        }
      }
    }
    if (__syncthreads_or(!ok)) {
      fail_chunk = c;
      break;
    }
    if (tid == 0 && c + kStages < nchunks) issue(c + kStages);
  }
  if (fail_chunk >= 0) {
    if (tid == 0) report(p.err, DEVERR_TIMEOUT);
    // let every copy already issued land before the CTA exits
    const int issued = min(fail_chunk + kStages, nchunks);
    for (int st = 0; st < kStages; ++st) {
      int last = -1;
      for (int c2 = st; c2 < issued; c2 += kStages) last = c2;
      if (last >= 0) mbar_wait(&bars[st], (last / kStages) & 1);
    }
    return;
  }

  // Merge the 16 streams (stages are all consumed; reuse their memory).
  float *sm_m = reinterpret_cast<float *>(smem);
  float *sm_l = sm_m + kStreams * G;
  float *sm_o = sm_l + kStreams * G;  // [stream][G][D]
  const int stream = warp * 4 + grp;
  if (sub == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      sm_m[stream * G + h] = m[h];
      sm_l[stream * G + h] = l[h];
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int e = 0; e < E; ++e)
      sm_o[(stream * G + h) * D + elem_index<D, DT>(sub, e)] = o[h][e];
  }
  __syncthreads();
  const float vs = DT == DT_FP8 ? p.v_scale[hkv] : 1.0f;
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int h = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int s2 = 0; s2 < kStreams; ++s2) M = fmaxf(M, sm_m[s2 * G + h]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < kStreams; ++s2) {
      const float ms = sm_m[s2 * G + h];
      const float wgt = ms == -INFINITY ? 0.f : ex2(ms - M);
      L = fmaf(sm_l[s2 * G + h], wgt, L);
      acc = fmaf(sm_o[(s2 * G + h) * D + d], wgt, acc);
    }
    const float res = acc / L * vs;
    const float lse_nat = (M + log2f(L)) * 0.69314718055994531f;
    const long bh = (long)b * p.n_h + h0 + h;
    if (p.n_splits == 1) {
      p.out[bh * D + d] = f2bf(res);
      if (d == 0 && p.lse) p.lse[bh] = lse_nat;
    } else {
      p.ws_o[(bh * p.n_splits + split) * D + d] = res;
      if (d == 0) p.ws_lse[bh * p.n_splits + split] = lse_nat;
    }
  }
  if (p.n_splits > 1) {
    const int n_valid = (T + p.split_len - 1) / p.split_len;
    merge_if_last(p, b, hkv, G, D, n_valid);
  }
}

template <int D, int G, int DT>
cudaError_t launch_t(const DecodeParams &p, cudaStream_t s) {
  constexpr int ROW = D * (DT == DT_BF16 ? 2 : 1);
  constexpr int SMEM = 2 * kStages * kStageRows * ROW + kStages * 8;
  static_assert(kStreams * G * (D + 2) * 4 <= 2 * kStages * kStageRows * ROW,
                "stream merge must fit in the stage buffers");
  auto kern = decode_simt_kernel<D, G, DT>;
  static bool done[64] = {};  // one table per instantiation
  cudaError_t e = set_smem_once(kern, SMEM, done);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_splits, p.n_kv, p.batch);
  kern<<<grid, kThreads, SMEM, s>>>(p);
  return cudaGetLastError();
}

template <int D, int DT>
cudaError_t launch_g(const DecodeParams &p, cudaStream_t s) {
  switch (p.n_h / p.n_kv) {
    case 1: return launch_t<D, 1, DT>(p, s);
    case 2: return launch_t<D, 2, DT>(p, s);
    case 4: return launch_t<D, 4, DT>(p, s);
  }
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeParams &p, cudaStream_t s) {
  const bool fp8 = p.dtype == DT_FP8;
  if (p.dk == 128) return fp8 ? launch_g<128, DT_FP8>(p, s)
                              : launch_g<128, DT_BF16>(p, s);
  if (p.dk == 64) return fp8 ? launch_g<64, DT_FP8>(p, s)
                             : launch_g<64, DT_BF16>(p, s);
  return cudaErrorNotSupported;
}

}  // namespace kvd

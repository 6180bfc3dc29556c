// Log-sum-exp merge of split-K partials. Each split s of a (sequence, head)
// produced o_s (normalised over its own positions) and lse_s; the attention
// over the union of the splits is
//   out = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M),  M = max_s lse_s,
//   lse = M + log sum_s exp(lse_s - M).
// Splitting a softmax this way is exact up to rounding, the same reason
// FlashAttention is exact (the My Weird Prompts 640482 transcript). Splits
// past a dense sequence's length are skipped; a split with lse = -inf
// (nothing selected) adds nothing; no split at all gives out = 0, lse = -inf.
#include <cmath>

#include "kvd_common.cuh"

namespace kvd {
namespace {

constexpr int kMaxSplits = 1024;

__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
  __shared__ float wts[kMaxSplits];
  __shared__ float s_max, s_sum;
  const int bh = blockIdx.x;
  const int b = bh / p.n_h;
  const int tid = threadIdx.x;
  int n_valid = p.n_splits;
  if (p.seq_lens) {
    int T = min(max(p.seq_lens[b], 0), p.max_seq_len);
    n_valid = min(p.n_splits, (T + p.split_len - 1) / p.split_len);
  }
  const float *lse_s = p.ws_lse + (long)bh * p.n_splits;
  if (tid == 0) {
    float M = -INFINITY;
    for (int s = 0; s < n_valid; ++s) M = fmaxf(M, lse_s[s]);
    float W = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < n_valid; ++s) {
        const float w = lse_s[s] == -INFINITY ? 0.f : expf(lse_s[s] - M);
        wts[s] = w;
        W += w;
      }
    }
    s_max = M;
    s_sum = W;
  }
  __syncthreads();
  const float M = s_max, W = s_sum;
  uint16_t *out = p.out + (long)bh * p.dv;
  if (M == -INFINITY) {
    for (int d = tid; d < p.dv; d += blockDim.x) out[d] = 0;
    if (tid == 0 && p.lse) p.lse[bh] = -INFINITY;
    return;
  }
  const float inv = 1.0f / W;
  const float *o_s = p.ws_o + (long)bh * p.n_splits * p.dv;
  for (int d = tid; d < p.dv; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < n_valid; ++s) {
      if (wts[s] != 0.f) acc = fmaf(wts[s], o_s[(long)s * p.dv + d], acc);
    }
    out[d] = f2bf(acc * inv);
  }
  if (tid == 0 && p.lse) p.lse[bh] = M + logf(W);
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t s) {
  if (p.n_splits > kMaxSplits) return cudaErrorNotSupported;
  const long n = (long)p.batch * p.n_h;
  if (n == 0) return cudaSuccess;
  merge_kernel<<<(unsigned)n, 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvd

// Load-balancing statistics of a routed batch and the post-batch bias controller.
//
// Section 10 "Routing, Capacity, and Load Balancing":
//   P_i = (1/T) sum_t p_t,i, the mean score of expert i normalised across experts
//         (softmax probabilities, or sigmoid scores divided by their sum, Section 10.7.1);
//   f_i = C_i^req / (K T) and L_LBL = N sum_i f_i P_i                      (Eq. 30, 38)
//   I_max(x) = n max(x) / sum(x)                                           (Eq. 22, 39)
//   I_H(x) = 1 - H(x / sum x) / log n, the coefficient of variation and the
//   never-selected count (Section 10.2); delta_route = sum D / (K T)       (Eq. 27)
//   b_i <- b_i + gamma sign(mean(C) - C_i)                                  (Eq. 36-37)
//
// The score sums are deterministic: one CTA per 256-token tile writes per-expert
// partial sums in token order, and one CTA adds the tiles in order.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kTile = 256;

__global__ void __launch_bounds__(256) score_partial_kernel(const float* logits, int64_t T, int N,
                                                            int score, float* partial) {
  __shared__ float s_max[kTile];
  __shared__ float s_sum[kTile];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTile;
  const int rows = static_cast<int>(min(static_cast<int64_t>(kTile), T - t0));
  // per-token normaliser: softmax (max, sum of exp) or the sum of sigmoid scores
  for (int r = warp; r < rows; r += 8) {
    const float* z = logits + (t0 + r) * N;
    float m = -INFINITY;
    if (score == MOE_SCORE_SOFTMAX) {
      for (int e = lane; e < N; e += 32) m = fmaxf(m, z[e]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    }
    float s = 0.f;
    for (int e = lane; e < N; e += 32)
      s += score == MOE_SCORE_SOFTMAX ? expf(z[e] - m) : 1.f / (1.f + expf(-z[e]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
      s_max[r] = m;
      s_sum[r] = s;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    float acc = 0.f;
    for (int r = 0; r < rows; ++r) {
      const float z = logits[(t0 + r) * N + e];
      const float q = score == MOE_SCORE_SOFTMAX ? expf(z - s_max[r]) : 1.f / (1.f + expf(-z));
      acc += q / s_sum[r];
    }
    partial[static_cast<int64_t>(blockIdx.x) * N + e] = acc;
  }
}

struct StatsArgs {
  const float* partial;   // [tiles][N] or nullptr (no scores)
  int64_t tiles, T;
  int32_t N, K, M;
  const int32_t* counts_req;
  const int32_t* counts_keep;
  const int32_t* R_req;
  const int32_t* R_keep;
  float* P;
  float* f;
  float* stats;
};

__device__ double imax(const int32_t* x, int n) {
  double mx = 0.0, s = 0.0;
  for (int i = 0; i < n; ++i) {
    mx = fmax(mx, static_cast<double>(x[i]));
    s += x[i];
  }
  return s > 0 ? n * mx / s : 0.0;
}

__device__ double hdef(const int32_t* x, int n) {
  double s = 0.0, h = 0.0;
  for (int i = 0; i < n; ++i) s += x[i];
  if (s <= 0 || n < 2) return 0.0;
  for (int i = 0; i < n; ++i)
    if (x[i] > 0) {
      const double pi = x[i] / s;
      h -= pi * log(pi);
    }
  return 1.0 - h / log(static_cast<double>(n));
}

__global__ void __launch_bounds__(256) stats_kernel(StatsArgs a) {
  __shared__ double s_fp[kMaxExperts];
  const double KT = static_cast<double>(a.K) * static_cast<double>(a.T);
  for (int e = threadIdx.x; e < a.N; e += blockDim.x) {
    const double fe = KT > 0 ? a.counts_req[e] / KT : 0.0;
    double Pe = 0.0;
    if (a.partial) {
      for (int64_t t = 0; t < a.tiles; ++t) Pe += a.partial[t * a.N + e];
      Pe = a.T > 0 ? Pe / static_cast<double>(a.T) : 0.0;
    }
    if (a.P) a.P[e] = static_cast<float>(Pe);
    if (a.f) a.f[e] = static_cast<float>(fe);
    s_fp[e] = fe * Pe;
  }
  __syncthreads();
  if (threadIdx.x != 0 || a.stats == nullptr) return;
  double L = 0.0;
  for (int e = 0; e < a.N; ++e) L += s_fp[e];
  double mean = 0.0, var = 0.0;
  int never = 0;
  long long dropped = 0;
  for (int e = 0; e < a.N; ++e) {
    mean += a.counts_req[e];
    never += a.counts_req[e] == 0;
    if (a.counts_keep) dropped += a.counts_req[e] - a.counts_keep[e];
  }
  mean /= a.N;
  for (int e = 0; e < a.N; ++e) var += (a.counts_req[e] - mean) * (a.counts_req[e] - mean);
  var /= a.N;
  float* o = a.stats;
  o[MOE_STAT_LBL] = a.partial ? static_cast<float>(a.N * L) : NAN;
  o[MOE_STAT_IMAX_REQ] = static_cast<float>(imax(a.counts_req, a.N));
  o[MOE_STAT_IMAX_KEEP] = a.counts_keep ? static_cast<float>(imax(a.counts_keep, a.N)) : NAN;
  o[MOE_STAT_IMAX_RANK_REQ] = a.R_req ? static_cast<float>(imax(a.R_req, a.M)) : NAN;
  o[MOE_STAT_IMAX_RANK_KEEP] = a.R_keep ? static_cast<float>(imax(a.R_keep, a.M)) : NAN;
  o[MOE_STAT_IH_REQ] = static_cast<float>(hdef(a.counts_req, a.N));
  o[MOE_STAT_IH_KEEP] = a.counts_keep ? static_cast<float>(hdef(a.counts_keep, a.N)) : NAN;
  o[MOE_STAT_CV_REQ] = mean > 0 ? static_cast<float>(sqrt(var) / mean) : 0.f;
  o[MOE_STAT_NEVER_SELECTED] = static_cast<float>(never);
  o[MOE_STAT_DROP_FRACTION] = (a.counts_keep && KT > 0) ? static_cast<float>(dropped / KT) : NAN;
}

__global__ void bias_update_kernel(int N, const int32_t* counts, float gamma, float* bias) {
  __shared__ double s_mean;
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int e = 0; e < N; ++e) s += counts[e];
    s_mean = s / N;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    const double d = s_mean - counts[e];
    const float step = d > 0 ? 1.f : (d < 0 ? -1.f : 0.f);
    bias[e] = bias[e] + gamma * step;
  }
}

}  // namespace

cudaError_t launch_balance_stats(const moe_config& c, const float* logits, float* partial,
                                 const int32_t* counts_req, const int32_t* counts_keep,
                                 const int32_t* R_req, const int32_t* R_keep, float* P, float* f,
                                 float* stats, cudaStream_t s) {
  const int64_t tiles = (c.T + kTile - 1) / kTile;
  if (logits && c.T > 0) {
    score_partial_kernel<<<static_cast<unsigned>(tiles), 256, 0, s>>>(logits, c.T, c.N, c.score,
                                                                      partial);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  StatsArgs a{};
  a.partial = (logits && c.T > 0) ? partial : nullptr;
  a.tiles = tiles;
  a.T = c.T;
  a.N = c.N;
  a.K = c.K;
  a.M = c.num_ranks;
  a.counts_req = counts_req;
  a.counts_keep = counts_keep;
  a.R_req = R_req;
  a.R_keep = R_keep;
  a.P = P;
  a.f = f;
  a.stats = stats;
  stats_kernel<<<1, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bias_update(int32_t N, const int32_t* counts, float gamma, float* bias,
                               cudaStream_t s) {
  bias_update_kernel<<<1, 256, 0, s>>>(N, counts, gamma, bias);
  return cudaGetLastError();
}

}  // namespace moe

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
// The score sums are deterministic: one CTA per 64-token tile, each lane summing its rows in
// token order, the row groups and warps combined in a fixed order; then one CTA adds the tiles
// in order (compensated fp32).  Counts are reduced exactly in integers and the remaining float
// sums run in a fixed shuffle-tree order, so every output is reproducible run to run.  Double
// precision is kept to a few scalar operations: its rate on this part is far below fp32's.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kTile = kScoreTile;   // tokens per CTA of the score pass
constexpr int kWarps = 8;
constexpr int kRowsInFlight = 8;    // row steps whose loads a warp issues together

// W lanes share one row (W = N rounded up to a power of two, at most 32), so a warp covers
// 32 / W rows per step and each lane holds C = ceil(N / W) experts: lane l of its group owns
// experts l, l + W, ...
template <int W, int C>
__global__ void __launch_bounds__(256) score_partial_kernel(const float* logits, int64_t T, int N,
                                                            int score, float* partial) {
  constexpr int kGroups = 32 / W;             // rows per warp step
  constexpr int kStep = kWarps * kGroups;     // rows per CTA step
  __shared__ float s_part[kWarps][kGroups][W * C];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int grp = lane / W, l = lane % W;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTile;
  const int rows = static_cast<int>(min(static_cast<int64_t>(kTile), T - t0));
  const bool softmax = score == MOE_SCORE_SOFTMAX;
  float acc[C];
#pragma unroll
  for (int j = 0; j < C; ++j) acc[j] = 0.f;
  // row of (step u, warp, group): base + u * kStep + warp * kGroups + grp
  for (int base = 0; base < rows; base += kStep * kRowsInFlight) {
    float z[kRowsInFlight][C];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int r = base + u * kStep + warp * kGroups + grp;
#pragma unroll
      for (int j = 0; j < C; ++j) {
        const int e = l + W * j;
        z[u][j] = (r < rows && e < N) ? logits[(t0 + r) * N + e] : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      if (base + u * kStep >= rows) break;   // the same for every lane of the CTA
      const bool row_ok = base + u * kStep + warp * kGroups + grp < rows;
      // the row's normaliser: softmax (max, sum of exp) or the sum of sigmoid scores
      float m = -INFINITY;
      if (softmax) {
#pragma unroll
        for (int j = 0; j < C; ++j) m = fmaxf(m, z[u][j]);
#pragma unroll
        for (int off = W / 2; off > 0; off >>= 1)
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      }
      float q[C], ssum = 0.f;
#pragma unroll
      for (int j = 0; j < C; ++j) {
        const bool ok = row_ok && l + W * j < N;
        q[j] = !ok ? 0.f : (softmax ? expf(z[u][j] - m) : 1.f / (1.f + expf(-z[u][j])));
        ssum += q[j];
      }
#pragma unroll
      for (int off = W / 2; off > 0; off >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, off);
      if (row_ok) {
        const float inv = 1.f / ssum;
#pragma unroll
        for (int j = 0; j < C; ++j) acc[j] += q[j] * inv;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < C; ++j) s_part[warp][grp][l + W * j] = acc[j];
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
#pragma unroll
      for (int g = 0; g < kGroups; ++g) v += s_part[w][g][e];
    partial[static_cast<int64_t>(blockIdx.x) * N + e] = v;
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

// s + x with the rounding error carried in c (Neumaier's variant of compensated summation).
__device__ __forceinline__ void comp_add(float& s, float& c, float x) {
  const float t = s + x;
  c += fabsf(s) >= fabsf(x) ? (s - t) + x : (x - t) + s;
  s = t;
}

__device__ __forceinline__ long long warp_sum(long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ long long warp_max(long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// a butterfly: every lane ends with the same, order-fixed sum
__device__ __forceinline__ float warp_sumf(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// phi(x) = x log x - x + 1 at x = n c / S, written with u = x - 1 = (n c - S) / S: the
// entropy deficit of counts c is sum_i phi(x_i) / (n log n), a sum of non-negative terms
// (log n - H(c / S) = sum_i p_i log(n p_i) and sum_i (p_i - 1/n) = 0).
__device__ __forceinline__ float phi_term(long long c, long long S, int n) {
  if (c == 0) return 1.f;
  const float u = static_cast<float>(static_cast<long long>(n) * c - S) / static_cast<float>(S);
  return (1.f + u) * log1pf(u) - u;
}

// Integer slots of the first block reduction (sums, maxima, sums of squares, counters).
enum { kSumReq, kMaxReq, kSumKeep, kMaxKeep, kSumRR, kMaxRR, kSumRK, kMaxRK, kNever, kDropped,
       kSqReq, kIntSlots };

constexpr int kStatsThreads = 1024;

// One CTA of 1024 threads.  The tile sums of P spread over all of them; the statistics of
// the count vectors use the first 256, one thread per expert (N <= 256) and per rank
// (M <= 256).
__global__ void __launch_bounds__(kStatsThreads) stats_kernel(StatsArgs a) {
  __shared__ float s_sum[kStatsThreads];
  __shared__ long long s_int[kWarps][kIntSlots];
  __shared__ float s_flt[kWarps][3];
  const int i = threadIdx.x, warp = i / 32, lane = i % 32;
  const int N = a.N, M = a.M;
  const long long KT = static_cast<long long>(a.K) * a.T;

  // P_i: G = 1024 / Np threads per expert (Np = N rounded up to a power of two), thread
  // (g, e) adding tiles g, g + G, ... in order (compensated); the G sums of an expert are
  // then added pairwise in a fixed tree.
  int Np = 1;
  while (Np < N) Np <<= 1;
  const int G = kStatsThreads / Np;
  if (a.partial) {
    const int e = i % Np, g = i / Np;
    float sum = 0.f, cmp = 0.f;
    if (e < N) {
#pragma unroll 8
      for (int64_t t = g; t < a.tiles; t += G) comp_add(sum, cmp, a.partial[t * N + e]);
    }
    s_sum[i] = sum + cmp;
    __syncthreads();
    for (int st = G / 2; st > 0; st >>= 1) {
      if (g < st) s_sum[i] += s_sum[i + st * Np];
      __syncthreads();
    }
  }
  float fP = 0.f;
  if (i < N) {
    const float Pe = (a.partial && a.T > 0) ? s_sum[i] / static_cast<float>(a.T) : 0.f;
    const float fe = KT > 0 ? static_cast<float>(a.counts_req[i]) / static_cast<float>(KT) : 0.f;
    if (a.P) a.P[i] = Pe;
    if (a.f) a.f[i] = fe;
    fP = fe * Pe;
  }
  if (a.stats == nullptr) return;   // uniform over the block

  // exact integer reductions and the L sum, one pass
  const long long c = i < N ? a.counts_req[i] : 0;
  const long long ck = (a.counts_keep && i < N) ? a.counts_keep[i] : 0;
  const long long rr = (a.R_req && i < M) ? a.R_req[i] : 0;
  const long long rk = (a.R_keep && i < M) ? a.R_keep[i] : 0;
  long long v[kIntSlots] = {c, c, ck, ck, rr, rr, rk, rk, (i < N && c == 0) ? 1 : 0, c - ck, c * c};
  if (!a.counts_keep) v[kDropped] = 0;
  if (warp < kWarps) {   // whole warps: threads 0..255 hold every expert and rank
#pragma unroll
    for (int k = 0; k < kIntSlots; ++k)
      v[k] = (k == kMaxReq || k == kMaxKeep || k == kMaxRR || k == kMaxRK) ? warp_max(v[k])
                                                                             : warp_sum(v[k]);
    const float L_w = warp_sumf(fP);
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < kIntSlots; ++k) s_int[warp][k] = v[k];
      s_flt[warp][0] = L_w;
    }
  }
  __syncthreads();
  if (warp >= kWarps) return;   // only named barrier 1 (256 threads) follows
  long long tot[kIntSlots];
#pragma unroll
  for (int k = 0; k < kIntSlots; ++k) {
    const bool is_max = k == kMaxReq || k == kMaxKeep || k == kMaxRR || k == kMaxRK;
    tot[k] = s_int[0][k];
    for (int w = 1; w < kWarps; ++w) tot[k] = is_max ? max(tot[k], s_int[w][k]) : tot[k] + s_int[w][k];
  }

  // entropy-deficit terms, which need the totals
  const float ph = (i < N && tot[kSumReq] > 0) ? phi_term(c, tot[kSumReq], N) : 0.f;
  const float phk = (a.counts_keep && i < N && tot[kSumKeep] > 0) ? phi_term(ck, tot[kSumKeep], N) : 0.f;
  const float ph_w = warp_sumf(ph), phk_w = warp_sumf(phk);
  if (lane == 0) {
    s_flt[warp][1] = ph_w;
    s_flt[warp][2] = phk_w;
  }
  // a barrier of the first 256 threads only (named barrier 1; the others have returned)
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (i != 0) return;
  float L = 0.f, Phi = 0.f, Phik = 0.f;
  for (int w = 0; w < kWarps; ++w) {
    L += s_flt[w][0];
    Phi += s_flt[w][1];
    Phik += s_flt[w][2];
  }
  auto imax = [](long long mx, long long S, int n) {
    return S > 0 ? static_cast<float>(static_cast<long long>(n) * mx) / static_cast<float>(S) : 0.f;
  };
  auto hdef = [](float phi_sum, long long S, int n) {
    return (S > 0 && n >= 2) ? phi_sum / (static_cast<float>(n) * logf(static_cast<float>(n))) : 0.f;
  };
  const long long S = tot[kSumReq];
  // cv = sqrt(N sum c^2 - S^2) / S; the difference (exact in integers up to rounding of the
  // two products to double) is where the cancellation sits
  const double var_n2 = static_cast<double>(N) * static_cast<double>(tot[kSqReq]) -
                        static_cast<double>(S) * static_cast<double>(S);
  float* o = a.stats;
  o[MOE_STAT_LBL] = a.partial ? static_cast<float>(N) * L : NAN;
  o[MOE_STAT_IMAX_REQ] = imax(tot[kMaxReq], S, N);
  o[MOE_STAT_IMAX_KEEP] = a.counts_keep ? imax(tot[kMaxKeep], tot[kSumKeep], N) : NAN;
  o[MOE_STAT_IMAX_RANK_REQ] = a.R_req ? imax(tot[kMaxRR], tot[kSumRR], M) : NAN;
  o[MOE_STAT_IMAX_RANK_KEEP] = a.R_keep ? imax(tot[kMaxRK], tot[kSumRK], M) : NAN;
  o[MOE_STAT_IH_REQ] = hdef(Phi, S, N);
  o[MOE_STAT_IH_KEEP] = a.counts_keep ? hdef(Phik, tot[kSumKeep], N) : NAN;
  o[MOE_STAT_CV_REQ] = S > 0 ? sqrtf(static_cast<float>(fmax(var_n2, 0.0))) / static_cast<float>(S) : 0.f;
  o[MOE_STAT_NEVER_SELECTED] = static_cast<float>(tot[kNever]);
  o[MOE_STAT_DROP_FRACTION] =
      (a.counts_keep && KT > 0) ? static_cast<float>(tot[kDropped]) / static_cast<float>(KT) : NAN;
}

// One CTA of 256 threads, one per expert.  sign(mean(C) - C_i) = sign(S - N C_i) with S the
// exact integer sum, so no division is needed.
__global__ void __launch_bounds__(256) bias_update_kernel(int N, const int32_t* counts, float gamma,
                                                          float* bias) {
  __shared__ long long s_tot[kWarps];
  const int e = threadIdx.x;
  const long long c = e < N ? counts[e] : 0;
  const long long w = warp_sum(c);
  if (e % 32 == 0) s_tot[e / 32] = w;
  __syncthreads();
  long long S = 0;
  for (int k = 0; k < kWarps; ++k) S += s_tot[k];
  if (e < N) {
    const long long d = S - static_cast<long long>(N) * c;
    const float step = d > 0 ? 1.f : (d < 0 ? -1.f : 0.f);
    bias[e] = bias[e] + gamma * step;
  }
}

}  // namespace

// the score pass's lane mapping for N experts: W lanes per row, C experts per lane
static cudaError_t launch_score_partial(unsigned tiles, const float* logits, int64_t T, int N,
                                        int score, float* partial, cudaStream_t s) {
  if (N <= 1) score_partial_kernel<1, 1><<<tiles, 256, 0, s>>>(logits, T, N, score, partial);
  else if (N <= 2) score_partial_kernel<2, 1><<<tiles, 256, 0, s>>>(logits, T, N, score, partial);
  else if (N <= 4) score_partial_kernel<4, 1><<<tiles, 256, 0, s>>>(logits, T, N, score, partial);
  else if (N <= 8) score_partial_kernel<8, 1><<<tiles, 256, 0, s>>>(logits, T, N, score, partial);
  else if (N <= 16) score_partial_kernel<16, 1><<<tiles, 256, 0, s>>>(logits, T, N, score, partial);
  else if (N <= 32) score_partial_kernel<32, 1><<<tiles, 256, 0, s>>>(logits, T, N, score, partial);
  else if (N <= 64) score_partial_kernel<32, 2><<<tiles, 256, 0, s>>>(logits, T, N, score, partial);
  else if (N <= 128) score_partial_kernel<32, 4><<<tiles, 256, 0, s>>>(logits, T, N, score, partial);
  else score_partial_kernel<32, 8><<<tiles, 256, 0, s>>>(logits, T, N, score, partial);
  return cudaGetLastError();
}

cudaError_t launch_balance_stats(const moe_config& c, const float* logits, float* partial,
                                 const int32_t* counts_req, const int32_t* counts_keep,
                                 const int32_t* R_req, const int32_t* R_keep, float* P, float* f,
                                 float* stats, cudaStream_t s) {
  const int64_t tiles = (c.T + kTile - 1) / kTile;   // kScoreTile-token tiles
  if (logits && c.T > 0) {
    cudaError_t e = launch_score_partial(static_cast<unsigned>(tiles), logits, c.T, c.N, c.score,
                                         partial, s);
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
  stats_kernel<<<1, kStatsThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bias_update(int32_t N, const int32_t* counts, float gamma, float* bias,
                               cudaStream_t s) {
  bias_update_kernel<<<1, 256, 0, s>>>(N, counts, gamma, bias);
  return cudaGetLastError();
}

}  // namespace moe

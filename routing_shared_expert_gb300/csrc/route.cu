// Router: logits, scores, top-K selection and merge coefficients.
//
// Follows Section 10 "Routing, Capacity, and Load Balancing" (Table 16: router
// projection and gating function; Eq. 35: softmax routing selects on the logits),
// Appendix E "Expert-Merge Normalization in Public MoE Models" (Table 52: softmax
// or sigmoid scores, selected renormalisation, routed scale alpha, softmax over
// the selected logits, learned sigmoid shared gate) and Section 21 "Merging
// Routed and Shared Expert Activations" (Eq. 80 coefficients r and s).
//
// This file holds the CUDA-core router, used for fp32 layers (bf16 layers use the
// tensor-core router in route_tc.cu).  One CTA handles 32 tokens.  Phase 1 computes the fp32 logits of its tokens for
// all N experts (plus the shared-gate column w_s when the layer has one) with a
// register-tiled dot product over d staged through shared memory.  Phase 2 gives
// each warp four tokens: the warp holds a token's N logits (8 per lane at most),
// takes K rounds of a warp arg-max on (logit desc, index asc), and evaluates the
// scores and coefficients of the selected experts in registers.
#include "common.cuh"
#include "internal.h"
#include "route_norm.cuh"

namespace moe {
namespace {

constexpr int kTokens = 32;      // tokens per CTA
constexpr int kChunk = 32;       // d elements per shared-memory stage
constexpr int kThreads = 256;

template <typename T, int MAXC>
__global__ void __launch_bounds__(kThreads) route_kernel(RouteParams p) {
  extern __shared__ float sm[];
  const int ncols = p.N + (p.shared_mode == MOE_SHARED_SIGMOID_GATE ? 1 : 0);
  const int cpt = (ncols + 15) / 16;                 // columns per thread
  float* xs = sm;                                    // [kTokens][kChunk + 1]
  float* ws = xs + kTokens * (kChunk + 1);           // [ncols][kChunk + 1]
  float* zl = ws + ncols * (kChunk + 1);             // [kTokens][ncols + 1]

  const int tid = threadIdx.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokens;
  const T* x = static_cast<const T*>(p.x);
  const T* W = static_cast<const T*>(p.W_router);
  const T* wsg = static_cast<const T*>(p.shared_gate_w);

  // ---------------- phase 1: logits ----------------
  const int tp = tid / 16;   // token pair 0..15
  const int cg = tid % 16;   // column group
  float acc0[MAXC], acc1[MAXC];
#pragma unroll
  for (int j = 0; j < MAXC; ++j) acc0[j] = acc1[j] = 0.f;

  for (int k0 = 0; k0 < p.d; k0 += kChunk) {
    for (int i = tid; i < kTokens * kChunk; i += kThreads) {
      const int r = i / kChunk, c = i % kChunk;
      const int64_t t = t0 + r;
      const int k = k0 + c;
      xs[r * (kChunk + 1) + c] = (t < p.T && k < p.d) ? to_f32(x[t * p.d + k]) : 0.f;
    }
    for (int i = tid; i < ncols * kChunk; i += kThreads) {
      const int r = i / kChunk, c = i % kChunk;
      const int k = k0 + c;
      float v = 0.f;
      if (k < p.d) v = (r < p.N) ? to_f32(W[static_cast<int64_t>(r) * p.d + k]) : to_f32(wsg[k]);
      ws[r * (kChunk + 1) + c] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kChunk; ++c) {
      const float xa = xs[(2 * tp) * (kChunk + 1) + c];
      const float xb = xs[(2 * tp + 1) * (kChunk + 1) + c];
#pragma unroll
      for (int j = 0; j < MAXC; ++j) {
        const int col = cg + 16 * j;
        if (j < cpt && col < ncols) {
          const float w = ws[col * (kChunk + 1) + c];
          acc0[j] = fmaf(xa, w, acc0[j]);
          acc1[j] = fmaf(xb, w, acc1[j]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    const int col = cg + 16 * j;
    if (j < cpt && col < ncols) {
      const float b = (col < p.N && p.router_bias) ? p.router_bias[col] : 0.f;
      // The selection key is the fp32 logit with the bias added in fp32.
      zl[(2 * tp) * (ncols + 1) + col] = acc0[j] + b;
      zl[(2 * tp + 1) * (ncols + 1) + col] = acc1[j] + b;
    }
  }
  __syncthreads();

  // ---------------- phase 2: selection and coefficients ----------------
  const int warp = tid / 32, lane = tid % 32;
  for (int r = warp; r < kTokens; r += kThreads / 32) {
    const int64_t t = t0 + r;
    if (t >= p.T) break;
    const float* z = zl + r * (ncols + 1);
    float v[8], key[8];   // unbiased logit z, and the selection key z + b_sel
    bool live[8];
    float zmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      live[j] = e < p.N;
      v[j] = live[j] ? z[e] : 0.f;
      key[j] = (live[j] && p.selection_bias) ? v[j] + p.selection_bias[e] : v[j];
      if (live[j]) zmax = fmaxf(zmax, v[j]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, off));
    if (p.logits) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (live[j]) p.logits[t * p.N + lane + 32 * j] = v[j];
    }
    int sel_i[kMaxTopK];
    float sel_z[kMaxTopK];
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) { sel_i[k] = 0; sel_z[k] = 0.f; }
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
      if (k >= p.K) break;
      // this lane's best remaining candidate: larger key, then lower index
      float bv = 0.f, bz = 0.f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = lane + 32 * j;
        if (live[j] && (bi == 0x7fffffff || key[j] > bv)) { bv = key[j]; bz = v[j]; bi = e; }
      }
      // warp arg-max (ties to the lower index; lanes without candidates carry bi = INT_MAX)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const float oz = __shfl_xor_sync(0xffffffffu, bz, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        const bool take = (oi != 0x7fffffff) &&
                          (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
        if (take) { bv = ov; bz = oz; bi = oi; }
      }
      sel_i[k] = bi;
      sel_z[k] = bz;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (bi == lane + 32 * j) live[j] = false;
    }

    // scores of the selected experts and their weights w; r = alpha * w
    float w[kMaxTopK];
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) w[k] = 0.f;
    if (p.norm == MOE_NORM_SOFTMAX_SELECTED) {
      float s = 0.f, msel = sel_z[0];
#pragma unroll
      for (int k = 1; k < kMaxTopK; ++k)
        if (k < p.K) msel = fmaxf(msel, sel_z[k]);
#pragma unroll
      for (int k = 0; k < kMaxTopK; ++k)
        if (k < p.K) { w[k] = expf(sel_z[k] - msel); s += w[k]; }
#pragma unroll
      for (int k = 0; k < kMaxTopK; ++k)
        if (k < p.K) w[k] /= s;
    } else {
      if (p.score == MOE_SCORE_SOFTMAX) {
        // full softmax over all N (unbiased logits)
        const float m = zmax;
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int e = lane + 32 * j;
          if (e < p.N) s += expf(z[e] - m);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
          if (k < p.K) w[k] = expf(sel_z[k] - m) / s;
      } else {
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
          if (k < p.K) w[k] = 1.f / (1.f + expf(-sel_z[k]));
      }
      if (p.norm == MOE_NORM_L1_SELECTED) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
          if (k < p.K) s += w[k];
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
          if (k < p.K) w[k] /= s;
      } else if (p.norm == MOE_NORM_LP_SELECTED) {
        lp_normalise(w, p.K, p.norm_p);
      }
    }
    if (lane < p.K) {
      float wk = 0.f;
      int ik = 0;
#pragma unroll
      for (int k = 0; k < kMaxTopK; ++k)
        if (k == lane) { wk = w[k]; ik = sel_i[k]; }
      p.topk_idx[t * p.K + lane] = ik;
      p.topk_w[t * p.K + lane] = p.alpha * wk;
    }
    if (lane == 0 && p.shared_coef) {
      float s = 0.f;
      if (p.shared_mode == MOE_SHARED_CONST) s = p.shared_gain;
      else if (p.shared_mode == MOE_SHARED_SIGMOID_GATE) s = 1.f / (1.f + expf(-z[p.N]));
      p.shared_coef[t] = s;
    }
  }
}

template <typename T, int MAXC>
cudaError_t launch_t(const RouteParams& p, cudaStream_t s) {
  const int ncols = p.N + (p.shared_mode == MOE_SHARED_SIGMOID_GATE ? 1 : 0);
  const size_t smem =
      sizeof(float) * (kTokens * (kChunk + 1) + ncols * (kChunk + 1) + kTokens * (ncols + 1));
  auto kern = route_kernel<T, MAXC>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (p.T + kTokens - 1) / kTokens;
  kern<<<static_cast<unsigned>(blocks), kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dt(const RouteParams& p, cudaStream_t s) {
  const int ncols = p.N + (p.shared_mode == MOE_SHARED_SIGMOID_GATE ? 1 : 0);
  const int cpt = (ncols + 15) / 16;
  if (cpt <= 2) return launch_t<T, 2>(p, s);
  if (cpt <= 4) return launch_t<T, 4>(p, s);
  if (cpt <= 8) return launch_t<T, 8>(p, s);
  return launch_t<T, 17>(p, s);
}

}  // namespace

cudaError_t launch_route(const RouteParams& p, int32_t dtype, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  return dtype == MOE_F32 ? launch_dt<float>(p, s) : launch_route_tc(p, s);
}

}  // namespace moe

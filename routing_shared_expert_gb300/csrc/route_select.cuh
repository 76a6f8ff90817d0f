// Selection, scores and coefficients of one token from its router accumulators (the bf16
// router's epilogue, route_tc.cu), behind a column loader so that the selection does not
// depend on where the accumulators live.
//
// Section 10 "Routing, Capacity, and Load Balancing" (Table 16, Eq. 35), Appendix E
// "Expert-Merge Normalization in Public MoE Models" (Table 52) and Section 21 (Eq. 80
// coefficients): the key z (+ the Eq. 35 selection-only bias) picks the top K experts,
// lower index first on equal keys; the scores of the selected experts come from the
// unbiased logits z = x W_router^T (+ the logit bias); the selected weights follow the
// layer's rule and r = alpha * w; s(x) is the constant gain or sigmoid(w_s . x).
#pragma once

#include "common.cuh"
#include "internal.h"
#include "route_norm.cuh"

namespace moe {

// One thread per token.  load32(c0, r) fills r[0..31] with the fp32 accumulators (bit
// patterns) of columns c0 .. c0 + 31 of this token's row; it is called with the same c0 by
// every thread of the warp (the tensor-memory load it may wrap is warp-collective).
// gate_raw is the shared-gate logit w_s . x when the layer has a learned gate.  s_bias and
// s_sel hold the logit bias and the selection-only bias per expert (zeros when absent).
// L is the length of the sorted list, any L >= K (the list's first K entries are the
// selection whatever L is; a shorter list takes fewer and shorter insertions).
template <int L, class Load32>
__device__ __forceinline__ void route_one_token(const RouteParams& p, const float* s_bias,
                                                const float* s_sel, int64_t t, bool valid,
                                                Load32&& load32, float gate_raw) {
  constexpr int EMPTY = 0x7fffffff;
  float bv[L], bz[L];   // selection key and unbiased logit of each slot
  int bi[L];
#pragma unroll
  for (int j = 0; j < L; ++j) { bv[j] = 0.f; bz[j] = 0.f; bi[j] = EMPTY; }
  float zmax = -INFINITY;
  const bool sel = p.selection_bias != nullptr;
  float* lrow = (p.logits && valid) ? p.logits + t * p.N : nullptr;
  // pass 1: keys, logits output, top-8 list
  for (int c0 = 0; c0 < p.N; c0 += 32) {
    uint32_t r[32];
    load32(c0, r);
    float z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = __uint_as_float(r[i]) + (c0 + i < p.N ? s_bias[c0 + i] : 0.f);
    if (lrow) {
      if (c0 + 32 <= p.N && (p.N & 3) == 0 && (reinterpret_cast<uintptr_t>(p.logits) & 15) == 0) {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          *reinterpret_cast<float4*>(lrow + c0 + 4 * v) =
              make_float4(z[4 * v], z[4 * v + 1], z[4 * v + 2], z[4 * v + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i < p.N) lrow[c0 + i] = z[i];
      }
    }
    // Candidates that beat the list's last key as it stands at the start of the chunk:
    // a mask built without branches.  Only those are then inserted, in ascending expert
    // index (a later candidate with an equal key never displaces an earlier one), each
    // checked again against the last key, which rises as the list fills.  The tokens of a
    // warp insert at different candidates, so a branch per candidate would run the
    // insertion for nearly every candidate of the warp; the mask loop runs as often as the
    // warp's busiest token has survivors.
    float cvs[32];
    uint32_t mask = 0;
    const bool full = bi[L - 1] != EMPTY;
    const float thr = bv[L - 1];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      cvs[i] = sel && c0 + i < p.N ? z[i] + s_sel[c0 + i] : z[i];
      if (c0 + i < p.N) {
        zmax = fmaxf(zmax, z[i]);
        if (!full || cvs[i] > thr) mask |= 1u << i;
      }
    }
    while (mask != 0u) {
      const int i = __ffs(mask) - 1;
      mask &= mask - 1u;
      const float cv = cvs[i];
      if (bi[L - 1] == EMPTY || cv > bv[L - 1]) {
        const float cz = z[i];
        const int ci = c0 + i;
        // The kept keys are a descending prefix of the list; the new key goes behind
        // every kept key it does not exceed.  Its place is a count and the shift is per
        // slot, so one insertion is a few dependent steps rather than a chain along the
        // list.
        int pos = 0;
#pragma unroll
        for (int j = 0; j < L; ++j) pos += (bi[j] != EMPTY && !(cv > bv[j])) ? 1 : 0;
#pragma unroll
        for (int j = L - 1; j > 0; --j) {
          const bool shift = j > pos, here = j == pos;
          bv[j] = shift ? bv[j - 1] : (here ? cv : bv[j]);
          bz[j] = shift ? bz[j - 1] : (here ? cz : bz[j]);
          bi[j] = shift ? bi[j - 1] : (here ? ci : bi[j]);
        }
        if (pos == 0) { bv[0] = cv; bz[0] = cz; bi[0] = ci; }
      }
    }
  }
  // scores and weights of the selected experts
  float w[L];
#pragma unroll
  for (int j = 0; j < L; ++j) w[j] = 0.f;
  if (p.norm == MOE_NORM_SOFTMAX_SELECTED) {
    float s = 0.f, msel = bz[0];
#pragma unroll
    for (int j = 1; j < L; ++j)
      if (j < p.K) msel = fmaxf(msel, bz[j]);
#pragma unroll
    for (int j = 0; j < L; ++j)
      if (j < p.K) { w[j] = expf(bz[j] - msel); s += w[j]; }
#pragma unroll
    for (int j = 0; j < L; ++j)
      if (j < p.K) w[j] /= s;
  } else {
    if (p.score == MOE_SCORE_SOFTMAX) {
      // pass 2: softmax denominator over all N experts (unbiased logits)
      const float m = zmax;
      float s = 0.f;
      for (int c0 = 0; c0 < p.N; c0 += 32) {
        uint32_t r[32];
        load32(c0, r);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i < p.N) s += expf(__uint_as_float(r[i]) + s_bias[c0 + i] - m);
      }
#pragma unroll
      for (int j = 0; j < L; ++j)
        if (j < p.K) w[j] = expf(bz[j] - m) / s;
    } else {
#pragma unroll
      for (int j = 0; j < L; ++j)
        if (j < p.K) w[j] = 1.f / (1.f + expf(-bz[j]));
    }
    if (p.norm == MOE_NORM_L1_SELECTED) {
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < L; ++j)
        if (j < p.K) s += w[j];
#pragma unroll
      for (int j = 0; j < L; ++j)
        if (j < p.K) w[j] /= s;
    } else if (p.norm == MOE_NORM_LP_SELECTED) {
      lp_normalise(w, p.K, p.norm_p);
    }
  }
  float shared = 0.f;
  if (p.shared_mode == MOE_SHARED_CONST) {
    shared = p.shared_gain;
  } else if (p.shared_mode == MOE_SHARED_SIGMOID_GATE) {
    shared = 1.f / (1.f + expf(-gate_raw));
  }
  if (valid) {
#pragma unroll
    for (int j = 0; j < L; ++j)
      if (j < p.K) {
        p.topk_idx[t * p.K + j] = bi[j];
        p.topk_w[t * p.K + j] = p.alpha * w[j];
      }
    if (p.shared_coef) p.shared_coef[t] = shared;
  }
}

}  // namespace moe

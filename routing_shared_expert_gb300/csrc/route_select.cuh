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

constexpr int kRouteEmpty = 0x7fffffff;   // expert index of an unused list slot

// Inserts one candidate (key cv, unbiased logit cz, column ci) into the descending list
// when it beats the last kept key.  The kept keys are a descending prefix of the list; the
// new key goes behind every kept key it does not exceed (an equal key of a lower column,
// inserted earlier, stays in front).  Its place is a count and the shift is per slot, so
// one insertion is a few dependent steps rather than a chain along the list.
template <int L>
__device__ __forceinline__ void list_insert(float cv, float cz, int ci, float (&bv)[L],
                                            float (&bz)[L], int (&bi)[L]) {
  if (bi[L - 1] == kRouteEmpty || cv > bv[L - 1]) {
    int pos = 0;
#pragma unroll
    for (int j = 0; j < L; ++j) pos += (bi[j] != kRouteEmpty && !(cv > bv[j])) ? 1 : 0;
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

template <int L>
__device__ __forceinline__ void list_clear(float (&bv)[L], float (&bz)[L], int (&bi)[L]) {
#pragma unroll
  for (int j = 0; j < L; ++j) { bv[j] = 0.f; bz[j] = 0.f; bi[j] = kRouteEmpty; }
}

// Compare-exchange into descending order.
__device__ __forceinline__ void cx_desc(float& a, float& b) {
  const float hi = fmaxf(a, b), lo = fminf(a, b);
  a = hi;
  b = lo;
}

// Sorts v[o .. o + 7] descending (the 19-comparator network for eight inputs).
__device__ __forceinline__ void sort8_desc(float (&v)[32], int o) {
  cx_desc(v[o + 0], v[o + 2]); cx_desc(v[o + 1], v[o + 3]);
  cx_desc(v[o + 4], v[o + 6]); cx_desc(v[o + 5], v[o + 7]);
  cx_desc(v[o + 0], v[o + 4]); cx_desc(v[o + 1], v[o + 5]);
  cx_desc(v[o + 2], v[o + 6]); cx_desc(v[o + 3], v[o + 7]);
  cx_desc(v[o + 0], v[o + 1]); cx_desc(v[o + 2], v[o + 3]);
  cx_desc(v[o + 4], v[o + 5]); cx_desc(v[o + 6], v[o + 7]);
  cx_desc(v[o + 2], v[o + 4]); cx_desc(v[o + 3], v[o + 5]);
  cx_desc(v[o + 1], v[o + 4]); cx_desc(v[o + 3], v[o + 6]);
  cx_desc(v[o + 1], v[o + 2]); cx_desc(v[o + 3], v[o + 4]); cx_desc(v[o + 5], v[o + 6]);
}

// v[a .. a + 7] <- the eight largest of the two descending runs v[a ..] and v[b ..], in
// descending order: the pairwise maxima of one run against the other reversed form a
// bitonic sequence holding the eight largest, which three half-cleaner stages sort.
__device__ __forceinline__ void merge_top8_desc(float (&v)[32], int a, int b) {
#pragma unroll
  for (int i = 0; i < 8; ++i) v[a + i] = fmaxf(v[a + i], v[b + 7 - i]);
#pragma unroll
  for (int i = 0; i < 4; ++i) cx_desc(v[a + i], v[a + i + 4]);
#pragma unroll
  for (int i = 0; i < 8; i += 4) { cx_desc(v[a + i], v[a + i + 2]); cx_desc(v[a + i + 1], v[a + i + 3]); }
#pragma unroll
  for (int i = 0; i < 8; i += 2) cx_desc(v[a + i], v[a + i + 1]);
}

// The L-th largest (L <= 8) of 32 values, none NaN.
template <int L>
__device__ __forceinline__ float lth_largest32(float (&v)[32]) {
  static_assert(L >= 1 && L <= 8, "list length");
#pragma unroll
  for (int o = 0; o < 32; o += 8) sort8_desc(v, o);
  merge_top8_desc(v, 0, 8);
  merge_top8_desc(v, 16, 24);
  merge_top8_desc(v, 0, 16);
  return v[L - 1];
}

// Pass 1 over one 32-column chunk: the logits z (+ the logit bias), the logits output, the
// running maximum logit and, per column slot, the largest key (z + the selection-only
// bias).  BIAS / SEL: the layer has that bias; FULL: every column of the chunk is below N
// (no range checks).  NaN keys are ignored by the maxima.
template <bool BIAS, bool SEL, bool FULL>
__device__ __forceinline__ void chunk_pass1(const RouteParams& p, const float* s_bias,
                                            const float* s_sel, int c0, const uint32_t (&r)[32],
                                            float* lrow, float (&slot_max)[32], float& zmax) {
  float z[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    z[i] = __uint_as_float(r[i]);
    if (BIAS && (FULL || c0 + i < p.N)) z[i] += s_bias[c0 + i];
  }
  if (lrow) {
    if (FULL && (p.N & 3) == 0 && (reinterpret_cast<uintptr_t>(p.logits) & 15) == 0) {
#pragma unroll
      for (int v = 0; v < 8; ++v)
        *reinterpret_cast<float4*>(lrow + c0 + 4 * v) =
            make_float4(z[4 * v], z[4 * v + 1], z[4 * v + 2], z[4 * v + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (FULL || c0 + i < p.N) lrow[c0 + i] = z[i];
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (FULL || c0 + i < p.N) {
      zmax = fmaxf(zmax, z[i]);
      slot_max[i] = fmaxf(slot_max[i], SEL ? z[i] + s_sel[c0 + i] : z[i]);
    }
}

// Pass 2 over one chunk: the candidates whose key is not below thr, inserted in ascending
// column order.  Their keys and logits are staged in this thread's shared-memory scratch
// rows (entry i at i * stride; the key row only when it differs from the logit): the
// candidates are picked by a run-time index, which on registers would place the chunk in
// local memory.  The tokens of a warp insert at different candidates, so the loop runs
// over a mask rather than branching per candidate; it runs as often as the warp's busiest
// token has candidates.
template <int L, bool BIAS, bool SEL, bool FULL>
__device__ __forceinline__ void chunk_pass2(const RouteParams& p, const float* s_bias,
                                            const float* s_sel, int c0, const uint32_t (&r)[32],
                                            float thr, float* s_cv, float* s_z, int stride,
                                            float (&bv)[L], float (&bz)[L], int (&bi)[L]) {
  uint32_t mask = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float z = __uint_as_float(r[i]);
    if (BIAS && (FULL || c0 + i < p.N)) z += s_bias[c0 + i];
    float cv = z;
    if (SEL && (FULL || c0 + i < p.N)) cv = z + s_sel[c0 + i];
    s_z[i * stride] = z;
    if (SEL) s_cv[i * stride] = cv;
    if ((FULL || c0 + i < p.N) && !(cv < thr)) mask |= 1u << i;
  }
  while (mask != 0u) {
    const int i = __ffs(mask) - 1;
    mask &= mask - 1u;
    const float z = s_z[i * stride];
    list_insert<L>(SEL ? s_cv[i * stride] : z, z, c0 + i, bv, bz, bi);
  }
}

template <int L, bool BIAS, bool SEL, class Load32>
__device__ __forceinline__ void list_columns_impl(const RouteParams& p, const float* s_bias,
                                                  const float* s_sel, int c_lo, int c_hi,
                                                  float* lrow, float* s_cv, float* s_z,
                                                  int stride, Load32&& load32, float (&bv)[L],
                                                  float (&bz)[L], int (&bi)[L], float& zmax) {
  float slot_max[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) slot_max[i] = -INFINITY;
  for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
    uint32_t r[32];
    load32(c0, r);
    if (c0 + 32 <= p.N)
      chunk_pass1<BIAS, SEL, true>(p, s_bias, s_sel, c0, r, lrow, slot_max, zmax);
    else
      chunk_pass1<BIAS, SEL, false>(p, s_bias, s_sel, c0, r, lrow, slot_max, zmax);
  }
  const float thr = lth_largest32<L>(slot_max);
  for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
    uint32_t r[32];
    load32(c0, r);
    if (c0 + 32 <= p.N)
      chunk_pass2<L, BIAS, SEL, true>(p, s_bias, s_sel, c0, r, thr, s_cv, s_z, stride, bv, bz, bi);
    else
      chunk_pass2<L, BIAS, SEL, false>(p, s_bias, s_sel, c0, r, thr, s_cv, s_z, stride, bv, bz, bi);
  }
}

// Selection over the columns [c_lo, c_hi) (c_lo a multiple of 32) of one token: the keys
// z (+ the selection-only bias), the logits output row (when lrow is given), the maximum
// logit and the sorted list.  load32(c0, r) fills r[0..31] with the fp32 accumulators (bit
// patterns) of columns c0 .. c0 + 31; every thread of the warp calls it with the same c0
// (the tensor-memory load it may wrap is warp-collective).  s_cv and s_z are this thread's
// 32-entry scratch rows in shared memory, entry i at index i * stride.
//
// Two passes.  The first keeps, for each of the 32 column slots of a chunk, the largest
// key over the chunks; those are maxima of distinct columns, so the L-th largest of them
// is at most the L-th largest key overall, and no column below it can be selected.  The
// second pass inserts, in ascending column order, only the columns whose key is not below
// that threshold (a handful), so the result is the selection over all columns with the
// lower index first on equal keys.  A single pass would insert every candidate of the
// first chunk (the list starts empty), each insertion a chain of dependent steps.  The
// layer's biases pick one of four compiled variants, so a layer without them issues no
// instruction for them.
template <int L, class Load32>
__device__ __forceinline__ void list_columns(const RouteParams& p, const float* s_bias,
                                             const float* s_sel, int c_lo, int c_hi, float* lrow,
                                             float* s_cv, float* s_z, int stride, Load32&& load32,
                                             float (&bv)[L], float (&bz)[L], int (&bi)[L],
                                             float& zmax) {
  const bool bias = p.router_bias != nullptr, sel = p.selection_bias != nullptr;
  if (bias) {
    if (sel)
      list_columns_impl<L, true, true>(p, s_bias, s_sel, c_lo, c_hi, lrow, s_cv, s_z, stride,
                                       load32, bv, bz, bi, zmax);
    else
      list_columns_impl<L, true, false>(p, s_bias, s_sel, c_lo, c_hi, lrow, s_cv, s_z, stride,
                                        load32, bv, bz, bi, zmax);
  } else {
    if (sel)
      list_columns_impl<L, false, true>(p, s_bias, s_sel, c_lo, c_hi, lrow, s_cv, s_z, stride,
                                        load32, bv, bz, bi, zmax);
    else
      list_columns_impl<L, false, false>(p, s_bias, s_sel, c_lo, c_hi, lrow, s_cv, s_z, stride,
                                         load32, bv, bz, bi, zmax);
  }
}

// Sum of exp(z - m) over the columns [c_lo, c_hi) below N (the softmax denominator's part).
template <bool BIAS, class Load32>
__device__ __forceinline__ float exp_sum_impl(const RouteParams& p, const float* s_bias, int c_lo,
                                              int c_hi, float m, Load32&& load32) {
  float s = 0.f;
  for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
    uint32_t r[32];
    load32(c0, r);
    if (c0 + 32 <= p.N) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        s += expf(__uint_as_float(r[i]) + (BIAS ? s_bias[c0 + i] : 0.f) - m);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (c0 + i < p.N) s += expf(__uint_as_float(r[i]) + (BIAS ? s_bias[c0 + i] : 0.f) - m);
    }
  }
  return s;
}

template <class Load32>
__device__ __forceinline__ float exp_sum_columns(const RouteParams& p, const float* s_bias,
                                                 int c_lo, int c_hi, float m, Load32&& load32) {
  return p.router_bias ? exp_sum_impl<true>(p, s_bias, c_lo, c_hi, m, load32)
                       : exp_sum_impl<false>(p, s_bias, c_lo, c_hi, m, load32);
}

// Whether the scores need the softmax denominator over all N experts.
__device__ __forceinline__ bool needs_full_softmax(const RouteParams& p) {
  return p.norm != MOE_NORM_SOFTMAX_SELECTED && p.score == MOE_SCORE_SOFTMAX;
}

// Scores, weights and coefficients of one token from its final list: bz / bi the unbiased
// logits and experts of the selected entries (the first K), m and s the maximum logit
// over all N and the sum of exp(z - m) (used by softmax scores over all experts).
template <int L>
__device__ __forceinline__ void finish_token(const RouteParams& p, int64_t t, bool valid,
                                             const float (&bz)[L], const int (&bi)[L], float m,
                                             float s_all, float gate_raw) {
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
#pragma unroll
      for (int j = 0; j < L; ++j)
        if (j < p.K) w[j] = expf(bz[j] - m) / s_all;
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

// One thread per token over all N columns (s_cv, s_z, stride: its scratch rows, as for
// list_columns).  gate_raw is the shared-gate logit w_s . x when the layer has a learned
// gate.  s_bias and s_sel hold the logit bias and the
// selection-only bias per expert (zeros when absent).  L is the length of the sorted
// list, any L >= K (the list's first K entries are the selection whatever L is; a shorter
// list takes fewer and shorter insertions).
template <int L, class Load32>
__device__ __forceinline__ void route_one_token(const RouteParams& p, const float* s_bias,
                                                const float* s_sel, int64_t t, bool valid,
                                                float* s_cv, float* s_z, int stride,
                                                Load32&& load32, float gate_raw) {
  float bv[L], bz[L];   // selection key and unbiased logit of each slot
  int bi[L];
  list_clear<L>(bv, bz, bi);
  float zmax = -INFINITY;
  float* lrow = (p.logits && valid) ? p.logits + t * p.N : nullptr;
  list_columns<L>(p, s_bias, s_sel, 0, p.N, lrow, s_cv, s_z, stride, load32, bv, bz, bi, zmax);
  const float s_all = needs_full_softmax(p) ? exp_sum_columns(p, s_bias, 0, p.N, zmax, load32) : 0.f;
  finish_token<L>(p, t, valid, bz, bi, zmax, s_all, gate_raw);
}

}  // namespace moe

// L_p normalisation of a token's selected weights (Appendix E, Table 52, MegaBlocks row):
// w_k <- w_k / (sum_j w_j^p)^(1/p).  The weights are scaled by their maximum first, so every
// power lies in (0, 1] with the largest term exactly 1: no underflow for large p or small
// scores.  Shared by the SIMT and tensor-core routers.
#pragma once

#include "internal.h"

namespace moe {

template <int KMAX>
__device__ __forceinline__ void lp_normalise(float (&w)[KMAX], int K, float p) {
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
    if (k < K) m = fmaxf(m, w[k]);
  if (!(m > 0.f)) return;
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
    if (k < K) s += powf(w[k] / m, p);
  const float n = m * powf(s, 1.f / p);
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
    if (k < K) w[k] /= n;
}

}  // namespace moe

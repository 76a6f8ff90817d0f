// Backward pass of the layer with the router coefficients held fixed: the expert-path
// Jacobian of the backward study of "Section 21: Merging Routed and Shared Expert
// Activations" (Figure 70 (b) "router coefficients fixed", (c) the routed and shared
// down-projection weight gradients), for the SwiGLU experts of "Section 20: One Shared
// Expert Is All You Need", Eq. 74, merged by Eq. 80.
//
// Given dy = dL/dy, per kept route (t, k) of expert e with coefficient r = r_tk (and per
// token for the shared expert with s_t):
//   gf = r dy_t;  [a | b] = x_t [W_g^e | W_u^e]^T (recomputed);  h = SiLU(a) b
//   dh = gf W_d^e;  da = dh b SiLU'(a);  db = dh SiLU(a)
//   dx_t += da W_g^e + db W_u^e;  dW_d^e += gf^T h;  dW_g^e += da^T x_t;  dW_u^e += db^T x_t
// Dropped routes carry no gradient.  The routed rows are laid out per expert segment,
// each padded to a multiple of 64 rows with zero rows, so that the weight-gradient GEMMs
// (K = the segment's rows) need no masking; the padded start of expert e is
// seg_pad[e] = sum_{i<e} ceil(C_i^keep / 64) * 64.
//
// Kernels here: the padded offsets, the gather of x and of the scaled upstream gradient
// into the padded rows, the scaled upstream gradient of the shared expert, and the
// fixed-order sum of each token's route gradients and shared gradient into dx.  The GEMMs
// are in gemm_bwd.cu.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__global__ void pad_offsets_kernel(const int32_t* counts_keep, int N, int32_t* seg_pad) {
  if (threadIdx.x == 0) {
    int32_t o = 0;
    for (int e = 0; e < N; ++e) {
      seg_pad[e] = o;
      o += (counts_keep[e] + 63) / 64 * 64;
    }
    seg_pad[N] = o;
  }
}

// One warp per padded row: the row of x and the scaled upstream gradient of its route,
// or zeros for a padding row.
__global__ void __launch_bounds__(256) bwd_rows_kernel(BwdRowsParams p) {
  __shared__ int32_t s_pad[kMaxExperts + 1];
  for (int i = threadIdx.x; i <= p.N; i += blockDim.x) s_pad[i] = p.seg_pad[i];
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t pp = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (pp >= s_pad[p.N]) return;
  int lo = 0, hi = p.N;   // s_pad[lo] <= pp < s_pad[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pad[mid] <= pp) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int64_t local = pp - s_pad[e];
  uint4* xo = reinterpret_cast<uint4*>(p.x_pad + pp * p.d);
  uint4* go = reinterpret_cast<uint4*>(p.gf + pp * p.d);
  const int vecs = p.d / 8;
  if (local >= p.counts_keep[e]) {
    for (int v = lane; v < vecs; v += 32) {
      xo[v] = make_uint4(0, 0, 0, 0);
      go[v] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const int64_t pos = p.offsets[e] + local;
  const int32_t t = p.perm_src[pos];
  if (t < 0 || t >= p.T) {
    if (lane == 0) set_status(p.status, MOE_ERR_DEVICE_BOUNDS);
    return;
  }
  float r = 0.f;
  bool found = false;
  for (int k = 0; k < p.K; ++k)
    if (p.route_pos[static_cast<int64_t>(t) * p.K + k] == pos) {
      r = p.topk_w[static_cast<int64_t>(t) * p.K + k];
      found = true;
    }
  if (!found) {
    if (lane == 0) set_status(p.status, MOE_ERR_DEVICE_BOUNDS);
    return;
  }
  const uint4* xi = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.x) + static_cast<int64_t>(t) * p.d);
  const float4* dyi = reinterpret_cast<const float4*>(p.dy + static_cast<int64_t>(t) * p.d);
  for (int v = lane; v < vecs; v += 32) {
    xo[v] = xi[v];
    const float4 a = dyi[2 * v], b = dyi[2 * v + 1];
    go[v] = make_uint4(pack_bf16x2(r * a.x, r * a.y), pack_bf16x2(r * a.z, r * a.w),
                       pack_bf16x2(r * b.x, r * b.y), pack_bf16x2(r * b.z, r * b.w));
  }
}

// gs[t] = s_t dy_t (bf16), one warp per token.
__global__ void __launch_bounds__(256) shared_scale_kernel(const float* dy, const float* s, int64_t T,
                                                           int d, __nv_bfloat16* gs) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (t >= T) return;
  const float c = s[t];
  const float4* dyi = reinterpret_cast<const float4*>(dy + t * d);
  uint4* o = reinterpret_cast<uint4*>(gs + t * d);
  for (int v = lane; v < d / 8; v += 32) {
    const float4 a = dyi[2 * v], b = dyi[2 * v + 1];
    o[v] = make_uint4(pack_bf16x2(c * a.x, c * a.y), pack_bf16x2(c * a.z, c * a.w),
                      pack_bf16x2(c * b.x, c * b.y), pack_bf16x2(c * b.z, c * b.w));
  }
}

// dx_t = sum over kept slots k (in slot order) of the route's dx row, plus the shared
// expert's dx row; one CTA per token, 4 fp32 per thread.
__global__ void __launch_bounds__(256) dx_combine_kernel(BwdCombineParams p) {
  const int64_t t = blockIdx.x;
  __shared__ int64_t s_row[kMaxTopK];
  if (threadIdx.x < p.K) {
    const int k = threadIdx.x;
    const int32_t pos = p.route_pos[t * p.K + k];
    int64_t row = -1;
    if (pos >= 0) {
      const int e = p.topk_idx[t * p.K + k];
      if (e < 0 || e >= p.N || pos < p.offsets[e] || pos >= p.offsets[e + 1])
        set_status(p.status, MOE_ERR_DEVICE_BOUNDS);
      else
        row = p.seg_pad[e] + (pos - p.offsets[e]);
    }
    s_row[k] = row;
  }
  __syncthreads();
  for (int c = threadIdx.x * 4; c < p.d; c += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < p.K; ++k) {
      if (s_row[k] < 0) continue;
      const float4 v = *reinterpret_cast<const float4*>(p.dxr + s_row[k] * p.d + c);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (p.dxs) {
      const float4 v = *reinterpret_cast<const float4*>(p.dxs + t * p.d + c);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    *reinterpret_cast<float4*>(p.dx + t * p.d + c) = acc;
  }
}

}  // namespace

cudaError_t launch_pad_offsets(const int32_t* counts_keep, int N, int32_t* seg_pad, cudaStream_t s) {
  pad_offsets_kernel<<<1, 32, 0, s>>>(counts_keep, N, seg_pad);
  return cudaGetLastError();
}

cudaError_t launch_bwd_rows(const BwdRowsParams& p, int64_t rows_cap, cudaStream_t s) {
  if (rows_cap <= 0) return cudaSuccess;
  bwd_rows_kernel<<<static_cast<unsigned>((rows_cap + 7) / 8), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_shared_scale(const float* dy, const float* sc, int64_t T, int d, __nv_bfloat16* gs,
                                cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  shared_scale_kernel<<<static_cast<unsigned>((T + 7) / 8), 256, 0, s>>>(dy, sc, T, d, gs);
  return cudaGetLastError();
}

cudaError_t launch_dx_combine(const BwdCombineParams& p, cudaStream_t s) {
  if (p.T <= 0) return cudaSuccess;
  dx_combine_kernel<<<static_cast<unsigned>(p.T), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe

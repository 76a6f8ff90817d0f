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

// Offsets of the segments padded to multiples of 64 rows: one warp, an exclusive prefix
// sum 32 experts at a time.
__global__ void pad_offsets_kernel(const int32_t* counts_keep, int N, int32_t* seg_pad) {
  const int lane = threadIdx.x;
  int32_t run = 0;
  for (int base = 0; base < N; base += 32) {
    const int e = base + lane;
    const int32_t v = e < N ? (counts_keep[e] + 63) / 64 * 64 : 0;
    int32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (e < N) seg_pad[e] = run + incl - v;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) seg_pad[N] = run;
}

// One warp per token: the row of x and the upstream gradient dy (as bf16, unscaled) are
// read once and written to the padded rows of all of the token's kept routes, with each
// route's coefficient r (applied in the GEMM epilogues).  Reading per token rather than
// per padded row fetches x and dy once instead of once per route.
__global__ void __launch_bounds__(256) bwd_rows_kernel(BwdRowsParams p) {
  __shared__ int32_t s_pad[kMaxExperts + 1];
  for (int i = threadIdx.x; i <= p.N; i += blockDim.x) s_pad[i] = p.seg_pad[i];
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (t >= p.T) return;
  int64_t dst[kMaxTopK];   // padded row of slot k, or -1 (dropped or no slot)
#pragma unroll
  for (int k = 0; k < kMaxTopK; ++k) {
    dst[k] = -1;
    if (k < p.K) {
      const int32_t pos = p.route_pos[t * p.K + k];
      if (pos < 0) continue;
      const int32_t e = p.topk_idx[t * p.K + k];
      if (e < 0 || e >= p.N) {
        if (lane == 0) set_status(p.status, MOE_ERR_DEVICE_BOUNDS);
        continue;
      }
      const int64_t local = static_cast<int64_t>(pos) - p.offsets[e];
      const int64_t row = s_pad[e] + local;
      if (local < 0 || local >= p.counts_keep[e] || row >= s_pad[e + 1] || row < 0 ||
          row >= p.rows_cap) {
        if (lane == 0) set_status(p.status, MOE_ERR_DEVICE_BOUNDS);
        continue;
      }
      dst[k] = row;
      if (lane == 0) p.r_pad[dst[k]] = p.topk_w[t * p.K + k];
    }
  }
  const int vecs = p.d / 8;
  const uint4* __restrict__ xi =
      reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.x) + t * p.d);
  const float4* __restrict__ dyi = reinterpret_cast<const float4*>(p.dy + t * p.d);
  uint4* __restrict__ xo = reinterpret_cast<uint4*>(p.x_pad);
  uint4* __restrict__ go = reinterpret_cast<uint4*>(p.gf);
  for (int v = lane; v < vecs; v += 32) {
    const uint4 xv = xi[v];
    const float4 a = dyi[2 * v], b = dyi[2 * v + 1];
    const uint4 gv = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k)
      if (dst[k] >= 0) {
        xo[dst[k] * vecs + v] = xv;
        go[dst[k] * vecs + v] = gv;
      }
  }
}

// The padding rows of each expert's segment (from its kept count up to the next multiple
// of 64): zeros and r = 0.  One warp per (expert, padding row) pair.
__global__ void __launch_bounds__(256) bwd_pad_rows_kernel(BwdRowsParams p) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  const int e = static_cast<int>(w / 64);
  if (e >= p.N) return;
  const int32_t kept = p.counts_keep[e];
  const int64_t row = static_cast<int64_t>(p.seg_pad[e]) + kept + (w % 64);
  if (kept < 0 || p.seg_pad[e] < 0 || row >= p.seg_pad[e + 1] || row >= p.rows_cap) return;
  const int vecs = p.d / 8;
  uint4* xo = reinterpret_cast<uint4*>(p.x_pad + row * p.d);
  uint4* go = reinterpret_cast<uint4*>(p.gf + row * p.d);
  for (int v = lane; v < vecs; v += 32) {
    xo[v] = make_uint4(0, 0, 0, 0);
    go[v] = make_uint4(0, 0, 0, 0);
  }
  if (lane == 0) p.r_pad[row] = 0.f;
}

// gs[t] = dy_t (bf16) and s_pad[t] = s_t (0 for the rows up to T rounded to 64), one
// warp per row.
__global__ void __launch_bounds__(256) shared_scale_kernel(const float* dy, const float* s, int64_t T,
                                                           int64_t t_pad, int d, __nv_bfloat16* gs,
                                                           float* s_pad) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (t >= t_pad) return;
  if (t >= T) {
    if (lane == 0) s_pad[t] = 0.f;
    return;
  }
  if (lane == 0) s_pad[t] = s[t];
  const float4* dyi = reinterpret_cast<const float4*>(dy + t * d);
  uint4* o = reinterpret_cast<uint4*>(gs + t * d);
  for (int v = lane; v < d / 8; v += 32) {
    const float4 a = dyi[2 * v], b = dyi[2 * v + 1];
    o[v] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                      pack_bf16x2(b.z, b.w));
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
    if (p.dxz) {   // through the router: dz W_r
      const float4 v = *reinterpret_cast<const float4*>(p.dxz + t * p.d + c);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (p.du) {    // through a learned shared gate: du w_s
      const float u = p.du[t];
      const float4 w = make_float4(to_f32(p.gate_w[c]), to_f32(p.gate_w[c + 1]),
                                   to_f32(p.gate_w[c + 2]), to_f32(p.gate_w[c + 3]));
      acc.x += u * w.x; acc.y += u * w.y; acc.z += u * w.z; acc.w += u * w.w;
    }
    *reinterpret_cast<float4*>(p.dx + t * p.d + c) = acc;
  }
}

// Gradient through the router coefficients, one warp per token (Table 52 rules; the
// selection held fixed): dr_k = dy . f_k = sum over tiles of dh_u . h of the route's row
// (zero for a dropped route), dw = alpha dr, then
//   softmax over the selected logits:  dz_S = w (dw - sum_k w_k dw_k)
//   otherwise dq_S from the rule (none: dw; L1: (dw - sum w dw) / sum q_S;
//   L_p: dw / n - (sum w dw) w^(p-1) / n) and dz = q (dq - sum_S q dq) for softmax
//   scores, dz_S = dq_S q_S (1 - q_S) for sigmoid scores.
// A learned shared gate s = sigma(u) adds du = (dy . g) s (1 - s), dy . g likewise from
// the shared expert's tiles.
__global__ void __launch_bounds__(256) router_bwd_kernel(RouterBwdParams p) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (t >= p.T) return;
  const float* z = p.logits + t * p.N;
  // coefficient gradients of the K slots
  float dw[kMaxTopK], zs[kMaxTopK];
  int si[kMaxTopK];
#pragma unroll
  for (int k = 0; k < kMaxTopK; ++k) {
    dw[k] = 0.f;
    zs[k] = 0.f;
    si[k] = -1;
    if (k < p.K) {
      const int e = p.topk_idx[t * p.K + k];
      si[k] = e;
      zs[k] = (e >= 0 && e < p.N) ? z[e] : 0.f;
      const int32_t pos = p.route_pos[t * p.K + k];
      if (pos >= 0 && e >= 0 && e < p.N) {
        const int64_t row = p.seg_pad[e] + (pos - p.offsets[e]);
        float acc = 0.f;
        for (int n = 0; n < p.nt; ++n) acc += p.dot_part[row * p.nt + n];
        dw[k] = p.alpha * acc;
      }
    }
  }
  float dzS[kMaxTopK];
  float c = 0.f;          // softmax scores: sum_S q dq
  float m = -INFINITY, sum = 0.f;
  const bool soft = p.score == MOE_SCORE_SOFTMAX;
  if (p.norm == MOE_NORM_SOFTMAX_SELECTED) {
    float ms = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k)
      if (k < p.K) ms = fmaxf(ms, zs[k]);
    float w[kMaxTopK], tot = 0.f, wdw = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
      w[k] = k < p.K ? expf(zs[k] - ms) : 0.f;
      tot += w[k];
    }
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
      w[k] /= tot;
      wdw += w[k] * dw[k];
    }
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) dzS[k] = k < p.K ? w[k] * (dw[k] - wdw) : 0.f;
  } else {
    float q[kMaxTopK];
    if (soft) {
      for (int j = lane; j < p.N; j += 32) m = fmaxf(m, z[j]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      for (int j = lane; j < p.N; j += 32) sum += expf(z[j] - m);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    }
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k)
      q[k] = k < p.K ? (soft ? expf(zs[k] - m) / sum : 1.f / (1.f + expf(-zs[k]))) : 0.f;
    float dq[kMaxTopK];
    if (p.norm == MOE_NORM_NONE) {
#pragma unroll
      for (int k = 0; k < kMaxTopK; ++k) dq[k] = dw[k];
    } else {
      float S = 0.f;
      if (p.norm == MOE_NORM_L1_SELECTED) {
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k) S += q[k];
      } else {   // L_p: n = (sum q^p)^(1/p), scaled by the largest q
        float mx = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k) mx = fmaxf(mx, q[k]);
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
          if (k < p.K) acc += powf(q[k] / mx, p.norm_p);
        S = mx * powf(acc, 1.f / p.norm_p);
      }
      float w[kMaxTopK], wdw = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxTopK; ++k) {
        w[k] = q[k] / S;
        wdw += w[k] * dw[k];
      }
#pragma unroll
      for (int k = 0; k < kMaxTopK; ++k) {
        if (p.norm == MOE_NORM_L1_SELECTED)
          dq[k] = (dw[k] - wdw) / S;
        else
          dq[k] = k < p.K ? dw[k] / S - wdw * powf(w[k], p.norm_p - 1.f) / S : 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
      if (soft) c += q[k] * dq[k];
      dzS[k] = k < p.K ? (soft ? q[k] * dq[k] : dq[k] * q[k] * (1.f - q[k])) : 0.f;
    }
  }
  // dz over all columns: selected ones get their slot term; with softmax scores every
  // column also gets -q_j c
  __nv_bfloat16* out = p.dz + t * p.n128;
  for (int j = lane; j < p.n128; j += 32) {
    float v = 0.f;
    if (j < p.N) {
#pragma unroll
      for (int k = 0; k < kMaxTopK; ++k)
        if (k < p.K && si[k] == j) v += dzS[k];
      if (soft && p.norm != MOE_NORM_SOFTMAX_SELECTED) v -= expf(z[j] - m) / sum * c;
    }
    out[j] = __float2bfloat16(v);
  }
  if (p.du != nullptr && lane == 0) {
    float ds = 0.f;
    for (int n = 0; n < p.nt_s; ++n) ds += p.dot_part_s[t * p.nt_s + n];
    const float s = p.shared_coef[t];
    p.du[t] = ds * s * (1.f - s);
  }
}

// dw_s = sum_t du_t x_t: partial sums over 64 chunks of tokens, then their ordered sum.
__global__ void __launch_bounds__(256) dws_partial_kernel(const float* du, const __nv_bfloat16* x,
                                                          int64_t T, int d, float* part) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d) return;
  const int64_t per = (T + gridDim.y - 1) / gridDim.y;
  const int64_t t0 = blockIdx.y * per;
  const int64_t t1 = t0 + per < T ? t0 + per : T;
  float acc = 0.f;
  for (int64_t t = t0; t < t1; ++t) acc += du[t] * __bfloat162float(x[t * d + i]);
  part[static_cast<int64_t>(blockIdx.y) * d + i] = acc;
}

__global__ void __launch_bounds__(256) dws_final_kernel(const float* part, int chunks, int d, float* dws) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d) return;
  float acc = 0.f;
  for (int c = 0; c < chunks; ++c) acc += part[static_cast<int64_t>(c) * d + i];
  dws[i] = acc;
}

}  // namespace

cudaError_t launch_router_bwd(const RouterBwdParams& p, cudaStream_t s) {
  if (p.T <= 0) return cudaSuccess;
  router_bwd_kernel<<<static_cast<unsigned>((p.T + 7) / 8), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dws(const float* du, const void* x, int64_t T, int d, float* part, float* dws,
                       cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((d + 255) / 256), kDwsChunks);
  dws_partial_kernel<<<grid, 256, 0, s>>>(du, static_cast<const __nv_bfloat16*>(x), T, d, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dws_final_kernel<<<static_cast<unsigned>((d + 255) / 256), 256, 0, s>>>(part, kDwsChunks, d, dws);
  return cudaGetLastError();
}

cudaError_t launch_pad_offsets(const int32_t* counts_keep, int N, int32_t* seg_pad, cudaStream_t s) {
  pad_offsets_kernel<<<1, 32, 0, s>>>(counts_keep, N, seg_pad);
  return cudaGetLastError();
}

cudaError_t launch_bwd_rows(const BwdRowsParams& p, cudaStream_t s) {
  if (p.T > 0) {
    bwd_rows_kernel<<<static_cast<unsigned>((p.T + 7) / 8), 256, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  bwd_pad_rows_kernel<<<static_cast<unsigned>(p.N * 8), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_shared_scale(const float* dy, const float* sc, int64_t T, int64_t t_pad, int d,
                                __nv_bfloat16* gs, float* s_pad, cudaStream_t s) {
  if (t_pad <= 0) return cudaSuccess;
  shared_scale_kernel<<<static_cast<unsigned>((t_pad + 7) / 8), 256, 0, s>>>(dy, sc, T, t_pad, d, gs,
                                                                            s_pad);
  return cudaGetLastError();
}

cudaError_t launch_dx_combine(const BwdCombineParams& p, cudaStream_t s) {
  if (p.T <= 0) return cudaSuccess;
  dx_combine_kernel<<<static_cast<unsigned>(p.T), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe

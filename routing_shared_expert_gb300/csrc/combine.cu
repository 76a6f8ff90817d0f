// Weighted combine, Section 21 "Merging Routed and Shared Expert Activations", Eq. 80:
//   y_t = sum_{k : route kept} r_{t,k} f[route_pos_{t,k}] + s_t g_t
// Dropped routes add nothing and the kept coefficients are not renormalised
// (Section 10.3: combine masks the tail-dropped routes).
//
// f and g are fp32, or fp16 under the fp16 intermediate of bf16 layers, where they hold
// f 2^-h_scale_log2 (the scale is folded into the coefficients here: exact, a power of
// two).  Rounding them to bf16 instead would cost about 2^-9 of the largest |f| per
// element, most of a 1.5e-2 relative budget; fp16 costs 2^-12.
// One CTA per token; each thread owns 16 bytes of a row (4 fp32) and
// accumulates in fp32 in a fixed order (slot 0..K-1, then the shared term), so
// the result does not depend on scheduling.  Loads and stores are 16-byte vectors;
// the pieces of all kept routes and of g are first requested into L2 together, so
// the in-order loads that follow do not each wait out a DRAM round trip.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

template <typename T>
struct Vec;
template <>
struct Vec<__half> {
  static constexpr int N = 8;
  __device__ static void load(const __half* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 b = *reinterpret_cast<const __half2*>(&w[i]);
      const float2 f = __half22float2(b);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float (&v)[4]) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
  }
};

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <typename T>
__global__ void __launch_bounds__(1024) combine_kernel(CombineParams p) {
  constexpr int V = Vec<T>::N;
  const int64_t t = blockIdx.x;
  __shared__ int s_pos[kMaxTopK];
  __shared__ float s_w[kMaxTopK];
  if (threadIdx.x < p.K) {
    int pos = p.route_pos[t * p.K + threadIdx.x];
    if (pos >= p.f_rows) {
      set_status(p.status, MOE_ERR_DEVICE_BOUNDS);
      pos = -1;
    }
    s_pos[threadIdx.x] = pos;
    s_w[threadIdx.x] = p.topk_w[t * p.K + threadIdx.x] * p.out_scale;
  }
  __syncthreads();
  const T* f = static_cast<const T*>(p.f);
  const T* g = static_cast<const T*>(p.g);
  const float s = (g != nullptr && p.shared_coef != nullptr) ? p.shared_coef[t] * p.out_scale : 0.f;
  for (int c = threadIdx.x * V; c < p.d; c += blockDim.x * V) {
    for (int k = 0; k < p.K; ++k)
      if (s_pos[k] >= 0) prefetch_l2(f + static_cast<int64_t>(s_pos[k]) * p.d + c);
    if (g != nullptr && p.shared_coef != nullptr) prefetch_l2(g + t * p.d + c);
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    for (int k = 0; k < p.K; ++k) {
      const int pos = s_pos[k];
      if (pos < 0) continue;
      float v[V];
      Vec<T>::load(f + static_cast<int64_t>(pos) * p.d + c, v);
      const float w = s_w[k];
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(w, v[i], acc[i]);
    }
    if (g != nullptr && p.shared_coef != nullptr) {
      float v[V];
      Vec<T>::load(g + t * p.d + c, v);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(s, v[i], acc[i]);
    }
    float* y = p.y + t * p.d + c;
#pragma unroll
    for (int i = 0; i < V; i += 4)
      *reinterpret_cast<float4*>(y + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
  }
}

template <typename T>
cudaError_t launch_t(const CombineParams& p, cudaStream_t s) {
  constexpr int V = Vec<T>::N;
  int threads = (p.d / V + 31) / 32 * 32;
  if (threads > 1024) threads = 1024;
  if (threads < 32) threads = 32;
  combine_kernel<T><<<static_cast<unsigned>(p.T), threads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  return p.f16 ? launch_t<__half>(p, s) : launch_t<float>(p, s);
}

}  // namespace moe

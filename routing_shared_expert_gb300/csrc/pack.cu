// Packing of a bf16 down-projection tensor into the fp16 layout read by the expert GEMMs
// of the fp16 intermediate format (MOE_H_F16).
//
// The down projection f = h W_d (Section 20 "One Shared Expert Is All You Need", Eq. 74)
// runs on the tensor cores with both operands of one type.  Holding h in fp16 (11
// significant bits) instead of bf16 (8) cuts the rounding error of the intermediate
// eightfold at the same MMA rate, so W_d is given to the MMA in fp16 too.  A bf16 weight
// has 8 significant bits and fits fp16's 11 exactly as long as its exponent lies in
// fp16's range, so the tensor is scaled by one power of two 2^k chosen from its largest
// magnitude (max |W| 2^k in [2^14, 2^15)): every bf16 value above max |W| 2^-31 or so
// converts exactly, and the GEMM epilogue multiplies the fp32 accumulator by 2^-k.
//
// Buffer: a PackHeader in the first 256 bytes (magic, max |W|, k, 2^-k, element count,
// flags), then the fp16 values in the order of the input.  Two grid-stride kernels: a
// max-magnitude reduction into the header, then the scaled conversion.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kPackThreads = 256;

__device__ __forceinline__ void fold(float v, float& m, int& bad) {
  if (!isfinite(v)) bad = 1;
  else m = fmaxf(m, fabsf(v));
}

__global__ void __launch_bounds__(kPackThreads) absmax_kernel(const __nv_bfloat16* __restrict__ W,
                                                              int64_t n, PackHeader* hdr) {
  float m = 0.f;
  int bad = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n8 = n / 8;
  const uint4* W8 = reinterpret_cast<const uint4*>(W);
  for (int64_t i = first; i < n8; i += stride) {
    const uint4 v = W8[i];
    const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(e[j]);
      fold(f.x, m, bad);
      fold(f.y, m, bad);
    }
  }
  for (int64_t i = n8 * 8 + first; i < n; i += stride) fold(__bfloat162float(W[i]), m, bad);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    bad |= __shfl_xor_sync(0xffffffffu, bad, off);
  }
  __shared__ float sm[kPackThreads / 32];
  __shared__ int sb[kPackThreads / 32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (lane == 0) {
    sm[warp] = m;
    sb[warp] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kPackThreads / 32; ++w) {
      m = fmaxf(m, sm[w]);
      bad |= sb[w];
    }
    // non-negative floats order like their bit patterns
    atomicMax(&hdr->absmax_bits, __float_as_uint(m));
    if (bad) atomicOr(&hdr->flags, kPackNonFinite);
  }
}

__device__ __forceinline__ int pack_exponent(float mx) {
  if (!(mx > 0.f) || !isfinite(mx)) return 0;
  int e = 0;
  frexpf(mx, &e);            // mx in [2^(e-1), 2^e)
  int k = 15 - e;            // mx 2^k in [2^14, 2^15)
  return k < -120 ? -120 : (k > 120 ? 120 : k);
}

__global__ void __launch_bounds__(kPackThreads) convert_kernel(const __nv_bfloat16* __restrict__ W,
                                                               int64_t n, PackHeader* hdr,
                                                               __half* __restrict__ out) {
  const int k = pack_exponent(__uint_as_float(hdr->absmax_bits));
  const float s = ldexpf(1.f, k);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n8 = n / 8;
  const uint4* W8 = reinterpret_cast<const uint4*>(W);
  uint4* O8 = reinterpret_cast<uint4*>(out);
  for (int64_t i = first; i < n8; i += stride) {
    const uint4 v = W8[i];
    const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(e[j]);
      o[j] = pack_f16x2(f.x * s, f.y * s);
    }
    O8[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  for (int64_t i = n8 * 8 + first; i < n; i += stride)
    out[i] = __float2half_rn(__bfloat162float(W[i]) * s);
  if (first == 0) {
    hdr->k = k;
    hdr->inv_scale = ldexpf(1.f, -k);
    hdr->elements = n;
    hdr->magic = kPackMagic;
  }
}

}  // namespace

cudaError_t launch_pack_f16(const void* W, int64_t elements, void* packed, cudaStream_t s) {
  PackHeader* hdr = static_cast<PackHeader*>(packed);
  cudaError_t e = cudaMemsetAsync(packed, 0, kPackHeaderBytes, s);
  if (e != cudaSuccess) return e;
  if (elements == 0) {
    // an empty tensor: header only (k = 0)
    convert_kernel<<<1, kPackThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(W), 0, hdr,
                                              nullptr);
    return cudaGetLastError();
  }
  const int64_t want = (elements / 8 + kPackThreads - 1) / kPackThreads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 4;
  const unsigned grid = static_cast<unsigned>(want < 1 ? 1 : (want < cap ? want : cap));
  const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(W);
  absmax_kernel<<<grid, kPackThreads, 0, s>>>(w, elements, hdr);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  __half* out = reinterpret_cast<__half*>(static_cast<char*>(packed) + kPackHeaderBytes);
  convert_kernel<<<grid, kPackThreads, 0, s>>>(w, elements, hdr, out);
  return cudaGetLastError();
}

}  // namespace moe

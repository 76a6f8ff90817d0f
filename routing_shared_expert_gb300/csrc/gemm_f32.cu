// fp32 SwiGLU experts on CUDA cores, for layers stored in fp32 (Section 20
// "One Shared Expert Is All You Need", Eq. 74, over the packed segments of
// Section 10, Eq. 26).  Tensor-core fp32 input (TF32) rounds operands to 10
// mantissa bits, far outside a 1e-5 relative budget, so this path stays on FFMA.
//
// Each CTA owns 32 packed rows x 64 output columns of one expert.  The rows'
// inputs and the weight rows are staged through shared memory in 32-wide K
// chunks; each thread accumulates 2 rows x 4 columns.  Row blocks never straddle
// two experts: the CTA walks the same m-tile table (32-row blocks here) that the
// offsets define.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int RB = 32;    // rows per CTA
constexpr int CB = 64;    // output columns per CTA
constexpr int KC = 32;    // K chunk
constexpr int THREADS = 256;

struct F32Args {
  const float* A;            // [rows][k_dim], or x when gathering
  const int32_t* gather_src; // packed row -> row of x, or nullptr
  int64_t src_rows;
  const int32_t* offsets;    // [groups+1] or nullptr (dense)
  int32_t groups;
  int64_t dense_rows;
  int64_t out_rows;
  int32_t k_dim, n_out;
  const float* B0;           // [groups][n_out][k_dim]  (gate, or down)
  const float* B1;           // [groups][n_out][k_dim]  (up) or nullptr
  float* out;                // [rows][n_out]
  int32_t* status;
};

// blockIdx.x: output column block; blockIdx.y: global 32-row block index over the
// concatenation of all segments' row blocks (found by walking the offsets).
template <bool SWIGLU>
__global__ void __launch_bounds__(THREADS) f32_mlp_kernel(F32Args a) {
  __shared__ float As[RB][KC + 1];
  __shared__ float Bg[CB][KC + 1];
  __shared__ float Bu[SWIGLU ? CB : 1][KC + 1];
  __shared__ int s_seg[3];   // group, segment start, segment end

  if (threadIdx.x == 0) {
    int64_t blk = blockIdx.y;
    int g = -1;
    int64_t start = 0, end = 0;
    if (a.offsets == nullptr) {
      g = 0;
      start = 0;
      end = a.dense_rows;
      if (blk * RB >= end) g = -1;
      else start = blk * RB;
    } else {
      for (int e = 0; e < a.groups; ++e) {
        const int64_t lo = a.offsets[e], hi = a.offsets[e + 1];
        const int64_t nb = hi > lo ? (hi - lo + RB - 1) / RB : 0;
        if (blk < nb) { g = e; start = lo + blk * RB; end = hi; break; }
        blk -= nb;
      }
    }
    s_seg[0] = g;
    s_seg[1] = static_cast<int>(start);
    s_seg[2] = static_cast<int>(min(end, a.out_rows));
  }
  __syncthreads();
  const int g = s_seg[0];
  if (g < 0) return;
  const int64_t r0 = s_seg[1], rend = s_seg[2];
  const int c0 = blockIdx.x * CB;

  const int tr = threadIdx.x / 16;   // 0..15 -> rows 2*tr, 2*tr+1
  const int tc = threadIdx.x % 16;   // 0..15 -> cols tc + 16*j
  float ag[2][4] = {}, au[2][4] = {};
  const float* B0 = a.B0 + static_cast<int64_t>(g) * a.n_out * a.k_dim;
  const float* B1 = SWIGLU ? a.B1 + static_cast<int64_t>(g) * a.n_out * a.k_dim : nullptr;

  for (int k0 = 0; k0 < a.k_dim; k0 += KC) {
    for (int i = threadIdx.x; i < RB * KC; i += THREADS) {
      const int r = i / KC, c = i % KC;
      const int64_t row = r0 + r;
      float v = 0.f;
      if (row < rend && k0 + c < a.k_dim) {
        int64_t src = row;
        if (a.gather_src) {
          src = a.gather_src[row];
          if (src < 0 || src >= a.src_rows) {
            set_status(a.status, MOE_ERR_DEVICE_BOUNDS);
            src = -1;
          }
        }
        if (src >= 0) v = a.A[src * a.k_dim + k0 + c];
      }
      As[r][c] = v;
    }
    for (int i = threadIdx.x; i < CB * KC; i += THREADS) {
      const int r = i / KC, c = i % KC;
      const int col = c0 + r;
      const bool ok = col < a.n_out && k0 + c < a.k_dim;
      Bg[r][c] = ok ? B0[static_cast<int64_t>(col) * a.k_dim + k0 + c] : 0.f;
      if (SWIGLU) Bu[r][c] = ok ? B1[static_cast<int64_t>(col) * a.k_dim + k0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < KC; ++c) {
      const float x0 = As[2 * tr][c], x1 = As[2 * tr + 1][c];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float wg = Bg[tc + 16 * j][c];
        ag[0][j] = fmaf(x0, wg, ag[0][j]);
        ag[1][j] = fmaf(x1, wg, ag[1][j]);
        if (SWIGLU) {
          const float wu = Bu[tc + 16 * j][c];
          au[0][j] = fmaf(x0, wu, au[0][j]);
          au[1][j] = fmaf(x1, wu, au[1][j]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int64_t row = r0 + 2 * tr + i;
    if (row >= rend) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = c0 + tc + 16 * j;
      if (col >= a.n_out) continue;
      float v = ag[i][j];
      if (SWIGLU) v = (v / (1.0f + expf(-v))) * au[i][j];
      a.out[row * a.n_out + col] = v;
    }
  }
}

}  // namespace

cudaError_t launch_mlp_f32(const MlpParams& p, cudaStream_t s) {
  const bool dense = p.offsets == nullptr;
  if (p.a_rows == 0 || (dense && p.dense_rows == 0)) return cudaSuccess;
  const int64_t rb_ub = dense ? (p.dense_rows + RB - 1) / RB : (p.a_rows + RB - 1) / RB + p.groups;
  F32Args a{};
  a.offsets = p.offsets;
  a.groups = p.groups;
  a.dense_rows = p.dense_rows;
  a.out_rows = p.a_rows;
  a.status = p.status;

  a.A = static_cast<const float*>(p.A);
  a.gather_src = p.gather_src;
  a.src_rows = p.src_rows;
  a.k_dim = p.d;
  a.n_out = p.width;
  a.B0 = static_cast<const float*>(p.W_gate);
  a.B1 = static_cast<const float*>(p.W_up);
  a.out = static_cast<float*>(p.h);
  dim3 g1((p.width + CB - 1) / CB, static_cast<unsigned>(rb_ub));
  f32_mlp_kernel<true><<<g1, THREADS, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  a.A = static_cast<const float*>(p.h);
  a.gather_src = nullptr;
  a.k_dim = p.width;
  a.n_out = p.d;
  a.B0 = static_cast<const float*>(p.W_down);
  a.B1 = nullptr;
  a.out = static_cast<float*>(p.out);   // fp32 layers: fp32 outputs
  dim3 g2((p.d + CB - 1) / CB, static_cast<unsigned>(rb_ub));
  f32_mlp_kernel<false><<<g2, THREADS, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

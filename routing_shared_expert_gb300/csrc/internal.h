// Internal declarations of the MoE layer library: the workspace layout and the
// kernel launchers.  Every launcher enqueues on the given stream and returns the
// CUDA error of the launch (cudaSuccess on success).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

constexpr int kMaxExperts = 256;   // N limit (routing keeps up to 8 logits per lane of a warp)
constexpr int kMaxTopK = 8;
constexpr int kHistTile = 256;     // tokens per counting tile of the permutation
constexpr int kTcRows = 128;       // rows per tensor-core tile (tcgen05 M)

// Byte offsets of the regions of one workspace (each region 256-byte aligned).
struct Layout {
  size_t status, hist, tile_prefix, topk_idx, topk_w, shared_coef, logits, counts_req,
      counts_keep, offsets, route_pos, perm_src, R_req, R_keep, drop_stats, score_partial, x_perm, h, f,
      hs, g;
  size_t total;
  int64_t hist_tiles;
};

Layout make_layout(const moe_config& c);

// Capacity budget of the layer: b (per expert, Eq. 25) or B (per rank, Eq. 23); 0 without capacity.
int32_t capacity_budget(const moe_config& c);

inline size_t elem_bytes(const moe_config& c) { return c.dtype == MOE_F32 ? 4 : 2; }

// ---- routing -----------------------------------------------------------------
struct RouteParams {
  const void* x;
  const void* W_router;
  const float* router_bias;
  const float* selection_bias;   // Eq. 35 b_i: added to the selection key only (nullable)
  const void* shared_gate_w;
  int64_t T;
  int32_t d, N, K, score, norm, shared_mode;
  float alpha, shared_gain;
  float norm_p;                  // p of the L_p rule
  int32_t* topk_idx;
  float* topk_w;
  float* shared_coef;
  float* logits;
  int32_t* status;
};
cudaError_t launch_route(const RouteParams& p, int32_t dtype, cudaStream_t s);
// bf16 router on the tensor cores (route_tc.cu); launch_route dispatches to it.
cudaError_t launch_route_tc(const RouteParams& p, cudaStream_t s);

// 2-D bf16 tensor map of a dense row-major [rows][inner] tensor: box 64 x box_rows,
// 128-byte swizzle, zero fill out of bounds.  False if the driver rejects it.
bool make_bf16_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);

// Raise a kernel's dynamic shared-memory limit once per device (host-side cache).
cudaError_t set_smem_once(const void* func, size_t bytes);
// Multiprocessor count of the current device (cached).
int device_sm_count();

// ---- counting, capacity, permutation ----------------------------------------
struct PermuteParams {
  const void* x;
  const int32_t* topk_idx;
  int64_t T;
  int32_t d, N, K;
  int32_t cap_policy;
  int32_t cap;            // per-expert budget b or per-rank budget B (ignored without capacity)
  int32_t num_ranks;
  int32_t rho[kMaxExperts];
  int32_t elem_bytes;
  int32_t* hist;          // [hist_tiles][N] workspace
  int64_t hist_tiles;
  int32_t* counts_req;
  int32_t* counts_keep;
  int32_t* offsets;
  int32_t* tile_prefix;   // [N+1] m-tile prefix for the grouped GEMMs
  int32_t* route_pos;
  int32_t* perm_src;
  void* x_perm;
  int32_t* R_req;
  int32_t* R_keep;
  int32_t* drop_stats;
  int32_t* status;
};
cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s);

// m-tile prefix of packed segments: tile_prefix[e] = sum_{i<e} ceil((offsets[i+1]-offsets[i]) / 128).
cudaError_t launch_tile_prefix(const int32_t* offsets, int32_t N, int32_t* tile_prefix,
                               int32_t* status, cudaStream_t s);

// ---- combine -------------------------------------------------------------------
struct CombineParams {
  const void* f;
  const int32_t* route_pos;
  const float* topk_w;
  const void* g;
  const float* shared_coef;
  float* y;
  int64_t T;
  int32_t d, K;
  int64_t f_rows;             // rows of f (positions must be below)
  int32_t* status;
};
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);

// ---- expert GEMMs -------------------------------------------------------------
// One grouped SwiGLU MLP over packed segments (groups = N routed experts) or over
// one dense block of rows (groups = 1, offsets == nullptr, rows = dense_rows).
struct MlpParams {
  const void* A;              // [a_rows][d] input rows, or x [src_rows][d] when gathering
  int64_t a_rows;             // packed rows (capacity of h and out, and of gather_src)
  const int32_t* gather_src;  // [a_rows] source row of each packed row, or nullptr (A is packed)
  int64_t src_rows;           // rows of x when gathering
  const int32_t* offsets;     // [groups+1] device, or nullptr for one dense group
  const int32_t* tile_prefix; // [groups+1] device, or nullptr for one dense group
  int64_t dense_rows;
  int32_t groups;
  int32_t d;                  // model width (K of gate/up, N of down)
  int32_t width;              // intermediate width per group
  const void* W_gate;         // [groups][width][d]
  const void* W_up;           // [groups][width][d]
  const void* W_down;         // [groups][d][width]
  void* h;                    // [a_rows][width] intermediate (workspace), layer dtype
  float* out;                 // [a_rows][d] fp32
  int32_t* status;
};
cudaError_t launch_mlp_bf16(const MlpParams& p, cudaStream_t s);        // 1-SM, 128-row tiles
cudaError_t launch_mlp_bf16_pair(const MlpParams& p, cudaStream_t s);   // CTA pairs, 256-row tiles

// Tile shape choice for the bf16 expert GEMMs: 256-row pair tiles load half the
// bytes per multiply-add of 128-row single-SM tiles and win once segments average
// about 192 rows (measured on GB300: +1.7% on 256-row segments); shorter segments
// waste less on 128-row tiles.
inline bool use_pair_tiles(int64_t rows, int32_t groups) { return rows >= 192LL * groups; }
cudaError_t launch_mlp_f32(const MlpParams& p, cudaStream_t s);



// ---- balancing statistics ------------------------------------------------------
cudaError_t launch_balance_stats(const moe_config& c, const float* logits, float* partial,
                                 const int32_t* counts_req, const int32_t* counts_keep,
                                 const int32_t* R_req, const int32_t* R_keep, float* P, float* f,
                                 float* stats, cudaStream_t s);
cudaError_t launch_bias_update(int32_t N, const int32_t* counts, float gamma, float* bias,
                               cudaStream_t s);

}  // namespace moe

// Internal declarations of the MoE layer library: the workspace layout and the
// kernel launchers.  Every launcher enqueues on the given stream and returns the
// CUDA error of the launch (cudaSuccess on success).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

constexpr int kMaxExperts = 256;   // N limit (routing keeps up to 8 logits per lane of a warp)
constexpr int kMaxTopK = 8;
constexpr int kHistTile = 256;     // tokens per counting tile of the permutation
constexpr int kScoreTile = 64;     // tokens per partial-sum tile of the balance statistics
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
// The fp16 intermediate format of a bf16 layer (MOE_H_F16): h, f and g are fp16.
inline bool h_f16(const moe_config& c) { return c.dtype == MOE_BF16 && c.h_format == MOE_H_F16; }
// Bytes of one element of the expert outputs f and g: fp16 (holding f 2^-h_scale_log2)
// under the fp16 intermediate, fp32 otherwise.
inline size_t out_bytes(const moe_config& c) { return h_f16(c) ? 2 : 4; }

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
// The same on CTA pairs for 128 < N <= 256 without a learned shared gate (route_pair.cu);
// launch_route_tc hands those layers to it.
bool route_pair_applies(const RouteParams& p);
cudaError_t launch_route_pair(const RouteParams& p, cudaStream_t s);

// 2-D bf16 tensor map of a dense row-major [rows][inner] tensor: box 64 x box_rows,
// 128-byte swizzle, zero fill out of bounds.  False if the driver rejects it.
bool make_bf16_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);
bool make_f32_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows);
bool make_bf16_store_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows);
bool make_f16_store_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows);

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
  // Grid-barrier words of the one-launch permutation (count, then generation, on separate
  // 64-byte lines of the workspace header, zero after moe_workspace_init); nullptr: the
  // launch-per-step permutation.
  unsigned* barrier;
};
constexpr size_t kBarrierOffset = 64;   // bytes into the workspace header
cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s);

// m-tile prefix of packed segments: tile_prefix[e] = sum_{i<e} ceil((offsets[i+1]-offsets[i]) / 128).
cudaError_t launch_tile_prefix(const int32_t* offsets, int32_t N, int32_t* tile_prefix,
                               int32_t* status, cudaStream_t s);

// ---- combine -------------------------------------------------------------------
struct CombineParams {
  const void* f;              // fp32, or fp16 holding f 2^-out_log2 (f16 set); g likewise
  bool f16;
  float out_scale;            // 2^out_log2: multiplies the fp16 f and g
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
  void* h;                    // [a_rows][width] intermediate (workspace), 2-byte elements
  void* out;                  // [a_rows][d] fp32, or fp16 holding out 2^-h_scale_log2 (h_f16)
  int32_t* status;
  // fp16 intermediate (MOE_H_F16): h is stored as fp16(h * h_scale), W_down points at a
  // packed buffer (PackHeader, then fp16 W * 2^k) and out holds fp16(accumulator * 2^-k),
  // which is the output times h_scale.
  bool h_f16;
  float h_scale;              // 2^-h_scale_log2
};

// Header of a packed fp16 down-projection tensor (moe_pack_weights): the first
// kPackHeaderBytes bytes of the buffer; elements fp16 values W * 2^k follow.
struct PackHeader {
  uint32_t magic;             // kPackMagic once the pack is complete
  uint32_t absmax_bits;       // fp32 bits of max |W| (reduced by the pack)
  int32_t k;                  // scale exponent: packed value = W * 2^k
  float inv_scale;            // 2^-k
  int64_t elements;
  int32_t flags;              // kPackNonFinite: a weight was infinite or NaN
};
constexpr uint32_t kPackMagic = 0x3631444du;   // "MD16"
constexpr int32_t kPackNonFinite = 1;
constexpr size_t kPackHeaderBytes = 256;
// Largest magnitude an fp16 intermediate may hold before rounding to infinity.
constexpr float kF16RoundsToInf = 65520.f;

cudaError_t launch_pack_f16(const void* W, int64_t elements, void* packed, cudaStream_t s);
// The fp16 values of a packed down-projection tensor (after its header).
inline const void* down_values(const struct MlpParams& p) {
  return static_cast<const char*>(p.W_down) + kPackHeaderBytes;
}
bool make_f16_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);
cudaError_t launch_mlp_bf16(const MlpParams& p, cudaStream_t s);        // 1-SM, 128-row tiles
cudaError_t launch_mlp_bf16_pair(const MlpParams& p, cudaStream_t s);   // CTA pairs, 256-row tiles

// ---- backward pass ------------------------------------------------------------
// Epilogues and kinds of the backward GEMM kernel (gemm_bwd.cu).
constexpr int kBwdEpiF32 = 0;      // fp32 C rows / blocks
constexpr int kBwdEpiSwiglu = 1;   // SwiGLU backward of dh: da | db and h (bf16)
constexpr int kBwdRowsKMajorB = 0;
constexpr int kBwdRowsMnB = 1;
constexpr int kBwdRowsMnBSwiglu = 2;
constexpr int kBwdWeightGrad = 3;

struct BwdGemmArgs {
  // C_g = A_g B_g^T per group g of segment rows [seg_off[g], seg_off[g+1]) (multiples of
  // 64; nullptr = one group of dense_rows).  Row mode (A K-major): M = the segment rows,
  // K = k_dim.  Weight-gradient mode (A MN-major): K = the segment rows, M = m_dim.
  const int32_t* seg_off;
  int32_t dense_rows;
  int32_t groups;
  int32_t m_dim;
  int32_t n_dim;
  int32_t k_dim;
  // B: K-major rows g * b_group_rows + n (second map past b_split_n), or MN-major rows
  // g * b_group_rows + k (second map past b_split_k); b_group_rows < 0: MN-major rows are
  // the segment rows.
  int32_t b_group_rows;
  int32_t b_split_k;
  int32_t b_split_n;
  // fp32 epilogue: rows of C at out (row mode: segment rows; weight mode: group block
  // g at out + g * group_stride, rows >= out_split_m at out2)
  float* out;
  float* out2;
  int32_t out_split_m;
  int64_t group_stride;
  int64_t ldo;
  // SwiGLU-backward epilogue: the accumulator is dh_u = W_d^T dy of a row whose
  // coefficient is row_scale[row] (r or s); dh = row_scale * dh_u
  const float* ab;            // [rows][2 * width] fp32: a | b
  __nv_bfloat16* dab;         // [rows][2 * width] bf16: da | db
  __nv_bfloat16* hout;        // [rows][width] bf16: row_scale * SiLU(a) * b
  const float* row_scale;     // [rows]
  float* dot_part;            // [rows][ceil(width / 256)]: sum over the tile's columns of dh_u * h
  int32_t width;
  int32_t* status;
};
cudaError_t launch_bwd_gemm(int kind, const CUtensorMap& a, const CUtensorMap& b0,
                            const CUtensorMap& b1, const BwdGemmArgs& args, int64_t max_tiles,
                            cudaStream_t s);

struct BwdRowsParams {
  const void* x;              // [T][d] bf16
  const float* dy;            // [T][d]
  const int32_t* counts_keep; // [N]
  const int32_t* offsets;     // [N+1] packed offsets of the forward
  const int32_t* topk_idx;    // [T][K]
  const int32_t* route_pos;   // [T][K]
  const float* topk_w;        // [T][K]
  const int32_t* seg_pad;     // [N+1] padded offsets
  __nv_bfloat16* x_pad;       // [rows][d]
  __nv_bfloat16* gf;          // [rows][d] dy of the row's token (bf16)
  float* r_pad;               // [rows] the row's coefficient r (0 for padding rows)
  int64_t rows_cap;           // rows of x_pad, gf and r_pad
  int64_t T;
  int32_t d, N, K;
  int32_t* status;
};
struct BwdCombineParams {
  const float* dxr;           // [rows][d] route rows (padded layout)
  const float* dxs;           // [T][d] shared rows, or nullptr
  const float* dxz;           // [T][d] dz W_r (gradient through the router), or nullptr
  const float* du;            // [T] gradient of the shared-gate logit, or nullptr
  const __nv_bfloat16* gate_w;   // [d] w_s when du is given
  const int32_t* route_pos;   // [T][K]
  const int32_t* topk_idx;    // [T][K]
  const int32_t* offsets;     // [N+1]
  const int32_t* seg_pad;     // [N+1]
  float* dx;                  // [T][d]
  int64_t T;
  int32_t d, N, K;
  int32_t* status;
};
struct RouterBwdParams {
  const float* logits;        // [T][N] z (+ logit bias) of the forward call
  const int32_t* topk_idx;    // [T][K]
  const int32_t* route_pos;   // [T][K]
  const int32_t* offsets;     // [N+1]
  const int32_t* seg_pad;     // [N+1]
  const float* dot_part;      // [rows][nt] routed dh_u . h per tile
  int32_t nt;
  const float* dot_part_s;    // [t_pad][nt_s] shared, when du is wanted
  int32_t nt_s;
  const float* shared_coef;   // [T]
  int64_t T;
  int32_t N, K, score, norm;
  float alpha, norm_p;
  __nv_bfloat16* dz;          // [T][n128]
  int32_t n128;
  float* du;                  // [T] or nullptr
  int32_t* status;
};
constexpr int kDwsChunks = 64;
cudaError_t launch_router_bwd(const RouterBwdParams& p, cudaStream_t s);
cudaError_t launch_dws(const float* du, const void* x, int64_t T, int d, float* part, float* dws,
                       cudaStream_t s);
cudaError_t launch_pad_offsets(const int32_t* counts_keep, int N, int32_t* seg_pad, cudaStream_t s);
cudaError_t launch_bwd_rows(const BwdRowsParams& p, cudaStream_t s);
cudaError_t launch_shared_scale(const float* dy, const float* sc, int64_t T, int64_t t_pad, int d,
                                __nv_bfloat16* gs, float* s_pad, cudaStream_t s);
cudaError_t launch_dx_combine(const BwdCombineParams& p, cudaStream_t s);

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

// One CTA waits, bounded by limit_ns, on a barrier nothing arrives on (csrc/selfcheck.cu).
cudaError_t launch_wait_bound_check(int32_t* status, uint64_t limit_ns, cudaStream_t s);

}  // namespace moe

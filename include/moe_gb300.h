/*
 * moe_gb300.h - C ABI of the routed + shared-expert MoE layer forward on one GB300 (sm_103a).
 *
 * The layer (Section 21 "Merging Routed and Shared Expert Activations", Eq. 80):
 *
 *     y(x) = sum_{i in S(x)} r_i(x) f_i(x) + s(x) g(x),        |S(x)| = K,
 *
 * with f_i the SwiGLU routed experts and g the shared SwiGLU expert (Section 20
 * "One Shared Expert Is All You Need", Eq. 74), the router, the scores, the
 * selection and the coefficient rules of Appendix E "Expert-Merge Normalization
 * in Public MoE Models" (Table 52), and the requested / kept counts, capacity
 * policies and packed per-expert segments of Section 10 "Routing, Capacity, and
 * Load Balancing" (Eq. 19-27).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named in the argument lists are DEVICE pointers unless marked
 *   "host".  The caller owns every buffer; the library allocates nothing and
 *   frees nothing.  Scratch memory comes from a caller-provided workspace of
 *   at least moe_workspace_size() bytes, 256-byte aligned.
 * - Tensors are dense row-major.  Element type of activations and weights is
 *   cfg->dtype (fp32 or bf16).  Router logits, coefficients, the shared
 *   coefficient and y are fp32 for every dtype.  Indices and counts are int32.
 * - Intermediate format of bf16 layers (cfg->h_format, see moe_h_format): h is
 *   rounded to bf16 and multiplied by the bf16 down projections as given, with the
 *   expert outputs f and the shared output g in fp32; or h is rounded to fp16 and
 *   multiplied by down projections packed to fp16 once by moe_pack_weights, with f
 *   and g in fp16 holding f 2^-h_scale_log2 and g 2^-h_scale_log2.  fp32 layers keep
 *   h, f and g in fp32.
 * - Weight storage: W_router [N][d] (one row per expert, z = x W_router^T);
 *   W_gate, W_up [N][d_expert][d] (one row per intermediate unit, the columns
 *   of W_g / W_u of Eq. 74); W_down [N][d][d_expert] (one row per output
 *   dimension, the columns of W_d); shared Ws_gate, Ws_up [d_shared][d],
 *   Ws_down [d][d_shared].
 * - All work is enqueued on the given stream.  No entry point synchronises
 *   the host with the device or copies device data to the host, except
 *   moe_read_status() which says so.  Arguments are validated on the host
 *   before anything is enqueued; an invalid call returns an error status and
 *   enqueues nothing.  A launch failure returns MOE_ERR_CUDA.
 * - Kernels never trap.  Anything a kernel detects (a bounded wait that ran
 *   out, an index out of range) is written to a status word inside the
 *   workspace; moe_read_status() returns and clears it.
 * - Thread safety: calls on different streams must use different workspaces.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,        /* a null pointer, a size out of range, an unknown enum */
  MOE_ERR_UNSUPPORTED = -2,        /* valid layer, but a shape this build has no kernel for */
  MOE_ERR_CUDA = -3,               /* a CUDA runtime call or launch failed */
  MOE_ERR_WORKSPACE_TOO_SMALL = -4,
  MOE_ERR_TIMEOUT = -5,            /* device status: a bounded wait inside a kernel ran out */
  MOE_ERR_DEVICE_BOUNDS = -6,      /* device status: a kernel saw an index out of range */
  MOE_ERR_MISALIGNED = -7,         /* a pointer is not 16-byte aligned */
  MOE_ERR_RANGE = -8,              /* device status: a value of the fp16 intermediate format
                                    * (h, f or g) left the fp16 range (|v| 2^-h_scale_log2 >=
                                    * 65520), or a packed weight tensor held a non-finite
                                    * value; the outputs are not valid */
  MOE_ERR_BAD_PACK = -9            /* device status: a down-projection pointer of an MOE_H_F16
                                    * call is not a complete moe_pack_weights buffer of the
                                    * layer's size */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Router score (Appendix E, Table 52): softmax over all N experts, or sigmoid affinities. */
typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score;

/* Selected-weight rule (Appendix E, Table 52):
 *   NONE              w = q_S (routed mass m_K < 1 for a softmax over N > K)
 *   L1_SELECTED       w = q_S / sum_S q (Section 21.1; the Olmo and DeepSeek-V3 rows)
 *   SOFTMAX_SELECTED  w = softmax(z_S), the softmax over the selected logits (Mixtral row)
 *   LP_SELECTED       w = q_S / (sum_S q^p)^(1/p), the L_p normalisation the MegaBlocks row
 *                     offers; p = moe_config.norm_p in [1, 64] (p = 1 is L1_SELECTED)
 * The routed coefficients are r = alpha * w.  The same row's option of routed coefficient
 * K/(K+1) and shared coefficient 1/(K+1) is alpha = K/(K+1) with MOE_SHARED_CONST gain 1/(K+1). */
typedef enum {
  MOE_NORM_NONE = 0,
  MOE_NORM_L1_SELECTED = 1,
  MOE_NORM_SOFTMAX_SELECTED = 2,
  MOE_NORM_LP_SELECTED = 3
} moe_norm;

/* Shared coefficient s(x) of Eq. 80: none (0), a constant gain, or sigmoid(w_s . x) (Eq. 77). */
typedef enum { MOE_SHARED_NONE = 0, MOE_SHARED_CONST = 1, MOE_SHARED_SIGMOID_GATE = 2 } moe_shared_mode;

/* Capacity (Section 10.3): none; per expert b = max(1, ceil(c K T / N)) (Eq. 25);
 * rank-wide B = max(1, ceil(c K T / M_E)) shared by the experts rho maps to one rank (Eq. 23),
 * admitted in ascending local expert order.  Kept routes of an expert are its first
 * requests in token order. */
typedef enum { MOE_CAP_NONE = 0, MOE_CAP_PER_EXPERT = 1, MOE_CAP_RANK_WIDE = 2 } moe_cap_policy;

/* Format of the expert intermediate h = SiLU(x W_g) * (x W_u) of bf16 layers (Section 20,
 * Eq. 74), which is the A operand of the down projection f = h W_d on the tensor cores.
 * Both operands of one tensor-core product share one type, so the format also fixes how
 * W_down and Ws_down are passed:
 *   MOE_H_BF16  h rounded to bf16 (8 significant bits, the range of fp32); W_down and
 *               Ws_down are the bf16 tensors of the layout above.
 *   MOE_H_F16   h 2^-h_scale_log2 rounded to fp16 (11 significant bits: eight times less
 *               rounding error, at the same tensor-core rate); W_down and Ws_down are
 *               buffers written by moe_pack_weights (fp16 copies scaled by a power of two,
 *               exact for bf16 weights).  The expert outputs f and g go to the combine in
 *               fp16 as f 2^-h_scale_log2 and g 2^-h_scale_log2 (half the bytes of fp32;
 *               rounding error 2^-12 of each value).  |h|, |f| and |g| times
 *               2^-h_scale_log2 must stay below 65520: a larger value becomes an infinity
 *               and the call leaves MOE_ERR_RANGE in the status word (raise h_scale_log2,
 *               or use MOE_H_BF16).
 * The fp32 layers keep h, f and g in fp32 and ignore the field. */
typedef enum { MOE_H_BF16 = 0, MOE_H_F16 = 1 } moe_h_format;

typedef struct moe_config {
  int64_t T;              /* tokens in the batch, >= 0 */
  int32_t d_model;        /* d */
  int32_t N;              /* routed experts, 1..256 */
  int32_t K;              /* selected per token, 1..min(N, 8) */
  int32_t d_expert;       /* routed intermediate width d_r */
  int32_t d_shared;       /* shared intermediate width d_s, 0 = no shared expert */
  int32_t dtype;          /* moe_dtype */
  int32_t score;          /* moe_score */
  int32_t norm;           /* moe_norm */
  float alpha;            /* routed scale, finite */
  int32_t shared_mode;    /* moe_shared_mode */
  float shared_gain;      /* s for MOE_SHARED_CONST */
  int32_t cap_policy;     /* moe_cap_policy */
  double capacity_factor; /* c > 0 when a capacity policy is set */
  int32_t num_ranks;      /* M_E >= 1: destination ranks of rho (Eq. 20) */
  const int32_t* rho;     /* HOST [N], values in [0, num_ranks); NULL means rho(i) = i mod num_ranks */
  float norm_p;           /* p of MOE_NORM_LP_SELECTED, finite, 1 <= p <= 64; ignored otherwise */
  int32_t h_format;       /* moe_h_format (bf16 layers); 0 = MOE_H_BF16 */
  int32_t h_scale_log2;   /* MOE_H_F16: h is stored as fp16(h 2^-h_scale_log2), -64..64; usually 0 */
} moe_config;

/* Weights of one layer (device pointers, layouts above).  router_bias, selection_bias and
 * shared_gate_w [d] may be NULL; shared weights are ignored when d_shared == 0.  With
 * h_format MOE_H_F16, W_down and Ws_down are moe_pack_weights buffers of the same tensors. */
typedef struct moe_weights {
  const void* W_router;
  const float* router_bias;       /* [N] fp32 logit bias (enters selection and scores), or NULL */
  const float* selection_bias;    /* [N] fp32 Eq. 35 bias b (enters the selection key only), or NULL */
  const void* shared_gate_w;
  const void* W_gate;
  const void* W_up;
  const void* W_down;
  const void* Ws_gate;
  const void* Ws_up;
  const void* Ws_down;
} moe_weights;

/* Outputs of moe_layer_forward (device pointers).  y is required when T > 0; every
 * other pointer may be NULL, in which case that result is kept in the workspace. */
typedef struct moe_outputs {
  float* y;               /* [T][d] fp32 */
  int32_t* topk_idx;      /* [T][K] selected experts, slot order = descending key, lower index on ties */
  float* topk_w;          /* [T][K] r = alpha * w */
  float* shared_coef;     /* [T]    s(x) */
  float* logits;          /* [T][N] router logits z (+ bias) as used for selection */
  int32_t* counts_req;    /* [N]    C^req (Eq. 19) */
  int32_t* counts_keep;   /* [N]    C^keep (Eq. 21) */
  int32_t* offsets;       /* [N+1]  o_e = sum_{i<e} C_i^keep (Eq. 26, exclusive form) */
  int32_t* route_pos;     /* [T][K] packed row of each route, -1 if dropped */
  int32_t* perm_src;      /* [K*T]  token of each packed row; rows >= offsets[N] are unspecified */
  int32_t* R_req;         /* [num_ranks] destination totals (Eq. 20) */
  int32_t* R_keep;        /* [num_ranks] (Eq. 21) */
  int32_t* drop_stats;    /* [4] dropped routes, tokens losing >= 1 route, tokens losing all K, 0 */
} moe_outputs;

/* Library version string (host). */
const char* moe_version(void);

/* Human-readable name of a status code (host). */
const char* moe_status_string(int32_t status);

/* Workspace bytes needed by every entry point for this layer (host only, no CUDA call).
 * Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for a layer the library cannot run. */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Router, scores, top-K and coefficients for every token (Section 10, Table 16 first row;
 * Appendix E, Table 52; Eq. 80 coefficients r and s).
 *   x [T][d]; W_router [N][d]; router_bias [N] fp32 or NULL (a logit bias: part of z);
 *   selection_bias [N] fp32 or NULL (Section 10.6, Eq. 35: added to the selection key only,
 *   the weights come from the unbiased logits); shared_gate_w [d] or NULL (required iff
 *   shared_mode is the sigmoid gate).
 * Out: topk_idx [T][K]; topk_w [T][K]; shared_coef [T] (may be NULL); logits [T][N] (may be
 * NULL) = z, the logits with router_bias and without selection_bias.
 * The selection key is the fp32 value z (+ selection_bias); ties go to the lower expert index. */
moe_status moe_route(const moe_config* cfg, const void* x, const void* W_router,
                     const float* router_bias, const float* selection_bias,
                     const void* shared_gate_w, int32_t* topk_idx, float* topk_w,
                     float* shared_coef, float* logits, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/* Requested and kept counts, capacity, packed offsets and the row permutation
 * (Section 10.1, Eq. 19-21; Section 10.3, Eq. 23, 25, 26, 27).
 *   x [T][d]; topk_idx [T][K] as produced by moe_route (values in [0, N)).
 * Out: counts_req [N], counts_keep [N], offsets [N+1], route_pos [T][K], perm_src [K*T],
 *   R_req / R_keep [num_ranks], drop_stats [4], and optionally x_perm [K*T][d] (rows
 *   [0, offsets[N]) hold x[perm_src[row]], the rest unspecified).  counts_req, R_req, R_keep,
 *   drop_stats and x_perm may be NULL; without x_perm no rows are copied and x may be NULL
 *   (moe_grouped_swiglu can read the rows of x through perm_src instead).
 * Within one expert, packed rows ascend with the token index.  Deterministic. */
moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                       int32_t* counts_req, int32_t* counts_keep, int32_t* offsets,
                       int32_t* route_pos, int32_t* perm_src, void* x_perm,
                       int32_t* R_req, int32_t* R_keep, int32_t* drop_stats,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* moe_permute without a workspace, for callers that cannot allocate device memory (a process
 * whose device memory is fully planned up front, or a plugin host that passes only inputs and
 * outputs).  The pages have no counterpart: this is a packaging variant of moe_permute with the
 * same arguments minus the workspace, and the same results, bit for bit.
 * Its scratch is one static device array built into the library (every GPU that loads the
 * library holds it, 258 KiB, until the process exits): it fits ceil(T / 256) * N <= 65536
 * (for example T <= 65536 at N = 256, T <= 524288 at N = 32); larger layers return
 * MOE_ERR_UNSUPPORTED before anything is enqueued.  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current, so make that first
 * call before any stream capture.  All calls share the array: calls that overlap on the GPU
 * race and must be serialised.  Calls no cudaMalloc / cudaFree.  Device-side index errors are
 * not reported (there is no status word); out-of-range expert ids are skipped. */
moe_status moe_permute_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                               int32_t* counts_req, int32_t* counts_keep, int32_t* offsets,
                               int32_t* route_pos, int32_t* perm_src, void* x_perm,
                               int32_t* R_req, int32_t* R_keep, int32_t* drop_stats,
                               cudaStream_t stream);

/* Bytes of the buffer moe_pack_weights writes for a tensor of `elements` values (host only). */
moe_status moe_packed_weights_size(int64_t elements, size_t* bytes);

/* Pack one bf16 down-projection tensor (W_down [N][d][d_expert], N * d * d_expert elements,
 * or Ws_down [d][d_shared], d * d_shared elements) for the fp16 intermediate (MOE_H_F16).
 * No counterpart on the pages: a storage conversion done once per layer, before the first
 * forward call.  Writes into `packed` (device, 256-byte aligned, moe_packed_weights_size
 * bytes, caller-owned): a 256-byte header (a magic word, the scale exponent k, 2^-k, the
 * element count, a flag for non-finite weights), then the fp16 values W 2^k in the order of
 * W, with k = 15 - e for the largest magnitude max |W| in [2^(e-1), 2^e) (so the largest
 * packed value lies in [2^14, 2^15)): bf16 weights convert exactly down to about
 * max |W| 2^-31.  The expert GEMMs read k from the header and scale their accumulators
 * by 2^-k.  W [elements] bf16 device, 16-byte aligned; W and packed must not overlap.
 * Asynchronous on the stream; no host synchronisation.  Errors: MOE_ERR_INVALID_ARG (NULL,
 * negative count, packed_bytes too small), MOE_ERR_MISALIGNED, MOE_ERR_CUDA.  A non-finite
 * weight is flagged in the header, and a forward call that reads it reports MOE_ERR_RANGE. */
moe_status moe_pack_weights(const void* W, int64_t elements, void* packed, size_t packed_bytes,
                            cudaStream_t stream);

/* Routed experts over densely packed segments (Section 20.1 Eq. 74 per segment; Section 10.3,
 * Eq. 26: packed rows [offsets[e], offsets[e+1]) belong to expert e, nothing else is computed).
 *   offsets [N+1] (device; read on the device, never copied to the host).
 *   perm_src NULL:  x_rows is x_perm [K*T][d], packed row r is x_rows[r].
 *   perm_src [K*T]: x_rows is x [T][d] and packed row r is x[perm_src[r]]; the rows are
 *                   gathered inside the GEMM's operand load, so no K*T x d buffer is
 *                   needed.  Same results bit for bit; on a GB300 this form measured about
 *                   1.5x slower on bf16 layers with 256-row tiles (the rows arrive by
 *                   16-byte asynchronous copies, slower than tile loads) and about 2.7x
 *                   with 128-row tiles (four-row TMA gathers), so moe_layer_forward uses
 *                   the packed form.
 * Out: f [K*T][d]: f[row] = SwiGLU_e(packed row) for rows < offsets[N], fp32 (fp16 holding
 * f 2^-h_scale_log2 under MOE_H_F16).  The intermediate h = SiLU(x W_g) * (x W_u) is kept
 * in the workspace (bf16 or fp16 per cfg->h_format; W_down is a moe_pack_weights buffer
 * under MOE_H_F16). */
moe_status moe_grouped_swiglu(const moe_config* cfg, const void* x_rows, const int32_t* offsets,
                              const int32_t* perm_src, const void* W_gate, const void* W_up,
                              const void* W_down, void* f, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* The one (merged) shared expert over all tokens (Section 20.1, Eq. 74-76).
 *   x [T][d]; Ws_gate, Ws_up [d_shared][d]; Ws_down [d][d_shared] (a moe_pack_weights
 *   buffer under MOE_H_F16).
 * Out: g [T][d] fp32 (fp16 holding g 2^-h_scale_log2 under MOE_H_F16).  Requires
 * d_shared > 0. */
moe_status moe_shared_mlp(const moe_config* cfg, const void* x, const void* Ws_gate,
                          const void* Ws_up, const void* Ws_down, void* g,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Weighted combine, Eq. 80: y_t = sum_{k: route_pos[t][k] >= 0} topk_w[t][k] * f[route_pos[t][k]]
 *   + shared_coef[t] * g_t, accumulated in fp32 in slot order, then the shared term.
 *   f [K*T][d] and g [T][d] as moe_grouped_swiglu / moe_shared_mlp write them (fp32, or fp16
 *   holding f 2^-h_scale_log2 under MOE_H_F16: the combine multiplies the coefficients by
 *   2^h_scale_log2); route_pos, topk_w [T][K]; g and shared_coef [T] may both be NULL (no
 *   shared term).  Out: y [T][d] fp32.  Dropped routes add nothing and the kept
 *   coefficients are not renormalised. */
moe_status moe_combine(const moe_config* cfg, const void* f, const int32_t* route_pos,
                       const float* topk_w, const void* g, const float* shared_coef, float* y,
                       cudaStream_t stream);

/* The whole layer: moe_route, moe_permute, moe_grouped_swiglu, moe_shared_mlp, moe_combine,
 * with intermediates in the workspace.  No host synchronisation.  The shared expert, which
 * needs only x, runs on a second stream beside the router, the permutation and the routed
 * experts: the call records an event on `stream`, makes the second stream wait for it,
 * enqueues the shared expert there and makes `stream` wait for it before the combine, so to
 * the caller the call is ordered on `stream` as if it ran there alone (graph capture of
 * `stream` takes in both).  The second stream and its two events belong to the calling host
 * thread and the current device; they are created on the first call and kept for the
 * thread's lifetime.  Failure to create them returns MOE_ERR_CUDA. */
moe_status moe_layer_forward(const moe_config* cfg, const moe_weights* w, const void* x,
                             const moe_outputs* out, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream);

/* moe_layer_forward that also records five caller-created CUDA events on the stream: before
 * the router, and after the router, the permutation, the routed experts, and the combine
 * (per-stage timing of the exact call a user makes; the shared expert runs concurrently
 * with the first three stages, and the last interval holds any wait for it).  events:
 * HOST array of 5 events. */
moe_status moe_layer_forward_profiled(const moe_config* cfg, const moe_weights* w, const void* x,
                                      const moe_outputs* out, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream,
                                      cudaEvent_t* events);

/* Eq. 75: merge n_parts ungated shared experts into one.  Part j has width widths[j] (HOST array);
 * gate_parts[j], up_parts[j] are [widths[j]][d], down_parts[j] is [d][widths[j]] (HOST arrays of
 * DEVICE pointers).  Out: Ws_gate, Ws_up [sum widths][d] (rows concatenated), Ws_down
 * [d][sum widths] (columns concatenated).  Device-to-device copies on the stream. */
moe_status moe_merge_shared(int32_t d_model, int32_t dtype, int32_t n_parts, const int32_t* widths,
                            const void* const* gate_parts, const void* const* up_parts,
                            const void* const* down_parts, void* Ws_gate, void* Ws_up,
                            void* Ws_down, cudaStream_t stream);

/* Indices into the stats array of moe_balance_stats. */
typedef enum {
  MOE_STAT_LBL = 0,            /* L = N sum_i f_i P_i (Eq. 30); NaN without logits */
  MOE_STAT_IMAX_REQ = 1,       /* I_max of C^req (Eq. 22, 39) */
  MOE_STAT_IMAX_KEEP = 2,      /* I_max of C^keep; NaN without counts_keep */
  MOE_STAT_IMAX_RANK_REQ = 3,  /* I_max of R^req; NaN without R_req */
  MOE_STAT_IMAX_RANK_KEEP = 4, /* I_max of R^keep; NaN without R_keep */
  MOE_STAT_IH_REQ = 5,         /* entropy deficit 1 - H(pi)/log N of C^req (Section 10.2); 0 for N = 1 */
  MOE_STAT_IH_KEEP = 6,        /* entropy deficit of C^keep; NaN without counts_keep */
  MOE_STAT_CV_REQ = 7,         /* coefficient of variation of C^req */
  MOE_STAT_NEVER_SELECTED = 8, /* experts with C^req = 0 */
  MOE_STAT_DROP_FRACTION = 9,  /* delta_route = sum D / (K T) (Eq. 27); NaN without counts_keep */
  MOE_STAT_COUNT = 10
} moe_stat;
/* I_max, I_H and the coefficient of variation of a load vector that sums to 0 are reported as 0. */

/* Load-balancing statistics of one routed batch (Section 10.5, Eq. 30 and 38; Section 10.2,
 * Eq. 22; Eq. 27).  logits [T][N] fp32 as moe_route wrote them (may be NULL: no P, no LBL);
 * counts_req [N] (required), counts_keep [N], R_req / R_keep [num_ranks] (may be NULL).
 * Out (device, each may be NULL): P [N] = mean over tokens of the scores normalised across
 * experts (softmax probabilities; sigmoid scores divided by their sum, Section 10.7.1);
 * f [N] = C_req / (K T); stats [MOE_STAT_COUNT] fp32.  Deterministic (fixed summation order). */
moe_status moe_balance_stats(const moe_config* cfg, const float* logits, const int32_t* counts_req,
                             const int32_t* counts_keep, const int32_t* R_req,
                             const int32_t* R_keep, float* P, float* f, float* stats,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Post-batch bias controller (Section 10.6, Eq. 36-37): bias[i] += gamma * sign(mean(C) - C[i])
 * for the selection-only bias of Eq. 35.  counts [N] int32 (requested counts of the feedback
 * window), bias [N] fp32 updated in place; both device.  Asynchronous on the stream. */
moe_status moe_bias_update(int32_t N, const int32_t* counts, float gamma, float* bias,
                           cudaStream_t stream);

/* ---- Backward pass (router coefficients held fixed) ------------------------------------
 * The expert-path backward of Eq. 74 / Eq. 80 (Section 21, the backward study of Figure
 * 70: input gradient with the router coefficients fixed, routed and shared weight
 * gradients).  Per kept route (t, k) of expert e, gf = topk_w[t][k] dy_t and
 *   dx_t += (W_g^e)^T da + (W_u^e)^T db,  dW_d^e += gf h^T,  dW_g^e += da x_t^T,  dW_u^e += db x_t^T
 * with a = W_g^e x_t, b = W_u^e x_t (recomputed), h = SiLU(a) b, dh = (W_d^e)^T gf,
 * da = dh b SiLU'(a), db = dh SiLU(a); the shared expert likewise with gf = s_t dy_t.
 * Dropped routes carry no gradient.  With grads->dW_router given, the coefficients carry
 * gradient too (Figure 70 (b) "including router gradient"): dr_tk = dy_t . f_{e_tk}(x_t),
 * ds_t = dy_t . g(x_t), differentiated through the selected-weight rule and the scores
 * (Table 52) back to the logits z (the selection held fixed): dW_r = dz^T x, dx += dz W_r,
 * and for a learned shared gate dw_s = sum_t ds_t s_t (1 - s_t) x_t, dx += that times w_s.
 * bf16 layers only, with d_model, d_expert and d_shared multiples of 128 (others:
 * MOE_ERR_UNSUPPORTED); GEMM operands are bf16 (dy, da, db, r h and dz rounded once),
 * accumulation fp32.  The backward takes the down projections as bf16 tensors: call it with
 * h_format MOE_H_BF16 (an MOE_H_F16 configuration returns MOE_ERR_UNSUPPORTED). */
typedef struct moe_grads {
  float* dx;        /* [T][d] fp32 */
  float* dW_gate;   /* [N][d_r][d] fp32 (overwritten) */
  float* dW_up;     /* [N][d_r][d] fp32 */
  float* dW_down;   /* [N][d][d_r] fp32 */
  float* dWs_gate;  /* [d_s][d] fp32; required when d_shared > 0 */
  float* dWs_up;    /* [d_s][d] fp32 */
  float* dWs_down;  /* [d][d_s] fp32 */
  float* dW_router;        /* [N][d] fp32, or NULL: when given, the gradient through the router
                            * coefficients is included (dx too); needs fwd->logits */
  float* dshared_gate_w;   /* [d] fp32: with dW_router and a learned shared gate (Eq. 77) */
} moe_grads;

/* ---- Expert parallelism across ranks (Section 10.3, Eq. 23 and 26, Figure 41) -------------
 * With M ranks each holding a batch of tokens and the experts rho maps to it, every rank
 * all-gathers the requested split counts counts[s][e] (the routes of source rank s's tokens to
 * expert e; C^req of each source's batch from moe_permute) and derives the same keep matrix:
 * destination rank q, with budget B = max(1, ceil(c K T / M)) for the T tokens of all ranks
 * (recovered from the counts: K requests per token), flattens its experts in ascending index
 * and, within an expert, the sources in ascending rank, and admits routes cumulatively until
 * B is used (MOE_CAP_RANK_WIDE; MOE_CAP_NONE keeps everything); source s keeps the first
 * keep[s][e] of its requests to e in token order.  Destination q packs, per expert in
 * ascending index, the rows of source 0, then 1, ...: recv_off[s][e] is the first row of split
 * (s, e) in q's buffer (Eq. 26 over q's experts), R_req[q] / R_keep[q] its requested and kept
 * totals (Eq. 20-21).  On one batch the result equals the single-device rank-wide rule applied
 * to the ranks' batches concatenated in rank order.  The exchange of rows and outputs itself is
 * the caller's (NCCL or peer stores to recv rows); these entries only plan it.
 *
 * moe_ep_keep_matrix: counts, keep, recv_off [M][N] int32 device; R_req, R_keep [M] device or
 * NULL; rho HOST [N] with values in [0, M).  One kernel on the stream, no host synchronisation.
 * Errors: MOE_ERR_INVALID_ARG (sizes, rho, NULL), MOE_ERR_UNSUPPORTED (per-expert capacity:
 * use the rank-wide budget across ranks), MOE_ERR_CUDA. */
moe_status moe_ep_keep_matrix(int32_t M, int32_t N, int32_t K, const int32_t* rho,
                              int32_t cap_policy, double capacity_factor, const int32_t* counts,
                              int32_t* keep, int32_t* recv_off, int32_t* R_req, int32_t* R_keep,
                              cudaStream_t stream);

/* Destination rows of source rank src_rank's routes: dst_row[t][k] = recv_off[src][e] + (rank of
 * route (t, k) among the source's requests to its expert e in token order) when that rank is
 * below keep[src][e], else -1 (dropped); the destination rank is rho[e].  topk_idx, route_pos
 * and offsets are those of a moe_permute of the source's batch under a configuration without
 * capacity (route_pos - offsets[e] is the rank); keep and recv_off from moe_ep_keep_matrix.
 * All device; M is the number of source ranks (rows of keep / recv_off), src_rank in [0, M).
 * workspace: a workspace of the layer (its status word records an expert id out of range, with
 * dst_row -1).  Errors: MOE_ERR_INVALID_ARG (sizes, src_rank, NULL), MOE_ERR_CUDA. */
moe_status moe_ep_place(int32_t M, int32_t src_rank, int64_t T, int32_t N, int32_t K,
                        const int32_t* topk_idx,
                        const int32_t* route_pos, const int32_t* offsets, const int32_t* keep,
                        const int32_t* recv_off, int32_t* dst_row, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/* The same two steps on HOST arrays, with no CUDA call (the planning logic alone, for hosts that
 * gather the counts themselves).  moe_ep_place_host ranks the routes itself from topk_idx in
 * (token, slot) order.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED as above. */
moe_status moe_ep_keep_matrix_host(int32_t M, int32_t N, int32_t K, const int32_t* rho,
                                   int32_t cap_policy, double capacity_factor,
                                   const int32_t* counts, int32_t* keep, int32_t* recv_off,
                                   int32_t* R_req, int32_t* R_keep);
moe_status moe_ep_place_host(int32_t M, int32_t src_rank, int64_t T, int32_t N, int32_t K,
                             const int32_t* topk_idx, const int32_t* keep,
                             const int32_t* recv_off, int32_t* dst_row);

/* The exchange buffers of the dispatch (Section 10.3, Figure 41).  Source src_rank's send
 * buffer holds, for each destination rank in ascending order, the rows it sends there in the
 * destination's buffer order (its experts ascending, each split's kept prefix in token
 * order), so a destination receives, per source in ascending rank, one contiguous block.
 *
 * moe_ep_send_pos: send_pos[t][k] = the send-buffer row of route (t, k), -1 when dropped;
 * send_counts[q] (may be NULL) = rows sent to rank q.  topk_idx, dst_row [T][K] (dst_row from
 * moe_ep_place), keep, recv_off [M][N], send_pos, send_counts: device.  rho HOST [N].
 * workspace: a layer workspace (its status word records expert ids out of range, with
 * send_pos -1).  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA.
 *
 * moe_ep_recv_rows: for destination dst_rank, recv_row[j] = the row of its packed buffer
 * (per local expert ascending, sources ascending: recv_off) that row j of its receive
 * buffer (source blocks in ascending rank) belongs to; R_keep[dst_rank] entries, at most
 * recv_cap written (more records MOE_ERR_DEVICE_BOUNDS in the workspace).  Device arrays,
 * rho HOST.  Errors as above.
 *
 * moe_rows_copy: for i in [0, n): dst row dst_index[i] (i when dst_index is NULL) = src row
 * src_index[i] (i / src_div when src_index is NULL; src_div = K maps route t K + k to token
 * t).  A negative destination skips the row; a negative source writes zeros when
 * zero_missing is set, else skips.  Rows of row_bytes bytes (a multiple of 16), src and dst
 * 16-byte aligned and not overlapping; src [src_rows] and dst [dst_rows] rows bound the
 * indices (an index past them records MOE_ERR_DEVICE_BOUNDS and skips the row).  One warp
 * per row.  Device arrays.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED (row_bytes not a
 * multiple of 16), MOE_ERR_MISALIGNED, MOE_ERR_CUDA.
 *
 * The _host twins take host arrays, make no CUDA call and return MOE_ERR_INVALID_ARG for an
 * index out of range. */
moe_status moe_ep_send_pos(int32_t M, int32_t src_rank, int64_t T, int32_t N, int32_t K,
                           const int32_t* rho, const int32_t* topk_idx, const int32_t* keep,
                           const int32_t* recv_off, const int32_t* dst_row, int32_t* send_pos,
                           int32_t* send_counts, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);
moe_status moe_ep_recv_rows(int32_t M, int32_t dst_rank, int32_t N, const int32_t* rho,
                            const int32_t* keep, const int32_t* recv_off, int32_t* recv_row,
                            int64_t recv_cap, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);
moe_status moe_rows_copy(const void* src, int64_t src_rows, const int32_t* src_index,
                         int64_t src_div, void* dst, int64_t dst_rows, const int32_t* dst_index,
                         int64_t n, int64_t row_bytes, int32_t zero_missing, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream);
moe_status moe_ep_send_pos_host(int32_t M, int32_t src_rank, int64_t T, int32_t N, int32_t K,
                                const int32_t* rho, const int32_t* topk_idx, const int32_t* keep,
                                const int32_t* recv_off, const int32_t* dst_row,
                                int32_t* send_pos, int32_t* send_counts);
moe_status moe_ep_recv_rows_host(int32_t M, int32_t dst_rank, int32_t N, const int32_t* rho,
                                 const int32_t* keep, const int32_t* recv_off, int32_t* recv_row,
                                 int64_t recv_cap);
moe_status moe_rows_copy_host(const void* src, int64_t src_rows, const int32_t* src_index,
                              int64_t src_div, void* dst, int64_t dst_rows,
                              const int32_t* dst_index, int64_t n, int64_t row_bytes,
                              int32_t zero_missing);

/* Bytes of scratch moe_layer_backward needs (256-byte aligned; prepare it with
 * moe_workspace_init before its first use). */
moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes);

/* The backward pass for upstream gradient dy [T][d] fp32 (device).  x and the weights are
 * those of the forward call; fwd holds that call's routing results (device): topk_idx,
 * topk_w, counts_keep, offsets, route_pos, perm_src, shared_coef when d_shared > 0, and
 * logits when grads->dW_router is given.
 * Writes every array of grads (device, caller-owned).  Asynchronous on the stream; no
 * host synchronisation. */
moe_status moe_layer_backward(const moe_config* cfg, const moe_weights* w, const void* x,
                              const moe_outputs* fwd, const float* dy, const moe_grads* grads,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Prepare a fresh workspace: zero its device status word (the first 256 bytes).  Call once
 * after allocating a workspace, before its first use.  Asynchronous on the stream. */
moe_status moe_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Self-check of the device-side wait bound (no counterpart on the pages): one CTA waits on a
 * barrier that nothing arrives on, bounded by limit_ns (1 ns .. 2 s) of %globaltimer, the same
 * bounded wait every tensor-core kernel uses.  The wait runs out, MOE_ERR_TIMEOUT lands in the
 * workspace status word and the CTA exits; the context stays usable.  Asynchronous on the stream;
 * read the result with moe_read_status().  Errors: MOE_ERR_INVALID_ARG (NULL or < 256-byte
 * workspace, limit out of range), MOE_ERR_MISALIGNED, MOE_ERR_CUDA (launch failure). */
moe_status moe_check_wait_bound(void* workspace, size_t workspace_bytes, int64_t limit_ns,
                                cudaStream_t stream);

/* Read and clear the device status word of a workspace.  Synchronises the stream and copies
 * 4 bytes to the host.  *code (host) receives MOE_OK or the first device-detected error.  The
 * whole 256-byte header of the workspace is reset (as by moe_workspace_init), so a workspace
 * is ready for the next call after any device-detected error. */
moe_status moe_read_status(void* workspace, int32_t* code, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */

// C ABI of the MoE layer library: argument validation, the workspace layout and
// the entry points declared in moe_gb300.h.  Validation happens on the host
// before anything is enqueued; every entry point is asynchronous on its stream.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <type_traits>
#include <utility>
#include <vector>

#include "internal.h"

namespace moe {

namespace {

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_cfg(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->T > (int64_t{1} << 28)) return MOE_ERR_INVALID_ARG;
  if (c->d_model < 1 || c->N < 1 || c->K < 1 || c->d_expert < 1 || c->d_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->N > kMaxExperts || c->K > kMaxTopK || c->K > c->N) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (c->norm < MOE_NORM_NONE || c->norm > MOE_NORM_LP_SELECTED) return MOE_ERR_INVALID_ARG;
  if (c->norm == MOE_NORM_LP_SELECTED &&
      !(std::isfinite(c->norm_p) && c->norm_p >= 1.f && c->norm_p <= 64.f))
    return MOE_ERR_INVALID_ARG;
  if (c->shared_mode < MOE_SHARED_NONE || c->shared_mode > MOE_SHARED_SIGMOID_GATE)
    return MOE_ERR_INVALID_ARG;
  if ((c->d_shared > 0) != (c->shared_mode != MOE_SHARED_NONE)) return MOE_ERR_INVALID_ARG;
  if (c->cap_policy < MOE_CAP_NONE || c->cap_policy > MOE_CAP_RANK_WIDE) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->alpha) || !std::isfinite(c->shared_gain)) return MOE_ERR_INVALID_ARG;
  if (c->cap_policy != MOE_CAP_NONE &&
      (!std::isfinite(c->capacity_factor) || c->capacity_factor <= 0.0))
    return MOE_ERR_INVALID_ARG;
  if (c->num_ranks < 1 || c->num_ranks > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (c->h_format != MOE_H_BF16 && c->h_format != MOE_H_F16) return MOE_ERR_INVALID_ARG;
  if (c->h_scale_log2 < -64 || c->h_scale_log2 > 64) return MOE_ERR_INVALID_ARG;
  if (c->rho) {
    for (int i = 0; i < c->N; ++i)
      if (c->rho[i] < 0 || c->rho[i] >= c->num_ranks) return MOE_ERR_INVALID_ARG;
  }
  const int64_t d = c->d_model, dr = c->d_expert, ds = c->d_shared;
  if (c->dtype == MOE_BF16) {
    // 16-byte rows for TMA and vector copies, and at least one 64-wide K block.
    if (d % 8 || dr % 8 || ds % 8 || d < 64 || dr < 64 || (ds > 0 && ds < 64))
      return MOE_ERR_UNSUPPORTED;
  } else {
    if (d % 4) return MOE_ERR_UNSUPPORTED;
  }
  if (c->T * c->K * std::max<int64_t>(d, std::max(dr, ds)) > (int64_t{1} << 40))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

moe_status check_ws(const moe_config& c, void* ws, size_t bytes, Layout* L) {
  *L = make_layout(c);
  if (!ws) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_MISALIGNED;
  if (bytes < L->total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

RouteParams route_params(const moe_config& c, const void* x, const void* W_router,
                         const float* bias, const float* sel_bias, const void* gate_w,
                         int32_t* idx, float* w, float* s, float* logits, int32_t* status) {
  RouteParams p{};
  p.x = x;
  p.W_router = W_router;
  p.router_bias = bias;
  p.selection_bias = sel_bias;
  p.shared_gate_w = gate_w;
  p.T = c.T;
  p.d = c.d_model;
  p.N = c.N;
  p.K = c.K;
  p.score = c.score;
  p.norm = c.norm;
  p.shared_mode = c.shared_mode;
  p.alpha = c.alpha;
  p.shared_gain = c.shared_gain;
  p.norm_p = c.norm_p;
  p.topk_idx = idx;
  p.topk_w = w;
  p.shared_coef = s;
  p.logits = logits;
  p.status = status;
  return p;
}

moe_status do_route(const moe_config& c, const void* x, const void* W_router, const float* bias,
                    const float* sel_bias, const void* gate_w, int32_t* idx, float* w, float* s,
                    float* logits, int32_t* status, cudaStream_t st) {
  if (c.T > 0 && (!x || !W_router || !idx || !w)) return MOE_ERR_INVALID_ARG;
  if (c.shared_mode == MOE_SHARED_SIGMOID_GATE && !gate_w) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_route(
      route_params(c, x, W_router, bias, sel_bias, gate_w, idx, w, s, logits, status), c.dtype, st));
}

struct PermOut {
  int32_t *counts_req, *counts_keep, *offsets, *route_pos, *perm_src, *R_req, *R_keep, *drops;
  void* x_perm;
};

moe_status do_permute(const moe_config& c, const Layout& L, void* ws, const void* x,
                      const int32_t* topk_idx, const PermOut& o, cudaStream_t st) {
  if (c.T > 0 && (!topk_idx || !o.route_pos || !o.perm_src)) return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && o.x_perm && !x) return MOE_ERR_INVALID_ARG;
  if (!o.counts_keep || !o.offsets) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(o.x_perm)) return MOE_ERR_MISALIGNED;
  PermuteParams p{};
  p.x = x;
  p.topk_idx = topk_idx;
  p.T = c.T;
  p.d = c.d_model;
  p.N = c.N;
  p.K = c.K;
  p.cap_policy = c.cap_policy;
  p.cap = capacity_budget(c);
  p.num_ranks = c.num_ranks;
  for (int i = 0; i < c.N; ++i) p.rho[i] = c.rho ? c.rho[i] : i % c.num_ranks;
  p.elem_bytes = static_cast<int32_t>(elem_bytes(c));
  p.hist = at<int32_t>(ws, L.hist);
  p.hist_tiles = L.hist_tiles;
  p.counts_req = o.counts_req;
  p.counts_keep = o.counts_keep;
  p.offsets = o.offsets;
  p.tile_prefix = at<int32_t>(ws, L.tile_prefix);
  p.route_pos = o.route_pos;
  p.perm_src = o.perm_src;
  p.x_perm = o.x_perm;
  p.R_req = o.R_req;
  p.R_keep = o.R_keep;
  p.drop_stats = o.drops;
  p.status = at<int32_t>(ws, L.status);
  p.barrier = at<unsigned>(ws, L.status + kBarrierOffset);
  return cuda_status(launch_permute(p, st));
}

// The intermediate format of a bf16 layer's expert GEMMs (moe_h_format).
void set_h_format(const moe_config& c, MlpParams* p) {
  p->h_f16 = h_f16(c);
  p->h_scale = std::ldexp(1.0f, -c.h_scale_log2);
}

moe_status do_grouped(const moe_config& c, const Layout& L, void* ws, const void* x_rows,
                      const int32_t* offsets, const int32_t* perm_src, const void* Wg,
                      const void* Wu, const void* Wd, void* f, bool tile_prefix_ready,
                      cudaStream_t st) {
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if (!x_rows || !Wg || !Wu || !Wd || !f) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_rows) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) || !aligned16(f))
    return MOE_ERR_MISALIGNED;
  int32_t* status = at<int32_t>(ws, L.status);
  int32_t* tp = at<int32_t>(ws, L.tile_prefix);
  if (!tile_prefix_ready) {
    moe_status s = cuda_status(launch_tile_prefix(offsets, c.N, tp, status, st));
    if (s != MOE_OK) return s;
  }
  MlpParams p{};
  p.A = x_rows;
  p.a_rows = c.T * c.K;
  p.gather_src = perm_src;
  p.src_rows = c.T;
  p.offsets = offsets;
  p.tile_prefix = tp;
  p.groups = c.N;
  p.d = c.d_model;
  p.width = c.d_expert;
  p.W_gate = Wg;
  p.W_up = Wu;
  p.W_down = Wd;
  p.h = at<void>(ws, L.h);
  p.out = f;
  p.status = status;
  set_h_format(c, &p);
  if (c.dtype == MOE_F32) return cuda_status(launch_mlp_f32(p, st));
  return cuda_status(use_pair_tiles(c.T * c.K, c.N) ? launch_mlp_bf16_pair(p, st)
                                                    : launch_mlp_bf16(p, st));
}

moe_status do_shared(const moe_config& c, const Layout& L, void* ws, const void* x,
                     const void* Wg, const void* Wu, const void* Wd, void* g, cudaStream_t st) {
  if (c.d_shared == 0) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if (!x || !Wg || !Wu || !Wd || !g) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) || !aligned16(g))
    return MOE_ERR_MISALIGNED;
  MlpParams p{};
  p.A = x;
  p.a_rows = c.T;
  p.offsets = nullptr;
  p.tile_prefix = nullptr;
  p.dense_rows = c.T;
  p.groups = 1;
  p.d = c.d_model;
  p.width = c.d_shared;
  p.W_gate = Wg;
  p.W_up = Wu;
  p.W_down = Wd;
  p.h = at<void>(ws, L.hs);
  p.out = g;
  p.status = at<int32_t>(ws, L.status);
  set_h_format(c, &p);
  if (c.dtype == MOE_F32) return cuda_status(launch_mlp_f32(p, st));
  return cuda_status(use_pair_tiles(c.T, 1) ? launch_mlp_bf16_pair(p, st) : launch_mlp_bf16(p, st));
}

moe_status do_combine(const moe_config& c, const void* f, const int32_t* route_pos,
                      const float* topk_w, const void* g, const float* s, float* y,
                      int32_t* status, cudaStream_t st) {
  if (c.T == 0) return MOE_OK;
  if (!f || !route_pos || !topk_w || !y) return MOE_ERR_INVALID_ARG;
  if ((g == nullptr) != (s == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(f) || !aligned16(y) || (g && !aligned16(g))) return MOE_ERR_MISALIGNED;
  CombineParams p{};
  p.f = f;
  p.f16 = h_f16(c);
  p.out_scale = std::ldexp(1.0f, c.h_scale_log2);
  p.route_pos = route_pos;
  p.topk_w = topk_w;
  p.g = g;
  p.shared_coef = s;
  p.y = y;
  p.T = c.T;
  p.d = c.d_model;
  p.K = c.K;
  p.f_rows = c.T * c.K;
  p.status = status;
  return cuda_status(launch_combine(p, st));
}

}  // namespace

int32_t capacity_budget(const moe_config& c) {
  if (c.cap_policy == MOE_CAP_NONE) return 0;
  const double routes = static_cast<double>(c.K) * static_cast<double>(c.T);
  const double denom = c.cap_policy == MOE_CAP_PER_EXPERT ? c.N : c.num_ranks;
  const double b = std::ceil(c.capacity_factor * routes / denom);
  if (b < 1.0) return 1;
  if (b > 2147483647.0) return 2147483647;
  return static_cast<int32_t>(b);
}

Layout make_layout(const moe_config& c) {
  Layout L{};
  const size_t T = static_cast<size_t>(c.T), N = c.N, K = c.K, d = c.d_model, dr = c.d_expert,
               ds = c.d_shared, eb = elem_bytes(c), M = c.num_ranks;
  L.hist_tiles = (c.T + kHistTile - 1) / kHistTile;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.status = take(256);
  L.hist = take(static_cast<size_t>(L.hist_tiles) * N * 4);
  L.tile_prefix = take((N + 1) * 4);
  L.topk_idx = take(T * K * 4);
  L.topk_w = take(T * K * 4);
  L.shared_coef = take(T * 4);
  L.logits = take(T * N * 4);
  L.counts_req = take(N * 4);
  L.counts_keep = take(N * 4);
  L.offsets = take((N + 1) * 4);
  L.route_pos = take(T * K * 4);
  L.perm_src = take(T * K * 4);
  L.R_req = take(M * 4);
  L.R_keep = take(M * 4);
  L.drop_stats = take(16);
  L.score_partial = take(static_cast<size_t>((c.T + kScoreTile - 1) / kScoreTile) * N * 4);
  L.x_perm = take(T * K * d * eb);
  L.h = take(T * K * dr * eb);
  L.f = take(T * K * d * out_bytes(c));
  L.hs = take(T * ds * eb);
  L.g = take(T * d * out_bytes(c));
  L.total = o;
  return L;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_version(void) { return "moe_gb300 0.1 (sm_103a)"; }

const char* moe_status_string(int32_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape for this build";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_BOUNDS: return "device index out of range";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MOE_ERR_RANGE: return "a value left the range of the fp16 intermediate format";
    case MOE_ERR_BAD_PACK: return "down projection is not a packed buffer of the layer's size";
    default: return "unknown status";
  }
}

moe_status moe_packed_weights_size(int64_t elements, size_t* bytes) {
  if (elements < 0 || !bytes || elements > (int64_t{1} << 40)) return MOE_ERR_INVALID_ARG;
  *bytes = moe::kPackHeaderBytes + ((static_cast<size_t>(elements) * 2 + 255) & ~size_t{255});
  return MOE_OK;
}

moe_status moe_pack_weights(const void* W, int64_t elements, void* packed, size_t packed_bytes,
                            cudaStream_t stream) {
  size_t need = 0;
  moe_status s = moe_packed_weights_size(elements, &need);
  if (s != MOE_OK) return s;
  if (!packed || (elements > 0 && !W) || packed_bytes < need) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(packed) & 255u) != 0 || (reinterpret_cast<uintptr_t>(W) & 15u))
    return MOE_ERR_MISALIGNED;
  const char* w0 = static_cast<const char*>(W);
  const char* p0 = static_cast<const char*>(packed);
  if (elements > 0 && w0 < p0 + need && p0 < w0 + elements * 2) return MOE_ERR_INVALID_ARG;
  return moe::launch_pack_f16(W, elements, packed, stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, const void* x, const void* W_router,
                     const float* router_bias, const float* selection_bias,
                     const void* shared_gate_w, int32_t* topk_idx, float* topk_w,
                     float* shared_coef, float* logits, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  Layout L;
  if ((s = check_ws(*cfg, workspace, workspace_bytes, &L)) != MOE_OK) return s;
  return do_route(*cfg, x, W_router, router_bias, selection_bias, shared_gate_w, topk_idx, topk_w,
                  shared_coef, logits, at<int32_t>(workspace, L.status), stream);
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                       int32_t* counts_req, int32_t* counts_keep, int32_t* offsets,
                       int32_t* route_pos, int32_t* perm_src, void* x_perm, int32_t* R_req,
                       int32_t* R_keep, int32_t* drop_stats, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  Layout L;
  if ((s = check_ws(*cfg, workspace, workspace_bytes, &L)) != MOE_OK) return s;
  PermOut o{counts_req, counts_keep, offsets, route_pos, perm_src, R_req, R_keep, drop_stats,
            x_perm};
  return do_permute(*cfg, L, workspace, x, topk_idx, o, stream);
}

moe_status moe_grouped_swiglu(const moe_config* cfg, const void* x_rows, const int32_t* offsets,
                              const int32_t* perm_src, const void* W_gate, const void* W_up,
                              const void* W_down, void* f, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  Layout L;
  if ((s = check_ws(*cfg, workspace, workspace_bytes, &L)) != MOE_OK) return s;
  return do_grouped(*cfg, L, workspace, x_rows, offsets, perm_src, W_gate, W_up, W_down, f, false,
                    stream);
}

moe_status moe_shared_mlp(const moe_config* cfg, const void* x, const void* Ws_gate,
                          const void* Ws_up, const void* Ws_down, void* g, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  Layout L;
  if ((s = check_ws(*cfg, workspace, workspace_bytes, &L)) != MOE_OK) return s;
  return do_shared(*cfg, L, workspace, x, Ws_gate, Ws_up, Ws_down, g, stream);
}

moe_status moe_combine(const moe_config* cfg, const void* f, const int32_t* route_pos,
                       const float* topk_w, const void* g, const float* shared_coef, float* y,
                       cudaStream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  return do_combine(*cfg, f, route_pos, topk_w, g, shared_coef, y, nullptr, stream);
}

}  // extern "C"

namespace moe {
namespace {

// The layer forward; when `ev` is non-null, events [0..4] are recorded on the stream before
// the router and after the router, the permutation, the routed experts, and the shared
// expert + combine.
// A second stream of the calling host thread on the current device, with a fork and a
// join event, created on first use and kept for the thread's lifetime.  The shared
// expert runs on it, concurrently with the router, the permutation and the routed
// experts; it needs none of their results.
struct AuxStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

struct AuxStreams {
  std::vector<std::pair<int, AuxStream>> per_device;
  ~AuxStreams() {
    for (auto& e : per_device) {   // errors at process teardown are of no consequence
      cudaEventDestroy(e.second.fork);
      cudaEventDestroy(e.second.join);
      cudaStreamDestroy(e.second.stream);
    }
  }
};

bool aux_stream(AuxStream* out) {
  thread_local AuxStreams cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  for (auto& e : cache.per_device)
    if (e.first == dev) {
      *out = e.second;
      return true;
    }
  AuxStream a;
  if (cudaStreamCreateWithFlags(&a.stream, cudaStreamNonBlocking) != cudaSuccess) return false;
  if (cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming) != cudaSuccess) {
    if (a.fork) cudaEventDestroy(a.fork);
    cudaStreamDestroy(a.stream);
    return false;
  }
  cache.per_device.emplace_back(dev, a);
  *out = a;
  return true;
}

moe_status layer_forward(const moe_config* cfg, const moe_weights* w, const void* x,
                         const moe_outputs* out, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream, cudaEvent_t* ev) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!w || !out || (!out->y && cfg->T > 0)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if ((s = check_ws(*cfg, workspace, workspace_bytes, &L)) != MOE_OK) return s;
  const moe_config& c = *cfg;
  void* ws = workspace;
  auto pick = [&](auto* user, size_t off) {
    using P = std::remove_pointer_t<decltype(user)>;
    return user ? user : at<P>(ws, off);
  };
  auto mark = [&](int i) {
    return (ev && cudaEventRecord(ev[i], stream) != cudaSuccess) ? MOE_ERR_CUDA : MOE_OK;
  };
  int32_t* idx = pick(out->topk_idx, L.topk_idx);
  float* tw = pick(out->topk_w, L.topk_w);
  float* sc = pick(out->shared_coef, L.shared_coef);
  int32_t* status = at<int32_t>(ws, L.status);
  if ((s = mark(0)) != MOE_OK) return s;
  // Fork: the shared expert (Eq. 74-76 on x) is enqueued on the auxiliary stream right
  // after the router, so the GPU runs it beside the router, the permutation and the
  // routed experts; the combine waits for it.
  AuxStream aux;
  const bool shared = c.d_shared > 0;
  if (shared) {
    if (!aux_stream(&aux)) return MOE_ERR_CUDA;
    if (cudaEventRecord(aux.fork, stream) != cudaSuccess ||
        cudaStreamWaitEvent(aux.stream, aux.fork, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if ((s = do_route(c, x, w->W_router, w->router_bias, w->selection_bias, w->shared_gate_w, idx,
                    tw, sc, out->logits, status, stream)) != MOE_OK)
    return s;
  void* g = nullptr;
  if (shared) {
    g = at<void>(ws, L.g);
    if ((s = do_shared(c, L, ws, x, w->Ws_gate, w->Ws_up, w->Ws_down, g, aux.stream)) != MOE_OK)
      return s;
    if (cudaEventRecord(aux.join, aux.stream) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if ((s = mark(1)) != MOE_OK) return s;
  PermOut po{pick(out->counts_req, L.counts_req), pick(out->counts_keep, L.counts_keep),
             pick(out->offsets, L.offsets),       pick(out->route_pos, L.route_pos),
             pick(out->perm_src, L.perm_src),     pick(out->R_req, L.R_req),
             pick(out->R_keep, L.R_keep),         pick(out->drop_stats, L.drop_stats),
             at<void>(ws, L.x_perm)};
  if ((s = do_permute(c, L, ws, x, idx, po, stream)) != MOE_OK) return s;
  if ((s = mark(2)) != MOE_OK) return s;
  void* f = at<void>(ws, L.f);
  // Packed rows: one copy pass, then plain tile loads in the GEMM.  Rows gathered inside
  // the GEMM (TMA four-row gathers, or cp.async by gatherer warps) arrive too slowly to feed
  // the tensor cores: the layer runs 1.4-1.5x slower that way.
  if ((s = do_grouped(c, L, ws, po.x_perm, po.offsets, nullptr, w->W_gate, w->W_up, w->W_down, f,
                      true, stream)) != MOE_OK)
    return s;
  if ((s = mark(3)) != MOE_OK) return s;
  if (shared && cudaStreamWaitEvent(stream, aux.join, 0) != cudaSuccess) return MOE_ERR_CUDA;
  if ((s = do_combine(c, f, po.route_pos, tw, g, g ? sc : nullptr, out->y, status, stream)) != MOE_OK)
    return s;
  return mark(4);
}


// ---- backward -------------------------------------------------------------------
struct BwdLayout {
  size_t status, seg_pad, x_pad, gf, r_pad, ab, dab, h, dxr, dot, gs, s_pad, ab_s, dab_s, h_s, dx_s,
      dot_s, dz, dxz, du, dws_part;
  size_t total;
  int64_t rows_cap;   // padded routed rows
  int64_t t_pad;      // T rounded up to 64
  int32_t nt, nt_s;   // 256-column tiles of d_r and d_s (partial dot products per row)
  int32_t n128;       // N rounded up to 128 (columns of dz)
};

BwdLayout make_bwd_layout(const moe_config& c) {
  BwdLayout L{};
  const size_t T = static_cast<size_t>(c.T), N = c.N, K = c.K, d = c.d_model, dr = c.d_expert,
               ds = c.d_shared;
  L.rows_cap = static_cast<int64_t>(K * T + 64 * N);
  L.t_pad = (c.T + 63) / 64 * 64;
  const size_t R = static_cast<size_t>(L.rows_cap), Tp = static_cast<size_t>(L.t_pad);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.nt = static_cast<int32_t>((dr + 255) / 256);
  L.nt_s = static_cast<int32_t>((ds + 255) / 256);
  L.n128 = static_cast<int32_t>((N + 127) / 128 * 128);
  L.status = take(256);
  L.seg_pad = take((N + 1) * 4);
  L.x_pad = take(R * d * 2);
  L.gf = take(R * d * 2);
  L.r_pad = take(R * 4);
  L.ab = take(R * 2 * dr * 4);
  L.dab = take(R * 2 * dr * 2);
  L.h = take(R * dr * 2);
  L.dxr = take(R * d * 4);
  L.dot = take(R * L.nt * 4);
  L.gs = take(T * d * 2);
  L.s_pad = take(Tp * 4);
  L.ab_s = take(Tp * 2 * ds * 4);
  L.dab_s = take(Tp * 2 * ds * 2);
  L.h_s = take(Tp * ds * 2);
  L.dx_s = take(Tp * d * 4);
  L.dot_s = take(Tp * static_cast<size_t>(L.nt_s) * 4);
  L.dz = take(T * static_cast<size_t>(L.n128) * 2);
  L.dxz = take(Tp * d * 4);
  L.du = take(T * 4);
  L.dws_part = take(static_cast<size_t>(kDwsChunks) * d * 4);
  L.total = o;
  return L;
}

moe_status check_bwd_cfg(const moe_config* c) {
  moe_status s = check_cfg(c);
  if (s != MOE_OK) return s;
  if (c->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (c->h_format != MOE_H_BF16) return MOE_ERR_UNSUPPORTED;   // needs the bf16 down projections
  if (c->d_model % 128 != 0 || c->d_expert % 128 != 0 || c->d_shared % 128 != 0)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// The five GEMMs of one expert family (routed: groups of padded segments; shared: one
// dense group of T rows), then nothing else: the caller combines dx.
moe_status bwd_family(const moe_config& c, bool routed, const int32_t* seg_pad, int64_t rows,
                      const void* x_rows, const __nv_bfloat16* gf, const float* row_scale,
                      float* dot_part, float* ab, __nv_bfloat16* dab, __nv_bfloat16* h, float* dxr,
                      const void* Wg, const void* Wu, const void* Wd, float* dWg, float* dWu,
                      float* dWd, int32_t* status, cudaStream_t st) {
  const int G = routed ? c.N : 1;
  const int64_t d = c.d_model, w = routed ? c.d_expert : c.d_shared;
  // rows of the row-major activation maps: routed rows_cap; shared: x and gf have T rows
  // (TMA fills the rows up to T rounded to 64 with zeros), the others t_pad
  const uint64_t in_rows = routed ? static_cast<uint64_t>(rows) : static_cast<uint64_t>(c.T);
  CUtensorMap mX, mGf, mDab, mWg, mWu, mWd, mWgMn, mWuMn, mGfMn, mHMn, mDabMn, mXMn;
  if (!make_bf16_map(&mX, x_rows, d, in_rows, 128) || !make_bf16_map(&mGf, gf, d, in_rows, 128) ||
      !make_bf16_map(&mDab, dab, 2 * w, rows, 128) ||
      !make_bf16_map(&mWg, Wg, d, static_cast<uint64_t>(G) * w, 128) ||
      !make_bf16_map(&mWu, Wu, d, static_cast<uint64_t>(G) * w, 128) ||
      !make_bf16_map(&mWd, Wd, w, static_cast<uint64_t>(G) * d, 64) ||
      !make_bf16_map(&mWgMn, Wg, d, static_cast<uint64_t>(G) * w, 64) ||
      !make_bf16_map(&mWuMn, Wu, d, static_cast<uint64_t>(G) * w, 64) ||
      !make_bf16_map(&mGfMn, gf, d, in_rows, 64) || !make_bf16_map(&mHMn, h, w, rows, 64) ||
      !make_bf16_map(&mDabMn, dab, 2 * w, rows, 64) || !make_bf16_map(&mXMn, x_rows, d, in_rows, 64))
    return MOE_ERR_CUDA;
  BwdGemmArgs a{};
  a.seg_off = routed ? seg_pad : nullptr;
  a.dense_rows = static_cast<int32_t>(rows);
  a.groups = G;
  a.status = status;
  const int64_t sms = device_sm_count();
  const int64_t row_tiles = rows / 128 + G;   // upper bound of 128-row tiles over all segments
  auto st_ok = [](cudaError_t e) { return e == cudaSuccess; };

  // recompute [a | b] = x [W_g | W_u]^T  (fp32)
  a.k_dim = static_cast<int32_t>(d);
  a.n_dim = static_cast<int32_t>(2 * w);
  a.b_group_rows = static_cast<int32_t>(w);
  a.b_split_n = static_cast<int32_t>(w);
  a.out = ab;
  a.ldo = 2 * w;
  if (!st_ok(launch_bwd_gemm(kBwdRowsKMajorB, mX, mWg, mWu, a, row_tiles * (2 * w / 128), st)))
    return MOE_ERR_CUDA;
  // dh = gf W_d, then da | db and h
  a.k_dim = static_cast<int32_t>(d);
  a.n_dim = static_cast<int32_t>(w);
  a.b_group_rows = static_cast<int32_t>(d);
  a.b_split_n = 0;
  a.b_split_k = 0;
  a.ab = ab;
  a.dab = dab;
  a.hout = h;
  a.row_scale = row_scale;
  a.dot_part = dot_part;
  a.width = static_cast<int32_t>(w);
  if (!st_ok(launch_bwd_gemm(kBwdRowsMnBSwiglu, mGf, mWd, mWd, a, row_tiles * (w / 128), st)))
    return MOE_ERR_CUDA;
  // dx rows = da W_g + db W_u
  a.k_dim = static_cast<int32_t>(2 * w);
  a.n_dim = static_cast<int32_t>(d);
  a.b_group_rows = static_cast<int32_t>(w);
  a.b_split_k = static_cast<int32_t>(w);
  a.out = dxr;
  a.ldo = d;
  if (!st_ok(launch_bwd_gemm(kBwdRowsMnB, mDab, mWgMn, mWuMn, a, row_tiles * (d / 128), st)))
    return MOE_ERR_CUDA;
  // dW_d = gf^T h
  a.b_split_k = 0;
  a.b_group_rows = -1;
  a.m_dim = static_cast<int32_t>(d);
  a.n_dim = static_cast<int32_t>(w);
  a.out = dWd;
  a.out2 = nullptr;
  a.out_split_m = 0;
  a.group_stride = d * w;
  a.ldo = w;
  if (!st_ok(launch_bwd_gemm(kBwdWeightGrad, mGfMn, mHMn, mHMn, a, G * (d / 128) * (w / 128), st)))
    return MOE_ERR_CUDA;
  // dW_g | dW_u = (da | db)^T x
  a.m_dim = static_cast<int32_t>(2 * w);
  a.n_dim = static_cast<int32_t>(d);
  a.out = dWg;
  a.out2 = dWu;
  a.out_split_m = static_cast<int32_t>(w);
  a.group_stride = w * d;
  a.ldo = d;
  if (!st_ok(launch_bwd_gemm(kBwdWeightGrad, mDabMn, mXMn, mXMn, a, G * (2 * w / 128) * (d / 128), st)))
    return MOE_ERR_CUDA;
  (void)sms;
  return MOE_OK;
}

moe_status layer_backward(const moe_config* cfg, const moe_weights* w, const void* x,
                          const moe_outputs* fwd, const float* dy, const moe_grads* g,
                          void* ws, size_t ws_bytes, cudaStream_t st) {
  moe_status s = check_bwd_cfg(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (!w || !fwd || !g || !ws) return MOE_ERR_INVALID_ARG;
  const bool shared = c.d_shared > 0;
  if (!g->dx || !g->dW_gate || !g->dW_up || !g->dW_down) return MOE_ERR_INVALID_ARG;
  if (shared && (!g->dWs_gate || !g->dWs_up || !g->dWs_down || !fwd->shared_coef))
    return MOE_ERR_INVALID_ARG;
  if (!fwd->topk_idx || !fwd->topk_w || !fwd->counts_keep || !fwd->offsets || !fwd->route_pos ||
      !fwd->perm_src)
    return MOE_ERR_INVALID_ARG;
  if (!w->W_gate || !w->W_up || !w->W_down || (shared && (!w->Ws_gate || !w->Ws_up || !w->Ws_down)))
    return MOE_ERR_INVALID_ARG;
  // the gradient through the router coefficients, when dW_router is given
  const bool router = g->dW_router != nullptr;
  const bool gate = router && shared && c.shared_mode == MOE_SHARED_SIGMOID_GATE;
  if (router && (!fwd->logits || !w->W_router)) return MOE_ERR_INVALID_ARG;
  if (gate && (!g->dshared_gate_w || !w->shared_gate_w)) return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && (!x || !dy)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_MISALIGNED;
  const BwdLayout L = make_bwd_layout(c);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(g->dx)) return MOE_ERR_MISALIGNED;
  int32_t* status = at<int32_t>(ws, L.status);
  int32_t* seg_pad = at<int32_t>(ws, L.seg_pad);
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (!ok(launch_pad_offsets(fwd->counts_keep, c.N, seg_pad, st))) return MOE_ERR_CUDA;
  if (c.T == 0) return MOE_OK;
  BwdRowsParams rp{};
  rp.x = x;
  rp.dy = dy;
  rp.counts_keep = fwd->counts_keep;
  rp.offsets = fwd->offsets;
  rp.topk_idx = fwd->topk_idx;
  rp.route_pos = fwd->route_pos;
  rp.topk_w = fwd->topk_w;
  rp.seg_pad = seg_pad;
  rp.x_pad = at<__nv_bfloat16>(ws, L.x_pad);
  rp.gf = at<__nv_bfloat16>(ws, L.gf);
  rp.r_pad = at<float>(ws, L.r_pad);
  rp.rows_cap = L.rows_cap;
  rp.T = c.T;
  rp.d = c.d_model;
  rp.N = c.N;
  rp.K = c.K;
  rp.status = status;
  if (!ok(launch_bwd_rows(rp, st))) return MOE_ERR_CUDA;
  s = bwd_family(c, true, seg_pad, L.rows_cap, rp.x_pad, rp.gf, rp.r_pad,
                 router ? at<float>(ws, L.dot) : nullptr, at<float>(ws, L.ab),
                 at<__nv_bfloat16>(ws, L.dab), at<__nv_bfloat16>(ws, L.h), at<float>(ws, L.dxr),
                 w->W_gate, w->W_up, w->W_down, g->dW_gate, g->dW_up, g->dW_down, status, st);
  if (s != MOE_OK) return s;
  float* dxs = nullptr;
  if (shared) {
    __nv_bfloat16* gs = at<__nv_bfloat16>(ws, L.gs);
    float* s_pad = at<float>(ws, L.s_pad);
    if (!ok(launch_shared_scale(dy, fwd->shared_coef, c.T, L.t_pad, c.d_model, gs, s_pad, st)))
      return MOE_ERR_CUDA;
    dxs = at<float>(ws, L.dx_s);
    s = bwd_family(c, false, nullptr, L.t_pad, x, gs, s_pad, gate ? at<float>(ws, L.dot_s) : nullptr,
                   at<float>(ws, L.ab_s), at<__nv_bfloat16>(ws, L.dab_s),
                   at<__nv_bfloat16>(ws, L.h_s), dxs, w->Ws_gate, w->Ws_up, w->Ws_down,
                   g->dWs_gate, g->dWs_up, g->dWs_down, status, st);
    if (s != MOE_OK) return s;
  }
  float* dxz = nullptr;
  float* du = nullptr;
  if (router) {
    // dz per token, then dW_r = dz^T x and dz W_r
    __nv_bfloat16* dz = at<__nv_bfloat16>(ws, L.dz);
    RouterBwdParams zp{};
    zp.logits = fwd->logits;
    zp.topk_idx = fwd->topk_idx;
    zp.route_pos = fwd->route_pos;
    zp.offsets = fwd->offsets;
    zp.seg_pad = seg_pad;
    zp.dot_part = at<float>(ws, L.dot);
    zp.nt = L.nt;
    zp.dot_part_s = gate ? at<float>(ws, L.dot_s) : nullptr;
    zp.nt_s = L.nt_s;
    zp.shared_coef = fwd->shared_coef;
    zp.T = c.T;
    zp.N = c.N;
    zp.K = c.K;
    zp.score = c.score;
    zp.norm = c.norm;
    zp.alpha = c.alpha;
    zp.norm_p = c.norm_p;
    zp.dz = dz;
    zp.n128 = L.n128;
    du = gate ? at<float>(ws, L.du) : nullptr;
    zp.du = du;
    zp.status = status;
    if (!ok(launch_router_bwd(zp, st))) return MOE_ERR_CUDA;
    CUtensorMap mZk, mZm, mWr, mX;
    if (!make_bf16_map(&mZk, dz, L.n128, c.T, 128) || !make_bf16_map(&mZm, dz, L.n128, c.T, 64) ||
        !make_bf16_map(&mWr, w->W_router, c.d_model, c.N, 64) ||
        !make_bf16_map(&mX, x, c.d_model, c.T, 64))
      return MOE_ERR_CUDA;
    BwdGemmArgs a{};
    a.seg_off = nullptr;
    a.dense_rows = static_cast<int32_t>(L.t_pad);
    a.groups = 1;
    a.status = status;
    // dW_r [N][d] = dz^T x (K = tokens)
    a.m_dim = c.N;
    a.n_dim = c.d_model;
    a.b_group_rows = -1;
    a.out = g->dW_router;
    a.ldo = c.d_model;
    if (!ok(launch_bwd_gemm(kBwdWeightGrad, mZm, mX, mX, a,
                            ((c.N + 255) / 256) * ((c.d_model + 255) / 256), st)))
      return MOE_ERR_CUDA;
    // dz W_r [T][d] (K = N rounded up to 128; dz is zero past N and W_r reads zero past N)
    dxz = at<float>(ws, L.dxz);
    a.m_dim = 0;
    a.k_dim = L.n128;
    a.n_dim = c.d_model;
    a.b_group_rows = 0;
    a.out = dxz;
    a.ldo = c.d_model;
    if (!ok(launch_bwd_gemm(kBwdRowsMnB, mZk, mWr, mWr, a,
                            (L.t_pad / 256 + 1) * ((c.d_model + 255) / 256), st)))
      return MOE_ERR_CUDA;
    if (gate && !ok(launch_dws(du, x, c.T, c.d_model, at<float>(ws, L.dws_part), g->dshared_gate_w, st)))
      return MOE_ERR_CUDA;
  }
  BwdCombineParams cp{};
  cp.dxr = at<float>(ws, L.dxr);
  cp.dxs = dxs;
  cp.dxz = dxz;
  cp.du = du;
  cp.gate_w = static_cast<const __nv_bfloat16*>(w->shared_gate_w);
  cp.route_pos = fwd->route_pos;
  cp.topk_idx = fwd->topk_idx;
  cp.offsets = fwd->offsets;
  cp.seg_pad = seg_pad;
  cp.dx = g->dx;
  cp.T = c.T;
  cp.d = c.d_model;
  cp.N = c.N;
  cp.K = c.K;
  cp.status = status;
  return ok(launch_dx_combine(cp, st)) ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_layer_forward(const moe_config* cfg, const moe_weights* w, const void* x,
                             const moe_outputs* out, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
  return layer_forward(cfg, w, x, out, workspace, workspace_bytes, stream, nullptr);
}

moe_status moe_layer_forward_profiled(const moe_config* cfg, const moe_weights* w, const void* x,
                                      const moe_outputs* out, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream,
                                      cudaEvent_t* events) {
  if (!events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 5; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return layer_forward(cfg, w, x, out, workspace, workspace_bytes, stream, events);
}

moe_status moe_merge_shared(int32_t d_model, int32_t dtype, int32_t n_parts, const int32_t* widths,
                            const void* const* gate_parts, const void* const* up_parts,
                            const void* const* down_parts, void* Ws_gate, void* Ws_up,
                            void* Ws_down, cudaStream_t stream) {
  if (d_model < 1 || n_parts < 1 || !widths || !gate_parts || !up_parts || !down_parts ||
      !Ws_gate || !Ws_up || !Ws_down)
    return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  const size_t eb = dtype == MOE_F32 ? 4 : 2;
  size_t total = 0;
  for (int j = 0; j < n_parts; ++j) {
    if (widths[j] < 1 || !gate_parts[j] || !up_parts[j] || !down_parts[j])
      return MOE_ERR_INVALID_ARG;
    total += static_cast<size_t>(widths[j]);
  }
  size_t row = 0;
  for (int j = 0; j < n_parts; ++j) {
    const size_t w = static_cast<size_t>(widths[j]);
    const size_t rows_bytes = w * d_model * eb;
    cudaError_t e = cudaMemcpyAsync(static_cast<char*>(Ws_gate) + row * d_model * eb,
                                    gate_parts[j], rows_bytes, cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<char*>(Ws_up) + row * d_model * eb, up_parts[j], rows_bytes,
                          cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(static_cast<char*>(Ws_down) + row * eb, total * eb, down_parts[j],
                            w * eb, w * eb, static_cast<size_t>(d_model),
                            cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    row += w;
  }
  return MOE_OK;
}

moe_status moe_balance_stats(const moe_config* cfg, const float* logits, const int32_t* counts_req,
                             const int32_t* counts_keep, const int32_t* R_req,
                             const int32_t* R_keep, float* P, float* f, float* stats,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  Layout L;
  if ((s = check_ws(*cfg, workspace, workspace_bytes, &L)) != MOE_OK) return s;
  if (!counts_req) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_balance_stats(*cfg, logits, at<float>(workspace, L.score_partial),
                                          counts_req, counts_keep, R_req, R_keep, P, f, stats,
                                          stream));
}

moe_status moe_bias_update(int32_t N, const int32_t* counts, float gamma, float* bias,
                           cudaStream_t stream) {
  if (N < 1 || N > kMaxExperts || !counts || !bias || !std::isfinite(gamma))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_bias_update(N, counts, gamma, bias, stream));
}

moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  moe_status s = check_bwd_cfg(cfg);
  if (s != MOE_OK) return s;
  *bytes = make_bwd_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_layer_backward(const moe_config* cfg, const moe_weights* w, const void* x,
                              const moe_outputs* fwd, const float* dy, const moe_grads* grads,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return layer_backward(cfg, w, x, fwd, dy, grads, workspace, workspace_bytes, stream);
}

moe_status moe_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!workspace || workspace_bytes < 256) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_MISALIGNED;
  return cudaMemsetAsync(workspace, 0, 256, stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_check_wait_bound(void* workspace, size_t workspace_bytes, int64_t limit_ns,
                                cudaStream_t stream) {
  if (!workspace || workspace_bytes < 256 || limit_ns <= 0 || limit_ns > 2000000000LL)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_MISALIGNED;
  return launch_wait_bound_check(static_cast<int32_t*>(workspace), static_cast<uint64_t>(limit_ns),
                                 stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_read_status(void* workspace, int32_t* code, cudaStream_t stream) {
  if (!workspace || !code) return MOE_ERR_INVALID_ARG;
  int32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  // the stream is idle: clear the whole header (the status word and the permutation's
  // grid-barrier words, which a barrier that ran out may have left set)
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, 256, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  *code = host;
  return MOE_OK;
}

}  // extern "C"

// moe_permute_noalloc: the counting / capacity / permutation step for callers
// that cannot allocate device memory.
//
// Who needs it: code that must not call cudaMalloc and has no workspace to hand
// over - for example a serving process whose device memory is fully planned and
// reserved at start-up, or a host plugin interface that passes only the input
// and output pointers of each call.  The regular moe_permute takes its scratch
// (per-tile expert histograms and the m-tile prefix) from a caller workspace;
// this variant takes it from one fixed array compiled into the library instead.
//
// The array below lives in device global memory of every GPU that loads the
// library, for the life of the process.  In host code its name is only a
// host-side stand-in for the symbol, so the host never passes it to a kernel:
// the first call on each device looks up the array's device address with
// cudaGetSymbolAddress (with that device current) and caches it together with
// the device's current CUDA context.  That first call should therefore come
// before any stream capture on that device.  A device reset replaces the
// context (and may move the array): a call that finds another context looks the
// address up again, so that call too should come before any stream capture.
//
// Every call on a device shares the array and leaves its last contents in it.
// Nothing in it needs clearing: each call overwrites every histogram entry and
// prefix entry it later reads.  Two calls that overlap on the GPU (different
// streams, or a second call enqueued on another stream before the first has
// finished) race on the array and give wrong results; serialise them.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// Capacity of the static scratch: per-tile expert histograms [ceil(T/256)][N]
// (at most 65536 int32, 256 KiB) plus the m-tile prefix (N + 1 <= 257 int32).
constexpr int64_t kNoAllocHistInts = 65536;
constexpr int64_t kNoAllocPrefixInts = 512;

static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocPrefixInts + kNoAllocHistInts];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int32_t* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The driver's cuCtxGetCurrent, found through the runtime (the library does not link the
// driver library itself).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch array on the current device, looked up once per device
// and context.
cudaError_t scratch_on_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return cudaErrorDeviceUninitialized;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (ctx == nullptr || g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    // the lookup binds the device's primary context to this thread if nothing has yet
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute_noalloc(const moe_config* cfg, const void* x,
                                          const int32_t* topk_idx, int32_t* counts_req,
                                          int32_t* counts_keep, int32_t* offsets,
                                          int32_t* route_pos, int32_t* perm_src, void* x_perm,
                                          int32_t* R_req, int32_t* R_keep, int32_t* drop_stats,
                                          cudaStream_t stream) {
  size_t unused = 0;
  moe_status s = moe_workspace_size(cfg, &unused);   // validates the layer (host only)
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  const int64_t tiles = (c.T + kHistTile - 1) / kHistTile;
  if (tiles * c.N > kNoAllocHistInts) return MOE_ERR_UNSUPPORTED;   // beyond the static scratch
  // the same argument rules as moe_permute: x is needed only to fill x_perm
  if (c.T > 0 && (!topk_idx || !route_pos || !perm_src)) return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && x_perm && !x) return MOE_ERR_INVALID_ARG;
  if (!counts_keep || !offsets) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x_perm) & 15u))
    return MOE_ERR_MISALIGNED;

  int32_t* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;

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
  p.tile_prefix = scratch;
  p.hist = scratch + kNoAllocPrefixInts;
  p.hist_tiles = tiles;
  p.counts_req = counts_req;
  p.counts_keep = counts_keep;
  p.offsets = offsets;
  p.route_pos = route_pos;
  p.perm_src = perm_src;
  p.x_perm = x_perm;
  p.R_req = R_req;
  p.R_keep = R_keep;
  p.drop_stats = drop_stats;
  p.status = nullptr;   // no workspace, so no status word: out-of-range expert ids are skipped
  return launch_permute(p, stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Requested and kept counts, capacity, packed offsets and the row permutation.
//
// Follows Section 10 "Routing, Capacity, and Load Balancing": Eq. 19 (requested
// counts), Eq. 20-21 (destination totals, kept counts, drops), Eq. 23 / Eq. 25
// (rank-wide and per-expert budgets), the admission order of Section 10.3
// (local-expert-major, a prefix of each expert's requests in token order),
// Eq. 26 (kept rows packed densely per expert, offsets o_e) and Eq. 27 (drops).
//
// A stable counting sort, no atomics on positions.  Layers whose 256-token tiles fit on
// the GPU at once (up to a few tens of thousands of tokens) run steps 1-3 as one
// cooperative launch with a grid barrier (permute_fused_kernel); larger ones, and callers
// without a workspace, run them as three launches:
//   1. count   - one CTA per tile of 256 tokens: per-tile histogram of experts.
//   2. scan    - one CTA: per-expert exclusive prefix over tiles (C^req falls out),
//                the capacity rule (C^keep), offsets, destination totals, the
//                m-tile prefix the grouped GEMMs walk, and the dropped-route total.
//   3. place   - one CTA per tile: ranks each route among the requests to its expert
//                in (token, slot) order (warp-level __match_any_sync, then a prefix
//                over the tile's warps), and writes the packed position of every
//                kept route (-1 if dropped) and its source token.
//   4. gather  - one warp per token: copies x[t] into the packed rows of t's kept
//                routes (only when the caller passes x_perm).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) count_kernel(PermuteParams p) {
  __shared__ int hist[kMaxExperts];
  for (int e = threadIdx.x; e < p.N; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kHistTile;
  const int64_t t1 = min(t0 + kHistTile, p.T);
  const int64_t r0 = t0 * p.K, r1 = t1 * p.K;
  for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const int e = p.topk_idx[r];
    if (e < 0 || e >= p.N) {
      set_status(p.status, MOE_ERR_DEVICE_BOUNDS);
      continue;
    }
    atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < p.N; e += blockDim.x)
    p.hist[blockIdx.x * static_cast<int64_t>(p.N) + e] = hist[e];
}

__device__ void capacity_and_offsets(const PermuteParams& p, const int* creq, int* ckeep, int* offs,
                                     int* tprefix, int* rreq, int* rkeep, int* dropped);
__device__ void write_layer_results(const PermuteParams& p, const int* creq, const int* ckeep,
                                    const int* offs, const int* tprefix, const int* rreq,
                                    const int* rkeep, int dropped, bool zero_tokens);

__global__ void __launch_bounds__(1024) scan_kernel(PermuteParams p) {
  __shared__ int creq[kMaxExperts];
  __shared__ int ckeep[kMaxExperts];
  __shared__ int offs[kMaxExperts + 1];
  __shared__ int tprefix[kMaxExperts + 1];
  __shared__ int rreq[kMaxExperts];
  __shared__ int rkeep[kMaxExperts];
  __shared__ int dropped;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = blockDim.x / 32;

  // 1. per-expert exclusive prefix over tiles, in place; C^req is the total.
  for (int e = warp; e < p.N; e += nwarps) {
    int running = 0;
    for (int64_t base = 0; base < p.hist_tiles; base += 32) {
      const int64_t tile = base + lane;
      const int v = tile < p.hist_tiles ? p.hist[tile * p.N + e] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (tile < p.hist_tiles) p.hist[tile * p.N + e] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) creq[e] = running;
  }
  __syncthreads();
  capacity_and_offsets(p, creq, ckeep, offs, tprefix, rreq, rkeep, &dropped);
  write_layer_results(p, creq, ckeep, offs, tprefix, rreq, rkeep, dropped, true);
}

// Kept counts (the capacity rule), destination totals, offsets (Eq. 26), the prefix of
// 128-row tiles and the dropped-route total, from the requested counts creq; every array
// in shared memory; all threads of the block call it.
__device__ void capacity_and_offsets(const PermuteParams& p, const int* creq, int* ckeep, int* offs,
                                     int* tprefix, int* rreq, int* rkeep, int* dropped) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // 2. kept counts and destination totals.  The per-expert and unlimited rules decide
  //    each expert alone.  The rank-wide budget is shared by a rank's experts in
  //    ascending expert index (the local-expert-major admission order of the rank-wide
  //    rule): one thread per rank walks its experts in that order.
  if (p.cap_policy == MOE_CAP_RANK_WIDE) {
    for (int q = threadIdx.x; q < p.num_ranks; q += blockDim.x) {
      int used = 0, req = 0;
      for (int e = 0; e < p.N; ++e) {
        if (p.rho[e] != q) continue;
        const int keep = min(creq[e], p.cap - used);
        ckeep[e] = keep;
        used += keep;
        req += creq[e];
      }
      rreq[q] = req;
      rkeep[q] = used;
    }
  } else {
    for (int q = threadIdx.x; q < p.num_ranks; q += blockDim.x) { rreq[q] = 0; rkeep[q] = 0; }
    __syncthreads();
    for (int e = threadIdx.x; e < p.N; e += blockDim.x) {
      const int keep = p.cap_policy == MOE_CAP_PER_EXPERT ? min(creq[e], p.cap) : creq[e];
      ckeep[e] = keep;
      atomicAdd(&rreq[p.rho[e]], creq[e]);
      atomicAdd(&rkeep[p.rho[e]], keep);
    }
  }
  __syncthreads();
  // 3. offsets (Eq. 26), the prefix of 128-row tiles, and the dropped-route total: one
  //    warp scans the experts 32 at a time.
  if (warp == 0) {
    int run_o = 0, run_t = 0, drop = 0;
    for (int base = 0; base < p.N; base += 32) {
      const int e = base + lane;
      const int k = e < p.N ? ckeep[e] : 0;
      const int nt = (k + kTcRows - 1) / kTcRows;
      if (e < p.N) drop += creq[e] - k;
      int io = k, it = nt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o1 = __shfl_up_sync(0xffffffffu, io, off);
        const int o2 = __shfl_up_sync(0xffffffffu, it, off);
        if (lane >= off) { io += o1; it += o2; }
      }
      if (e < p.N) {
        offs[e + 1] = run_o + io;
        tprefix[e + 1] = run_t + it;
      }
      run_o += __shfl_sync(0xffffffffu, io, 31);
      run_t += __shfl_sync(0xffffffffu, it, 31);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) drop += __shfl_xor_sync(0xffffffffu, drop, off);
    if (lane == 0) {
      offs[0] = 0;
      tprefix[0] = 0;
      *dropped = drop;
    }
  }
  __syncthreads();
}

// The layer-wide results of the counting pass; with `zero_tokens` the two per-token drop
// tallies are reset (the placing pass adds to them afterwards).
__device__ void write_layer_results(const PermuteParams& p, const int* creq, const int* ckeep,
                                    const int* offs, const int* tprefix, const int* rreq,
                                    const int* rkeep, int dropped, bool zero_tokens) {
  for (int e = threadIdx.x; e < p.N; e += blockDim.x) {
    if (p.counts_req) p.counts_req[e] = creq[e];
    p.counts_keep[e] = ckeep[e];
  }
  for (int e = threadIdx.x; e <= p.N; e += blockDim.x) {
    p.offsets[e] = offs[e];
    p.tile_prefix[e] = tprefix[e];
  }
  for (int q = threadIdx.x; q < p.num_ranks; q += blockDim.x) {
    if (p.R_req) p.R_req[q] = rreq[q];
    if (p.R_keep) p.R_keep[q] = rkeep[q];
  }
  if (threadIdx.x == 0 && p.drop_stats) {
    p.drop_stats[0] = dropped;
    if (zero_tokens) {
      p.drop_stats[1] = 0;
      p.drop_stats[2] = 0;
    }
    p.drop_stats[3] = 0;
  }
}

// One CTA (8 warps) per 256-token tile.  Warp w owns tokens [32w, 32w+32) of the
// tile; its 32*K routes in (token, slot) order are ranked within the warp with
// __match_any_sync (round k holds routes [32k, 32k+32) of the warp's range).  A
// per-expert exclusive prefix over the warps, seeded with the routes to that
// expert from earlier tiles, then gives every route its rank among all requests
// to its expert in token order.
// The placing step for one tile (256 threads): ckeep and offs in shared memory, seed[e] the
// requests to expert e from earlier tiles (shared or global memory).  wcnt (per-warp counts
// of the tile, then per-warp bases within the tile: at most 256 K <= 2048, so 16 bits) and
// drops are shared-memory scratch of the caller.
__device__ void place_tile(const PermuteParams& p, int64_t tile, const int* ckeep, const int* offs,
                           const int* seed, uint16_t (*wcnt)[kMaxExperts], int* drops) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int e = threadIdx.x; e < p.N; e += blockDim.x) {
#pragma unroll
    for (int w = 0; w < 8; ++w) wcnt[w][e] = 0;
  }
  for (int i = threadIdx.x; i < kHistTile; i += blockDim.x) drops[i] = 0;
  __syncthreads();

  const int64_t t0 = tile * kHistTile;
  const int64_t t1 = min(t0 + kHistTile, p.T);
  const int64_t w0 = min(t0 + 32 * warp, t1), w1 = min(w0 + 32, t1);
  const int64_t r0 = w0 * p.K, r1 = w1 * p.K;
  const unsigned lt_mask = (1u << lane) - 1u;
  int my_e[kMaxTopK], my_rank[kMaxTopK];
#pragma unroll
  for (int k = 0; k < kMaxTopK; ++k) {
    my_e[k] = -1;
    my_rank[k] = 0;
    if (k >= p.K) continue;
    const int64_t r = r0 + 32 * k + lane;
    int e = -1;
    if (r < r1) {
      e = p.topk_idx[r];
      if (e < 0 || e >= p.N) e = -1;   // reported by the count kernel
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & lt_mask);
    int base = 0;
    if (e >= 0) base = wcnt[warp][e];
    __syncwarp();
    if (e >= 0 && rank == 0) wcnt[warp][e] = static_cast<uint16_t>(base + __popc(same));
    __syncwarp();
    my_e[k] = e;
    my_rank[k] = base + rank;
  }
  __syncthreads();
  // exclusive prefix over the tile's warps (the routes from earlier tiles are added below)
  for (int e = threadIdx.x; e < p.N; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int c = wcnt[w][e];
      wcnt[w][e] = static_cast<uint16_t>(run);
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kMaxTopK; ++k) {
    if (k >= p.K) continue;
    const int64_t r = r0 + 32 * k + lane;
    if (r >= r1) continue;
    const int e = my_e[k];
    const int64_t t = r / p.K;
    const int g = e >= 0 ? seed[e] + wcnt[warp][e] + my_rank[k] : 0;
    if (e >= 0 && g < ckeep[e]) {
      const int pos = offs[e] + g;
      p.route_pos[r] = pos;
      p.perm_src[pos] = static_cast<int32_t>(t);
    } else {
      p.route_pos[r] = -1;
      atomicAdd(&drops[t - t0], 1);
    }
  }
  __syncthreads();
  if (p.drop_stats && warp == 0) {
    int lost_any = 0, lost_all = 0;
    for (int64_t t = t0 + lane; t < t1; t += 32) {
      const int d = drops[t - t0];
      lost_any += d > 0;
      lost_all += d == p.K;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      lost_any += __shfl_xor_sync(0xffffffffu, lost_any, off);
      lost_all += __shfl_xor_sync(0xffffffffu, lost_all, off);
    }
    if (lane == 0) {
      if (lost_any) atomicAdd(&p.drop_stats[1], lost_any);
      if (lost_all) atomicAdd(&p.drop_stats[2], lost_all);
    }
  }
}

__global__ void __launch_bounds__(256) place_kernel(PermuteParams p) {
  __shared__ int ckeep[kMaxExperts];
  __shared__ int offs[kMaxExperts];
  __shared__ uint16_t wcnt[8][kMaxExperts];
  __shared__ int drops[kHistTile];
  for (int e = threadIdx.x; e < p.N; e += blockDim.x) {
    ckeep[e] = p.counts_keep[e];
    offs[e] = p.offsets[e];
  }
  __syncthreads();
  // after the scan, hist holds the per-expert exclusive prefix over tiles
  place_tile(p, blockIdx.x, ckeep, offs, p.hist + static_cast<int64_t>(blockIdx.x) * p.N, wcnt,
             drops);
}

// Grid barrier of a cooperative launch (every CTA resident at once).  count and gen sit on
// separate lines of the workspace header: both zero after moe_workspace_init, and count is
// zero again after every barrier (the last CTA to arrive resets it, then advances gen).
// The wait is bounded by %globaltimer: a barrier that runs out records MOE_ERR_TIMEOUT and
// the CTAs that gave up return false.
constexpr uint64_t kBarrierLimitNs = 1000000000ull;

__device__ bool grid_barrier(unsigned* count, unsigned* gen, unsigned nblocks, int32_t* status) {
  __shared__ int ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile unsigned* vgen = gen;
    const unsigned g0 = *vgen;   // read before arriving: gen cannot advance without us
    ok = 1;
    __threadfence();             // this CTA's writes before its arrival
    if (atomicAdd(count, 1u) == nblocks - 1) {
      atomicExch(count, 0u);
      __threadfence();
      atomicAdd(gen, 1u);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (*vgen == g0) {
        if (globaltimer_ns() - t0 > kBarrierLimitNs) {
          set_status(status, MOE_ERR_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
  return ok != 0;
}

// The whole counting / capacity / placing pass in one launch: one CTA per tile of 256
// tokens, all resident (cooperative launch).  Each CTA counts its tile into hist, waits
// at a grid barrier, sums the histograms of all tiles per expert (the requests from
// earlier tiles and in total: every CTA the same totals), applies the capacity rule and
// the offsets in shared memory, and places its tile's routes; CTA 0 writes the layer-wide
// results.  The same results as count, scan and place, bit for bit.
__global__ void __launch_bounds__(256) permute_fused_kernel(PermuteParams p) {
  // About 9 KB of shared memory, so that a CTA fits on an SM beside a running expert-GEMM
  // CTA (which leaves ~14 KB) and the cooperative launch need not wait for those to end.
  // One region serves, in turn, as this tile's histogram, as the capacity step's prefix of
  // 128-row tiles and destination totals, and as the placing step's per-warp counters.
  __shared__ __align__(16) uint16_t region[8][kMaxExperts];
  __shared__ int before[kMaxExperts];   // requests to each expert from earlier tiles
  __shared__ int creq[kMaxExperts];
  __shared__ int ckeep[kMaxExperts];
  __shared__ int offs[kMaxExperts + 1];
  __shared__ int drops[kHistTile];
  __shared__ int dropped;
  static_assert(sizeof(region) >= sizeof(int) * (3 * kMaxExperts + 1), "region too small");
  int* cnt = reinterpret_cast<int*>(region);
  int* tprefix = reinterpret_cast<int*>(region);
  int* rreq = tprefix + kMaxExperts + 1;
  int* rkeep = rreq + kMaxExperts;
  const int64_t tile = blockIdx.x;
  const int ntiles = gridDim.x;
  for (int e = threadIdx.x; e < p.N; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int64_t t0 = tile * kHistTile;
  const int64_t t1 = min(t0 + kHistTile, p.T);
  for (int64_t r = t0 * p.K + threadIdx.x; r < t1 * p.K; r += blockDim.x) {
    const int e = p.topk_idx[r];
    if (e < 0 || e >= p.N) {
      set_status(p.status, MOE_ERR_DEVICE_BOUNDS);
      continue;
    }
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < p.N; e += blockDim.x) p.hist[tile * p.N + e] = cnt[e];
  __syncthreads();   // the region is reused after the barrier
  // the per-token drop tallies start at zero before any CTA adds to them
  if (tile == 0 && threadIdx.x == 0 && p.drop_stats) {
    p.drop_stats[1] = 0;
    p.drop_stats[2] = 0;
  }
  if (!grid_barrier(p.barrier, p.barrier + 16, static_cast<unsigned>(ntiles), p.status)) return;
  for (int e = threadIdx.x; e < p.N; e += blockDim.x) {
    int b = 0, total = 0;
    for (int t = 0; t < ntiles; ++t) {
      const int v = __ldcg(p.hist + static_cast<int64_t>(t) * p.N + e);
      b += t < tile ? v : 0;
      total += v;
    }
    before[e] = b;
    creq[e] = total;
  }
  __syncthreads();
  capacity_and_offsets(p, creq, ckeep, offs, tprefix, rreq, rkeep, &dropped);
  if (tile == 0) write_layer_results(p, creq, ckeep, offs, tprefix, rreq, rkeep, dropped, false);
  __syncthreads();   // the region becomes the placing step's counters
  place_tile(p, tile, ckeep, offs, before, region, drops);
}

// One warp per token: each 16-byte piece of x[t] is read once and written to the
// packed rows of all of t's kept routes.  A lane issues four loads before their stores
// (the source and destination never overlap), so each warp keeps several reads in flight.
__global__ void __launch_bounds__(256) gather_kernel(PermuteParams p) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (t >= p.T) return;
  const int64_t cap = p.T * p.K;
  int64_t dst[kMaxTopK];   // packed row of slot k, or -1 (dropped or no slot)
#pragma unroll
  for (int k = 0; k < kMaxTopK; ++k) {
    dst[k] = -1;
    if (k < p.K) {
      const int32_t pos = p.route_pos[t * p.K + k];
      if (pos >= cap) set_status(p.status, MOE_ERR_DEVICE_BOUNDS);
      else if (pos >= 0) dst[k] = pos;
    }
  }
  const int64_t nvec = static_cast<int64_t>(p.d) * p.elem_bytes / 16;
  const int4* __restrict__ src =
      reinterpret_cast<const int4*>(static_cast<const char*>(p.x) + t * nvec * 16);
  int4* __restrict__ out = static_cast<int4*>(p.x_perm);
  constexpr int U = 4;
  for (int64_t v0 = lane; v0 < nvec; v0 += 32 * U) {
    int4 val[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (v0 + u * 32 < nvec) val[u] = src[v0 + u * 32];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + u * 32;
      if (v < nvec) {
#pragma unroll
        for (int k = 0; k < kMaxTopK; ++k)
          if (dst[k] >= 0) out[dst[k] * nvec + v] = val[u];
      }
    }
  }
}

__global__ void tile_prefix_kernel(const int32_t* offsets, int32_t N, int32_t* tile_prefix,
                                   int32_t* status) {
  if (threadIdx.x != 0) return;
  int acc = 0;
  tile_prefix[0] = 0;
  for (int e = 0; e < N; ++e) {
    const int m = offsets[e + 1] - offsets[e];
    if (m < 0) {
      set_status(status, MOE_ERR_DEVICE_BOUNDS);
      acc = 0x3fffffff;  // no valid tile walk exists; make every later prefix huge but finite
    } else {
      acc += (m + kTcRows - 1) / kTcRows;
    }
    tile_prefix[e + 1] = acc;
  }
}

}  // namespace

// Largest grid of the one-launch permutation that is resident at once (cached per device).
int fused_permute_capacity() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, permute_fused_kernel, 256, 0) !=
      cudaSuccess)
    per_sm = 0;
  const int cap = per_sm * device_sm_count();
  if (dev >= 0 && dev < 64) cached[dev] = cap > 0 ? cap : -1;
  return cap;
}

cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s) {
  const unsigned tiles = static_cast<unsigned>(p.hist_tiles);
  if (p.T > 0 && p.barrier != nullptr && static_cast<int64_t>(tiles) <= fused_permute_capacity()) {
    // count, scan and place in one cooperative launch
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, permute_fused_kernel, p);
    if (e != cudaSuccess) return e;
    if (p.x_perm == nullptr) return cudaSuccess;
    gather_kernel<<<static_cast<unsigned>((p.T + 7) / 8), 256, 0, s>>>(p);
    return cudaGetLastError();
  }
  if (p.T > 0) {
    count_kernel<<<tiles, 256, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  scan_kernel<<<1, 1024, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.T == 0) return e;
  place_kernel<<<tiles, 256, 0, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.x_perm == nullptr) return cudaSuccess;   // the expert GEMM gathers rows itself
  gather_kernel<<<static_cast<unsigned>((p.T + 7) / 8), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tile_prefix(const int32_t* offsets, int32_t N, int32_t* tile_prefix,
                               int32_t* status, cudaStream_t s) {
  tile_prefix_kernel<<<1, 32, 0, s>>>(offsets, N, tile_prefix, status);
  return cudaGetLastError();
}

}  // namespace moe

// Requested and kept counts, capacity, packed offsets and the row permutation.
//
// Follows Section 10 "Routing, Capacity, and Load Balancing": Eq. 19 (requested
// counts), Eq. 20-21 (destination totals, kept counts, drops), Eq. 23 / Eq. 25
// (rank-wide and per-expert budgets), the admission order of Section 10.3
// (local-expert-major, a prefix of each expert's requests in token order),
// Eq. 26 (kept rows packed densely per expert, offsets o_e) and Eq. 27 (drops).
//
// A stable counting sort, four launches, no atomics on positions:
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
      dropped = drop;
    }
  }
  __syncthreads();

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
    p.drop_stats[1] = 0;
    p.drop_stats[2] = 0;
    p.drop_stats[3] = 0;
  }
}

// One CTA (8 warps) per 256-token tile.  Warp w owns tokens [32w, 32w+32) of the
// tile; its 32*K routes in (token, slot) order are ranked within the warp with
// __match_any_sync (round k holds routes [32k, 32k+32) of the warp's range).  A
// per-expert exclusive prefix over the warps, seeded with the routes to that
// expert from earlier tiles, then gives every route its rank among all requests
// to its expert in token order.
__global__ void __launch_bounds__(256) place_kernel(PermuteParams p) {
  __shared__ int wcnt[8][kMaxExperts];   // per-warp counts, then per-warp bases
  __shared__ int ckeep[kMaxExperts];
  __shared__ int offs[kMaxExperts];
  __shared__ int drops[kHistTile];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t tile = blockIdx.x;
  for (int e = threadIdx.x; e < p.N; e += blockDim.x) {
    ckeep[e] = p.counts_keep[e];
    offs[e] = p.offsets[e];
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
    if (e >= 0 && rank == 0) wcnt[warp][e] = base + __popc(same);
    __syncwarp();
    my_e[k] = e;
    my_rank[k] = base + rank;
  }
  __syncthreads();
  // exclusive prefix over warps, seeded with the routes from earlier tiles
  for (int e = threadIdx.x; e < p.N; e += blockDim.x) {
    int run = p.hist[tile * p.N + e];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int c = wcnt[w][e];
      wcnt[w][e] = run;
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
    const int g = e >= 0 ? wcnt[warp][e] + my_rank[k] : 0;
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

cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s) {
  const unsigned tiles = static_cast<unsigned>(p.hist_tiles);
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

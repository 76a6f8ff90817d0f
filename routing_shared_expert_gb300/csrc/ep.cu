// Expert-parallel capacity agreement and dispatch plan (Section 10.3): the keep matrix every
// rank derives from the all-gathered requested split counts, each route's destination row,
// the send and receive layouts of the exchange, and the indexed row copies that fill and
// drain the exchange buffers (ep_plan.h holds the rules, shared by the device kernels and
// the host entry points).
//
// The device entries are sync-free: the gathered counts stay on the device, the token
// count over all sources is recovered from them (K requests per token), and a source's
// routes get their destination rows from the stable ranks moe_permute computes.
#include <cstring>

#include "common.cuh"
#include "ep_plan.h"
#include "internal.h"

namespace moe {
namespace {

struct EpKeepArgs {
  const int32_t* counts;   // [M][N] device
  int32_t M, N, K, cap_policy;
  double capacity_factor;
  int32_t rho[kMaxExperts];
  int32_t* keep;
  int32_t* recv_off;
  int32_t* R_req;
  int32_t* R_keep;
};

constexpr int kEpThreads = 256;   // every kernel below: one thread per expert fits (N <= 256)

// Exclusive prefix of v over the kEpThreads threads of the block in thread order; *total
// receives the block's sum.  Every thread of the block calls it.
__device__ int64_t block_exclusive_scan(int64_t v, int64_t* total) {
  __shared__ int64_t warp_sums[kEpThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  int64_t before = 0, all = 0;
#pragma unroll
  for (int i = 0; i < kEpThreads / 32; ++i) {
    const int64_t ws = warp_sums[i];
    before += i < w ? ws : 0;
    all += ws;
  }
  __syncthreads();   // warp_sums is reused by the next call
  *total = all;
  return before + x - v;
}

// One block per destination rank q: the rule of ep_keep_dest in parallel.  Along q's
// sequence of splits (its experts in ascending index, within an expert the sources in
// ascending rank), with P the requests of the splits before one and B the budget, the
// cumulative admission keeps min(c, max(0, B - P)) of a split's c requests at row
// min(P, B) of q's buffer (no policy: all c at row P): a prefix sum of the requests.
__global__ void __launch_bounds__(kEpThreads) ep_keep_kernel(EpKeepArgs a) {
  __shared__ int32_t local[kMaxExperts];   // q's experts in ascending index
  const int q = blockIdx.x;
  const int64_t splits = static_cast<int64_t>(a.M) * a.N;
  // tokens over all sources (K requests each) give the budget
  int64_t part = 0;
  for (int64_t i = threadIdx.x; i < splits; i += kEpThreads) part += a.counts[i];
  int64_t routes = 0;
  block_exclusive_scan(part, &routes);
  const int64_t B = ep_rank_budget(a.capacity_factor, a.K, routes / a.K, a.M);
  const int e = threadIdx.x;
  const bool mine = e < a.N && a.rho[e] == q;
  int64_t n_local = 0;
  const int64_t li = block_exclusive_scan(mine ? 1 : 0, &n_local);
  if (mine) local[li] = e;
  __syncthreads();
  const int64_t L = n_local * a.M;
  int64_t carry = 0;   // requests of the splits before this chunk
  for (int64_t base = 0; base < L; base += kEpThreads) {
    const int64_t j = base + threadIdx.x;
    int64_t c = 0, idx = -1;
    if (j < L) {
      const int ee = local[j / a.M], src = static_cast<int>(j % a.M);
      idx = static_cast<int64_t>(src) * a.N + ee;
      c = a.counts[idx];
    }
    int64_t chunk = 0;
    const int64_t P = carry + block_exclusive_scan(c, &chunk);
    if (idx >= 0) {
      int64_t k = c, row = P;
      if (a.cap_policy == MOE_CAP_RANK_WIDE) {
        const int64_t left = B - P;
        k = left < c ? (left > 0 ? left : 0) : c;
        row = P < B ? P : B;
      }
      a.keep[idx] = static_cast<int32_t>(k);
      a.recv_off[idx] = static_cast<int32_t>(row);
    }
    carry += chunk;
  }
  if (threadIdx.x == 0) {
    if (a.R_req) a.R_req[q] = static_cast<int32_t>(carry);
    if (a.R_keep)
      a.R_keep[q] = static_cast<int32_t>(a.cap_policy == MOE_CAP_RANK_WIDE && carry > B ? B : carry);
  }
}

// One thread per route of the source rank: its rank among the source's requests to its
// expert is route_pos - offsets[e] of a capacity-free moe_permute of the source's batch.
__global__ void ep_place_kernel(const int32_t* topk_idx, const int32_t* route_pos,
                                const int32_t* offsets, const int32_t* keep,
                                const int32_t* recv_off, int64_t routes, int32_t N, int32_t src,
                                int32_t* dst_row, int32_t* status) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= routes) return;
  const int e = topk_idx[r];
  const int pos = route_pos[r];
  if (e < 0 || e >= N || pos < 0) {
    set_status(status, MOE_ERR_DEVICE_BOUNDS);
    dst_row[r] = -1;
    return;
  }
  dst_row[r] = ep_place_route(src, N, e, pos - offsets[e], keep, recv_off);
}

struct EpSendArgs {
  int32_t rho[kMaxExperts];
  int32_t M, N, K, src;
  int64_t routes;
  const int32_t* topk_idx;
  const int32_t* keep;
  const int32_t* recv_off;
  const int32_t* dst_row;
  int32_t* send_pos;
  int32_t* send_counts;
  int32_t* status;
};

// One thread per route.  Every block first lays out the source's send buffer (the rule of
// ep_send_base, one thread per expert): base[e] sums the source's kept routes of the
// experts before e in the order (destination rank, expert index).
__global__ void __launch_bounds__(kEpThreads) ep_send_pos_kernel(EpSendArgs a) {
  __shared__ int32_t base[kMaxExperts];
  __shared__ int32_t kept[kMaxExperts];
  for (int e = threadIdx.x; e < a.N; e += kEpThreads)
    kept[e] = a.keep[static_cast<int64_t>(a.src) * a.N + e];
  __syncthreads();
  for (int e = threadIdx.x; e < a.N; e += kEpThreads) {
    const int q = a.rho[e];
    int64_t b = 0;
    for (int e2 = 0; e2 < a.N; ++e2) {
      const int q2 = a.rho[e2];
      b += (q2 < q || (q2 == q && e2 < e)) ? kept[e2] : 0;
    }
    base[e] = static_cast<int32_t>(b);
  }
  if (blockIdx.x == 0 && a.send_counts) {
    for (int q = threadIdx.x; q < a.M; q += kEpThreads) {
      int64_t n = 0;
      for (int e2 = 0; e2 < a.N; ++e2) n += a.rho[e2] == q ? kept[e2] : 0;
      a.send_counts[q] = static_cast<int32_t>(n);
    }
  }
  __syncthreads();
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= a.routes) return;
  const int e = a.topk_idx[r];
  if (e < 0 || e >= a.N) {
    set_status(a.status, MOE_ERR_DEVICE_BOUNDS);
    a.send_pos[r] = -1;
    return;
  }
  a.send_pos[r] = ep_send_pos_route(a.src, a.N, e, a.dst_row[r], base, a.recv_off);
}

struct EpRecvArgs {
  int32_t rho[kMaxExperts];
  int32_t M, N, q;
  const int32_t* keep;
  const int32_t* recv_off;
  int32_t* recv_row;
  int64_t cap;
  int32_t* status;
};

// One block per source s: its rows sit in the receive buffer after the earlier sources'
// (the rule of ep_recv_rows), and within source s its splits of q's experts follow in
// ascending expert index; a block sum and a scan over the experts give each split's first
// receive row, then the block writes the split's rows one after another.
__global__ void __launch_bounds__(kEpThreads) ep_recv_rows_kernel(EpRecvArgs a) {
  __shared__ int64_t first[kMaxExperts];
  __shared__ int32_t rho[kMaxExperts];
  for (int e = threadIdx.x; e < a.N; e += kEpThreads) rho[e] = a.rho[e];
  __syncthreads();
  const int s = blockIdx.x;
  int64_t part = 0;   // rows of q's receive buffer from sources before s
  for (int64_t i = threadIdx.x; i < static_cast<int64_t>(s) * a.N; i += kEpThreads)
    part += rho[i % a.N] == a.q ? a.keep[i] : 0;
  int64_t before = 0;
  block_exclusive_scan(part, &before);
  const int e = threadIdx.x;
  const bool mine = e < a.N && a.rho[e] == a.q;
  int64_t total = 0;
  const int64_t pre =
      block_exclusive_scan(mine ? a.keep[static_cast<int64_t>(s) * a.N + e] : 0, &total);
  if (e < a.N) first[e] = before + pre;
  __syncthreads();
  for (int e2 = 0; e2 < a.N; ++e2) {
    if (a.rho[e2] != a.q) continue;
    const int64_t i = static_cast<int64_t>(s) * a.N + e2;
    const int32_t n = a.keep[i], off = a.recv_off[i];
    const int64_t j0 = first[e2];
    for (int32_t r = threadIdx.x; r < n; r += kEpThreads) {
      if (j0 + r >= a.cap) {
        set_status(a.status, MOE_ERR_DEVICE_BOUNDS);
        break;
      }
      a.recv_row[j0 + r] = off + r;
    }
  }
}

struct RowsCopyArgs {
  const int4* src;
  int64_t src_rows;
  const int32_t* src_index;
  int64_t src_div;
  int4* dst;
  int64_t dst_rows;
  const int32_t* dst_index;
  int64_t n;
  int64_t nvec;   // 16-byte vectors per row
  int32_t zero_missing;
  int32_t* status;
};

// One warp per copied row: dst[dst row] = src[src row], four 16-byte loads in flight per lane.
__global__ void __launch_bounds__(256) rows_copy_kernel(RowsCopyArgs a) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (i >= a.n) return;
  const int64_t t = a.dst_index ? a.dst_index[i] : i;
  if (t < 0) return;
  const int64_t sr = a.src_index ? a.src_index[i] : i / a.src_div;
  if (t >= a.dst_rows || sr >= a.src_rows) {
    if (lane == 0) set_status(a.status, MOE_ERR_DEVICE_BOUNDS);
    return;
  }
  int4* out = a.dst + t * a.nvec;
  if (sr < 0) {
    if (a.zero_missing)
      for (int64_t v = lane; v < a.nvec; v += 32) out[v] = make_int4(0, 0, 0, 0);
    return;
  }
  const int4* __restrict__ in = a.src + sr * a.nvec;
  constexpr int U = 4;
  for (int64_t v0 = lane; v0 < a.nvec; v0 += 32 * U) {
    int4 val[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (v0 + u * 32 < a.nvec) val[u] = in[v0 + u * 32];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (v0 + u * 32 < a.nvec) out[v0 + u * 32] = val[u];
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

namespace {

moe_status check_rho(int32_t M, int32_t N, const int32_t* rho) {
  if (M < 1 || M > kMaxExperts || N < 1 || N > kMaxExperts || !rho) return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < N; ++e)
    if (rho[e] < 0 || rho[e] >= M) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status check_rows_copy(const void* src, int64_t src_rows, int64_t src_div, const void* dst,
                           int64_t dst_rows, int64_t n, int64_t row_bytes) {
  if (n < 0 || src_rows < 0 || dst_rows < 0 || row_bytes <= 0 || src_div < 1) return MOE_ERR_INVALID_ARG;
  if (row_bytes % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if (n > 0 && (!dst || (src_rows > 0 && !src))) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u))
    return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

moe_status check_ep(int32_t M, int32_t N, int32_t K, int32_t cap_policy, double c,
                    const int32_t* rho) {
  if (M < 1 || M > kMaxExperts || N < 1 || N > kMaxExperts || K < 1 || K > N || !rho)
    return MOE_ERR_INVALID_ARG;
  if (cap_policy != MOE_CAP_NONE && cap_policy != MOE_CAP_RANK_WIDE) return MOE_ERR_UNSUPPORTED;
  if (cap_policy == MOE_CAP_RANK_WIDE && !(c > 0.0 && c < 1e9)) return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < N; ++e)
    if (rho[e] < 0 || rho[e] >= M) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_ep_keep_matrix(int32_t M, int32_t N, int32_t K, const int32_t* rho,
                              int32_t cap_policy, double capacity_factor, const int32_t* counts,
                              int32_t* keep, int32_t* recv_off, int32_t* R_req, int32_t* R_keep,
                              cudaStream_t stream) {
  moe_status s = check_ep(M, N, K, cap_policy, capacity_factor, rho);
  if (s != MOE_OK) return s;
  if (!counts || !keep || !recv_off) return MOE_ERR_INVALID_ARG;
  EpKeepArgs a{};
  a.counts = counts;
  a.M = M;
  a.N = N;
  a.K = K;
  a.cap_policy = cap_policy;
  a.capacity_factor = capacity_factor;
  std::memcpy(a.rho, rho, sizeof(int32_t) * N);
  a.keep = keep;
  a.recv_off = recv_off;
  a.R_req = R_req;
  a.R_keep = R_keep;
  ep_keep_kernel<<<static_cast<unsigned>(M), kEpThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_ep_place(int32_t M, int32_t src_rank, int64_t T, int32_t N, int32_t K,
                        const int32_t* topk_idx,
                        const int32_t* route_pos, const int32_t* offsets, const int32_t* keep,
                        const int32_t* recv_off, int32_t* dst_row, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  if (M < 1 || M > kMaxExperts || T < 0 || N < 1 || N > kMaxExperts || K < 1 || K > N ||
      src_rank < 0 || src_rank >= M)
    return MOE_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < 256) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!topk_idx || !route_pos || !offsets || !keep || !recv_off || !dst_row) return MOE_ERR_INVALID_ARG;
  const int64_t routes = T * K;
  ep_place_kernel<<<static_cast<unsigned>((routes + 255) / 256), 256, 0, stream>>>(
      topk_idx, route_pos, offsets, keep, recv_off, routes, N, src_rank, dst_row,
      static_cast<int32_t*>(workspace));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_ep_keep_matrix_host(int32_t M, int32_t N, int32_t K, const int32_t* rho,
                                   int32_t cap_policy, double capacity_factor,
                                   const int32_t* counts, int32_t* keep, int32_t* recv_off,
                                   int32_t* R_req, int32_t* R_keep) {
  moe_status s = check_ep(M, N, K, cap_policy, capacity_factor, rho);
  if (s != MOE_OK) return s;
  if (!counts || !keep || !recv_off) return MOE_ERR_INVALID_ARG;
  for (int64_t i = 0; i < static_cast<int64_t>(M) * N; ++i)
    if (counts[i] < 0) return MOE_ERR_INVALID_ARG;
  ep_keep_matrix(counts, M, N, rho, cap_policy, capacity_factor, K, keep, recv_off, R_req, R_keep);
  return MOE_OK;
}

moe_status moe_ep_place_host(int32_t M, int32_t src_rank, int64_t T, int32_t N, int32_t K,
                             const int32_t* topk_idx, const int32_t* keep,
                             const int32_t* recv_off, int32_t* dst_row) {
  if (M < 1 || M > kMaxExperts || T < 0 || N < 1 || N > kMaxExperts || K < 1 || K > N ||
      src_rank < 0 || src_rank >= M)
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!topk_idx || !keep || !recv_off || !dst_row) return MOE_ERR_INVALID_ARG;
  int32_t seen[kMaxExperts] = {};
  for (int64_t r = 0; r < T * K; ++r) {   // (token, slot) order: token order per expert
    const int32_t e = topk_idx[r];
    if (e < 0 || e >= N) return MOE_ERR_INVALID_ARG;
    dst_row[r] = ep_place_route(src_rank, N, e, seen[e]++, keep, recv_off);
  }
  return MOE_OK;
}

}  // extern "C"

extern "C" {

moe_status moe_ep_send_pos(int32_t M, int32_t src_rank, int64_t T, int32_t N, int32_t K,
                           const int32_t* rho, const int32_t* topk_idx, const int32_t* keep,
                           const int32_t* recv_off, const int32_t* dst_row, int32_t* send_pos,
                           int32_t* send_counts, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  moe_status s = check_rho(M, N, rho);
  if (s != MOE_OK) return s;
  if (T < 0 || K < 1 || K > N || src_rank < 0 || src_rank >= M) return MOE_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < 256 || !keep) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !recv_off || !dst_row || !send_pos)) return MOE_ERR_INVALID_ARG;
  EpSendArgs a{};
  std::memcpy(a.rho, rho, sizeof(int32_t) * N);
  a.M = M;
  a.N = N;
  a.K = K;
  a.src = src_rank;
  a.routes = T * K;
  a.topk_idx = topk_idx;
  a.keep = keep;
  a.recv_off = recv_off;
  a.dst_row = dst_row;
  a.send_pos = send_pos;
  a.send_counts = send_counts;
  a.status = static_cast<int32_t*>(workspace);
  const int64_t blocks = a.routes > 0 ? (a.routes + 255) / 256 : 1;   // block 0 writes the counts
  ep_send_pos_kernel<<<static_cast<unsigned>(blocks), kEpThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_ep_recv_rows(int32_t M, int32_t dst_rank, int32_t N, const int32_t* rho,
                            const int32_t* keep, const int32_t* recv_off, int32_t* recv_row,
                            int64_t recv_cap, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  moe_status s = check_rho(M, N, rho);
  if (s != MOE_OK) return s;
  if (dst_rank < 0 || dst_rank >= M || recv_cap < 0) return MOE_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < 256 || !keep || !recv_off) return MOE_ERR_INVALID_ARG;
  if (recv_cap > 0 && !recv_row) return MOE_ERR_INVALID_ARG;
  EpRecvArgs a{};
  std::memcpy(a.rho, rho, sizeof(int32_t) * N);
  a.M = M;
  a.N = N;
  a.q = dst_rank;
  a.keep = keep;
  a.recv_off = recv_off;
  a.recv_row = recv_row;
  a.cap = recv_cap;
  a.status = static_cast<int32_t*>(workspace);
  ep_recv_rows_kernel<<<static_cast<unsigned>(M), kEpThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_rows_copy(const void* src, int64_t src_rows, const int32_t* src_index,
                         int64_t src_div, void* dst, int64_t dst_rows, const int32_t* dst_index,
                         int64_t n, int64_t row_bytes, int32_t zero_missing, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  moe_status s = check_rows_copy(src, src_rows, src_div, dst, dst_rows, n, row_bytes);
  if (s != MOE_OK) return s;
  if (!workspace || workspace_bytes < 256) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  RowsCopyArgs a{};
  a.src = static_cast<const int4*>(src);
  a.src_rows = src_rows;
  a.src_index = src_index;
  a.src_div = src_div;
  a.dst = static_cast<int4*>(dst);
  a.dst_rows = dst_rows;
  a.dst_index = dst_index;
  a.n = n;
  a.nvec = row_bytes / 16;
  a.zero_missing = zero_missing ? 1 : 0;
  a.status = static_cast<int32_t*>(workspace);
  rows_copy_kernel<<<static_cast<unsigned>((n + 7) / 8), 256, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_ep_send_pos_host(int32_t M, int32_t src_rank, int64_t T, int32_t N, int32_t K,
                                const int32_t* rho, const int32_t* topk_idx, const int32_t* keep,
                                const int32_t* recv_off, const int32_t* dst_row,
                                int32_t* send_pos, int32_t* send_counts) {
  moe_status s = check_rho(M, N, rho);
  if (s != MOE_OK) return s;
  if (T < 0 || K < 1 || K > N || src_rank < 0 || src_rank >= M || !keep) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !recv_off || !dst_row || !send_pos)) return MOE_ERR_INVALID_ARG;
  int32_t base[kMaxExperts];
  ep_send_base(src_rank, M, N, rho, keep, base, send_counts);
  for (int64_t r = 0; r < T * K; ++r) {
    const int32_t e = topk_idx[r];
    if (e < 0 || e >= N) return MOE_ERR_INVALID_ARG;
    send_pos[r] = ep_send_pos_route(src_rank, N, e, dst_row[r], base, recv_off);
  }
  return MOE_OK;
}

moe_status moe_ep_recv_rows_host(int32_t M, int32_t dst_rank, int32_t N, const int32_t* rho,
                                 const int32_t* keep, const int32_t* recv_off, int32_t* recv_row,
                                 int64_t recv_cap) {
  moe_status s = check_rho(M, N, rho);
  if (s != MOE_OK) return s;
  if (dst_rank < 0 || dst_rank >= M || recv_cap < 0 || !keep || !recv_off) return MOE_ERR_INVALID_ARG;
  int64_t need = 0;
  for (int32_t q = 0; q < M; ++q)
    for (int32_t e = 0; e < N; ++e)
      if (rho[e] == dst_rank) need += keep[static_cast<int64_t>(q) * N + e];
  if (need > recv_cap || (need > 0 && !recv_row)) return MOE_ERR_INVALID_ARG;
  ep_recv_rows(dst_rank, M, N, rho, keep, recv_off, recv_row);
  return MOE_OK;
}

moe_status moe_rows_copy_host(const void* src, int64_t src_rows, const int32_t* src_index,
                              int64_t src_div, void* dst, int64_t dst_rows,
                              const int32_t* dst_index, int64_t n, int64_t row_bytes,
                              int32_t zero_missing) {
  moe_status s = check_rows_copy(src, src_rows, src_div, dst, dst_rows, n, row_bytes);
  if (s != MOE_OK) return s;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t t = dst_index ? dst_index[i] : i;
    if (t < 0) continue;
    const int64_t sr = src_index ? src_index[i] : i / src_div;
    if (t >= dst_rows || sr >= src_rows) return MOE_ERR_INVALID_ARG;
    char* out = static_cast<char*>(dst) + t * row_bytes;
    if (sr < 0) {
      if (zero_missing) std::memset(out, 0, static_cast<size_t>(row_bytes));
      continue;
    }
    std::memcpy(out, static_cast<const char*>(src) + sr * row_bytes, static_cast<size_t>(row_bytes));
  }
  return MOE_OK;
}

}  // extern "C"

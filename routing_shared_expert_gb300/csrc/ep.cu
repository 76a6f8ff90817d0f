// Expert-parallel capacity agreement and dispatch plan (Section 10.3): the keep matrix every
// rank derives from the all-gathered requested split counts, and each route's destination
// row (ep_plan.h holds the rules, shared by the device kernels and the host entry points).
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

// One thread per destination rank; every thread recomputes the (small) route total.
__global__ void ep_keep_kernel(EpKeepArgs a) {
  const int q = threadIdx.x;
  if (q >= a.M) return;
  const int64_t B =
      ep_rank_budget(a.capacity_factor, a.K, ep_total_tokens(a.counts, a.M, a.N, a.K), a.M);
  ep_keep_dest(q, a.counts, a.M, a.N, a.rho, a.cap_policy, B, a.keep, a.recv_off, a.R_req,
               a.R_keep);
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

}  // namespace
}  // namespace moe

using namespace moe;

namespace {

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
  ep_keep_kernel<<<1, 256, 0, stream>>>(a);
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

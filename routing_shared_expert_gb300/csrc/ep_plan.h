// Expert-parallel capacity agreement and dispatch plan (Section 10 "Routing, Capacity, and
// Load Balancing", Section 10.3 and Eq. 23, Eq. 26, Figure 41), written once for the host
// and the device.
//
// With M source ranks, every rank all-gathers the requested split counts C^req[s][e] (the
// routes rank s's tokens send to expert e) and derives the same keep matrix: each
// destination rank q, with budget B = max(1, ceil(c K T / M)) for T tokens over all
// sources (Eq. 23, T_route = K T / M per source), flattens its local experts (those with
// rho(e) = q) in ascending expert index, and within an expert the sources in ascending
// rank, and admits routes cumulatively until B is used; a source keeps a prefix, in its
// token order, of each of its splits.  The destination packs, per local expert in
// ascending index, the rows of source 0, then source 1, ... (Eq. 26 offsets over the
// local experts): recv_off[s][e] is the first row of split (s, e) in that buffer.
// Without a capacity policy every request is kept.
#pragma once

#include <stdint.h>

#include "moe_gb300.h"

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__
#else
#define MOE_HD
#endif

namespace moe {

// Budget of one destination rank: B = max(1, ceil(c K T / M)) computed in double, as the
// single-device rank-wide rule with the batch spread evenly over the M ranks.
MOE_HD inline int64_t ep_rank_budget(double capacity_factor, int32_t K, int64_t T_total,
                                     int32_t M) {
  const double v = capacity_factor * static_cast<double>(K) * static_cast<double>(T_total) /
                   static_cast<double>(M);
  int64_t b = static_cast<int64_t>(v);
  if (static_cast<double>(b) < v) ++b;
  return b < 1 ? 1 : b;
}

// Destination rank q's part of the keep matrix (destinations are independent): keep and
// recv_off of the splits (s, e) with rho[e] = q; R_req[q] / R_keep[q] when given.
// cap_policy: MOE_CAP_NONE keeps every request, MOE_CAP_RANK_WIDE applies budget B.
MOE_HD inline void ep_keep_dest(int32_t q, const int32_t* counts, int32_t M, int32_t N,
                                const int32_t* rho, int32_t cap_policy, int64_t B, int32_t* keep,
                                int32_t* recv_off, int32_t* R_req, int32_t* R_keep) {
  {
    int64_t used = 0, req = 0;
    int64_t row = 0;   // next row of destination q's packed buffer
    for (int32_t e = 0; e < N; ++e) {
      if (rho[e] != q) continue;
      for (int32_t s = 0; s < M; ++s) {
        const int64_t c = counts[static_cast<int64_t>(s) * N + e];
        int64_t k = c;
        if (cap_policy == MOE_CAP_RANK_WIDE) {
          const int64_t left = B - used;
          k = left < c ? (left > 0 ? left : 0) : c;
        }
        keep[static_cast<int64_t>(s) * N + e] = static_cast<int32_t>(k);
        recv_off[static_cast<int64_t>(s) * N + e] = static_cast<int32_t>(row);
        used += k;
        req += c;
        row += k;
      }
    }
    if (R_req) R_req[q] = static_cast<int32_t>(req);
    if (R_keep) R_keep[q] = static_cast<int32_t>(used);
  }
}

// Tokens over all sources: every token requests exactly K routes.
MOE_HD inline int64_t ep_total_tokens(const int32_t* counts, int32_t M, int32_t N, int32_t K) {
  int64_t routes = 0;
  for (int64_t i = 0; i < static_cast<int64_t>(M) * N; ++i) routes += counts[i];
  return routes / K;
}

// keep[s * N + e], recv_off[s * N + e] from counts[s * N + e] (M sources, N experts, rho[e]
// the destination rank of expert e); R_req / R_keep [M] per destination (may be null).
MOE_HD inline void ep_keep_matrix(const int32_t* counts, int32_t M, int32_t N, const int32_t* rho,
                                  int32_t cap_policy, double capacity_factor, int32_t K,
                                  int32_t* keep, int32_t* recv_off, int32_t* R_req,
                                  int32_t* R_keep) {
  const int64_t B = ep_rank_budget(capacity_factor, K, ep_total_tokens(counts, M, N, K), M);
  for (int32_t q = 0; q < M; ++q)
    ep_keep_dest(q, counts, M, N, rho, cap_policy, B, keep, recv_off, R_req, R_keep);
}

// Placement of one route of source rank `src`: expert e, its rank among src's requests to
// e in token order.  Returns the destination row in rho[e]'s packed buffer, or -1 when
// the route is dropped (its rank is past the split's kept prefix).
MOE_HD inline int32_t ep_place_route(int32_t src, int32_t N, int32_t e, int32_t rank,
                                     const int32_t* keep, const int32_t* recv_off) {
  const int64_t i = static_cast<int64_t>(src) * N + e;
  return rank < keep[i] ? recv_off[i] + rank : -1;
}

// A source's send buffer holds, for each destination rank q in ascending order, the rows it
// sends to q in q's buffer order (q's experts in ascending index, each split's kept prefix in
// token order).  base[e] is the send-buffer position of the first kept route of split
// (src, e); send_counts[q] (may be null) the rows the source sends to q.  base [N], rho [N].
MOE_HD inline void ep_send_base(int32_t src, int32_t M, int32_t N, const int32_t* rho,
                                const int32_t* keep, int32_t* base, int32_t* send_counts) {
  int64_t pos = 0;
  for (int32_t q = 0; q < M; ++q) {
    int64_t n = 0;
    for (int32_t e = 0; e < N; ++e) {
      if (rho[e] != q) continue;
      base[e] = static_cast<int32_t>(pos + n);
      n += keep[static_cast<int64_t>(src) * N + e];
    }
    if (send_counts) send_counts[q] = static_cast<int32_t>(n);
    pos += n;
  }
}

// Send-buffer position of a route of source `src` placed at destination row `row` (from
// ep_place_route) for expert e, or -1 when the route is dropped (row < 0).
MOE_HD inline int32_t ep_send_pos_route(int32_t src, int32_t N, int32_t e, int32_t row,
                                        const int32_t* base, const int32_t* recv_off) {
  return row < 0 ? -1 : base[e] + (row - recv_off[static_cast<int64_t>(src) * N + e]);
}

// Destination q's receive buffer from the exchange: the blocks of sources 0, 1, ... in
// order, each in the source's send order for q.  recv_row[j] is the row of q's packed
// buffer that received row j belongs to.  Writes R_keep[q] entries; returns their count.
MOE_HD inline int64_t ep_recv_rows(int32_t q, int32_t M, int32_t N, const int32_t* rho,
                                   const int32_t* keep, const int32_t* recv_off,
                                   int32_t* recv_row) {
  int64_t j = 0;
  for (int32_t s = 0; s < M; ++s)
    for (int32_t e = 0; e < N; ++e) {
      if (rho[e] != q) continue;
      const int64_t i = static_cast<int64_t>(s) * N + e;
      for (int32_t r = 0; r < keep[i]; ++r) recv_row[j++] = recv_off[i] + r;
    }
  return j;
}

}  // namespace moe

// Router for many experts (128 < N <= 256, bf16, no learned shared gate) on CTA pairs.
//
// Computes the same as route_tc.cu (Section 10 "Routing, Capacity, and Load Balancing",
// Table 16 and Eq. 35; Appendix E, Table 52; Section 21, Eq. 80 coefficients), laid out
// so that no CTA streams all of W_router nor scans all N columns of a token alone:
//   - a cluster of two CTAs takes 128 tokens, 64 per CTA.  The even CTA issues
//     tcgen05.mma.cta_group::2 with M = 128 (64 A rows from each CTA) and N = 256 (B
//     columns 0-127, the first 128 experts, from the even CTA's shared memory, 128-255
//     from the odd CTA's), so each CTA reads its own tokens' x and half of W_router per
//     K block (24 KB instead of 40), and the MMAs take half the cycles of a one-CTA
//     M = 128 x N = 256 step whose rows are half empty;
//   - a ring stage holds two K blocks, so the issuing thread waits once per 8 MMAs
//     (a wait costs it about as long as 4 MMAs of this shape take to run);
//   - each CTA's accumulator holds its 64 tokens: TMEM lane l < 64 carries experts
//     0-127 of token l, lane 64 + l experts 128-255 of the same token.  The four
//     epilogue warps therefore work on all 128 lanes: each thread builds the sorted list
//     of its half of a token's experts, the upper half passes its list, maximum logit
//     and partial softmax denominator through shared memory, and the lower half merges
//     them (its entries have the lower indices, so they win ties) and finishes the
//     token.  The softmax denominator over all N is the two partial sums rescaled to
//     the larger of the two maxima.
// Every wait is bounded; a wait that runs out records MOE_ERR_TIMEOUT, the CTA drains what
// it issued, and both CTAs meet at the final cluster barrier before TMEM is released.
#include "common.cuh"
#include "internal.h"
#include "route_select.cuh"

namespace moe {
namespace {

constexpr int kRows = 64;                     // tokens per CTA (128 per pair)
constexpr int kBK = 64;
constexpr int kHalfN = 128;                   // experts per CTA's B half
constexpr int kA = kRows * kBK * 2;           // 8 KB
constexpr int kB = kHalfN * kBK * 2;          // 16 KB
constexpr int kSub = kA + kB;                 // one K block
constexpr int kKsub = 2;                      // K blocks per ring stage
constexpr int kStages = 4;
constexpr int kStage = kKsub * kSub;
constexpr int kRing = kStages * kStage;       // 192 KB
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 100000000ull;

template <int L>
struct Exchange {      // the upper half of each token's columns, passed to the lower half
  float v[kRows][L];
  float z[kRows][L];
  int i[kRows][L];
  float zmax[kRows];
  float zsum[kRows];
  int ready[4];
};

template <int L>
constexpr size_t smem_bytes() {
  return 1024 + kRing + 8 * (2 * kStages + 2) + 16 + 2 * sizeof(float) * kMaxExperts +
         sizeof(Exchange<L>) + 64;
}

__device__ __forceinline__ void epilogue_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
}

template <int L>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    route_pair_kernel(const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmW, const RouteParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRing);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* never = const_cast<int*>(abort_flag) + 1;
  float* s_bias = reinterpret_cast<float*>(never + 2);   // 16-byte aligned
  float* s_sel = s_bias + kMaxExperts;
  Exchange<L>* xch = reinterpret_cast<Exchange<L>*>(s_sel + kMaxExperts);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int k_blocks = (p.d + kBK - 1) / kBK;
  const uint32_t smem_base = smem_u32(smem);
  const int64_t t_cta = static_cast<int64_t>(blockIdx.x >> 1) * (2 * kRows) + rank * kRows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    *never = 0;
    mbar_fence_init();
  }
  for (int i = threadIdx.x; i < p.N; i += kThreads) {
    s_bias[i] = p.router_bias ? p.router_bias[i] : 0.f;
    s_sel[i] = p.selection_bias ? p.selection_bias[i] : 0.f;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmX);
    tma_prefetch_map(&tmW);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_holder), kTmemCols);
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();   // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ---------------- producer (both CTAs): this CTA's tokens and its half of W_router
    if (lane == 0) {
      constexpr uint32_t tx = 2u * kSub;   // both CTAs' bytes land on the even CTA's barrier
      int stage = 0;
      uint32_t phase = 0;
      int issued_parity[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) issued_parity[s] = -1;
      bool ok = true;
      for (int kb0 = 0; kb0 < k_blocks; kb0 += kKsub) {
        if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p.status,
                               kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t fb_local = smem_u32(&full[stage]);
        const uint32_t fb_leader = mapa_shared(fb_local, 0);
        const int nv = min(kKsub, k_blocks - kb0);
        if (leader) mbar_arrive_expect_tx(fb_local, tx * static_cast<uint32_t>(nv));
        for (int u = 0; u < nv; ++u) {
          const int kb = kb0 + u;
          const uint32_t sA = smem_base + stage * kStage + u * kSub;
          tma_load_2d_pair(sA, &tmX, kb * kBK, static_cast<int32_t>(t_cta), fb_leader);
          tma_load_2d_pair(sA + kA, &tmW, kb * kBK, static_cast<int32_t>(rank) * kHalfN,
                           fb_leader);
        }
        issued_parity[stage] = static_cast<int>(phase);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok && leader) {
        // the even CTA's full barriers count both CTAs' copies: wait for them to land
        for (int s = 0; s < kStages; ++s)
          if (issued_parity[s] >= 0)
            mbar_wait_bounded(smem_u32(&full[s]), static_cast<uint32_t>(issued_parity[s]), never,
                              nullptr, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kRows, 2 * kHalfN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb0 = 0; kb0 < k_blocks; kb0 += kKsub) {
        if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, p.status,
                               kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int nv = min(kKsub, k_blocks - kb0);
        for (int u = 0; u < nv; ++u) {
          const uint32_t sA = smem_base + stage * kStage + u * kSub;
          const uint64_t a_desc = sw128_kmajor_desc(sA);
          const uint64_t b_desc = sw128_kmajor_desc(sA + kA);
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j)
            tc_mma_bf16_pair(tmem_base, a_desc + 2 * j, b_desc + 2 * j, idesc,
                             (kb0 + u > 0 || j > 0) ? 1u : 0u);
        }
        tc_commit_pair(smem_u32(&empty[stage]), 0x3);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (ok) {
        tc_commit_pair(smem_u32(acc_full), 0x3);
      } else {
        tc_commit_pair(smem_u32(drain), 0x1);
        mbar_wait_bounded(smem_u32(drain), 0, never, nullptr, kDrainLimitNs);
      }
    }
  } else {
    // ---------------- epilogue (both CTAs): two threads per token
    const int q = warp & 3;                  // TMEM lane quadrant of this warp
    const bool upper = q >= 2;               // experts 128-255
    const int tok = (q & 1) * 32 + lane;     // token within the CTA
    const int64_t t = t_cta + tok;
    const bool valid = t < p.T;
    bool ready = true;
    if (lane == 0)
      ready = mbar_wait_bounded(smem_u32(acc_full), 0, abort_flag, p.status, kWaitLimitNs);
    if (lane == 0) xch->ready[q] = ready ? 1 : 0;
    __syncwarp();
    epilogue_bar();
    // the same decision in all four warps, so that every warp reaches the second barrier
    const bool go = xch->ready[0] && xch->ready[1] && xch->ready[2] && xch->ready[3];
    float bv[L], bz[L];
    int bi[L];
    list_clear<L>(bv, bz, bi);
    float zmax = -INFINITY, zsum = 0.f;
    if (go) {
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int c_lo = upper ? kHalfN : 0;
      const int c_hi = min(c_lo + kHalfN, p.N);
      auto load32 = [&](int c0, uint32_t(&r)[32]) {
        tmem_ld32(taddr + static_cast<uint32_t>(c0 - c_lo), r);
      };
      float* lrow = (p.logits && valid) ? p.logits + t * p.N : nullptr;
      // the ring is free once the accumulator is complete: two 32-entry scratch rows per
      // thread, thread-interleaved so that every access is free of bank conflicts
      float* scratch = reinterpret_cast<float*>(smem) + q * 32 + lane;
      list_columns<L>(p, s_bias, s_sel, c_lo, c_hi, lrow, scratch, scratch + 32 * 128, 128,
                      load32, bv, bz, bi, zmax);
      if (needs_full_softmax(p)) zsum = exp_sum_columns(p, s_bias, c_lo, c_hi, zmax, load32);
      if (upper) {
#pragma unroll
        for (int j = 0; j < L; ++j) {
          xch->v[tok][j] = bv[j];
          xch->z[tok][j] = bz[j];
          xch->i[tok][j] = bi[j];
        }
        xch->zmax[tok] = zmax;
        xch->zsum[tok] = zsum;
      }
    }
    __syncwarp();
    epilogue_bar();
    if (go && !upper) {
      // The upper list's experts all follow this list's: inserting them in their order
      // with strict comparisons keeps the lower index first on equal keys.
#pragma unroll
      for (int j = 0; j < L; ++j) {
        const int ci = xch->i[tok][j];
        if (ci != kRouteEmpty) list_insert<L>(xch->v[tok][j], xch->z[tok][j], ci, bv, bz, bi);
      }
      const float zm_up = xch->zmax[tok];
      const float m = fmaxf(zmax, zm_up);
      const float s_all =
          needs_full_softmax(p) ? zsum * expf(zmax - m) + xch->zsum[tok] * expf(zm_up - m) : 0.f;
      finish_token<L>(p, t, valid, bz, bi, m, s_all, 0.f);
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync_all();   // no CTA leaves while its partner may still use its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <int L>
cudaError_t launch_list(const CUtensorMap& mX, const CUtensorMap& mW, const RouteParams& p,
                        cudaStream_t s) {
  constexpr size_t smem = smem_bytes<L>();
  static_assert(smem <= 227 * 1024, "pair router shared memory");
  auto kern = route_pair_kernel<L>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int64_t pairs = (p.T + 2 * kRows - 1) / (2 * kRows);
  kern<<<static_cast<unsigned>(2 * pairs), kThreads, smem, s>>>(mX, mW, p);
  return cudaGetLastError();
}

}  // namespace

bool route_pair_applies(const RouteParams& p) {
  return p.N > kHalfN && p.N <= 2 * kHalfN && p.shared_mode != MOE_SHARED_SIGMOID_GATE;
}

cudaError_t launch_route_pair(const RouteParams& p, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  if (!route_pair_applies(p)) return cudaErrorInvalidValue;
  CUtensorMap mX, mW;
  // x: 64-row boxes (one CTA's tokens; rows past T read as zeros); W_router: 128-row boxes
  // (one CTA's experts; rows past N read as zeros and are never selected)
  if (!make_bf16_map(&mX, p.x, p.d, p.T, kRows) || !make_bf16_map(&mW, p.W_router, p.d, p.N, kHalfN))
    return cudaErrorInvalidValue;
  if (p.K <= 2) return launch_list<2>(mX, mW, p, s);
  if (p.K <= 4) return launch_list<4>(mX, mW, p, s);
  return launch_list<kMaxTopK>(mX, mW, p, s);
}

}  // namespace moe

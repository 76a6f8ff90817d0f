// Router on the tensor cores for bf16 layers: logits, scores, top-K and coefficients.
//
// Same step as route.cu (Section 10 "Routing, Capacity, and Load Balancing",
// Table 16 and Eq. 35; Appendix E "Expert-Merge Normalization in Public MoE
// Models", Table 52; Section 21, Eq. 80 coefficients), organised for sm_103a:
//   - one CTA per R tokens (R = 32, 64 or 128, so that the grid covers the SMs: the
//     step streams x once and is bound by HBM, not by the tensor cores); warp 0
//     streams x and W_router K-blocks with TMA (128-byte swizzle) through a
//     shared-memory ring, warp 1 issues tcgen05.mma (M = 128 rows, of which the
//     first R are this CTA's tokens and the rest are ignored; N = N rounded up to
//     16; fp32 accumulators in TMEM), plus an N = 16 MMA against the shared-gate
//     vector w_s when the layer has a learned shared gate (its logit lands in TMEM
//     column N_pad).  With few experts a CTA takes a quarter of the SM's shared
//     memory and TMEM, so several run per SM;
//   - warps 2-5 read the accumulators with tcgen05.ld, one token row per
//     thread, so the selection runs in registers: a sorted list of 2, 4 or 8
//     entries (the smallest that holds K) with
//     strict comparisons (an equal later expert never displaces an earlier one,
//     which gives the lower-index tie rule) on the key z (+ the Eq. 35
//     selection-only bias), then the scores of the selected experts from the
//     unbiased logits, the selected weights and r = alpha * w.
// Every wait is bounded; a wait that runs out records MOE_ERR_TIMEOUT.
#include "common.cuh"
#include "internal.h"
#include "route_select.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                    // MMA rows (and A slot rows)
constexpr int BK = 64;
constexpr int THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;
constexpr int G_BYTES = 16 * BK * 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 100000000ull;

struct RouteTcArgs {
  RouteParams p;
  int32_t n_pad;       // N rounded up to 16
  int32_t gated;       // 1 when the shared gate column is computed
  int32_t stages;
  int32_t stage_bytes;
  int32_t rows;        // tokens per CTA (R)
  uint32_t tmem_cols;  // power of two >= n_pad (+16 when gated)
};

// L: length of the per-token sorted list (2, 4 or 8, the smallest that holds K); one
// kernel per length, so each carries only its own selection code.
template <int L>
__global__ void __launch_bounds__(THREADS, 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmG, const RouteTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const RouteParams& p = a.p;
  const int S = a.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * a.stage_bytes);
  uint64_t* empty = full + 8;
  uint64_t* acc_full = empty + 8;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* never = const_cast<int*>(abort_flag) + 1;
  float* s_bias = reinterpret_cast<float*>(never + 1);   // [kMaxExperts] logit bias
  float* s_sel = s_bias + kMaxExperts;                    // [kMaxExperts] selection-only bias

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int k_blocks = (p.d + BK - 1) / BK;
  const uint32_t smem_base = smem_u32(smem);
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * a.rows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    *never = 0;
    mbar_fence_init();
  }
  for (int i = threadIdx.x; i < p.N; i += THREADS) {
    s_bias[i] = p.router_bias ? p.router_bias[i] : 0.f;
    s_sel[i] = p.selection_bias ? p.selection_bias[i] : 0.f;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmX);
    tma_prefetch_map(&tmW);
    if (a.gated) tma_prefetch_map(&tmG);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), a.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint32_t tx_bytes =
      static_cast<uint32_t>(a.rows * BK * 2 + a.n_pad * BK * 2 + (a.gated ? G_BYTES : 0));

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued_parity[8];
      for (int s = 0; s < 8; ++s) issued_parity[s] = -1;
      bool ok = true;
      for (int kb = 0; kb < k_blocks; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p.status,
                               kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&full[stage]);
        mbar_arrive_expect_tx(fb, tx_bytes);
        const uint32_t sA = smem_base + stage * a.stage_bytes;
        const uint32_t sB = sA + A_BYTES;
        tma_load_2d(sA, &tmX, kb * BK, static_cast<int32_t>(t0), fb);
        tma_load_2d(sB, &tmW, kb * BK, 0, fb);
        if (a.gated) tma_load_2d(sB + a.n_pad * BK * 2, &tmG, kb * BK, 0, fb);
        issued_parity[stage] = static_cast<int>(phase);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok)
        for (int s = 0; s < S; ++s)
          if (issued_parity[s] >= 0)
            mbar_wait_bounded(smem_u32(&full[s]), static_cast<uint32_t>(issued_parity[s]), never,
                              nullptr, kDrainLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, a.n_pad);
      const uint32_t idesc_g = idesc_bf16_f32(BM, 16);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < k_blocks; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, p.status, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sA = smem_base + stage * a.stage_bytes;
        const uint32_t sB = sA + A_BYTES;
        const uint64_t a_desc = sw128_kmajor_desc(sA);
        const uint64_t b_desc = sw128_kmajor_desc(sB);
        const uint64_t g_desc = sw128_kmajor_desc(sB + a.n_pad * BK * 2);
#pragma unroll
        for (int j = 0; j < BK / 16; ++j) {
          const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
          tc_mma_bf16(tmem_base, a_desc + 2 * j, b_desc + 2 * j, idesc, acc);
          if (a.gated)
            tc_mma_bf16(tmem_base + a.n_pad, a_desc + 2 * j, g_desc + 2 * j, idesc_g, acc);
        }
        tc_commit(smem_u32(&empty[stage]));
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (ok) {
        tc_commit(smem_u32(acc_full));
      } else {
        tc_commit(smem_u32(drain));
        mbar_wait_bounded(smem_u32(drain), 0, never, nullptr, kDrainLimitNs);
      }
    }
  } else {
    // ---------------- epilogue: one token row per thread ----------------
    const int q = warp & 3;
    if (q * 32 >= a.rows) goto done;   // TMEM lanes of rows this CTA does not own
    {
    bool ready = true;
    if (lane == 0)
      ready = mbar_wait_bounded(smem_u32(acc_full), 0, abort_flag, p.status, kWaitLimitNs);
    ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
    if (ready) {
      tc_fence_after();
      const int64_t t = t0 + q * 32 + lane;
      const bool valid = t < p.T;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      float gate_raw = 0.f;
      if (p.shared_mode == MOE_SHARED_SIGMOID_GATE) {
        uint32_t r[32];
        tmem_ld32(taddr + a.n_pad, r);
        gate_raw = __uint_as_float(r[0]);
      }
      // the ring is free once the accumulator is complete: two 32-entry scratch rows per
      // thread, thread-interleaved so that every access is free of bank conflicts
      float* scratch = reinterpret_cast<float*>(smem) + q * 32 + lane;
      route_one_token<L>(p, s_bias, s_sel, t, valid, scratch, scratch + 32 * BM, BM,
                         [&](int c0, uint32_t(&r)[32]) { tmem_ld32(taddr + c0, r); }, gate_raw);
    }
    }
  }

done:
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

}  // namespace

cudaError_t launch_route_tc(const RouteParams& p, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  if (route_pair_applies(p)) return launch_route_pair(p, s);
  const bool gated = p.shared_mode == MOE_SHARED_SIGMOID_GATE;
  const int n_pad = (p.N + 15) / 16 * 16;
  // Tokens per CTA: the smallest of 32, 64, 128 whose grid fits the SMs at once (two
  // CTAs per SM with few experts; one with many, where each CTA's MMAs over all N
  // columns and its reads of W_router cost the same for any R, so R stays >= 64).
  const int64_t sms = device_sm_count() > 0 ? device_sm_count() : 1;
  const bool wide = n_pad > 128;
  int rows = wide ? 64 : 32;
  while (rows < BM && (p.T + rows - 1) / rows > (wide ? 1 : 2) * sms) rows *= 2;
  CUtensorMap mX, mW, mG;
  if (!make_bf16_map(&mX, p.x, p.d, p.T, static_cast<uint32_t>(rows)) ||
      !make_bf16_map(&mW, p.W_router, p.d, p.N, n_pad))
    return cudaErrorInvalidValue;
  if (gated) {
    if (!make_bf16_map(&mG, p.shared_gate_w, p.d, 1, 16)) return cudaErrorInvalidValue;
  } else {
    mG = mW;
  }
  RouteTcArgs a{};
  a.p = p;
  a.n_pad = n_pad;
  a.gated = gated ? 1 : 0;
  a.rows = rows;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(n_pad + (gated ? 16 : 0))) cols *= 2;
  a.tmem_cols = cols;
  a.stage_bytes = A_BYTES + n_pad * BK * 2 + (gated ? G_BYTES : 0);
  // With at most 128 TMEM columns a CTA leaves room for others on its SM: a ring of
  // about 100 KB lets two run per SM; otherwise the ring takes most of the 227 KB.
  const int ring = cols <= 128 ? 100 * 1024 : 200 * 1024;
  a.stages = ring / a.stage_bytes;
  if (a.stages > 8) a.stages = 8;
  if (a.stages < 2) a.stages = 2;
  const size_t smem = 1024 + static_cast<size_t>(a.stages) * a.stage_bytes + 8 * 20 + 16 +
                      2 * sizeof(float) * kMaxExperts + 64;
  using Kernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const RouteTcArgs);
  const Kernel kern = p.K <= 2   ? static_cast<Kernel>(route_tc_kernel<2>)
                      : p.K <= 4 ? static_cast<Kernel>(route_tc_kernel<4>)
                                 : static_cast<Kernel>(route_tc_kernel<kMaxTopK>);
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>((p.T + rows - 1) / rows);
  kern<<<grid, THREADS, smem, s>>>(mX, mW, mG, a);
  return cudaGetLastError();
}

}  // namespace moe

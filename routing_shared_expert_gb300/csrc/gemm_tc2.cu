// Grouped SwiGLU expert GEMMs on CTA pairs: tcgen05 with cta_group::2 (2-SM MMA).
//
// Computes the same as gemm_tc.cu (Section 20 "One Shared Expert Is All You
// Need", Eq. 74, per packed segment of Section 10, Eq. 26):
//   gate/up:  h[row] = SiLU(x[row] W_g^e) * (x[row] W_u^e)     (bf16 h)
//   down:     f[row] = h[row] W_d^e                            (fp32 f)
// but a cluster of two CTAs on two SMs computes each 256-row tile together.
// The even CTA issues tcgen05.mma with M = 256, N = 256: A rows 0-127 come from
// its own shared memory and rows 128-255 from its partner's; B columns 0-127
// from its own and 128-255 from its partner's.  Each CTA therefore loads only
// 16 KB of A and 16 KB of B per 64-wide K step (half the bytes per multiply-add
// of a one-SM 128 x 256 tile), which lets six K blocks sit in shared memory and
// keeps the tensor pipe fed from L2.  Each CTA's TMEM holds the fp32
// accumulator rows of its own 128 rows for all 256 columns.
//   SwiGLU mode: a tile covers 128 h columns.  In a full tile the even CTA loads
//                their 128 gate weight rows and the odd CTA their 128 up rows,
//                so TMEM columns [0,128) hold x W_g and [128,256) x W_u.  In a
//                half tile each CTA loads the gate and the up rows of 64 of the
//                h columns (two 64-row boxes), so that gate and up of one h
//                column land in the same TMEM lane, 64 columns apart.
//   Plain mode:  each CTA loads 128 of the 256 output columns' weight rows.
// The last tile of a segment is a half tile (M = 128: 64 A rows per CTA) when at
// most 128 of its rows are real.  A cta_group::2 MMA with M = 128 issues at twice
// the rate of one with M = 256 (each SM computes 64 rows), so a short tail costs
// half a tile instead of a whole one, once the issuer's waits are spread over
// enough MMAs (the ring stage width below).  Its accumulator lands in TMEM lanes 0-63 for
// B columns [0,128) and lanes 64-127 for columns [128,256), TMEM columns 0-127,
// rows 64 r + (lane mod 64) in CTA r.
// The gate/up A rows are either read from a packed buffer (one TMA tile load) or
// gathered straight from x through the packed-row source table, so that the row
// permutation of Section 10.3 costs no extra pass over memory.  Gathering, six more
// warps per CTA, one per K block of the ring, copy the CTA's A rows of their K block with
// 16-byte cp.async pieces (a warp instruction moves four whole 128-byte row pieces), wait
// for them, make them visible to the tensor core's proxy and arrive on the even CTA's
// stage barrier, which then counts the producer's arrival, the gatherer arrivals of both
// CTAs and the B bytes.
// Roles per CTA (192 threads, 384 gathering): warp 0 TMA producer (both CTAs;
// completions are counted on the even CTA's barrier), warp 1 TMEM allocation and, in
// the even CTA only, the MMA issuer; warps 2-5 epilogue; warps 6-11 A-row gatherers.
// The epilogue stages each
// 32 x 32 block through shared memory: h blocks go out as row-contiguous lane stores,
// fp32 f blocks as TMA bulk tensor stores (lane stores at a segment's end).
// Every wait is bounded by %globaltimer; a wait that runs out records
// MOE_ERR_TIMEOUT and the CTA drains what it issued before the final cluster
// barrier and TMEM release.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128;                    // rows per CTA
constexpr int PM = 256;                    // rows per pair tile
constexpr int HM = 64;                     // rows per CTA of a half tile (M = 128)
constexpr int BK = 64;
// The ring holds six K blocks of 64 (32 KB each).  A ring stage is one K block, or two
// (three stages of 64 KB) when the launch asks for it: the MMA issuer then waits once
// per 8 MMAs instead of once per 4, which matters when an MMA group is short (a half
// tile's 4 MMAs take 256 cycles, less than one wait-to-issue round trip of the issuer),
// while the finer ring keeps more bytes in flight for weight-streaming launches.
constexpr int RING_BLOCKS = 6;
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int B_BYTES = 128 * BK * 2;      // 16 KB
constexpr int SUB_BYTES = A_BYTES + B_BYTES;
constexpr int RING_BYTES = RING_BLOCKS * SUB_BYTES;
constexpr int EPI_LD = 36;                 // 32-bit words per staged row (16-byte aligned)
constexpr int EPI_WARP_WORDS = 32 * EPI_LD;
constexpr int EPI_BYTES = 4 * EPI_WARP_WORDS * 4;
constexpr int THREADS = 192;
constexpr int GATHER_THREADS = THREADS + 32 * RING_BLOCKS;   // one gatherer warp per ring K block
constexpr int GATHER_WARP0 = 6;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 100000000ull;

struct PairArgs {
  const int32_t* offsets;    // [groups+1] device, or nullptr for one dense group
  int32_t dense_rows;
  int32_t groups;
  int32_t k_dim;
  int32_t n_out;             // output columns per group
  int32_t b_rows_per_group;  // rows between groups in the 2-D view of B
  int64_t out_rows;          // rows of the output buffer
  void* out;                 // SwiGLU: bf16 h; plain: fp32 f
  int64_t ldo;
  int32_t* status;
  const int32_t* gather_src; // non-null: A rows are gathered from x through this table
  int64_t gather_cap;        // entries of gather_src
  int64_t src_rows;          // rows of x
  const uint16_t* gather_x;  // x [src_rows][k_dim] (16-bit elements, 16-byte aligned rows)
  // fp16 intermediate: SwiGLU mode stores fp16(h * h_scale); plain mode reads the packed
  // weights' header and writes fp16(accumulator * 2^-k)
  float h_scale;
  const PackHeader* down_hdr;
  int64_t down_elements;     // elements the packed tensor must hold
};

// Epilogue modes of the pair kernel.
constexpr int kSwiGLU = 0;    // h = SiLU(gate) * up, bf16
constexpr int kPlain = 1;     // fp32 rows

struct Tile {
  int g, m, n, seg_start, seg_end;
  bool half;   // at most BM real rows: an M = 128 tile
};

// Tile t of a launch: groups in order; within a group, by default the row tiles of one
// output-column block together (the tiles that read one weight slice run at once), or with
// rows_first the column blocks of one row tile together (dense launches: a block of rows is
// read once while the whole weight matrix, reused by every row tile, stays in L2).
__device__ __forceinline__ bool pair_tile(const int* s_tp, const int* s_off, int G, int n_tiles,
                                          int64_t t, Tile& o, bool rows_first = false) {
  if (t >= static_cast<int64_t>(s_tp[G]) * n_tiles) return false;
  int lo = 0, hi = G;   // s_tp[lo] * n_tiles <= t < s_tp[hi] * n_tiles
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(s_tp[mid]) * n_tiles <= t) lo = mid; else hi = mid;
  }
  const int mt = s_tp[lo + 1] - s_tp[lo];
  const int64_t local = t - static_cast<int64_t>(s_tp[lo]) * n_tiles;
  o.g = lo;
  o.n = static_cast<int>(rows_first ? local % n_tiles : local / mt);
  o.m = static_cast<int>(rows_first ? local / n_tiles : local % mt);
  o.seg_start = s_off[lo];
  o.seg_end = s_off[lo + 1];
  o.half = o.seg_end - (o.seg_start + o.m * PM) <= BM;
  return true;
}

// First weight row of this CTA's B half for a tile (rows of the 2-D [groups * rows][k] view).
template <bool SWIGLU>
__device__ __forceinline__ int b_first_row(const PairArgs& args, const Tile& tl, uint32_t rank) {
  const int base = tl.g * args.b_rows_per_group;
  if (!SWIGLU) return base + tl.n * 256 + static_cast<int>(rank) * 128;
  return base + tl.n * 128 + (tl.half ? static_cast<int>(rank) * 64 : 0);
}

// Loads this CTA's 16 KB B half of one K block.  Plain: 128 weight rows.  SwiGLU full
// tile: the even CTA's gate rows, the odd CTA's up rows (128 each).  SwiGLU half tile:
// 64 gate rows then the same 64 up rows.
template <bool SWIGLU>
__device__ __forceinline__ void load_b(uint32_t sB, bool half, bool leader, const CUtensorMap* b0,
                                       const CUtensorMap* b1, const CUtensorMap* b0h,
                                       const CUtensorMap* b1h, int k, int row, uint32_t bar) {
  if (!SWIGLU) {
    tma_load_2d_pair(sB, b0, k, row, bar);
  } else if (!half) {
    tma_load_2d_pair(sB, leader ? b0 : b1, k, row, bar);
  } else {
    tma_load_2d_pair(sB, b0h, k, row, bar);
    tma_load_2d_pair(sB + B_BYTES / 2, b1h, k, row, bar);
  }
}

template <int MODE, bool GATHER, int KSUB, bool H16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GATHER ? GATHER_THREADS : THREADS, 1)
    tc_pair_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA64,
                 const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                 const __grid_constant__ CUtensorMap tmB0h, const __grid_constant__ CUtensorMap tmB1h,
                 const __grid_constant__ CUtensorMap tmOut, const PairArgs args) {
  constexpr bool SWIGLU = MODE == kSwiGLU;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint32_t* epi = reinterpret_cast<uint32_t*>(smem + RING_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES + EPI_BYTES);
  uint64_t* empty = full + RING_BLOCKS;
  uint64_t* tfull = empty + RING_BLOCKS;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* never = const_cast<int*>(abort_flag) + 1;
  const int G = args.offsets ? args.groups : 1;
  int* s_off = never + 1;       // [G+1]
  int* s_tp = s_off + (G + 1);  // [G+1] pair-tile prefix

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  constexpr int BN_OUT = SWIGLU ? 128 : 256;
  const int n_tiles = (args.n_out + BN_OUT - 1) / BN_OUT;
  const int k_blocks = (args.k_dim + BK - 1) / BK;
  constexpr int ksub = KSUB;
  constexpr int stages = RING_BLOCKS / KSUB;
  constexpr int stage_bytes = KSUB * SUB_BYTES;
  const uint32_t smem_base = smem_u32(smem);
  const int64_t pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const bool dense_rows_first = args.offsets == nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RING_BLOCKS; ++s) {
      // gathering: the producer and, in each CTA, one gatherer warp per K block of the stage
      mbar_init(smem_u32(&full[s]), GATHER ? 1 + 2 * KSUB : 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 8);   // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    *never = 0;
    mbar_fence_init();
  }
  if (warp == 3) {
    // segment table and prefix of 256-row tiles per group
    if (args.offsets == nullptr) {
      if (lane == 0) {
        s_off[0] = 0;
        s_off[1] = args.dense_rows;
        s_tp[0] = 0;
        s_tp[1] = (args.dense_rows + PM - 1) / PM;
      }
    } else {
      for (int i = lane; i <= G; i += 32) s_off[i] = args.offsets[i];
      __syncwarp();
      int running = 0;
      for (int base = 0; base < G; base += 32) {
        const int g = base + lane;
        int v = 0;
        if (g < G) {
          const int len = s_off[g + 1] - s_off[g];
          if (len < 0) set_status(args.status, MOE_ERR_DEVICE_BOUNDS);
          v = len > 0 ? (len + PM - 1) / PM : 0;
        }
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        if (g < G) s_tp[g + 1] = running + incl;
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) s_tp[0] = 0;
    }
  }
  if (warp == 0 && lane == 0) {
    if (!GATHER) {
      tma_prefetch_map(&tmA);
      tma_prefetch_map(&tmA64);
    }
    tma_prefetch_map(&tmB0);
    if (SWIGLU) {
      tma_prefetch_map(&tmB1);
      tma_prefetch_map(&tmB0h);
      tma_prefetch_map(&tmB1h);
    }
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_holder), TMEM_COLS);
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();   // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    int stage = 0;
    uint32_t phase = 0;
    int issued_parity[RING_BLOCKS];
#pragma unroll
    for (int s = 0; s < RING_BLOCKS; ++s) issued_parity[s] = -1;
    bool ok = true;
    Tile tl;
    // Lane 0 alone: wait for a free stage, arm the even CTA's barrier, load A (unless the
    // gatherer warps copy it) and B.
    if (lane == 0) {
      for (int64_t t = pair_id; ok && pair_tile(s_tp, s_off, G, n_tiles, t, tl, dense_rows_first); t += n_pairs) {
        int a_row = tl.seg_start + tl.m * PM + static_cast<int>(rank) * (tl.half ? HM : BM);
        // A CTA whose A rows all lie past the segment (the odd CTA of a half tile over a tail
        // of at most 64 rows) loads its box from past the last row of the buffer instead:
        // TMA fills it with zeros, reads no memory, and the MMAs on those rows (whose results
        // are never stored) multiply zeros instead of the next segment's rows.
        if (a_row >= tl.seg_end) a_row = static_cast<int>(args.out_rows);
        const CUtensorMap* mapA = tl.half ? &tmA64 : &tmA;
        const uint32_t tx =
            GATHER ? 2u * B_BYTES : 2u * ((tl.half ? A_BYTES / 2 : A_BYTES) + B_BYTES);
        const int b_row = b_first_row<SWIGLU>(args, tl, rank);
        for (int kb0 = 0; kb0 < k_blocks; kb0 += ksub) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.status,
                                 kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = smem_u32(&full[stage]);
          const uint32_t fb_leader = mapa_shared(fb_local, 0);
          const int nv = ksub == 1 ? 1 : min(ksub, k_blocks - kb0);
          if (leader) mbar_arrive_expect_tx(fb_local, tx * static_cast<uint32_t>(nv));
#pragma unroll
          for (int u = 0; u < nv; ++u) {
            const int kb = kb0 + u;
            const uint32_t sA = smem_base + stage * stage_bytes + u * SUB_BYTES;
            if (!GATHER) tma_load_2d_pair(sA, mapA, kb * BK, a_row, fb_leader);
            load_b<SWIGLU>(sA + A_BYTES, tl.half, leader, &tmB0, &tmB1, &tmB0h, &tmB1h, kb * BK,
                           b_row, fb_leader);
          }
          issued_parity[stage] = static_cast<int>(phase);
          if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
      }
    }
    if (!ok && leader && lane == 0) {
      // The even CTA's full barriers count both CTAs' copies: wait for them to land.
      for (int s = 0; s < stages; ++s)
        if (issued_parity[s] >= 0)
          mbar_wait_bounded(smem_u32(&full[s]), static_cast<uint32_t>(issued_parity[s]), never,
                            nullptr, kDrainLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      // gate/up multiply bf16 x by bf16 weights; the down GEMM of the fp16 intermediate
      // multiplies fp16 h by the packed fp16 weights
      constexpr bool kF16Ops = H16 && !SWIGLU;
      constexpr uint32_t idesc_full = idesc_f32acc<kF16Ops>(PM, 256);
      constexpr uint32_t idesc_half = idesc_f32acc<kF16Ops>(2 * HM, 256);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Tile tl;
      int64_t local = 0;
      for (int64_t t = pair_id; ok && pair_tile(s_tp, s_off, G, n_tiles, t, tl, dense_rows_first);
           t += n_pairs, ++local) {
        const int buf = static_cast<int>(local & 1);
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait_bounded(smem_u32(&tempty[buf]), (use & 1u) ^ 1u, abort_flag, args.status,
                               kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_acc = tmem_base + static_cast<uint32_t>(buf * 256);
        const uint32_t idesc = tl.half ? idesc_half : idesc_full;
        for (int kb0 = 0; kb0 < k_blocks; kb0 += ksub) {
          // gathered A rows: the partner's gatherers release their rows at cluster scope
          if (!mbar_wait_bounded<GATHER>(smem_u32(&full[stage]), phase, abort_flag, args.status,
                                         kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nv = ksub == 1 ? 1 : min(ksub, k_blocks - kb0);
#pragma unroll
          for (int u = 0; u < nv; ++u) {
            const uint32_t sA = smem_base + stage * stage_bytes + u * SUB_BYTES;
            const uint64_t a_desc = sw128_kmajor_desc(sA);
            const uint64_t b_desc = sw128_kmajor_desc(sA + A_BYTES);
#pragma unroll
            for (int j = 0; j < BK / 16; ++j)
              tc_mma_bf16_pair(d_acc, a_desc + 2 * j, b_desc + 2 * j, idesc,
                               (kb0 + u > 0 || j > 0) ? 1u : 0u);
          }
          tc_commit_pair(smem_u32(&empty[stage]), 0x3);
          if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit_pair(smem_u32(&tfull[buf]), 0x3);
      }
      if (!ok) {
        tc_commit_pair(smem_u32(drain), 0x1);
        mbar_wait_bounded(smem_u32(drain), 0, never, nullptr, kDrainLimitNs);
      }
    }
  } else if (warp < GATHER_WARP0) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    uint32_t* stg = epi + (warp - 2) * EPI_WARP_WORDS;
    // plain mode of the fp16 intermediate: the packed weights' scale, checked once; the
    // output holds f 2^-h_scale_log2 = accumulator 2^-k in fp16
    float out_mul = 1.f;
    if (H16 && !SWIGLU) {
      const PackHeader* hd = args.down_hdr;
      out_mul = hd->inv_scale;
      if (lane == 0 && (hd->magic != kPackMagic || hd->elements != args.down_elements))
        set_status(args.status, MOE_ERR_BAD_PACK);
      if (lane == 0 && (hd->flags & kPackNonFinite)) set_status(args.status, MOE_ERR_RANGE);
    }
    Tile tl;
    int64_t local = 0;
    for (int64_t t = pair_id; pair_tile(s_tp, s_off, G, n_tiles, t, tl, dense_rows_first); t += n_pairs, ++local) {
      const int buf = static_cast<int>(local & 1);
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      bool ready = true;
      if (lane == 0)
        ready = mbar_wait_bounded(smem_u32(&tfull[buf]), use & 1u, abort_flag, args.status,
                                  kWaitLimitNs);
      ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
      if (!ready) break;
      tc_fence_after();
      // Full tile: warp q holds rows 128 r + 32 q .. of all 256 accumulator columns.
      // Half tile: warp q holds rows 64 r + 32 (q mod 2) .. of accumulator columns
      // [128 (q / 2), 128 (q / 2) + 128), found in TMEM columns 0-127.
      const int hq = q >> 1;
      const int64_t row0 = static_cast<int64_t>(tl.seg_start) + tl.m * PM +
                           (tl.half ? rank * HM + (q & 1) * 32 : rank * BM + q * 32);
      const int64_t row_end = tl.seg_end < args.out_rows ? tl.seg_end : args.out_rows;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(buf * 256);
      if (SWIGLU) {
        // full tile: gate of h column j in TMEM column j, up in 128 + j; half tile: the
        // warp's 64 h columns with gate in TMEM columns [0,64) and up in [64,128)
        uint16_t* out = static_cast<uint16_t*>(args.out);
        float amax = 0.f;
        const int chunks = tl.half ? 2 : 4;
        const int up_off = tl.half ? 64 : 128;
#pragma unroll 1
        for (int c = 0; c < chunks; ++c) {
          const int hcol = tl.n * 128 + (tl.half ? hq * 64 : 0) + 32 * c;
          uint32_t gr[32], ur[32];
          tmem_ld32x2(taddr + 32 * c, taddr + 32 * c + up_off, gr, ur);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int e = 8 * v + 2 * i;
              const float h0 = silu(__uint_as_float(gr[e])) * __uint_as_float(ur[e]);
              const float h1 = silu(__uint_as_float(gr[e + 1])) * __uint_as_float(ur[e + 1]);
              if constexpr (H16) {
                const float s0 = h0 * args.h_scale, s1 = h1 * args.h_scale;
                amax = fmaxf(amax, fmaxf(fabsf(s0), fabsf(s1)));
                w4[i] = pack_f16x2(s0, s1);
              } else {
                w4[i] = pack_bf16x2(h0, h1);
              }
            }
            *reinterpret_cast<uint4*>(stg + lane * EPI_LD + 4 * v) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
          __syncwarp();
          // four lanes per row (16 bytes each), eight rows per pass
#pragma unroll
          for (int pass = 0; pass < 4; ++pass) {
            const int r = pass * 8 + lane / 4;
            const int64_t row = row0 + r;
            const int col = hcol + (lane % 4) * 8;
            const uint4 val = *reinterpret_cast<const uint4*>(stg + r * EPI_LD + (lane % 4) * 4);
            if (row < row_end && col + 8 <= args.n_out)
              *reinterpret_cast<uint4*>(out + row * args.ldo + col) = val;
          }
          __syncwarp();
        }
        // an h value of this lane's row past the fp16 range became an infinity: report it
        // (rows past the segment's end are never stored, and are not checked)
        if (H16 && row0 + lane < row_end && !(amax < kF16RoundsToInf))
          set_status(args.status, MOE_ERR_RANGE);
      } else {
        // One 32 x 32 fp32 block per chunk, staged in the 128-byte swizzled layout of the
        // output map (16-byte piece v of row r at piece v ^ (r mod 8): conflict-free) and
        // written by one TMA store when it lies inside the segment and the width; blocks
        // crossing the segment's end (the next rows belong to another segment) or the width
        // are written by the lanes.
        float* out = static_cast<float*>(args.out);
        const int chunks = tl.half ? 4 : 8;
        const int col_base = tl.n * 256 + (tl.half ? hq * 128 : 0);
        uint8_t* blk = reinterpret_cast<uint8_t*>(epi) + (warp - 2) * 4096;
        const bool rows_in = row0 + 32 <= row_end;
#pragma unroll 1
        for (int c = 0; c < chunks; ++c) {
          uint32_t ar[32];
          tmem_ld32(taddr + c * 32, ar);
          const int col0 = col_base + c * 32;
          if constexpr (H16) {
            // fp16 32 x 32 block, staged in the 64-byte swizzled layout of the output map
            // (16-byte piece v of row r at piece v ^ ((r / 2) mod 4)) and written by one TMA
            // store inside the segment and the width; else each lane stores its own row
            uint32_t pk[16];
            float m = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float v0 = __uint_as_float(ar[2 * i]) * out_mul;
              const float v1 = __uint_as_float(ar[2 * i + 1]) * out_mul;
              m = fmaxf(m, fmaxf(fabsf(v0), fabsf(v1)));
              pk[i] = pack_f16x2(v0, v1);
            }
            const int64_t row = row0 + lane;
            if (row < row_end && !(m < kF16RoundsToInf)) set_status(args.status, MOE_ERR_RANGE);
            if (rows_in && col0 + 32 <= args.n_out) {
              if (lane == 0) bulk_wait_read_all();   // the previous block has been read out
              __syncwarp();
#pragma unroll
              for (int v = 0; v < 4; ++v)
                *reinterpret_cast<uint4*>(blk + lane * 64 + ((v ^ ((lane >> 1) & 3)) * 16)) =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmOut, col0, static_cast<int32_t>(row0), smem_u32(blk));
                bulk_commit();
              }
            } else if (row < row_end) {
              uint16_t* orow = static_cast<uint16_t*>(args.out) + row * args.ldo;
#pragma unroll
              for (int v = 0; v < 4; ++v)
                if (col0 + 8 * v + 8 <= args.n_out)
                  __stcs(reinterpret_cast<uint4*>(orow + col0 + 8 * v),
                         make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]));
            }
            continue;
          }
          if (lane == 0) bulk_wait_read_all();   // the previous block has been read out
          __syncwarp();
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<uint4*>(blk + lane * 128 + ((v ^ (lane & 7)) * 16)) =
                make_uint4(ar[4 * v], ar[4 * v + 1], ar[4 * v + 2], ar[4 * v + 3]);
          if (rows_in && col0 + 32 <= args.n_out) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, col0, static_cast<int32_t>(row0), smem_u32(blk));
              bulk_commit();
            }
          } else {
            __syncwarp();
            // eight lanes per row (16 bytes each), four rows per pass
#pragma unroll
            for (int pass = 0; pass < 8; ++pass) {
              const int r = pass * 4 + lane / 8;
              const int64_t row = row0 + r;
              const int col = col0 + (lane % 8) * 4;
              const uint4 val =
                  *reinterpret_cast<const uint4*>(blk + r * 128 + (((lane % 8) ^ (r & 7)) * 16));
              if (row < row_end && col + 4 <= args.n_out)
                __stcs(reinterpret_cast<uint4*>(out + row * args.ldo + col), val);
            }
            __syncwarp();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[buf]), 0));
    }
    if (!SWIGLU && lane == 0) bulk_wait_all();   // the output blocks are written
  } else if constexpr (GATHER) {
    // ------------------------------------------------------------ A-row gatherers (both CTAs)
    // One warp per ring slot and K block of a stage (six warps): warp gw fills K block
    // gw / stages of slot gw mod stages at every use of that slot, with all R A rows of the
    // CTA (R = 128, or 64 in a half tile).  Lanes 8j..8j+7 take the eight 16-byte pieces of
    // one row, so a warp instruction moves four whole 128-byte row pieces; piece v of row r
    // lands at piece v ^ (r mod 8) of the row's 128 bytes (the 128-byte swizzle the MMA
    // descriptors expect).  Rows past the segment are zero-filled.  The warp waits for its
    // own copies, fences them into the async proxy and arrives once on the even CTA's
    // stage barrier, so every slot refills as soon as the MMAs release it, independently
    // of the others.
    constexpr int kGatherWarps = (GATHER_THREADS - THREADS) / 32;
    static_assert(kGatherWarps == RING_BLOCKS, "one gatherer warp per ring K block");
    const int gw = warp - GATHER_WARP0;
    const int my_slot = gw % stages, my_u = gw / stages;
    const int sub = lane >> 3, piece = lane & 7;
    const int64_t ld_bytes = static_cast<int64_t>(args.k_dim) * 2;
    const char* xb = reinterpret_cast<const char*>(args.gather_x);
    const int stages_per_tile = (k_blocks + ksub - 1) / ksub;
    int64_t j0 = 0;   // ring stages of the tiles before this one
    bool ok = true;
    Tile tl;
    for (int64_t t = pair_id; ok && pair_tile(s_tp, s_off, G, n_tiles, t, tl, dense_rows_first);
         t += n_pairs, j0 += stages_per_tile) {
      // this warp's first stage of the tile: the first j >= j0 with j mod stages == my_slot
      int q = static_cast<int>((my_slot - j0 % stages + stages) % stages);
      if (q >= stages_per_tile) continue;
      const int rows = tl.half ? HM : BM;
      const int n_i = rows / 4;   // instructions per K block: 32 (full tile) or 16 (half)
      const int64_t a_row = static_cast<int64_t>(tl.seg_start) + tl.m * PM + rank * rows;
      int32_t tok[32];
      uint32_t valid = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int64_t pr = a_row + 4 * i + sub;
        int32_t v = 0;
        if (i < n_i && pr < tl.seg_end && pr < args.gather_cap) {
          v = args.gather_src[pr];
          if (v < 0 || v >= args.src_rows) {
            set_status(args.status, MOE_ERR_DEVICE_BOUNDS);
            v = 0;
          } else {
            valid |= 1u << i;
          }
        }
        tok[i] = v;
      }
      for (; q < stages_per_tile; q += stages) {
        const int64_t j = j0 + q;
        const uint32_t phase = static_cast<uint32_t>((j / stages) & 1);
        bool go = true;
        if (lane == 0)
          go = mbar_wait_bounded(smem_u32(&empty[my_slot]), phase ^ 1u, abort_flag, args.status,
                                 kWaitLimitNs);
        go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
        if (!go) {
          ok = false;
          break;
        }
        const int kb = q * ksub + my_u;
        if (kb < k_blocks) {
          const uint32_t sA = smem_base + my_slot * stage_bytes + my_u * SUB_BYTES;
          const bool in_k = kb * BK + piece * 8 < args.k_dim;
          // a piece past the width reads nothing (zero fill); its address stays in the row
          const int64_t koff = in_k ? static_cast<int64_t>(kb) * (BK * 2) + piece * 16 : 0;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i < n_i) {
              const int r = 4 * i + sub;
              cp_async16(sA + r * 128 + ((piece ^ (r & 7)) * 16), xb + tok[i] * ld_bytes + koff,
                         (in_k && (valid >> i & 1u)) ? 16u : 0u);
            }
          }
          cp_async_commit();
          cp_async_wait<0>();
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&full[my_slot]), 0));
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync_all();   // no CTA leaves while its partner may still use its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

size_t pair_smem_bytes(int groups) {
  return 1024 + RING_BYTES + EPI_BYTES + 8 * (2 * RING_BLOCKS + 5) + 16 +
         8 * (static_cast<size_t>(groups) + 1) + 64;
}

template <int MODE, bool GATHER, int KSUB, bool H16>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& a64, const CUtensorMap& b0,
                        const CUtensorMap& b1, const CUtensorMap& b0h, const CUtensorMap& b1h,
                        const CUtensorMap& out, const PairArgs& args, int64_t max_pair_tiles,
                        cudaStream_t s) {
  if (max_pair_tiles <= 0) return cudaSuccess;
  const size_t smem = pair_smem_bytes(args.offsets ? args.groups : 1);
  auto kern = tc_pair_gemm<MODE, GATHER, KSUB, H16>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int64_t pairs_max = device_sm_count() >= 2 ? device_sm_count() / 2 : 1;
  const int64_t pairs = max_pair_tiles < pairs_max ? max_pair_tiles : pairs_max;
  kern<<<static_cast<unsigned>(2 * pairs), GATHER ? GATHER_THREADS : THREADS, smem, s>>>(
      a, a64, b0, b1, b0h, b1h, out, args);
  return cudaGetLastError();
}

}  // namespace

template <bool H16>
cudaError_t run_pair(const MlpParams& p, cudaStream_t s) {
  const bool dense = p.offsets == nullptr;
  const int64_t rows_cap = p.a_rows;
  if (rows_cap == 0 || (dense && p.dense_rows == 0)) return cudaSuccess;
  const int64_t mt_ub = dense ? (p.dense_rows + PM - 1) / PM : (rows_cap + PM - 1) / PM + p.groups;

  // Full-tile boxes of 128 rows and half-tile boxes of 64 (a gathered A is copied by the
  // gatherer warps and needs no map).
  CUtensorMap mA, mA64, mG, mU, mG64, mU64, mH, mH64, mD;
  const bool gather = p.gather_src != nullptr;
  const uint64_t w_rows = static_cast<uint64_t>(p.groups) * p.width;
  if ((!gather && !make_bf16_map(&mA, p.A, p.d, rows_cap, BM)) ||
      (!gather && !make_bf16_map(&mA64, p.A, p.d, rows_cap, HM)) ||
      !make_bf16_map(&mG, p.W_gate, p.d, w_rows, 128) ||
      !make_bf16_map(&mU, p.W_up, p.d, w_rows, 128) ||
      !make_bf16_map(&mG64, p.W_gate, p.d, w_rows, HM) ||
      !make_bf16_map(&mU64, p.W_up, p.d, w_rows, HM) ||
      !(H16 ? make_f16_map(&mH, p.h, p.width, rows_cap, BM)
            : make_bf16_map(&mH, p.h, p.width, rows_cap, BM)) ||
      !(H16 ? make_f16_map(&mH64, p.h, p.width, rows_cap, HM)
            : make_bf16_map(&mH64, p.h, p.width, rows_cap, HM)) ||
      !(H16 ? make_f16_map(&mD, down_values(p), p.width, static_cast<uint64_t>(p.groups) * p.d, 128)
            : make_bf16_map(&mD, p.W_down, p.width, static_cast<uint64_t>(p.groups) * p.d, 128)))
    return cudaErrorInvalidValue;
  if (gather) mA = mA64 = mG;   // unused placeholders

  PairArgs a{};
  a.offsets = p.offsets;
  a.dense_rows = static_cast<int32_t>(p.dense_rows);
  a.groups = p.groups;
  a.out_rows = rows_cap;
  a.status = p.status;
  a.gather_src = p.gather_src;
  a.gather_cap = rows_cap;
  a.src_rows = p.src_rows;
  a.gather_x = static_cast<const uint16_t*>(p.A);
  a.h_scale = p.h_scale;
  a.down_hdr = H16 ? static_cast<const PackHeader*>(p.W_down) : nullptr;
  a.down_elements = static_cast<int64_t>(p.groups) * p.d * p.width;
  // Two K blocks per ring stage when the average group has at least 512 rows (each
  // weight byte feeds enough rows for the tensor pipe to bound the launch); one
  // otherwise.
  const bool wide = (dense ? p.dense_rows : rows_cap / (p.groups > 0 ? p.groups : 1)) >= 512;

  a.k_dim = p.d;
  a.n_out = p.width;
  a.b_rows_per_group = p.width;
  a.out = p.h;
  a.ldo = p.width;
  const int64_t gu_tiles = mt_ub * ((p.width + 127) / 128);
  cudaError_t e =
      gather ? (wide ? launch_pair<kSwiGLU, true, 2, H16>(mA, mA64, mG, mU, mG64, mU64, mA, a, gu_tiles, s)
                     : launch_pair<kSwiGLU, true, 1, H16>(mA, mA64, mG, mU, mG64, mU64, mA, a, gu_tiles, s))
      : wide ? launch_pair<kSwiGLU, false, 2, H16>(mA, mA64, mG, mU, mG64, mU64, mA, a, gu_tiles, s)
             : launch_pair<kSwiGLU, false, 1, H16>(mA, mA64, mG, mU, mG64, mU64, mA, a, gu_tiles, s);
  if (e != cudaSuccess) return e;

  a.k_dim = p.width;
  a.n_out = p.d;
  a.b_rows_per_group = p.d;
  a.out = p.out;
  a.ldo = p.d;
  a.gather_src = nullptr;    // h is packed
  const int64_t d_tiles = mt_ub * ((p.d + 255) / 256);
  CUtensorMap mF;
  if (!(H16 ? make_f16_store_map(&mF, p.out, p.d, rows_cap) : make_f32_map(&mF, p.out, p.d, rows_cap)))
    return cudaErrorInvalidValue;
  return wide ? launch_pair<kPlain, false, 2, H16>(mH, mH64, mD, mD, mD, mD, mF, a, d_tiles, s)
              : launch_pair<kPlain, false, 1, H16>(mH, mH64, mD, mD, mD, mD, mF, a, d_tiles, s);
}

cudaError_t launch_mlp_bf16_pair(const MlpParams& p, cudaStream_t s) {
  return p.h_f16 ? run_pair<true>(p, s) : run_pair<false>(p, s);
}

}  // namespace moe

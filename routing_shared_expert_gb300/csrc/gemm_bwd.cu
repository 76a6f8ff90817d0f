// Grouped GEMMs of the layer's backward pass on the tensor cores (tcgen05 + TMEM, fed by TMA).
//
// The backward pass of Eq. 74 / Eq. 80 ("Section 21: Merging Routed and Shared Expert
// Activations", the backward study of Figure 70; "Section 20: One Shared Expert Is All
// You Need", Eq. 74) needs, per expert segment of packed rows, products whose operands
// sit in row-major buffers in either orientation:
//   recompute   [a | b] = x W_g^T | x W_u^T          A = rows (K-major), B = weights (K-major)
//   dgrad down  dh      = gf W_d                      A = rows (K-major), B = W_d (MN-major)
//   dgrad g/u   dx      = da W_g + db W_u             A = rows (K-major), B = W_g ; W_u (MN-major)
//   wgrad down  dW_d    = gf^T h                      A, B = rows read across (MN-major), K = segment
//   wgrad g/u   dW_g|u  = (da|db)^T x                 A, B = rows read across (MN-major), K = segment
// One kernel template covers them: C = A B^T with A and B each K-major (K contiguous) or
// MN-major (M or N contiguous), both loaded by TMA with 128-byte swizzle.  An MN-major
// operand tile is two 64-column boxes of 64 K-rows (8 KB apart: the descriptor's leading
// byte offset), K-rows 1024 bytes per 8 (its stride byte offset), and a K step of 16
// advances the start address by 2048 bytes; the instruction descriptor's bits 15 / 16 mark
// A / B as MN-major.
//
// Segments are padded to multiples of 64 rows with zero rows (the caller's layout), so a
// GEMM whose K runs over a segment's rows needs no masking.  Two epilogues: fp32 rows
// (dx, dW), and the SwiGLU backward for the down dgrad, which reads the recomputed a, b
// and writes da, db (bf16, the next GEMMs' operands) and h = SiLU(a) b (bf16):
//   da = dh * b * SiLU'(a),  db = dh * SiLU(a),  SiLU'(a) = sigma(a) (1 + a (1 - sigma(a))).
//
// Kernel design (persistent CTA pairs, cluster of 2, 192 threads each): a 256 x 256 tile
// per pair, the even CTA issuing tcgen05.mma cta_group::2 (M = 256, N = 256, K = 16); each
// CTA loads its 128 rows (or columns) of A and its 128 columns of B per 64-wide K block
// (32 KB, 6-stage ring), completing on the even CTA's barrier; each CTA's TMEM holds the
// fp32 accumulators of its 128 rows, double buffered; warp 0 TMA producer, warp 1 TMEM
// allocation (and MMA issue in the even CTA), warps 2-5 epilogue.  The epilogue stages
// each warp's 32 x 32 output blocks in shared memory in the swizzled layout of a store
// tensor map and writes them with TMA bulk tensor stores; blocks reaching past a segment's
// end or the width are written by the lanes instead.
// Every wait is bounded; a wait that runs out records MOE_ERR_TIMEOUT and the CTA drains
// what it issued before freeing its TMEM.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BMC = 128;                  // M rows (or columns) per CTA
constexpr int BM = 256;                   // M per pair tile
constexpr int BNC = 128;                  // N columns per CTA
constexpr int BN = 256;                   // N per pair tile
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int A_BYTES = BMC * BK * 2;
constexpr int B_BYTES = BNC * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
// Output staging per epilogue warp: one 32 x 32 fp32 block, or the da, db and h 32 x 32
// bf16 blocks of the SwiGLU epilogue (2 KB each).
constexpr int EPI_WARP_BYTES = 6144;
constexpr int EPI_BYTES = 4 * EPI_WARP_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 100000000ull;
constexpr uint32_t kMnLbo = 8192;   // bytes between the two 64-wide MN halves of a CTA's tile
constexpr uint32_t kMnSbo = 1024;   // bytes between groups of 8 K-rows

// SMEM descriptor of an MN-major, 128-byte-swizzled operand tile.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((kMnLbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((kMnSbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

struct BwdTile {
  int g, m, n;
  int seg_start, seg_end;   // padded segment rows of group g
};

// Tile t of a launch.  Within a group the tiles of one output-column block run together
// (the operand block they share is read once while the other streams), except in dense
// launches (one group, no segments: the shared expert's and the router's GEMMs) whose row
// operand is the larger one: there the column blocks of one row block run together, so the
// rows are read once while the smaller column operand, reused by every row block, stays in
// L2.
__device__ __forceinline__ bool bwd_tile(const BwdGemmArgs& a, bool k_seg, const int* s_off,
                                         const int* s_tp, int n_tiles, int64_t t, BwdTile& o) {
  const int G = a.seg_off ? a.groups : 1;
  if (k_seg) {
    const int mt = (a.m_dim + BM - 1) / BM;
    const int64_t per = static_cast<int64_t>(mt) * n_tiles;
    if (t >= per * G) return false;
    o.g = static_cast<int>(t / per);
    const int64_t local = t - static_cast<int64_t>(o.g) * per;
    const bool rows_first = a.seg_off == nullptr && a.m_dim > a.n_dim;
    o.n = static_cast<int>(rows_first ? local % n_tiles : local / mt);
    o.m = static_cast<int>(rows_first ? local / n_tiles : local % mt);
  } else {
    if (t >= static_cast<int64_t>(s_tp[G]) * n_tiles) return false;
    int lo = 0, hi = G;   // s_tp[lo] * n_tiles <= t < s_tp[hi] * n_tiles
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (static_cast<int64_t>(s_tp[mid]) * n_tiles <= t) lo = mid; else hi = mid;
    }
    const int mt = s_tp[lo + 1] - s_tp[lo];
    const int64_t local = t - static_cast<int64_t>(s_tp[lo]) * n_tiles;
    o.g = lo;
    const bool rows_first = a.seg_off == nullptr && a.dense_rows > a.n_dim;
    o.n = static_cast<int>(rows_first ? local % n_tiles : local / mt);
    o.m = static_cast<int>(rows_first ? local / n_tiles : local % mt);
  }
  o.seg_start = s_off[o.g];
  o.seg_end = s_off[o.g + 1];
  return true;
}

template <bool A_MN, bool B_MN, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    tc_bwd_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO,
                const __grid_constant__ CUtensorMap tmO2, const BwdGemmArgs args) {
  // A_MN: K runs over the segment rows (weight gradients); otherwise the rows are M.
  constexpr bool K_SEG = A_MN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint32_t* epi = reinterpret_cast<uint32_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + EPI_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* never = const_cast<int*>(abort_flag) + 1;
  const int G = args.seg_off ? args.groups : 1;
  int* s_off = never + 1;       // [G+1]
  int* s_tp = s_off + (G + 1);  // [G+1] pair m-tile prefix (row mode)

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int n_tiles = (args.n_dim + BN - 1) / BN;
  const uint32_t smem_base = smem_u32(smem);
  const int64_t pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
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
    if (args.seg_off == nullptr) {
      if (lane == 0) {
        s_off[0] = 0;
        s_off[1] = args.dense_rows;
        s_tp[0] = 0;
        s_tp[1] = (args.dense_rows + BM - 1) / BM;
      }
    } else {
      for (int i = lane; i <= G; i += 32) s_off[i] = args.seg_off[i];
      __syncwarp();
      int running = 0;
      for (int base = 0; base < G; base += 32) {
        const int g = base + lane;
        int v = 0;
        if (g < G) {
          const int len = s_off[g + 1] - s_off[g];
          if (len < 0 || (len & (BK - 1)) != 0) set_status(args.status, MOE_ERR_DEVICE_BOUNDS);
          v = len > 0 ? (len + BM - 1) / BM : 0;
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
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB0);
    tma_prefetch_map(&tmB1);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_holder), TMEM_COLS);
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();   // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  auto k_blocks_of = [&](const BwdTile& tl) {
    return K_SEG ? (tl.seg_end - tl.seg_start) / BK : args.k_dim / BK;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued_parity[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
      bool ok = true;
      BwdTile tl;
      for (int64_t t = pair_id; ok && bwd_tile(args, K_SEG, s_off, s_tp, n_tiles, t, tl);
           t += n_pairs) {
        const int kbs = k_blocks_of(tl);
        // this CTA's halves: M (rows or columns) m0.., N columns n0..
        const int m0 = tl.m * BM + static_cast<int>(rank) * BMC;
        const int n0 = tl.n * BN + static_cast<int>(rank) * BNC;
        for (int kb = 0; kb < kbs; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.status,
                                 kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = smem_u32(&full[stage]);
          const uint32_t fb = mapa_shared(fb_local, 0);
          if (leader) mbar_arrive_expect_tx(fb_local, 2 * STAGE_BYTES);
          const uint32_t sA = smem_base + stage * STAGE_BYTES;
          const uint32_t sB = sA + A_BYTES;
          const int k0 = kb * BK;
          if (A_MN) {
            const int row = tl.seg_start + k0;
            tma_load_2d_pair(sA, &tmA, m0, row, fb);
            tma_load_2d_pair(sA + kMnLbo, &tmA, m0 + 64, row, fb);
          } else {
            tma_load_2d_pair(sA, &tmA, k0, tl.seg_start + m0, fb);
          }
          if (B_MN) {
            // B[n][k] = view[row(k)][n]: weights (group rows) or segment rows
            const CUtensorMap* mb = &tmB0;
            int row;
            if (args.b_group_rows < 0) {
              row = tl.seg_start + k0;
            } else if (args.b_split_k > 0 && k0 >= args.b_split_k) {
              mb = &tmB1;
              row = tl.g * args.b_group_rows + (k0 - args.b_split_k);
            } else {
              row = tl.g * args.b_group_rows + k0;
            }
            tma_load_2d_pair(sB, mb, n0, row, fb);
            tma_load_2d_pair(sB + kMnLbo, mb, n0 + 64, row, fb);
          } else {
            // B[n][k] = view[g * b_group_rows + n][k], the second map past b_split_n
            const CUtensorMap* mb = &tmB0;
            int nn = n0;
            if (args.b_split_n > 0 && n0 >= args.b_split_n) {
              mb = &tmB1;
              nn = n0 - args.b_split_n;
            }
            tma_load_2d_pair(sB, mb, k0, tl.g * args.b_group_rows + nn, fb);
          }
          issued_parity[stage] = static_cast<int>(phase);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok && leader)
        for (int s = 0; s < STAGES; ++s)
          if (issued_parity[s] >= 0)
            mbar_wait_bounded(smem_u32(&full[s]), static_cast<uint32_t>(issued_parity[s]), never,
                              nullptr, kDrainLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN) | (A_MN ? (1u << 15) : 0u) |
                                 (B_MN ? (1u << 16) : 0u);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      BwdTile tl;
      int64_t local = 0;
      for (int64_t t = pair_id; ok && bwd_tile(args, K_SEG, s_off, s_tp, n_tiles, t, tl);
           t += n_pairs, ++local) {
        const int buf = static_cast<int>(local & 1);
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait_bounded(smem_u32(&tempty[buf]), (use & 1u) ^ 1u, abort_flag, args.status,
                               kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_acc = tmem_base + static_cast<uint32_t>(buf * BN);
        const int kbs = k_blocks_of(tl);
        for (int kb = 0; kb < kbs; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, args.status,
                                 kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_base + stage * STAGE_BYTES;
          const uint32_t sB = sA + A_BYTES;
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            const uint64_t ad = A_MN ? sw128_mnmajor_desc(sA + j * 2048) : sw128_kmajor_desc(sA) + 2 * j;
            const uint64_t bd = B_MN ? sw128_mnmajor_desc(sB + j * 2048) : sw128_kmajor_desc(sB) + 2 * j;
            tc_mma_bf16_pair(d_acc, ad, bd, idesc, (kb > 0 || j > 0) ? 1u : 0u);
          }
          tc_commit_pair(smem_u32(&empty[stage]), 0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit_pair(smem_u32(&tfull[buf]), 0x3);   // with no K blocks this arrives at once
      }
      if (!ok) {
        tc_commit_pair(smem_u32(drain), 0x1);
        mbar_wait_bounded(smem_u32(drain), 0, never, nullptr, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    BwdTile tl;
    int64_t local = 0;
    for (int64_t t = pair_id; bwd_tile(args, K_SEG, s_off, s_tp, n_tiles, t, tl);
         t += n_pairs, ++local) {
      const int buf = static_cast<int>(local & 1);
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      bool ready = true;
      if (lane == 0)
        ready = mbar_wait_bounded(smem_u32(&tfull[buf]), use & 1u, abort_flag, args.status,
                                  kWaitLimitNs);
      ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
      if (!ready) break;
      tc_fence_after();
      const bool empty_k = k_blocks_of(tl) == 0;   // no rows: the product is zero
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(buf * BN);
      const int r0 = tl.m * BM + static_cast<int>(rank) * BMC + q * 32;   // first tile row of the warp
      // destination of the warp's 32 rows (fp32 epilogue); rows past the end are dropped
      float* obase = args.out;
      int64_t orow0 = 0;
      int64_t rows_left = 0;
      int64_t map_row = 0;        // first row of the warp's block in the store map
      bool second = false;        // the block goes to out2
      if (EPI == kBwdEpiF32) {
        if (K_SEG) {
          // groups of rpg rows, group_stride apart (one group: m_dim rows)
          const int64_t rpg = args.group_stride > 0 ? args.group_stride / args.ldo : args.m_dim;
          orow0 = r0;
          obase = args.out + static_cast<int64_t>(tl.g) * args.group_stride;
          if (args.out_split_m > 0 && r0 >= args.out_split_m) {
            obase = args.out2 + static_cast<int64_t>(tl.g) * args.group_stride;
            orow0 = r0 - args.out_split_m;
            second = true;
          }
          rows_left = args.m_dim - r0;
          map_row = static_cast<int64_t>(tl.g) * rpg + orow0;
        } else {
          orow0 = tl.seg_start + r0;
          rows_left = tl.seg_end - orow0;
          map_row = orow0;
        }
      }
      uint8_t* blk = reinterpret_cast<uint8_t*>(epi) + (warp - 2) * EPI_WARP_BYTES;   // output staging
      float dot = 0.f;   // SwiGLU epilogue: this row's sum of dh_u * h over the tile's columns
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int col = tl.n * BN + c * 32;
        if (col >= args.n_dim) break;
        uint32_t v[32];
        if (empty_k) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        } else {
          tmem_ld32(taddr + c * 32, v);
        }
        if (EPI == kBwdEpiF32) {
          // The 32 x 32 block, staged in the 128-byte swizzled layout of the store maps
          // (16-byte piece j of row r at piece j ^ (r mod 8)), goes out by one TMA store when
          // all its rows and columns are inside; else the lanes write the rows that are.
          if (lane == 0) bulk_wait_read_all();   // the previous block has been read out
          __syncwarp();
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            *reinterpret_cast<uint4*>(blk + lane * 128 + ((v4 ^ (lane & 7)) * 16)) =
                make_uint4(v[4 * v4], v[4 * v4 + 1], v[4 * v4 + 2], v[4 * v4 + 3]);
          if (rows_left >= 32 && col + 32 <= args.n_dim) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(second ? &tmO2 : &tmO, col, static_cast<int32_t>(map_row), smem_u32(blk));
              bulk_commit();
            }
          } else {
            __syncwarp();
            // eight lanes per row (16 bytes each), four rows per pass
#pragma unroll
            for (int pass = 0; pass < 8; ++pass) {
              const int rr = pass * 4 + lane / 8;
              const uint4 val =
                  *reinterpret_cast<const uint4*>(blk + rr * 128 + (((lane % 8) ^ (rr & 7)) * 16));
              if (rr < rows_left)
                *reinterpret_cast<uint4*>(obase + (orow0 + rr) * args.ldo + col + (lane % 8) * 4) = val;
            }
            __syncwarp();
          }
        } else {
          // SwiGLU backward: dh_u in v; a, b from ab; da | db and scale * h out (bf16).  When
          // all 32 rows of the warp lie in the segment the three 32 x 32 blocks are staged in
          // the 64-byte swizzled layout of the store maps (16-byte piece j of row r at piece
          // j ^ ((r / 2) mod 4)) and go out by TMA; else each lane stores its own row.
          const int64_t row = tl.seg_start + r0 + lane;
          const bool block_in = tl.seg_start + r0 + 32 <= tl.seg_end;
          if (block_in) {
            if (lane == 0) bulk_wait_read_all();   // the previous blocks have been read out
            __syncwarp();
          }
          if (row < tl.seg_end) {
            const float sc = args.row_scale[row];
            const float4* arow =
                reinterpret_cast<const float4*>(args.ab + row * (2 * static_cast<int64_t>(args.width)) + col);
            const float4* brow = reinterpret_cast<const float4*>(
                args.ab + row * (2 * static_cast<int64_t>(args.width)) + args.width + col);
            __nv_bfloat16* drow = args.dab + row * (2 * static_cast<int64_t>(args.width));
            __nv_bfloat16* hrow = args.hout + row * static_cast<int64_t>(args.width);
            // all 16 loads of the chunk issued before any store (no aliasing assumed)
            float4 a4[8], b4[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              a4[i] = __ldg(arow + i);
              b4[i] = __ldg(brow + i);
            }
#pragma unroll
            for (int v8 = 0; v8 < 4; ++v8) {
              const float4 a0 = a4[2 * v8], a1 = a4[2 * v8 + 1];
              const float4 b0 = b4[2 * v8], b1 = b4[2 * v8 + 1];
              const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
              const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
              uint32_t da2[4], db2[4], h2[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float dav[2], dbv[2], hv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float a = av[2 * i + e];
                  const float b = bv[2 * i + e];
                  const float dhu = __uint_as_float(v[8 * v8 + 2 * i + e]);
                  const float dh = sc * dhu;
                  const float sg = 1.0f / (1.0f + __expf(-a));
                  const float sl = a * sg;
                  dav[e] = dh * b * (sg * (1.0f + a * (1.0f - sg)));
                  dbv[e] = dh * sl;
                  hv[e] = sc * (sl * b);
                  dot += dhu * (sl * b);
                }
                da2[i] = pack_bf16x2(dav[0], dav[1]);
                db2[i] = pack_bf16x2(dbv[0], dbv[1]);
                h2[i] = pack_bf16x2(hv[0], hv[1]);
              }
              if (block_in) {
                const int off = lane * 64 + ((v8 ^ ((lane >> 1) & 3)) * 16);
                *reinterpret_cast<uint4*>(blk + off) = make_uint4(da2[0], da2[1], da2[2], da2[3]);
                *reinterpret_cast<uint4*>(blk + 2048 + off) = make_uint4(db2[0], db2[1], db2[2], db2[3]);
                *reinterpret_cast<uint4*>(blk + 4096 + off) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
              } else {
                const int j0 = col + 8 * v8;
                *reinterpret_cast<uint4*>(drow + j0) = make_uint4(da2[0], da2[1], da2[2], da2[3]);
                *reinterpret_cast<uint4*>(drow + args.width + j0) = make_uint4(db2[0], db2[1], db2[2], db2[3]);
                *reinterpret_cast<uint4*>(hrow + j0) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
              }
            }
          }
          if (block_in) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int32_t brow = static_cast<int32_t>(tl.seg_start + r0);
              tma_store_2d(&tmO, col, brow, smem_u32(blk));                     // da
              tma_store_2d(&tmO, args.width + col, brow, smem_u32(blk + 2048));  // db
              tma_store_2d(&tmO2, col, brow, smem_u32(blk + 4096));             // scale * h
              bulk_commit();
            }
          }
        }
      }
      if (EPI == kBwdEpiSwiglu && args.dot_part != nullptr) {
        const int64_t row = tl.seg_start + r0 + lane;
        if (row < tl.seg_end) args.dot_part[row * ((args.width + BN - 1) / BN) + tl.n] = dot;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[buf]), 0));
    }
    if (lane == 0) bulk_wait_all();   // the output blocks are written
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync_all();   // no CTA leaves while its partner may still use its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

size_t bwd_smem_bytes(int groups) {
  return 1024 + STAGES * STAGE_BYTES + EPI_BYTES + 8 * (2 * STAGES + 5) + 16 +
         8 * (static_cast<size_t>(groups) + 1) + 64;
}

template <bool A_MN, bool B_MN, int EPI>
cudaError_t launch_one_bwd(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                           const BwdGemmArgs& args, int64_t max_tiles, cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  const size_t smem = bwd_smem_bytes(args.seg_off ? args.groups : 1);
  // store maps of the outputs: fp32 out (and out2 of a split output), or the SwiGLU
  // epilogue's bf16 da | db and h
  CUtensorMap mo = a, mo2 = a;
  if (EPI == kBwdEpiSwiglu) {
    const uint64_t rows = static_cast<uint64_t>(args.dense_rows);
    if (!make_bf16_store_map(&mo, args.dab, 2 * static_cast<uint64_t>(args.width), rows) ||
        !make_bf16_store_map(&mo2, args.hout, static_cast<uint64_t>(args.width), rows))
      return cudaErrorInvalidValue;
  }
  if (EPI == kBwdEpiF32) {
    const int64_t rpg = args.group_stride > 0 ? args.group_stride / args.ldo : args.m_dim;
    const int64_t rows = A_MN ? static_cast<int64_t>(args.seg_off ? args.groups : 1) * rpg
                              : static_cast<int64_t>(args.dense_rows);
    if (!make_f32_map(&mo, args.out, static_cast<uint64_t>(args.ldo), static_cast<uint64_t>(rows)))
      return cudaErrorInvalidValue;
    if (args.out2 && !make_f32_map(&mo2, args.out2, static_cast<uint64_t>(args.ldo),
                                   static_cast<uint64_t>(rows)))
      return cudaErrorInvalidValue;
  }
  auto kern = tc_bwd_gemm<A_MN, B_MN, EPI>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int64_t pairs_max = device_sm_count() >= 2 ? device_sm_count() / 2 : 1;
  const int64_t pairs = max_tiles < pairs_max ? max_tiles : pairs_max;
  kern<<<static_cast<unsigned>(2 * pairs), THREADS, smem, s>>>(a, b0, b1, mo, mo2, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_gemm(int kind, const CUtensorMap& a, const CUtensorMap& b0,
                            const CUtensorMap& b1, const BwdGemmArgs& args, int64_t max_tiles,
                            cudaStream_t s) {
  switch (kind) {
    case kBwdRowsKMajorB:   // recompute: A rows, B weights K-major, fp32 out
      return launch_one_bwd<false, false, kBwdEpiF32>(a, b0, b1, args, max_tiles, s);
    case kBwdRowsMnB:       // dgrad gate/up: A rows, B weights MN-major, fp32 out
      return launch_one_bwd<false, true, kBwdEpiF32>(a, b0, b1, args, max_tiles, s);
    case kBwdRowsMnBSwiglu: // dgrad down + SwiGLU backward
      return launch_one_bwd<false, true, kBwdEpiSwiglu>(a, b0, b1, args, max_tiles, s);
    case kBwdWeightGrad:    // wgrad: A, B MN-major over segment rows, fp32 blocks
      return launch_one_bwd<true, true, kBwdEpiF32>(a, b0, b1, args, max_tiles, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe

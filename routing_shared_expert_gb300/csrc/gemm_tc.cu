// Grouped SwiGLU expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM, fed by TMA).
//
// What is computed (Section 20 "One Shared Expert Is All You Need", Eq. 74, per
// packed segment of Section 10 "Routing, Capacity, and Load Balancing", Eq. 26):
//   gate/up:  h[row] = SiLU(x[row] W_g^e) * (x[row] W_u^e)      rows of expert e's segment
//   down:     f[row] = h[row] W_d^e        (fp32 output)
// Only rows [offsets[e], offsets[e+1]) are written; the offsets are read on the
// device, so no count ever travels to the host.  The shared expert is the same
// kernel over one dense group of T rows.
//
// Kernel design (one CTA per SM, persistent, 192 threads):
//   warp 0      TMA producer: per 64-wide K block, one 128-row A tile and the B
//               tile(s) into a 4-stage shared-memory ring (128-byte swizzle).
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16 (bf16 in,
//               fp32 accumulate in TMEM), M = 128; commits free ring stages and
//               publish finished accumulators.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator rows (one TMEM lane per
//               thread), SiLU(gate) * up to bf16 h, or the fp32 rows of f; row-masked stores.
// The accumulator is double buffered in TMEM (2 x 256 columns), so the epilogue
// of one tile overlaps the MMAs of the next.
//   SwiGLU mode: a tile is 128 rows x 128 h columns; the gate and up weight tiles
//                (128 rows each) feed two N = 128 MMAs into TMEM columns [0,128) and
//                [128,256), so SiLU(gate) * up pairs columns of one thread's row.
//   Plain mode:  a tile is 128 rows x 256 output columns, one N = 256 MMA per K step.
// Tiles are numbered group-major, then by output column block, then by row block,
// so CTAs that run together share the same weight tile through L2.
// Every wait is bounded (%globaltimer); a wait that runs out records
// MOE_ERR_TIMEOUT, the CTA drains what it issued, frees its TMEM and exits.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128;                   // rows per tile (MMA M)
constexpr int BK = 64;                    // K elements per stage = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BYTES = 256 * BK * 2;     // 32 KB: plain N = 256, or gate 128 + up 128
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint64_t kDrainLimitNs = 100000000ull;   // 100 ms

struct TcArgs {
  const int32_t* offsets;      // [groups+1] or nullptr (one dense group)
  const int32_t* tile_prefix;  // [groups+1] or nullptr
  int32_t dense_rows;
  int32_t groups;
  int32_t k_dim;
  int32_t n_out;               // output columns per group
  int32_t b_rows_per_group;    // rows between groups in the 2-D view of B
  int64_t out_rows;            // rows of the output buffer (stores beyond are dropped)
  void* out;                   // SwiGLU mode: bf16 h; plain mode: fp32 f
  int64_t ldo;
  int32_t* status;
  const int32_t* gather_src;   // non-null: A rows are gathered from x through this table
  int64_t gather_cap;
  int64_t src_rows;
  // fp16 intermediate: SwiGLU mode stores fp16(h * h_scale); plain mode reads the packed
  // weights' header and writes fp16(accumulator * 2^-k)
  float h_scale;
  const PackHeader* down_hdr;
  int64_t down_elements;
};

struct Tile {
  int g, m, n, seg_start, seg_end;
};

// Tile t -> (group, row block, column block).  s_tp / s_off are shared-memory
// copies of tile_prefix / offsets.
__device__ __forceinline__ bool tile_coords(const TcArgs& a, const int* s_tp, const int* s_off,
                                            int n_tiles, int64_t t, Tile& o) {
  if (a.tile_prefix == nullptr) {
    const int mt = (a.dense_rows + BM - 1) / BM;
    if (t >= static_cast<int64_t>(mt) * n_tiles) return false;
    o.g = 0;
    o.n = static_cast<int>(t / mt);
    o.m = static_cast<int>(t % mt);
    o.seg_start = 0;
    o.seg_end = a.dense_rows;
    return true;
  }
  const int G = a.groups;
  if (t >= static_cast<int64_t>(s_tp[G]) * n_tiles) return false;
  int lo = 0, hi = G;   // invariant: s_tp[lo] * n_tiles <= t < s_tp[hi] * n_tiles
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(s_tp[mid]) * n_tiles <= t) lo = mid; else hi = mid;
  }
  const int mt = s_tp[lo + 1] - s_tp[lo];
  const int64_t local = t - static_cast<int64_t>(s_tp[lo]) * n_tiles;
  o.g = lo;
  o.n = static_cast<int>(local / mt);
  o.m = static_cast<int>(local % mt);
  o.seg_start = s_off[lo];
  o.seg_end = s_off[lo + 1];
  return true;
}

template <bool SWIGLU, bool GATHER, bool H16>
__global__ void __launch_bounds__(THREADS, 1)
    tc_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const TcArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* never = const_cast<int*>(abort_flag) + 1;   // stays 0: drain waits ignore aborts
  int* s_tp = never + 1;
  int* s_off = s_tp + (args.groups + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int BN_OUT = SWIGLU ? 128 : 256;
  const int n_tiles = (args.n_out + BN_OUT - 1) / BN_OUT;
  const int k_blocks = (args.k_dim + BK - 1) / BK;
  const uint32_t smem_base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 4);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    *never = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB0);
    if (SWIGLU) tma_prefetch_map(&tmB1);
  }
  if (args.tile_prefix != nullptr) {
    for (int i = threadIdx.x; i <= args.groups; i += THREADS) {
      s_tp[i] = args.tile_prefix[i];
      s_off[i] = args.offsets[i];
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    int issued_parity[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
    bool ok = true;
    Tile tl;
    if constexpr (!GATHER) {
      // Lane 0 alone: wait for a free stage, arm its barrier, load A and B.
      if (lane == 0) {
        for (int64_t t = blockIdx.x; ok && tile_coords(args, s_tp, s_off, n_tiles, t, tl);
             t += gridDim.x) {
          const int a_row = tl.seg_start + tl.m * BM;
          const int b_row = tl.g * args.b_rows_per_group + tl.n * BN_OUT;
          for (int kb = 0; kb < k_blocks; ++kb) {
            if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.status,
                                   kWaitLimitNs)) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(&full[stage]);
            mbar_arrive_expect_tx(fb, STAGE_BYTES);
            const uint32_t sA = smem_base + stage * STAGE_BYTES;
            const uint32_t sB = sA + A_BYTES;
            tma_load_2d(sA, &tmA, kb * BK, a_row, fb);
            tma_load_2d(sB, &tmB0, kb * BK, b_row, fb);
            if (SWIGLU) tma_load_2d(sB + B_BYTES / 2, &tmB1, kb * BK, b_row, fb);
            issued_parity[stage] = static_cast<int>(phase);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
    } else {
      // Whole warp: lane 0 waits and loads B; every lane gathers four of the 128 A rows.
      for (int64_t t = blockIdx.x; ok && tile_coords(args, s_tp, s_off, n_tiles, t, tl);
           t += gridDim.x) {
        const int a_row = tl.seg_start + tl.m * BM;
        const int b_row = tl.g * args.b_rows_per_group + tl.n * BN_OUT;
        int32_t src[4];
        gather_rows4(args.gather_src, args.gather_cap, a_row + 4 * lane, tl.seg_start, tl.seg_end,
                     args.src_rows, args.status, src);
        for (int kb = 0; kb < k_blocks; ++kb) {
          bool go = true;
          if (lane == 0)
            go = mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.status,
                                   kWaitLimitNs);
          go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
          if (!go) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          const uint32_t sA = smem_base + stage * STAGE_BYTES;
          const uint32_t sB = sA + A_BYTES;
          if (lane == 0) {
            mbar_arrive_expect_tx(fb, STAGE_BYTES);
            tma_load_2d(sB, &tmB0, kb * BK, b_row, fb);
            if (SWIGLU) tma_load_2d(sB + B_BYTES / 2, &tmB1, kb * BK, b_row, fb);
            issued_parity[stage] = static_cast<int>(phase);
          }
          tma_gather4(sA + lane * 512, &tmA, kb * BK, src, fb);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
    if (!ok && lane == 0) {
      // Let every copy this warp started land before the CTA can exit.
      for (int s = 0; s < STAGES; ++s)
        if (issued_parity[s] >= 0)
          mbar_wait_bounded(smem_u32(&full[s]), static_cast<uint32_t>(issued_parity[s]), never,
                            nullptr, kDrainLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // gate/up multiply bf16 x by bf16 weights; the down GEMM of the fp16 intermediate
      // multiplies fp16 h by the packed fp16 weights
      constexpr uint32_t idesc =
          SWIGLU ? idesc_bf16_f32(BM, 128) : idesc_f32acc<H16>(BM, 256);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Tile tl;
      int64_t local = 0;
      for (int64_t t = blockIdx.x; ok && tile_coords(args, s_tp, s_off, n_tiles, t, tl);
           t += gridDim.x, ++local) {
        const int buf = static_cast<int>(local & 1);
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait_bounded(smem_u32(&tempty[buf]), (use & 1u) ^ 1u, abort_flag, args.status,
                               kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_acc = tmem_base + static_cast<uint32_t>(buf * 256);
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, args.status,
                                 kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_base + stage * STAGE_BYTES;
          const uint32_t sB = sA + A_BYTES;
          const uint64_t a_desc = sw128_kmajor_desc(sA);
          const uint64_t b_desc = sw128_kmajor_desc(sB);
          const uint64_t b1_desc = sw128_kmajor_desc(sB + B_BYTES / 2);
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            // K step j starts 32 bytes further into each 128-byte swizzled row.
            const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
            tc_mma_bf16(d_acc, a_desc + 2 * j, b_desc + 2 * j, idesc, acc);
            if (SWIGLU) tc_mma_bf16(d_acc + 128, a_desc + 2 * j, b1_desc + 2 * j, idesc, acc);
          }
          tc_commit(smem_u32(&empty[stage]));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tfull[buf]));
      }
      if (!ok) {
        // Let every MMA this thread issued finish before TMEM is released.
        tc_commit(smem_u32(drain));
        mbar_wait_bounded(smem_u32(drain), 0, never, nullptr, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may access
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
    for (int64_t t = blockIdx.x; tile_coords(args, s_tp, s_off, n_tiles, t, tl);
         t += gridDim.x, ++local) {
      const int buf = static_cast<int>(local & 1);
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      bool ready = true;
      if (lane == 0)
        ready = mbar_wait_bounded(smem_u32(&tfull[buf]), use & 1u, abort_flag, args.status,
                                  kWaitLimitNs);
      ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
      if (!ready) break;
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(tl.seg_start) + tl.m * BM + q * 32 + lane;
      const bool valid = row < tl.seg_end && row < args.out_rows;
      uint16_t* out_row = static_cast<uint16_t*>(args.out) + (valid ? row : 0) * args.ldo;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(buf * 256);
      if (SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t gr[32], ur[32];
          tmem_ld32x2(taddr + c * 32, taddr + 128 + c * 32, gr, ur);
          const int col0 = tl.n * 128 + c * 32;
          if (valid) {
            uint32_t pk[16];
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(gr[2 * i]), g1 = __uint_as_float(gr[2 * i + 1]);
              const float u0 = __uint_as_float(ur[2 * i]), u1 = __uint_as_float(ur[2 * i + 1]);
              if constexpr (H16) {
                const float s0 = silu(g0) * u0 * args.h_scale, s1 = silu(g1) * u1 * args.h_scale;
                amax = fmaxf(amax, fmaxf(fabsf(s0), fabsf(s1)));
                pk[i] = pack_f16x2(s0, s1);
              } else {
                pk[i] = pack_bf16x2(silu(g0) * u0, silu(g1) * u1);
              }
            }
            // an h value past the fp16 range became an infinity: report it
            if (H16 && !(amax < kF16RoundsToInf)) set_status(args.status, MOE_ERR_RANGE);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              if (col0 + v * 8 + 8 <= args.n_out)
                *reinterpret_cast<uint4*>(out_row + col0 + v * 8) =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else {
        // plain mode: output rows, fp32 (or fp16 of the fp16 intermediate, where they hold
        // f 2^-h_scale_log2)
        float* out_f = static_cast<float*>(args.out) + (valid ? row : 0) * args.ldo;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t ar[32], br[32];
          tmem_ld32x2(taddr + c * 64, taddr + c * 64 + 32, ar, br);
          const int col0 = tl.n * 256 + c * 64;
          if constexpr (H16) {
            if (valid) {
              uint16_t* orow = static_cast<uint16_t*>(args.out) + row * args.ldo;
              float m = 0.f;
              uint32_t pk[32];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float a0 = __uint_as_float(ar[2 * i]) * out_mul;
                const float a1 = __uint_as_float(ar[2 * i + 1]) * out_mul;
                const float b0 = __uint_as_float(br[2 * i]) * out_mul;
                const float b1 = __uint_as_float(br[2 * i + 1]) * out_mul;
                m = fmaxf(m, fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(b0), fabsf(b1))));
                pk[i] = pack_f16x2(a0, a1);
                pk[16 + i] = pack_f16x2(b0, b1);
              }
              if (!(m < kF16RoundsToInf)) set_status(args.status, MOE_ERR_RANGE);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                if (col0 + v * 8 + 8 <= args.n_out)
                  *reinterpret_cast<uint4*>(orow + col0 + v * 8) =
                      make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
            continue;
          }
          if (valid) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              if (col0 + v * 4 + 4 <= args.n_out)
                *reinterpret_cast<uint4*>(out_f + col0 + v * 4) =
                    make_uint4(ar[4 * v], ar[4 * v + 1], ar[4 * v + 2], ar[4 * v + 3]);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              if (col0 + 32 + v * 4 + 4 <= args.n_out)
                *reinterpret_cast<uint4*>(out_f + col0 + 32 + v * 4) =
                    make_uint4(br[4 * v], br[4 * v + 1], br[4 * v + 2], br[4 * v + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

size_t smem_bytes(int groups) {
  return 1024 + STAGES * STAGE_BYTES + 8 * (2 * STAGES + 5) + 16 + 8 * (groups + 1) + 64;
}

template <bool SWIGLU, bool GATHER, bool H16>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                       const TcArgs& args, int64_t max_tiles, cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  const size_t smem = smem_bytes(args.groups);
  auto kern = tc_grouped_gemm<SWIGLU, GATHER, H16>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  const int grid = static_cast<int>(max_tiles < sms ? max_tiles : sms);
  kern<<<grid, THREADS, smem, s>>>(a, b0, b1, args);
  return cudaGetLastError();
}

}  // namespace

namespace {

// 2-D tensor [rows][inner] (row-major, dense), box box_inner x box_rows, with the given
// shared-memory swizzle.  Encoded maps are cached (keyed by device, element type, address,
// shape, box and swizzle) so that repeated layer calls on the same buffers cost no driver
// work on the host.
bool make_map_2d(CUtensorMap* m, CUtensorMapDataType type, uint32_t elem_bytes, const void* base,
                 uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle) {
  struct Entry {
    int dev;
    CUtensorMapDataType type;
    const void* base;
    uint64_t inner, rows;
    uint32_t box_inner, box_rows;
    CUtensorMapSwizzle swizzle;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int n = 0, next = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
      if (cache[i].dev == dev && cache[i].type == type && cache[i].base == base &&
          cache[i].inner == inner && cache[i].rows == rows && cache[i].box_inner == box_inner &&
          cache[i].box_rows == box_rows && cache[i].swizzle == swizzle) {
        *m = cache[i].map;
        return true;
      }
  }
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  if (enc(m, type, 2, const_cast<void*>(base), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(mu);
  Entry& e = cache[next];
  e.dev = dev;
  e.type = type;
  e.base = base;
  e.inner = inner;
  e.rows = rows;
  e.box_inner = box_inner;
  e.box_rows = box_rows;
  e.swizzle = swizzle;
  e.map = *m;
  next = (next + 1) % 64;
  if (n < 64) ++n;
  return true;
}

}  // namespace

// bf16 [rows][inner], box 64 x box_rows (128-byte rows of the box), 128-byte swizzle.
bool make_bf16_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, rows, BK, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// fp16 [rows][inner]: the same boxes as make_bf16_map (fp16 intermediate h and packed
// down-projection weights).
bool make_f16_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, inner, rows, BK, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// fp16 [rows][inner], box 32 x 32 (64-byte rows), 64-byte swizzle: the fp16 output blocks
// (expert outputs of the fp16 intermediate) the expert GEMM epilogues store with TMA.
bool make_f16_store_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows) {
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, inner, rows, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_64B);
}

// fp32 [rows][inner], box 32 x 32 (128-byte rows), 128-byte swizzle: the output blocks the
// expert GEMM epilogues store with TMA.
bool make_f32_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows) {
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, inner, rows, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// bf16 [rows][inner], box 32 x 32 (64-byte rows), 64-byte swizzle: the 32-column blocks the
// backward SwiGLU epilogue stores with TMA.
bool make_bf16_store_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows) {
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, rows, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_64B);
}

cudaError_t set_smem_once(const void* func, size_t bytes) {
  struct Entry {
    const void* func;
    int dev;
    size_t bytes;
  };
  static std::mutex mu;
  static Entry seen[64];
  static int n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (seen[i].func == func && seen[i].dev == dev && seen[i].bytes >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n; ++i)
    if (seen[i].func == func && seen[i].dev == dev) {
      seen[i].bytes = bytes;
      return cudaSuccess;
    }
  if (n < 64) seen[n++] = Entry{func, dev, bytes};
  return cudaSuccess;
}

int device_sm_count() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

namespace {

template <bool H16>
cudaError_t run_one(const MlpParams& p, cudaStream_t s) {
  const bool dense = p.offsets == nullptr;
  const int64_t rows_cap = p.a_rows;
  if (rows_cap == 0 || (dense && p.dense_rows == 0)) return cudaSuccess;
  // Upper bound on row blocks without reading counts: each group adds at most one partial block.
  const int64_t mt_ub = dense ? (p.dense_rows + BM - 1) / BM : (rows_cap + BM - 1) / BM + p.groups;

  CUtensorMap mA, mG, mU, mH, mD;
  const bool gather = p.gather_src != nullptr;
  if (!make_bf16_map(&mA, p.A, p.d, gather ? p.src_rows : rows_cap, gather ? 1 : BM) ||
      !make_bf16_map(&mG, p.W_gate, p.d, static_cast<uint64_t>(p.groups) * p.width, 128) ||
      !make_bf16_map(&mU, p.W_up, p.d, static_cast<uint64_t>(p.groups) * p.width, 128) ||
      !(H16 ? make_f16_map(&mH, p.h, p.width, rows_cap, BM)
            : make_bf16_map(&mH, p.h, p.width, rows_cap, BM)) ||
      !(H16 ? make_f16_map(&mD, down_values(p), p.width, static_cast<uint64_t>(p.groups) * p.d, 256)
            : make_bf16_map(&mD, p.W_down, p.width, static_cast<uint64_t>(p.groups) * p.d, 256)))
    return cudaErrorInvalidValue;

  TcArgs a{};
  a.offsets = p.offsets;
  a.tile_prefix = p.tile_prefix;
  a.dense_rows = static_cast<int32_t>(p.dense_rows);
  a.groups = p.groups;
  a.status = p.status;
  a.out_rows = rows_cap;
  a.gather_src = p.gather_src;
  a.gather_cap = rows_cap;
  a.src_rows = p.src_rows;
  a.h_scale = p.h_scale;
  a.down_hdr = H16 ? static_cast<const PackHeader*>(p.W_down) : nullptr;
  a.down_elements = static_cast<int64_t>(p.groups) * p.d * p.width;

  // gate/up + SiLU -> h
  a.k_dim = p.d;
  a.n_out = p.width;
  a.b_rows_per_group = p.width;
  a.out = p.h;
  a.ldo = p.width;
  const int64_t gu_tiles = mt_ub * ((p.width + 127) / 128);
  cudaError_t e = gather ? launch_one<true, true, H16>(mA, mG, mU, a, gu_tiles, s)
                         : launch_one<true, false, H16>(mA, mG, mU, a, gu_tiles, s);
  if (e != cudaSuccess) return e;

  // down -> out (h is packed)
  a.gather_src = nullptr;
  a.k_dim = p.width;
  a.n_out = p.d;
  a.b_rows_per_group = p.d;
  a.out = p.out;
  a.ldo = p.d;
  return launch_one<false, false, H16>(mH, mD, mD, a, mt_ub * ((p.d + 255) / 256), s);
}

}  // namespace

cudaError_t launch_mlp_bf16(const MlpParams& p, cudaStream_t s) {
  return p.h_f16 ? run_one<true>(p, s) : run_one<false>(p, s);
}

}  // namespace moe

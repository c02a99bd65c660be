// K6, small-batch path: experts with few rows (EPS-MoE review, "GroupGemm vs
// DenseGemm": below a crossover the grouped GEMM wastes its tile on a handful
// of tokens, so small per-expert batches take a different kernel).
//
// For an expert with fewer than `small_threshold` rows the grouped kernels'
// 128-row tile would be mostly padding.  Here the product is computed
// transposed, Y^T = W^T X^T ("swap AB"):
//   MMA M = 128 output features (the weights, read as stored: features are
//           contiguous, i.e. an MN-major A operand),
//   MMA N = the group's rows, rounded up to 16 (at most 64 per tile),
//   MMA K = 16, accumulating in TMEM (lanes = features, columns = tokens).
// A 10-row expert thus costs an N=16 MMA instead of an M=128 one, and the
// kernel becomes a pure weight stream: 8 stages of 16 KB weights + 8 KB
// activations (GeLU / down projection) or 5 stages of 32 KB + 8 KB (SwiGLU,
// gate and up side by side).  Tiles are (unit = an expert's adjacent groups,
// 128-feature slice, 64-token chunk), chunks fastest, so tiles sharing a
// weight slice run together.
// Epilogue: 4 warps, lane = feature; for each token, a warp writes 32
// consecutive features (64 B).  The same warp roles, TMEM double buffering and
// bounded waits as the grouped kernel (ffn.cuh).
#pragma once
#include <cstddef>

#include "ffn.cuh"

namespace ffn_small {

using namespace sm100;
using ffn::gelu_erf;
using ffn::kGelu;
using ffn::kStore;
using ffn::kSwiglu;
using ffn::Params;
using ffn::wait_phase;

constexpr int BMF = 128;                  // output features per tile (MMA M)
constexpr int BT = 64;                    // tokens per tile at most (MMA N <= 64)
constexpr int BK = 64;
constexpr int W_BOX_BYTES = 64 * BK * 2;  // 8 KB: 64 features x 64 k
constexpr int W_BYTES = BMF * BK * 2;     // 16 KB per weight operand
constexpr int X_BYTES = BT * BK * 2;      // 8 KB: 64 token rows x 64 k
constexpr int EPI_WARPS = 4;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int MAX_G = 512;
static_assert(BT % 4 == 0 && BT / 4 <= 32 && BK * 2 == 128, "a gathered X tile is BT/4 lanes x 4 rows of 128 bytes");

template <int EPI>
struct Cfg {
  static constexpr int NW = (EPI == kSwiglu) ? 2 : 1;       // weight operands per stage
  static constexpr int STAGE = NW * W_BYTES + X_BYTES;       // 24 or 40 KB
  static constexpr int STAGES = (EPI == kSwiglu) ? 5 : 8;
  static constexpr uint32_t ACC_COLS = NW * BT;              // TMEM columns per accumulator buffer
  static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS <= 32 ? 32 : (2 * ACC_COLS <= 64 ? 64 : (2 * ACC_COLS <= 128 ? 128 : 256));
};

template <int EPI>
struct Smem {
  uint8_t stage[Cfg<EPI>::STAGES][Cfg<EPI>::STAGE];  // weights (NW x 16 KB) then X (8 KB)
  uint64_t full[Cfg<EPI>::STAGES];
  uint64_t empty[Cfg<EPI>::STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  int32_t total_tiles;
  int32_t u_count;
  int32_t goff[MAX_G + 1];   // staged group offsets
  int32_t us[MAX_G + 1];     // unit first rows (ffn::build_units)
  int32_t tstart[MAX_G + 1];
  int32_t nchunk[MAX_G];     // 64-token chunks of each small unit (0 = not handled here)
  int32_t ex[MAX_G];         // unit experts
  long long red[8];          // ffn::small_sms scratch
};

template <int EPI>
constexpr size_t smem_bytes() {
  return sizeof(Smem<EPI>) + 1024;
}
static_assert(sizeof(Smem<kSwiglu>) + 1024 <= 232448 && sizeof(Smem<kGelu>) + 1024 <= 232448,
              "shared memory beyond the 227 KB per-block opt-in limit");
static_assert(Cfg<kSwiglu>::STAGE % 1024 == 0 && Cfg<kGelu>::STAGE % 1024 == 0, "stages must stay 1024-aligned");

// 32 lanes x 16 consecutive 32-bit TMEM columns; waits for completion.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

struct Tile {
  int g, ft, rows;
  long long row0;
};

template <int EPI>
__device__ __forceinline__ Tile decode(const Smem<EPI>& s, int U, int tile) {
  int lo = 0, hi = U;  // tstart[lo] <= tile < tstart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tstart[mid] <= tile) lo = mid; else hi = mid;
  }
  Tile t;
  t.g = lo;
  const int local = tile - s.tstart[lo];
  const int nc = s.nchunk[lo];
  t.ft = local / nc;
  t.row0 = (long long)s.us[lo] + (long long)(local % nc) * BT;
  const long long left = (long long)s.us[lo + 1] - t.row0;
  t.rows = left < BT ? (int)left : BT;
  return t;
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    small_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW0,
                 const __grid_constant__ CUtensorMap tmW1, const Params p) {
  using C = Cfg<EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem<EPI>& s = *reinterpret_cast<Smem<EPI>*>(base);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- units (an expert's adjacent groups) with fewer than small_threshold
  // rows, in 64-token chunks
  const int U = ffn::build_units<THREADS>(p, s.goff, s.us, s.ex, &s.u_count);
  // with an SM split (ffn::small_sms) this kernel runs on S SMs, or not at
  // all when S = 0 (the grouped kernels then take the small experts too)
  const int S = ffn::small_sms<THREADS>(p, U, s.us, s.ex, s.red);
  ffn::unit_tile_prefix<THREADS>(p, U, s.us, s.ex, s.nchunk, s.tstart, &s.total_tiles, BT,
                                 [&](int rows) { return S != 0 && rows < p.small_threshold; });
  __syncthreads();
  const int nctas = (S > 0 && S < (int)gridDim.x) ? S : (int)gridDim.x;
  // no tiles, or a CTA beyond this kernel's share: exit before any barrier or TMEM set-up
  if (s.total_tiles == 0 || (int)blockIdx.x >= nctas) return;
  s.red[1] = nctas;  // read back per tile: the loops below keep no register for it
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], EPI_WARPS);
    }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW0);
    if (EPI == kSwiglu) tma_prefetch_desc(&tmW1);
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(&s.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;
  const int total = s.total_tiles;
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // lane 0 waits, arms the stage and loads the weights (and X when stored
    // in row order); a gathered X is copied by lanes 0..15, four rows each
    const bool gather = p.a_src != nullptr;
    uint32_t stage = 0, phase = 0, issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += (int)*(volatile long long*)&s.red[1]) {
      const Tile t = decode(s, U, tile);
      const int wrow = s.ex[t.g] * p.K;
      const int f0 = t.ft * BMF;
      const int4 src = (gather && lane < BT / 4) ? ffn::gather_src4(p, t.row0, lane) : make_int4(0, 0, 0, 0);
      for (int kb = 0; kb < kblocks; ++kb) {
        bool w = true;
        if (lane == 0) w = wait_phase(&s.empty[stage], phase ^ 1, &s.abort_flag);
        if (!__shfl_sync(0xffffffffu, (int)w, 0)) {
          ok = false;
          break;
        }
        uint8_t* st = s.stage[stage];
        if (lane == 0) {
          mbar_arrive_expect_tx(&s.full[stage], C::STAGE);
#pragma unroll
          for (int op = 0; op < C::NW; ++op) {
            const CUtensorMap* m = op == 0 ? &tmW0 : &tmW1;
            tma_load_2d(st + op * W_BYTES, m, &s.full[stage], f0, wrow + kb * BK);
            tma_load_2d(st + op * W_BYTES + W_BOX_BYTES, m, &s.full[stage], f0 + 64, wrow + kb * BK);
          }
          if (!gather) tma_load_2d(st + C::NW * W_BYTES, &tmX, &s.full[stage], kb * BK, (int)t.row0);
        }
        __syncwarp();
        if (gather && lane < BT / 4) tma_gather4(st + C::NW * W_BYTES + lane * 512, &tmX, &s.full[stage], kb * BK, src);
        ++issued;
        if (++stage == (uint32_t)C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (lane == 0) {
      for (uint32_t st = 0; st < (uint32_t)C::STAGES; ++st) {
        if (issued > st) {
          const uint32_t last = issued - 1 - ((issued - 1 - st) % C::STAGES);
          wait_phase(&s.full[st], (last / C::STAGES) & 1u, &s.abort_flag, true);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, any_mma = false;
      // weights: MN-major A (64-feature boxes 8 KB apart, 8 k-rows 1024 B
      // apart, K step of 16 = +128 in the start field); activations: K-major B
      // (128-byte rows, 8-row groups 1024 B apart, K step of 16 = +2)
      const uint64_t wdesc0 = smem_desc_sw128(smem_u32(s.stage[0]), W_BOX_BYTES, 1024);
      const uint64_t xdesc0 = smem_desc_sw128(smem_u32(s.stage[0]) + C::NW * W_BYTES, 16, 1024);
      for (int tile = blockIdx.x; tile < total && ok; tile += (int)*(volatile long long*)&s.red[1]) {
        const Tile t = decode(s, U, tile);
        const int npad = (t.rows + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(BMF, npad, true, false);
        if (!wait_phase(&s.tempty[acc], acc_phase ^ 1, &s.abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * C::ACC_COLS;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_phase(&s.full[stage], phase, &s.abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)(stage * (C::STAGE >> 4));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t xd = xdesc0 + so + (uint64_t)(kk * 2);
#pragma unroll
            for (int op = 0; op < C::NW; ++op)
              mma_bf16(d + op * BT, wdesc0 + so + (uint64_t)(op * (W_BYTES >> 4) + kk * 128), xd, idesc,
                       (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&s.empty[stage]);
          any_mma = true;
          if (++stage == (uint32_t)C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&s.tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (any_mma) {
        mma_commit(&s.drain);
        wait_phase(&s.drain, 0, &s.abort_flag, true);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes (features) 32*quarter .. +31
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += (int)*(volatile long long*)&s.red[1]) {
      const Tile t = decode(s, U, tile);
      if (!__all_sync(0xffffffffu, wait_phase(&s.tfull[acc], acc_phase, &s.abort_flag))) break;
      tc_fence_after();
      const int f = t.ft * BMF + quarter * 32 + lane;  // this thread's output feature
      const bool f_ok = f < p.N_out;
      const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * C::ACC_COLS;
      uint16_t* ocol = p.out + (size_t)t.row0 * p.N_out + (f_ok ? f : 0);
#pragma unroll 1
      for (int c0 = 0; c0 < t.rows; c0 += 16) {
        uint32_t g[16];
        __syncwarp();
        tmem_ld16(tb + c0, g);
        float v[16];
        if (EPI == kSwiglu) {
          uint32_t u[16];
          tmem_ld16(tb + BT + c0, u);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float z = __uint_as_float(g[i]);
            v[i] = __fdividef(z, 1.0f + __expf(-z)) * __uint_as_float(u[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float z = __uint_as_float(g[i]);
            v[i] = (EPI == kGelu) ? gelu_erf(z) : z;
          }
        }
        if (EPI == ffn::kCombine) {
          // each token row: its gate weight times the value, added into the
          // row's token in the fp32 accumulator (32 consecutive features per warp)
#pragma unroll 1
          for (int i = 0; i < 16; ++i) {
            if (c0 + i >= t.rows) break;
            float wt;
            float* arow = ffn::comb_target(p, t.row0 + c0 + i, t.row0 + t.rows, wt);
            if (arow && f_ok)
              asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(arow + f), "f"(wt * v[i]) : "memory");
          }
        } else if (f_ok) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (c0 + i < t.rows) {
              __nv_bfloat16 b = __float2bfloat16_rn(v[i]);
              ocol[(size_t)(c0 + i) * p.N_out] = *reinterpret_cast<uint16_t*>(&b);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace ffn_small

// K6: grouped expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// PopFetcher (ATC'25) review: MoE-GPT experts are GeLU MLPs with F = alpha*H.
// EPS-MoE review, "MoE architecture analysis": the gate, up and down GEMMs are
// the compute-bound part of the layer; "GroupGemm vs DenseGemm": all experts'
// GEMMs run in one kernel (GroupGemm), with a separate path for small
// per-expert batches.
//
// Two launches of one persistent, warp-specialised kernel template:
//   GEMM1: inter[A, F] = act(xp[A, H] . W1[e])            (GeLU)
//          inter[A, F] = silu(xp . W1[e]) * (xp . W3[e])  (SwiGLU)
//   GEMM2: y[A, H]     = inter[A, F] . W2[e]
// Rows are grouped by expert (or replica group); group sizes live only on the
// device, so every CTA reads the group offsets and enumerates the tiles
// (group, n-tile, m-tile) itself, m fastest so that CTAs running at the same
// time share the expert's weight tile in L2.  CTA c takes tiles c, c+grid, ...
//
// Per CTA (one per SM, 320 threads):
//   warp 0      TMA producer: A tile 128x64 (K-major) and B tile 64x256
//               (weights as stored, N contiguous = MN-major), 128-byte
//               swizzle, into a 4-stage ring guarded by full/empty mbarriers.
//   warp 1      TMEM allocator and MMA issuer: one thread issues
//               tcgen05.mma (M=128, N=256, K=16, bf16 in, fp32 accumulate in
//               TMEM) and tcgen05.commit frees each smem stage; two TMEM
//               accumulators (2 x 256 columns) let the epilogue of one tile
//               overlap the main loop of the next.
//   warps 2..9  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4).., half the columns each), activation in
//               fp32, bf16 rounding, row-masked stores (rows past the
//               group's end belong to another group and are not written).
// For SwiGLU the B tile holds 128 columns of W1 then the same 128 columns of
// W3, so one N=256 MMA yields gate and up side by side in TMEM.
//
// Every mbarrier wait is bounded (2 s of %globaltimer): on expiry the
// waiting role raises the CTA's abort flag and the device timeout bit, the
// other roles leave their loops at their next wait, the producer waits for
// the copies it issued, the MMA thread for its MMAs, and TMEM is freed before
// the CTA exits.
#pragma once
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace ffn {

using namespace sm100;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;  // 8 KB: 64 columns x 64 k-rows
constexpr int B_BYTES = BN * BK * 2;      // 32 KB
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr int MAX_G = 512;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint64_t kWaitBudgetNs = 2000000000ull;
constexpr uint32_t kMaxPolls = 1u << 30;

enum Epi : int { kGelu = 0, kSwiglu = 1, kStore = 2 };

struct Params {
  const int32_t* group_offsets;  // [G+1]
  const int32_t* group_expert;   // [G] or null (group g = expert g)
  int G;
  int E;
  long long A_rows;  // rows of the A operand and of the output
  int K;             // reduction length, multiple of BK
  int N_out;         // output columns, multiple of 64
  int n_tiles;       // N tiles per group
  uint16_t* out;     // [A_rows, N_out] bf16
  int flags;         // bit 0: CTA 0 withholds its first accumulator signal (timeout self-test)
};

struct Smem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  int32_t total_tiles;
  int32_t goff[MAX_G + 1];
  int32_t tstart[MAX_G + 1];
  int32_t mt[MAX_G];
  int32_t ex[MAX_G];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack

// Wait for the phase of `bar` with parity `parity`.  Returns false when another
// role of this CTA aborted (unless ignore_abort) or after the time budget, in
// which case it raises the abort flag and the device timeout bit.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint32_t* abort_flag,
                                           bool ignore_abort = false) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  volatile uint32_t* ab = abort_flag;
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((i & 127) == 127) {
      if (!ignore_abort && *ab) return false;
      if (globaltimer_ns() - t0 > kWaitBudgetNs) break;
    }
  }
  *ab = 1;
  moe_flag_error(MOE_DEVERR_TIMEOUT);
  return false;
}

struct Tile {
  int g, nt, rows;
  long long row0;
};

__device__ __forceinline__ Tile decode(const Smem& s, int G, int tile) {
  int lo = 0, hi = G;  // tstart[lo] <= tile < tstart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tstart[mid] <= tile) lo = mid; else hi = mid;
  }
  Tile t;
  t.g = lo;
  const int local = tile - s.tstart[lo];
  const int m = s.mt[lo];
  t.nt = local / m;
  t.row0 = (long long)s.goff[lo] + (long long)(local % m) * BM;
  const long long left = (long long)s.goff[lo + 1] - t.row0;
  t.rows = left < BM ? (int)left : BM;
  return t;
}

__device__ __forceinline__ float gelu_erf(float x) { return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f)); }

__device__ __forceinline__ void store32(uint16_t* dst, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 o;
    o.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    o.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    o.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    o.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    st_v4(dst + 8 * q, o);
  }
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmB1, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem& s = *reinterpret_cast<Smem*>(base);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
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
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    if (EPI == kSwiglu) tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) {
    __syncwarp();  // .sync.aligned: whole warp, converged
    tmem_alloc(&s.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }

  // ---- group table: validate offsets, m-tiles per group, tile prefix
  for (int g = threadIdx.x; g <= G; g += THREADS) s.goff[g] = p.group_offsets[g];
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += THREADS) {
    const long long lo = s.goff[g], hi = s.goff[g + 1];
    long long rows = hi - lo;
    const int e = p.group_expert ? p.group_expert[g] : g;
    bool bad = lo < 0 || hi < lo || hi > p.A_rows;
    if (!bad && rows > 0 && (e < 0 || e >= p.E)) bad = true;
    if (bad) {
      moe_flag_error(MOE_DEVERR_DATA);
      rows = 0;
    }
    s.mt[g] = (int)((rows + BM - 1) / BM);
    s.ex[g] = e;
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int c0 = 0; c0 < G; c0 += 32) {
      const int g = c0 + lane;
      const int v = g < G ? s.mt[g] * p.n_tiles : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += u;
      }
      if (g < G) s.tstart[g] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s.tstart[G] = carry;
      s.total_tiles = carry;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;
  const int total = s.total_tiles;
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = decode(s, G, tile);
        const int brow = s.ex[t.g] * p.K;
        const int arow = (int)t.row0;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_phase(&s.empty[stage], phase ^ 1, &s.abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.full[stage], A_BYTES + B_BYTES);
          tma_load_2d(s.a[stage], &tmA, &s.full[stage], kb * BK, arow);
          if (EPI == kSwiglu) {
            const int n0 = t.nt * (BN / 2);
            tma_load_2d(s.b[stage] + 0 * B_BOX_BYTES, &tmB0, &s.full[stage], n0, brow + kb * BK);
            tma_load_2d(s.b[stage] + 1 * B_BOX_BYTES, &tmB0, &s.full[stage], n0 + 64, brow + kb * BK);
            tma_load_2d(s.b[stage] + 2 * B_BOX_BYTES, &tmB1, &s.full[stage], n0, brow + kb * BK);
            tma_load_2d(s.b[stage] + 3 * B_BOX_BYTES, &tmB1, &s.full[stage], n0 + 64, brow + kb * BK);
          } else {
            const int n0 = t.nt * BN;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              tma_load_2d(s.b[stage] + c * B_BOX_BYTES, &tmB0, &s.full[stage], n0 + 64 * c, brow + kb * BK);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // every stage's latest copy must have landed before the CTA may exit
      for (uint32_t st = 0; st < (uint32_t)STAGES; ++st) {
        if (issued > st) {
          const uint32_t last = issued - 1 - ((issued - 1 - st) % STAGES);
          wait_phase(&s.full[st], (last / STAGES) & 1u, &s.abort_flag, true);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false, true);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, withheld = false, any_mma = false;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        if (!wait_phase(&s.tempty[acc], acc_phase ^ 1, &s.abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_phase(&s.full[stage], phase, &s.abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(s.a[stage]);
          const uint32_t b0 = smem_u32(s.b[stage]);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A: K-major, 128-byte rows, 8-row groups 1024 B apart; K step = 32 B.
            // B: MN-major, 64-column boxes 8 KB apart (LBO), 8 k-rows 1024 B apart (SBO);
            //    K step of 16 rows = 2048 B.
            mma_bf16(d, smem_desc_sw128(a0 + kk * 32, 16, 1024), smem_desc_sw128(b0 + kk * 2048, B_BOX_BYTES, 1024),
                     idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&s.empty[stage]);
          any_mma = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if ((p.flags & 1) && blockIdx.x == 0 && !withheld)
          withheld = true;  // self-test: this accumulator is never signalled
        else
          mma_commit(&s.tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (any_mma) {  // all issued MMAs must finish before TMEM is freed
        mma_commit(&s.drain);
        wait_phase(&s.drain, 0, &s.abort_flag, true);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode(s, G, tile);
      // every lane waits; the vote keeps the warp converged for tcgen05.ld
      if (!__all_sync(0xffffffffu, wait_phase(&s.tfull[acc], acc_phase, &s.abort_flag))) break;
      tc_fence_after();
      const int r = quarter * 32 + lane;
      const bool row_ok = r < t.rows;
      uint16_t* orow = p.out + (size_t)(t.row0 + (row_ok ? r : 0)) * p.N_out;
      const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (EPI == kSwiglu) {
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          const int c = half * 64 + cc * 32;
          uint32_t gr[32], ur[32];
          __syncwarp();
          tmem_ld32(tb + c, gr);
          tmem_ld32(tb + BN / 2 + c, ur);
          const int col = t.nt * (BN / 2) + c;
          if (row_ok && col < p.N_out) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float g = __uint_as_float(gr[i]);
              v[i] = g / (1.0f + __expf(-g)) * __uint_as_float(ur[i]);
            }
            store32(orow + col, v);
          }
        }
      } else {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          const int c = half * (BN / 2) + cc * 32;
          uint32_t raw[32];
          __syncwarp();
          tmem_ld32(tb + c, raw);
          const int col = t.nt * BN + c;
          if (row_ok && col < p.N_out) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float z = __uint_as_float(raw[i]);
              v[i] = (EPI == kGelu) ? gelu_erf(z) : z;
            }
            store32(orow + col, v);
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

  // ---- teardown: every role has left its loop (all waits are bounded)
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace ffn

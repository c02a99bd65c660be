// K6, fused form: both GEMMs of the expert FFN in one persistent CTA-pair
// kernel (EPS-MoE review, "GroupGemm": every expert's GEMM in one kernel).
//
// The two-launch form (ffn_pair.cuh) loses two things on this part: GEMM2's
// last wave (its few long tiles run alone at the end) and GEMM1's activation
// epilogue, which is on GEMM1's critical path because its tiles have half
// GEMM2's k-blocks.  Here one launch runs the tiles of both GEMMs over the
// same 256-row blocks of the dispatched rows, in one order known to every
// role of every pair:
//   block b = (unit, 256-row tile of the unit), B blocks in all;
//   N1 GEMM1 tiles and N2 GEMM2 tiles per block;
//   order: the GEMM1 tiles of blocks 0..D-1, then for b = D..B-1 the GEMM1
//   tiles of block b followed by the GEMM2 tiles of block b-D, then the
//   GEMM2 tiles of blocks B-D..B-1.
// Pair c takes positions c, c + pairs, ...  so every pair alternates short
// GEMM1 tiles (heavy epilogue) with long GEMM2 tiles, and the epilogue of one
// overlaps the main loop of the next; the lag D (about three rounds of tiles)
// lets a block's GEMM1 tiles finish before its GEMM2 tiles come up.
//
// Dependency: a GEMM2 tile reads the bf16 intermediate rows of its block,
// written by the block's GEMM1 epilogues.  Every epilogue warp of a GEMM1
// tile, after its stores, fences (gpu scope) and adds 1 to the block's
// counter; the producers of a GEMM2 tile wait (bounded) until the counter
// reaches 2 CTAs x 16 warps x N1, then order those generic-proxy writes
// before their tensor copies (fence.proxy.async) and load.  Every tile a
// GEMM2 tile waits for sits earlier in the order, and every pair runs its
// tiles in order, so the smallest unfinished position can always proceed
// (no cycle).  The grid is at most the number of co-resident pairs, and no
// other kernel waits on this one, so a pair that is not resident at first
// (SMs held by the small-batch kernels on the side stream) becomes resident
// when those finish; every wait is bounded all the same.
// Each tile's arithmetic is exactly the two-launch kernel's (same tiles,
// same k order), so the output is bit-identical to it.
#pragma once
#include "ffn_pair.cuh"

namespace ffn3 {

using namespace sm100;
using ffn::kGelu;
using ffn::kStore;
using ffn::kSwiglu;
using ffn::Params;
using ffn::pack32;
using ffn::store_rows32;
using ffn::gelu_erf;
using ffn2::A_BYTES;
using ffn2::B_BOX_BYTES;
using ffn2::B_HALF_BYTES;
using ffn2::BK;
using ffn2::BM;
using ffn2::BMP;
using ffn2::BN;
using ffn2::EPI_SLICES;
using ffn2::EPI_WARPS;
using ffn2::Smem;
using ffn2::STAGES;
using ffn2::THREADS;
using ffn2::TMEM_COLS;
using ffn2::wait_phase;
using ffn2::kSmemBytes;

struct FusedParams {
  Params p1;          // GEMM1: K = H, N_out = F, out = intermediate
  Params p2;          // GEMM2: K = F, N_out = H, out = y
  uint32_t* done;     // [blocks] GEMM1 epilogue warps finished per block; zero at launch
  int lag;            // D
};

constexpr uint64_t kDepBudgetNs = 2000000000ull;

struct FTile {
  int phase;          // 1 or 2
  int u;              // unit
  int nt;             // n-tile
  int b;              // block
  long long row0;     // first row of the pair tile
};

// Position -> tile (the order described at the top of this file).  bstart[u]
// = first block of unit u (tstart of unit_tile_prefix with one tile per block).
__device__ __forceinline__ FTile decode(const Smem& s, int U, int B, int N1, int N2, int D, int pos) {
  FTile t;
  int b, n;
  const int head = D * N1;
  if (pos < head) {
    t.phase = 1;
    b = pos / N1;
    n = pos % N1;
  } else {
    const int q = pos - head;
    const int mid = (B - D) * (N1 + N2);
    if (q < mid) {
      const int sb = q / (N1 + N2), r = q % (N1 + N2);
      if (r < N1) {
        t.phase = 1;
        b = D + sb;
        n = r;
      } else {
        t.phase = 2;
        b = sb;
        n = r - N1;
      }
    } else {
      const int q2 = q - mid;
      t.phase = 2;
      b = (B - D) + q2 / N2;
      n = q2 % N2;
    }
  }
  int lo = 0, hi = U;  // tstart[lo] <= b < tstart[hi]
  while (hi - lo > 1) {
    const int m = (lo + hi) >> 1;
    if (s.tstart[m] <= b) lo = m; else hi = m;
  }
  t.u = lo;
  t.nt = n;
  t.b = b;
  t.row0 = (long long)s.us[lo] + (long long)(b - s.tstart[lo]) * BMP;
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait for a block's GEMM1 tiles.  False after the budget (abort
// flag and timeout bit raised) or when another role aborted.
__device__ __forceinline__ bool wait_block(const uint32_t* counter, uint32_t target, uint32_t* abort_flag) {
  if (ld_acquire_gpu(counter) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  volatile uint32_t* ab = abort_flag;
  for (uint32_t i = 0; i < ffn::kMaxPolls; ++i) {
    if (ld_acquire_gpu(counter) >= target) return true;
    if ((i & 63) == 63) {
      if (*ab) return false;
      if (globaltimer_ns() - t0 > kDepBudgetNs) break;
    }
    __nanosleep(64);
  }
  *ab = 1;
  moe_flag_error(MOE_DEVERR_TIMEOUT);
  return false;
}

template <int EPI1>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    ffn_fused_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmW1,
                     const __grid_constant__ CUtensorMap tmW3, const __grid_constant__ CUtensorMap tmA2,
                     const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ FusedParams fp) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem& s = *reinterpret_cast<Smem*>(base);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const Params& p1 = fp.p1;
  const Params& p2 = fp.p2;

  // ---- units and their 256-row blocks (identical in every CTA)
  Params pb = p1;
  pb.n_tiles = 1;
  const int U = ffn::build_units<THREADS>(pb, s.goff, s.us, s.ex, &s.u_count);
  // with an SM split (ffn::small_sms) the small-batch experts are left to the
  // small-batch kernels only when they get SMs (S > 0), and the pairs beyond
  // this kernel's (split_ctas - S) / 2 exit.  The pairs that stay are
  // co-resident once the exiting CTAs and the small-batch kernels' CTAs
  // beyond their own share have left, which they do without waiting on
  // anything, so the dependency waits below still always progress.
  const int S = ffn::small_sms<THREADS>(pb, U, s.us, s.ex, s.red);
  const bool skip_small = pb.small_threshold > 0 && S != 0;
  ffn::unit_tile_prefix<THREADS>(pb, U, s.us, s.ex, s.mt, s.tstart, &s.total_tiles, BMP,
                                 [&](int rows) { return !skip_small || rows >= pb.small_threshold; });
  __syncthreads();
  const int B = s.total_tiles;
  const int npairs = (S > 0 && (pb.split_ctas - S) / 2 < (int)(gridDim.x >> 1)) ? (pb.split_ctas - S) / 2
                                                                                   : (int)(gridDim.x >> 1);
  // no tiles, or a pair beyond this kernel's share: exit before any barrier or TMEM set-up
  if (B == 0 || pair >= npairs) return;
  s.red[1] = npairs;  // read back per tile: the loops below keep no register for it
  const int N1 = p1.n_tiles, N2 = p2.n_tiles;
  const int D = fp.lag < B ? fp.lag : B;
  const int total = B * (N1 + N2);
  const uint32_t dep_target = 2u * EPI_WARPS * (uint32_t)N1;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 2 * EPI_WARPS);
    }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmW1);
    if (EPI1 == kSwiglu) tma_prefetch_desc(&tmW3);
    tma_prefetch_desc(&tmA2);
    tma_prefetch_desc(&tmW2);
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc_pair(&s.tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      const uint32_t full0 = mapa_shared(smem_u32(&s.full[0]), 0);  // leader's barriers
      for (int pos = pair; pos < total && ok; pos += (int)*(volatile long long*)&s.red[1]) {
        const FTile t = decode(s, U, B, N1, N2, D, pos);
        const bool g1 = t.phase == 1;
        const Params& p = g1 ? p1 : p2;
        const CUtensorMap* mA = g1 ? &tmA1 : &tmA2;
        const CUtensorMap* mB = g1 ? ((EPI1 == kSwiglu && !leader) ? &tmW3 : &tmW1) : &tmW2;
        const int brow = s.ex[t.u] * p.K;
        const int arow = (int)(t.row0 + BM * rank);
        const int n0 = (g1 && EPI1 == kSwiglu) ? t.nt * (BN / 2) : t.nt * BN + (int)rank * (BN / 2);
        if (!g1) {
          if (!wait_block(fp.done + t.b, dep_target, &s.abort_flag)) {
            ok = false;
            break;
          }
          asm volatile("fence.proxy.async;" ::: "memory");  // the block's rows, stored by other SMs
        }
        const int kblocks = p.K / BK;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_phase<true>(&s.empty[stage], phase ^ 1, &s.abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + stage * (uint32_t)sizeof(uint64_t);
          if (leader) mbar_arrive_expect_tx(&s.full[stage], 2 * (A_BYTES + B_HALF_BYTES));
          tma_load_2d_pair(s.a[stage], mA, fb, kb * BK, arow);
          if (p.b3d) {
            tma_load_3d_pair(s.b[stage], mB, fb, 0, brow + kb * BK, n0 / 64);
          } else {
            tma_load_2d_pair(s.b[stage], mB, fb, n0, brow + kb * BK);
            tma_load_2d_pair(s.b[stage] + B_BOX_BYTES, mB, fb, n0 + 64, brow + kb * BK);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (ok) {
        for (uint32_t st = 0; st < (uint32_t)STAGES; ++st) {
          if (issued > st) {
            const uint32_t last = issued - 1 - ((issued - 1 - st) % STAGES);
            wait_phase<true>(&s.empty[st], (last / STAGES) & 1u, &s.abort_flag);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer (leader)
      constexpr uint32_t idesc = idesc_bf16_f32(BMP, BN, false, true);
      const uint64_t adesc0 = smem_desc_sw128(smem_u32(s.a[0]), 16, 1024);
      const uint64_t bdesc0 = smem_desc_sw128(smem_u32(s.b[0]), B_BOX_BYTES, 1024);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, withheld = false, any_mma = false;
      for (int pos = pair; pos < total && ok; pos += (int)*(volatile long long*)&s.red[1]) {
        const FTile t = decode(s, U, B, N1, N2, D, pos);
        const int kblocks = (t.phase == 1 ? p1.K : p2.K) / BK;
        if (!wait_phase<true>(&s.tempty[acc], acc_phase ^ 1, &s.abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_phase<true>(&s.full[stage], phase, &s.abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = adesc0 + (uint64_t)(stage * (A_BYTES >> 4));
          const uint64_t bd = bdesc0 + (uint64_t)(stage * (B_HALF_BYTES >> 4));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16_pair(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 128), idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit_pair_multicast(&s.empty[stage], 0x3);
          any_mma = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if ((p1.flags & 1) && pair == 0 && !withheld)
          withheld = true;  // self-test: this accumulator is never signalled
        else
          mma_commit_pair_multicast(&s.tfull[acc], 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (any_mma) {
        mma_commit_pair(&s.drain);
        wait_phase<false>(&s.drain, 0, &s.abort_flag, true);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;
    const int slice = (warp - 2) >> 2;
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&s.tempty[0]), 0);
    uint32_t acc = 0, acc_phase = 0;
    for (int pos = pair; pos < total; pos += (int)*(volatile long long*)&s.red[1]) {
      const FTile t = decode(s, U, B, N1, N2, D, pos);
      if (!__all_sync(0xffffffffu, wait_phase<true>(&s.tfull[acc], acc_phase, &s.abort_flag))) break;
      tc_fence_after();
      const bool g1 = t.phase == 1;
      const Params& p = g1 ? p1 : p2;
      const long long myrow0 = t.row0 + BM * rank;
      const long long left = (long long)s.us[t.u + 1] - myrow0;
      const int rows = left <= 0 ? 0 : (left < BM ? (int)left : BM);
      const int wrows = rows - quarter * 32;  // rows of this warp's 32 that belong to the unit
      uint16_t* wbase = p.out + (size_t)(myrow0 + quarter * 32) * p.N_out;
      const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (g1 && EPI1 == kSwiglu) {
        constexpr int W = (BN / 2) / EPI_SLICES;
#pragma unroll 1
        for (int cc = 0; cc < W; cc += 32) {
          const int c = slice * W + cc;
          uint32_t gr[32], ur[32];
          __syncwarp();
          tmem_ld32(tb + c, gr);
          tmem_ld32(tb + BN / 2 + c, ur);
          const int col = t.nt * (BN / 2) + c;
          if (col < p.N_out) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float g = __uint_as_float(gr[i]);
              v[i] = __fdividef(g, 1.0f + __expf(-g)) * __uint_as_float(ur[i]);
            }
            uint32_t pk[16];
            pack32(v, pk);
            store_rows32(s.stg[warp - 2], wbase + col, (size_t)p.N_out, wrows, pk, lane);
          }
        }
      } else {
        constexpr int W = BN / EPI_SLICES;
        const bool gelu = g1 && EPI1 == kGelu;
#pragma unroll 1
        for (int cc = 0; cc < W; cc += 32) {
          const int c = slice * W + cc;
          uint32_t raw[32];
          __syncwarp();
          tmem_ld32(tb + c, raw);
          const int col = t.nt * BN + c;
          if (col < p.N_out) {
            float v[32];
            if (gelu) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = gelu_erf(__uint_as_float(raw[i]));
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]);
            }
            uint32_t pk[16];
            pack32(v, pk);
            store_rows32(s.stg[warp - 2], wbase + col, (size_t)p.N_out, wrows, pk, lane);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&s.tempty[acc]);
        else
          mbar_arrive_cluster(tempty_leader0 + acc * (uint32_t)sizeof(uint64_t));
      }
      if (g1) {
        // the block's intermediate rows of this warp are stored: publish them
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(fp.done + t.b, 1u);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  // ---- teardown (as in the two-launch kernel)
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  const uint32_t peer_abort = ld_shared_cluster_u32(mapa_shared(smem_u32(&s.abort_flag), rank ^ 1u));
  cluster_sync();  // neither CTA exits while the other reads its shared memory
  if (s.abort_flag || peer_abort) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) {
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace ffn3

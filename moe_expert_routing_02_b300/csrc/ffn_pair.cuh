// K6, CTA-pair form: the grouped expert GEMM on pairs of SMs
// (tcgen05.mma.cta_group::2).
//
// Same computation, tile enumeration and epilogues as ffn.cuh (EPS-MoE review,
// "GroupGemm": every expert's GEMM in one persistent kernel), with the MMA
// spread over a cluster of two CTAs:
//   * a pair tile is 256 rows x 256 columns; CTA r of the pair holds rows
//     128r..128r+127 of A and columns 128r..128r+127 of B in its shared
//     memory, and receives all 256 accumulator columns of its 128 rows in its
//     own TMEM.  Each SM therefore streams 32 KB per 64-deep k-block instead
//     of 48 KB, halving the B operand traffic from L2 -- the resource that
//     limits the single-CTA kernel when all 148 SMs run -- and six stages fit
//     in shared memory;
//   * SwiGLU: CTA 0 holds 128 W1 (gate) columns and CTA 1 the same 128 W3 (up)
//     columns, so every CTA's TMEM holds [gate | up] for its rows;
//   * the leader CTA (rank 0) issues the MMAs; its commits are multicast to
//     both CTAs' "stage free" and "accumulator ready" barriers;
//   * both CTAs' TMA loads complete their bytes on the LEADER's "stage full"
//     barrier (the cta_group::2 form of the tensor copy), which the leader's
//     producer arms with the bytes of both CTAs; the peer's epilogue warps
//     arrive remotely on the leader's "accumulator free" barrier;
//   * teardown: each producer waits until the pair's MMAs released its last
//     stages (which implies its copies landed), the MMA thread until its MMAs
//     finished, then a cluster barrier, then the pair-collective TMEM
//     release.  After an abort (bounded wait expired) the CTAs wait a fixed
//     100 us instead, far longer than any copy or arrival takes to land.
// All waits are bounded exactly as in the single-CTA kernel.
#pragma once
#include <cstddef>
#include "ffn.cuh"

namespace ffn2 {

using namespace sm100;
using ffn::gelu_erf;
using ffn::kGelu;
using ffn::kStore;
using ffn::kSwiglu;
using ffn::kWaitBudgetNs;
using ffn::kMaxPolls;
using ffn::Params;
using ffn::pack32;
using ffn::store_rows32;

constexpr int BM = 128;                   // rows per CTA
constexpr int BMP = 2 * BM;               // rows per pair tile
constexpr int BN = 256;                   // MMA N (each CTA holds BN/2 columns of B)
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;  // 8 KB
constexpr int B_HALF_BYTES = (BN / 2) * BK * 2;  // 16 KB: two boxes
constexpr int EPI_WARPS = 16;
constexpr int EPI_SLICES = EPI_WARPS / 4;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr int MAX_G = 512;
constexpr uint32_t TMEM_COLS = 2 * BN;
static_assert(BM == 4 * 32 && BK * 2 == 128, "a gathered A tile is 32 lanes x 4 rows of 128 bytes");

struct Smem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_HALF_BYTES];
  uint64_t full[STAGES];    // leader: both CTAs' copies of the stage landed
  uint64_t empty[STAGES];   // the pair's MMAs finished reading the stage (multicast)
  uint64_t tfull[2];        // accumulator ready (multicast)
  uint64_t tempty[2];       // leader: accumulator drained by both CTAs' epilogues
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  int32_t total_tiles;
  int32_t total_a;           // tiles of the weight-streaming class (ffn::unit_tile_prefix)
  int32_t u_count;
  int32_t goff[MAX_G + 1];   // staged group offsets
  int32_t us[MAX_G + 1];     // unit first rows (ffn::build_units)
  int32_t tstart[MAX_G + 1]; // first tile of the i-th unit in class order
  int32_t mt[MAX_G];
  int32_t ex[MAX_G];         // unit experts
  int32_t ord[MAX_G];        // units in class order
  long long red[8];          // ffn::small_sms scratch
  alignas(128) uint8_t stg[EPI_WARPS][1024];  // per-warp output staging (store_rows32; 16-byte accesses)
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory beyond the 227 KB per-block opt-in limit");
static_assert(offsetof(Smem, stg) % 128 == 0 && offsetof(Smem, b) % 1024 == 0, "staging / stage buffers misaligned");

// Bounded parity wait; CLUSTER selects cluster-scope acquire (the phase was
// completed by the other CTA of the pair).
template <bool CLUSTER>
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint32_t* abort_flag,
                                           bool ignore_abort = false) {
  const uint32_t addr = smem_u32(bar);
  auto poll = [&]() { return CLUSTER ? mbar_try_wait_cluster(addr, parity) : mbar_try_wait(addr, parity); };
  if (poll()) return true;
  const uint64_t t0 = globaltimer_ns();
  volatile uint32_t* ab = abort_flag;
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    if (poll()) return true;
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
  int g, nt;
  long long row0;  // first row of the pair tile
};

// Schedule position -> pair tile (units in class order, ffn::unit_tile_prefix;
// positions spread over the classes by ffn::interleave).
__device__ __forceinline__ Tile decode(const Smem& s, int U, int pos) {
  const int tile = ffn::interleave(pos, s.total_a, s.total_tiles);
  int lo = 0, hi = U;  // tstart[lo] <= tile < tstart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tstart[mid] <= tile) lo = mid; else hi = mid;
  }
  const int u = s.ord[lo];
  Tile t;
  t.g = u;
  const int local = tile - s.tstart[lo];
  const int m = s.mt[u];
  t.nt = local / m;
  t.row0 = (long long)s.us[u] + (long long)(local % m) * BMP;
  return t;
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmB1, const Params p) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem& s = *reinterpret_cast<Smem*>(base);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;

  // ---- units and their tiles (identical in both CTAs of the pair); experts
  // below the small-batch threshold are left to the small-batch kernel
  const int U = ffn::build_units<THREADS>(p, s.goff, s.us, s.ex, &s.u_count);
  // with an SM split (ffn::small_sms) the small-batch experts are left to the
  // small-batch kernels only when they get SMs (S > 0), and the pairs beyond
  // this kernel's (split_ctas - S) / 2 exit
  const int S = ffn::small_sms<THREADS>(p, U, s.us, s.ex, s.red);
  const bool skip_small = p.small_threshold > 0 && S != 0;
  ffn::unit_tile_prefix<THREADS>(p, U, s.us, s.ex, s.mt, s.tstart, &s.total_tiles, BMP,
                                 [&](int rows) { return !skip_small || rows >= p.small_threshold; },
                                 s.ord, &s.total_a);
  __syncthreads();
  const int npairs = (S > 0 && (p.split_ctas - S) / 2 < (int)(gridDim.x >> 1)) ? (p.split_ctas - S) / 2
                                                                                 : (int)(gridDim.x >> 1);
  // no tiles, or a pair beyond this kernel's share (both CTAs of a pair agree):
  // exit before any barrier or TMEM set-up
  if (s.total_tiles == 0 || pair >= npairs) return;
  s.red[1] = npairs;  // read back per tile: the loops below keep no register for it
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
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    if (EPI == kSwiglu) tma_prefetch_desc(&tmB1);
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
  const int total = s.total_tiles;
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    // lane 0 waits, arms (leader) and loads B (and A when stored in row
    // order); a gathered A is copied by all 32 lanes, four rows each
    const bool gather = p.a_src != nullptr;
    uint32_t stage = 0, phase = 0, issued = 0;
    bool ok = true;
    const CUtensorMap* mB = (EPI == kSwiglu && !leader) ? &tmB1 : &tmB0;
    const uint32_t full0 = mapa_shared(smem_u32(&s.full[0]), 0);  // leader's barriers
    for (int tile = pair; tile < total && ok; tile += (int)*(volatile long long*)&s.red[1]) {
      const Tile t = decode(s, U, tile);
      const int brow = s.ex[t.g] * p.K;
      const int arow = (int)(t.row0 + BM * rank);
      const int n0 = (EPI == kSwiglu) ? t.nt * (BN / 2) : t.nt * BN + (int)rank * (BN / 2);
      const int4 src = gather ? ffn::gather_src4(p, t.row0 + BM * rank, lane) : make_int4(0, 0, 0, 0);
      for (int kb = 0; kb < kblocks; ++kb) {
        bool w = true;
        if (lane == 0) w = wait_phase<true>(&s.empty[stage], phase ^ 1, &s.abort_flag);
        if (!__shfl_sync(0xffffffffu, (int)w, 0)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + stage * (uint32_t)sizeof(uint64_t);
        if (lane == 0) {
          if (leader) mbar_arrive_expect_tx(&s.full[stage], 2 * (A_BYTES + B_HALF_BYTES));
          if (!gather) tma_load_2d_pair(s.a[stage], &tmA, fb, kb * BK, arow);
          if (p.b3d) {
            tma_load_3d_pair(s.b[stage], mB, fb, 0, brow + kb * BK, n0 / 64);
          } else {
            tma_load_2d_pair(s.b[stage], mB, fb, n0, brow + kb * BK);
            tma_load_2d_pair(s.b[stage] + B_BOX_BYTES, mB, fb, n0 + 64, brow + kb * BK);
          }
        }
        __syncwarp();
        if (gather) tma_gather4_pair(s.a[stage] + lane * 512, &tmA, fb, kb * BK, src);
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // normal path: the pair's MMAs released every stage this CTA filled, so
    // its copies landed and no commit arrival is still travelling here
    if (ok && lane == 0) {
      for (uint32_t st = 0; st < (uint32_t)STAGES; ++st) {
        if (issued > st) {
          const uint32_t last = issued - 1 - ((issued - 1 - st) % STAGES);
          wait_phase<true>(&s.empty[st], (last / STAGES) & 1u, &s.abort_flag);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer (leader)
      constexpr uint32_t idesc = idesc_bf16_f32(BMP, BN, false, true);
      // stage-0 descriptors; stage s adds s * (stage bytes >> 4) to the
      // start-address field, a K step of 16 adds 2 (A, 32 B) or 128 (B, 2048 B)
      const uint64_t adesc0 = smem_desc_sw128(smem_u32(s.a[0]), 16, 1024);
      const uint64_t bdesc0 = smem_desc_sw128(smem_u32(s.b[0]), B_BOX_BYTES, 1024);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, withheld = false, any_mma = false;
      for (int tile = pair; tile < total && ok; tile += (int)*(volatile long long*)&s.red[1]) {
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
        if ((p.flags & 1) && pair == 0 && !withheld)
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
    for (int tile = pair; tile < total; tile += (int)*(volatile long long*)&s.red[1]) {
      const Tile t = decode(s, U, tile);
      if (!__all_sync(0xffffffffu, wait_phase<true>(&s.tfull[acc], acc_phase, &s.abort_flag))) break;
      tc_fence_after();
      const long long myrow0 = t.row0 + BM * rank;
      const long long left = (long long)s.us[t.g + 1] - myrow0;
      const int rows = left <= 0 ? 0 : (left < BM ? (int)left : BM);
      const int wrows = rows - quarter * 32;  // rows of this warp's 32 that belong to the group
      uint16_t* wbase = p.out + (size_t)(myrow0 + quarter * 32) * p.N_out;
      const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (EPI == ffn::kCombine) {
        constexpr int W = BN / EPI_SLICES;
        float wt;
        float* arow = ffn::comb_target(p, myrow0 + quarter * 32 + lane, myrow0 + rows, wt);
#pragma unroll 1
        for (int cc = 0; cc < W; cc += 32) {
          const int c = slice * W + cc;
          uint32_t raw[32];
          __syncwarp();
          tmem_ld32(tb + c, raw);
          const int col = t.nt * BN + c;
          if (col < p.N_out && arow) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]);
            ffn::red_add32(arow + col, v, wt);
          }
        }
      } else if (EPI == kSwiglu) {
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
#pragma unroll 1
        for (int cc = 0; cc < W; cc += 32) {
          const int c = slice * W + cc;
          uint32_t raw[32];
          __syncwarp();
          tmem_ld32(tb + c, raw);
          const int col = t.nt * BN + c;
          if (col < p.N_out) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float z = __uint_as_float(raw[i]);
              v[i] = (EPI == kGelu) ? gelu_erf(z) : z;
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
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  const uint32_t peer_abort = ld_shared_cluster_u32(mapa_shared(smem_u32(&s.abort_flag), rank ^ 1u));
  cluster_sync();  // neither CTA exits while the other reads its shared memory
  if (s.abort_flag || peer_abort) {
    // an aborted pair may still have arrivals in flight: give them time to land
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

}  // namespace ffn2

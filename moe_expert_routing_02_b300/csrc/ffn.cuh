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
// The same kernel serves the backward pass (ffn_backward.cu): dgrad GEMMs
// with the weights as a K-major B operand (kStoreKM), GEMM1 recomputed with
// an epilogue that writes the activation and its derivative factors
// (kBwdGelu, kBwdSwiglu), and dA = dY W2^T multiplied by those factors in its
// epilogue (kStoreKMMul, kStoreKMMul2); see the Epi modes below.
//
// Rows are grouped by expert (or replica group); group sizes live only on the
// device, so every CTA reads the group offsets, folds adjacent groups of the
// same expert into one row range ("unit", build_units) and enumerates the
// tiles (unit, n-tile, m-tile) itself, m fastest so that CTAs running at the
// same time share the expert's weight tile in L2.  CTA c takes tiles c,
// c+grid, ...  Experts below the small-batch threshold are left to
// ffn_small.cuh.
//
// Per CTA (one per SM, 576 threads):
//   warp 0      TMA producer: A tile 128x64 (K-major) and B tile 64x256
//               (weights as stored, N contiguous = MN-major), 128-byte
//               swizzle, into a 4-stage ring guarded by full/empty mbarriers.
//   warp 1      TMEM allocator and MMA issuer: one thread issues
//               tcgen05.mma (M=128, N=256, K=16, bf16 in, fp32 accumulate in
//               TMEM) and tcgen05.commit frees each smem stage; two TMEM
//               accumulators (2 x 256 columns) let the epilogue of one tile
//               overlap the main loop of the next.
//   warps 2..17 epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4).., a quarter of the columns each), activation
//               in fp32, bf16 rounding, row-masked stores (rows past the
//               group's end belong to another group and are not written).
//               Four warps per SM sub-partition keep the issue slots busy:
//               GeLU's epilogue costs about as many instructions per tile as
//               the main loop has cycles when H = 1024.
// For SwiGLU the B tile holds 128 columns of W1 then the same 128 columns of
// W3, so one N=256 MMA yields gate and up side by side in TMEM.
//
// Every mbarrier wait is bounded (2 s of %globaltimer): on expiry the
// waiting role raises the CTA's abort flag and the device timeout bit, the
// other roles leave their loops at their next wait, the producer waits for
// the copies it issued, the MMA thread for its MMAs, and TMEM is freed before
// the CTA exits.
#pragma once
#include <climits>
#include <cstddef>
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace ffn {

using namespace sm100;

#ifndef MOE_FFN_BN
#define MOE_FFN_BN 256
#endif
#ifndef MOE_FFN_STAGES
#define MOE_FFN_STAGES 4
#endif
#ifndef MOE_FFN_EPI_WARPS
#define MOE_FFN_EPI_WARPS 16
#endif
constexpr int BM = 128;
constexpr int BN = MOE_FFN_BN;          // MMA N: 256 (or 128)
constexpr int BK = 64;
constexpr int STAGES = MOE_FFN_STAGES;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;  // 8 KB: 64 columns x 64 k-rows
constexpr int B_BYTES = BN * BK * 2;      // 32 KB
constexpr int EPI_WARPS = MOE_FFN_EPI_WARPS;
constexpr int B_BOXES = BN / 64;       // 64-column TMA boxes per B stage
static_assert(BN % 128 == 0 && BN <= 256, "BN must be 128 or 256");
static_assert(BM == 4 * 32 && BK * 2 == 128, "a gathered A tile is 32 lanes x 4 rows of 128 bytes");
constexpr int EPI_SLICES = EPI_WARPS / 4;  // column slices per TMEM lane quarter
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr int MAX_G = 512;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint64_t kWaitBudgetNs = 2000000000ull;
constexpr uint32_t kMaxPolls = 1u << 30;

// kGelu / kSwiglu / kStore: forward GEMM1 and GEMM2 (B = weights as stored,
// MN-major).  kStoreKM: data gradient, B = the transpose of the weights as
// stored (K-major rows of the weight tensor), K optionally split between two
// weight tensors at k_split blocks.  kBwdGelu / kBwdSwiglu: GEMM1 recomputed in
// the backward pass; the epilogue writes the activation (out) and the factors
// that turn dA into the pre-activation gradients (out2): gelu'(z), or
// [u silu'(g) | silu(g)] for SwiGLU.  kStoreKMMul: dA = dY W2^T (K-major B);
// the epilogue multiplies dA by those factors in place (out), giving dz;
// kStoreKMMul2 likewise with the SwiGLU pair of factors, giving [dg | du].
// kCombine: GEMM2 with the combine in its epilogue: row i's result, times
// its gate weight w[perm[i]], is added (fp32 reductions) into row
// perm[i] / k of an fp32 [T, N_out] accumulator instead of being stored.
enum Epi : int {
  kGelu = 0, kSwiglu = 1, kStore = 2, kStoreKM = 3, kBwdGelu = 4, kBwdSwiglu = 5, kStoreKMMul = 6, kStoreKMMul2 = 7,
  kCombine = 8
};

__host__ __device__ constexpr bool epi_pair_b(int e) { return e == kSwiglu || e == kBwdSwiglu; }
__host__ __device__ constexpr bool epi_kmajor_b(int e) { return e == kStoreKM || e == kStoreKMMul || e == kStoreKMMul2; }

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
  const int32_t* rep_base;  // [E+1] or null: groups of expert e are rep_base[e]..rep_base[e+1]-1
  int small_threshold;      // experts with fewer rows take the small-batch kernel (0 = none)
  int b3d;                  // the MN-major weight maps are 3-D (64, rows, N/64): one load per stage and matrix
  // Gathered A operand (GEMM1 only): row i of A is row a_src[i] / a_src_div
  // of the tensor behind tmA (a token of x, a_src = the dispatch permutation,
  // a_src_div = k); null = A is stored in row order.
  const int32_t* a_src;
  int a_src_div;
  int a_src_rows;  // rows of that tensor (T)
  // kStoreKM: k-blocks below k_split read the first weight tensor, the rest
  // the second (at k-block kb - k_split).  kStoreKMMul / kStoreKMMul2: K/BK
  // (kStoreKMMul passes the factor tensor, 16-column x 32-row boxes, as the
  // second tensor map).
  int k_split;
  // kBwdGelu / kBwdSwiglu: out = activation [A_rows, N_out]; out2 = the
  // factors, [A_rows, N_out] (GeLU) or [A_rows, 2 N_out] (SwiGLU).
  // kStoreKMMul / kStoreKMMul2: out = those factors, overwritten with the
  // products.
  uint16_t* out2;
  // kCombine: the dispatch permutation, the gate weights [T*k], k and the
  // fp32 accumulator [T, N_out] (zero before the call)
  const int32_t* comb_perm;
  const float* comb_w;
  int comb_k;
  float* comb_acc;
  // SM split between the small-batch kernels and the grouped kernels of one
  // forward FFN call (small_sms below).  split_ctas = 0: no split -- the
  // grouped kernels skip the experts below small_threshold and the
  // small-batch kernels take them with their whole grid.  Otherwise every
  // kernel of the call gets the same values: split_ctas = the SMs they share,
  // split_force = -1 (the model decides) or the small-batch kernels' SMs
  // (0 = no small-batch path), split_pair = the grouped kernel runs CTA
  // pairs, split_rows = rows per grouped tile, ffn_H / ffn_F / ffn_mats = the
  // whole FFN's shape and weight matrices per expert (2 GeLU, 3 SwiGLU).
  int split_ctas;
  int split_force;
  int split_pair;
  int split_rows;
  int ffn_H, ffn_F, ffn_mats;
};

// Rates of the split model (per SM unless stated): the small-batch kernel
// streams about kSplitSmallBytesPerNs bytes of weights per ns on one SM
// (measured on B300: 59-63 GB/s per SM with 8 to 48 SMs given to it on the
// DeepSeekV2-shaped layer; about 200 KB of stages in flight against the HBM
// latency under load); the grouped kernel executes about kSplitGroupFlopPerNs
// padded-tile flops per ns on one SM; HBM moves about kSplitHbmBytesPerNs
// bytes per ns in all.
#ifndef MOE_SPLIT_SMALL_BPNS
#define MOE_SPLIT_SMALL_BPNS 60
#endif
#ifndef MOE_SPLIT_GROUP_FPNS
#define MOE_SPLIT_GROUP_FPNS 8000
#endif
constexpr long long kSplitSmallBytesPerNs = MOE_SPLIT_SMALL_BPNS;
constexpr long long kSplitGroupFlopPerNs = MOE_SPLIT_GROUP_FPNS;
constexpr long long kSplitHbmBytesPerNs = 6000;

// The SMs that the small-batch kernels of this FFN call take (0: no
// small-batch path this call; the grouped kernels then take every expert).
// A two-resource model (the small-batch kernel is a weight stream, bound by
// HBM; the grouped kernel's large experts are bound by the tensor pipe):
// with S SMs for the small-batch experts and the rest for the grouped ones,
//   t(S) = max(small weights / min(S rate, HBM), grouped flops / ((N-S) rate),
//              all weights / HBM),
// against t(0) = the grouped kernels alone on every SM, the small experts as
// padded tiles, which a split must beat by 1/8.  The first term falls and the
// second rises with S, so the
// best S sits where they cross, S* = N Ws Rt / (Ws Rt + Fg Rs), capped where
// the small-batch kernel alone would saturate HBM; the lanes of warp 0 score
// the split sizes next to it and t(0), and the smallest t wins (the smaller
// S on ties).  Only from the unit table and the call's parameters, with
// integer sums and explicitly rounded fp32 operations, so every kernel of the
// call computes the same S.  Call from all NT threads
// after build_units; `red` is shared scratch of 8 long longs.
template <int NT>
__device__ int small_sms(const Params& p, int U, const int32_t* us, const int32_t* ue, long long* red) {
  if (p.split_ctas <= 0 || p.small_threshold <= 0) {
    __syncthreads();
    return -1;  // no split: legacy behaviour
  }
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    long long small_chunks = 0, small_units = 0, small_pad = 0, grp_pad = 0, grp_units = 0;
    const long long gr = p.split_rows;
    for (int c0 = 0; c0 < U; c0 += 32) {
      const int u = c0 + lane;
      long long sc = 0, su = 0, sp = 0, gp = 0, gu = 0;
      if (u < U) {
        const long long rows = us[u + 1] - us[u];
        if (rows > 0 && ue[u] >= 0) {
          if (rows < p.small_threshold) {
            sc = (rows + 63) / 64;
            su = 1;
            sp = (rows + gr - 1) / gr * gr;
          } else {
            gp = (rows + gr - 1) / gr * gr;
            gu = 1;
          }
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        sc += __shfl_xor_sync(0xffffffffu, sc, off);
        su += __shfl_xor_sync(0xffffffffu, su, off);
        sp += __shfl_xor_sync(0xffffffffu, sp, off);
        gp += __shfl_xor_sync(0xffffffffu, gp, off);
        gu += __shfl_xor_sync(0xffffffffu, gu, off);
      }
      small_chunks += sc;
      small_units += su;
      small_pad += sp;
      grp_pad += gp;
      grp_units += gu;
    }
    const long long N = p.split_ctas, step = p.split_pair ? 2 : 1;
    long long S = 0;
    if (small_units > 0 && p.split_force > 0) {
      S = p.split_force;
    } else if (small_units > 0 && p.split_force < 0) {
      // times in ns as fp32 with explicitly rounded operations (never
      // contracted), so every kernel reaches the same S; a wrong S only costs
      // time, never a result
      const float wb = __fmul_rn(__fmul_rn((float)p.ffn_mats, (float)p.ffn_H), __fmul_rn((float)p.ffn_F, 2.f));
      const float fl = wb;  // flops per row = 2 * mats * H * F = the weight bytes of an expert
      const float Ws = __fmul_rn((float)small_chunks, wb), Bs = __fmul_rn((float)small_units, wb);
      const float Bg = __fmul_rn((float)grp_units, wb);
      const float Fg = __fmul_rn((float)grp_pad, fl), F0 = __fmul_rn((float)(grp_pad + small_pad), fl);
      const float rs1 = (float)kSplitSmallBytesPerNs, rt1 = (float)kSplitGroupFlopPerNs;
      const float bw = (float)kSplitHbmBytesPerNs, Nf = (float)N;
      const long long hi = N - step;
      long long cap = kSplitHbmBytesPerNs / kSplitSmallBytesPerNs;
      if (cap > hi) cap = hi;
      // crossing of the small-batch and grouped times: S* = N Ws Rt / (Ws Rt + Fg Rs)
      const float a = __fmul_rn(Ws, rt1);
      const float xf = __fdiv_rn(__fmul_rn(Nf, a), __fadd_rn(a, __fmul_rn(Fg, rs1)));
      long long xs = (long long)xf;  // truncation toward zero of a non-negative value
      if (xs > cap) xs = cap;
      long long cand = (xs / step + (lane - 4)) * step;  // lanes 1..8: -3 .. +4 steps around it
      float t = __int_as_float(0x7f800000);            // +inf
      if (lane == 0) {
        // a split must beat the grouped-only time by 1/8: giving SMs away
        // also costs what the model leaves out (measured: 2 SMs taken from
        // the fused CTA-pair kernel on the moe_gpt_stream layer cost 8%, as the
        // small-batch CTAs break up SM pairs the clusters need)
        cand = 0;
        t = __fmul_rn(fmaxf(__fdiv_rn(F0, __fmul_rn(Nf, rt1)), __fdiv_rn(__fadd_rn(Bs, Bg), bw)), 0.875f);
      } else if (lane <= 8 && cand >= step && cand <= hi) {
        const float rs = fminf(__fmul_rn((float)cand, rs1), bw);
        t = __fdiv_rn(Ws, rs);
        if (grp_units) t = fmaxf(t, __fdiv_rn(Fg, __fmul_rn((float)(N - cand), rt1)));
        t = fmaxf(t, __fdiv_rn(__fadd_rn(Ws, Bg), bw));
      }
      // the smallest (t, S) over the warp
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const float ot = __shfl_xor_sync(0xffffffffu, t, off);
        const long long oc = __shfl_xor_sync(0xffffffffu, cand, off);
        if (ot < t || (ot == t && oc < cand)) {
          t = ot;
          cand = oc;
        }
      }
      S = cand;
    }
    if (S > N - step) S = N - step;
    if (S < 0) S = 0;
    if (step == 2) S &= ~1LL;
    if (lane == 0) red[0] = S;
  }
  __syncthreads();
  return (int)red[0];
}

// acc[t, c .. c+31] += wt * v[0 .. 31] with vector fp32 reductions (8 per
// row segment).  For k = 2 every accumulator element receives exactly two
// additions onto zero, so the result does not depend on their order.
__device__ __forceinline__ void red_add32(float* dst, const float (&v)[32], float wt) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * j),
                 "f"(wt * v[4 * j]), "f"(wt * v[4 * j + 1]), "f"(wt * v[4 * j + 2]), "f"(wt * v[4 * j + 3])
                 : "memory");
}

// Token row and gate weight of dispatched row `row` (kCombine); a row
// outside [0, rows) or an invalid permutation entry gives wt = 0 and
// acc_row = null (flagged).
__device__ __forceinline__ float* comb_target(const Params& p, long long row, long long rows_valid_end, float& wt) {
  wt = 0.f;
  if (row >= rows_valid_end) return nullptr;
  const int f = __ldg(p.comb_perm + row);
  if (f < 0 || (long long)f >= p.A_rows) {
    moe_flag_error(MOE_DEVERR_DATA);
    return nullptr;
  }
  wt = __ldg(p.comb_w + f);
  return p.comb_acc + (size_t)(f / p.comb_k) * p.N_out;
}


struct Smem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t fbar[EPI_WARPS][3];  // kStoreKMMul: per-warp factor buffers
  uint32_t tmem_base;
  uint32_t abort_flag;
  int32_t total_tiles;
  int32_t total_a;           // tiles of the weight-streaming class (unit_tile_prefix)
  int32_t u_count;
  int32_t goff[MAX_G + 1];   // staged group offsets
  int32_t us[MAX_G + 1];     // unit first rows (build_units)
  int32_t tstart[MAX_G + 1]; // first tile of the i-th unit in class order
  int32_t mt[MAX_G];
  int32_t ex[MAX_G];         // unit experts
  int32_t ord[MAX_G];        // units in class order
  long long red[8];          // small_sms scratch
  alignas(128) uint8_t stg[EPI_WARPS][1024];  // per-warp output staging (store_rows32; 16-byte accesses)
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory beyond the 227 KB per-block opt-in limit");
static_assert(offsetof(Smem, stg) % 128 == 0 && offsetof(Smem, b) % 1024 == 0, "staging / stage buffers misaligned");

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

// Group table -> "units": maximal runs of consecutive groups that serve the
// same expert.  The replica groups of an expert are adjacent in the dispatched
// layout and alias that expert's weights, so a unit is tiled as one row range:
// every row's result is the same as when its replica group is tiled alone
// (same weights, same K order), without a partial tile per replica.  A unit's
// rows are the expert's total rows, so the kernel path chosen from them is
// the same for all replicas of an expert.
//   us[u] first row of unit u, us[U] = end of the last unit; ue[u] its expert
//   (-1: no valid expert; such a unit gets no tiles).  Offsets are clamped to
//   [0, A_rows]; decreasing or out-of-range offsets and unknown experts are
//   flagged as invalid data.  Call from all NT threads; returns U.
template <int NT>
__device__ int build_units(const Params& p, int32_t* goff, int32_t* us, int32_t* ue, int32_t* u_count) {
  const int G = p.G;
  const int lane = threadIdx.x & 31;
  for (int g = threadIdx.x; g <= G; g += NT) {
    long long v = p.group_offsets[g];
    if (v < 0 || v > p.A_rows) {
      moe_flag_error(MOE_DEVERR_DATA);
      v = v < 0 ? 0 : p.A_rows;
    }
    goff[g] = (int32_t)v;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    int carry = 0, prev_e = INT_MIN;
    for (int c0 = 0; c0 < G; c0 += 32) {
      const int g = c0 + lane;
      int e = INT_MIN;
      if (g < G) e = p.group_expert ? p.group_expert[g] : g;
      int pe = __shfl_up_sync(0xffffffffu, e, 1);
      if (lane == 0) pe = prev_e;
      const bool start = g < G && (g == 0 || e != pe);
      const unsigned starts = __ballot_sync(0xffffffffu, start);
      const int u = carry + __popc(starts & ((1u << lane) - 1u));
      if (start) {
        us[u] = goff[g];
        ue[u] = e;
      }
      if (g < G && goff[g + 1] < goff[g]) moe_flag_error(MOE_DEVERR_DATA);
      carry += __popc(starts);
      prev_e = __shfl_sync(0xffffffffu, e, 31);
    }
    if (lane == 0) {
      us[carry] = goff[G];
      *u_count = carry;
    }
  }
  __syncthreads();
  const int U = *u_count;
  for (int u = threadIdx.x; u < U; u += NT) {
    const int rows = us[u + 1] - us[u];
    if (rows > 0 && (ue[u] < 0 || ue[u] >= p.E)) {
      moe_flag_error(MOE_DEVERR_DATA);
      ue[u] = -1;
    }
  }
  __syncthreads();
  return U;
}

// Tiles of each unit and their prefix (warp 0): tiles_u = ceil(rows_u / tile_rows)
// * n_tiles for units the caller's filter keeps (keep(rows) -> bool), else 0.
// Without `ord`, tstart[u] is unit u's first tile (units in row order).  With
// `ord`, the units are taken in class order -- first those of one row tile
// (mt == 1: each weight tile serves one row tile, so they stream weights and
// are bound by HBM), then the others (bound by the tensor pipe) -- ord[i] is
// the i-th unit of that order, tstart[i] its first tile and *total_a the
// tiles of the first class; interleave() then spreads the two classes over
// the schedule.
template <int NT, typename Keep>
__device__ void unit_tile_prefix(const Params& p, int U, const int32_t* us, const int32_t* ue, int32_t* mt,
                                 int32_t* tstart, int32_t* total, int tile_rows, Keep keep,
                                 int32_t* ord = nullptr, int32_t* total_a = nullptr) {
  const int lane = threadIdx.x & 31;
  for (int u = threadIdx.x; u < U; u += NT) {
    const int rows = us[u + 1] - us[u];
    mt[u] = (rows > 0 && ue[u] >= 0 && keep(rows)) ? (rows + tile_rows - 1) / tile_rows : 0;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    int carry = 0, pos = 0;
    for (int cls = 0; cls < (ord ? 2 : 1); ++cls) {
      for (int c0 = 0; c0 < U; c0 += 32) {
        const int u = c0 + lane;
        const bool in = u < U && (!ord || ((mt[u] == 1) == (cls == 0)));
        const unsigned m = __ballot_sync(0xffffffffu, in);
        const int v = in ? mt[u] * p.n_tiles : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int w = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += w;
        }
        const int i = pos + __popc(m & ((1u << lane) - 1u));
        if (in) {
          tstart[i] = carry + incl - v;
          if (ord) ord[i] = u;
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
        pos += __popc(m);
      }
      if (cls == 0 && total_a && lane == 0) *total_a = carry;
    }
    if (lane == 0) {
      tstart[U] = carry;
      *total = carry;
    }
  }
}

// Schedule position -> tile index in class order: the first-class tiles
// [0, ta) are spread evenly over the positions (position q is one of them iff
// floor((q + 1) ta / total) > floor(q ta / total)), the rest keep their order,
// so every round of the persistent grid mixes weight-streaming tiles with
// tensor-bound ones in the proportion of their totals.  A bijection on
// [0, total); the identity when ta is 0 or total.
__device__ __forceinline__ int interleave(int q, int ta, int total) {
  if (ta <= 0 || ta >= total) return q;
  const int a0 = (int)((long long)q * ta / total);
  const int a1 = (int)((long long)(q + 1) * ta / total);
  return a1 > a0 ? a0 : ta + (q - a0);
}

struct Tile {
  int g, nt, rows;
  long long row0;
};

// Schedule position -> tile (units in class order, see unit_tile_prefix).
__device__ __forceinline__ Tile decode(const Smem& s, int U, int pos) {
  const int tile = interleave(pos, s.total_a, s.total_tiles);
  int lo = 0, hi = U;  // tstart[lo] <= tile < tstart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tstart[mid] <= tile) lo = mid; else hi = mid;
  }
  const int u = s.ord[lo];
  Tile t;
  t.g = u;  // unit
  const int local = tile - s.tstart[lo];
  const int m = s.mt[u];
  t.nt = local / m;
  t.row0 = (long long)s.us[u] + (long long)(local % m) * BM;
  const long long left = (long long)s.us[u + 1] - t.row0;
  t.rows = left < BM ? (int)left : BM;
  return t;
}

// Source rows of A rows row0 + 4*q .. row0 + 4*q + 3 (gathered A operand).
// Rows past the operand's end read row 0: they fill the ragged tail of the
// last tile, whose results are never stored.  A source outside [0, rows)
// is invalid device data: flagged, and row 0 is read instead.
__device__ __forceinline__ int4 gather_src4(const Params& p, long long row0, int q) {
  int r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const long long row = row0 + 4 * q + j;
    int src = 0;
    if (row < p.A_rows) {
      src = __ldg(p.a_src + row) / p.a_src_div;
      if ((unsigned)src >= (unsigned)p.a_src_rows) {
        moe_flag_error(MOE_DEVERR_DATA);
        src = 0;
      }
    }
    r[j] = src;
  }
  return make_int4(r[0], r[1], r[2], r[3]);
}

// erf by Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26 (Hastings' rational approximation): for x >= 0,
//   erf(x) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-x^2),
//   t = 1 / (1 + p x),  |error| <= 1.5e-7,
// extended to x < 0 by oddness.  In fp32 with the fast reciprocal and
// exponential the error stays near 3e-7, far below the bf16 rounding of the
// output (2^-9 relative).  Two MUFU operations and ten FMA-pipe operations.
__device__ __forceinline__ float erf_as7126(float x) {
  const float ax = fabsf(x);
  const float t = __fdividef(1.0f, fmaf(0.3275911f, ax, 1.0f));
  float q = fmaf(1.061405429f, t, -1.453152027f);
  q = fmaf(q, t, 1.421413741f);
  q = fmaf(q, t, -0.284496736f);
  q = fmaf(q, t, 0.254829592f);
  q *= t;
  const float r = fmaf(-q, __expf(-ax * ax), 1.0f);
  return copysignf(r, x);
}

// Exact-erf GeLU: z * Phi(z) = z/2 * (1 + erf(z / sqrt 2)).
__device__ __forceinline__ float gelu_erf(float z) {
  const float h = 0.5f * z;
  return fmaf(h, erf_as7126(z * 0.70710678118654752f), h);
}

// GeLU and its derivative from one exponential:
//   gelu(z) = z Phi(z),  gelu'(z) = Phi(z) + z phi(z),
//   Phi(z) = (1 + erf(z / sqrt 2)) / 2,  phi(z) = exp(-z^2 / 2) / sqrt(2 pi),
// with erf by the same 7.1.26 approximation, whose exp(-x^2) at x = z/sqrt 2
// is exp(-z^2 / 2).
__device__ __forceinline__ void gelu_and_grad(float z, float& a, float& da) {
  const float x = z * 0.70710678118654752f;
  const float ax = fabsf(x);
  const float t = __fdividef(1.0f, fmaf(0.3275911f, ax, 1.0f));
  float q = fmaf(1.061405429f, t, -1.453152027f);
  q = fmaf(q, t, 1.421413741f);
  q = fmaf(q, t, -0.284496736f);
  q = fmaf(q, t, 0.254829592f);
  q *= t;
  const float ex = __expf(-ax * ax);
  const float erfv = copysignf(fmaf(-q, ex, 1.0f), x);
  const float Phi = fmaf(0.5f, erfv, 0.5f);
  a = z * Phi;
  da = fmaf(z * 0.39894228040143268f, ex, Phi);
}

// gelu_and_grad on a pair (z0, z1), on packed fp32 pairs where the two
// halves share an instruction; the same operations in the same order as the
// scalar form, so each half's results are bit-identical to it.  The erf
// polynomial is evaluated with negated coefficients (each step exactly the
// negation of the scalar step), which gives 1 - q e as one fused step.
__device__ __forceinline__ void gelu_and_grad2(f32x2 z, f32x2& a, f32x2& da) {
  const f32x2 x = f2_mul(z, f2_splat(0.70710678118654752f));
  float x0, x1;
  f2_unpack(x, x0, x1);
  const f32x2 ax = f2_pack(fabsf(x0), fabsf(x1));
  float d0, d1;
  f2_unpack(f2_fma(f2_splat(0.3275911f), ax, f2_splat(1.0f)), d0, d1);
  const f32x2 t = f2_pack(__fdividef(1.0f, d0), __fdividef(1.0f, d1));
  f32x2 nq = f2_fma(f2_splat(-1.061405429f), t, f2_splat(1.453152027f));
  nq = f2_fma(nq, t, f2_splat(-1.421413741f));
  nq = f2_fma(nq, t, f2_splat(0.284496736f));
  nq = f2_fma(nq, t, f2_splat(-0.254829592f));
  nq = f2_mul(nq, t);
  float s0, s1;
  f2_unpack(f2_mul(ax, ax), s0, s1);
  const f32x2 ex = f2_pack(__expf(-s0), __expf(-s1));
  float r0, r1;
  f2_unpack(f2_fma(nq, ex, f2_splat(1.0f)), r0, r1);
  const f32x2 Phi = f2_fma(f2_splat(0.5f), f2_pack(copysignf(r0, x0), copysignf(r1, x1)), f2_splat(0.5f));
  a = f2_mul(z, Phi);
  da = f2_fma(f2_mul(z, f2_splat(0.39894228040143268f)), ex, Phi);
}

// bf16 pair (packed as in pack_bf16x2) -> fp32 pair
__device__ __forceinline__ f32x2 bf16x2_to_f2(uint32_t v) { return f2_pack(bf16lo(v), bf16hi(v)); }

__device__ __forceinline__ uint32_t f2_to_bf16x2(f32x2 v) {
  float lo, hi;
  f2_unpack(v, lo, hi);
  return pack_bf16x2(lo, hi);
}

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

// Write a warp's 32 rows x 32 bf16 columns (lane i holds row i, packed in
// pk) through 1 KB of shared memory, 16 rows at a time, so that each global
// store instruction covers 8 whole 64-byte row segments instead of 32 rows x
// 16 bytes.  In the buffer, 16-byte chunk j of row r sits at slot
// (j + r/2) mod 4 of the row: conflict-free for both the row-wise writes and
// the chunk-wise reads.  Rows >= rows_valid (another group's rows) are not
// written.
__device__ __forceinline__ void store_rows32(uint8_t* stg, uint16_t* out, size_t ld, int rows_valid,
                                             const uint32_t (&pk)[16], int lane) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    __syncwarp();
    if ((lane >> 4) == h) {
      const int r = lane & 15;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(stg + r * 64 + (((j + (r >> 1)) & 3) << 4)) =
            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    }
    __syncwarp();
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int idx = pass * 32 + lane;
      const int r = idx >> 2, c = idx & 3;
      const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 64 + (((c + (r >> 1)) & 3) << 4));
      const int row = h * 16 + r;
      if (row < rows_valid) st_v4(out + (size_t)row * ld + c * 8, v);
    }
  }
}

// The reverse of store_rows32: lane i receives row i's 32 bf16 columns of
// src (packed pairs in pk), read through 1 KB of shared memory with whole
// 64-byte row segments per load instruction.  Rows >= rows_valid read as 0.
__device__ __forceinline__ void load_rows32(uint8_t* stg, const uint16_t* src, size_t ld, int rows_valid,
                                            uint32_t (&pk)[16], int lane) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    __syncwarp();
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int idx = pass * 32 + lane;
      const int r = idx >> 2, c = idx & 3;
      const int row = h * 16 + r;
      const uint4 v = row < rows_valid ? ld_nc_v4(src + (size_t)row * ld + c * 8) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(stg + r * 64 + (((c + (r >> 1)) & 3) << 4)) = v;
    }
    __syncwarp();
    if ((lane >> 4) == h) {
      const int r = lane & 15;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 64 + (((j + (r >> 1)) & 3) << 4));
        pk[4 * j] = v.x;
        pk[4 * j + 1] = v.y;
        pk[4 * j + 2] = v.z;
        pk[4 * j + 3] = v.w;
      }
    }
  }
}

// Coalesced read of a warp's 32 rows x 16 bf16 columns of src (row stride
// ld) into registers: two 16-byte loads per lane, each instruction covering
// 16 whole 32-byte row segments.  Rows >= rows_valid read as 0.
__device__ __forceinline__ void prefetch_rows16(const uint16_t* src, size_t ld, int rows_valid, int lane,
                                                uint4 (&v)[2]) {
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int idx = pass * 32 + lane;
    const int r = idx >> 1, c = idx & 1;
    v[pass] = r < rows_valid ? ld_nc_v4(src + (size_t)r * ld + c * 8) : make_uint4(0, 0, 0, 0);
  }
}

// prefetch_rows16's registers -> lane i holds row i's 16 columns (8 packed
// pairs), through the staging buffer in store_rows16's slot layout.
__device__ __forceinline__ void transpose_rows16(uint8_t* stg, const uint4 (&v)[2], int lane, uint32_t (&dv)[8]) {
  __syncwarp();
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int idx = pass * 32 + lane;
    const int r = idx >> 1, c = idx & 1;
    *reinterpret_cast<uint4*>(stg + r * 32 + (((c + (r >> 2)) & 1) << 4)) = v[pass];
  }
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint4 q = *reinterpret_cast<const uint4*>(stg + lane * 32 + (((j + (lane >> 2)) & 1) << 4));
    dv[4 * j] = q.x;
    dv[4 * j + 1] = q.y;
    dv[4 * j + 2] = q.z;
    dv[4 * j + 3] = q.w;
  }
}

// store_rows32 for 16 columns: lane i holds row i's 16 bf16 columns (8
// packed pairs); through 1 KB of staging, each row's two 16-byte chunks at
// slots (j + r/4) mod 2, so that the writes (8 lanes per phase, rows r and
// r+4 in different slots) and the reads (4 whole 32-byte rows per phase) are
// free of bank conflicts.  Rows >= rows_valid are not written.
__device__ __forceinline__ void store_rows16(uint8_t* stg, uint16_t* out, size_t ld, int rows_valid,
                                             const uint32_t (&pk)[8], int lane) {
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 2; ++j)
    *reinterpret_cast<uint4*>(stg + lane * 32 + (((j + (lane >> 2)) & 1) << 4)) =
        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
  __syncwarp();
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int idx = pass * 32 + lane;
    const int r = idx >> 1, c = idx & 1;
    const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 32 + (((c + (r >> 2)) & 1) << 4));
    if (r < rows_valid) st_v4(out + (size_t)r * ld + c * 8, v);
  }
}

__device__ __forceinline__ void pack32(const float (&v)[32], uint32_t (&pk)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
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
  // ---- units (an expert's adjacent groups), their tiles and prefix; experts
  // below the small-batch threshold are left to the small-batch kernel
  const int U = build_units<THREADS>(p, s.goff, s.us, s.ex, &s.u_count);
  // with an SM split (small_sms) the small-batch experts are left to the
  // small-batch kernels only when they get SMs (S > 0), and this kernel runs
  // on the other split_ctas - S SMs
  const int S = small_sms<THREADS>(p, U, s.us, s.ex, s.red);
  const bool skip_small = p.small_threshold > 0 && S != 0;
  unit_tile_prefix<THREADS>(p, U, s.us, s.ex, s.mt, s.tstart, &s.total_tiles, BM,
                            [&](int rows) { return !skip_small || rows >= p.small_threshold; },
                            s.ord, &s.total_a);
  __syncthreads();
  const int nctas = (S > 0 && p.split_ctas - S < (int)gridDim.x) ? p.split_ctas - S : (int)gridDim.x;
  // no tiles, or a CTA beyond this kernel's share: exit before any barrier or TMEM set-up
  if (s.total_tiles == 0 || (int)blockIdx.x >= nctas) return;
  s.red[1] = nctas;  // read back per tile: the loops below keep no register for it
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int w = 0; w < EPI_WARPS; ++w) {
      for (int b = 0; b < 3; ++b) mbar_init(&s.fbar[w][b], 1);
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
    if (epi_pair_b(EPI) || epi_kmajor_b(EPI)) tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) {
    __syncwarp();  // .sync.aligned: whole warp, converged
    tmem_alloc(&s.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;
  const int total = s.total_tiles;
  const int kblocks = p.K / BK;
  // kStoreKMMul keeps the last stage's buffers for its epilogue's factor
  // tiles (16 warps x three 1 KB buffers: two in the B buffer, one in the A
  // buffer) and runs the operand ring on the rest
  constexpr int NST = EPI == kStoreKMMul ? STAGES - 1 : STAGES;
  static_assert(EPI_WARPS * 2 * 1024 <= B_BYTES && EPI_WARPS * 1024 <= A_BYTES, "factor buffers exceed a stage");

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // lane 0 waits, arms the stage and loads B (and A when stored in row
    // order); a gathered A is copied by all 32 lanes, four rows each
    const bool gather = p.a_src != nullptr;
    uint32_t stage = 0, phase = 0, issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += (int)*(volatile long long*)&s.red[1]) {
      const Tile t = decode(s, U, tile);
      const int brow = epi_kmajor_b(EPI) ? s.ex[t.g] * p.N_out + t.nt * BN : s.ex[t.g] * p.K;
      const int arow = (int)t.row0;
      const int4 src = gather ? gather_src4(p, t.row0, lane) : make_int4(0, 0, 0, 0);
      for (int kb = 0; kb < kblocks; ++kb) {
        bool w = true;
        if (lane == 0) w = wait_phase(&s.empty[stage], phase ^ 1, &s.abort_flag);
        if (!__shfl_sync(0xffffffffu, (int)w, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&s.full[stage], A_BYTES + B_BYTES);
          if (!gather) tma_load_2d(s.a[stage], &tmA, &s.full[stage], kb * BK, arow);
          if (epi_kmajor_b(EPI)) {
            // B = rows n0.. of the expert's [N_out, K] weight block, K-major: one 128 x BN box
            if (kb < p.k_split)
              tma_load_2d(s.b[stage], &tmB0, &s.full[stage], kb * BK, brow);
            else
              tma_load_2d(s.b[stage], &tmB1, &s.full[stage], (kb - p.k_split) * BK, brow);
          } else if (epi_pair_b(EPI)) {
            // first half of the B tile: W1 (gate) columns, second half: the same W3 (up) columns
            const int n0 = t.nt * (BN / 2);
            if (p.b3d) {
              tma_load_3d(s.b[stage], &tmB0, &s.full[stage], 0, brow + kb * BK, n0 / 64);
              tma_load_3d(s.b[stage] + (B_BOXES / 2) * B_BOX_BYTES, &tmB1, &s.full[stage], 0, brow + kb * BK,
                          n0 / 64);
            } else {
#pragma unroll
              for (int c = 0; c < B_BOXES / 2; ++c) {
                tma_load_2d(s.b[stage] + c * B_BOX_BYTES, &tmB0, &s.full[stage], n0 + 64 * c, brow + kb * BK);
                tma_load_2d(s.b[stage] + (c + B_BOXES / 2) * B_BOX_BYTES, &tmB1, &s.full[stage], n0 + 64 * c,
                            brow + kb * BK);
              }
            }
          } else {
            const int n0 = t.nt * BN;
            if (p.b3d) {
              tma_load_3d(s.b[stage], &tmB0, &s.full[stage], 0, brow + kb * BK, n0 / 64);
            } else {
#pragma unroll
              for (int c = 0; c < B_BOXES; ++c)
                tma_load_2d(s.b[stage] + c * B_BOX_BYTES, &tmB0, &s.full[stage], n0 + 64 * c, brow + kb * BK);
            }
          }
        }
        __syncwarp();
        if (gather) tma_gather4(s.a[stage] + lane * 512, &tmA, &s.full[stage], kb * BK, src);
        ++issued;
        if (++stage == NST) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // every stage's latest copy must have landed before the CTA may exit
    if (lane == 0) {
      for (uint32_t st = 0; st < (uint32_t)NST; ++st) {
        if (issued > st) {
          const uint32_t last = issued - 1 - ((issued - 1 - st) % NST);
          wait_phase(&s.full[st], (last / NST) & 1u, &s.abort_flag, true);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr bool kmb = epi_kmajor_b(EPI);
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false, !kmb);
      // B K-major (kStoreKM): BN rows of 128 bytes like the A tile; a K step
      // of 16 is +2 in the start-address field
      constexpr uint32_t kBStep = kmb ? 2u : 128u;
      // descriptors of stage 0; stages are contiguous, so stage s adds
      // s * (stage bytes >> 4) to the start-address field
      const uint64_t adesc0 = smem_desc_sw128(smem_u32(s.a[0]), 16, 1024);
      const uint64_t bdesc0 = smem_desc_sw128(smem_u32(s.b[0]), kmb ? 16u : (uint32_t)B_BOX_BYTES, 1024);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, withheld = false, any_mma = false;
      for (int tile = blockIdx.x; tile < total && ok; tile += (int)*(volatile long long*)&s.red[1]) {
        if (!wait_phase(&s.tempty[acc], acc_phase ^ 1, &s.abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_phase(&s.full[stage], phase, &s.abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // A: K-major, 128-byte rows, 8-row groups 1024 B apart; a K step of 16 is
          //    32 B, i.e. +2 in the descriptor's start-address field (16-B units).
          // B: MN-major, 64-column boxes 8 KB apart (LBO), 8 k-rows 1024 B apart
          //    (SBO); a K step of 16 rows is 2048 B, i.e. +128 in that field.
          const uint64_t ad = adesc0 + (uint64_t)(stage * (A_BYTES >> 4));
          const uint64_t bd = bdesc0 + (uint64_t)(stage * (B_BYTES >> 4));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * kBStep), idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit(&s.empty[stage]);
          any_mma = true;
          if (++stage == NST) {
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
    const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
    const int slice = (warp - 2) >> 2;         // column slice 0..EPI_SLICES-1
    uint32_t acc = 0, acc_phase = 0;
    // kStoreKMMul: this warp's two factor buffers, their next phases and
    // whether a copy into them is outstanding
    uint8_t* fb3[3] = {s.b[STAGES - 1] + (warp - 2) * 2048, s.b[STAGES - 1] + (warp - 2) * 2048 + 1024,
                       s.a[STAGES - 1] + (warp - 2) * 1024};
    uint32_t fph[3] = {0u, 0u, 0u};
    bool fpend[3] = {false, false, false};
    for (int tile = blockIdx.x; tile < total; tile += (int)*(volatile long long*)&s.red[1]) {
      const Tile t = decode(s, U, tile);
      // Multiply epilogues: the factor rows of the warp's 64 columns are
      // requested before the accumulator wait.  kStoreKMMul: two 32x16 TMA
      // boxes into the warp's factor buffers (pieces 2, 3 follow as 0, 1 are
      // read); kStoreKMMul2 (SwiGLU, two factors): plain loads, the first
      // factor's whole slice ahead and the second one piece ahead.
      constexpr bool kMul = EPI == kStoreKMMul || EPI == kStoreKMMul2;
      constexpr bool kPair = EPI == kStoreKMMul2;
      constexpr int kMulW = BN / EPI_SLICES;
      constexpr int kMulNP = kMulW / 16;
      const int mcol0 = t.nt * BN + slice * kMulW;
      const size_t mld = (kPair ? 2 : 1) * (size_t)p.N_out;
      const int mrow = (int)t.row0 + quarter * 32;
      uint16_t* mbase = kMul ? p.out + (size_t)mrow * mld : nullptr;
      uint4 pre[kPair ? kMulNP : 1][2];
      uint4 preu[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
      if (EPI == kStoreKMMul) {
        // pieces 0, 1, 2 into buffers 0, 1, 2; piece 3 follows into buffer 0
#pragma unroll
        if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // last tile's reads first
        for (int q = 0; q < 3; ++q) {
          if (q < kMulNP && mcol0 + 16 * q < p.N_out) {
            if (lane == 0) {
              mbar_arrive_expect_tx(&s.fbar[warp - 2][q], 1024);
              tma_load_2d(fb3[q], &tmB1, &s.fbar[warp - 2][q], mcol0 + 16 * q, mrow);
            }
            fpend[q] = true;
          }
        }
      } else if (kPair) {
#pragma unroll
        for (int pc = 0; pc < kMulNP; ++pc) {
          pre[pc][0] = pre[pc][1] = make_uint4(0, 0, 0, 0);
          if (mcol0 + 16 * pc < p.N_out)
            prefetch_rows16(mbase + mcol0 + 16 * pc, mld, t.rows - quarter * 32, lane, pre[pc]);
        }
        if (mcol0 < p.N_out) prefetch_rows16(mbase + p.N_out + mcol0, mld, t.rows - quarter * 32, lane, preu);
      }
      // every lane waits; the vote keeps the warp converged for tcgen05.ld
      if (!__all_sync(0xffffffffu, wait_phase(&s.tfull[acc], acc_phase, &s.abort_flag))) break;
      tc_fence_after();
      // this warp's 32 rows: tile rows quarter*32 .. +31, of which wrows are the group's
      const int wrows = t.rows - quarter * 32;
      uint16_t* wbase = p.out + (size_t)(t.row0 + quarter * 32) * p.N_out;
      const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (EPI == kStoreKMMul) {
        // dz = dA * gelu'(z) over the factors in place; 16-column pieces,
        // factor pieces from the TMA buffers, the next piece's TMEM load
        // issued before this piece's stores
        constexpr int NP = kMulNP;
        bool ok = true;
        uint32_t raw[16];
        __syncwarp();
        if (mcol0 < p.N_out) {
          tmem_ld16_issue(tb + slice * kMulW, raw);
          tmem_wait16(raw);
        }
#pragma unroll
        for (int pc = 0; pc < NP; ++pc) {
          const int col = mcol0 + pc * 16;
          if (col >= p.N_out) break;  // warp-uniform; later pieces lie further right
          const int b = pc % 3;
          if (!__all_sync(0xffffffffu, wait_phase(&s.fbar[warp - 2][b], fph[b], &s.abort_flag))) {
            ok = false;
            break;
          }
          fph[b] ^= 1u;
          fpend[b] = false;
          const uint4 q0 = *reinterpret_cast<const uint4*>(fb3[b] + lane * 32);
          const uint4 q1 = *reinterpret_cast<const uint4*>(fb3[b] + lane * 32 + 16);
          const uint32_t fv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
          __syncwarp();
          if (pc + 3 < NP && col + 48 < p.N_out) {
            if (lane == 0) {
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // reads above, then the copy
              mbar_arrive_expect_tx(&s.fbar[warp - 2][b], 1024);
              tma_load_2d(fb3[b], &tmB1, &s.fbar[warp - 2][b], col + 48, mrow);
            }
            fpend[b] = true;
          }
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o[i] = f2_to_bf16x2(f2_mul(f2_pack(__uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1])),
                                       bf16x2_to_f2(fv[i])));
          const bool next = pc + 1 < NP && col + 16 < p.N_out;  // warp-uniform
          if (next) tmem_ld16_issue(tb + slice * kMulW + (pc + 1) * 16, raw);
          store_rows16(s.stg[warp - 2], mbase + col, mld, wrows, o, lane);
          if (next) tmem_wait16(raw);
        }
        if (!ok) break;
      } else if (kPair) {
        // dg = dA * u silu'(g), du = dA * silu(g) over the factors in place
        constexpr int NP = kMulNP;
#pragma unroll
        for (int pc = 0; pc < NP; ++pc) {
          const int col = mcol0 + pc * 16;
          if (col >= p.N_out) break;  // warp-uniform
          uint32_t fv[8], fu[8];
          transpose_rows16(s.stg[warp - 2], pre[pc], lane, fv);
          transpose_rows16(s.stg[warp - 2], preu, lane, fu);
          if (pc + 1 < NP && col + 16 < p.N_out)
            prefetch_rows16(mbase + p.N_out + col + 16, mld, wrows, lane, preu);
          __syncwarp();
          uint32_t raw[16];
          tmem_ld16(tb + slice * kMulW + pc * 16, raw);
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o[i] = f2_to_bf16x2(f2_mul(f2_pack(__uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1])),
                                       bf16x2_to_f2(fv[i])));
          store_rows16(s.stg[warp - 2], mbase + col, mld, wrows, o, lane);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o[i] = f2_to_bf16x2(f2_mul(f2_pack(__uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1])),
                                       bf16x2_to_f2(fu[i])));
          store_rows16(s.stg[warp - 2], mbase + p.N_out + col, mld, wrows, o, lane);
        }
      } else if (EPI == kBwdGelu) {
        // 16-column pieces: a = gelu(z) and the factor gelu'(z).  The next
        // piece's TMEM load is issued once this piece's values are packed, so
        // that it completes under this piece's stores.
        constexpr int W = BN / EPI_SLICES;
        constexpr int NP = W / 16;
        const int col0 = t.nt * BN + slice * W;
        uint16_t* w2base = p.out2 + (size_t)(t.row0 + quarter * 32) * p.N_out;
        uint32_t raw[16];
        __syncwarp();
        if (col0 < p.N_out) {
          tmem_ld16_issue(tb + slice * W, raw);
          tmem_wait16(raw);
        }
#pragma unroll 1
        for (int pc = 0; pc < NP; ++pc) {
          const int col = col0 + pc * 16;
          if (col >= p.N_out) break;  // warp-uniform; later pieces lie further right
          uint32_t pa[8], pd[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            f32x2 a, g;
            gelu_and_grad2(f2_pack(__uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1])), a, g);
            pa[i] = f2_to_bf16x2(a);
            pd[i] = f2_to_bf16x2(g);
          }
          const bool next = pc + 1 < NP && col + 16 < p.N_out;  // warp-uniform
          __syncwarp();
          if (next) tmem_ld16_issue(tb + slice * W + (pc + 1) * 16, raw);
          store_rows16(s.stg[warp - 2], wbase + col, (size_t)p.N_out, wrows, pa, lane);
          store_rows16(s.stg[warp - 2], w2base + col, (size_t)p.N_out, wrows, pd, lane);
          if (next) tmem_wait16(raw);
        }
      } else if (EPI == kBwdSwiglu) {
        // 16-column pieces: a = silu(g) u and the factors u silu'(g) and
        // silu(g), with silu(g) = g s, silu'(g) = s (1 + g (1 - s)),
        // s = 1 / (1 + exp(-g)).
        constexpr int W = (BN / 2) / EPI_SLICES;
        constexpr int NP = W / 16;
        const int col0 = t.nt * (BN / 2) + slice * W;
        const size_t ld2 = 2 * (size_t)p.N_out;
        uint16_t* w2base = p.out2 + (size_t)(t.row0 + quarter * 32) * ld2;
#pragma unroll 1
        for (int pc = 0; pc < NP; ++pc) {
          const int col = col0 + pc * 16;
          if (col >= p.N_out) break;  // warp-uniform
          const int c = slice * W + pc * 16;  // TMEM column
          __syncwarp();
          uint32_t gr[16], ur[16];
          tmem_ld16x2(tb + c, tb + BN / 2 + c, gr, ur);
          uint32_t pa[8], pg[8], pu[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float g0 = __uint_as_float(gr[2 * i]), g1 = __uint_as_float(gr[2 * i + 1]);
            const f32x2 g = f2_pack(g0, g1);
            const f32x2 u = f2_pack(__uint_as_float(ur[2 * i]), __uint_as_float(ur[2 * i + 1]));
            float e0, e1;
            f2_unpack(f2_add(f2_pack(__expf(-g0), __expf(-g1)), f2_splat(1.0f)), e0, e1);
            const f32x2 sg = f2_pack(__fdividef(1.0f, e0), __fdividef(1.0f, e1));
            const f32x2 silu = f2_mul(g, sg);
            const f32x2 oms = f2_add(f2_splat(1.0f), f2_mul(sg, f2_splat(-1.0f)));
            pa[i] = f2_to_bf16x2(f2_mul(silu, u));
            pg[i] = f2_to_bf16x2(f2_mul(f2_mul(u, sg), f2_fma(g, oms, f2_splat(1.0f))));
            pu[i] = f2_to_bf16x2(silu);
          }
          store_rows16(s.stg[warp - 2], wbase + col, (size_t)p.N_out, wrows, pa, lane);
          store_rows16(s.stg[warp - 2], w2base + col, ld2, wrows, pg, lane);
          store_rows16(s.stg[warp - 2], w2base + p.N_out + col, ld2, wrows, pu, lane);
        }
      } else if (EPI == kCombine) {
        constexpr int W = BN / EPI_SLICES;
        float wt;
        float* arow = comb_target(p, t.row0 + quarter * 32 + lane, t.row0 + t.rows, wt);
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
            red_add32(arow + col, v, wt);
          }
        }
      } else if (EPI == kSwiglu) {
        constexpr int W = (BN / 2) / EPI_SLICES;   // output columns per warp
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
      if (lane == 0) mbar_arrive(&s.tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    // factor copies still in flight (a role aborted) land before the exit
    if (EPI == kStoreKMMul && lane == 0) {
      for (int b = 0; b < 3; ++b)
        if (fpend[b]) wait_phase(&s.fbar[warp - 2][b], fph[b], &s.abort_flag, true);
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

// K4: replica counts for hot experts.
//
// MoE-GPS blog, section 2.1 (duplicate_experts): target load = total / slots;
// an expert loaded above 1.2 x target gets ceil(load / target) - 1 extra
// copies.  MoE-MPMC summary, contribution 3: copies are capped by a capacity
// bound.  On one GPU each expert owns one slot, so target = total / E and, in
// exact integers,
//   hot    <=>  load * E * den > num * total
//   copies  =   (load * E + total - 1) / total - 1.
// With loads summing to at most `total`, copies_e < load_e * E / total, so the
// copies sum to less than E and there are at most 2E - 1 groups.
//
// A memory budget (MoE-MPMC summary, contribution 3: replica counts limited
// by a predefined GPU memory budget) bounds the total of the copies: experts
// in order of decreasing load (lower expert first on equal loads) keep
// min(their copies, what is left of the budget); budget < 0: no bound.
//
// Loads from a prediction (moe_replicate_predicted): the largest-remainder
// apportionment of `total` in proportion to the predicted float32 shares --
// quotas q_e = p_e * total exact (p_e = m * 2^x with m a 24-bit integer, so
// m * total is an exact 64-bit product and the remainder an exact double
// for total < 2^29), floors, then one more for the experts with the largest
// remainders (lower expert first), repeated while any is left; floors above
// the total give one back from the smallest remainders (higher expert first)
// among positive floors.
#pragma once
#include "common.cuh"

namespace replicate {

constexpr int kThreads = 256;

// Block-level body (blockDim.x == kThreads, E <= kThreads).
__device__ __forceinline__ void replicate_block(const int32_t* __restrict__ load, int E, long long total, int num,
                                                int den, int max_copies, int32_t* __restrict__ copies_out,
                                                int32_t* __restrict__ rep_base,
                                                int32_t* __restrict__ group_expert, int budget = -1) {
  __shared__ int warp_sum[kThreads / 32];
  __shared__ long long load_sum[kThreads / 32];
  __shared__ int bad_sh;
  __shared__ int c_sh[kThreads];
  __shared__ int ld_sh[kThreads];
  const int e = threadIdx.x, lane = e & 31, wid = e >> 5;
  if (e == 0) bad_sh = 0;
  __syncthreads();
  long long ld = 0;
  int c = 0;
  if (e < E) {
    ld = load[e];
    if (ld < 0) bad_sh = 1;
    if (total > 0 && ld * E * den > (long long)num * total) {
      c = (int)((ld * E + total - 1) / total - 1);
      if (max_copies >= 0 && c > max_copies) c = max_copies;
    }
  }
  if (budget >= 0) {
    // hottest first: copies granted to the experts ranked before e
    c_sh[e] = c;
    ld_sh[e] = (int)ld;
    __syncthreads();
    if (e < E) {
      long long before = 0;
      for (int o = 0; o < E; ++o)
        if (ld_sh[o] > ld_sh[e] || (ld_sh[o] == ld_sh[e] && o < e)) before += c_sh[o];
      const long long room = (long long)budget - before;
      c = room <= 0 ? 0 : (room < c ? (int)room : c);
    }
  }
  // load sum check and exclusive scan of n = copies + 1 (one block)
  long long ls = ld;
  int n = (e < E) ? c + 1 : 0, incl = n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
    ls += __shfl_xor_sync(0xffffffffu, ls, off);
  }
  if (lane == 31) warp_sum[wid] = incl;
  if (lane == 0) load_sum[wid] = ls;
  __syncthreads();
  int before = 0, all = 0;
  long long lsum = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < wid) before += warp_sum[w];
    all += warp_sum[w];
    lsum += load_sum[w];
  }
  const bool bad = bad_sh || (total > 0 && lsum > total) || all > 2 * E;
  if (bad) {
    // precondition broken: flag it and emit the no-replication table
    if (e == 0) moe_flag_error(MOE_DEVERR_DATA);
    if (e < E) {
      copies_out[e] = 0;
      rep_base[e] = e;
      group_expert[e] = e;
      group_expert[E + e] = -1;
    }
    if (e == 0) rep_base[E] = E;
    return;
  }
  const int excl = before + incl - n;
  if (e < E) {
    copies_out[e] = c;
    rep_base[e] = excl;
    for (int q = 0; q < n; ++q) group_expert[excl + q] = e;
  }
  if (e == 0) rep_base[E] = all;
  for (int g = all + e; g < 2 * E; g += kThreads) group_expert[g] = -1;
}

// Largest-remainder apportionment of `total` over E experts by the float32
// shares p (see the header of this file).  Leaves the loads in load_out.
__device__ __forceinline__ void apportion_block(const float* __restrict__ p, int E, long long total,
                                                int32_t* __restrict__ load_out) {
  __shared__ double rem_sh[kThreads];
  __shared__ long long fl_sh[kThreads];
  __shared__ long long fsum_w[kThreads / 32];
  __shared__ int rank_sh[kThreads];
  const int e = threadIdx.x, lane = e & 31, wid = e >> 5;
  long long f = 0;
  double r = 0.0;
  if (e < E) {
    float v = p[e];
    if (!(v >= 0.f)) {  // negative or NaN share: counts as 0
      if (v != v) moe_flag_error(MOE_DEVERR_DATA);
      v = 0.f;
    }
    const uint32_t bits = __float_as_uint(v);
    const int be = (int)((bits >> 23) & 0xffu);
    const unsigned long long m = (bits & 0x7fffffu) | (be ? 0x800000u : 0u);
    const int sh = 150 - (be ? be : 1);  // v = m * 2^-sh
    const unsigned long long prod = m * (unsigned long long)total;
    if (sh <= 0) {  // v >= 2^23: not a share
      moe_flag_error(MOE_DEVERR_DATA);
      f = total;
      r = 0.0;
    } else if (sh >= 64) {
      f = 0;
      r = ldexp((double)prod, -sh);
    } else {
      f = (long long)(prod >> sh);
      r = ldexp((double)(prod & ((1ull << sh) - 1ull)), -sh);
    }
  }
  rem_sh[e] = e < E ? r : -1.0;
  fl_sh[e] = f;
  long long fs = f;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) fs += __shfl_xor_sync(0xffffffffu, fs, off);
  if (lane == 0) fsum_w[wid] = fs;
  __syncthreads();
  long long fsum = 0;
  for (int w = 0; w < kThreads / 32; ++w) fsum += fsum_w[w];
  // rank by (remainder descending, expert ascending)
  int rank = 0;
  if (e < E)
    for (int o = 0; o < E; ++o) rank += (rem_sh[o] > r || (rem_sh[o] == r && o < e)) ? 1 : 0;
  rank_sh[e] = e < E ? rank : kThreads;
  const long long left = total - fsum;
  if (left >= 0) {
    if (e < E) load_out[e] = (int32_t)(f + left / E + (rank < left % E ? 1 : 0));
    return;
  }
  // floors above the total: one back at a time from the smallest remainder
  // (highest rank first) among positive floors, cycling (one thread; |left|
  // is at most a few units when the shares sum to 1 within rounding)
  __syncthreads();
  if (e == 0) {
    __shared__ int order[kThreads];
    for (int o = 0; o < E; ++o) order[rank_sh[o]] = o;
    long long need = -left;
    int guard = 0;
    while (need > 0 && guard < 1 << 20) {
      bool moved = false;
      for (int q = E - 1; q >= 0 && need > 0; --q) {
        const int o = order[q];
        if (fl_sh[o] > 0) {
          --fl_sh[o];
          --need;
          moved = true;
        }
      }
      if (!moved) break;
      ++guard;
    }
    if (need > 0) moe_flag_error(MOE_DEVERR_DATA);
  }
  __syncthreads();
  if (e < E) load_out[e] = (int32_t)fl_sh[e];
}

__global__ void __launch_bounds__(kThreads) replicate_predicted_kernel(const float* __restrict__ p, int E,
                                                                       long long total, int num, int den,
                                                                       int max_copies, int budget,
                                                                       int32_t* __restrict__ load_out,
                                                                       int32_t* __restrict__ copies_out,
                                                                       int32_t* __restrict__ rep_base,
                                                                       int32_t* __restrict__ group_expert) {
  apportion_block(p, E, total, load_out);
  __syncthreads();  // the loads are global writes of this block: visible to it after the barrier
  replicate_block(load_out, E, total, num, den, max_copies, copies_out, rep_base, group_expert, budget);
}

__global__ void __launch_bounds__(kThreads) replicate_kernel(const int32_t* __restrict__ load, int E,
                                                             long long total, int num, int den, int max_copies,
                                                             int32_t* __restrict__ copies_out,
                                                             int32_t* __restrict__ rep_base,
                                                             int32_t* __restrict__ group_expert) {
  replicate_block(load, E, total, num, den, max_copies, copies_out, rep_base, group_expert);
}

static cudaError_t launch_predicted(const float* p, int E, long long total, int num, int den, int max_copies,
                                    int budget, int32_t* load_out, int32_t* copies, int32_t* rep_base,
                                    int32_t* group_expert, cudaStream_t st) {
  replicate_predicted_kernel<<<1, kThreads, 0, st>>>(p, E, total, num, den, max_copies, budget, load_out, copies,
                                                     rep_base, group_expert);
  return cudaGetLastError();
}

static cudaError_t launch(const int32_t* load, int E, long long total, int num, int den, int max_copies,
                          int32_t* copies, int32_t* rep_base, int32_t* group_expert, cudaStream_t st) {
  replicate_kernel<<<1, kThreads, 0, st>>>(load, E, total, num, den, max_copies, copies, rep_base, group_expert);
  return cudaGetLastError();
}

}  // namespace replicate

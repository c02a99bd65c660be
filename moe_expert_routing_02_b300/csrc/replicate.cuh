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
#pragma once
#include "common.cuh"

namespace replicate {

constexpr int kThreads = 256;

// Block-level body (blockDim.x == kThreads, E <= kThreads).
__device__ __forceinline__ void replicate_block(const int32_t* __restrict__ load, int E, long long total, int num,
                                                int den, int max_copies, int32_t* __restrict__ copies_out,
                                                int32_t* __restrict__ rep_base,
                                                int32_t* __restrict__ group_expert) {
  __shared__ int warp_sum[kThreads / 32];
  __shared__ long long load_sum[kThreads / 32];
  __shared__ int bad_sh;
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

__global__ void __launch_bounds__(kThreads) replicate_kernel(const int32_t* __restrict__ load, int E,
                                                             long long total, int num, int den, int max_copies,
                                                             int32_t* __restrict__ copies_out,
                                                             int32_t* __restrict__ rep_base,
                                                             int32_t* __restrict__ group_expert) {
  replicate_block(load, E, total, num, den, max_copies, copies_out, rep_base, group_expert);
}

static cudaError_t launch(const int32_t* load, int E, long long total, int num, int den, int max_copies,
                          int32_t* copies, int32_t* rep_base, int32_t* group_expert, cudaStream_t st) {
  replicate_kernel<<<1, kThreads, 0, st>>>(load, E, total, num, den, max_copies, copies, rep_base, group_expert);
  return cudaGetLastError();
}

}  // namespace replicate

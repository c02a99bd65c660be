// Physical replica copies of hot experts' weights (MoE-MPMC summary,
// contribution 2: predicted experts physically replicated on the GPU;
// PopFetcher review: expert copies fetched on a separate stream).
//
// The replica table lives on the device (moe_replicate / the front's plan),
// so the copies are made by a kernel that reads it, not by host-issued
// memory copies (which would need the table on the host first).  Layout of
// the caller's weight buffer: slots 0..E-1 hold the experts' weights, slots
// E.. the extra replicas in expert order; expert e's q-th extra replica
// (q = 1 .. n_e - 1, n_e = rep_base[e+1] - rep_base[e]) is slot
// E + (rep_base[e] - e) + q - 1.  group_slot[g] = weight slot of group g
// (-1 past the last group): the primary group of an expert reads its own
// slot, the replica groups their copies.
#pragma once
#include "common.cuh"

namespace replica_copy {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) slots_kernel(const int32_t* __restrict__ rep_base, int E,
                                                         int32_t* __restrict__ group_slot) {
  const int n_groups = rep_base[E];
  for (int g = threadIdx.x + blockIdx.x * kThreads; g < 2 * E; g += gridDim.x * kThreads) {
    int slot = -1;
    if (g < n_groups) {
      int lo = 0, hi = E;  // expert e with rep_base[e] <= g < rep_base[e+1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (rep_base[mid] <= g) lo = mid; else hi = mid;
      }
      const int q = g - rep_base[lo];
      slot = q == 0 ? lo : E + (rep_base[lo] - lo) + q - 1;
    }
    group_slot[g] = slot;
  }
}

// Copies every extra replica (16-byte vectors, grid-stride over all of them).
__global__ void __launch_bounds__(kThreads) copy_kernel(const int32_t* __restrict__ rep_base, int E,
                                                        uint4* __restrict__ w_all, long long slot_vecs) {
  const int extras = rep_base[E] - E;
  if (extras <= 0) return;
  const long long total = (long long)extras * slot_vecs;
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < total; i += (long long)gridDim.x * kThreads) {
    const int r = (int)(i / slot_vecs);
    const long long v = i - (long long)r * slot_vecs;
    int lo = 0, hi = E;  // expert e with rep_base[e] - e <= r < rep_base[e+1] - (e+1)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (rep_base[mid] - mid <= r) lo = mid; else hi = mid;
    }
    w_all[(size_t)(E + r) * slot_vecs + v] = w_all[(size_t)lo * slot_vecs + v];
  }
}

static cudaError_t launch(const int32_t* rep_base, int E, uint16_t* w_all, long long slot_elems, int32_t* group_slot,
                          int num_sms, cudaStream_t st) {
  if (group_slot) slots_kernel<<<1, kThreads, 0, st>>>(rep_base, E, group_slot);
  if (w_all) {
    copy_kernel<<<(unsigned)(num_sms * 4), kThreads, 0, st>>>(rep_base, E, reinterpret_cast<uint4*>(w_all),
                                                                slot_elems / 8);
  }
  return cudaGetLastError();
}

}  // namespace replica_copy

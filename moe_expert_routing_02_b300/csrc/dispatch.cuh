// K5: stable dispatch by expert, then replica (round-robin), and the
//     permuted copy of the token rows.
//
// PopFetcher (ATC'25) review, problem statement: tokens are dispatched to
// their experts before the expert FFN and collected afterwards.  MoE-MPMC
// summary (physical replication): tokens needing the same expert are spread
// over its distinct physical replicas.
//
// Assignment f = t*k + r.  Expert e's assignments, in ascending f, get ranks
// m = 0, 1, ...; rank m goes to replica q = m mod n_e at position
// floor(m / n_e) of group g = rep_base[e] + q.  Group sizes follow in closed
// form: floor(h_e / n_e) + [q < h_e mod n_e], so
//   slot(e, m) = base_e + q * floor(h_e/n_e) + min(q, h_e mod n_e) + floor(m/n_e)
// with base_e the exclusive scan of the expert totals h_e.
//
// Four launches, all deterministic (no slot depends on atomic order):
//   count   : per tile of 1024 assignments, per-expert counts (warp-aggregated
//             shared atomics) -> workspace
//   scan    : one block; per expert an exclusive scan over tiles (-> each
//             tile's starting rank), expert totals, group offsets
//   scatter : per tile, the stable in-tile rank of every assignment
//             (__match_any_sync rank inside the warp + earlier warps' counts +
//             earlier rounds' counts) -> slot -> perm / inv_perm
//   gather  : one warp per slot row, 128-bit loads/stores: xp[slot] = x[perm[slot]/k]
#pragma once
#include "common.cuh"

namespace dispatch {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 1024;
constexpr int kRounds = kTile / kThreads;
constexpr int kScanChunk = 8192;  // int32 counts staged per pass of the scan

// Workspace: counts[ntiles][E] int32, then info[4][E] int32 (base, n, h, unused).
__host__ __device__ inline long long num_tiles(long long A) { return (A + kTile - 1) / kTile; }
__host__ inline size_t workspace_bytes(long long A, int E) {
  const long long nt = num_tiles(A) > 0 ? num_tiles(A) : 1;
  return (size_t)(nt * E + 4LL * E) * sizeof(int32_t);
}

__global__ void __launch_bounds__(kThreads) count_kernel(const int32_t* __restrict__ idx, long long A, int E,
                                                         int32_t* __restrict__ counts) {
  extern __shared__ int32_t sh_cnt[];
  for (int i = threadIdx.x; i < E; i += kThreads) sh_cnt[i] = 0;
  __syncthreads();
  const long long f0 = (long long)blockIdx.x * kTile;
  bool bad = false;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const long long f = f0 + r * kThreads + threadIdx.x;
    int e = -1;
    if (f < A) {
      e = idx[f];
      if ((unsigned)e >= (unsigned)E) {
        bad = true;
        e = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&sh_cnt[e], __popc(peers));
  }
  if (bad) moe_flag_error(MOE_DEVERR_DATA);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += kThreads) counts[(size_t)blockIdx.x * E + i] = sh_cnt[i];
}

__global__ void __launch_bounds__(kThreads) scan_kernel(int32_t* __restrict__ counts, long long ntiles, int E,
                                                        long long A, const int32_t* __restrict__ rep_base,
                                                        int32_t* __restrict__ info,
                                                        int32_t* __restrict__ group_offsets) {
  __shared__ int32_t warp_tot[kWarps];
  __shared__ int bad_sh;
  const int e = threadIdx.x, lane = e & 31, wid = e >> 5;
  if (e == 0) bad_sh = 0;
  __syncthreads();
  // per-expert exclusive scan over tiles, staged through shared memory in
  // chunks (coalesced loads; the serial walk runs on shared memory)
  __shared__ int32_t chunk[kScanChunk];
  int h = 0, n = 1, rb = e;
  const long long per = kScanChunk / E;  // tiles per chunk
  for (long long b0 = 0; b0 < ntiles; b0 += per) {
    const long long nb = (ntiles - b0 < per) ? (ntiles - b0) : per;
    const long long cnt = nb * E;
    for (long long i = e; i < cnt; i += kThreads) chunk[i] = counts[b0 * E + i];
    __syncthreads();
    if (e < E) {
      for (long long b = 0; b < nb; ++b) {
        const int c = chunk[b * E + e];
        chunk[b * E + e] = h;
        h += c;
      }
    }
    __syncthreads();
    for (long long i = e; i < cnt; i += kThreads) counts[b0 * E + i] = chunk[i];
    __syncthreads();
  }
  if (e < E) {
    if (rep_base) {
      rb = rep_base[e];
      n = rep_base[e + 1] - rb;
      if (n < 1 || rb < 0 || (e == 0 && rb != 0) || rep_base[e + 1] > 2 * E) bad_sh = 1;
    }
  }
  __syncthreads();
  const bool use_rep = rep_base != nullptr && !bad_sh;
  if (!use_rep) {
    // invalid replica table: flag it and lay out one group per expert
    if (rep_base != nullptr && e == 0) moe_flag_error(MOE_DEVERR_DATA);
    n = 1;
    rb = e;
  }
  // exclusive scan of h over experts
  int incl = (e < E) ? h : 0;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < wid; ++w) before += warp_tot[w];
  const int base = before + incl - ((e < E) ? h : 0);
  if (e < E) {
    info[e] = base;
    info[E + e] = n;
    info[2 * E + e] = h;
    const int qs = h / n, qr = h % n;
    for (int q = 0; q < n; ++q) group_offsets[rb + q] = base + q * qs + (q < qr ? q : qr);
  }
  // entries past the last group equal A
  const int ngroups = use_rep ? rep_base[E] : E;
  for (int g = ngroups + e; g <= 2 * E; g += kThreads) group_offsets[g] = (int32_t)A;
}

__global__ void __launch_bounds__(kThreads) scatter_kernel(const int32_t* __restrict__ idx, long long A, int E,
                                                           const int32_t* __restrict__ tile_base,
                                                           const int32_t* __restrict__ info,
                                                           int32_t* __restrict__ perm,
                                                           int32_t* __restrict__ inv_perm) {
  extern __shared__ int32_t sm[];
  int32_t* warp_cnt = sm;            // [kWarps][E]
  int32_t* run = sm + kWarps * E;    // [E]
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int i = tid; i < kWarps * E; i += kThreads) warp_cnt[i] = 0;
  for (int i = tid; i < E; i += kThreads) run[i] = tile_base[(size_t)blockIdx.x * E + i];
  __syncthreads();
  const long long f0 = (long long)blockIdx.x * kTile;
  for (int r = 0; r < kRounds; ++r) {
    const long long f = f0 + r * kThreads + tid;
    int e = -1;
    if (f < A) {
      e = idx[f];
      if ((unsigned)e >= (unsigned)E) e = -1;  // flagged by count_kernel
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) warp_cnt[wid * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int m = run[e] + __popc(peers & lanemask_lt());
      for (int w = 0; w < wid; ++w) m += warp_cnt[w * E + e];
      const int base = info[e], n = info[E + e], h = info[2 * E + e];
      const int q = m % n, pos = m / n, qs = h / n, qr = h % n;
      const int slot = base + q * qs + (q < qr ? q : qr) + pos;
      if ((unsigned long long)slot < (unsigned long long)A) {
        perm[slot] = (int32_t)f;
        inv_perm[f] = slot;
      } else {
        inv_perm[f] = -1;
      }
    } else if (f < A) {
      inv_perm[f] = -1;  // expert out of range (flagged by count_kernel): no slot
    }
    __syncthreads();
    for (int i = tid; i < E; i += kThreads) {
      int s = 0;
      for (int w = 0; w < kWarps; ++w) {
        s += warp_cnt[w * E + i];
        warp_cnt[w * E + i] = 0;
      }
      run[i] += s;
    }
    __syncthreads();
  }
}

// xp[inv_perm[t k + r], :] = x[t, :] for every assignment with a slot: two tokens per
// warp, each token row read once, 16-byte vectors.
__global__ void __launch_bounds__(kThreads) gather_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ inv_perm, long long T, int k,
                                                          int H, uint16_t* __restrict__ xp) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * kWarps;
  const long long A = T * k;
  const int chunks = H / 8;
  // two tokens per warp (eight 16-byte loads in flight per lane); each token
  // row is read once and stored to the slots of all k of its assignments
  for (long long t = (((long long)blockIdx.x * kThreads + threadIdx.x) >> 5) * 2; t < T; t += 2 * warps) {
    const bool has1 = t + 1 < T;
    const uint16_t* src0 = x + t * H;
    const uint16_t* src1 = src0 + H;
    for (int c = lane; c < chunks; c += 128) {
      uint4 v0[4], v1[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int cu = c + 32 * u;
        if (cu < chunks) {
          v0[u] = ld_nc_v4(src0 + (size_t)cu * 8);
          if (has1) v1[u] = ld_nc_v4(src1 + (size_t)cu * 8);
        }
      }
      for (int r = 0; r < k; ++r) {
        const int32_t s0 = inv_perm[t * k + r];
        if ((unsigned long long)s0 < (unsigned long long)A) {  // -1: no slot (invalid routing)
          uint16_t* dst = xp + (size_t)s0 * H;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (c + 32 * u < chunks) st_v4(dst + (size_t)(c + 32 * u) * 8, v0[u]);
        }
        const int32_t s1 = has1 ? inv_perm[(t + 1) * k + r] : -1;
        if ((unsigned long long)s1 < (unsigned long long)A) {
          uint16_t* dst = xp + (size_t)s1 * H;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (c + 32 * u < chunks) st_v4(dst + (size_t)(c + 32 * u) * 8, v1[u]);
        }
      }
    }
  }
}

struct Args {
  const uint16_t* x;
  const int32_t* idx;
  long long T;
  int k, H, E;
  const int32_t* rep_base;
  int32_t* group_offsets;
  int32_t* perm;
  int32_t* inv_perm;
  uint16_t* xp;
  void* ws;
};

static cudaError_t launch(const Args& a, int num_sms, cudaStream_t st) {
  const long long A = a.T * a.k;
  const int E = a.E;
  if (A == 0) {
    // empty batch: every offset is 0
    return cudaMemsetAsync(a.group_offsets, 0, sizeof(int32_t) * (2 * E + 1), st);
  }
  const long long nt = num_tiles(A);
  int32_t* counts = reinterpret_cast<int32_t*>(a.ws);
  int32_t* info = counts + nt * E;
  count_kernel<<<(unsigned)nt, kThreads, sizeof(int32_t) * E, st>>>(a.idx, A, E, counts);
  scan_kernel<<<1, kThreads, 0, st>>>(counts, nt, E, A, a.rep_base, info, a.group_offsets);
  scatter_kernel<<<(unsigned)nt, kThreads, sizeof(int32_t) * (kWarps + 1) * E, st>>>(a.idx, A, E, counts, info,
                                                                                      a.perm, a.inv_perm);
  if (a.x != nullptr) {
    long long blocks = (a.T + 2 * kWarps - 1) / (2 * kWarps);
    const long long cap = (long long)num_sms * 16;
    if (blocks > cap) blocks = cap;
    gather_kernel<<<(unsigned)blocks, kThreads, 0, st>>>(a.x, a.inv_perm, a.T, a.k, a.H, a.xp);
  }
  return cudaGetLastError();
}

}  // namespace dispatch

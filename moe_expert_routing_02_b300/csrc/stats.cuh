// K2: per-expert histogram and layer j-1 -> j co-selection counts, written to
//     the window ring and folded into running window sums.
// K3: window popularity, conditional probability and next-layer prediction.
//
// PopFetcher (ATC'25) review: observation 1 (token allocation per expert),
// observation 2 / Fig. 6 (inter-layer conditional probability), core method
// (Routing Information Collector with a sliding window of s iterations;
// Eq. (1) sequence popularity, Eq. (2)(3) next-layer popularity).  MoE-GPS
// blog, section 2.1: p_i = n_i / N averaged over a sliding window.
//
// K2 is one launch: blocks walk the tokens grid-stride, each thread with the
// choices of kTokensAhead tokens loaded before it counts them, and count into
// shared memory with plain atomics (E bins, and the E*E co-selection bins
// when E <= 64); blocks flush the non-zero bins to a global accumulator, and
// the last block to finish (ticket counter after a fence) moves the
// accumulator into ring slot iter % s, updates the window sums by
// (new - old) and zeroes the accumulator for the next call.  Counts are
// integers, so the result does not depend on the order in which atomics land.
#pragma once
#include "common.cuh"

namespace stats {

constexpr int kThreads = 256;
constexpr int kSmemCoselMaxE = 64;  // E*E counters in shared memory up to E = 64

struct UpdateArgs {
  const int32_t* idx_cur;   // [T,k]
  const int32_t* idx_prev;  // [T,k] (read only when has_prev and T > 0)
  int has_prev;             // layer > 0: co-selection counts are kept
  int T, k, E;
  uint32_t* acc_h;          // [E]   zero between calls
  uint32_t* acc_c;          // [E*E] zero between calls
  uint32_t* ticket;         // zero between calls
  uint32_t* ring_h;         // slot of layer j   [E]
  unsigned long long* hsum; // window sum layer j [E]
  uint32_t* ring_c;         // slot of pair j-1  [E*E] or null
  unsigned long long* csum; // window sum pair j-1 [E*E] or null
  int32_t* hist_out;        // [E] or null
};

constexpr int kTokensAhead = 4;

// The last block to finish (ticket after a fence) moves the accumulated
// totals into ring slot iter % s, updates the window sums by (new - old) and
// zeroes the accumulator and the ticket for the next call.
template <int NT>
__device__ __forceinline__ void fold_last_block(const UpdateArgs& a) {
  __shared__ bool is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < a.E; i += NT) {
    const uint32_t nw = atomicExch(a.acc_h + i, 0u);
    const uint32_t old = a.ring_h[i];
    a.ring_h[i] = nw;
    a.hsum[i] = a.hsum[i] + nw - old;
    if (a.hist_out) a.hist_out[i] = (int32_t)nw;
  }
  if (a.has_prev) {
    for (int i = threadIdx.x; i < a.E * a.E; i += NT) {
      const uint32_t nw = atomicExch(a.acc_c + i, 0u);
      const uint32_t old = a.ring_c[i];
      a.ring_c[i] = nw;
      a.csum[i] = a.csum[i] + nw - old;
    }
  }
  if (threadIdx.x == 0) *a.ticket = 0;
}

__global__ void __launch_bounds__(kThreads) update_kernel(UpdateArgs a) {
  extern __shared__ uint32_t sh[];
  const int E = a.E, k = a.k;
  const bool cos = a.has_prev != 0;
  const bool cos_smem = cos && E <= kSmemCoselMaxE;
  uint32_t* sh_h = sh;
  uint32_t* sh_c = sh + E;
  uint32_t* cbase = cos_smem ? sh_c : a.acc_c;
  const int nsh = E + (cos_smem ? E * E : 0);
  for (int i = threadIdx.x; i < nsh; i += kThreads) sh[i] = 0;
  __syncthreads();

  constexpr int U = kTokensAhead;
  const long long stride = (long long)gridDim.x * kThreads * U;
  bool bad = false;
  for (long long base = (long long)blockIdx.x * kThreads * U + threadIdx.x; base < a.T; base += stride) {
    // tokens base, base + kThreads, ... (coalesced across the block)
    int cur[U][8], prv[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long t = base + (long long)u * kThreads;
      const bool live = t < a.T;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        cur[u][r] = -1;
        prv[u][r] = -1;
        if (r < k && live) {
          cur[u][r] = a.idx_cur[t * k + r];
          if (cos) prv[u][r] = a.idx_prev[t * k + r];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool live = base + (long long)u * kThreads < a.T;
      if (!live) continue;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r < k) {
          if ((unsigned)cur[u][r] < (unsigned)E)
            atomicAdd(sh_h + cur[u][r], 1u);
          else
            bad = true;
        }
      }
      if (cos) {
#pragma unroll
        for (int r1 = 0; r1 < 8; ++r1) {
          if (r1 < k) {
            const int p = prv[u][r1];
            if ((unsigned)p >= (unsigned)E) {
              bad = true;
              continue;
            }
#pragma unroll
            for (int r2 = 0; r2 < 8; ++r2)
              if (r2 < k && (unsigned)cur[u][r2] < (unsigned)E) atomicAdd(cbase + p * E + cur[u][r2], 1u);
          }
        }
      }
    }
  }
  if (bad) moe_flag_error(MOE_DEVERR_DATA);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += kThreads)
    if (sh_h[i]) atomicAdd(a.acc_h + i, sh_h[i]);
  if (cos_smem)
    for (int i = threadIdx.x; i < E * E; i += kThreads)
      if (sh_c[i]) atomicAdd(a.acc_c + i, sh_c[i]);

  fold_last_block<kThreads>(a);
}

// E <= 16: the histogram lives in 16 registers per thread (a compare-and-add
// per bin, no dynamic indexing), so the Zipf-skewed hot bins take no atomics
// at all; each warp counts its co-selection pairs into its own E*E bins in
// shared memory (8 KB per block), so shared atomics meet only the other lanes
// of their warp, not the whole block.  At the end the warps' bins are summed
// per bin, the histogram per warp by shuffles, each block adds its non-zero
// bins to the global accumulator, and the last block folds as update_kernel
// does.
constexpr int kSmallE = 16;
constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;

// KM: the largest k the instance handles (2 covers top-1 and top-2 with far
// fewer registers; 8 the rest).
template <int KM>
__global__ void __launch_bounds__(kSmallThreads, 2) update_small_kernel(UpdateArgs a) {
  __shared__ uint32_t wb[kSmallWarps][kSmallE * kSmallE];  // per-warp co-selection bins p * 16 + c
  __shared__ uint32_t hs[kSmallE];
  const int E = a.E, k = a.k;
  const bool cos = a.has_prev != 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < kSmallE) hs[threadIdx.x] = 0;
  if (cos)
    for (int i = threadIdx.x; i < kSmallWarps * kSmallE * kSmallE; i += kSmallThreads) (&wb[0][0])[i] = 0u;
  __syncthreads();
  uint32_t* mb = wb[warp];
  uint32_t h[kSmallE];
#pragma unroll
  for (int q = 0; q < kSmallE; ++q) h[q] = 0u;

  // tokens in flight per thread (the loop is bound by the latency of its
  // loads), within 128 registers; top-2 rows are read as one 8-byte load when
  // both index arrays are 8-byte aligned
  constexpr int U = KM <= 2 ? 6 : 2;
  const bool pair_loads = KM == 2 && k == 2 &&
                          ((reinterpret_cast<uintptr_t>(a.idx_cur) | reinterpret_cast<uintptr_t>(a.idx_prev)) & 7) == 0;
  const long long stride = (long long)gridDim.x * kSmallThreads * U;
  bool bad = false;
  for (long long base = (long long)blockIdx.x * kSmallThreads * U + threadIdx.x; base < a.T; base += stride) {
    int cur[U][KM], prv[U][KM];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long t = base + (long long)u * kSmallThreads;
      const bool live = t < a.T;
#pragma unroll
      for (int r = 0; r < KM; ++r) {
        cur[u][r] = -1;
        prv[u][r] = -1;
      }
      if (pair_loads) {
        if (live) {
          const int2 c2 = *reinterpret_cast<const int2*>(a.idx_cur + t * 2);
          cur[u][0] = c2.x;
          cur[u][KM - 1] = c2.y;
          if (cos) {
            const int2 p2 = *reinterpret_cast<const int2*>(a.idx_prev + t * 2);
            prv[u][0] = p2.x;
            prv[u][KM - 1] = p2.y;
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < KM; ++r) {
          if (r < k && live) {
            cur[u][r] = a.idx_cur[t * k + r];
            if (cos) prv[u][r] = a.idx_prev[t * k + r];
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (base + (long long)u * kSmallThreads >= a.T) continue;
#pragma unroll
      for (int r = 0; r < KM; ++r) {
        if (r < k) {
          const int e = cur[u][r];
          if ((unsigned)e >= (unsigned)E) {
            bad = true;
            continue;
          }
#pragma unroll
          for (int q = 0; q < kSmallE; ++q) h[q] += (e == q) ? 1u : 0u;
        }
      }
      if (cos) {
#pragma unroll
        for (int r1 = 0; r1 < KM; ++r1) {
          if (r1 < k) {
            const int pe = prv[u][r1];
            if ((unsigned)pe >= (unsigned)E) {
              bad = true;
              continue;
            }
#pragma unroll
            for (int r2 = 0; r2 < KM; ++r2)
              if (r2 < k && (unsigned)cur[u][r2] < (unsigned)E) atomicAdd(mb + pe * kSmallE + cur[u][r2], 1u);
          }
        }
      }
    }
  }
  if (bad) moe_flag_error(MOE_DEVERR_DATA);
  // histogram: warp sums by butterflies, then one shared add per warp and bin
#pragma unroll
  for (int q = 0; q < kSmallE; ++q) {
    uint32_t v = h[q];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    h[q] = v;
  }
  if (lane == 0) {
#pragma unroll
    for (int q = 0; q < kSmallE; ++q)
      if (h[q]) atomicAdd(&hs[q], h[q]);
  }
  __syncthreads();
  if (cos) {
    const int b = threadIdx.x;  // kSmallThreads == 16 * 16 bins
    uint32_t v = 0;
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) v += wb[w][b];
    const int p = b / kSmallE, c = b % kSmallE;
    if (v && p < E && c < E) atomicAdd(a.acc_c + p * E + c, v);
  }
  if (threadIdx.x < E && hs[threadIdx.x]) atomicAdd(a.acc_h + threadIdx.x, hs[threadIdx.x]);
  fold_last_block<kSmallThreads>(a);
}
static_assert(kSmallThreads == kSmallE * kSmallE, "one thread per co-selection bin in the block sum");

static cudaError_t launch_update(const UpdateArgs& a, int num_sms, cudaStream_t st) {
  if (a.E <= kSmallE) {
    long long blocks = ((long long)a.T + kTokensAhead * kSmallThreads - 1) / (kTokensAhead * kSmallThreads);
    if (blocks > 2LL * num_sms) blocks = 2LL * num_sms;  // each block flushes up to E + E*E bins
    if (blocks < 1) blocks = 1;
    if (a.k <= 2)
      update_small_kernel<2><<<(int)blocks, kSmallThreads, 0, st>>>(a);
    else
      update_small_kernel<8><<<(int)blocks, kSmallThreads, 0, st>>>(a);
    return cudaGetLastError();
  }
  const bool cos_smem = a.has_prev != 0 && a.E <= kSmemCoselMaxE;
  const size_t smem = sizeof(uint32_t) * (a.E + (cos_smem ? a.E * a.E : 0));
  long long blocks = ((long long)a.T + kTokensAhead * kThreads - 1) / (kTokensAhead * kThreads);
  if (blocks > 2LL * num_sms) blocks = 2LL * num_sms;  // each block flushes up to E + E*E bins
  if (blocks < 1) blocks = 1;
  update_kernel<<<(int)blocks, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- K3
// One block, fp64 throughout (window sums are integers, converted exactly).
// Every read is a cooperative, coalesced load into shared memory first; the
// row sums of Cbar are one warp per row.  Pr(e'|e) = Cbar[e,e'] / row[e] is
// formed as Cbar * (1 / row) -- within one fp64 ulp of the division, far below
// the fp32 output rounding.
constexpr int kPredictSmemE = 64;  // Cbar staged in shared memory up to E = 64

// Block-level body (blockDim.x == kThreads).  Callable from any kernel whose
// block reaches it with all threads.  S is the type of the window sums:
// unsigned long long (plain window) or double (decay-weighted window; integer
// sums are exact in double, so both give the same result for equal sums).
// Cbar is staged in shared memory for E <= STAGE_E (a kernel that runs this
// in one of many blocks keeps STAGE_E small, since the staging array is part
// of every block's static shared memory); the result does not depend on it.
template <typename S, int STAGE_E = kPredictSmemE>
__device__ __forceinline__ void predict_block(const S* __restrict__ hsum, const S* __restrict__ csum, int E,
                                              float* __restrict__ p_seq, float* __restrict__ cond,
                                              float* __restrict__ p_next) {
  __shared__ double ps[256];
  __shared__ double rinv[256];   // 1 / row sum, or 0 for an empty row
  __shared__ S rsum[256];
  __shared__ S wsum[kThreads / 32];
  __shared__ S cs[STAGE_E * STAGE_E];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool stage = csum != nullptr && E <= STAGE_E;
  S h = tid < E ? hsum[tid] : S(0);
  if (stage)
    for (int i = tid; i < E * E; i += kThreads) cs[i] = csum[i];
  S tot = h;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
  if (lane == 0) wsum[wid] = tot;
  __syncthreads();
  // row sums of Cbar: one warp per row
  if (csum) {
    for (int e = wid; e < E; e += kThreads / 32) {
      S r = 0;
      for (int e2 = lane; e2 < E; e2 += 32) r += stage ? cs[e * E + e2] : csum[(size_t)e * E + e2];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
      if (lane == 0) rsum[e] = r;
    }
  }
  tot = 0;
  for (int w = 0; w < kThreads / 32; ++w) tot += wsum[w];
  __syncthreads();
  // the two divisions of each expert run side by side in its thread
  if (tid < E) {
    const double p = tot > 0 ? (double)h / (double)tot : 1.0 / (double)E;
    ps[tid] = p;
    p_seq[tid] = (float)p;
    if (csum) {
      const S r = rsum[tid];
      rinv[tid] = r > 0 ? 1.0 / (double)r : 0.0;
    }
  }
  if (!csum) return;
  __syncthreads();
  const double uni = 1.0 / (double)E;
  if (cond) {
    for (int i = tid; i < E * E; i += kThreads) {
      const double ri = rinv[i / E];
      const S cv = stage ? cs[i] : csum[i];
      cond[i] = (float)(ri > 0 ? (double)cv * ri : uni);
    }
  }
  if (p_next) {
    // p_next[e'] = sum_e p_seq[e] * Pr(e'|e).  Thread t works on column
    // e' = t / P and rows e = q, q + P, ... (q = t % P, P a power of two with
    // P * E <= 256), two interleaved accumulators; the P partial sums of a
    // column sit in P adjacent lanes and are added by a butterfly, so the
    // order of the additions is fixed (the result is deterministic)
    int P = 1;
    while (P * 2 * E <= kThreads && P < 32) P *= 2;
    const int col = tid / P, q = tid % P;
    double a0 = 0.0, a1 = 0.0;
    if (col < E) {
      int e = q;
      for (; e + P < E; e += 2 * P) {
        const double r0 = rinv[e], r1 = rinv[e + P];
        const S c0 = stage ? cs[e * E + col] : csum[(size_t)e * E + col];
        const S c1 = stage ? cs[(e + P) * E + col] : csum[(size_t)(e + P) * E + col];
        a0 = fma(ps[e], r0 > 0 ? (double)c0 * r0 : uni, a0);
        a1 = fma(ps[e + P], r1 > 0 ? (double)c1 * r1 : uni, a1);
      }
      if (e < E) {
        const double r0 = rinv[e];
        const S c0 = stage ? cs[e * E + col] : csum[(size_t)e * E + col];
        a0 = fma(ps[e], r0 > 0 ? (double)c0 * r0 : uni, a0);
      }
    }
    double acc = a0 + a1;
    for (int off = 1; off < P; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (col < E && q == 0) p_next[col] = (float)acc;
  }
}

__global__ void __launch_bounds__(kThreads) predict_kernel(const unsigned long long* __restrict__ hsum,
                                                           const unsigned long long* __restrict__ csum, int E,
                                                           float* __restrict__ p_seq, float* __restrict__ cond,
                                                           float* __restrict__ p_next) {
  predict_block<unsigned long long>(hsum, csum, E, p_seq, cond, p_next);
}

// Decay-weighted window (MoE-GPS blog section 2.1: sliding-window average
// with a decay factor against drift).  Under the causal order (layer j
// recorded at iteration `iter`, then predicted, then layer j+1 recorded),
// ring slot (iter - a) mod s of h_j and slot (iter - 1 - a) mod s of C_j
// weigh lam^a, a = 0 .. s-1 (weights lam^a by repeated multiplication in
// fp64, lam^0 = 1).  The weighted sums go to `scratch` ([E + E*E] doubles),
// then the block predicts from them as from the plain window sums.
__global__ void __launch_bounds__(kThreads) predict_decay_kernel(const uint32_t* __restrict__ ring_h,
                                                                 const uint32_t* __restrict__ ring_c, int E, int s,
                                                                 long long iter, double lam,
                                                                 double* __restrict__ scratch,
                                                                 float* __restrict__ p_seq,
                                                                 float* __restrict__ cond,
                                                                 float* __restrict__ p_next) {
  __shared__ double w[1024];
  for (int a = threadIdx.x; a < s; a += kThreads) {
    double v = 1.0;
    for (int q = 0; q < a; ++q) v *= lam;
    w[a] = v;
  }
  __syncthreads();
  double* H = scratch;
  double* C = scratch + E;
  for (int e = threadIdx.x; e < E; e += kThreads) {
    double acc = 0.0;
    for (int a = 0; a < s; ++a) {
      const long long slot = ((iter - a) % s + s) % s;
      acc += w[a] * (double)ring_h[(size_t)slot * E + e];
    }
    H[e] = acc;
  }
  if (ring_c) {
    for (int i = threadIdx.x; i < E * E; i += kThreads) {
      double acc = 0.0;
      for (int a = 0; a < s; ++a) {
        const long long slot = ((iter - 1 - a) % s + s) % s;
        acc += w[a] * (double)ring_c[(size_t)slot * E * E + i];
      }
      C[i] = acc;
    }
  }
  __syncthreads();  // the block's global writes are visible to the block after the barrier
  predict_block<double>(H, ring_c ? C : nullptr, E, p_seq, cond, p_next);
}

}  // namespace stats

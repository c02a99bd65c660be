// K1: top-k gate over router logits.
//
// PopFetcher (ATC'25) review: naive top-k gate; EPS-MoE review, experiments:
// top-2 / top-4 / top-6 with softmax-renormalised gate weights.
//
// A group of G lanes (G = 1..32, a power of two) owns one token: the token's
// E logits are read with 128-bit loads, lane g holding float4 chunks
// g, g+G, ... (at most two chunks, eight values, since E <= 256).  The k
// winners are taken one at a time: every lane offers its best unchosen value,
// a butterfly over the G lanes keeps the larger value (lower expert index on
// equal values; -0.0 == +0.0), and the owning lane retires it.  Logits are
// read once; the kernel is bound by HBM bandwidth (or launch latency at small T).
#pragma once
#include "common.cuh"

namespace route {

constexpr int kThreads = 256;

__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

// Top-k of one token's logits by its group of G lanes (all G lanes call it,
// `live` false for a lane group past the last token).  On return every lane
// of the group holds the k winners (sel_i, rank order) and their logits
// (sel_v); *denom is the softmax denominator of the chosen weighting, so
// w_r = expf(sel_v[r] - sel_v[0]) / *denom.
template <int G, bool VEC>
__device__ __forceinline__ void topk_token(const float* __restrict__ row, bool live, int E, int k, int renorm,
                                           float (&sel_v)[8], int (&sel_i)[8], float* denom_out) {
  const int gl = (threadIdx.x & 31) % G;
  float v[8];
  int id[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    v[s] = -INFINITY;
    id[s] = 0x7fffffff;
  }
  if (live) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int chunk = gl + c * G;
      const int e0 = chunk * 4;
      if (VEC) {
        if (e0 < E) {
          float4 q = __ldg(reinterpret_cast<const float4*>(row + e0));
          v[c * 4 + 0] = q.x; v[c * 4 + 1] = q.y; v[c * 4 + 2] = q.z; v[c * 4 + 3] = q.w;
#pragma unroll
          for (int u = 0; u < 4; ++u) id[c * 4 + u] = e0 + u;
        }
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (e0 + u < E) {
            v[c * 4 + u] = __ldg(row + e0 + u);
            id[c * 4 + u] = e0 + u;
          }
        }
      }
    }
  }

  unsigned chosen = 0;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    sel_v[r] = -INFINITY;
    sel_i[r] = 0;
    if (r < k) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        if (id[s] != 0x7fffffff && !((chosen >> s) & 1u) && better(v[s], id[s], bv, bi)) {
          bv = v[s];
          bi = id[s];
        }
      }
#pragma unroll
      for (int off = G / 2; off >= 1; off >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (id[s] == bi) chosen |= 1u << s;
      sel_v[r] = bv;
      sel_i[r] = bi;
    }
  }

  // gate-weight denominator
  float denom = 0.f;
  const float ref = sel_v[0];
  if (renorm) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < k) denom += expf(sel_v[r] - ref);
  } else {
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (id[s] != 0x7fffffff) denom += expf(v[s] - ref);
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
  }
  *denom_out = denom;
}

// Lane gl of the token's group writes ranks r with r % G == gl.
template <int G>
__device__ __forceinline__ void write_token(long long t, int k, const float (&sel_v)[8], const int (&sel_i)[8],
                                            float denom, int32_t* __restrict__ idx, float* __restrict__ wout) {
  const int gl = (threadIdx.x & 31) % G;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    if (r < k && (r % G) == gl) {
      idx[(size_t)t * k + r] = sel_i[r];
      wout[(size_t)t * k + r] = expf(sel_v[r] - sel_v[0]) / denom;
    }
  }
}

template <int G, bool VEC>
__global__ void __launch_bounds__(kThreads) topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                        int renorm, int32_t* __restrict__ idx,
                                                        float* __restrict__ wout) {
  constexpr int TPW = 32 / G;  // tokens per warp
  const int lane = threadIdx.x & 31;
  const long long warp_id = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const long long t = warp_id * TPW + lane / G;
  const bool live = t < T;
  float sel_v[8], denom;
  int sel_i[8];
  topk_token<G, VEC>(logits + (size_t)(live ? t : 0) * E, live, E, k, renorm, sel_v, sel_i, &denom);
  if (live) write_token<G>(t, k, sel_v, sel_i, denom, idx, wout);
}

template <int G>
static cudaError_t launch_g(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                            cudaStream_t st) {
  constexpr int tokens_per_block = (kThreads / 32) * (32 / G);
  const int blocks = (T + tokens_per_block - 1) / tokens_per_block;
  const bool vec = (E % 4 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  if (vec)
    topk_kernel<G, true><<<blocks, kThreads, 0, st>>>(logits, T, E, k, renorm, idx, w);
  else
    topk_kernel<G, false><<<blocks, kThreads, 0, st>>>(logits, T, E, k, renorm, idx, w);
  return cudaGetLastError();
}

// Lanes per token: smallest power of two with G*8 >= E (<= 2 float4 per lane).
static cudaError_t launch(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                          cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (E <= 8) return launch_g<1>(logits, T, E, k, renorm, idx, w, st);
  if (E <= 16) return launch_g<2>(logits, T, E, k, renorm, idx, w, st);
  if (E <= 32) return launch_g<4>(logits, T, E, k, renorm, idx, w, st);
  if (E <= 64) return launch_g<8>(logits, T, E, k, renorm, idx, w, st);
  if (E <= 128) return launch_g<16>(logits, T, E, k, renorm, idx, w, st);
  return launch_g<32>(logits, T, E, k, renorm, idx, w, st);
}

}  // namespace route

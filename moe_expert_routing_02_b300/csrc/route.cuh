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
// read once.  moe_route's kernel has the rank count as a template parameter
// and compares (value, expert) as one 64-bit key; the fused front
// (front.cuh) uses the generic-k device functions below.
#pragma once
#include "common.cuh"

namespace route {

constexpr int kThreads = 256;

__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

// Logits of one token for its group of G lanes: lane gl holds float4 chunks
// gl and gl + G (values past E, or of a dead token, are -inf).
template <int G, bool VEC>
__device__ __forceinline__ void load_token(const float* __restrict__ row, bool live, int E, float (&v)[8]) {
  const int gl = (threadIdx.x & 31) % G;
#pragma unroll
  for (int s = 0; s < 8; ++s) v[s] = -INFINITY;
  if (!live) return;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int e0 = (gl + c * G) * 4;
    if (VEC) {
      if (e0 < E) {
        const float4 q = __ldg(reinterpret_cast<const float4*>(row + e0));
        v[c * 4 + 0] = q.x; v[c * 4 + 1] = q.y; v[c * 4 + 2] = q.z; v[c * 4 + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e0 + u < E) v[c * 4 + u] = __ldg(row + e0 + u);
    }
  }
}

// Top-k of one token from its loaded values, by its group of G lanes (all G
// lanes call it).  ex[r] = expf(sel_v[r] - sel_v[0]) for the k winners.  On return every lane of the group holds the k winners
// (sel_i, rank order) and their logits (sel_v); *denom is the softmax
// denominator of the chosen weighting, so w_r = expf(sel_v[r] - sel_v[0]) / *denom.
template <int G>
__device__ __forceinline__ void select_token_ex(const float (&v)[8], bool live, int E, int k, int renorm,
                                                float (&sel_v)[8], int (&sel_i)[8], float (&ex)[8],
                                                float* denom_out) {
  const int gl = (threadIdx.x & 31) % G;
  int id[8];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = (gl + c * G) * 4 + u;
      id[c * 4 + u] = (live && e < E) ? e : 0x7fffffff;
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
#pragma unroll
  for (int r = 0; r < 8; ++r) ex[r] = r < k ? expf(sel_v[r] - ref) : 0.f;
  if (renorm) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < k) denom += ex[r];
  } else {
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (id[s] != 0x7fffffff) denom += expf(v[s] - ref);
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
  }
  *denom_out = denom;
}

template <int G>
__device__ __forceinline__ void select_token(const float (&v)[8], bool live, int E, int k, int renorm,
                                             float (&sel_v)[8], int (&sel_i)[8], float* denom_out) {
  float ex[8];
  select_token_ex<G>(v, live, E, k, renorm, sel_v, sel_i, ex, denom_out);
}

// Both steps for one token.
template <int G, bool VEC>
__device__ __forceinline__ void topk_token(const float* __restrict__ row, bool live, int E, int k, int renorm,
                                           float (&sel_v)[8], int (&sel_i)[8], float* denom_out) {
  float v[8];
  load_token<G, VEC>(row, live, E, v);
  select_token<G>(v, live, E, k, renorm, sel_v, sel_i, denom_out);
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

// ---- moe_route's kernel.  A group of G lanes owns a token, each lane up to
// 16 logits (float4 chunks gl, gl+G, gl+2G, gl+3G), so G = 1 up to E = 16.
// The rank count K is a template parameter (exactly K rounds).  A round: the
// group's largest remaining logit (float max over the lane's slots still in
// its mask, then a butterfly), then the lowest expert holding that value
// (each lane's lowest matching slot from a bitmask, then a butterfly min);
// the owning lane clears that slot's bit.  Equal logits -- including -0.0
// and +0.0, which compare equal -- go to the lower expert; a logit of -inf
// stays selectable, since removal is by mask, not by value.
template <int G, bool VEC>
__device__ __forceinline__ void load_token16(const float* __restrict__ row, bool live, int E, float (&v)[16],
                                             unsigned& valid) {
  const int gl = (threadIdx.x & 31) % G;
  valid = 0u;
#pragma unroll
  for (int s = 0; s < 16; ++s) v[s] = -INFINITY;
  if (!live) return;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int e0 = (gl + c * G) * 4;
    if (VEC) {
      if (e0 < E) {
        const float4 q = __ldg(reinterpret_cast<const float4*>(row + e0));
        v[c * 4 + 0] = q.x; v[c * 4 + 1] = q.y; v[c * 4 + 2] = q.z; v[c * 4 + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e0 + u < E) v[c * 4 + u] = __ldg(row + e0 + u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (e0 + u < E) valid |= 1u << (c * 4 + u);
  }
}

template <int G, int K>
__device__ __forceinline__ void select_k16(const float (&v)[16], unsigned valid, bool live, int E, int renorm,
                                           int (&sel_i)[K], float (&ex)[K], float* denom_out) {
  const int gl = (threadIdx.x & 31) % G;
  unsigned rem = valid;
  float sel_v[K];
#pragma unroll
  for (int r = 0; r < K; ++r) {
    float b = -INFINITY;
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if ((rem >> s) & 1u) b = fmaxf(b, v[s]);
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1) b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, off));
    unsigned m = 0u;
#pragma unroll
    for (int s = 0; s < 16; ++s) m |= (v[s] == b ? 1u : 0u) << s;
    m &= rem;
    // slot s holds expert (gl + (s/4)*G)*4 + s%4: lower slot, lower expert
    const int s0 = m ? __ffs(m) - 1 : 0;
    int id = m ? (gl + (s0 >> 2) * G) * 4 + (s0 & 3) : 0x7fffffff;
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1) id = min(id, __shfl_xor_sync(0xffffffffu, id, off));
    if (m && (gl + (s0 >> 2) * G) * 4 + (s0 & 3) == id) rem &= ~(1u << s0);
    sel_i[r] = id;
    sel_v[r] = b;
  }
  const float ref = sel_v[0];
  float denom = 0.f;
#pragma unroll
  for (int r = 0; r < K; ++r) ex[r] = expf(sel_v[r] - ref);
  if (renorm) {
#pragma unroll
    for (int r = 0; r < K; ++r) denom += ex[r];
  } else {
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if ((valid >> s) & 1u) denom += expf(v[s] - ref);
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
  }
  (void)live;
  (void)E;
  *denom_out = denom;
}

// One token per lane group; 8 warps * (32/G) tokens per block.
template <int G, bool VEC, int K>
__global__ void __launch_bounds__(kThreads) topk_kernel(const float* __restrict__ logits, int T, int E,
                                                        int renorm, int32_t* __restrict__ idx,
                                                        float* __restrict__ wout, int vec_store) {
  constexpr int TPW = 32 / G;
  const int lane = threadIdx.x & 31, gl = lane % G;
  const long long t = (((long long)blockIdx.x * kThreads + threadIdx.x) >> 5) * TPW + lane / G;
  const bool live = t < T;
  float v[16], ex[K], denom;
  unsigned valid;
  int sel_i[K];
  load_token16<G, VEC>(logits + (size_t)(live ? t : 0) * E, live, E, v, valid);
  select_k16<G, K>(v, valid, live, E, renorm, sel_i, ex, &denom);
  if (!live) return;
  if (G == 1 && (K == 2 || K == 4 || K == 8) && vec_store) {
    // one lane holds the whole token: its K indices and weights as vector
    // stores (K * 4 bytes at t * K * 4; vec_store says idx and w are
    // 16-byte aligned)
#pragma unroll
    for (int r = 0; r < K; r += (K == 2 ? 2 : 4)) {
      if (K == 2) {
        *reinterpret_cast<int2*>(idx + (size_t)t * K + r) = make_int2(sel_i[r], sel_i[r + 1]);
        *reinterpret_cast<float2*>(wout + (size_t)t * K + r) = make_float2(ex[r] / denom, ex[r + 1] / denom);
      } else {
        *reinterpret_cast<int4*>(idx + (size_t)t * K + r) =
            make_int4(sel_i[r], sel_i[r + 1], sel_i[r + 2], sel_i[r + 3]);
        *reinterpret_cast<float4*>(wout + (size_t)t * K + r) =
            make_float4(ex[r] / denom, ex[r + 1] / denom, ex[r + 2] / denom, ex[r + 3] / denom);
      }
    }
    return;
  }
#pragma unroll
  for (int r = 0; r < K; ++r) {
    if ((r % G) == gl) {
      idx[(size_t)t * K + r] = sel_i[r];
      wout[(size_t)t * K + r] = ex[r] / denom;
    }
  }
}

template <int G, int K>
static cudaError_t launch_gk(const float* logits, int T, int E, int renorm, int32_t* idx, float* w, cudaStream_t st) {
  constexpr int tokens_per_block = (kThreads / 32) * (32 / G);
  const long long blocks = ((long long)T + tokens_per_block - 1) / tokens_per_block;
  const bool vec = (E % 4 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  const int vst = ((reinterpret_cast<uintptr_t>(idx) | reinterpret_cast<uintptr_t>(w)) & 15) == 0 ? 1 : 0;
  if (vec)
    topk_kernel<G, true, K><<<(unsigned)blocks, kThreads, 0, st>>>(logits, T, E, renorm, idx, w, vst);
  else
    topk_kernel<G, false, K><<<(unsigned)blocks, kThreads, 0, st>>>(logits, T, E, renorm, idx, w, vst);
  return cudaGetLastError();
}

template <int G>
static cudaError_t launch_g(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                            cudaStream_t st) {
  switch (k) {
    case 1: return launch_gk<G, 1>(logits, T, E, renorm, idx, w, st);
    case 2: return launch_gk<G, 2>(logits, T, E, renorm, idx, w, st);
    case 3: return launch_gk<G, 3>(logits, T, E, renorm, idx, w, st);
    case 4: return launch_gk<G, 4>(logits, T, E, renorm, idx, w, st);
    case 5: return launch_gk<G, 5>(logits, T, E, renorm, idx, w, st);
    case 6: return launch_gk<G, 6>(logits, T, E, renorm, idx, w, st);
    case 7: return launch_gk<G, 7>(logits, T, E, renorm, idx, w, st);
    default: return launch_gk<G, 8>(logits, T, E, renorm, idx, w, st);
  }
}

// Lanes per token for moe_route: smallest power of two with G*16 >= E.
static cudaError_t launch(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                          cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (E <= 16) return launch_g<1>(logits, T, E, k, renorm, idx, w, st);
  if (E <= 32) return launch_g<2>(logits, T, E, k, renorm, idx, w, st);
  if (E <= 64) return launch_g<4>(logits, T, E, k, renorm, idx, w, st);
  if (E <= 128) return launch_g<8>(logits, T, E, k, renorm, idx, w, st);
  return launch_g<16>(logits, T, E, k, renorm, idx, w, st);
}

}  // namespace route

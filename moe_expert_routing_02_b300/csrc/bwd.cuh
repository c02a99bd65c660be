// Backward of the routed expert layer around the GEMMs: the padded row
// layout, the gather of the backward's row operands, the token gradient and
// the gate's gradient.
//
// PopFetcher (ATC'25) review: the system trains MoE models, so every step of
// the forward layer has a backward.  The forward steps being inverted are
// EPS-MoE's LocalReduce (combine: out[t] = sum_r w[t,r] Y[slot(t,r)]), the
// dispatch copy (xp[slot] = x[t]) and the top-k gate of the PopFetcher and
// EPS-MoE reviews (softmax weights over the chosen experts, or over all).
//
// Padded row space: the rows of each unit (an expert's adjacent groups) are
// laid out from a multiple of 64 and padded with zero rows to a multiple of
// 64.  Every 64-row block then holds one expert, so the weight gradients
// (ffn_wgrad.cuh) need no masking, and every intermediate of the backward
// GEMMs is exactly zero on the padding rows.
#pragma once
#include <climits>
#include "common.cuh"

namespace bwd {

constexpr int kMaxG = 512;
constexpr int kLayoutThreads = 512;

// One block.  Units as in the forward GEMMs: maximal runs of consecutive
// groups of one expert.  Outputs, with U units:
//   pgoff[0..G]   padded first row of unit u (u <= U); pgoff[u > U] = pgoff[U]
//   pue[0..G-1]   expert of unit u (u < U), -1 after
//   ustart[0..G]  first dispatched row of unit u; ustart[u > U] = ustart[U]
//   pbeg[e], pcnt[e]  the padded range of expert e (0, 0 when it has no rows)
// An expert with rows in two units, an expert outside [0, E) with rows, and
// offsets outside [0, A] or decreasing are flagged as invalid device data.
__global__ void __launch_bounds__(kLayoutThreads)
    layout_kernel(const int32_t* goff_in, const int32_t* gexp, int G, int E, int A, int32_t* pgoff, int32_t* pue,
                  int32_t* ustart, int32_t* pbeg, int32_t* pcnt) {
  __shared__ int32_t goff[kMaxG + 1];
  __shared__ int32_t us[kMaxG + 1];
  __shared__ int32_t ue[kMaxG];
  __shared__ int32_t pst[kMaxG + 1];
  __shared__ int32_t owner[256];
  __shared__ int32_t U_s;
  const int lane = threadIdx.x & 31;
  for (int g = threadIdx.x; g <= G; g += blockDim.x) {
    int v = goff_in[g];
    if (v < 0 || v > A) {
      moe_flag_error(MOE_DEVERR_DATA);
      v = v < 0 ? 0 : A;
    }
    goff[g] = v;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) owner[e] = -1;
  __syncthreads();
  if (threadIdx.x == 0) {
    // decreasing offsets are invalid data; clamping them to a running maximum
    // keeps the units' rows within [0, A], so the padded space fits its bound
    for (int g = 1; g <= G; ++g)
      if (goff[g] < goff[g - 1]) {
        moe_flag_error(MOE_DEVERR_DATA);
        goff[g] = goff[g - 1];
      }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    int carry = 0, prev_e = INT_MIN;
    for (int c0 = 0; c0 < G; c0 += 32) {
      const int g = c0 + lane;
      int e = INT_MIN;
      if (g < G) e = gexp ? gexp[g] : g;
      int pe = __shfl_up_sync(0xffffffffu, e, 1);
      if (lane == 0) pe = prev_e;
      const bool start = g < G && (g == 0 || e != pe);
      const unsigned starts = __ballot_sync(0xffffffffu, start);
      const int u = carry + __popc(starts & ((1u << lane) - 1u));
      if (start) {
        us[u] = goff[g];
        ue[u] = e;
      }
      carry += __popc(starts);
      prev_e = __shfl_sync(0xffffffffu, e, 31);
    }
    if (lane == 0) {
      us[carry] = goff[G];
      U_s = carry;
    }
    __syncwarp();
    // padded prefix over units
    const int U = carry;
    int run = 0;
    for (int c0 = 0; c0 < U; c0 += 32) {
      const int u = c0 + lane;
      int v = 0;
      if (u < U) {
        const int rows = us[u + 1] - us[u];
        v = rows > 0 ? (rows + 63) & ~63 : 0;
      }
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int w = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += w;
      }
      if (u < U) pst[u] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pst[U] = run;
  }
  __syncthreads();
  const int U = U_s;
  for (int u = threadIdx.x; u < U; u += blockDim.x) {
    const int rows = us[u + 1] - us[u];
    int e = ue[u];
    if (rows > 0) {
      if (e < 0 || e >= E) {
        moe_flag_error(MOE_DEVERR_DATA);
        e = -1;
      } else if (atomicCAS(&owner[e], -1, u) != -1) {
        moe_flag_error(MOE_DEVERR_DATA);  // the expert's rows are not adjacent
        e = -1;
      }
    } else if (e < 0 || e >= E) {
      e = -1;
    }
    ue[u] = e;
  }
  __syncthreads();
  for (int u = threadIdx.x; u <= G; u += blockDim.x) {
    pgoff[u] = pst[u <= U ? u : U];
    ustart[u] = us[u <= U ? u : U];
    if (u < G) pue[u] = u < U ? ue[u] : -1;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int u = owner[e];
    if (u >= 0 && ue[u] == e) {
      pbeg[e] = pst[u];
      pcnt[e] = pst[u + 1] - pst[u];
    } else {
      pbeg[e] = 0;
      pcnt[e] = 0;
    }
  }
}

// One warp per padded row pr < pgoff[G].  A real row (dispatched row i of
// unit u) takes token t = perm[i] / k, rank r = perm[i] % k:
//   xp[pr] = x[t];  dy[pr] = bf16(w[t,r] dout[t]);  prow[i] = pr;
//   dw[t,r] = <dout[t], y[i]>   (fp32; only when y is given)
// A padding row gets zeros in xp and dy.
__global__ void __launch_bounds__(256)
    gather_kernel(const int32_t* pgoff_in, const int32_t* ustart_in, int G, const int32_t* perm, int T, int k,
                  const uint16_t* x, const uint16_t* dout, const float* w, const uint16_t* y, int H, uint16_t* xp,
                  uint16_t* dy, float* dw, int32_t* prow) {
  __shared__ int32_t pgoff[kMaxG + 1];
  __shared__ int32_t ustart[kMaxG + 1];
  for (int g = threadIdx.x; g <= G; g += blockDim.x) {
    pgoff[g] = pgoff_in[g];
    ustart[g] = ustart_in[g];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int P = pgoff[G];
  const int H8 = H >> 3;
  const long long A = (long long)T * k;
  for (long long pr = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pr < P;
       pr += (long long)gridDim.x * (blockDim.x >> 5)) {
    int lo = 0, hi = G;  // last u with pgoff[u] <= pr
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pgoff[mid] <= pr) lo = mid; else hi = mid;
    }
    const int local = (int)(pr - pgoff[lo]);
    const int rows = ustart[lo + 1] - ustart[lo];
    uint4* xo = reinterpret_cast<uint4*>(xp + pr * H);
    uint4* yo = reinterpret_cast<uint4*>(dy + pr * H);
    int f = -1;
    if (local < rows) {
      const int i = ustart[lo] + local;
      f = perm[i];
      if (f < 0 || f >= A) {
        moe_flag_error(MOE_DEVERR_DATA);
        f = -1;
      } else if (lane == 0) {
        prow[i] = (int32_t)pr;
      }
    }
    if (f < 0) {
      for (int c = lane; c < H8; c += 32) {
        xo[c] = make_uint4(0, 0, 0, 0);
        yo[c] = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    const int t = f / k;
    const float wt = w[f];
    const uint4* xi = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const uint4* gi = reinterpret_cast<const uint4*>(dout + (size_t)t * H);
    const uint4* yi = y ? reinterpret_cast<const uint4*>(y + (size_t)(ustart[lo] + local) * H) : nullptr;
    float dot = 0.f;
    for (int c = lane; c < H8; c += 32) {
      xo[c] = ld_nc_v4(xi + c);
      const uint4 g = ld_nc_v4(gi + c);
      const uint32_t gv[4] = {g.x, g.y, g.z, g.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = pack_bf16x2(wt * bf16lo(gv[q]), wt * bf16hi(gv[q]));
      yo[c] = make_uint4(o[0], o[1], o[2], o[3]);
      if (yi) {
        const uint4 yy = ld_nc_v4(yi + c);
        const uint32_t yv[4] = {yy.x, yy.y, yy.z, yy.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dot = fmaf(bf16lo(gv[q]), bf16lo(yv[q]), dot);
          dot = fmaf(bf16hi(gv[q]), bf16hi(yv[q]), dot);
        }
      }
    }
    if (yi) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      if (lane == 0) dw[f] = dot;
    }
  }
}

// dx[t] = sum_r dxp[prow[inv_perm[t k + r]]], fp32 in r order, one bf16
// rounding (the backward of the dispatch copy).  One warp per token.
__global__ void __launch_bounds__(256)
    scatter_kernel(const uint16_t* dxp, const int32_t* prow, const int32_t* inv_perm, int T, int k, int H,
                   long long P_rows, uint16_t* dx) {
  const int lane = threadIdx.x & 31;
  const int H8 = H >> 3;
  const long long A = (long long)T * k;
  for (long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
       t += (long long)gridDim.x * (blockDim.x >> 5)) {
    int src[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      src[r] = -1;
      if (r < k) {
        const int i = inv_perm[t * k + r];
        int pr = (i >= 0 && i < A) ? prow[i] : -1;
        if (pr < 0 || pr >= P_rows) {
          if (lane == 0) moe_flag_error(MOE_DEVERR_DATA);
          pr = -1;
        }
        src[r] = pr;
      }
    }
    for (int c = lane; c < H8; c += 32) {
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r < k && src[r] >= 0) {
          const uint4 v = ld_nc_v4(reinterpret_cast<const uint4*>(dxp + (size_t)src[r] * H) + c);
          acc[0] += bf16lo(v.x);
          acc[1] += bf16hi(v.x);
          acc[2] += bf16lo(v.y);
          acc[3] += bf16hi(v.y);
          acc[4] += bf16lo(v.z);
          acc[5] += bf16hi(v.z);
          acc[6] += bf16lo(v.w);
          acc[7] += bf16hi(v.w);
        }
      }
      reinterpret_cast<uint4*>(dx + (size_t)t * H)[c] =
          make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                     pack_bf16x2(acc[6], acc[7]));
    }
  }
}

// Gradient of the gate weights with respect to the router logits, the chosen
// experts held fixed.  One thread per token (the work per token is a few
// dependent loads and k..E exponentials, so a warp per token leaves most
// lanes idle and the grid latency-bound), fp32.
//   renorm: w_r = softmax over the chosen logits;
//           dl[e_r] = w_r (dw_r - sum_s w_s dw_s), 0 for the other experts
//   full:   w_r = p[e_r], p = softmax over all E logits;
//           dl[j] = p_j (g_j - sum_r dw_r p[e_r]), g_j = dw_r if j = e_r else 0
__global__ void __launch_bounds__(256)
    route_bwd_kernel(const float* logits, const int32_t* idx, const float* dwt, int T, int E, int k, int renorm,
                     float* dl) {
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < T; t += (long long)gridDim.x * blockDim.x) {
    const float* l = logits + t * E;
    float* o = dl + t * E;
    int e[8];
    float d[8], lr[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      e[r] = 0;
      d[r] = 0.f;
      if (r < k) {
        e[r] = idx[t * k + r];
        if (e[r] < 0 || e[r] >= E) {
          moe_flag_error(MOE_DEVERR_DATA);
          e[r] = 0;
        }
        d[r] = dwt[t * k + r];
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) lr[r] = r < k ? l[e[r]] : -INFINITY;
    if (renorm) {
      float m = lr[0];
#pragma unroll
      for (int r = 1; r < 8; ++r) m = fmaxf(m, lr[r]);
      float z[8], sum = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        z[r] = r < k ? expf(lr[r] - m) : 0.f;
        sum += z[r];
      }
      float c = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        z[r] /= sum;  // w_r
        c = fmaf(z[r], d[r], c);
      }
      for (int j = 0; j < E; ++j) o[j] = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < k) o[e[r]] = z[r] * (d[r] - c);
    } else {
      float m = -INFINITY;
      for (int j = 0; j < E; ++j) m = fmaxf(m, l[j]);
      float sum = 0.f;
      for (int j = 0; j < E; ++j) sum += expf(l[j] - m);
      const float inv = 1.0f / sum;
      float c = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < k) c = fmaf(d[r], expf(lr[r] - m) * inv, c);
      for (int j = 0; j < E; ++j) {
        float g = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < k && e[r] == j) g = d[r];
        o[j] = expf(l[j] - m) * inv * (g - c);
      }
    }
  }
}

}  // namespace bwd

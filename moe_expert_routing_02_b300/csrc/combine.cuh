// K7: gate-weighted combine of each token's k expert outputs.
//
// EPS-MoE review, compute/communication overlap: the LocalReduce of expert
// outputs is a memory-bound step; PopFetcher review: result collect.
//   out[t] = sum_{r<k} w[t,r] * y[inv_perm[t*k+r]]
// One warp per token row; each lane owns 16-byte chunks (8 bf16), issues the
// k gathered row loads of several chunks before accumulating each chunk in
// fp32 in rank order r = 0..k-1, rounding once to bf16.  Bound by HBM
// bandwidth: A*H*2 bytes read, T*H*2 written, plus the small index/weight reads.
#pragma once
#include "common.cuh"

namespace combine {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// The row's chunks are taken NC at a time (NC * K <= 8 loads of 16 bytes in
// flight per lane, all issued before any is used), so a warp keeps a whole
// 1024-wide row of top-2 outputs in flight instead of one chunk per lane.
template <int K>
__device__ __forceinline__ void combine_row(const uint16_t* __restrict__ y, const long long* slot, const float* wr,
                                            int H, uint16_t* __restrict__ dst, int lane) {
  constexpr int NC = K <= 2 ? 4 : (K <= 4 ? 2 : 1);
  const int chunks = H / 8;
  for (int c0 = lane; c0 < chunks; c0 += 32 * NC) {
    uint4 v[NC][K];
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = c0 + 32 * j;
#pragma unroll
      for (int r = 0; r < K; ++r)
        if (c < chunks) v[j][r] = ld_nc_v4(y + slot[r] * H + (size_t)c * 8);
    }
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = c0 + 32 * j;
      if (c >= chunks) break;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
      for (int r = 0; r < K; ++r) {
        const uint32_t u[4] = {v[j][r].x, v[j][r].y, v[j][r].z, v[j][r].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(wr[r], bf16lo(u[i]), acc[2 * i]);
          acc[2 * i + 1] = fmaf(wr[r], bf16hi(u[i]), acc[2 * i + 1]);
        }
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      st_v4(dst + (size_t)c * 8, o);
    }
  }
}

template <int K>
__global__ void __launch_bounds__(kThreads) combine_kernel(const uint16_t* __restrict__ y,
                                                           const int32_t* __restrict__ inv_perm,
                                                           const float* __restrict__ w, long long T, int H,
                                                           long long A, uint16_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * kWarps;
  pdl_wait();
  for (long long t = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5; t < T; t += warps) {
    long long slot[K];
    float wr[K];
    bool ok = true;
#pragma unroll
    for (int r = 0; r < K; ++r) {
      const int32_t s = inv_perm[t * K + r];
      ok &= (unsigned long long)s < (unsigned long long)A;
      slot[r] = ok ? s : 0;
      wr[r] = w[t * K + r];
    }
    if (!ok) {  // hole left by invalid routing (flagged upstream)
      if (lane == 0) moe_flag_error(MOE_DEVERR_DATA);
      continue;
    }
    combine_row<K>(y, slot, wr, H, out + t * H, lane);
  }
}

static cudaError_t launch(const uint16_t* y, const int32_t* inv_perm, const float* w, long long T, int k, int H,
                          uint16_t* out, int num_sms, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  long long blocks = (T + kWarps - 1) / kWarps;
  const long long cap = (long long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  const long long A = T * k;
  switch (k) {
#define MOE_COMBINE_CASE(KK) \
  case KK: return launch_pdl(combine_kernel<KK>, dim3((unsigned)blocks), dim3(kThreads), 0, st, y, inv_perm, w, T, \
                             H, A, out);
    MOE_COMBINE_CASE(1)
    MOE_COMBINE_CASE(2)
    MOE_COMBINE_CASE(3)
    MOE_COMBINE_CASE(4)
    MOE_COMBINE_CASE(5)
    MOE_COMBINE_CASE(6)
    MOE_COMBINE_CASE(7)
    MOE_COMBINE_CASE(8)
#undef MOE_COMBINE_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// The combine fused into the FFN's second GEMM leaves its sums in an fp32
// [T, H] accumulator; this rounds them once to bf16 (8 values per thread).
__global__ void __launch_bounds__(kThreads) finalize_kernel(const float* __restrict__ acc, long long n8,
                                                           uint16_t* __restrict__ out) {
  pdl_wait();
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < n8; i += (long long)gridDim.x * kThreads) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    reinterpret_cast<uint4*>(out)[i] =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
}

static cudaError_t launch_finalize(const float* acc, long long T, int H, uint16_t* out, int num_sms, cudaStream_t st) {
  const long long n8 = T * H / 8;
  if (n8 == 0) return cudaSuccess;
  long long blocks = (n8 + kThreads - 1) / kThreads;
  if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
  return launch_pdl(finalize_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, st, acc, n8, out);
}

}  // namespace combine

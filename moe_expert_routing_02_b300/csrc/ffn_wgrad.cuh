// Weight gradients of the grouped expert FFN (backward of K6) on tcgen05.
//
// PopFetcher (ATC'25) review: the system trains MoE models; its core method
// and design trade-offs state that the backward pass of a replicated expert
// sends the copies' gradients back to the primary expert and reduces them
// there.  On one GPU that reduction is the sum over every row routed to the
// expert, whichever replica group served the row:
//
//   dW[e] = L_e^T R_e    [M_out, N_out], fp32 (or dW[e] += ..., accumulate;
//                         or rounded once to bf16),
//
// where L_e [rows_e, M_out] and R_e [rows_e, N_out] are expert e's rows of two
// row-major bf16 activation tensors (the reduction runs over rows).  The rows
// of an expert form one range of a padded row space: it starts at a multiple
// of 64 and its length is padded with zero rows to a multiple of 64, so every
// 64-row k-block belongs to one expert and no tail needs masking.  Up to three
// "jobs" (GeLU: dW2 and dW1; SwiGLU: dW2, dW1 and dW3) share one persistent
// launch; tiles run expert-major, so the CTAs working at the same time read
// the same expert's rows (L2 reuse across jobs and tiles).
//
// Per CTA (one per SM), the roles of ffn::gemm_kernel:
//   warp 0      TMA producer: A tile = 64 rows x 128 columns of L (two
//               64x64 boxes), B tile = 64 rows x 256 columns of R (four
//               boxes); both MN-major with the 128-byte swizzle.
//   warp 1      MMA issuer (M=128, N=256, K=16, both operands MN-major),
//               two TMEM accumulators.
//   warps 2..17 epilogue: fp32 results, 8 rows x 128 bytes per store
//               instruction through a staging buffer.
// Every wait is bounded as in ffn::gemm_kernel.
#pragma once
#include "ffn.cuh"

namespace ffn_wg {

using namespace sm100;
using ffn::A_BYTES;
using ffn::B_BOX_BYTES;
using ffn::B_BYTES;
using ffn::BK;
using ffn::BM;
using ffn::BN;
using ffn::EPI_SLICES;
using ffn::EPI_WARPS;
using ffn::STAGES;
using ffn::THREADS;
using ffn::TMEM_COLS;
using ffn::wait_phase;

constexpr int MAX_JOBS = 3;
constexpr int MAX_E = 256;

struct Job {
  void* out;          // [E, M_out, N_out] fp32, or bf16 with out_bf16
  int M_out, N_out;   // multiples of 64
  int m_tiles, n_tiles;
  int a_col0, b_col0;  // first column of the job's L and R in their tensors
};

struct Maps {
  CUtensorMap a[MAX_JOBS];  // L tensors, box 64 columns x 64 rows
  CUtensorMap b[MAX_JOBS];  // R tensors, box 64 columns x 64 rows
};

struct WParams {
  const int32_t* pbeg;  // [E] first row of expert e's range (multiple of 64)
  const int32_t* pcnt;  // [E] rows of the range (multiple of 64; 0 = no rows, dW[e] = 0)
  int E;
  int jobs;
  int tiles_per_expert;  // sum over jobs of m_tiles * n_tiles
  long long rows;        // rows of the operand tensors
  int accumulate;        // 1: dW += result (gradient accumulation), 0: dW = result
  int out_bf16;          // 1: results rounded once to bf16 (no accumulation)
  Job job[MAX_JOBS];
};

struct Smem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  int32_t krow[MAX_E];  // first row of each expert's range
  int32_t kbn[MAX_E];   // its k-blocks
  alignas(128) uint8_t stg[EPI_WARPS][1024];
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory beyond the 227 KB per-block opt-in limit");
static_assert(offsetof(Smem, b) % 1024 == 0 && offsetof(Smem, stg) % 128 == 0, "stage buffers misaligned");

struct WTile {
  int e, j, mt, nt;
};

__device__ __forceinline__ WTile wdecode(const WParams& p, int tile) {
  WTile t;
  t.e = tile / p.tiles_per_expert;
  int r = tile - t.e * p.tiles_per_expert;
  int j = 0;
  while (j + 1 < p.jobs && r >= p.job[j].m_tiles * p.job[j].n_tiles) {
    r -= p.job[j].m_tiles * p.job[j].n_tiles;
    ++j;
  }
  t.j = j;
  t.nt = r / p.job[j].m_tiles;  // m fastest: CTAs side by side share the R columns
  t.mt = r - t.nt * p.job[j].m_tiles;
  return t;
}

// Lane i holds row i's 32 fp32 columns; rows >= rows_valid are not written.
// Through 1 KB of shared memory, 8 rows at a time: chunk j (16 bytes) of row
// r sits at slot (j + r) mod 8, so the writes (8 lanes, one row each) and the
// reads (8 lanes per row, one 128-byte row segment per 8 lanes) are free of
// bank conflicts.  accumulate: each 16-byte chunk is added to what the output
// holds (read with the same coalesced pattern) instead of replacing it.
__device__ __forceinline__ void store_rows32_f32(uint8_t* stg, float* out, size_t ld, int rows_valid,
                                                 const uint32_t (&v)[32], int lane, bool accumulate) {
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    __syncwarp();
    if ((lane >> 3) == h) {
      const int r = lane & 7;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(stg + r * 128 + (((j + r) & 7) << 4)) =
            make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    __syncwarp();
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int idx = pass * 32 + lane;
      const int r = idx >> 3, c = idx & 7;
      uint4 q = *reinterpret_cast<const uint4*>(stg + r * 128 + (((c + r) & 7) << 4));
      const int row = h * 8 + r;
      if (row < rows_valid) {
        float* dst = out + (size_t)row * ld + c * 4;
        if (accumulate) {
          const float4 o = *reinterpret_cast<const float4*>(dst);
          q = make_uint4(__float_as_uint(o.x + __uint_as_float(q.x)), __float_as_uint(o.y + __uint_as_float(q.y)),
                         __float_as_uint(o.z + __uint_as_float(q.z)), __float_as_uint(o.w + __uint_as_float(q.w)));
        }
        st_v4(dst, q);
      }
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1)
    wgrad_kernel(const __grid_constant__ Maps m, const __grid_constant__ WParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem& s = *reinterpret_cast<Smem*>(base);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // ---- each expert's row range, checked against the tensors
  for (int e = threadIdx.x; e < p.E; e += THREADS) {
    const long long b = p.pbeg[e], c = p.pcnt[e];
    if (c == 0) {
      s.krow[e] = 0;
      s.kbn[e] = 0;
    } else if (b < 0 || c < 0 || (b & 63) || (c & 63) || b + c > p.rows) {
      moe_flag_error(MOE_DEVERR_DATA);
      s.krow[e] = 0;
      s.kbn[e] = 0;
    } else {
      s.krow[e] = (int32_t)b;
      s.kbn[e] = (int32_t)(c / BK);
    }
  }
  const int total = p.E * p.tiles_per_expert;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], EPI_WARPS);
    }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_mbar_init();
    for (int j = 0; j < p.jobs; ++j) {
      tma_prefetch_desc(&m.a[j]);
      tma_prefetch_desc(&m.b[j]);
    }
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(&s.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const WTile t = wdecode(p, tile);
        const Job& J = p.job[t.j];
        const CUtensorMap* ma = &m.a[t.j];
        const CUtensorMap* mb = &m.b[t.j];
        const int kbn = s.kbn[t.e];
        const int krow = s.krow[t.e];
        const int ax = J.a_col0 + t.mt * BM;
        const int bx = J.b_col0 + t.nt * BN;
        for (int kb = 0; kb < kbn; ++kb) {
          if (!wait_phase(&s.empty[stage], phase ^ 1, &s.abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.full[stage], A_BYTES + B_BYTES);
          const int y = krow + kb * BK;
#pragma unroll
          for (int c = 0; c < BM / 64; ++c) tma_load_2d(s.a[stage] + c * B_BOX_BYTES, ma, &s.full[stage], ax + 64 * c, y);
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) tma_load_2d(s.b[stage] + c * B_BOX_BYTES, mb, &s.full[stage], bx + 64 * c, y);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      for (uint32_t st = 0; st < (uint32_t)STAGES; ++st) {
        if (issued > st) {
          const uint32_t last = issued - 1 - ((issued - 1 - st) % STAGES);
          wait_phase(&s.full[st], (last / STAGES) & 1u, &s.abort_flag, true);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, true, true);
      // both operands MN-major: 64-column boxes 8 KB apart (LBO), 8 k-rows
      // 1024 B apart (SBO); a K step of 16 rows is 2048 B (+128 in the field)
      const uint64_t adesc0 = smem_desc_sw128(smem_u32(s.a[0]), B_BOX_BYTES, 1024);
      const uint64_t bdesc0 = smem_desc_sw128(smem_u32(s.b[0]), B_BOX_BYTES, 1024);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, any_mma = false;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const WTile t = wdecode(p, tile);
        const int kbn = s.kbn[t.e];
        if (!wait_phase(&s.tempty[acc], acc_phase ^ 1, &s.abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < kbn; ++kb) {
          if (!wait_phase(&s.full[stage], phase, &s.abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = adesc0 + (uint64_t)(stage * (A_BYTES >> 4));
          const uint64_t bd = bdesc0 + (uint64_t)(stage * (B_BYTES >> 4));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16(d, ad + (uint64_t)(kk * 128), bd + (uint64_t)(kk * 128), idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit(&s.empty[stage]);
          any_mma = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        // an expert without rows commits no MMA: the epilogue writes zeros
        mma_commit(&s.tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (any_mma) {
        mma_commit(&s.drain);
        wait_phase(&s.drain, 0, &s.abort_flag, true);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int slice = (warp - 2) >> 2;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const WTile t = wdecode(p, tile);
      const Job& J = p.job[t.j];
      const bool empty = s.kbn[t.e] == 0;
      if (!__all_sync(0xffffffffu, wait_phase(&s.tfull[acc], acc_phase, &s.abort_flag))) break;
      tc_fence_after();
      const int row0 = t.mt * BM + quarter * 32;
      const int wrows = J.M_out - row0;
      const size_t ooff = ((size_t)t.e * J.M_out + row0) * J.N_out;
      const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      constexpr int W = BN / EPI_SLICES;
#pragma unroll 1
      for (int cc = 0; cc < W; cc += 32) {
        const int c = slice * W + cc;
        const int col = t.nt * BN + c;
        uint32_t raw[32];
        if (empty) {
#pragma unroll
          for (int i = 0; i < 32; ++i) raw[i] = 0;
        } else {
          __syncwarp();
          tmem_ld32(tb + c, raw);
        }
        if (col < J.N_out && wrows > 0) {
          if (p.out_bf16) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1]));
            ffn::store_rows32(s.stg[warp - 2], static_cast<uint16_t*>(J.out) + ooff + col, (size_t)J.N_out, wrows, pk,
                              lane);
          } else {
            store_rows32_f32(s.stg[warp - 2], static_cast<float*>(J.out) + ooff + col, (size_t)J.N_out, wrows, raw,
                             lane, p.accumulate != 0);
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace ffn_wg

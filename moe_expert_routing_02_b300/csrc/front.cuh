// Fused front of the layer: top-k gate, token statistics and window, next-layer
// prediction, replica counts and the dispatch, in two launches.
//
// Same results as moe_route -> moe_stats_update -> moe_predict ->
// moe_replicate -> moe_dispatch (PopFetcher review: gate, Routing Information
// Collector with Eq. (1)-(3); MoE-GPS blog section 2.1 duplicate_experts;
// MoE-MPMC summary, replica dispatch), with five fewer launches:
//
//   F1 (route_count_kernel), one block per tiles_per_block tiles of TT tokens:
//      top-k of each token (route::topk_token), idx / w written; per tile the
//      expert counts (shared atomics), written as the tile's exclusive prefix
//      within the block, and the block's totals (blk_tot, and added to the
//      histogram accumulator and to the totals of the block's segment of
//      kSegBlocks route blocks); the co-selection pairs with the previous
//      layer's routing (shared atomics, flushed to the window state's
//      accumulator).
//   F2 (scatter_copy_kernel), one block per tile plus one statistics block.
//      Every block first issues all its independent loads at once (the
//      histogram; for a tile, its prefix, the segment and block totals before
//      it, its first expert ids).  The statistics block folds the histogram
//      and the co-selection counts into the window ring and sums (as
//      stats::update_kernel does) and predicts the next layer
//      (stats::predict_block); the dispatch reads none of that, so it runs
//      beside the tiles.  Each tile block computes the replica counts and the
//      group layout itself -- O(E) integer work, the same in every block: one
//      scan for replicas from the histogram, the block forms
//      (replicate::replicate_block, after replicate::apportion_block for a
//      predicted popularity) with a copies budget -- then the tile's starting
//      rank per expert, stable in-tile ranks -> slots -> perm / inv_perm, and
//      the copy of the rows of the tile's assignments to their slots with
//      16-byte vectors.  For short rows the route blocks let this kernel
//      start as soon as they passed their own wait, and each tile block first
//      asks L2 for its token rows, so that read overlaps the routing and the
//      plan.  The paths few blocks take (statistics, budget or shares, table
//      writes) are out of line: the code every tile block runs stays compact,
//      which measured ~3 us shorter than with everything inlined.
// No block waits for a single planner: the plan that one block used to run
// after all the routing (histogram fold, prediction, replica table, layout)
// is spread over the blocks that need it.  Counts are integers, so nothing
// depends on the order of atomics.
#pragma once
#include "common.cuh"
#include "dispatch.cuh"
#include "replicate.cuh"
#include "route.cuh"
#include "sm100_ptx.cuh"
#include "stats.cuh"

namespace front {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSmemCoselMaxE = 64;

// Tokens per dispatch tile, from T alone (so workspace sizes need no device):
// the smallest power of two in [16, 128] giving at most 512 tiles.
__host__ __device__ inline int tile_tokens(long long T) {
  int tt = 16;
  while (tt < 128 && (T + tt - 1) / tt > 512) tt <<= 1;
  return tt;
}
__host__ inline long long num_tiles(long long T) { return (T + tile_tokens(T) - 1) / tile_tokens(T); }
// Route blocks: at most kMaxRouteBlocks (the F2 prologue reads the totals
// of the blocks before its own), and at least one pass of every warp.
constexpr int kMaxRouteBlocks = 128;
// Route blocks are grouped in segments of kSegBlocks; each route block also
// adds its totals to its segment's, so a tile's starting ranks need at most
// kSegments - 1 segment totals and kSegBlocks - 1 block totals.
constexpr int kSegBlocks = 8;
constexpr int kSegments = kMaxRouteBlocks / kSegBlocks;
// Those totals are loaded kPreLoads per thread at once (more in a loop).
constexpr int kPreLoads = 8;
// The one-launch front (front_coop_kernel) groups tiles in segments of
// kSegTiles; the statistics handle keeps kSegSlots segment rows, enough for
// both forms (the one-launch front runs at most kSegTiles * kSegSlots tiles).
constexpr int kSegTiles = 32;
constexpr int kSegSlots = 32;
static_assert(kSegSlots >= kSegments, "segment rows of the two-launch front");
// Workspace: tile prefixes [ntiles][E], block totals [<= ntiles][E] (the
// size keeps room for [4][E] more words).
__host__ inline size_t workspace_bytes(long long T, int E) {
  const long long nt = num_tiles(T) > 0 ? num_tiles(T) : 1;
  return (size_t)(2 * nt * E + 4LL * E) * sizeof(int32_t);
}

struct Args {
  // route
  const float* logits;
  int T, E, k, renorm;
  int32_t* idx;
  float* w;
  // window update (pointers into the stats handle for this layer / pair)
  int has_prev;
  const int32_t* idx_prev;
  uint32_t* acc_h;   // [E] histogram accumulator (zero between calls)
  uint32_t* acc_c;   // [E*E] co-selection accumulator (zero between calls)
  uint32_t* seg_tot; // [kSegSlots][E] totals per segment of route blocks or tiles (zero between calls)
  uint32_t* ticket;  // F2 blocks that left (zero between calls)
  uint32_t* arrive;  // blocks past the routing of the one-launch front (zero between calls)
  uint32_t* ring_h;
  unsigned long long* hsum;
  uint32_t* ring_c;
  unsigned long long* csum;
  int32_t* hist_out;
  // prediction (p_seq == null: skipped); pred_csum null for the last layer
  const unsigned long long* pred_csum;
  float* p_seq;
  float* cond;
  float* p_next;
  // replication
  int replicate, num, den, max_copies, budget;
  const float* rep_share;  // [E] shares for the replica decision, or null (own histogram)
  int32_t* copies;
  int32_t* rep_base;
  int32_t* group_expert;
  // dispatch
  int TT;            // tokens per tile
  int tiles_per_block;
  long long ntiles;
  int32_t* counts;   // [ntiles][E]: tile's exclusive prefix within its route block
  int32_t* blk_tot;  // [route blocks][E]: block totals
  int32_t* group_offsets;
  int release_early;  // route blocks let the scatter/copy kernel start once they passed their wait
};

// The layer's co-selection counts into window ring slot and sums (pair j-1, j).
__device__ __forceinline__ void fold_cosel(const Args& a) {
  for (int i = threadIdx.x; i < a.E * a.E; i += kThreads) {
    const uint32_t nw = atomicExch(a.acc_c + i, 0u);
    const uint32_t old = a.ring_c[i];
    a.ring_c[i] = nw;
    a.csum[i] = a.csum[i] + nw - old;
  }
}

// The statistics block of F2: the histogram into the window ring and sums,
// the co-selection counts likewise, then the prediction for the next layer.
// Nothing in the dispatch reads these, so the block runs beside the copy.
__device__ __noinline__ void stats_tail(const Args& a, const int32_t* hist_s) {
  for (int e = threadIdx.x; e < a.E; e += kThreads) {
    const int32_t h = hist_s[e];
    const uint32_t old = a.ring_h[e];
    a.ring_h[e] = (uint32_t)h;
    a.hsum[e] = a.hsum[e] + (uint32_t)h - old;
    if (a.hist_out) a.hist_out[e] = h;
  }
  if (a.has_prev) fold_cosel(a);
  __syncthreads();  // hsum and csum written above are read by other threads below
  if (a.p_seq) stats::predict_block<unsigned long long, 16>(a.hsum, a.pred_csum, a.E, a.p_seq, a.cond, a.p_next);
}

template <int G, bool VEC>
__global__ void __launch_bounds__(kThreads) route_count_kernel(Args a) {
  pdl_wait();
  // The scatter/copy kernel may start now: before its own wait it only reads
  // x, which the wait above has seen completed.
  if (a.release_early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint32_t dsm[];  // cnt[tiles_per_block][E], then cosel[E*E] (small E)
  constexpr int TPW = 32 / G;
  const int E = a.E, k = a.k;
  const bool cos = a.has_prev != 0;
  const bool cos_smem = cos && E <= kSmemCoselMaxE;
  const int tpb = a.tiles_per_block;
  uint32_t* cnt = dsm;
  uint32_t* cs = dsm + tpb * E;
  const int nsh = tpb * E + (cos_smem ? E * E : 0);
  for (int i = threadIdx.x; i < nsh; i += kThreads) dsm[i] = 0;
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gl = lane % G;
  const long long tb0 = (long long)blockIdx.x * tpb * a.TT;  // first token of the block
  long long tb1 = tb0 + (long long)tpb * a.TT;
  if (tb1 > a.T) tb1 = a.T;
  bool bad = false;
  for (long long t0 = tb0 + (long long)warp * TPW; t0 < tb1; t0 += (long long)kWarps * TPW) {
    const long long t = t0 + lane / G;
    const bool live = t < tb1;
    // the previous layer's choices of the token, loaded ahead of the top-k
    int pe[8];
#pragma unroll
    for (int r1 = 0; r1 < 8; ++r1) pe[r1] = (cos && live && gl == 0 && r1 < k) ? a.idx_prev[t * k + r1] : 0;
    float sel_v[8], denom;
    int sel_i[8];
    route::topk_token<G, VEC>(a.logits + (size_t)(live ? t : 0) * E, live, E, k, a.renorm, sel_v, sel_i, &denom);
    if (live) {
      route::write_token<G>(t, k, sel_v, sel_i, denom, a.idx, a.w);
      if (gl == 0) {
        uint32_t* c = cnt + (int)((t - tb0) / a.TT) * E;
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < k) atomicAdd(c + sel_i[r], 1u);
        if (cos) {
#pragma unroll
          for (int r1 = 0; r1 < 8; ++r1) {
            if (r1 < k) {
              if ((unsigned)pe[r1] >= (unsigned)E) {
                bad = true;
                continue;
              }
#pragma unroll
              for (int r2 = 0; r2 < 8; ++r2) {
                if (r2 < k) {
                  const int bin = pe[r1] * E + sel_i[r2];
                  if (cos_smem)
                    atomicAdd(cs + bin, 1u);
                  else
                    atomicAdd(a.acc_c + bin, 1u);
                }
              }
            }
          }
        }
      }
    }
  }
  if (bad) moe_flag_error(MOE_DEVERR_DATA);
  __syncthreads();
  // per expert: tile prefixes within the block, block total, histogram
  const long long tile0 = (long long)blockIdx.x * tpb;
  for (int e = threadIdx.x; e < E; e += kThreads) {
    uint32_t run = 0;
    for (int i = 0; i < tpb; ++i) {
      const long long tile = tile0 + i;
      if (tile < a.ntiles) a.counts[tile * E + e] = (int32_t)run;
      run += cnt[i * E + e];
    }
    a.blk_tot[(size_t)blockIdx.x * E + e] = (int32_t)run;
    if (run) {
      atomicAdd(a.acc_h + e, run);
      atomicAdd(a.seg_tot + (size_t)(blockIdx.x / kSegBlocks) * E + e, run);
    }
  }
  if (cos_smem)
    for (int i = threadIdx.x; i < E * E; i += kThreads)
      if (cs[i]) atomicAdd(a.acc_c + i, cs[i]);
}

// Offset of scatter_body's slot_s in its dynamic shared memory, in int32
// words (histogram, bases, groups, group bases, copies, group experts, loads,
// per-warp counts, running counts before it).
__host__ __device__ inline int scatter_slot_offset(int E) { return 9 * E + 1 + kWarps * E; }

// Dynamic shared memory of scatter_copy_kernel, in int32 words.
__host__ __device__ inline int scatter_smem_words(int E, int TT, int k) {
  return (16 + kWarps) * E + 1 + TT * k + kThreads;
}
// A tile's token rows are prefetched into L2 when they take at most this many
// bytes (measured: on 160 KB tiles of 10 KB rows the prefetch slowed the copy).
constexpr long long kPrefetchMaxBytes = 64 * 1024;

// The row copy of a tile, by token: one warp per two tokens (8 loads of 16
// bytes in flight per lane), each token row read once and stored to the
// slots of all k of its assignments (16-byte chunks).
__device__ __forceinline__ void copy_rows(const uint16_t* __restrict__ x, int H, uint16_t* __restrict__ xp, int k,
                                          long long f0, int nA, const int32_t* slot_s) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int chunks = H / 8;
  const long long t0 = f0 / k;
  const int nt = nA / k;
  for (int tt = 2 * wid; tt < nt; tt += 2 * kWarps) {
    const bool has1 = tt + 1 < nt;
    const uint16_t* src0 = x + (t0 + tt) * H;
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
        const int s0 = slot_s[tt * k + r];
        if (s0 >= 0) {
          uint16_t* dst = xp + (size_t)s0 * H;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (c + 32 * u < chunks) st_v4(dst + (size_t)(c + 32 * u) * 8, v0[u]);
        }
        const int s1 = has1 ? slot_s[(tt + 1) * k + r] : -1;
        if (s1 >= 0) {
          uint16_t* dst = xp + (size_t)s1 * H;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (c + 32 * u < chunks) st_v4(dst + (size_t)(c + 32 * u) * 8, v1[u]);
        }
      }
    }
  }
}

// Every block takes a ticket (thread 0) once it has read the histogram and
// segment accumulators; the ticket's value is first needed at the block's
// exit, where the last block to have taken one clears those accumulators and
// the ticket for the next call.
__device__ __forceinline__ unsigned take_ticket(const Args& a) {
  return threadIdx.x == 0 ? atomicAdd(a.ticket, 1u) : 0u;
}
__device__ __forceinline__ void leave_block(const Args& a, unsigned ticket) {
  __shared__ int last_s;
  if (threadIdx.x == 0) last_s = ticket == gridDim.x - 1;
  __syncthreads();
  if (last_s) {
    for (int i = threadIdx.x; i < a.E; i += kThreads) a.acc_h[i] = 0u;
    for (int i = threadIdx.x; i < kSegSlots * a.E; i += kThreads) a.seg_tot[i] = 0u;
    if (threadIdx.x == 0) {
      *a.ticket = 0u;
      *a.arrive = 0u;
    }
  }
}

// A load of a word another block may have written: through L2 (ld.cg) in the
// one-launch front, where the writer ran in the same launch.
template <bool THROUGH_L2>
__device__ __forceinline__ uint32_t ld_front(const uint32_t* p) {
  return THROUGH_L2 ? __ldcg(p) : *p;
}

// Shared-memory arrays of the plan in scatter_copy_kernel.
struct Plan {
  int32_t* hist;    // [E]   histogram
  int32_t* base;    // [E]   first slot of the expert's rows
  int32_t* n;       // [E]   replica groups of the expert
  int32_t* rb;      // [E+1] first group of the expert
  int32_t* copies;  // [E]
  int32_t* ge;      // [2E]  expert of each group
  int32_t* load;    // [E]   loads apportioned from the shares
};

// The plan with a copies budget or from predicted shares (the block forms of
// the replica rule), then the expert bases.  Kept out of line, like the other
// paths few blocks take, so the instructions every tile block runs stay
// together.
__device__ __noinline__ void plan_general(const Args& a, const Plan& pl, long long A) {
  __shared__ int32_t wtot[kWarps];
  const int E = a.E, e = threadIdx.x, lane = e & 31, wid = e >> 5;
  int32_t *hist_s = pl.hist, *base_s = pl.base, *n_s = pl.n, *rb_s = pl.rb, *copies_s = pl.copies, *ge_s = pl.ge,
          *load_s = pl.load;
  const int32_t* ld = hist_s;
  if (a.rep_share) {  // replicas from a prediction: loads apportioned by the shares
    replicate::apportion_block(a.rep_share, E, A, load_s);
    __syncthreads();
    ld = load_s;
  }
  replicate::replicate_block(ld, E, A, a.num, a.den, a.max_copies, copies_s, rb_s, ge_s, a.budget);
  __syncthreads();
  // expert bases: exclusive scan of the histogram (E <= kThreads)
  int incl = e < E ? hist_s[e] : 0;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) wtot[wid] = incl;
  __syncthreads();
  int before = 0;
  for (int ww = 0; ww < wid; ++ww) before += wtot[ww];
  if (e < E) {
    base_s[e] = before + incl - hist_s[e];
    n_s[e] = rb_s[e + 1] - rb_s[e];
  }
}

// Tile 0's block writes the replica table and the group offsets.
__device__ __noinline__ void write_tables(const Args& a, const Plan& pl, long long A) {
  const int E = a.E, e = threadIdx.x, tid = threadIdx.x;
  const int32_t *hist_s = pl.hist, *base_s = pl.base, *n_s = pl.n, *rb_s = pl.rb, *copies_s = pl.copies,
                *ge_s = pl.ge;
  const int ngroups = rb_s[E];
  if (e < E) {
    const int hh = hist_s[e], n = n_s[e], rb = rb_s[e], base = base_s[e];
    const int qs = hh / n, qr = hh % n;
    for (int q = 0; q < n; ++q) a.group_offsets[rb + q] = base + q * qs + (q < qr ? q : qr);
    if (a.replicate) {
      a.copies[e] = copies_s[e];
      a.rep_base[e] = rb;
    }
  }
  if (a.replicate) {
    if (tid == 0) a.rep_base[E] = ngroups;
    for (int g = tid; g < 2 * E; g += kThreads) a.group_expert[g] = ge_s[g];
  }
  for (int g = ngroups + tid; g <= 2 * E; g += kThreads) a.group_offsets[g] = (int32_t)A;
}

// F2.  Block 0 is the statistics block (stats_tail); block b >= 1 serves
// dispatch tile b - 1.  Every block first takes the layer's histogram from the
// accumulator the route blocks added their totals to; the last block to take
// it clears the accumulator (and the ticket) for the next call.  A tile block
// then computes the replica table and the group layout itself -- O(E) integer
// work, identical in every block -- so no block waits for a single planner;
// tile 0's block writes the tables out.  Then: the tile's starting rank per
// expert (totals of the route blocks before its own, plus its prefix within
// its block), stable in-tile ranks of its assignments (in f order), slots,
// perm / inv_perm, and the row copy xp[slot] = x[f / k].  With `prefetch`,
// each tile block asks L2 for its token rows before the wait on the previous
// kernel: x is the layer's input, complete before the route kernel of this
// call passed its own wait (and this kernel starts only after every route
// block has passed it), so the read may overlap everything that follows.
// The part of F2 after its wait (see scatter_copy_kernel), shared with the
// one-launch front (front_coop_kernel).  COOP: the tile's assignments were
// routed by this block (their experts are in slot_s), the starting ranks come
// from the totals of the tile segments before the tile's and of the tiles
// before it in its segment, and everything other blocks wrote in this launch
// is read through L2.
template <bool COOP>
__device__ __forceinline__ void scatter_body(const Args& a, const uint16_t* __restrict__ x, int H,
                                             uint16_t* __restrict__ xp, int32_t* __restrict__ perm,
                                             int32_t* __restrict__ inv_perm, int32_t* sm) {
  const int E = a.E, k = a.k;
  int32_t* hist_s = sm;                   // [E]
  int32_t* base_s = hist_s + E;           // [E]   first slot of the expert's rows
  int32_t* n_s = base_s + E;              // [E]   replica groups of the expert
  int32_t* rb_s = n_s + E;                // [E+1] first group of the expert
  int32_t* copies_s = rb_s + E + 1;       // [E]
  int32_t* ge_s = copies_s + E;           // [2E]
  int32_t* load_s = ge_s + 2 * E;         // [E]   loads apportioned from the shares
  int32_t* warp_cnt = load_s + E;         // [kWarps][E]
  int32_t* run = warp_cnt + kWarps * E;   // [E]
  int32_t* slot_s = sm + scatter_slot_offset(E);  // [TT*k], right after run
  int32_t* part_s = slot_s + a.TT * k;    // [kThreads] partial sums
  const Plan pl{hist_s, base_s, n_s, rb_s, copies_s, ge_s, load_s};
  __shared__ int32_t wtot[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int tile = (int)blockIdx.x - 1;
  const long long A = (long long)a.T * k;
  const long long f0 = tile >= 0 ? (long long)tile * a.TT * k : 0;
  long long f1 = tile >= 0 ? f0 + (long long)a.TT * k : 0;
  if (f1 > A) f1 = A;
  const int nA = (int)(f1 - f0);

  // Every load that does not depend on another is issued here at once: the
  // histogram, the tile's prefix within its route block, the totals of the
  // segments and route blocks before it, and the tile's first expert ids.
  // (COOP: segments of kSegTiles tiles, then the tiles before this one in
  // its segment, whose counts are in `counts`; otherwise segments of route
  // blocks, then the route blocks before the tile's, plus the tile's prefix
  // within its route block)
  int nseg, npre;
  const int32_t* blk_seg;
  if (COOP) {
    const int sg = tile >= 0 ? tile / kSegTiles : 0;
    nseg = sg * E;
    npre = nseg + (tile >= 0 ? tile - sg * kSegTiles : 0) * E;
    blk_seg = a.counts + (size_t)sg * kSegTiles * E;
  } else {
    const int rblk = tile >= 0 ? tile / a.tiles_per_block : 0;
    const int sg = rblk / kSegBlocks;
    nseg = sg * E;
    npre = nseg + (rblk - sg * kSegBlocks) * E;
    blk_seg = a.blk_tot + (size_t)sg * kSegBlocks * E;
  }
  int hv = 0, cv = 0, ex0 = -1;
  int pv[kPreLoads];
  if (tid < E) hv = (int32_t)ld_front<COOP>(a.acc_h + tid);
  if (tile >= 0) {
    if (!COOP && tid < E) cv = a.counts[(size_t)tile * E + tid];
#pragma unroll
    for (int u = 0; u < kPreLoads; ++u) {
      const int i = tid + u * kThreads;
      pv[u] = i < nseg ? (int32_t)ld_front<COOP>(a.seg_tot + i)
                       : i < npre ? (int32_t)ld_front<COOP>(reinterpret_cast<const uint32_t*>(blk_seg) + i - nseg) : 0;
    }
    if (tid < nA) ex0 = COOP ? slot_s[tid] : a.idx[f0 + tid];
  }
  if (tid < E) {
    hist_s[tid] = hv;
    run[tid] = cv;
  }
  for (int i = tid; i < kWarps * E; i += kThreads) warp_cnt[i] = 0;
  __syncthreads();
  if (tile < 0) {
    const unsigned ticket = take_ticket(a);
    stats_tail(a, hist_s);
    leave_block(a, ticket);
    return;
  }
  // starting rank of the tile per expert: its prefix within its route block
  // plus the totals before that block (integers: any order of the adds)
  if (kThreads % E == 0) {
    // every total this thread loads belongs to expert tid % E: add them here,
    // then across that expert's threads (shuffles, then shared memory), with
    // no atomics on the few hot bins
    int acc = 0;
#pragma unroll
    for (int u = 0; u < kPreLoads; ++u) acc += pv[u];
    for (int i0 = tid + kPreLoads * kThreads; i0 < npre; i0 += kPreLoads * kThreads) {
#pragma unroll
      for (int u = 0; u < kPreLoads; ++u) {
        const int i = i0 + u * kThreads;
        acc += i < nseg ? (int32_t)ld_front<COOP>(a.seg_tot + i)
                        : i < npre ? (int32_t)ld_front<COOP>(reinterpret_cast<const uint32_t*>(blk_seg) + i - nseg)
                                   : 0;
      }
    }
    if (E < 32) {
      for (int off = E; off < 32; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane < E) part_s[wid * E + lane] = acc;
    } else {
      part_s[tid] = acc;
    }
    __syncthreads();
    if (tid < E) {
      const int nparts = E < 32 ? kWarps : kThreads / E;
      int s2 = 0;
      for (int j = 0; j < nparts; ++j) s2 += part_s[j * E + tid];
      run[tid] += s2;
    }
  } else {
#pragma unroll
    for (int u = 0; u < kPreLoads; ++u)
      if (pv[u]) atomicAdd(&run[(tid + u * kThreads) % E], pv[u]);
    for (int i0 = tid + kPreLoads * kThreads; i0 < npre; i0 += kPreLoads * kThreads) {
#pragma unroll
      for (int u = 0; u < kPreLoads; ++u) {
        const int i = i0 + u * kThreads;
        pv[u] = i < nseg ? (int32_t)ld_front<COOP>(a.seg_tot + i)
                         : i < npre ? (int32_t)ld_front<COOP>(reinterpret_cast<const uint32_t*>(blk_seg) + i - nseg)
                                    : 0;
      }
#pragma unroll
      for (int u = 0; u < kPreLoads; ++u)
        if (pv[u]) atomicAdd(&run[(i0 + u * kThreads) % E], pv[u]);
    }
    __syncthreads();
  }
  // every thread's reads of the accumulators are done (both branches end in a barrier)
  const unsigned ticket = take_ticket(a);

  // ---- replica table and group layout
  const int e = tid;
  if (a.replicate && (a.rep_share || a.budget >= 0)) {
    plan_general(a, pl, A);
  } else {
    // Replicas from the histogram with no copies budget (or none at all): the
    // replica rule is a closed form per expert (replicate::replicate_block
    // states it), so the copies, the expert bases and the group bases come
    // from one scan of (load, groups) over the experts.
    __shared__ int32_t wtot_n[kWarps];
    const int h = e < E ? hist_s[e] : 0;
    int c = 0;
    if (a.replicate && e < E && A > 0 && (long long)h * E * a.den > (long long)a.num * A) {
      const long long q = (long long)h * E + A - 1;  // ceil(h * E / A) by a 32-bit division when it fits
      c = (q >> 31) == 0 ? (int)((unsigned)q / (unsigned)A) - 1 : (int)(q / A - 1);
      if (a.max_copies >= 0 && c > a.max_copies) c = a.max_copies;
    }
    const int n = e < E ? c + 1 : 0;
    int ih = h, in = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int vh = __shfl_up_sync(0xffffffffu, ih, off);
      const int vn = __shfl_up_sync(0xffffffffu, in, off);
      if (lane >= off) {
        ih += vh;
        in += vn;
      }
    }
    if (lane == 31) {
      wtot[wid] = ih;
      wtot_n[wid] = in;
    }
    const int any_negative = __syncthreads_or(e < E && h < 0);
    int bh = 0, bn = 0;
    long long all_h = 0;
    int all_n = 0;
    for (int ww = 0; ww < kWarps; ++ww) {
      if (ww < wid) {
        bh += wtot[ww];
        bn += wtot_n[ww];
      }
      all_h += wtot[ww];
      all_n += wtot_n[ww];
    }
    // the block form's precondition: loads non-negative and summing to at
    // most the total (then fewer than 2E groups); broken -> no replication
    const bool bad = a.replicate && (any_negative || (A > 0 && all_h > A) || all_n > 2 * E);
    if (bad && tid == 0) moe_flag_error(MOE_DEVERR_DATA);
    if (e < E) {
      base_s[e] = bh + ih - h;
      const int rb = bad ? e : bn + in - n;
      n_s[e] = bad ? 1 : n;
      rb_s[e] = rb;
      copies_s[e] = bad ? 0 : c;
      if (a.replicate && tile == 0) {
        ge_s[rb] = e;
        if (bad) ge_s[E + e] = -1;
        else
          for (int q = 1; q < n; ++q) ge_s[rb + q] = e;
      }
    }
    const int ngroups = bad ? E : all_n;
    if (tid == 0) rb_s[E] = ngroups;
    if (a.replicate && tile == 0)
      for (int g = ngroups + tid; g < 2 * E; g += kThreads) ge_s[g] = -1;
  }
  __syncthreads();
  if (tile == 0) write_tables(a, pl, A);

  // ---- stable in-tile ranks, slots, perm / inv_perm
  for (int r0 = 0; r0 < nA; r0 += kThreads) {
    const int i = r0 + tid;
    int ex = -1;
    if (i < nA) {
      ex = r0 == 0 ? ex0 : COOP ? slot_s[i] : a.idx[f0 + i];
      if ((unsigned)ex >= (unsigned)E) ex = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, ex);
    if (ex >= 0 && lane == __ffs(peers) - 1) warp_cnt[wid * E + ex] = __popc(peers);
    __syncthreads();
    int slot = -1;
    if (ex >= 0) {
      int m = run[ex] + __popc(peers & lanemask_lt());
      for (int w = 0; w < wid; ++w) m += warp_cnt[w * E + ex];
      const int base = base_s[ex], n = n_s[ex], h = hist_s[ex];
      const int q = m % n, pos = m / n, qs = h / n, qr = h % n;
      slot = base + q * qs + (q < qr ? q : qr) + pos;
      if ((unsigned long long)slot < (unsigned long long)A) {
        perm[slot] = (int32_t)(f0 + i);
        inv_perm[f0 + i] = slot;
      } else {
        slot = -1;
        inv_perm[f0 + i] = -1;
      }
    } else if (i < nA) {
      inv_perm[f0 + i] = -1;  // expert out of range (flagged): no slot
    }
    if (i < nA) slot_s[i] = slot;
    __syncthreads();
    for (int j = tid; j < E; j += kThreads) {
      int s2 = 0;
      for (int w = 0; w < kWarps; ++w) {
        s2 += warp_cnt[w * E + j];
        warp_cnt[w * E + j] = 0;
      }
      run[j] += s2;
    }
    __syncthreads();
  }
  if (x != nullptr) copy_rows(x, H, xp, k, f0, nA, slot_s);
  leave_block(a, ticket);
}

__global__ void __launch_bounds__(kThreads) scatter_copy_kernel(const Args a, const uint16_t* __restrict__ x, int H,
                                                                uint16_t* __restrict__ xp,
                                                                int32_t* __restrict__ perm,
                                                                int32_t* __restrict__ inv_perm, int prefetch) {
  extern __shared__ int32_t sm[];
  if (prefetch && blockIdx.x > 0 && threadIdx.x == 0) {
    const long long t0 = (long long)(blockIdx.x - 1) * a.TT;
    const long long nt = a.T - t0 < a.TT ? a.T - t0 : a.TT;
    sm100::bulk_prefetch_l2(x + t0 * H, (uint32_t)(nt * H * 2));
  }
  pdl_wait();
  scatter_body<false>(a, x, H, xp, perm, inv_perm, sm);
}

// Dynamic shared memory of route_count_kernel stays below 17 KB (tile counts
// plus, for E <= 64, the E*E co-selection bins); that of scatter_copy_kernel
// below 29 KB (E = 256, 128-token tiles of top-8), which with the static
// arrays of the replica, apportionment and prediction block functions can pass
// 48 KB.  The limits are raised once per device and kernel instance.
constexpr int kRouteDynSmemMax = 20 * 1024;
constexpr int kScatterDynSmemMax = 32 * 1024;

template <typename K>
static cudaError_t ensure_smem_attr(K kernel, bool* done_per_device, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done_per_device[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done_per_device[dev] = true;
  return e;
}

// ---------------------------------------------------------------- one launch
// The front in one cooperative launch (every block resident): each tile block
// routes its own TT tokens (the same per-token work as route_count_kernel),
// keeps their experts in shared memory, publishes its tile counts (to
// `counts`, the histogram accumulator and its tile segment's totals) and its
// co-selection pairs, then all blocks meet at a grid-wide barrier; after it,
// scatter_body<true> runs the dispatch as scatter_copy_kernel does, without a
// second launch and without reloading the tile's experts.

// Route the tile's tokens [t0, t0 + nt); counts into cnt_s, the experts of
// assignment f = (t - t0) * k + r into ex_s[f], co-selection pairs into cs_s
// (cos_smem) or the accumulator.
template <int G, bool VEC>
__device__ __forceinline__ void route_tile(const Args& a, long long t0, int nt, int32_t* cnt_s, uint32_t* cs_s,
                                           bool cos_smem, int32_t* ex_s) {
  constexpr int TPW = 32 / G;
  const int E = a.E, k = a.k;
  const bool cos = a.has_prev != 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gl = lane % G;
  bool bad = false;
  for (int tt0 = warp * TPW; tt0 < nt; tt0 += kWarps * TPW) {
    const int tt = tt0 + lane / G;
    const bool live = tt < nt;
    const long long t = t0 + tt;
    int pe[8];
#pragma unroll
    for (int r1 = 0; r1 < 8; ++r1) pe[r1] = (cos && live && gl == 0 && r1 < k) ? a.idx_prev[t * k + r1] : 0;
    float sel_v[8], denom;
    int sel_i[8];
    route::topk_token<G, VEC>(a.logits + (size_t)(live ? t : 0) * E, live, E, k, a.renorm, sel_v, sel_i, &denom);
    if (live) {
      route::write_token<G>(t, k, sel_v, sel_i, denom, a.idx, a.w);
      if (gl == 0) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (r < k) {
            atomicAdd(cnt_s + sel_i[r], 1);
            ex_s[tt * k + r] = sel_i[r];
          }
        }
        if (cos) {
#pragma unroll
          for (int r1 = 0; r1 < 8; ++r1) {
            if (r1 < k) {
              if ((unsigned)pe[r1] >= (unsigned)E) {
                bad = true;
                continue;
              }
#pragma unroll
              for (int r2 = 0; r2 < 8; ++r2) {
                if (r2 < k) {
                  const int bin = pe[r1] * E + sel_i[r2];
                  if (cos_smem)
                    atomicAdd(cs_s + bin, 1u);
                  else
                    atomicAdd(a.acc_c + bin, 1u);
                }
              }
            }
          }
        }
      }
    }
  }
  if (bad) moe_flag_error(MOE_DEVERR_DATA);
}

// Grid-wide barrier of the one-launch front: thread 0 of each block makes the
// block's writes visible, arrives, and polls the count with a bounded wait
// (~2 s, then the device timeout bit; the block goes on and the call's
// results are not to be used).
__device__ __forceinline__ void grid_barrier(const Args& a) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(a.arrive, 1u);
    const uint64_t start = sm100::globaltimer_ns();
    for (uint32_t i = 0; i < (1u << 28); ++i) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.arrive) : "memory");
      if (v >= gridDim.x) break;
      if ((i & 63) == 63 && sm100::globaltimer_ns() - start > 2000000000ull) {
        moe_flag_error(MOE_DEVERR_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
}

// Dynamic shared memory of front_coop_kernel, in int32 words: scatter_body's,
// then the tile counts [E] and, for E <= kSmemCoselMaxE, the co-selection
// bins [E*E].
__host__ __device__ inline int coop_smem_words(int E, int TT, int k, bool cos_smem) {
  return scatter_smem_words(E, TT, k) + E + (cos_smem ? E * E : 0);
}

template <int G, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) front_coop_kernel(const Args a, const uint16_t* __restrict__ x, int H,
                                                                 uint16_t* __restrict__ xp,
                                                                 int32_t* __restrict__ perm,
                                                                 int32_t* __restrict__ inv_perm, int prefetch) {
  extern __shared__ int32_t sm[];
  pdl_wait();
  const int E = a.E, k = a.k, tid = threadIdx.x;
  const int tile = (int)blockIdx.x - 1;
  const bool cos_smem = a.has_prev != 0 && E <= kSmemCoselMaxE;
  int32_t* ex_s = sm + scatter_slot_offset(E);  // scatter_body's slot_s: the tile's experts until its ranks
  int32_t* cnt_s = sm + scatter_smem_words(E, a.TT, k);
  uint32_t* cs_s = reinterpret_cast<uint32_t*>(cnt_s + E);
  if (tile >= 0) {
    const long long t0 = (long long)tile * a.TT;
    const int nt = (int)(a.T - t0 < a.TT ? a.T - t0 : a.TT);
    if (prefetch && tid == 0) sm100::bulk_prefetch_l2(x + t0 * H, (uint32_t)((long long)nt * H * 2));
    for (int i = tid; i < E + (cos_smem ? E * E : 0); i += kThreads) cnt_s[i] = 0;
    __syncthreads();
    route_tile<G, VEC>(a, t0, nt, cnt_s, cs_s, cos_smem, ex_s);
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
      const int c = cnt_s[e];
      a.counts[(size_t)tile * E + e] = c;
      if (c) {
        atomicAdd(a.acc_h + e, (uint32_t)c);
        atomicAdd(a.seg_tot + (size_t)(tile / kSegTiles) * E + e, (uint32_t)c);
      }
    }
    if (cos_smem)
      for (int i = tid; i < E * E; i += kThreads)
        if (cs_s[i]) atomicAdd(a.acc_c + i, cs_s[i]);
  }
  grid_barrier(a);
  scatter_body<true>(a, x, H, xp, perm, inv_perm, sm);
}

// Host side of the one-launch front: blocks per SM of the instance at this
// shared-memory size (0 if it cannot be resident), cached per device.
template <int G, bool VEC>
static cudaError_t launch_coop_g(const Args& a, const uint16_t* x, int H, uint16_t* xp, int32_t* perm,
                                 int32_t* inv_perm, int prefetch, int num_sms, bool* launched, cudaStream_t st) {
  *launched = false;
  static bool done[64] = {};
  const bool cos_smem = a.has_prev != 0 && a.E <= kSmemCoselMaxE;
  const size_t smem = sizeof(int32_t) * (size_t)coop_smem_words(a.E, a.TT, a.k, cos_smem);
  if (smem > (size_t)kScatterDynSmemMax) return cudaSuccess;
  cudaError_t e = ensure_smem_attr(front_coop_kernel<G, VEC>, done, kScatterDynSmemMax);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, front_coop_kernel<G, VEC>, kThreads, smem);
  if (e != cudaSuccess) return e;
  if ((long long)per_sm * num_sms < a.ntiles + 1) return cudaSuccess;  // not all resident: two launches
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.ntiles + 1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g_moe_pdl.load(std::memory_order_relaxed) ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, front_coop_kernel<G, VEC>, a, x, H, xp, perm, inv_perm, prefetch);
  if (e != cudaSuccess) return e;
  *launched = true;
  return cudaGetLastError();
}

// Tiles per route block: every warp gets at least one pass of tokens, and
// there are at most kMaxRouteBlocks blocks.
__host__ inline int route_tiles_per_block(long long T, int E) {
  const int G = E <= 8 ? 1 : E <= 16 ? 2 : E <= 32 ? 4 : E <= 64 ? 8 : E <= 128 ? 16 : 32;
  const int TT = tile_tokens(T);
  const int tokens_per_pass = kWarps * (32 / G);
  int tpb = tokens_per_pass >= TT ? tokens_per_pass / TT : 1;
  const long long nt = num_tiles(T);
  const long long need = (nt + kMaxRouteBlocks - 1) / kMaxRouteBlocks;
  if (need > tpb) tpb = (int)need;
  return tpb;
}

template <int G>
static cudaError_t launch_route_g(const Args& a, bool vec, cudaStream_t st) {
  static bool done_vec[64] = {}, done_scalar[64] = {};
  const long long tokens_per_block = (long long)a.tiles_per_block * a.TT;
  const long long blocks = (a.T + tokens_per_block - 1) / tokens_per_block;
  const bool cos_smem = a.has_prev && a.E <= kSmemCoselMaxE;
  const size_t smem = sizeof(uint32_t) * ((size_t)a.tiles_per_block * a.E + (cos_smem ? (size_t)a.E * a.E : 0));
  if (smem > (size_t)kRouteDynSmemMax) return cudaErrorInvalidValue;
  if (vec) {
    cudaError_t e = ensure_smem_attr(route_count_kernel<G, true>, done_vec, kRouteDynSmemMax);
    if (e != cudaSuccess) return e;
    e = launch_pdl(route_count_kernel<G, true>, dim3((unsigned)blocks), dim3(kThreads), smem, st, a);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = ensure_smem_attr(route_count_kernel<G, false>, done_scalar, kRouteDynSmemMax);
    if (e != cudaSuccess) return e;
    e = launch_pdl(route_count_kernel<G, false>, dim3((unsigned)blocks), dim3(kThreads), smem, st, a);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

// Process-wide choice of the front's form (moe_set_option(MOE_OPT_FRONT_ONE_LAUNCH)).
// Off by default: on the moe_gpt_stream layer the one launch measured slower
// (per-block stamps: routing in 513 blocks done at 6.1-7.4 us against 4.2 us
// in 128 route blocks -- 4x the co-selection flushes onto the same bins --
// and 2.5-3 us in the grid-wide barrier; last copy done at 29.7 against
// 23.8 us), and no faster on the single-layer workloads.
inline std::atomic<int> g_front_one_launch{0};

static cudaError_t launch(const Args& a0, const uint16_t* x, int H, uint16_t* xp, int32_t* perm, int32_t* inv_perm,
                          int num_sms, cudaStream_t st) {
  Args a = a0;
  a.tiles_per_block = route_tiles_per_block(a.T, a.E);
  // Short token rows: the scatter/copy blocks start while the route blocks
  // run and ask L2 for their rows first (measured better than the route
  // blocks prefetching them, which slowed the routing itself).
  const int prefetch = (x != nullptr && a.ntiles > 0 && (long long)a.TT * H * 2 <= kPrefetchMaxBytes) ? 1 : 0;
  const bool vec = (a.E % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.logits) & 15) == 0);
  cudaError_t e;
  if (g_front_one_launch.load(std::memory_order_relaxed) && a.ntiles > 0 &&
      a.ntiles <= (long long)kSegTiles * kSegSlots) {
    a.release_early = 0;
    bool launched = false;
    if (a.E <= 8) e = vec ? launch_coop_g<1, true>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st)
                          : launch_coop_g<1, false>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st);
    else if (a.E <= 16) e = vec ? launch_coop_g<2, true>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st)
                                : launch_coop_g<2, false>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st);
    else if (a.E <= 32) e = vec ? launch_coop_g<4, true>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st)
                                : launch_coop_g<4, false>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st);
    else if (a.E <= 64) e = vec ? launch_coop_g<8, true>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st)
                                : launch_coop_g<8, false>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st);
    else if (a.E <= 128)
      e = vec ? launch_coop_g<16, true>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st)
              : launch_coop_g<16, false>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st);
    else
      e = vec ? launch_coop_g<32, true>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st)
              : launch_coop_g<32, false>(a, x, H, xp, perm, inv_perm, prefetch, num_sms, &launched, st);
    if (e != cudaSuccess || launched) return e;
  }
  a.release_early = prefetch;
  if (a.E <= 8) e = launch_route_g<1>(a, vec, st);
  else if (a.E <= 16) e = launch_route_g<2>(a, vec, st);
  else if (a.E <= 32) e = launch_route_g<4>(a, vec, st);
  else if (a.E <= 64) e = launch_route_g<8>(a, vec, st);
  else if (a.E <= 128) e = launch_route_g<16>(a, vec, st);
  else e = launch_route_g<32>(a, vec, st);
  if (e != cudaSuccess) return e;
  static bool done_scatter[64] = {};
  const size_t smem = sizeof(int32_t) * (size_t)scatter_smem_words(a.E, a.TT, a.k);
  if (smem > (size_t)kScatterDynSmemMax) return cudaErrorInvalidValue;
  if ((e = ensure_smem_attr(scatter_copy_kernel, done_scatter, kScatterDynSmemMax)) != cudaSuccess) return e;
  e = launch_pdl(scatter_copy_kernel, dim3((unsigned)(a.ntiles + 1)), dim3(kThreads), smem, st, a, x, H, xp, perm,
                 inv_perm, prefetch);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Kernels one call of launch() makes for these sizes on the current device
// (T > 0): 1 when the one-launch form applies, else 2.  Host only.
static int launches(long long T, int E, int k, bool has_prev, int num_sms) {
  const long long nt = num_tiles(T);
  if (!g_front_one_launch.load(std::memory_order_relaxed) || nt <= 0 || nt > (long long)kSegTiles * kSegSlots)
    return 2;
  const bool cos_smem = has_prev && E <= kSmemCoselMaxE;
  const size_t smem = sizeof(int32_t) * (size_t)coop_smem_words(E, tile_tokens(T), k, cos_smem);
  if (smem > (size_t)kScatterDynSmemMax) return 2;
  int per_sm = 0;
  cudaError_t e;
  if (E <= 8) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, front_coop_kernel<1, true>, kThreads, smem);
  else if (E <= 16) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, front_coop_kernel<2, true>, kThreads, smem);
  else if (E <= 32) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, front_coop_kernel<4, true>, kThreads, smem);
  else if (E <= 64) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, front_coop_kernel<8, true>, kThreads, smem);
  else if (E <= 128)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, front_coop_kernel<16, true>, kThreads, smem);
  else
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, front_coop_kernel<32, true>, kThreads, smem);
  if (e != cudaSuccess) return 2;
  return (long long)per_sm * num_sms >= nt + 1 ? 1 : 2;
}

}  // namespace front

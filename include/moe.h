/*
 * moe.h -- C ABI of the B300 MoE routing-and-expert step (libmoe.so).
 *
 * One MoE layer, on one GPU, as seven stream-ordered calls:
 *
 *   moe_route         top-k gate over router logits
 *   moe_stats_update  per-expert histogram + layer j-1 -> j co-selection counts,
 *                     kept over a sliding window
 *   moe_predict       window popularity p_seq, conditional probability,
 *                     predicted next-layer popularity
 *   moe_replicate     replica counts for hot experts
 *   moe_dispatch      stable permutation of assignments by expert / replica,
 *                     and the permuted copy of the token rows
 *   moe_expert_ffn    grouped expert FFN (GeLU or SwiGLU) on tcgen05 tensor cores
 *   moe_combine       gate-weighted sum of each token's k expert outputs
 *
 * Fused forms of the same work: moe_layer_front (route through dispatch in
 * two launches), moe_expert_ffn_gather (the FFN reading the token rows in
 * place, so that dispatch writes only the permutation) and
 * moe_expert_ffn_combine (the combine in the second GEMM's epilogue).
 * Widened calls: moe_predict_decay and moe_replicate_predicted (replicas from
 * a prediction, with a copies budget), moe_replicate_weights and
 * moe_expert_ffn_slots (physical replica copies), moe_ffn_backward and
 * moe_route_backward (the layer's backward), and moe_dispatch_noalloc
 * (dispatch with library-owned scratch).
 *
 * Conventions
 *   T tokens, E experts, k experts per token, A = T*k assignments (assignment
 *   f = t*k + r is token t's r-th choice), H hidden size, F expert FFN width.
 *   Matrices are row-major and contiguous.  bf16 tensors are passed as
 *   uint16_t bit patterns.  Every pointer is a DEVICE pointer unless the
 *   argument says "host".  `stream` is a cudaStream_t (NULL = legacy stream).
 *
 * Ownership and ordering
 *   The caller owns every tensor and stream.  The library allocates device
 *   memory only in moe_stats_create (the window state) and frees it in
 *   moe_stats_destroy; scratch for moe_dispatch / moe_expert_ffn is passed in
 *   by the caller (size from moe_workspace_bytes).  Every call only enqueues
 *   work on `stream` and returns; none synchronises except moe_check,
 *   moe_stats_export and moe_stats_import.  Calls that share a moe_stats
 *   handle or a workspace must be ordered on one stream.  The expert FFN
 *   calls run their small-batch kernels on a library-owned stream per device
 *   (created with two events at the first call on that device, kept for the
 *   life of the process), forked from `stream` and joined back to it within
 *   the call, so callers see ordinary stream order; calls on different
 *   streams share that side stream (one fork/join at a time, under a
 *   process-wide lock).  The sharing adds an ordering between callers that
 *   work on independent streams: the side-stream part of a later call waits
 *   for the side-stream part of every earlier one on that device, and so does
 *   the caller's stream at the join.  Results are unaffected; only overlap
 *   between such callers is lost.  Under CUDA
 *   graph capture the side stream joins the capture through the fork event
 *   and stays part of it until the capture ends, so while one thread captures
 *   these calls no other thread may enqueue them on the same device; make the
 *   first call on a device before capturing (it creates the side stream).
 *
 * Errors
 *   Every call returns a moe_status.  Arguments are validated on the host
 *   before anything is enqueued: MOE_ERR_INVALID for null required pointers,
 *   out-of-range sizes (T < 0, E < 1 or E > 256, k < 1 or k > min(E, 8),
 *   H/F not multiples of the stated granule, A = T*k >= 2^31) and misaligned
 *   pointers; MOE_ERR_WORKSPACE for a workspace smaller than
 *   moe_workspace_bytes; MOE_ERR_CUDA when a launch fails (message from
 *   moe_last_error).  Kernels that meet invalid device data (an expert id
 *   outside [0, E), inconsistent group offsets) or a bounded wait that ran
 *   out skip the offending work and set a device error word; moe_check
 *   reports it (MOE_ERR_DEVICE / MOE_ERR_TIMEOUT) and clears it.  No C++
 *   exception crosses this ABI.  T = 0 is a valid empty batch.
 *
 * Source of each operation: the pages that define the method are reviews of
 * PopFetcher (ATC'25), MoE-GPS, EPS-MoE, MoE-MPMC and "Prediction Is All MoE
 * Needs"; each entry below names the passage it follows.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID = 1,      /* bad argument (host-side check)                 */
    MOE_ERR_UNSUPPORTED = 2,  /* valid request the library does not support      */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed           */
    MOE_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out (moe_check) */
    MOE_ERR_WORKSPACE = 5,    /* workspace too small                            */
    MOE_ERR_DEVICE = 6        /* invalid device data met by a kernel (moe_check) */
} moe_status;

typedef enum { MOE_ACT_GELU = 0, MOE_ACT_SWIGLU = 1 } moe_act;

typedef enum { MOE_OP_DISPATCH = 1, MOE_OP_EXPERT_FFN = 2, MOE_OP_LAYER_FRONT = 3, MOE_OP_EXPERT_FFN_COMBINE = 4 } moe_op;

/* Opaque window state: device ring buffers of per-layer histograms and
 * per-layer-pair co-selection counts, plus running window sums. */
typedef struct moe_stats moe_stats;

/* ---------------------------------------------------------------------------
 * moe_stats_create / moe_stats_destroy
 * PopFetcher review, core method (Routing Information Collector): token
 * allocation statistics are kept over a sliding window of s iterations
 * (s = 10 in the paper).
 *   st      (host) receives the handle
 *   L       MoE layers (1..1024);  E experts (1..256);  window s (1..1024)
 *   stream  used to zero the state (the call returns after the zeroing is
 *           enqueued; the handle is usable by later calls on any stream
 *           ordered after it)
 * Device memory: L*s*E*4 + L*E*8 + (L-1)*(s*E*E*4 + E*E*8) bytes + O(E*E).
 * ------------------------------------------------------------------------- */
moe_status moe_stats_create(moe_stats** st, int L, int E, int window, void* stream);
moe_status moe_stats_destroy(moe_stats* st);

/* ---------------------------------------------------------------------------
 * moe_route -- top-k gate.
 * PopFetcher review (naive top-k gate) and EPS-MoE review, experiments (top-2
 * Mixtral, top-4 DBRX, top-6 DeepSeekV2; softmax-renormalised gate weights).
 *   logits  [T,E] fp32, finite (not checked per element); 16-byte aligned
 *   idx     [T,k] int32 out: chosen experts by logit descending; equal logits
 *           (including -0.0 vs +0.0) -> lower expert index first
 *   w       [T,k] fp32 out: renorm=1: softmax over the k chosen logits;
 *           renorm=0: full softmax over all E logits, at the chosen experts
 * ------------------------------------------------------------------------- */
moe_status moe_route(const float* logits, int T, int E, int k, int renorm,
                     int32_t* idx, float* w, void* stream);

/* ---------------------------------------------------------------------------
 * moe_stats_update -- token allocation statistics of one layer.
 * PopFetcher review, observation 1 (per-expert token counts) and observation
 * 2 / Fig. 6 (layer-to-layer selection counts behind Pr(E^{h,j+1}|E^{i,j})).
 *   iter       iteration number (>= 0); the update goes to ring slot iter % s
 *              and replaces what that slot held for this layer
 *   layer      j in [0, L)
 *   idx_layer  [T,k] int32: layer j's routing (from moe_route)
 *   idx_prev   [T,k] int32: layer j-1's routing of the same tokens; required
 *              for j > 0 (co-selection counts C_{j-1}[e,e'] = number of
 *              tokens with e among their layer j-1 choices and e' among
 *              their layer j choices; all k*k pairs count), NULL for j = 0
 *   hist_out   [E] int32 out (nullable): this update's histogram h_j
 * Expert ids outside [0,E) are skipped and flagged (moe_check).
 * ------------------------------------------------------------------------- */
moe_status moe_stats_update(moe_stats* st, int64_t iter, int layer,
                            const int32_t* idx_layer, const int32_t* idx_prev,
                            int T, int k, int32_t* hist_out, void* stream);

/* ---------------------------------------------------------------------------
 * moe_predict -- window popularity and next-layer prediction.
 * PopFetcher review, core method: Eq. (1) sequence popularity p_seq over the
 * window; Eq. (2)(3) p(E^{j+1}) = sum_e p_seq^j(e) * Pr(e'|e).  MoE-GPS blog
 * section 2.1: p_i = n_i / N with a sliding-window average.
 *   layer   j; predicts layer j+1
 *   p_seq   [E] fp32 out: H_j[e] / sum H_j (window sums; 1/E while empty)
 *   cond    [E,E] fp32 out (nullable): Cbar_j[e,e'] / sum_e'' Cbar_j[e,e'']
 *           (1/E for a row with no counts)
 *   p_next  [E] fp32 out (nullable): sum_e p_seq[e] * cond[e,e']
 * Computed in fp64.  For j = L-1, cond and p_next must be NULL.
 * ------------------------------------------------------------------------- */
moe_status moe_predict(moe_stats* st, int layer, float* p_seq, float* cond,
                       float* p_next, void* stream);

/* ---------------------------------------------------------------------------
 * moe_predict_decay -- next-layer prediction from a decay-weighted window.
 * MoE-GPS blog section 2.1: the sliding-window estimate p_i = n_i / N carries
 * a decay factor against distribution drift (no formula printed).  Reading:
 * with the causal order of the calls (layer j recorded at iteration `iter`,
 * then predicted, then layer j+1 recorded), ring slot (iter - a) mod s of the
 * histogram and slot (iter - 1 - a) mod s of the co-selection counts weigh
 * lambda^a (a = 0 .. s-1, lambda^0 = 1); p_seq, cond and p_next are then
 * formed as in moe_predict.  lambda = 1 gives moe_predict's results bit for
 * bit; lambda = 0 uses the newest iteration only.
 *   iter    >= 0, the iteration of the newest histogram of layer j
 *   lambda  in [0, 1]
 *   p_seq, cond, p_next as in moe_predict (cond/p_next NULL for the last
 *           layer).  Computed in fp64 in one block; uses the handle's own
 *           scratch, so calls on one handle must be ordered on one stream.
 * ------------------------------------------------------------------------- */
moe_status moe_predict_decay(moe_stats* st, int layer, int64_t iter, double lambda,
                             float* p_seq, float* cond, float* p_next, void* stream);

/* ---------------------------------------------------------------------------
 * moe_replicate -- replica counts for hot experts.
 * MoE-GPS blog section 2.1 (duplicate_experts): target = total / E; an
 * expert whose load exceeds (thresh_num/thresh_den) * target (6/5 = 1.2)
 * gets ceil(load / target) - 1 extra copies.  MoE-MPMC summary, contribution
 * 3: a capacity bound caps the copies (max_copies; -1 = none).
 *   load          [E] int32 (device), e.g. hist_out of moe_stats_update;
 *                 must be >= 0 and sum to <= total
 *   total         (host) A = T*k
 *   copies        [E] int32 out
 *   rep_base      [E+1] int32 out: exclusive scan of copies+1; rep_base[E]
 *                 = number of groups G (<= 2E-1 when loads sum to <= total)
 *   group_expert  [2E] int32 out: expert of group g; -1 for g >= G
 * Exact integer arithmetic.  Loads that break the precondition set the
 * device error word and produce the no-replication table.
 * ------------------------------------------------------------------------- */
moe_status moe_replicate(const int32_t* load, int E, int64_t total, int thresh_num,
                         int thresh_den, int max_copies, int32_t* copies,
                         int32_t* rep_base, int32_t* group_expert, void* stream);

/* ---------------------------------------------------------------------------
 * moe_replicate_predicted -- replica table from a predicted popularity
 * (prediction-driven replication: replicas placed before the layer runs).
 * MoE-GPS blog section 2.1 (duplicate_experts rule on the predicted token
 * distribution); MoE-MPMC summary, contribution 3 (replica counts bounded by
 * a predefined memory budget).
 *   p_next     [E] fp32 predicted shares (moe_predict's p_next of the layer
 *              before); a negative share counts as 0, a NaN share also sets
 *              the device error word
 *   total      A = T*k assignments the prediction is for, 1 <= total < 2^29
 *   load_out   [E] int32 out: the largest-remainder apportionment of total
 *              by the shares (sums to total; quotas computed exactly from
 *              the fp32 values; ties: lower expert first)
 *   thresh_num/thresh_den, max_copies: the replica rule of moe_replicate on
 *              load_out
 *   budget     bound on the total number of extra copies (-1 = none); the
 *              hottest experts (by load_out, lower expert first on ties)
 *              keep their copies first
 *   copies [E], rep_base [E+1], group_expert [2E]: as moe_replicate
 * ------------------------------------------------------------------------- */
moe_status moe_replicate_predicted(const float* p_next, int E, int64_t total, int thresh_num,
                                   int thresh_den, int max_copies, int budget, int32_t* load_out,
                                   int32_t* copies, int32_t* rep_base, int32_t* group_expert,
                                   void* stream);

/* ---------------------------------------------------------------------------
 * moe_dispatch -- stable permutation by expert, then replica.
 * PopFetcher review, problem statement (token dispatch before the expert
 * FFN); MoE-MPMC summary (tokens of one expert spread over its physical
 * replicas).  Expert e's assignments are taken in ascending f; the m-th goes
 * to replica q = m mod n_e (n_e = rep_base[e+1]-rep_base[e]) at position
 * floor(m / n_e) of group g = rep_base[e] + q.
 *   x              [T,H] bf16; may be NULL together with xp (permutation only)
 *   idx            [T,k] int32 routing
 *   rep_base       [E+1] int32 from moe_replicate, or NULL (one group per expert)
 *   group_offsets  [2E+1] int32 out: row offset of each group in xp;
 *                  entries past the last group equal A
 *   perm           [A] int32 out: slot -> assignment f
 *   inv_perm       [A] int32 out: assignment f -> slot (-1 for an assignment
 *                  whose expert is out of range; the call flags that)
 *   xp             [A,H] bf16 out: xp[slot] = x[perm[slot] / k] (bit copy)
 *   workspace      ws_bytes >= moe_workspace_bytes(MOE_OP_DISPATCH, T, k, E, H, 0),
 *                  16-byte aligned
 * H must be a multiple of 8; x and xp 16-byte aligned.
 * ------------------------------------------------------------------------- */
moe_status moe_dispatch(const uint16_t* x, const int32_t* idx, int T, int k, int H, int E,
                        const int32_t* rep_base, int32_t* group_offsets, int32_t* perm,
                        int32_t* inv_perm, uint16_t* xp, void* workspace, size_t ws_bytes,
                        void* stream);

/* ---------------------------------------------------------------------------
 * moe_layer_front -- route, statistics, prediction, replicas and dispatch of one
 * layer in two launches.
 * The same results, bit for bit, as
 *   moe_route(logits) -> moe_stats_update(st, iter, layer, idx, idx_prev) ->
 *   moe_predict(st, layer) [when p_seq != NULL] -> moe_replicate(hist, T*k)
 *   [when replicate != 0] -> moe_dispatch(x, idx, rep_base or NULL)
 * (passages as for those calls: PopFetcher review, gate and Routing
 * Information Collector, Eq. (1)-(3); MoE-GPS blog section 2.1,
 * duplicate_experts; MoE-MPMC summary, replica dispatch), with the
 * arguments of those calls:
 *   logits [T,E] f32, x [T,H] bf16 (NULL with xp = NULL: permutation only),
 *   renorm, st / iter / layer / idx_prev (NULL for layer 0), replicate and its
 *   thresh_num / thresh_den / max_copies, and the outputs idx, w, hist_out
 *   (nullable), p_seq / cond / p_next (nullable; cond and p_next NULL for the
 *   last layer), copies / rep_base / group_expert (required when replicating),
 *   group_offsets [2E+1], perm, inv_perm, xp.
 *   workspace  ws_bytes >= moe_workspace_bytes(MOE_OP_LAYER_FRONT, T, k, E, H, 0),
 *              16-byte aligned
 * Replication before routing (prediction-driven): rep_share [E] fp32 (for
 * instance the p_next of the previous layer's prediction) makes the replica
 * table that of moe_replicate_predicted(rep_share, T*k, ..., budget) instead
 * of moe_replicate(hist, T*k) (T*k < 2^29); NULL keeps the layer's own
 * histogram.  budget bounds the total copies in both cases (-1 = none;
 * hottest experts first).  The tokens are still dispatched by their actual
 * choices, split over the replica groups of their expert.
 * The first launch routes tiles of tokens and counts them.  In the second,
 * one block folds the histogram and the co-selection counts into the window
 * and predicts, while every other block computes the replica table and the
 * group layout from the histogram (the same integers in each), then
 * scatters the permutation of its tile and copies its rows.  E must equal
 * the handle's E.
 * ------------------------------------------------------------------------- */
moe_status moe_layer_front(const float* logits, const uint16_t* x, int T, int E, int k, int H, int renorm,
                           moe_stats* st, int64_t iter, int layer, const int32_t* idx_prev, int replicate,
                           int thresh_num, int thresh_den, int max_copies, const float* rep_share, int budget,
                           int32_t* idx, float* w,
                           int32_t* hist_out, float* p_seq, float* cond, float* p_next, int32_t* copies,
                           int32_t* rep_base, int32_t* group_expert, int32_t* group_offsets, int32_t* perm,
                           int32_t* inv_perm, uint16_t* xp, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_expert_ffn -- grouped expert FFN over the dispatched rows.
 * PopFetcher review (MoE-GPT experts: GeLU MLP with F = alpha*H); EPS-MoE
 * review, "MoE architecture analysis" (gate, up, down GEMMs) and
 * "GroupGemm vs DenseGemm" (all experts in one grouped kernel, and a
 * separate path for small per-expert batches).
 *   xp             [A,H] bf16 dispatched rows
 *   group_offsets  [G+1] int32, G = 2E when group_expert is given, else E
 *   group_expert   [G] int32 expert of each group (-1 / empty groups
 *                  allowed) or NULL (group g = expert g)
 *   rep_base       [E+1] int32 or NULL; not needed by the kernels: adjacent
 *                  groups with the same expert (the layout moe_dispatch
 *                  writes) are treated as that expert's rows, tiled as one
 *                  range, and the kernel path is chosen from their total, so
 *                  every replica of an expert takes the same path and the
 *                  output does not depend on the replica split
 *   w1, w3         [E,H,F] bf16 (w1 = gate / first projection, w3 = up
 *                  projection, NULL for GeLU);  w2 [E,F,H] bf16
 *   act            MOE_ACT_GELU: y = gelu(x w1) w2 (exact erf)
 *                  MOE_ACT_SWIGLU: y = (silu(x w1) * (x w3)) w2
 *   small_group_threshold  experts with fewer rows use the small-batch kernel
 *                  (0 = never): Y^T = W^T X^T with the expert's rows as the
 *                  MMA N dimension (EPS-MoE review: DenseGemm below the
 *                  GroupGemm crossover); the others use the grouped kernel
 *   y              [A,H] bf16 out (fp32 accumulation, bf16 intermediate)
 *   workspace      ws_bytes >= moe_workspace_bytes(MOE_OP_EXPERT_FFN, T, k, E, H, F)
 *                  with T*k = A; 16-byte aligned (the bf16 intermediate
 *                  [A,F], then one counter per 256-row block for the fused
 *                  kernel, zeroed by the call)
 * H and F must be multiples of 64; all matrices 16-byte aligned.
 * ------------------------------------------------------------------------- */
moe_status moe_expert_ffn(const uint16_t* xp, const int32_t* group_offsets,
                          const int32_t* group_expert, const int32_t* rep_base, int E, int A,
                          const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                          int H, int F, moe_act act, int small_group_threshold, uint16_t* y,
                          void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_expert_ffn_gather -- the same grouped expert FFN, reading the token
 * rows in place: the dispatch copy is folded into the first GEMM's operand
 * loads (EPS-MoE review, expert pipeline: the dispatched rows are only an
 * input of the expert GEMMs), so moe_dispatch / moe_layer_front can be run
 * with x = xp = NULL (permutation only).
 *   x              [T,H] bf16 token rows (not permuted)
 *   perm           [T*k] int32 slot -> assignment f (moe_dispatch's perm);
 *                  dispatched row i is x[perm[i] / k].  A value outside
 *                  [0, T*k) sets the device error word (MOE_ERR_DEVICE from
 *                  moe_check) and row 0 is read in its place.
 *   the other arguments as in moe_expert_ffn, with A = T*k.
 * y is bit-identical to moe_expert_ffn on the copied rows.  T = 0 is a valid
 * empty batch; the workspace is moe_workspace_bytes(MOE_OP_EXPERT_FFN, T, k,
 * E, H, F) bytes.
 * ------------------------------------------------------------------------- */
moe_status moe_expert_ffn_gather(const uint16_t* x, int T, const int32_t* perm, int k,
                                 const int32_t* group_offsets, const int32_t* group_expert,
                                 const int32_t* rep_base, int E, const uint16_t* w1,
                                 const uint16_t* w3, const uint16_t* w2, int H, int F, moe_act act,
                                 int small_group_threshold, uint16_t* y, void* workspace,
                                 size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_replicate_weights -- physical replica copies of hot experts' weights.
 * MoE-MPMC summary, contribution 2 (predicted experts physically replicated
 * on the GPU); PopFetcher review (expert copies moved on a separate stream).
 * The replica table stays on the device, so a kernel makes the copies.
 *   rep_base   [E+1] int32 device: moe_replicate's table (groups of expert e
 *              are rep_base[e] .. rep_base[e+1]-1)
 *   w_all      [2E-1, rows, cols] bf16: slots 0..E-1 hold the experts'
 *              weights (the caller's); the call writes the extra replicas to
 *              slots E.., expert e's q-th extra copy (q >= 1) to slot
 *              E + (rep_base[e] - e) + q - 1.  NULL: only group_slot.
 *              rows*cols a multiple of 8, 16-byte aligned.
 *   group_slot [2E] int32 device out (nullable): weight slot of every group
 *              (the expert's own slot for its first group, a copy's slot
 *              for the others, -1 past the last group)
 * Call once per weight matrix (w1, w3, w2: rows x cols = H x F or F x H).
 * ------------------------------------------------------------------------- */
moe_status moe_replicate_weights(const int32_t* rep_base, int E, uint16_t* w_all, int rows, int cols,
                                 int32_t* group_slot, void* stream);

/* ---------------------------------------------------------------------------
 * moe_expert_ffn_slots -- the grouped expert FFN with each group reading
 * its own weight slot (physical replicas, moe_replicate_weights).
 * MoE-MPMC summary, methodology (the tokens of an expert spread over its
 * distinct physical replicas, each computing with its own copy); the
 * arithmetic is moe_expert_ffn's (EPS-MoE review: gate, up and down GEMMs).
 *   group_slot  [G] int32: weight slot of group g (-1 / empty groups
 *               allowed); G <= 512
 *   n_slots     weight slots in w1/w3/w2 ([n_slots,H,F] / [n_slots,F,H]),
 *               <= 512
 *   the other arguments as moe_expert_ffn; workspace as for moe_expert_ffn
 *   with G groups (moe_workspace_bytes(MOE_OP_EXPERT_FFN, T, k, E, H, F)
 *   covers G = 2E).
 * The output equals moe_expert_ffn's with the logical table when the slots
 * hold copies of the same weights (each row's arithmetic is the same).
 * ------------------------------------------------------------------------- */
moe_status moe_expert_ffn_slots(const uint16_t* xp, const int32_t* group_offsets, const int32_t* group_slot,
                                int G, int n_slots, int A, const uint16_t* w1, const uint16_t* w3,
                                const uint16_t* w2, int H, int F, moe_act act, int small_group_threshold,
                                uint16_t* y, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_expert_ffn_combine -- moe_expert_ffn and moe_combine in one call, the
 * combine done in the second GEMM's epilogue.
 * EPS-MoE review (expert pipelining: fusing the LocalReduce of expert outputs
 * into the expert computation).  Each dispatched row's GEMM2 result, times its
 * gate weight w[perm[i]], is added with fp32 reductions into row perm[i] / k of
 * an fp32 [T, H] accumulator in the workspace (zeroed by the call); a last
 * pass rounds it once to bf16 into out.  Y is never stored.
 *   Arguments as moe_expert_ffn (xp, group_offsets, group_expert, rep_base,
 *   E, weights, H, F, act, small_group_threshold) and moe_combine (perm from
 *   the same dispatch, w [T,k] f32, T, k); out bf16 [T,H].
 *   workspace  >= moe_workspace_bytes(MOE_OP_EXPERT_FFN_COMBINE, T, k, E, H, F),
 *              256-byte aligned.
 * Arithmetic: fp32 sums of w * (fp32 GEMM2 result) -- Y is not rounded to
 * bf16 first, so out can differ from moe_expert_ffn + moe_combine by about
 * one bf16 rounding; for k <= 2 every sum is two additions onto zero and the
 * result does not depend on their order (bit-reproducible); for k > 2 the
 * order of the reductions, and so the last bits, may vary between runs.
 * Uses the two-launch grouped kernels (not the fused one).
 * ------------------------------------------------------------------------- */
moe_status moe_expert_ffn_combine(const uint16_t* xp, const int32_t* group_offsets, const int32_t* group_expert,
                                  const int32_t* rep_base, int E, const int32_t* perm, const float* w, int T, int k,
                                  const uint16_t* w1, const uint16_t* w3, const uint16_t* w2, int H, int F,
                                  moe_act act, int small_group_threshold, uint16_t* out, void* workspace,
                                  size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_ffn_backward -- backward of the routed expert layer: combine, expert
 * FFN and dispatch copy.
 * PopFetcher (ATC'25) review: the system trains MoE models; in the backward
 * pass the gradients of an expert's replicas are reduced into the primary
 * expert (core method; design trade-offs).  Here every row routed to expert e,
 * in whichever of its replica groups, adds into the one gradient dW[e].
 *
 * Forward being differentiated (moe_dispatch -> moe_expert_ffn -> moe_combine):
 *   xp[i] = x[t(i)],  Y = FFN_e(xp),  out[t] = sum_r w[t,r] Y[inv_perm[t k + r]].
 * Given dout = dL/dout:
 *   dY[i] = w[t,r] dout[t];  dw[t,r] = <dout[t], Y[inv_perm[t k + r]]>;
 *   GeLU:   z = xp W1, a = gelu(z), dA = dY W2^T, dz = dA gelu'(z),
 *           dW2[e] = a^T dY, dW1[e] = xp^T dz, dxp = dz W1^T;
 *   SwiGLU: g = xp W1, u = xp W3, a = silu(g) u, dg = dA u silu'(g),
 *           du = dA silu(g), dW1 = xp^T dg, dW3 = xp^T du,
 *           dxp = dg W1^T + du W3^T;
 *   dx[t] = sum_r dxp[inv_perm[t k + r]].
 * Arithmetic: bf16 operands, fp32 accumulation; dY, a, the derivative
 * factors (gelu'(z); u silu'(g) and silu(g)), dz (dg, du) and dxp are rounded
 * to bf16 between the GEMMs (as the forward rounds its intermediate); dA
 * stays fp32 in the accumulator; the weight gradients and dw are fp32.
 *
 *   x, dout      bf16 [T, H]: the layer input and the output's gradient
 *   w            f32 [T, k] gate weights (moe_route)
 *   y            bf16 [A, H] the forward FFN output in dispatched order, or
 *                NULL: then dw is not computed (dw may be NULL)
 *   perm, inv_perm, group_offsets, group_expert, E: from moe_dispatch (or
 *                moe_layer_front) of the same routing; group_expert NULL =
 *                group g is expert g (E groups), else 2E groups.  The groups of
 *                one expert must be adjacent (as the dispatch writes them).
 *   w1, w3, w2   expert weights as in moe_expert_ffn (w3 NULL for GeLU)
 *   dx           bf16 [T, H] out
 *   dw           f32 [T, k] out (when y is given)
 *   dw1, dw3, dw2  [E, H, F], [E, H, F] (SwiGLU; else NULL), [E, F, H] out, f32
 *                (bf16 bit patterns with MOE_BWD_WGRAD_BF16): every expert's
 *                gradient is written (0 for experts without rows), or added to
 *                what they hold with MOE_BWD_ACCUMULATE_WGRAD
 *   flags        0 or a combination of MOE_BWD_ACCUMULATE_WGRAD (dW += this
 *                batch's gradient: gradient accumulation over micro-batches)
 *                and MOE_BWD_WGRAD_BF16 (the fp32 results rounded once to bf16:
 *                half the bytes written; not with accumulation); dx and dw are
 *                always written
 *   workspace    ws_bytes >= moe_ffn_backward_workspace_bytes(T, k, E, H, F),
 *                256-byte aligned; holds the padded intermediates (each
 *                expert's rows start at a multiple of 64, zero-padded).
 * Seven launches on `stream`.  Errors: MOE_ERR_INVALID (sizes as moe_expert_ffn,
 * null or misaligned pointers, y without dw), MOE_ERR_WORKSPACE; invalid device
 * data (offsets, permutation, an expert's groups not adjacent) sets the
 * device error word.
 * ------------------------------------------------------------------------- */
#define MOE_BWD_ACCUMULATE_WGRAD 1
#define MOE_BWD_WGRAD_BF16 2
size_t moe_ffn_backward_workspace_bytes(int T, int k, int E, int H, int F);
moe_status moe_ffn_backward(const uint16_t* x, const uint16_t* dout, const float* w, const uint16_t* y,
                            const int32_t* perm, const int32_t* inv_perm, int T, int k,
                            const int32_t* group_offsets, const int32_t* group_expert, int E,
                            const uint16_t* w1, const uint16_t* w3, const uint16_t* w2, int H, int F,
                            moe_act act, uint16_t* dx, float* dw, void* dw1, void* dw3, void* dw2,
                            int flags, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_route_backward -- gradient of the gate weights with respect to the
 * router logits, the chosen experts held fixed (the top-k choice is piecewise
 * constant).  PopFetcher and EPS-MoE reviews: softmax gate over the chosen
 * experts (renorm = 1) or over all E (renorm = 0), as moe_route.
 *   renorm = 1: dlogits[t, e_r] = w_r (dw_r - sum_s w_s dw_s), 0 elsewhere
 *   renorm = 0: dlogits[t, j] = p_j (g_j - sum_r dw_r p[e_r]),
 *               p = softmax(logits[t]), g_j = dw_r if j = e_r else 0
 *   logits f32 [T, E]; idx i32 [T, k] (moe_route); dw f32 [T, k];
 *   dlogits f32 [T, E] out.  fp32 arithmetic.  One launch.
 * ------------------------------------------------------------------------- */
moe_status moe_route_backward(const float* logits, const int32_t* idx, const float* dw, int T, int E, int k,
                              int renorm, float* dlogits, void* stream);

/* ---------------------------------------------------------------------------
 * moe_combine -- gate-weighted sum of each token's expert outputs.
 * EPS-MoE review, compute/communication overlap (LocalReduce of expert
 * outputs); PopFetcher review (result collect).
 *   out[t] = sum_{r<k} w[t,r] * y[inv_perm[t*k+r]], accumulated in fp32 in
 *   rank order r = 0..k-1, rounded once to bf16.
 *   y [A,H] bf16, inv_perm [A] int32, w [T,k] fp32, out [T,H] bf16.
 * H must be a multiple of 8; y and out 16-byte aligned.
 * ------------------------------------------------------------------------- */
moe_status moe_combine(const uint16_t* y, const int32_t* inv_perm, const float* w, int T,
                       int k, int H, uint16_t* out, void* stream);

/* ---------------------------------------------------------------------------
 * moe_dispatch_noalloc -- moe_dispatch without a caller-provided workspace.
 * The paper has no counterpart to this call.  It is for callers that cannot
 * allocate device memory at dispatch time: a host framework that owns all
 * device memory and forbids plug-ins from allocating, code enqueueing work
 * while a stream is being captured, or a latency-critical thread that must
 * not call cudaMalloc (it can synchronise the device).  The caller still
 * passes the inputs and outputs exactly as for moe_dispatch (same meaning,
 * layout and results); the scratch is a file-scope device array of
 * MOE_DISPATCH_NOALLOC_SCRATCH_BYTES (1 MiB) that every GPU loading the
 * library holds until the process exits.
 *   Limit   T*k assignments over E experts must need at most 1 MiB of
 *           scratch (moe_workspace_bytes(MOE_OP_DISPATCH, ...) <= 1 MiB:
 *           about 16.7M assignments at E = 16, 1.04M at E = 256); larger
 *           requests return MOE_ERR_WORKSPACE and enqueue nothing.
 *   Set-up  the first call on a device (with that device current) looks up
 *           the array's device address once; make that first call before
 *           any stream capture.  The address is kept for the life of the
 *           process: after cudaDeviceReset (or anything else that destroys
 *           the device's primary context) it is stale, and this call must
 *           not be used on that device again in the same process.
 *   Sharing every call on a device uses the same array, which keeps the last
 *           call's contents (each call writes every word it reads, so nothing
 *           needs clearing).  Calls whose work overlaps on the GPU (different
 *           streams, or different host threads) race on the array: order
 *           them on one stream.
 * Calls no cudaMalloc / cudaFree and no allocating library routine.
 * ------------------------------------------------------------------------- */
#define MOE_DISPATCH_NOALLOC_SCRATCH_BYTES (1u << 20)
moe_status moe_dispatch_noalloc(const uint16_t* x, const int32_t* idx, int T, int k, int H, int E,
                                const int32_t* rep_base, int32_t* group_offsets, int32_t* perm,
                                int32_t* inv_perm, uint16_t* xp, void* stream);

/* ---------------------------------------------------------------------------
 * Library options (process-wide, host side; no device work).
 *   MOE_OPT_FFN_KERNEL  which grouped-GEMM kernel moe_expert_ffn launches:
 *     MOE_FFN_KERNEL_AUTO   (default) when the experts average >= 256 rows
 *                           (A >= 256*E): a CTA-pair kernel (tcgen05
 *                           cta_group::2, 256-row tiles over two SMs) -- the
 *                           fused one (both GEMMs in one launch, tiles
 *                           interleaved block by block) when one expert's
 *                           weights take at most 16 MB, else the two-launch
 *                           one (moe_expert_ffn_gather always uses the
 *                           two-launch one); otherwise the single-CTA kernel
 *                           (128-row tiles).  The choice depends only on
 *                           (A, E, H, F, act).
 *     MOE_FFN_KERNEL_SINGLE / MOE_FFN_KERNEL_PAIR / MOE_FFN_KERNEL_FUSED
 *                           force one kernel (PAIR: two launches).
 * All kernels give bit-identical outputs except SINGLE vs the pair kernels
 * (different tiles; the same math, within the FFN tolerance).
 *   MOE_OPT_FFN_TIMEOUT_SELFTEST  value 1 arms a one-shot self-test of the
 *     bounded waits: in the next moe_expert_ffn call, the first GEMM's CTA
 *     (pair) 0 never signals its first accumulator, so its epilogue's wait
 *     runs out after ~2 s; the kernel then releases its resources and
 *     returns, and moe_check reports MOE_ERR_TIMEOUT (that call's output is
 *     incomplete).  The option resets itself after that call.
 *   MOE_OPT_PDL  1 (default): the route/plan, scatter/copy, grouped FFN and
 *     combine kernels are launched as programmatic dependents of the
 *     previous kernel in their stream (CUDA programmatic dependent launch):
 *     the hardware may start one once every block of the kernel before it
 *     has exited, and each waits for that kernel's completion (griddepcontrol
 *     .wait) before touching memory.  Only the front's route kernel releases
 *     its dependent early (for rows of at most 64 KB per dispatch tile: the
 *     scatter/copy blocks start while it runs and prefetch their token rows
 *     into L2, reading nothing the route kernel writes before their own wait).
 *     0: ordinary launches.  Results are identical either way.
 *   MOE_OPT_FFN_SMALL_SMS  how the SMs are shared between the small-batch
 *     kernels and the grouped kernels of an expert-FFN call whose
 *     small_group_threshold is > 0 (EPS-MoE review, "GroupGemm vs
 *     DenseGemm": experts with few tokens on a separate path):
 *       0 (default)   no small-batch path: the grouped kernels take every
 *                     expert (their schedule mixes the tiles of experts with
 *                     one row tile, which stream weights, with the others)
 *                     and the small-batch kernels are not launched.  On
 *                     B300 no split measured faster on the workloads this
 *                     library was tuned on, and the model below chose none,
 *                     so by default the two launches are left out;
 *       -1            each call's kernels choose from the group table, all
 *                     the same way: the small-batch kernels (a weight
 *                     stream, bound by HBM) get the SMs that balance their
 *                     time against the grouped kernels' (bound by the
 *                     tensor pipe) on the rest, and both run at once; when
 *                     running the small experts as padded grouped tiles on
 *                     every SM is expected to be faster, they do that
 *                     instead and the small-batch kernels exit at once;
 *       n > 0         the small-batch kernels use n SMs (even n with the
 *                     CTA-pair kernels), the grouped kernels the rest.
 *     The outputs are the same within the FFN tolerance whichever path an
 *     expert takes (bit-identical for the experts on the grouped kernels).
 *   MOE_OPT_FRONT_ONE_LAUNCH  0 (default): moe_layer_front makes two
 *     launches (route/count, then plan, statistics, ranks and copy).  1: it
 *     runs as one cooperative launch when all of its blocks (one per
 *     dispatch tile, plus one) can be resident on the device at once: each
 *     block routes its own tile, the blocks meet at a grid-wide barrier (a
 *     bounded wait: after ~2 s moe_check reports MOE_ERR_TIMEOUT and the
 *     call's outputs are not to be used), then the dispatch runs as in the
 *     two-launch form; other sizes take the two launches.  The outputs are
 *     bit-identical either way; on B300 the one launch measured slower on
 *     the 16K-token layer and no faster on the others.
 * Unknown options or values return MOE_ERR_INVALID.  Options are process-wide
 * and stored atomically; a call reads each one once when it is made, so a
 * set from another thread applies to the calls that start after it returns
 * (a call made at the same time sees the old or the new value).
 * ------------------------------------------------------------------------- */
typedef enum {
    MOE_OPT_FFN_KERNEL = 1,
    MOE_OPT_FFN_TIMEOUT_SELFTEST = 2,
    MOE_OPT_PDL = 3,
    MOE_OPT_FFN_SMALL_SMS = 4,
    MOE_OPT_FRONT_ONE_LAUNCH = 5
} moe_option;
typedef enum {
    MOE_FFN_KERNEL_AUTO = 0,
    MOE_FFN_KERNEL_SINGLE = 1,
    MOE_FFN_KERNEL_PAIR = 2,
    MOE_FFN_KERNEL_FUSED = 3
} moe_ffn_kernel;
moe_status moe_set_option(int option, int value);
moe_status moe_get_option(int option, int* value /* host */);

/* Kernel launches one moe_expert_ffn (gather = 0) or moe_expert_ffn_gather
 * (gather = 1) call makes under the current options: 1 (fused) or 2 grouped
 * launches, plus 2 small-batch launches when small_group_threshold > 0 and
 * MOE_OPT_FFN_SMALL_SMS is not 0.
 * 0 for sizes, activations or thresholds the FFN refuses.  Host only. */
int moe_ffn_launches(int A, int E, int H, int F, int act, int small_group_threshold, int gather);

/* Kernel launches one moe_layer_front call with T > 0 tokens makes on the
 * current device under the current options: 1 when it runs as one
 * cooperative launch (MOE_OPT_FRONT_ONE_LAUNCH on, and all of its blocks can
 * be resident at once), else 2.  has_prev: the call passes the previous
 * layer's choices (co-selection counts kept).  0 for T <= 0 (an empty batch
 * runs the separate calls instead), for sizes moe_layer_front refuses, or
 * when no device can be queried.  Host only (queries the device's occupancy). */
int moe_layer_front_launches(int T, int E, int k, int has_prev);

/* Workspace bytes for op (MOE_OP_DISPATCH, MOE_OP_EXPERT_FFN, MOE_OP_LAYER_FRONT or
 * MOE_OP_EXPERT_FFN_COMBINE); 0 for bad sizes. */
size_t moe_workspace_bytes(int op, int T, int k, int E, int H, int F);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device: MOE_ERR_TIMEOUT if a bounded wait ran out, MOE_ERR_DEVICE if
 * a kernel met invalid data, MOE_ERR_CUDA on an asynchronous CUDA error. */
moe_status moe_check(void* stream);

/* Raw device error word of the current device (bit 0: invalid data, bit 1:
 * timeout), without clearing it; synchronises the device. */
moe_status moe_error_word(uint32_t* word_out /* host */);

const char* moe_status_string(moe_status s);

/* Text of the last MOE_ERR_CUDA / MOE_ERR_INVALID raised by this thread. */
const char* moe_last_error(void);

/* Checkpoint / resume of the window state: moe_stats_bytes gives the size;
 * export copies ring buffers and window sums into host memory (synchronous,
 * after all work queued on the legacy stream), import restores them. */
size_t moe_stats_bytes(const moe_stats* st);
moe_status moe_stats_export(const moe_stats* st, void* host_buf, size_t bytes);
moe_status moe_stats_import(moe_stats* st, const void* host_buf, size_t bytes);

/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */

"""CPU oracle for the MoE routing-and-expert step (test infrastructure).

This module is test infrastructure, not product code.  Only the tests, the
`smoke()` check and the benchmark's CPU-baseline leg may import it; the
library's compute path never calls it and has no CPU fallback.

It is a plain, slow, obviously-correct restatement of what the step computes,
in float64 (integers exact), written from the pages:

  * top-k gate over router logits -- PopFetcher (ATC'25) review, "core method"
    and experiments (naive top-k gate); EPS-MoE review, experiment set-up
    (top-2 / top-4 / top-6 models); gate weights renormalised over the chosen
    experts (softmax over the k selected logits).
  * per-expert token histogram and layer j -> j+1 co-selection counts --
    PopFetcher review, observation 1 (token allocation statistics) and
    observation 2 / Fig. 6 (conditional probability Pr(E^{h,j+1} | E^{i,j})).
  * sliding-window popularity p_seq and predicted next-layer popularity --
    PopFetcher review, "core method": Routing Information Collector, window
    s = 10, Eq. (1) and Eq. (2)(3); MoE-GPS blog section 2.1 (maximum-
    likelihood p_i = n_i / N with a sliding-window average).
  * replica counts for hot experts -- MoE-GPS blog section 2.1,
    `duplicate_experts` (threshold 1.2 x target, copies = ceil(load/target)-1);
    MoE-MPMC summary, contributions 2 (physical replication) and 3 (capacity
    bound).
  * prediction-driven replication and prediction quality -- MoE-GPS blog
    section 2.1 (sliding-window estimate with a decay factor against drift),
    MoE-MPMC summary contribution 3 (replica counts bounded by a memory
    budget), PopFetcher review (top-5 next-layer prediction accuracy, s = 10),
    "Prediction Is All MoE Needs" (mean error of the predicted expert-load
    proportion).
  * backward of the routed FFN (PopFetcher trains the MoE models it routes:
    its prefetched expert copies send their gradients back to the primary
    expert for the reduction) -- the gradients of the expert FFN, the
    combine and the gate weights, with every replica's rows reducing into
    its expert's one gradient.
  * stable dispatch by expert / replica and the gate-weighted combine --
    PopFetcher review, problem statement (token dispatch + result collect);
    EPS-MoE review, compute/communication overlap (LocalReduce); MoE-MPMC
    summary (tokens of one expert spread over distinct replicas).
  * expert FFN (GeLU MLP for MoE-GPT; SwiGLU gate/up/down for Mixtral,
    DeepSeekV2, DBRX) -- PopFetcher review (alpha = F/H); EPS-MoE review,
    "MoE architecture analysis" (gate, up, down GEMMs).

Readings of points the pages leave open are stated where they are used; every
one is also listed in the repository's design notes.

Parity pins: every function here is pinned by `-m "not gpu"` tests against
brute force, hand-computed tables or closed forms.

Parity unpinned (the pages print no formula or value to pin against):
  * the numerical content of Eq. (1)-(3) beyond the "window sums of counts,
    normalised" reading -- that reading is pinned by the stationary-stream
    closed form and brute-force window sums, not by printed values;
  * the decay weighting of predict_decay beyond its reading (weights
    lam**age) -- pinned by hand-derived cases of that reading only.
"""
from __future__ import annotations

import math
from fractions import Fraction
from typing import Optional

import numpy as np
from scipy.special import erf as _erf

__all__ = ["bf16_to_f64", "topk_gate", "histogram", "coselection", "WindowStats",
           "replicate", "dispatch", "gather_rows", "expert_ffn_rows", "expert_ffn",
           "combine", "moe_layer"]


# ----------------------------------------------------------------------------
# bf16 decoding: a bf16 value is the top 16 bits of an IEEE binary32.
# ----------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Top-k gate
# ----------------------------------------------------------------------------
def topk_gate(logits: np.ndarray, k: int, renorm: bool = True):
    """Top-k gate (PopFetcher review: naive top-k gate).

    For every token, order the (logit, expert) pairs by logit descending and,
    on equal logits, by expert index ascending; the first k are the chosen
    experts in rank order.  (The tie rule is not on the pages; the lower index
    wins.  -0.0 and +0.0 are equal logits.)

    Gate weights (EPS-MoE review, Mixtral: softmax-renormalised):
      renorm=True : w_r = exp(l_r - l_0) / sum_{r'<k} exp(l_r' - l_0)
      renorm=False: w_r = exp(l_r - m) / sum_e exp(l_e - m), m = max_e l_e
    Returns idx int32 [T,k] and w float64 [T,k]."""
    l = np.asarray(logits)
    T, E = l.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    l64 = l.astype(np.float64)
    eidx = np.broadcast_to(np.arange(E), (T, E))
    # lexsort: last key is primary.  Primary: -logit ascending (= logit
    # descending); secondary: expert index ascending.
    order = np.lexsort((eidx, -l64), axis=-1)
    idx = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(l64, idx.astype(np.int64), axis=1)
    if renorm:
        z = np.exp(sel - sel[:, :1])
        w = z / z.sum(axis=1, keepdims=True)
    else:
        m = l64.max(axis=1, keepdims=True)
        z = np.exp(l64 - m)
        w = np.take_along_axis(z, idx.astype(np.int64), axis=1) / z.sum(axis=1, keepdims=True)
    return idx, w


# ----------------------------------------------------------------------------
# Token allocation statistics
# ----------------------------------------------------------------------------
def histogram(idx: np.ndarray, E: int) -> np.ndarray:
    """h[e] = number of (token, rank) assignments routed to expert e
    (PopFetcher review, observation 1: token allocation per expert)."""
    flat = np.asarray(idx).reshape(-1).astype(np.int64)
    return np.bincount(flat, minlength=E).astype(np.int64)


def coselection(idx_prev: np.ndarray, idx_cur: np.ndarray, E: int) -> np.ndarray:
    """C[e, e'] = number of tokens t with e in S_prev(t) and e' in S_cur(t)
    (PopFetcher review, observation 2 / Fig. 6: layer-to-layer selection
    counts behind Pr(E^{h,j+1} | E^{i,j})).

    Reading (the pages do not say which pairs count): every one of the k x k
    (previous choice, current choice) pairs of a token counts once."""
    a = np.asarray(idx_prev).astype(np.int64)
    b = np.asarray(idx_cur).astype(np.int64)
    C = np.zeros((E, E), dtype=np.int64)
    k_prev, k_cur = a.shape[1], b.shape[1]
    for r1 in range(k_prev):
        for r2 in range(k_cur):
            np.add.at(C, (a[:, r1], b[:, r2]), 1)
    return C


class WindowStats:
    """Sliding-window routing statistics and next-layer prediction.

    PopFetcher review, "core method" (Routing Information Collector): the
    token allocation of each layer is kept over a window of s = 10
    iterations; Eq. (1) gives the sequence popularity p_seq, Eq. (2)(3)
    propagate it through the inter-layer conditional probability to the next
    layer.  MoE-GPS blog section 2.1 states the same estimate as the MLE
    p_i = n_i / N averaged over a sliding window.

    Readings (Eq. (1)-(3) are named but not printed):
      * the window holds the last s updates of each layer, by ring slot
        (iteration mod s); an update for an iteration already in its slot
        replaces it;
      * p_seq_j[e]       = H_j[e] / sum_e H_j[e],  H_j = window sum of h_j
                           (uniform 1/E while the window is empty);
      * Pr_j(e' | e)     = Cbar_j[e,e'] / sum_e'' Cbar_j[e,e''],
                           Cbar_j = window sum of C_j (row of zeros: 1/E);
      * p_next_{j+1}[e'] = sum_e p_seq_j[e] * Pr_j(e' | e).
    This object keeps only the raw per-slot counts and re-sums the window
    on every query."""

    def __init__(self, L: int, E: int, window: int = 10):
        if L < 1 or E < 1 or window < 1:
            raise ValueError("bad sizes")
        self.L, self.E, self.s = L, E, window
        self.h = np.zeros((L, window, E), dtype=np.int64)
        self.C = np.zeros((max(L - 1, 0), window, E, E), dtype=np.int64)

    def update(self, it: int, layer: int, idx_layer: np.ndarray,
               idx_prev: Optional[np.ndarray] = None) -> np.ndarray:
        """Record layer `layer`'s routing at iteration `it`; with `idx_prev`
        (layer-1's routing of the same tokens) also the co-selection counts
        between layer-1 and layer.  Returns this update's histogram."""
        slot = it % self.s
        h = histogram(idx_layer, self.E)
        self.h[layer, slot] = h
        if layer > 0:
            if idx_prev is None:
                raise ValueError("layer > 0 needs the previous layer's routing")
            self.C[layer - 1, slot] = coselection(idx_prev, idx_layer, self.E)
        return h

    def window_hist(self, layer: int) -> np.ndarray:
        return self.h[layer].sum(axis=0)

    def window_cosel(self, layer: int) -> np.ndarray:
        """Cbar between `layer` and `layer`+1."""
        return self.C[layer].sum(axis=0)

    def predict(self, layer: int):
        """(p_seq_j, Pr_j, p_next_{j+1}); the last two are None for the last layer."""
        E = self.E
        H = self.window_hist(layer)
        tot = H.sum()
        p_seq = H / tot if tot > 0 else np.full(E, 1.0 / E)
        if layer >= self.L - 1:
            return p_seq, None, None
        Cb = self.window_cosel(layer).astype(np.float64)
        rows = Cb.sum(axis=1)
        cond = np.empty((E, E), dtype=np.float64)
        for e in range(E):
            cond[e] = Cb[e] / rows[e] if rows[e] > 0 else 1.0 / E
        p_next = p_seq @ cond
        return p_seq, cond, p_next

    def predict_decay(self, layer: int, it: int, lam: float):
        """Prediction from a decay-weighted window.  MoE-GPS blog section 2.1:
        the sliding-window average carries a decay factor against drift.

        Reading (no formula is printed): under the causal order (layer j
        updated at iteration `it`, then predicted, then layer j+1 updated),
        the ring slot of iteration it - a weighs lam**a in the histogram sums
        H_j, and the slot of iteration it - 1 - a weighs lam**a in the
        co-selection sums Cbar_j, a = 0 .. s-1; the three quantities are then
        formed exactly as in predict().  lam = 1 is predict(); lam = 0 keeps
        only the newest iteration (0**0 = 1)."""
        E, s = self.E, self.s
        if not (0.0 <= lam <= 1.0):
            raise ValueError("lam must lie in [0, 1]")
        wts = [1.0 if a == 0 else lam ** a for a in range(s)]
        H = np.zeros(E, dtype=np.float64)
        for a in range(s):
            H += wts[a] * self.h[layer, (it - a) % s].astype(np.float64)
        tot = H.sum()
        p_seq = H / tot if tot > 0 else np.full(E, 1.0 / E)
        if layer >= self.L - 1:
            return p_seq, None, None
        Cb = np.zeros((E, E), dtype=np.float64)
        for a in range(s):
            Cb += wts[a] * self.C[layer, (it - 1 - a) % s].astype(np.float64)
        rows = Cb.sum(axis=1)
        cond = np.empty((E, E), dtype=np.float64)
        for e in range(E):
            cond[e] = Cb[e] / rows[e] if rows[e] > 0 else 1.0 / E
        p_next = p_seq @ cond
        return p_seq, cond, p_next


# ----------------------------------------------------------------------------
# Prediction-driven replication and prediction quality
# ----------------------------------------------------------------------------
def apportion(p32: np.ndarray, total: int) -> np.ndarray:
    """Integer loads summing to `total` in proportion to the predicted
    popularity (so that replica counts can be taken from a prediction).

    Reading of "feed round(p * A) into the replica rule": plain rounding can
    miss the total, which the replica rule needs as its bound, so the loads
    are the largest-remainder apportionment of `total`: q_e = p_e * total
    computed exactly from the float32 values (p_e = m * 2**x, m an integer),
    floors first, then one more for the experts with the largest remainders
    (ties: lower expert first), repeated while any is left; a negative p
    counts as 0.  Should the floors exceed `total` (p summing above 1 by
    rounding), one is taken back from the experts with the smallest
    remainders among those with a positive floor (ties: higher expert first).
    Exact rational arithmetic throughout."""
    p32 = np.asarray(p32, dtype=np.float32).reshape(-1)
    E = p32.size
    q = [max(Fraction(float(v)), Fraction(0)) * total for v in p32]   # float32 -> exact rational
    f = [math.floor(v) for v in q]
    r = [q[e] - f[e] for e in range(E)]
    left = total - sum(f)
    order = sorted(range(E), key=lambda e: (-r[e], e))     # largest remainder, lower expert first
    while left > 0:
        for e in order:
            if left == 0:
                break
            f[e] += 1
            left -= 1
    back = list(reversed(order))                           # smallest remainder, higher expert first
    while left < 0:
        moved = False
        for e in back:
            if left == 0:
                break
            if f[e] > 0:
                f[e] -= 1
                left += 1
                moved = True
        if not moved:
            raise ValueError("cannot apportion")
    return np.array(f, dtype=np.int64)


def cap_copies(copies, load, budget: int):
    """Bound the total number of extra copies by a memory budget (MoE-MPMC
    summary, contribution 3: replica counts limited by a predefined GPU
    memory budget).  Reading: the hottest experts are served first -- experts
    in order of decreasing load (ties: lower expert first) each keep
    min(their copies, what is left of the budget).  budget < 0: no bound."""
    copies = [int(c) for c in copies]
    if budget < 0:
        return np.array(copies, dtype=np.int32)
    load = [int(v) for v in load]
    left = int(budget)
    out = [0] * len(copies)
    for e in sorted(range(len(copies)), key=lambda e: (-load[e], e)):
        out[e] = min(copies[e], left)
        left -= out[e]
    return np.array(out, dtype=np.int32)


def replicate_predicted(p32, total: int, thresh_num: int = 6, thresh_den: int = 5, max_copies: int = -1,
                        budget: int = -1):
    """Replica table from a predicted popularity: loads by apportion(), the
    replica rule of replicate(), then the budget bound of cap_copies().
    Returns (load, copies, rep_base, group_expert)."""
    load = apportion(p32, total)
    copies, _, _ = replicate(load, total, thresh_num, thresh_den, max_copies)
    copies = cap_copies(copies, load, budget)
    E = len(copies)
    rep_base = np.zeros(E + 1, dtype=np.int32)
    rep_base[1:] = np.cumsum(copies.astype(np.int64) + 1)
    group_expert = np.full(2 * E, -1, dtype=np.int32)
    g = 0
    for e in range(E):
        for _ in range(int(copies[e]) + 1):
            group_expert[g] = e
            g += 1
    return load.astype(np.int32), copies, rep_base, group_expert


def top_overlap(p_pred, load_actual, m: int = 5) -> float:
    """Top-m prediction accuracy (PopFetcher review: top-5 next-layer accuracy
    ~77% for the naive top-k gate at s = 10).  Reading: the share of the m
    most loaded experts of the layer (by its actual histogram) that are
    among the m most popular predicted ones; ties go to the lower expert on
    both sides."""
    p_pred = np.asarray(p_pred, dtype=np.float64).reshape(-1)
    load_actual = np.asarray(load_actual, dtype=np.int64).reshape(-1)
    m = min(m, p_pred.size)
    pred = sorted(range(p_pred.size), key=lambda e: (-p_pred[e], e))[:m]
    act = sorted(range(load_actual.size), key=lambda e: (-load_actual[e], e))[:m]
    return len(set(pred) & set(act)) / m


def load_proportion_error(p_pred, load_actual) -> float:
    """Mean error of the predicted expert-load proportion ("Prediction Is All
    MoE Needs": ~1.3% / ~1.8% for GPT3 350M).  Reading: mean over experts of
    |p_pred[e] - load[e] / sum(load)|, as a fraction (x100 for percent)."""
    p_pred = np.asarray(p_pred, dtype=np.float64).reshape(-1)
    load_actual = np.asarray(load_actual, dtype=np.float64).reshape(-1)
    tot = load_actual.sum()
    if tot <= 0:
        raise ValueError("empty load")
    return float(np.mean(np.abs(p_pred - load_actual / tot)))


# ----------------------------------------------------------------------------
# Replica counts
# ----------------------------------------------------------------------------
def replicate(load, total: int, thresh_num: int = 6, thresh_den: int = 5,
              max_copies: int = -1):
    """Replica counts for hot experts (MoE-GPS blog section 2.1,
    `duplicate_experts`): target = total / slots; an expert is hot when its
    load exceeds 1.2 x target, and then gets ceil(load / target) - 1 extra
    copies.  MoE-MPMC summary, contribution 3: a capacity bound caps the
    copies (`max_copies`, -1 = no cap).

    Readings: on one GPU every expert owns one slot, so slots = E and
    target = total / E; the garbled comparison is read as strict '>'.
    Exact rational arithmetic (Fraction), so the table is exact.

    Returns copies [E], rep_base [E+1] (exclusive scan of copies+1;
    rep_base[E] = number of groups) and group_expert [2E] (expert of each
    group, -1 past the last group)."""
    load = [int(v) for v in np.asarray(load).reshape(-1)]
    E = len(load)
    total = int(total)
    if total <= 0:
        raise ValueError("total must be positive")
    target = Fraction(total, E)
    thresh = Fraction(thresh_num, thresh_den)
    copies = []
    for ld in load:
        c = 0
        if ld > thresh * target:
            c = math.ceil(Fraction(ld) / target) - 1
        if max_copies >= 0:
            c = min(c, max_copies)
        copies.append(c)
    rep_base = [0]
    for c in copies:
        rep_base.append(rep_base[-1] + c + 1)
    group_expert = []
    for e, c in enumerate(copies):
        group_expert += [e] * (c + 1)
    if len(group_expert) > 2 * E:
        raise ValueError("more than 2E groups: loads exceed total")
    group_expert += [-1] * (2 * E - len(group_expert))
    return (np.array(copies, dtype=np.int32), np.array(rep_base, dtype=np.int32),
            np.array(group_expert, dtype=np.int32))


# ----------------------------------------------------------------------------
# Dispatch
# ----------------------------------------------------------------------------
def dispatch(idx: np.ndarray, E: int, rep_base: Optional[np.ndarray] = None):
    """Stable token permutation by expert, then replica.

    Assignments are numbered f = t*k + r.  An expert's assignments are taken
    in ascending f; the m-th (0-based) goes to replica q = m mod n_e of that
    expert (round-robin; MoE-MPMC summary: tokens of one expert are spread
    over distinct physical replicas), and within a replica keeps that order.
    Groups are ordered by expert, then replica: g = rep_base[e] + q.

    Returns group_offsets [2E+1] (exclusive scan of group sizes; entries past
    the last group equal A), perm [A] (slot -> f) and inv_perm [A] (f -> slot)."""
    idx = np.asarray(idx)
    T, k = idx.shape
    A = T * k
    if rep_base is None:
        rep_base = np.arange(E + 1, dtype=np.int64)
    rep_base = [int(v) for v in rep_base]
    n_groups = rep_base[E]
    groups = [[] for _ in range(n_groups)]
    seen = [0] * E
    flat = idx.reshape(-1)
    for f in range(A):
        e = int(flat[f])
        n_e = rep_base[e + 1] - rep_base[e]
        m = seen[e]
        seen[e] += 1
        groups[rep_base[e] + m % n_e].append(f)
    offsets = [0]
    for g in groups:
        offsets.append(offsets[-1] + len(g))
    offsets += [A] * (2 * E + 1 - len(offsets))
    perm = np.array([f for g in groups for f in g], dtype=np.int32)
    inv_perm = np.empty(A, dtype=np.int32)
    inv_perm[perm] = np.arange(A, dtype=np.int32)
    return np.array(offsets, dtype=np.int32), perm, inv_perm


def gather_rows(x: np.ndarray, perm: np.ndarray, k: int) -> np.ndarray:
    """Xp[slot] = X[perm[slot] // k] (bit copy)."""
    return np.asarray(x)[np.asarray(perm).astype(np.int64) // k]


# ----------------------------------------------------------------------------
# Expert FFN
# ----------------------------------------------------------------------------
def _gelu(z):
    # exact (erf) GeLU: z * Phi(z)
    return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))


def _silu(z):
    return z / (1.0 + np.exp(-z))


def expert_ffn_rows(x_rows: np.ndarray, experts: np.ndarray, w1, w3, w2, act: str) -> np.ndarray:
    """Expert FFN of individual rows, float64.

    x_rows: bf16 bits [n, H]; experts: [n] expert of each row; w1/w3: bf16
    bits [E,H,F] (w3 None for GeLU); w2: bf16 bits [E,F,H].
      GeLU  : y = gelu(x W1[e]) W2[e]
      SwiGLU: y = (silu(x W1[e]) * (x W3[e])) W2[e]
    (PopFetcher review: MoE-GPT experts, F = alpha*H; EPS-MoE review: gate,
    up and down GEMMs.)  Readings: exact-erf GeLU; no biases; w1 is the gate
    and w3 the up projection.  The intermediate stays float64."""
    x = bf16_to_f64(x_rows)
    experts = np.asarray(experts).astype(np.int64)
    n, H = x.shape
    y = np.zeros((n, w2.shape[2]), dtype=np.float64)
    for e in np.unique(experts):
        rows = np.nonzero(experts == e)[0]
        xe = x[rows]
        z = xe @ bf16_to_f64(w1[e])
        if act == "gelu":
            a = _gelu(z)
        elif act == "swiglu":
            a = _silu(z) * (xe @ bf16_to_f64(w3[e]))
        else:
            raise ValueError(act)
        y[rows] = a @ bf16_to_f64(w2[e])
    return y


def expert_ffn(xp: np.ndarray, group_offsets: np.ndarray, group_expert: Optional[np.ndarray],
               w1, w3, w2, act: str, slots: Optional[np.ndarray] = None) -> np.ndarray:
    """Y rows of the dispatched matrix Xp.  Slot s of group g is computed with
    expert group_expert[g] (identity when None).  `slots` restricts the work to
    those rows (returned in that order)."""
    go = np.asarray(group_offsets).astype(np.int64)
    A = int(go[-1])
    if slots is None:
        slots = np.arange(A)
    slots = np.asarray(slots).astype(np.int64)
    g = np.searchsorted(go, slots, side="right") - 1
    ge = np.arange(len(go)) if group_expert is None else np.asarray(group_expert)
    experts = np.asarray(ge)[g]
    return expert_ffn_rows(np.asarray(xp)[slots], experts, w1, w3, w2, act)


# ----------------------------------------------------------------------------
# Backward of the routed FFN
# ----------------------------------------------------------------------------
def _gelu_grad(z):
    # d/dz [z Phi(z)] = Phi(z) + z phi(z)
    return 0.5 * (1.0 + _erf(z / math.sqrt(2.0))) + z * np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)


def _silu_grad(z):
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def expert_ffn_backward_f64(x, experts, w1, w3, w2, act: str, dy):
    """Gradients of expert_ffn_rows, all in float64 (x [n,H], w1/w3 [E,H,F],
    w2 [E,F,H] and dy [n,H] float64).  Per row of expert e:
      GeLU  : z = x W1, a = gelu(z), y = a W2
              dA = dy W2^T, dz = dA * gelu'(z),
              dW2 += a^T dy, dW1 += x^T dz, dx = dz W1^T
      SwiGLU: g = x W1, u = x W3, a = silu(g) * u, y = a W2
              dA = dy W2^T, dg = dA * u * silu'(g), du = dA * silu(g),
              dW2 += a^T dy, dW1 += x^T dg, dW3 += x^T du,
              dx = dg W1^T + du W3^T
    Every row adds into its expert's gradients, so the rows of an expert's
    replica groups reduce into the expert's one gradient.
    Returns dx [n,H], dw1 [E,H,F], dw3 [E,H,F] or None, dw2 [E,F,H]."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    experts = np.asarray(experts).astype(np.int64)
    w1 = np.asarray(w1, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    w3 = None if w3 is None else np.asarray(w3, dtype=np.float64)
    dx = np.zeros_like(x)
    dw1 = np.zeros_like(w1)
    dw2 = np.zeros_like(w2)
    dw3 = None if w3 is None else np.zeros_like(w3)
    for e in np.unique(experts):
        rows = np.nonzero(experts == e)[0]
        xe, dye = x[rows], dy[rows]
        dA = dye @ w2[e].T
        if act == "gelu":
            z = xe @ w1[e]
            a = _gelu(z)
            dz = dA * _gelu_grad(z)
            dw1[e] += xe.T @ dz
            dx[rows] = dz @ w1[e].T
        elif act == "swiglu":
            g = xe @ w1[e]
            u = xe @ w3[e]
            a = _silu(g) * u
            dg = dA * u * _silu_grad(g)
            du = dA * _silu(g)
            dw1[e] += xe.T @ dg
            dw3[e] += xe.T @ du
            dx[rows] = dg @ w1[e].T + du @ w3[e].T
        else:
            raise ValueError(act)
        dw2[e] += a.T @ dye
    return dx, dw1, dw3, dw2


def combine_backward(dout, y, inv_perm, w):
    """Gradients of combine: out[t] = sum_r w[t,r] Y[slot(t,r)].
    dY[slot(t,r)] = w[t,r] dout[t];  dw[t,r] = <dout[t], Y[slot(t,r)]>.
    float64 in and out (y may be bf16 bits)."""
    dout = np.asarray(dout, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, k = w.shape
    yy = bf16_to_f64(y) if np.asarray(y).dtype == np.uint16 else np.asarray(y, dtype=np.float64)
    inv = np.asarray(inv_perm).astype(np.int64)
    dY = np.zeros_like(yy)
    dw = np.zeros((T, k), dtype=np.float64)
    for r in range(k):
        slots = inv[np.arange(T) * k + r]
        dY[slots] = w[:, r:r + 1] * dout
        dw[:, r] = np.sum(dout * yy[slots], axis=1)
    return dY, dw


def scatter_sum(dxp, inv_perm, T: int, k: int):
    """Token gradients from the dispatched rows: dx[t] = sum_r dxp[slot(t,r)]
    (the backward of the row copy xp[slot] = x[t])."""
    d = np.asarray(dxp, dtype=np.float64)
    inv = np.asarray(inv_perm).astype(np.int64)
    dx = np.zeros((T, d.shape[1]), dtype=np.float64)
    for r in range(k):
        dx += d[inv[np.arange(T) * k + r]]
    return dx


def router_backward(logits, idx, dw, renorm: bool = True):
    """Gradient of the gate weights with respect to the router logits, the
    choice of experts held fixed (it is piecewise constant).
      renorm: w_r = softmax over the k chosen logits ->
              dlogit[e_r] = w_r (dw_r - sum_s w_s dw_s), 0 elsewhere;
      full  : w_r = p[e_r], p = softmax over all E ->
              dlogit[j] = p_j (g_j - sum_r dw_r p[e_r]), g_j = dw_r if j = e_r else 0."""
    l = np.asarray(logits, dtype=np.float64)
    idx = np.asarray(idx).astype(np.int64)
    dw = np.asarray(dw, dtype=np.float64)
    T, E = l.shape
    out = np.zeros((T, E), dtype=np.float64)
    for t in range(T):
        sel = l[t, idx[t]]
        if renorm:
            z = np.exp(sel - sel.max())
            w = z / z.sum()
            out[t, idx[t]] = w * (dw[t] - np.dot(w, dw[t]))
        else:
            z = np.exp(l[t] - l[t].max())
            p = z / z.sum()
            g = np.zeros(E)
            g[idx[t]] = dw[t]
            out[t] = p * (g - np.dot(dw[t], p[idx[t]]))
    return out


# ----------------------------------------------------------------------------
# Combine
# ----------------------------------------------------------------------------
def combine(y: np.ndarray, inv_perm: np.ndarray, w: np.ndarray) -> np.ndarray:
    """out[t] = sum_r w[t,r] * Y[inv_perm[t*k + r]] (EPS-MoE review: the
    LocalReduce of expert outputs; PopFetcher review: result collect).
    y is float64 (or bf16 bits, decoded); result float64 [T, H]."""
    w = np.asarray(w, dtype=np.float64)
    T, k = w.shape
    yy = bf16_to_f64(y) if np.asarray(y).dtype == np.uint16 else np.asarray(y, dtype=np.float64)
    inv = np.asarray(inv_perm).astype(np.int64)
    out = np.zeros((T, yy.shape[1]), dtype=np.float64)
    for r in range(k):
        out += w[:, r:r + 1] * yy[inv[np.arange(T) * k + r]]
    return out


# ----------------------------------------------------------------------------
# Whole layer (end to end, for a subset of tokens if asked)
# ----------------------------------------------------------------------------
def moe_layer(logits, x_bits, k, w1, w3, w2, act, *, renorm=True, replicate_on=False,
              thresh=(6, 5), max_copies=-1, tokens: Optional[np.ndarray] = None):
    """Route -> (replicate) -> dispatch -> FFN -> combine for one layer.

    The routing, counts and dispatch cover all tokens (they are global);
    the FFN and combine are evaluated for `tokens` only (all when None).
    Returns a dict with every intermediate and out [len(tokens), H] float64."""
    logits = np.asarray(logits)
    T, E = logits.shape
    idx, w = topk_gate(logits, k, renorm)
    h = histogram(idx, E)
    rep = replicate(h, T * k, thresh[0], thresh[1], max_copies) if replicate_on else None
    go, perm, inv = dispatch(idx, E, None if rep is None else rep[1])
    tokens = np.arange(T) if tokens is None else np.asarray(tokens).astype(np.int64)
    slots = (inv.astype(np.int64)[tokens[:, None] * k + np.arange(k)[None, :]]).reshape(-1)
    xp_rows = gather_rows(x_bits, perm[slots], k)
    g = np.searchsorted(go.astype(np.int64), slots, side="right") - 1
    ge = rep[2] if rep is not None else np.arange(2 * E + 1)
    yrows = expert_ffn_rows(xp_rows, ge[g], w1, w3, w2, act).reshape(len(tokens), k, -1)
    out = np.einsum("tr,trh->th", w[tokens], yrows)
    return dict(idx=idx, w=w, hist=h, rep=rep, group_offsets=go, perm=perm, inv_perm=inv,
                slots=slots, out=out)

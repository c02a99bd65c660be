"""Plant plausible slips in the oracle (CPU only) and check that the pins in
test_oracle_pins.py catch every one of them."""
import math

import numpy as np
import pytest

from oracle import moe_oracle as O
import tests.test_oracle_pins as P
import tests.test_oracle_prediction as PP
import tests.test_oracle_backward as PB


def _topk_ties_reversed(logits, k, renorm=True):
    l = np.asarray(logits).astype(np.float64)
    T, E = l.shape
    eidx = np.broadcast_to(np.arange(E)[::-1], (T, E))  # higher index first on ties
    order = np.lexsort((eidx, -l), axis=-1)
    idx = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(l, idx.astype(np.int64), 1)
    z = np.exp(sel - sel[:, :1])
    return idx, z / z.sum(1, keepdims=True)


def _topk_weight_sign(logits, k, renorm=True):
    idx, w = ORIG["topk_gate"](logits, k, renorm)
    l = np.take_along_axis(np.asarray(logits, np.float64), idx.astype(np.int64), 1)
    z = np.exp(l[:, :1] - l)  # sign slip
    return idx, z / z.sum(1, keepdims=True)


def _cosel_transposed(a, b, E):
    return ORIG["coselection"](a, b, E).T


def _predict_transposed(self, layer):
    p, c, n = ORIG["predict"](self, layer)
    if c is None:
        return p, c, n
    return p, c, c @ p


def _predict_no_row_norm(self, layer):
    p, c, n = ORIG["predict"](self, layer)
    if c is None:
        return p, c, n
    Cb = self.window_cosel(layer).astype(np.float64)
    c2 = Cb / max(Cb.sum(), 1)
    return p, c2, p @ c2


def _replicate_ge(load, total, thresh_num=6, thresh_den=5, max_copies=-1):
    E = len(load)
    copies = []
    for ld in load:
        c = math.ceil(ld * E / total) - 1 if ld * E * thresh_den >= thresh_num * total else 0
        copies.append(min(c, max_copies) if max_copies >= 0 else c)
    return _tables(copies)


def _replicate_floor(load, total, thresh_num=6, thresh_den=5, max_copies=-1):
    E = len(load)
    copies = []
    for ld in load:
        c = (ld * E) // total - 1 if ld * E * thresh_den > thresh_num * total else 0
        copies.append(min(c, max_copies) if max_copies >= 0 else c)
    return _tables(copies)


def _tables(copies):
    E = len(copies)
    rb = np.concatenate([[0], np.cumsum(np.array(copies) + 1)]).astype(np.int32)
    ge = [e for e, c in enumerate(copies) for _ in range(c + 1)]
    ge += [-1] * (2 * E - len(ge))
    return np.array(copies, np.int32), rb, np.array(ge, np.int32)


def _dispatch_block_split(idx, E, rep_base=None):
    idx = np.asarray(idx)
    A = idx.size
    if rep_base is None:
        rep_base = np.arange(E + 1)
    flat = idx.reshape(-1)
    groups = []
    for e in range(E):
        fs = [f for f in range(A) if flat[f] == e]
        n_e = int(rep_base[e + 1] - rep_base[e])
        sz = [len(fs) // n_e + (1 if q < len(fs) % n_e else 0) for q in range(n_e)]
        p = 0
        for q in range(n_e):
            groups.append(fs[p:p + sz[q]])
            p += sz[q]
    off = [0]
    for g in groups:
        off.append(off[-1] + len(g))
    off += [A] * (2 * E + 1 - len(off))
    perm = np.array([f for g in groups for f in g], np.int32)
    inv = np.empty(A, np.int32)
    inv[perm] = np.arange(A)
    return np.array(off, np.int32), perm, inv


def _gelu_tanh(z):
    return 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))


def _ffn_drop_up(x_rows, experts, w1, w3, w2, act):
    return ORIG["expert_ffn_rows"](x_rows, experts, w1, w1 if w3 is not None else None, w2, act)


def _combine_rank_swap(y, inv_perm, w):
    return ORIG["combine"](y, inv_perm, np.asarray(w)[:, ::-1])


def _decay_age_off_by_one(self, layer, it, lam):
    return ORIG["predict_decay"](self, layer, it + 1, lam)


def _decay_cosel_same_age(self, layer, it, lam):
    # co-selection ages counted from `it` instead of it - 1
    E, s = self.E, self.s
    p, _, _ = ORIG["predict_decay"](self, layer, it, lam)
    if layer >= self.L - 1:
        return p, None, None
    Cb = sum((lam ** a if a else 1.0) * self.C[layer, (it - a) % s].astype(np.float64) for a in range(s))
    rows = Cb.sum(axis=1, keepdims=True)
    c = np.where(rows > 0, Cb / np.where(rows > 0, rows, 1), 1.0 / E)
    return p, c, p @ c


def _apportion_ties_high_first(p32, total):
    p32 = np.asarray(p32, np.float32)
    q = [max(float(v), 0.0) * total for v in p32]
    f = [math.floor(v) for v in q]
    left = total - sum(f)
    order = sorted(range(len(q)), key=lambda e: (-(q[e] - f[e]), -e))
    for e in order[:max(left, 0)]:
        f[e] += 1
    return np.array(f, np.int64)


def _apportion_plain_round(p32, total):
    return np.array([int(round(float(v) * total)) for v in np.asarray(p32, np.float32)], np.int64)


def _cap_coldest_first(copies, load, budget):
    copies = [int(c) for c in copies]
    if budget < 0:
        return np.array(copies, np.int32)
    left, out = int(budget), [0] * len(copies)
    for e in sorted(range(len(copies)), key=lambda e: (int(load[e]), e)):
        out[e] = min(copies[e], left)
        left -= out[e]
    return np.array(out, np.int32)


def _overlap_bottom(p_pred, load_actual, m=5):
    p_pred = np.asarray(p_pred, np.float64)
    load_actual = np.asarray(load_actual)
    pred = sorted(range(p_pred.size), key=lambda e: (p_pred[e], e))[:m]
    act = sorted(range(load_actual.size), key=lambda e: (-load_actual[e], e))[:m]
    return len(set(pred) & set(act)) / m


def _gelu_grad_cdf_only(z):
    return 0.5 * (1.0 + O._erf(z / math.sqrt(2.0)))


def _silu_grad_sign(z):
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * s)


def _combine_bwd_unweighted(dout, y, inv_perm, w):
    _, dw = ORIG["combine_backward"](dout, y, inv_perm, w)
    dY, _ = ORIG["combine_backward"](dout, y, inv_perm, np.ones_like(np.asarray(w, np.float64)))
    return dY, dw


def _scatter_sum_perm(dxp, inv_perm, T, k):
    perm = np.argsort(np.asarray(inv_perm))
    return ORIG["scatter_sum"](dxp, perm, T, k)


def _router_bwd_no_centering(logits, idx, dw, renorm=True):
    l = np.asarray(logits, np.float64)
    idx = np.asarray(idx).astype(np.int64)
    out = np.zeros_like(l)
    for t in range(l.shape[0]):
        z = np.exp(l[t, idx[t]] - l[t, idx[t]].max())
        w = z / z.sum()
        out[t, idx[t]] = w * np.asarray(dw, np.float64)[t]
    return out


def _topk_full_softmax_always(logits, k, renorm=True):
    return ORIG["topk_gate"](logits, k, False)


def _topk_renorm_always(logits, k, renorm=True):
    return ORIG["topk_gate"](logits, k, True)


def _hist_first_choice_only(idx, E):
    return np.bincount(np.asarray(idx)[:, 0].astype(np.int64), minlength=E).astype(np.int64)


def _cosel_same_rank_only(a, b, E):
    a = np.asarray(a).astype(np.int64)
    b = np.asarray(b).astype(np.int64)
    C = np.zeros((E, E), np.int64)
    for r in range(min(a.shape[1], b.shape[1])):
        np.add.at(C, (a[:, r], b[:, r]), 1)
    return C


def _update_accumulates(self, it, layer, idx_layer, idx_prev=None):
    # the ring slot is added to instead of replaced
    slot = it % self.s
    h = O.histogram(idx_layer, self.E)
    self.h[layer, slot] += h
    if layer > 0:
        self.C[layer - 1, slot] += O.coselection(idx_prev, idx_layer, self.E)
    return h


def _update_window_one_short(self, it, layer, idx_layer, idx_prev=None):
    # a ring of s - 1 slots
    slot = it % max(self.s - 1, 1)
    h = O.histogram(idx_layer, self.E)
    self.h[layer, slot] = h
    if layer > 0:
        self.C[layer - 1, slot] = O.coselection(idx_prev, idx_layer, self.E)
    return h


def _predict_unseen_rows_zero(self, layer):
    p, c, n = ORIG["predict"](self, layer)
    if c is None:
        return p, c, n
    rows = self.window_cosel(layer).sum(axis=1)
    c = c.copy()
    c[rows == 0] = 0.0
    return p, c, p @ c


def _replicate_no_cap(load, total, thresh_num=6, thresh_den=5, max_copies=-1):
    return ORIG["replicate"](load, total, thresh_num, thresh_den, -1)


def _replicate_no_minus_one(load, total, thresh_num=6, thresh_den=5, max_copies=-1):
    E = len(load)
    copies = []
    for ld in load:
        c = math.ceil(ld * E / total) if ld * E * thresh_den > thresh_num * total else 0
        copies.append(min(c, max_copies) if max_copies >= 0 else c)
    return _tables(copies)


def _dispatch_groups_reversed(idx, E, rep_base=None):
    go, perm, _ = ORIG["dispatch"](idx, E, rep_base)
    perm = perm.copy()
    for g in range(len(go) - 1):
        perm[go[g]:go[g + 1]] = perm[go[g]:go[g + 1]][::-1]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=perm.dtype)
    return go, perm, inv


def _gather_mod_k(x, perm, k):
    return np.asarray(x)[np.asarray(perm).astype(np.int64) % k]


def _bf16_shift15(bits):
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 15).view(np.float32).astype(np.float64)


def _silu_negated_gate(z):
    return z / (1.0 + np.exp(z))


def _combine_unweighted(y, inv_perm, w):
    return ORIG["combine"](y, inv_perm, np.ones_like(np.asarray(w, np.float64)))


def _replicate_predicted_no_budget(p32, total, thresh_num=6, thresh_den=5, max_copies=-1, budget=-1):
    return ORIG["replicate_predicted"](p32, total, thresh_num, thresh_den, max_copies, -1)


def _load_error_unnormalised(p_pred, load_actual):
    return float(np.mean(np.abs(np.asarray(p_pred, np.float64) - np.asarray(load_actual, np.float64))))


def _router_bwd_full_no_centering(logits, idx, dw, renorm=True):
    if renorm:
        return ORIG["router_backward"](logits, idx, dw, renorm)
    l = np.asarray(logits, np.float64)
    idx = np.asarray(idx).astype(np.int64)
    out = np.zeros_like(l)
    for t in range(l.shape[0]):
        z = np.exp(l[t] - l[t].max())
        p = z / z.sum()
        g = np.zeros(l.shape[1])
        g[idx[t]] = np.asarray(dw, np.float64)[t]
        out[t] = p * g
    return out


def _ffn_bwd_up_from_gate_preact(x, experts, w1, w3, w2, act, dy):
    # SwiGLU: du taken as dA * g (the gate's pre-activation) instead of dA * silu(g)
    if act != "swiglu":
        return ORIG["expert_ffn_backward_f64"](x, experts, w1, w3, w2, act, dy)
    x, dy = np.asarray(x, np.float64), np.asarray(dy, np.float64)
    w1, w3, w2 = (np.asarray(w, np.float64) for w in (w1, w3, w2))
    experts = np.asarray(experts).astype(np.int64)
    dx, dw1, dw3, dw2 = np.zeros_like(x), np.zeros_like(w1), np.zeros_like(w3), np.zeros_like(w2)
    for e in np.unique(experts):
        rows = np.nonzero(experts == e)[0]
        xe, dye = x[rows], dy[rows]
        g, u = xe @ w1[e], xe @ w3[e]
        a = O._silu(g) * u
        dA = dye @ w2[e].T
        dg = dA * u * O._silu_grad(g)
        du = dA * g
        dw1[e] += xe.T @ dg
        dw3[e] += xe.T @ du
        dw2[e] += a.T @ dye
        dx[rows] = dg @ w1[e].T + du @ w3[e].T
    return dx, dw1, dw3, dw2


ORIG = {
    "topk_gate": O.topk_gate,
    "coselection": O.coselection,
    "predict": O.WindowStats.predict,
    "expert_ffn_rows": O.expert_ffn_rows,
    "combine": O.combine,
    "predict_decay": O.WindowStats.predict_decay,
    "combine_backward": O.combine_backward,
    "scatter_sum": O.scatter_sum,
    "replicate": O.replicate,
    "dispatch": O.dispatch,
    "replicate_predicted": O.replicate_predicted,
    "router_backward": O.router_backward,
    "expert_ffn_backward_f64": O.expert_ffn_backward_f64,
}

MUTANTS = [
    ("topk_gate", _topk_ties_reversed, [P.test_topk_brute_force_with_many_ties]),
    ("topk_gate", _topk_weight_sign, [P.test_topk_hand_cases]),
    ("coselection", _cosel_transposed, [P.test_coselection_hand_case]),
    ("WindowStats.predict", _predict_transposed, [P.test_window_hand_case_ring_overwrite]),
    ("WindowStats.predict", _predict_no_row_norm, [P.test_window_stationary_stream_closed_form]),
    ("replicate", _replicate_ge, [P.test_replicate_hand_tables]),
    ("replicate", _replicate_floor, [P.test_replicate_hand_tables]),
    ("dispatch", _dispatch_block_split, [P.test_dispatch_hand_case]),
    ("_gelu", _gelu_tanh, [P.test_ffn_closed_form_values]),
    ("expert_ffn_rows", _ffn_drop_up, [lambda: P.test_ffn_matches_naive_triple_loop("swiglu")]),
    ("combine", _combine_rank_swap, [P.test_combine_hand_case]),
    ("WindowStats.predict_decay", _decay_age_off_by_one, [PP.test_decay_hand_cases]),
    ("WindowStats.predict_decay", _decay_cosel_same_age, [PP.test_decay_hand_cases]),
    ("apportion", _apportion_ties_high_first, [PP.test_apportion_hand_cases]),
    ("apportion", _apportion_plain_round, [PP.test_apportion_hand_cases]),
    ("cap_copies", _cap_coldest_first, [PP.test_budget_hand_cases]),
    ("top_overlap", _overlap_bottom, [PP.test_quality_hand_cases]),
    ("_gelu_grad", _gelu_grad_cdf_only, [lambda: PB.test_ffn_backward_matches_finite_differences("gelu")]),
    ("_silu_grad", _silu_grad_sign, [lambda: PB.test_ffn_backward_matches_finite_differences("swiglu")]),
    ("combine_backward", _combine_bwd_unweighted, [PB.test_combine_backward_matches_finite_differences]),
    ("scatter_sum", _scatter_sum_perm, [PB.test_scatter_sum_is_the_adjoint_of_the_row_copy]),
    ("router_backward", _router_bwd_no_centering, [lambda: PB.test_router_backward_matches_finite_differences(True)]),
    ("topk_gate", _topk_full_softmax_always, [P.test_gate_weights_closed_forms]),
    ("topk_gate", _topk_renorm_always, [P.test_gate_weights_closed_forms]),
    ("histogram", _hist_first_choice_only, [P.test_histogram_brute_force_and_sum]),
    ("coselection", _cosel_same_rank_only, [P.test_coselection_sums_and_brute_force]),
    ("WindowStats.update", _update_accumulates, [P.test_window_keeps_last_s_iterations]),
    ("WindowStats.update", _update_window_one_short, [P.test_window_keeps_last_s_iterations]),
    ("WindowStats.predict", _predict_unseen_rows_zero, [P.test_window_empty_and_unseen_rows]),
    ("replicate", _replicate_no_cap, [P.test_replicate_hand_tables]),
    ("replicate", _replicate_no_minus_one, [P.test_replicate_hand_tables, P.test_replicate_bound_and_float_rule]),
    ("dispatch", _dispatch_groups_reversed, [P.test_dispatch_hand_case, lambda: P.test_dispatch_properties(True)]),
    ("gather_rows", _gather_mod_k, [P.test_layer_replication_invariance]),
    ("bf16_to_f64", _bf16_shift15, [P.test_ffn_closed_form_values]),
    ("_silu", _silu_negated_gate, [P.test_ffn_closed_form_values]),
    ("combine", _combine_unweighted, [P.test_combine_hand_case]),
    ("replicate_predicted", _replicate_predicted_no_budget,
     [PP.test_replicate_predicted_reduces_to_replicate_on_exact_shares]),
    ("load_proportion_error", _load_error_unnormalised, [PP.test_quality_hand_cases]),
    ("router_backward", _router_bwd_full_no_centering,
     [lambda: PB.test_router_backward_matches_finite_differences(False)]),
    ("expert_ffn_backward_f64", _ffn_bwd_up_from_gate_preact,
     [lambda: PB.test_ffn_backward_matches_finite_differences("swiglu")]),
]


@pytest.mark.parametrize("name,mutant,pins", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_pins_catch_planted_slip(monkeypatch, name, mutant, pins):
    if name.startswith("WindowStats."):
        monkeypatch.setattr(O.WindowStats, name.split(".")[1], mutant)
    else:
        monkeypatch.setattr(O, name, mutant)
    for pin in pins:
        with pytest.raises(AssertionError):
            pin()

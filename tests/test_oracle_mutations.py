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


ORIG = {
    "topk_gate": O.topk_gate,
    "coselection": O.coselection,
    "predict": O.WindowStats.predict,
    "expert_ffn_rows": O.expert_ffn_rows,
    "combine": O.combine,
    "predict_decay": O.WindowStats.predict_decay,
    "combine_backward": O.combine_backward,
    "scatter_sum": O.scatter_sum,
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

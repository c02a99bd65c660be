"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here recomputes an oracle formula by retyping it: each check is brute
force on tiny inputs, a hand-derived table (tests/golden), a closed form, an
invariant, or an independent library routine.  Each one is chosen so that a
plausible slip in the oracle (a dropped term, a swapped index, a transposed
operand, an off-by-one at a threshold) makes it fail; test_oracle_mutations.py
plants such slips and checks that they are caught.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import moe_oracle as O
from moe_expert_routing_02_b300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def f32_to_bf16_bits(a):
    """Round fp32 values to bf16 bit patterns (round to nearest even)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------
# top-k gate
# ----------------------------------------------------------------------------
def brute_topk(row, k):
    """Brute force over every k-subset: the subset with the largest exact sum,
    lexicographically smallest (by sorted index list) among equal sums."""
    E = len(row)
    vals = [Fraction(float(v)) for v in row]
    best, best_sum = None, None
    for sub in itertools.combinations(range(E), k):
        s = sum(vals[i] for i in sub)
        if best is None or s > best_sum:
            best, best_sum = sub, s
    # rank order inside the set: value descending, index ascending
    return sorted(best, key=lambda i: (-vals[i], i))


@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_topk_matches_brute_force(k):
    cfg = W.config_by_name("tiny")
    lg = W.make_layer_logits(cfg, 0, T=48)[1]  # layer 2 carries the correlation boost
    idx, w = O.topk_gate(lg, k)
    for t in range(lg.shape[0]):
        assert list(idx[t]) == brute_topk(lg[t], k), t


def test_topk_brute_force_with_many_ties():
    rng = np.random.default_rng(7)
    lg = rng.integers(-2, 3, size=(64, 7)).astype(np.float32)  # heavy ties
    lg[rng.random(lg.shape) < 0.2] = -0.0
    for k in (1, 2, 4, 7):
        idx, _ = O.topk_gate(lg, k)
        for t in range(lg.shape[0]):
            assert list(idx[t]) == brute_topk(lg[t], k)


def test_topk_hand_cases():
    for c in gold("gate_hand.json")["cases"]:
        lg = np.array([c["logits"]], dtype=np.float32)
        idx, w = O.topk_gate(lg, c["k"])
        assert list(idx[0]) == c["idx"]
        if "w_renorm" in c:
            assert np.allclose(w[0], c["w_renorm"], atol=1e-7, rtol=0)


def test_gate_weights_closed_forms():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((200, 16)).astype(np.float32)
    for k in (1, 2, 6):
        idx, w = O.topk_gate(lg, k, renorm=True)
        assert np.allclose(w.sum(1), 1.0, atol=1e-12)
        assert np.all(np.diff(w, axis=1) <= 1e-15)  # rank order = weight order
        if k == 1:
            assert np.all(w == 1.0)
        # ratio of two chosen weights is exp of the logit difference
        if k >= 2:
            l0 = np.take_along_axis(lg.astype(np.float64), idx[:, :2].astype(np.int64), 1)
            assert np.allclose(w[:, 1] / w[:, 0], np.exp(l0[:, 1] - l0[:, 0]), rtol=1e-12)
    # full softmax agrees with scipy's softmax on the chosen entries
    from scipy.special import softmax
    idx, w = O.topk_gate(lg, 3, renorm=False)
    sm = softmax(lg.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(sm, idx.astype(np.int64), 1), rtol=1e-12, atol=0)
    # equal logits: uniform weights
    idx, w = O.topk_gate(np.zeros((3, 8), np.float32), 4, renorm=False)
    assert np.allclose(w, 1 / 8) and np.all(idx == np.arange(4))


# ----------------------------------------------------------------------------
# histogram and co-selection
# ----------------------------------------------------------------------------
def test_histogram_brute_force_and_sum():
    cfg = W.config_by_name("tiny")
    lg = W.make_layer_logits(cfg, 3)
    for j in range(2):
        idx, _ = O.topk_gate(lg[j], cfg.k)
        h = O.histogram(idx, cfg.E)
        assert h.sum() == cfg.T * cfg.k
        bf = [sum(1 for t in range(cfg.T) for r in range(cfg.k) if idx[t, r] == e) for e in range(cfg.E)]
        assert list(h) == bf


def test_coselection_hand_case():
    g = gold("coselect_hand.json")
    C = O.coselection(np.array(g["idx_prev"]), np.array(g["idx_cur"]), g["E"])
    assert C.tolist() == g["C"]


def test_coselection_sums_and_brute_force():
    cfg = W.config_by_name("tiny")
    lg = W.make_layer_logits(cfg, 5)
    a, _ = O.topk_gate(lg[0], cfg.k)
    b, _ = O.topk_gate(lg[1], cfg.k)
    C = O.coselection(a, b, cfg.E)
    k = cfg.k
    assert np.array_equal(C.sum(1), k * O.histogram(a, cfg.E))   # row sums = k * h_j
    assert np.array_equal(C.sum(0), k * O.histogram(b, cfg.E))   # column sums = k * h_{j+1}
    assert C.sum() == cfg.T * k * k
    bf = np.zeros_like(C)
    for t in range(cfg.T):
        for e in a[t]:
            for e2 in b[t]:
                bf[e, e2] += 1
    assert np.array_equal(C, bf)
    # k = 1: literally "row sums equal the layer-j histogram"
    C1 = O.coselection(a[:, :1], b[:, :1], cfg.E)
    assert np.array_equal(C1.sum(1), O.histogram(a[:, :1], cfg.E))


# ----------------------------------------------------------------------------
# sliding window and prediction
# ----------------------------------------------------------------------------
def test_window_hand_case_ring_overwrite():
    g = gold("window_hand.json")
    st = O.WindowStats(g["L"], g["E"], g["s"])
    for step in g["stream"]:
        it = step["it"]
        st.update(it, 0, np.array(step["layer0"]))
        if it == 2:
            p, c, n = st.predict(0)
            m = g["mid_it2"]
            assert np.allclose(p, m["p_seq"], atol=1e-15)
            assert np.allclose(c, m["cond"], atol=1e-15)
            assert np.allclose(n, m["p_next"], atol=1e-15)
        st.update(it, 1, np.array(step["layer1"]), np.array(step["layer0"]))
    p, c, n = st.predict(0)
    e = g["end_it2"]
    assert np.allclose(p, e["p_seq"], atol=1e-15)
    assert np.allclose(c, e["cond"], atol=1e-15)
    assert np.allclose(n, e["p_next"], atol=1e-15)
    p1, c1, n1 = st.predict(1)
    assert np.allclose(p1, e["p_seq_layer1"]) and c1 is None and n1 is None


def test_window_stationary_stream_closed_form():
    """If the same routing repeats every iteration, the predicted next-layer
    popularity equals the next layer's own popularity exactly:
    sum_e Cbar[e,e'] / (k * sum H_j) = H_{j+1}[e'] / sum H_{j+1}."""
    cfg = W.config_by_name("tiny")
    lg = W.make_layer_logits(cfg, 0)
    idx = [O.topk_gate(l, cfg.k)[0] for l in lg]
    st = O.WindowStats(cfg.L, cfg.E, 10)
    for it in range(13):
        st.update(it, 0, idx[0])
        st.update(it, 1, idx[1], idx[0])
    p0, cond, p_next = st.predict(0)
    p1, _, _ = st.predict(1)
    h1 = O.histogram(idx[1], cfg.E)
    assert np.allclose(p_next, p1, atol=1e-14)
    assert np.allclose(p1, h1 / h1.sum(), atol=1e-15)
    assert np.allclose(cond.sum(1), 1.0, atol=1e-14)
    assert abs(p_next.sum() - 1.0) < 1e-14


def test_window_empty_and_unseen_rows():
    st = O.WindowStats(2, 4, 10)
    p, c, n = st.predict(0)
    assert np.allclose(p, 0.25) and np.allclose(c, 0.25) and np.allclose(n, 0.25)
    st.update(0, 0, np.array([[0], [0]]))
    p, c, n = st.predict(0)
    assert np.allclose(p, [1, 0, 0, 0])
    assert np.allclose(n, 0.25)  # no co-selection yet: uniform rows


def test_window_keeps_last_s_iterations():
    """Brute force: window sums equal the sum over the last s iterations."""
    cfg = W.config_by_name("tiny")
    st = O.WindowStats(cfg.L, cfg.E, 4)
    hist_log, cos_log = [], []
    for it in range(9):
        lg = W.make_layer_logits(cfg, it, T=64)
        a = O.topk_gate(lg[0], cfg.k)[0]
        b = O.topk_gate(lg[1], cfg.k)[0]
        st.update(it, 0, a)
        st.update(it, 1, b, a)
        hist_log.append(O.histogram(a, cfg.E))
        cos_log.append(O.coselection(a, b, cfg.E))
        lo = max(0, it - 3)
        assert np.array_equal(st.window_hist(0), sum(hist_log[lo:it + 1]))
        assert np.array_equal(st.window_cosel(0), sum(cos_log[lo:it + 1]))


# ----------------------------------------------------------------------------
# replication
# ----------------------------------------------------------------------------
def test_replicate_hand_tables():
    for c in gold("replicate_table.json")["cases"]:
        copies, rep_base, ge = O.replicate(c["load"], c["total"], 6, 5, c.get("max_copies", -1))
        assert copies.tolist() == c["copies"], c["name"]
        assert rep_base.tolist() == c["rep_base"], c["name"]
        E = len(c["load"])
        assert len(ge) == 2 * E
        for e in range(E):
            assert all(ge[rep_base[e]:rep_base[e + 1]] == e)
        assert all(ge[rep_base[E]:] == -1)


def test_replicate_bound_and_float_rule():
    """E_phys <= 2E - 1 whenever loads sum to the total, and the exact table
    agrees with the rule evaluated in plain floating point away from ties."""
    rng = np.random.default_rng(11)
    for trial in range(300):
        E = int(rng.integers(1, 40))
        A = int(rng.integers(E, 5000))
        p = rng.dirichlet(np.full(E, rng.uniform(0.05, 3)))
        load = rng.multinomial(A, p)
        copies, rep_base, ge = O.replicate(load, A)
        assert rep_base[-1] <= 2 * E - 1
        target = A / E
        for e in range(E):
            x = load[e] / target
            if abs(x - 1.2) > 1e-9 and abs(x - round(x)) > 1e-9:
                want = math.ceil(x) - 1 if load[e] > 1.2 * target else 0
                assert copies[e] == want


# ----------------------------------------------------------------------------
# dispatch
# ----------------------------------------------------------------------------
def test_dispatch_hand_case():
    g = gold("dispatch_hand.json")
    go, perm, inv = O.dispatch(np.array(g["idx"]), g["E"], np.array(g["rep_base"]))
    assert go.tolist() == g["group_offsets"]
    assert perm.tolist() == g["perm"]
    assert inv.tolist() == g["inv_perm"]
    go, perm, inv = O.dispatch(np.array(g["idx"]), g["E"], None)
    assert go.tolist() == g["no_replica"]["group_offsets"]
    assert perm.tolist() == g["no_replica"]["perm"]


@pytest.mark.parametrize("replicated", [False, True])
def test_dispatch_properties(replicated):
    cfg = W.config_by_name("dbrx_replicated_layer")
    lg = W.make_layer_logits(cfg, 0, T=512)[0]
    idx, _ = O.topk_gate(lg, cfg.k)
    A = idx.size
    h = O.histogram(idx, cfg.E)
    rep = O.replicate(h, A) if replicated else None
    rb = rep[1] if rep is not None else np.arange(cfg.E + 1)
    go, perm, inv = O.dispatch(idx, cfg.E, None if rep is None else rep[1])
    assert sorted(perm.tolist()) == list(range(A))          # a permutation
    assert np.array_equal(inv[perm], np.arange(A))          # inv o perm = id
    flat = idx.reshape(-1)
    for e in range(cfg.E):
        n_e = rb[e + 1] - rb[e]
        for q in range(n_e):
            g = rb[e] + q
            seg = perm[go[g]:go[g + 1]]
            assert np.all(flat[seg] == e)
            assert np.all(np.diff(seg) > 0)                 # stable inside a group
            assert len(seg) == h[e] // n_e + (1 if q < h[e] % n_e else 0)
    if replicated:
        assert rb[-1] > cfg.E  # the skewed config does replicate
    else:
        # no replication: a stable counting sort by expert
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))


# ----------------------------------------------------------------------------
# expert FFN
# ----------------------------------------------------------------------------
def test_ffn_closed_form_values():
    one = f32_to_bf16_bits(np.float32(1.0))
    zero = f32_to_bf16_bits(np.float32(0.0))
    eye = np.array([[[one, zero], [zero, one]]], dtype=np.uint16)
    x = np.array([[one, zero]], dtype=np.uint16)
    y = O.expert_ffn_rows(x, np.array([0]), eye, None, eye, "gelu")
    assert abs(y[0, 0] - 0.8413447460685429) < 1e-15   # gelu(1) = Phi(1)
    assert y[0, 1] == 0.0
    y = O.expert_ffn_rows(x, np.array([0]), eye, eye, eye, "swiglu")
    assert abs(y[0, 0] - 0.7310585786300049) < 1e-15   # silu(1) * 1 = sigmoid(1)
    # GeLU is x * Phi(x): compare with scipy's normal cdf
    from scipy.stats import norm
    z = np.linspace(-6, 6, 101)
    assert np.allclose(O._gelu(z), z * norm.cdf(z), rtol=1e-13, atol=1e-15)


def naive_ffn(x, w1, w3, w2, act):
    """Triple loop in plain Python floats (no NumPy arithmetic)."""
    H = len(x)
    F = len(w1[0])
    a = []
    for f in range(F):
        z = sum(x[h] * w1[h][f] for h in range(H))
        if act == "gelu":
            a.append(0.5 * z * (1.0 + math.erf(z / math.sqrt(2.0))))
        else:
            u = sum(x[h] * w3[h][f] for h in range(H))
            a.append(z / (1.0 + math.exp(-z)) * u)
    return [sum(a[f] * w2[f][o] for f in range(F)) for o in range(len(w2[0]))]


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_ffn_matches_naive_triple_loop(act):
    rng = np.random.default_rng(5)
    E, H, F, n = 3, 8, 12, 10
    def rnd(*s, sc=1.0):
        return f32_to_bf16_bits((rng.standard_normal(s) * sc).astype(np.float32))
    w1, w3, w2 = rnd(E, H, F, sc=0.5), rnd(E, H, F, sc=0.5), rnd(E, F, H, sc=0.5)
    x = rnd(n, H)
    ex = rng.integers(0, E, n)
    y = O.expert_ffn_rows(x, ex, w1, w3 if act == "swiglu" else None, w2, act)
    X = O.bf16_to_f64(x)
    for i in range(n):
        e = ex[i]
        ref = naive_ffn(list(X[i]), O.bf16_to_f64(w1[e]).tolist(), O.bf16_to_f64(w3[e]).tolist(),
                        O.bf16_to_f64(w2[e]).tolist(), act)
        assert np.allclose(y[i], ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# combine and the whole layer
# ----------------------------------------------------------------------------
def test_combine_hand_case():
    # T=2, k=2, H=1; Y slots [10, 20, 30, 40]; token 0 -> slots 3,0; token 1 -> slots 1,2
    y = np.array([[10.0], [20.0], [30.0], [40.0]])
    inv = np.array([3, 0, 1, 2])
    w = np.array([[0.75, 0.25], [0.5, 0.5]])
    out = O.combine(y, inv, w)
    assert out[:, 0].tolist() == [0.75 * 40 + 0.25 * 10, 0.5 * 20 + 0.5 * 30]


def test_layer_replication_invariance():
    """Replicas compute the same expert, so per-token outputs are identical
    with and without replication (PopFetcher review: loss curves coincide
    with and without expert copies; MoE-MPMC summary: replication does not
    change the MoE computation)."""
    cfg = W.config_by_name("dbrx_replicated_layer")
    T, E, H, F = 96, cfg.E, 64, 128
    lg = W.make_layer_logits(cfg, 0, T=T)[0]
    x = W.bf16_bits(W.make_x(cfg, 0, 0, T=T).reshape(T, -1)[:, :H])
    w1, w3, w2 = (W.bf16_bits(t) for t in W.make_weights(cfg, 0, E=E, H=H, F=F))
    a = O.moe_layer(lg, x, cfg.k, w1, w3, w2, "swiglu", replicate_on=False)
    b = O.moe_layer(lg, x, cfg.k, w1, w3, w2, "swiglu", replicate_on=True)
    assert b["rep"][1][-1] > E
    assert np.array_equal(a["out"], b["out"])
    # and the whole layer equals a direct per-token evaluation
    idx, w = a["idx"], a["w"]
    for t in range(0, T, 17):
        ref = sum(w[t, r] * O.expert_ffn_rows(x[t:t + 1], [idx[t, r]], w1, w3, w2, "swiglu")[0]
                  for r in range(cfg.k))
        assert np.allclose(a["out"][t], ref, rtol=1e-12, atol=1e-14)

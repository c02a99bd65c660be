"""Property-based pins of the CPU oracle (hypothesis): random tiny inputs,
each checked against brute force or a property that the definition fixes
(ceil bounds of the replica rule, round-robin group sizes, the window as
the last s distinct iterations, linearity and adjoint identities, rows of
a softmax gradient summing to zero).  None of them restates an oracle
formula in the oracle's own form."""
import math
from fractions import Fraction

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import moe_oracle as O  # noqa: E402
from tests.test_oracle_pins import brute_topk  # noqa: E402

SETTINGS = settings(max_examples=60, deadline=None, derandomize=True)


@st.composite
def routing(draw, max_T=12, max_E=7, max_k=None):
    """idx [T, k]: k distinct experts per token, out of E."""
    E = draw(st.integers(1, max_E))
    k = draw(st.integers(1, min(E, max_k or E)))
    T = draw(st.integers(1, max_T))
    rows = [draw(st.permutations(range(E)))[:k] for _ in range(T)]
    return np.array(rows, dtype=np.int32).reshape(T, k), E


# ----------------------------------------------------------------------------
# gate
# ----------------------------------------------------------------------------
@SETTINGS
@given(st.data())
def test_topk_brute_force_with_ties(data):
    E = data.draw(st.integers(1, 8))
    k = data.draw(st.integers(1, E))
    T = data.draw(st.integers(1, 6))
    vals = st.sampled_from([-2.0, -1.0, -0.0, 0.0, 0.5, 1.0, 3.0])
    lg = np.array([[data.draw(vals) for _ in range(E)] for _ in range(T)], dtype=np.float32)
    idx, w = O.topk_gate(lg, k, renorm=True)
    _, wf = O.topk_gate(lg, k, renorm=False)
    for t in range(T):
        assert list(idx[t]) == brute_topk(lg[t], k)
    # renormalised weights sum to 1; the full-softmax ones are the same
    # numerators over a larger denominator, so never larger
    assert np.allclose(w.sum(1), 1.0, atol=1e-12)
    assert np.all(wf <= w + 1e-15)
    if k == E:
        assert np.allclose(wf, w, rtol=1e-12)


# ----------------------------------------------------------------------------
# histogram and co-selection
# ----------------------------------------------------------------------------
@SETTINGS
@given(routing(), st.data())
def test_coselection_brute_force_and_margins(r, data):
    a, E = r
    T = a.shape[0]
    kb = data.draw(st.integers(1, E))
    b = np.array([data.draw(st.permutations(range(E)))[:kb] for _ in range(T)], dtype=np.int32).reshape(T, kb)
    C = O.coselection(a, b, E)
    bf = np.zeros((E, E), dtype=np.int64)
    for t in range(T):
        for e in a[t]:
            for e2 in b[t]:
                bf[e, e2] += 1
    assert np.array_equal(C, bf)
    assert np.array_equal(C.sum(1), kb * O.histogram(a, E))
    assert np.array_equal(C.sum(0), a.shape[1] * O.histogram(b, E))


# ----------------------------------------------------------------------------
# sliding window
# ----------------------------------------------------------------------------
@SETTINGS
@given(st.data())
def test_window_is_the_last_s_distinct_iterations(data):
    """Iterations advance by 0 (an update that replaces the last one) or 1.
    The window sums must equal the sum, over the last s distinct iterations,
    of each iteration's latest update (an event log, not a ring)."""
    E = data.draw(st.integers(1, 5))
    s = data.draw(st.integers(1, 4))
    k = data.draw(st.integers(1, E))
    ws = O.WindowStats(2, E, s)
    log0, log1 = {}, {}
    it = 0
    for _ in range(data.draw(st.integers(1, 12))):
        it += data.draw(st.integers(0, 1))
        T = data.draw(st.integers(1, 5))
        a = np.array([data.draw(st.permutations(range(E)))[:k] for _ in range(T)], dtype=np.int32).reshape(T, k)
        b = np.array([data.draw(st.permutations(range(E)))[:k] for _ in range(T)], dtype=np.int32).reshape(T, k)
        ws.update(it, 0, a)
        ws.update(it, 1, b, a)
        log0[it] = a
        log1[it] = (a, b)
        recent = [j for j in log0 if j > it - s]
        H0 = sum(np.bincount(log0[j].reshape(-1), minlength=E) for j in recent)
        Cb = np.zeros((E, E), dtype=np.int64)
        for j in recent:
            pa, pb = log1[j]
            for t in range(pa.shape[0]):
                for e in pa[t]:
                    for e2 in pb[t]:
                        Cb[e, e2] += 1
        assert np.array_equal(ws.window_hist(0), H0)
        assert np.array_equal(ws.window_cosel(0), Cb)
        p, cond, pn = ws.predict(0)
        assert abs(p.sum() - 1) < 1e-12 and np.all(p >= 0)
        assert np.allclose(cond.sum(1), 1.0, atol=1e-12) and np.all(cond >= 0)
        assert abs(pn.sum() - 1) < 1e-12 and np.all(pn >= 0)


# ----------------------------------------------------------------------------
# replica counts
# ----------------------------------------------------------------------------
@SETTINGS
@given(st.data())
def test_replica_rule_ceil_bounds(data):
    """With target = total / E: a hot expert (load > 1.2 target) gets c copies
    with c < load / target <= c + 1 (the ceil of the rule); a cold one none;
    more load never gets fewer copies; at most 2E - 1 groups when the loads
    sum to the total; a cap bounds every count."""
    E = data.draw(st.integers(1, 12))
    loads = data.draw(st.lists(st.integers(0, 50), min_size=E, max_size=E))
    total = sum(loads)
    if total == 0:
        return
    cap = data.draw(st.sampled_from([-1, 0, 1, 2]))
    copies, rep_base, ge = O.replicate(loads, total, 6, 5, cap)
    target = Fraction(total, E)
    for e, ld in enumerate(loads):
        hot = Fraction(ld) > Fraction(6, 5) * target
        if not hot:
            assert copies[e] == 0
        elif cap < 0:
            c = int(copies[e])
            assert c < Fraction(ld) / target <= c + 1
        else:
            assert copies[e] == min(math.ceil(Fraction(ld) / target) - 1, cap)
    order = sorted(range(E), key=lambda e: loads[e])
    assert all(copies[order[i]] <= copies[order[i + 1]] for i in range(E - 1))
    assert rep_base[-1] <= 2 * E - 1
    assert rep_base[0] == 0 and all(rep_base[e + 1] - rep_base[e] == copies[e] + 1 for e in range(E))
    assert list(ge[:rep_base[-1]]) == [e for e in range(E) for _ in range(int(copies[e]) + 1)]


# ----------------------------------------------------------------------------
# dispatch
# ----------------------------------------------------------------------------
@SETTINGS
@given(routing(max_T=16, max_E=6), st.data())
def test_dispatch_round_robin_by_slicing(r, data):
    """Group q of expert e holds the assignments f = t*k + r of e (ascending)
    at positions q, q + n_e, q + 2 n_e, ... (a stride slice)."""
    idx, E = r
    copies = [data.draw(st.integers(0, 2)) for _ in range(E)]
    while sum(copies) > E - 1:      # the replica rule's bound: at most 2E - 1 groups
        copies[copies.index(max(copies))] -= 1
    rep_base = np.concatenate([[0], np.cumsum(np.array(copies) + 1)]).astype(np.int32)
    go, perm, inv = O.dispatch(idx, E, rep_base)
    flat = idx.reshape(-1)
    A = flat.size
    want = []
    for e in range(E):
        fs = [f for f in range(A) if flat[f] == e]
        n_e = copies[e] + 1
        for q in range(n_e):
            want.append(fs[q::n_e])
    assert [list(perm[go[g]:go[g + 1]]) for g in range(len(want))] == want
    assert np.all(go[len(want):] == A)
    assert np.array_equal(inv[perm], np.arange(A))


# ----------------------------------------------------------------------------
# combine, whole layer and backward identities
# ----------------------------------------------------------------------------
@SETTINGS
@given(routing(max_T=8, max_E=5), st.data())
def test_combine_linear_and_adjoint(r, data):
    idx, E = r
    T, k = idx.shape
    _, perm, inv = O.dispatch(idx, E)
    rng = np.random.default_rng(data.draw(st.integers(0, 2 ** 31)))
    y = rng.standard_normal((T * k, 3))
    w1, w2 = rng.standard_normal((T, k)), rng.standard_normal((T, k))
    a, b = 0.75, -1.5
    assert np.allclose(O.combine(y, inv, a * w1 + b * w2), a * O.combine(y, inv, w1) + b * O.combine(y, inv, w2),
                       rtol=1e-12, atol=1e-12)
    dout = rng.standard_normal((T, 3))
    dY, dw = O.combine_backward(dout, y, inv, w1)
    out = O.combine(y, inv, w1)
    # <dout, out> is bilinear in (w, Y): it equals <dY, Y> and <dw, w>
    assert math.isclose(np.sum(dout * out), np.sum(dY * y), rel_tol=1e-10, abs_tol=1e-10)
    assert math.isclose(np.sum(dout * out), np.sum(dw * w1), rel_tol=1e-10, abs_tol=1e-10)
    # every token's row is reached once per choice
    xs = rng.standard_normal((T, 3))
    xp = O.gather_rows(xs, perm, k)
    for slot in range(T * k):
        assert np.array_equal(xp[slot], xs[perm[slot] // k])


@SETTINGS
@given(st.data())
def test_router_gradient_rows_sum_to_zero(data):
    """Softmax weights are invariant to adding a constant to every logit, so
    every row of the gate gradient sums to zero (renormalised or not)."""
    E = data.draw(st.integers(1, 8))
    k = data.draw(st.integers(1, E))
    T = data.draw(st.integers(1, 5))
    rng = np.random.default_rng(data.draw(st.integers(0, 2 ** 31)))
    lg = rng.standard_normal((T, E)).astype(np.float32)
    for renorm in (True, False):
        idx, _ = O.topk_gate(lg, k, renorm)
        dw = rng.standard_normal((T, k))
        g = O.router_backward(lg, idx, dw, renorm)
        assert np.allclose(g.sum(1), 0.0, atol=1e-12)
        if renorm:   # only the chosen logits move the renormalised weights
            mask = np.ones((T, E), bool)
            np.put_along_axis(mask, idx.astype(np.int64), False, 1)
            assert np.all(g[mask] == 0)


def test_layer_token_subset_equals_rows_of_the_full_layer():
    from moe_expert_routing_02_b300 import workloads as W
    cfg = W.config_by_name("tiny")
    T, E, H, F = 40, cfg.E, 64, 128
    lg = W.make_layer_logits(cfg, 0, T=T)[0]
    x = W.bf16_bits(W.make_x(cfg, 0, 0, T=T).reshape(T, -1)[:, :H])
    w1, w3, w2 = (W.bf16_bits(t) if t is not None else None
                  for t in W.make_weights(cfg, 0, E=E, H=H, F=F))
    full = O.moe_layer(lg, x, cfg.k, w1, w3, w2, cfg.act, replicate_on=True)
    sub = np.array([3, 17, 0, 39, 17])
    part = O.moe_layer(lg, x, cfg.k, w1, w3, w2, cfg.act, replicate_on=True, tokens=sub)
    # same rows, other batch shapes for the float64 matmuls: equal to rounding
    assert np.allclose(part["out"], full["out"][sub], rtol=1e-12, atol=1e-15)
    assert np.array_equal(part["perm"], full["perm"])

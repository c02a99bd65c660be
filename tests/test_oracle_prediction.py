"""Pins of the oracle's prediction-driven replication and prediction-quality
functions (CPU only): hand-derived fixtures, reductions to the plain window,
and properties that hold for any input."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _window_stream():
    g = _load("window_hand.json")
    ws = O.WindowStats(g["L"], g["E"], g["s"])
    return g, ws


def test_decay_hand_cases():
    g, ws = _window_stream()
    st = g["stream"]
    for step in st[:2]:
        ws.update(step["it"], 0, np.array(step["layer0"]))
        ws.update(step["it"], 1, np.array(step["layer1"]), np.array(step["layer0"]))
    ws.update(2, 0, np.array(st[2]["layer0"]))
    d = _load("decay_hand.json")
    for case in d["cases"]:
        p, c, n = ws.predict_decay(0, 2, case["lam"])
        assert np.allclose(p, case["p_seq"], atol=1e-15, rtol=0)
        assert np.allclose(c, case["cond"], atol=1e-15, rtol=0)
        assert np.allclose(n, case["p_next"], atol=1e-15, rtol=0)


def _random_stream(seed=0, L=3, E=6, s=4, T=40, k=2, iters=9):
    rng = np.random.default_rng(seed)
    ws = O.WindowStats(L, E, s)
    idx_hist = []
    for it in range(iters):
        prev = None
        per = []
        for j in range(L):
            idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
            ws.update(it, j, idx, prev)
            per.append(idx)
            prev = idx
        idx_hist.append(per)
    return ws, idx_hist


def test_decay_one_is_the_plain_window():
    ws, _ = _random_stream()
    for j in range(3):
        a = ws.predict(j)
        b = ws.predict_decay(j, 8, 1.0)
        for x, y in zip(a, b):
            if x is None:
                assert y is None
            else:
                assert np.array_equal(x, y)


def test_decay_zero_is_the_newest_iteration():
    """lam = 0: p_seq from the histogram of the newest iteration, Pr from the
    co-selection counts of the iteration before (computed here directly from
    the routings, not through the window object)."""
    ws, hist = _random_stream(seed=3)
    it = 8
    for j in range(2):
        p, c, n = ws.predict_decay(j, it, 0.0)
        h = np.bincount(hist[it][j].reshape(-1), minlength=6).astype(np.float64)
        assert np.allclose(p, h / h.sum(), atol=1e-15)
        Cm = np.zeros((6, 6))
        for t in range(hist[it - 1][j].shape[0]):
            for a in hist[it - 1][j][t]:
                for b in hist[it - 1][j + 1][t]:
                    Cm[a, b] += 1
        rows = Cm.sum(1, keepdims=True)
        want = np.where(rows > 0, Cm / np.where(rows > 0, rows, 1), 1.0 / 6)
        assert np.allclose(c, want, atol=1e-15)
        assert np.allclose(n, (h / h.sum()) @ want, atol=1e-15)


@pytest.mark.parametrize("lam", [0.3, 0.9])
def test_decay_invariants(lam):
    ws, _ = _random_stream(seed=5)
    for it in (0, 2, 8):
        p, c, n = ws.predict_decay(0, it, lam)
        assert abs(p.sum() - 1) < 1e-12 and (p >= 0).all()
        assert np.allclose(c.sum(1), 1, atol=1e-12)
        assert abs(n.sum() - 1) < 1e-12
    with pytest.raises(ValueError):
        ws.predict_decay(0, 1, 1.5)


def test_apportion_hand_cases():
    for case in _load("replicate_predicted_hand.json")["apportion"]:
        got = O.apportion(np.array(case["p"], np.float32), case["total"])
        assert got.tolist() == case["load"], case


@pytest.mark.parametrize("seed", range(6))
def test_apportion_properties(seed):
    """Sum equals the total; each load is the floor or the ceiling of its
    exact quota when the float32 shares sum to 1 within rounding; an expert
    that got the extra unit has a remainder at least as large as any that did
    not (lower expert first on equal remainders)."""
    rng = np.random.default_rng(seed)
    E = int(rng.integers(2, 40))
    total = int(rng.integers(1, 100000))
    p = rng.dirichlet(np.ones(E) * 0.3).astype(np.float32)
    load = O.apportion(p, total)
    assert load.sum() == total and (load >= 0).all()
    q = [Fraction(float(v)) * total for v in p]
    import math
    fl = [math.floor(v) for v in q]
    if sum(fl) <= total <= sum(fl) + E:
        up = [e for e in range(E) if load[e] == fl[e] + 1]
        down = [e for e in range(E) if load[e] == fl[e]]
        assert len(up) + len(down) == E
        rem = [q[e] - fl[e] for e in range(E)]
        for a in up:
            for b in down:
                assert rem[a] > rem[b] or (rem[a] == rem[b] and a < b)


def test_budget_hand_cases():
    for case in _load("replicate_predicted_hand.json")["budget"]:
        copies, _, _ = O.replicate(case["load"], case["total"])
        got = O.cap_copies(copies, case["load"], case["budget"])
        assert got.tolist() == case["copies"], case


@pytest.mark.parametrize("seed", range(5))
def test_budget_properties(seed):
    rng = np.random.default_rng(seed)
    E = 12
    load = rng.multinomial(600, rng.dirichlet(np.ones(E) * 0.4))
    copies, _, _ = O.replicate(load, 600)
    budget = int(rng.integers(0, max(int(copies.sum()), 1) + 1))
    capped = O.cap_copies(copies, load, budget)
    assert capped.sum() <= budget and (capped <= copies).all() and (capped >= 0).all()
    order = sorted(range(E), key=lambda e: (-load[e], e))
    cut = [e for e in order if capped[e] < copies[e]]
    if cut:   # every expert served before the first cut one kept all its copies
        first = order.index(cut[0])
        assert all(capped[e] == copies[e] for e in order[:first])
        assert capped.sum() == budget


def test_replicate_predicted_reduces_to_replicate_on_exact_shares():
    """Shares that are exact in float32 and give integer quotas: the loads are
    the quotas and the table equals the histogram-driven one."""
    load = np.array([512, 256, 128, 64, 32, 16, 8, 8], np.int64)
    total = int(load.sum())
    p = (load / total).astype(np.float32)
    lp, copies, rb, ge = O.replicate_predicted(p, total)
    assert lp.tolist() == load.tolist()
    c2, rb2, ge2 = O.replicate(load, total)
    assert copies.tolist() == c2.tolist() and rb.tolist() == rb2.tolist() and ge.tolist() == ge2.tolist()
    _, c3, rb3, _ = O.replicate_predicted(p, total, budget=1)
    assert int(c3.sum()) <= 1 and rb3[-1] == 8 + int(c3.sum())


def test_quality_hand_cases():
    q = _load("replicate_predicted_hand.json")["quality"]
    assert O.top_overlap(q[0]["p"], q[0]["load"], q[0]["m"]) == q[0]["overlap"]
    assert O.load_proportion_error(q[1]["p"], q[1]["load"]) == q[1]["error"]
    assert O.top_overlap([0.1, 0.2, 0.3], [1, 2, 3], 3) == 1.0
    assert O.top_overlap([0.9, 0.05, 0.05, 0.0], [0, 0, 1, 9], 1) == 0.0
    assert O.load_proportion_error([0.25, 0.75], [1, 3]) == 0.0

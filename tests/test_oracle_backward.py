"""Pins of the oracle's backward (CPU only): every gradient against central
finite differences of a scalar loss in float64, and the replica reduction
(an expert's gradient is the sum over all of its rows, whatever groups they
sit in)."""
import numpy as np
import pytest

from oracle import moe_oracle as O

EPS = 1e-6


def _fwd(x, experts, w1, w3, w2, act):
    """Float64 forward of the expert FFN written out here (not the oracle's
    function), so the finite differences do not lean on the code under test."""
    y = np.zeros((x.shape[0], w2.shape[2]))
    for i in range(x.shape[0]):
        e = experts[i]
        z = x[i] @ w1[e]
        if act == "gelu":
            from scipy.stats import norm
            a = z * norm.cdf(z)
        else:
            u = x[i] @ w3[e]
            a = z / (1 + np.exp(-z)) * u
        y[i] = a @ w2[e]
    return y


def _fd(f, arr, rng, n=12):
    """Central differences of scalar f at n random entries of arr."""
    out = []
    for _ in range(n):
        i = tuple(int(rng.integers(0, s)) for s in arr.shape)
        old = arr[i]
        arr[i] = old + EPS
        fp = f()
        arr[i] = old - EPS
        fm = f()
        arr[i] = old
        out.append((i, (fp - fm) / (2 * EPS)))
    return out


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_ffn_backward_matches_finite_differences(act):
    rng = np.random.default_rng(0 if act == "gelu" else 1)
    n, E, H, F = 9, 3, 5, 7
    x = rng.normal(size=(n, H))
    experts = rng.integers(0, E, n)
    w1 = rng.normal(size=(E, H, F)) * 0.5
    w3 = rng.normal(size=(E, H, F)) * 0.5 if act == "swiglu" else None
    w2 = rng.normal(size=(E, F, H)) * 0.5
    dy = rng.normal(size=(n, H))
    dx, dw1, dw3, dw2 = O.expert_ffn_backward_f64(x, experts, w1, w3, w2, act, dy)
    loss = lambda: float(np.sum(dy * _fwd(x, experts, w1, w3, w2, act)))
    for arr, grad in ((x, dx), (w1, dw1), (w2, dw2)) + (((w3, dw3),) if act == "swiglu" else ()):
        for i, num in _fd(loss, arr, rng):
            assert abs(grad[i] - num) <= 1e-6 * max(1.0, abs(num)), (i, grad[i], num)


def test_replica_rows_reduce_into_the_expert():
    """Splitting an expert's rows over several groups changes nothing: its
    weight gradient is the sum of the per-row contributions."""
    rng = np.random.default_rng(2)
    n, E, H, F = 12, 2, 4, 6
    x = rng.normal(size=(n, H))
    experts = np.array([0] * 7 + [1] * 5)
    w1 = rng.normal(size=(E, H, F))
    w2 = rng.normal(size=(E, F, H))
    dy = rng.normal(size=(n, H))
    _, dw1, _, dw2 = O.expert_ffn_backward_f64(x, experts, w1, None, w2, "gelu", dy)
    acc1 = np.zeros_like(dw1)
    acc2 = np.zeros_like(dw2)
    for i in range(n):   # one row at a time: the finest replica split
        _, a1, _, a2 = O.expert_ffn_backward_f64(x[i:i + 1], experts[i:i + 1], w1, None, w2, "gelu", dy[i:i + 1])
        acc1 += a1
        acc2 += a2
    assert np.allclose(acc1, dw1, atol=1e-12) and np.allclose(acc2, dw2, atol=1e-12)


def test_combine_backward_matches_finite_differences():
    rng = np.random.default_rng(3)
    T, k, H = 6, 2, 4
    A = T * k
    y = rng.normal(size=(A, H))
    inv = rng.permutation(A)
    w = rng.random((T, k))
    dout = rng.normal(size=(T, H))
    dY, dw = O.combine_backward(dout, y, inv, w)

    def out():
        o = np.zeros((T, H))
        for t in range(T):
            for r in range(k):
                o[t] += w[t, r] * y[inv[t * k + r]]
        return o
    loss = lambda: float(np.sum(dout * out()))
    for arr, grad in ((y, dY), (w, dw)):
        for i, num in _fd(loss, arr, rng):
            assert abs(grad[i] - num) <= 1e-6 * max(1.0, abs(num))


def test_scatter_sum_is_the_adjoint_of_the_row_copy():
    rng = np.random.default_rng(4)
    T, k, H = 5, 3, 4
    inv = rng.permutation(T * k)
    dxp = rng.normal(size=(T * k, H))
    x = rng.normal(size=(T, H))
    xp = np.zeros((T * k, H))
    for t in range(T):
        for r in range(k):
            xp[inv[t * k + r]] = x[t]
    # <copy(x), dxp> = <x, scatter_sum(dxp)>
    assert abs(np.sum(xp * dxp) - np.sum(x * O.scatter_sum(dxp, inv, T, k))) < 1e-12


@pytest.mark.parametrize("renorm", [True, False])
def test_router_backward_matches_finite_differences(renorm):
    rng = np.random.default_rng(5 + renorm)
    T, E, k = 4, 7, 3
    logits = rng.normal(size=(T, E)) * 2
    idx, w = O.topk_gate(logits, k, renorm)
    dw = rng.normal(size=(T, k))
    g = O.router_backward(logits, idx, dw, renorm)

    def weights():
        out = np.zeros((T, k))
        for t in range(T):
            if renorm:
                z = np.exp(logits[t, idx[t]] - logits[t, idx[t]].max())
                out[t] = z / z.sum()
            else:
                z = np.exp(logits[t] - logits[t].max())
                out[t] = (z / z.sum())[idx[t]]
        return out
    loss = lambda: float(np.sum(dw * weights()))
    for i, num in _fd(loss, logits, rng, n=20):
        assert abs(g[i] - num) <= 1e-6 * max(1.0, abs(num)), (i, g[i], num)

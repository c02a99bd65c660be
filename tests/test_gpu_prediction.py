"""Prediction-driven replication on the GPU against the oracle: the
decay-weighted window prediction (moe_predict_decay) and the replica table
from a predicted popularity (moe_replicate_predicted)."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from moe_expert_routing_02_b300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402

PROB_TOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def _stream(name, iters, T=None, L=None):
    """Run the separate stats calls and the oracle side by side; yields
    (it, layer, gpu stats handle, oracle window) after each layer update."""
    c = W.config_by_name(name)
    L = c.L if L is None else L
    st = M.MoEStats(L, c.E, c.window)
    ws = O.WindowStats(L, c.E, c.window)
    for it in range(iters):
        lgs = W.make_layer_logits(c, it, T=T, layers=L)
        prev = prev_np = None
        for j in range(L):
            idx_np, _ = O.topk_gate(lgs[j], c.k)
            idx = dev(idx_np)
            M.moe_stats_update(st, it, j, idx, prev)
            ws.update(it, j, idx_np, prev_np)
            yield c, it, j, st, ws
            prev, prev_np = idx, idx_np


@pytest.mark.parametrize("name,T", [("tiny", None), ("moe_gpt_stream", 2048)])
def test_decay_one_is_moe_predict_bit_for_bit(name, T):
    for c, it, j, st, ws in _stream(name, 12, T=T, L=3):
        a = M.moe_predict(st, j)
        b = M.moe_predict_decay(st, j, it, 1.0)
        for x, y in zip(a, b):
            if x is None:
                assert y is None
            else:
                assert torch.equal(x, y), (it, j)


@pytest.mark.parametrize("lam", [0.0, 0.5, 0.9])
@pytest.mark.parametrize("name,T", [("tiny", None), ("moe_gpt_stream", 2048)])
def test_decay_matches_oracle(name, T, lam):
    """Every (iteration, layer) of a 13-iteration stream, including the first
    iterations where the window is not full yet."""
    for c, it, j, st, ws in _stream(name, 13, T=T, L=3):
        got = M.moe_predict_decay(st, j, it, lam)
        want = ws.predict_decay(j, it, lam)
        for g, w_ in zip(got, want):
            if w_ is None:
                assert g is None
                continue
            assert np.max(np.abs(host(g).astype(np.float64) - w_)) <= PROB_TOL, (it, j, lam)


def test_decay_rejects_bad_arguments():
    st = M.MoEStats(2, 8, 10)
    with pytest.raises(M.MoEError):
        M.moe_predict_decay(st, 0, 0, 1.5)
    with pytest.raises(M.MoEError):
        M.moe_predict_decay(st, 0, -1, 0.5)
    f32 = dict(dtype=torch.float32, device="cuda")
    with pytest.raises(M.MoEError):  # the last layer has no next layer
        M.moe_predict_decay(st, 1, 0, 0.5, out=(torch.empty(8, **f32), None, torch.empty(8, **f32)))


def _check_table(p32, total, thresh=(6, 5), max_copies=-1, budget=-1):
    load, copies, rb, ge = M.moe_replicate_predicted(dev(p32), total, thresh, max_copies, budget)
    M.moe_check()
    ol, oc, orb, oge = O.replicate_predicted(p32, total, thresh[0], thresh[1], max_copies, budget)
    assert host(load).tolist() == ol.tolist()
    assert host(copies).tolist() == oc.tolist()
    assert host(rb).tolist() == orb.tolist()
    assert host(ge).tolist() == oge.tolist()
    assert int(host(load).sum()) == total


@pytest.mark.parametrize("seed", range(8))
def test_replicate_predicted_matches_oracle(seed):
    """Seeded shares (Dirichlet, rounded to float32), drawn here and given to
    both sides; bit-exact loads and tables, with and without cap and budget."""
    rng = np.random.default_rng(seed)
    for E in (1, 2, 7, 16, 160, 256):
        p = rng.dirichlet(np.ones(E) * (0.2 + seed * 0.3)).astype(np.float32)
        total = int(rng.integers(1, 1 << 20))
        _check_table(p, total)
        _check_table(p, total, max_copies=1)
        _check_table(p, total, budget=int(rng.integers(0, 4)))
        _check_table(p, total, thresh=(3, 2), budget=E)


def test_replicate_predicted_edges():
    # hand cases of the golden file, and shares summing above / below 1
    _check_table(np.array([0.5, 0.25, 0.125, 0.125], np.float32), 10)
    _check_table(np.array([0.5, 0.5, 0.25], np.float32), 4)          # floors above the total
    _check_table(np.array([1 / 3] * 3, np.float32), 10)               # equal remainders
    _check_table(np.array([0.0, 1.0, 0.0], np.float32), 7)
    _check_table(np.array([0.2, 0.2, 0.2, 0.2], np.float32), 1000)    # shares below 1: leftovers cycle
    _check_table(np.array([1e-30, 1e-40, 0.5, 0.5], np.float32), 999)  # tiny and denormal shares
    _check_table(np.array([-0.1, 0.6, 0.5], np.float32), 50)           # a negative share counts as 0
    with pytest.raises(M.MoEError):
        M.moe_replicate_predicted(dev(np.ones(4, np.float32) / 4), 1 << 29)
    # a NaN share: counted as 0 and reported
    M.moe_replicate_predicted(dev(np.array([np.nan, 0.5, 0.5], np.float32)), 10)
    with pytest.raises(M.MoEError) as ei:
        M.moe_check()
    assert ei.value.status == M.MOE_ERR_DEVICE


def test_replicate_predicted_from_the_gpu_prediction():
    """The chain moe_predict -> moe_replicate_predicted against the oracle's
    own chain (its fp64 prediction rounded to float32).  The two float32
    predictions agree to an ulp, so loads must agree exactly unless an exact
    quota sits within that ulp of an integer or of a remainder tie; there only
    the validity of the result is checked (sum, floor/ceil of the quota)."""
    checked = exact = 0
    for c, it, j, st, ws in _stream("moe_gpt_stream", 12, T=4096, L=3):
        if j == c.L - 1 or j == 2:
            continue
        _, _, p_next = M.moe_predict(st, j)
        A = 4096 * c.k
        load, copies, rb, ge = M.moe_replicate_predicted(p_next, A)
        _, _, want_p = ws.predict(j)
        p32 = want_p.astype(np.float32)
        ol, oc, orb, oge = O.replicate_predicted(p32, A)
        gl = host(load)
        assert gl.sum() == A
        q = want_p * A
        ulp_q = A * np.abs(np.spacing(p32.astype(np.float32))).astype(np.float64) * 2
        frac = q - np.floor(q)
        near_int = np.minimum(frac, 1 - frac) <= ulp_q
        rem_sorted = np.sort(frac)
        near_tie = np.any(np.diff(rem_sorted) <= 2 * ulp_q.max())
        checked += 1
        if not near_int.any() and not near_tie:
            assert gl.tolist() == ol.tolist()
            assert host(copies).tolist() == oc.tolist() and host(rb).tolist() == orb.tolist()
            exact += 1
        else:
            assert np.all(np.abs(gl - q) < 1 + 1e-9)
    assert checked > 0 and exact > 0

"""moe_layer_front (route + statistics + prediction + replicas + dispatch in two
launches) against the separate calls, bit for bit, and against the oracle."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from moe_expert_routing_02_b300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()


def _separate(lg, x, st, it, j, k, idx_prev, predict, replicate):
    idx, w = M.moe_route(lg, k)
    E = lg.shape[1]
    hist = torch.empty(E, dtype=torch.int32, device="cuda")
    M.moe_stats_update(st, it, j, idx, idx_prev, hist_out=hist)
    out = {"idx": idx, "w": w, "hist": hist}
    if predict:
        out["p_seq"], out["cond"], out["p_next"] = M.moe_predict(st, j)
    rb = None
    if replicate:
        out["copies"], out["rep_base"], out["group_expert"] = M.moe_replicate(hist, idx.numel())
        rb = out["rep_base"]
    out["group_offsets"], out["perm"], out["inv_perm"], out["xp"] = M.moe_dispatch(x, idx, E, rb)
    return out


def _compare(a, b, keys):
    for key in keys:
        if a.get(key) is None and b.get(key) is None:
            continue
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("name", [c.name for c in W.CONFIGS])
@pytest.mark.parametrize("replicate", [False, True])
def test_front_matches_separate_calls(name, replicate):
    c = W.config_by_name(name)
    L = min(c.L, 3)
    st_a = M.MoEStats(c.L, c.E, c.window)
    st_b = M.MoEStats(c.L, c.E, c.window)
    keys = ["idx", "w", "hist", "p_seq", "cond", "p_next", "copies", "rep_base", "group_expert",
            "group_offsets", "perm", "inv_perm", "xp"]
    for it in range(3):
        lgs = W.make_layer_logits(c, it, layers=L)
        prev_a = prev_b = None
        for j in range(L):
            lg = torch.from_numpy(lgs[j]).cuda()
            x = W.make_x(c, it, j, device="cuda") if j == 0 or c.H <= 1024 else None
            a = _separate(lg, x, st_a, it, j, c.k, prev_a, True, replicate)
            b = M.moe_layer_front(lg, x, st_b, it, j, c.k, idx_prev=prev_b, predict=True, replicate=replicate)
            M.moe_check()
            _compare(a, b, keys)
            prev_a, prev_b = a["idx"], b["idx"]
    assert st_a.export_state() == st_b.export_state()


def test_front_edges_and_oracle():
    rng = np.random.default_rng(9)
    for T, E, k in [(1, 4, 2), (17, 8, 3), (1000, 160, 6), (2049, 256, 8), (5000, 16, 1), (333, 64, 4)]:
        st_a = M.MoEStats(2, E, 4)
        st_b = M.MoEStats(2, E, 4)
        prev_a = prev_b = None
        for j in range(2):
            lg_np = rng.standard_normal((T, E)).astype(np.float32)
            lg_np[:, ::5] = np.round(lg_np[:, ::5])
            lg = torch.from_numpy(lg_np).cuda()
            x = torch.randn((T, 64), device="cuda").to(torch.bfloat16)
            a = _separate(lg, x, st_a, 1, j, k, prev_a, True, True)
            b = M.moe_layer_front(lg, x, st_b, 1, j, k, idx_prev=prev_b, replicate=True)
            M.moe_check()
            _compare(a, b, list(a))
            oi, _ = O.topk_gate(lg_np, k)
            assert np.array_equal(b["idx"].cpu().numpy(), oi)
            go, perm, inv = O.dispatch(oi, E, b["rep_base"].cpu().numpy())
            assert np.array_equal(b["perm"].cpu().numpy(), perm)
            prev_a, prev_b = a["idx"], b["idx"]
        assert st_a.export_state() == st_b.export_state()
    # empty batch and permutation only
    st = M.MoEStats(1, 8, 4)
    out = M.moe_layer_front(torch.empty((0, 8), device="cuda"), None, st, 0, 0, 2)
    M.moe_check()
    assert out["group_offsets"].cpu().tolist() == [0] * 17


@pytest.mark.parametrize("budget", [-1, 0, 2])
def test_front_replicates_from_a_prediction(budget):
    """rep_share: the front's replica table equals moe_replicate_predicted on
    the same shares (and, with budget, the oracle's capped table); the rest of
    the front is unchanged."""
    c = W.config_by_name("moe_gpt_stream")
    T, L = 4096, 3
    st_a = M.MoEStats(L, c.E, c.window)
    st_b = M.MoEStats(L, c.E, c.window)
    lgs = W.make_layer_logits(c, 0, T=T, layers=L)
    x = W.make_x(c, 0, 0, device="cuda", T=T)
    prev_a = prev_b = None
    share = None
    for j in range(L):
        lg = torch.from_numpy(lgs[j]).cuda()
        a = M.moe_layer_front(lg, x, st_a, 0, j, c.k, idx_prev=prev_a, predict=True, replicate=True,
                              rep_share=share, budget=budget)
        b = _separate(lg, x, st_b, 0, j, c.k, prev_b, True, False)
        if share is not None:
            load, copies, rb, ge = M.moe_replicate_predicted(share, T * c.k, budget=budget)
            p32 = share.cpu().numpy()
            ol, oc, orb, oge = O.replicate_predicted(p32, T * c.k, budget=budget)
            assert copies.cpu().numpy().tolist() == oc.tolist()
        else:
            copies, rb, ge = M.moe_replicate(b["hist"], T * c.k)
            if budget >= 0:
                oc = O.cap_copies(copies.cpu().numpy(), b["hist"].cpu().numpy(), budget)
                copies = torch.from_numpy(oc).cuda()
                rb = torch.from_numpy(np.concatenate([[0], np.cumsum(oc.astype(np.int64) + 1)]).astype(np.int32)).cuda()
                ge_np = np.full(2 * c.E, -1, np.int32)
                ge_np[:int(rb[-1])] = np.repeat(np.arange(c.E), oc + 1)
                ge = torch.from_numpy(ge_np).cuda()
        assert torch.equal(a["copies"], copies) and torch.equal(a["rep_base"], rb) and torch.equal(a["group_expert"], ge)
        go, perm, inv, xp = M.moe_dispatch(x, b["idx"], c.E, rb)
        for key, ref in (("idx", b["idx"]), ("w", b["w"]), ("hist", b["hist"]), ("p_seq", b["p_seq"]),
                         ("group_offsets", go), ("perm", perm), ("inv_perm", inv), ("xp", xp)):
            assert torch.equal(a[key], ref), (j, key)
        if j < L - 1:
            assert torch.equal(a["p_next"], b["p_next"])
            share = a["p_next"].clone()
        prev_a, prev_b = a["idx"], b["idx"]
    M.moe_check()


def _front_vs_oracle(lg_np, x, st, ost, it, j, k, prev_d, prev_o, oracle_pred):
    """One fused-front call against the oracle at the same point of the
    stream: routing, histogram, window ring and sums, prediction, replica
    table and dispatch (with the row copy)."""
    E = lg_np.shape[1]
    lg = torch.from_numpy(lg_np).cuda()
    b = M.moe_layer_front(lg, x, st, it, j, k, idx_prev=prev_d, predict=True, replicate=True)
    M.moe_check()
    oi, ow = O.topk_gate(lg_np, k)
    assert np.array_equal(b["idx"].cpu().numpy(), oi), (it, j)
    assert np.abs(b["w"].cpu().numpy() - ow).max() <= 1e-6
    oh = ost.update(it, j, oi, prev_o)
    assert np.array_equal(b["hist"].cpu().numpy(), oh), (it, j)
    ring_h, hsum, ring_c, csum = st.state_arrays()
    assert np.array_equal(ring_h.astype(np.int64), ost.h), (it, j)
    assert np.array_equal(ring_c.astype(np.int64), ost.C), (it, j)
    assert np.array_equal(hsum[j].astype(np.int64), ost.window_hist(j)), (it, j)
    if j > 0:
        assert np.array_equal(csum[j - 1].astype(np.int64), ost.window_cosel(j - 1)), (it, j)
    op, oc, opn = oracle_pred(j)
    assert np.abs(b["p_seq"].cpu().numpy() - op).max() <= 1e-6, (it, j)
    if oc is not None:
        assert np.abs(b["cond"].cpu().numpy() - oc).max() <= 1e-6, (it, j)
        assert np.abs(b["p_next"].cpu().numpy() - opn).max() <= 1e-6, (it, j)
    copies, rb, ge = O.replicate(oh, oi.size)
    assert b["copies"].cpu().numpy().tolist() == copies.tolist(), (it, j)
    assert b["rep_base"].cpu().numpy().tolist() == rb.tolist(), (it, j)
    G = int(rb[-1])
    assert b["group_expert"].cpu().numpy()[:G].tolist() == ge[:G].tolist(), (it, j)
    go, perm, inv = O.dispatch(oi, E, rb)
    assert np.array_equal(b["group_offsets"].cpu().numpy(), go), (it, j)
    assert np.array_equal(b["perm"].cpu().numpy(), perm), (it, j)
    assert np.array_equal(b["inv_perm"].cpu().numpy(), inv), (it, j)
    if x is not None:
        src = b["perm"].long() // k
        assert torch.equal(b["xp"], x[src]), (it, j)
    return b, oi, G


def test_front_across_ring_wrap_moe_gpt_stream():
    """The fused front over the full-size moe_gpt_stream workload (12 layers,
    T = 16384, window s = 10) for 25 iterations -- the ring wraps twice, so
    every window sum has had slots replaced (new - old) -- and then for
    iterations 50..55 of the stationary skewed phase, where hot experts get
    replicas.  Every layer of every iteration is compared with the oracle's
    window (PopFetcher review, Routing Information Collector, s = 10)."""
    c = W.config_by_name("moe_gpt_stream")
    st = M.MoEStats(c.L, c.E, c.window)
    ost = O.WindowStats(c.L, c.E, c.window)
    extra = 0
    its = list(range(25)) + list(range(50, 56))
    for it in its:
        lgs = W.make_layer_logits(c, it)
        prev_d = prev_o = None
        for j in range(c.L):
            x = W.make_x(c, it, j, device="cuda") if j in (0, c.L - 1) else None
            b, oi, G = _front_vs_oracle(lgs[j], x, st, ost, it, j, c.k, prev_d, prev_o, ost.predict)
            if it >= 50:
                extra += G - c.E
            prev_d, prev_o = b["idx"], oi
    assert extra > 0   # the skewed phase does split hot experts


@pytest.mark.parametrize("T,E,k", [(1, 4, 2), (17, 8, 3), (1000, 160, 6), (2049, 256, 8), (5000, 16, 1),
                                   (333, 64, 4)])
def test_front_across_ring_wrap_edges(T, E, k):
    """Window s = 4 over 10 iterations of three layers (the ring wraps twice),
    tie-heavy logits, edge shapes: every call against the oracle."""
    rng = np.random.default_rng([T, E, k])
    L, s = 3, 4
    st = M.MoEStats(L, E, s)
    ost = O.WindowStats(L, E, s)
    for it in range(10):
        prev_d = prev_o = None
        for j in range(L):
            lg_np = rng.standard_normal((T, E)).astype(np.float32)
            lg_np[:, ::5] = np.round(lg_np[:, ::5])
            lg_np[:, 0] += 1.5 * (it % 3)     # drifting skew: replica tables change
            x = torch.randn((T, 64), device="cuda").to(torch.bfloat16)
            b, oi, _ = _front_vs_oracle(lg_np, x, st, ost, it, j, k, prev_d, prev_o, ost.predict)
            prev_d, prev_o = b["idx"], oi


@pytest.mark.parametrize("T,E,k,H", [(131149, 16, 2, 64), (200003, 160, 6, 8), (150001, 256, 8, 8),
                                     (70001, 63, 3, 16)])
def test_front_many_tiles(T, E, k, H):
    """Past 512 dispatch tiles (T > 65,536: 128-token tiles, many tiles per
    route block, every segment of route blocks in use; E dividing the block or
    not, so both ways of summing the earlier totals run), two layers: bit-identical
    to the separate calls, and routing, histogram and dispatch against the
    oracle."""
    rng = np.random.default_rng([11, T, E])
    st_a = M.MoEStats(2, E, 3)
    st_b = M.MoEStats(2, E, 3)
    prev_a = prev_b = None
    bias = -1.1 * np.log(np.arange(1, E + 1, dtype=np.float64))
    for j in range(2):
        lg_np = (rng.standard_normal((T, E)) + bias[None, :]).astype(np.float32)
        lg_np[:, ::7] = np.round(lg_np[:, ::7])
        lg = torch.from_numpy(lg_np).cuda()
        x = torch.randn((T, H), device="cuda").to(torch.bfloat16)
        a = _separate(lg, x, st_a, 2, j, k, prev_a, True, True)
        b = M.moe_layer_front(lg, x, st_b, 2, j, k, idx_prev=prev_b, predict=True, replicate=True)
        M.moe_check()
        _compare(a, b, list(a))
        oi, _ = O.topk_gate(lg_np, k)
        assert np.array_equal(b["idx"].cpu().numpy(), oi)
        oh = np.bincount(oi.ravel(), minlength=E)
        assert np.array_equal(b["hist"].cpu().numpy(), oh)
        go, perm, inv = O.dispatch(oi, E, b["rep_base"].cpu().numpy())
        assert np.array_equal(b["group_offsets"].cpu().numpy(), go)
        assert np.array_equal(b["perm"].cpu().numpy(), perm)
        assert np.array_equal(b["inv_perm"].cpu().numpy(), inv)
        prev_a, prev_b = a["idx"], b["idx"]
    assert st_a.export_state() == st_b.export_state()


@pytest.mark.parametrize("name", [c.name for c in W.CONFIGS])
def test_front_one_launch_matches_two_launches(name):
    """The one-launch front (cooperative, grid-wide barrier) against the two
    launches: every output and the window state bit-identical, over iterations
    that wrap the window ring, with replicas and the prediction on."""
    c = W.config_by_name(name)
    L = min(c.L, 3)
    st = {f: M.MoEStats(c.L, c.E, c.window) for f in (0, 1)}
    keys = ["idx", "w", "hist", "p_seq", "cond", "p_next", "copies", "rep_base", "group_expert",
            "group_offsets", "perm", "inv_perm", "xp"]
    try:
        for it in range(c.window + 2):
            lgs = W.make_layer_logits(c, it, layers=L)
            prev = {0: None, 1: None}
            for j in range(L):
                lg = torch.from_numpy(lgs[j]).cuda()
                x = W.make_x(c, it, j, device="cuda") if j == 0 or c.H <= 1024 else None
                out = {}
                for f in (0, 1):
                    M.moe_set_option(M.MOE_OPT_FRONT_ONE_LAUNCH, f)
                    out[f] = M.moe_layer_front(lg, x, st[f], it, j, c.k, idx_prev=prev[f], predict=True,
                                               replicate=True)
                    M.moe_check()
                    prev[f] = out[f]["idx"]
                _compare(out[0], out[1], keys)
    finally:
        M.moe_set_option(M.MOE_OPT_FRONT_ONE_LAUNCH, 0)
    assert st[0].export_state() == st[1].export_state()

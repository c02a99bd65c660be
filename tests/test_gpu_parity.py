"""GPU parity: every kernel, through the C ABI, against the CPU oracle on the
same seeded inputs.

Bars: bit-exact for indices, counts, replica tables, permutations and the
dispatched row copy; 1e-6 absolute for gate weights and the popularity /
probability outputs; 2e-2 relative Frobenius error for the bf16 FFN output
(fp32 accumulation, bf16 intermediate) against the fp64 oracle; the combine
within one bf16 rounding of the oracle fed the GPU's expert outputs.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O
from moe_expert_routing_02_b300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402

FFN_TOL = 2e-2
PROB_TOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()
    yield
    torch.cuda.synchronize()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def ok_check():
    M.moe_check()


KERNELS = {"auto": 0, "single": 1, "pair": 2}


@pytest.fixture
def ffn_kernel(request):
    """Force the grouped-GEMM kernel for one test, then restore the default."""
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, KERNELS[request.param])
    yield request.param
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, M.MOE_FFN_KERNEL_AUTO)


# ----------------------------------------------------------------------------
# K1 route
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("name", [c.name for c in W.CONFIGS])
def test_route_configs(name):
    c = W.config_by_name(name)
    for j, lg in enumerate(W.make_layer_logits(c, 3, layers=min(c.L, 3))):
        for renorm in (True, False):
            idx, w = M.moe_route(dev(lg), c.k, renorm)
            oi, ow = O.topk_gate(lg, c.k, renorm)
            assert np.array_equal(host(idx), oi), (name, j)
            assert np.abs(host(w) - ow).max() <= PROB_TOL
    ok_check()


@pytest.mark.parametrize("E", [1, 2, 3, 5, 8, 13, 16, 17, 31, 64, 100, 160, 255, 256])
def test_route_shapes_and_ties(E):
    rng = np.random.default_rng(E)
    for T in (1, 33, 1000):
        for k in sorted({1, min(2, E), min(E, 8)}):
            lg = rng.standard_normal((T, E)).astype(np.float32)
            lg[:, ::3] = np.round(lg[:, ::3])            # exact ties
            lg[rng.random(lg.shape) < 0.1] = -0.0         # -0.0 against +0.0
            lg[rng.random(lg.shape) < 0.1] = 0.0
            for renorm in (True, False):
                idx, w = M.moe_route(dev(lg), k, renorm)
                oi, ow = O.topk_gate(lg, k, renorm)
                assert np.array_equal(host(idx), oi), (T, k)
                assert np.abs(host(w) - ow).max() <= PROB_TOL
    # empty batch
    M.moe_route(torch.empty((0, E), dtype=torch.float32, device="cuda"), 1)
    ok_check()


# ----------------------------------------------------------------------------
# K2/K3 stats over a stream
# ----------------------------------------------------------------------------
def _stream_parity(c, iters, T=None, predict_every=1):
    st = M.MoEStats(c.L, c.E, c.window)
    ost = O.WindowStats(c.L, c.E, c.window)
    hist = torch.empty(c.E, dtype=torch.int32, device="cuda")
    for it in range(iters):
        lg = W.make_layer_logits(c, it, T=T)
        prev_d = prev_o = None
        for j in range(c.L):
            oi, _ = O.topk_gate(lg[j], c.k)
            di = dev(oi)
            M.moe_stats_update(st, it, j, di, prev_d, hist_out=hist)
            oh = ost.update(it, j, oi, prev_o)
            assert np.array_equal(host(hist), oh), (it, j)
            if it % predict_every == 0 or it == iters - 1:
                p, cond, pn = M.moe_predict(st, j)
                op, oc, opn = ost.predict(j)
                assert np.abs(host(p) - op).max() <= PROB_TOL, (it, j)
                if oc is not None:
                    assert np.abs(host(cond) - oc).max() <= PROB_TOL
                    assert np.abs(host(pn) - opn).max() <= PROB_TOL
                    assert abs(float(host(pn).sum()) - 1.0) < 1e-5
            prev_d, prev_o = di, oi
    ring_h, hsum, ring_c, csum = st.state_arrays()
    assert np.array_equal(ring_h.astype(np.int64), ost.h)
    assert np.array_equal(ring_c.astype(np.int64), ost.C)
    for j in range(c.L):
        assert np.array_equal(hsum[j].astype(np.int64), ost.window_hist(j))
    for j in range(c.L - 1):
        assert np.array_equal(csum[j].astype(np.int64), ost.window_cosel(j))
    ok_check()
    return st


def test_stats_tiny_stream():
    _stream_parity(W.config_by_name("tiny"), 10)


def test_stats_moe_gpt_stream_full_size():
    # 25 iterations: the ring wraps twice and the skew is still ramping
    _stream_parity(W.config_by_name("moe_gpt_stream"), 25, predict_every=4)


def test_stats_ring_overwrite_hand_case():
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "window_hand.json")))
    st = M.MoEStats(g["L"], g["E"], g["s"])
    for step in g["stream"]:
        it = step["it"]
        a = dev(np.array(step["layer0"], np.int32))
        M.moe_stats_update(st, it, 0, a)
        if it == 2:
            p, cond, pn = M.moe_predict(st, 0)
            assert np.allclose(host(pn), g["mid_it2"]["p_next"], atol=PROB_TOL)
        M.moe_stats_update(st, it, 1, dev(np.array(step["layer1"], np.int32)), a)
    p, cond, pn = M.moe_predict(st, 0)
    assert np.allclose(host(p), g["end_it2"]["p_seq"], atol=PROB_TOL)
    assert np.allclose(host(cond), g["end_it2"]["cond"], atol=PROB_TOL)
    assert np.allclose(host(pn), g["end_it2"]["p_next"], atol=PROB_TOL)
    ok_check()


def test_stats_checkpoint_resume():
    c = W.config_by_name("tiny")
    a = M.MoEStats(c.L, c.E, c.window)
    b = M.MoEStats(c.L, c.E, c.window)
    for it in range(7):
        lg = W.make_layer_logits(c, it)
        i0 = M.moe_route(dev(lg[0]), c.k)[0]
        i1 = M.moe_route(dev(lg[1]), c.k)[0]
        M.moe_stats_update(a, it, 0, i0)
        M.moe_stats_update(a, it, 1, i1, i0)
        if it == 3:
            b.import_state(a.export_state())
        elif it > 3:
            M.moe_stats_update(b, it, 0, i0)
            M.moe_stats_update(b, it, 1, i1, i0)
    assert a.export_state() == b.export_state()
    pa, pb = M.moe_predict(a, 0), M.moe_predict(b, 0)
    for x, y in zip(pa, pb):
        assert torch.equal(x, y)


@pytest.mark.parametrize("E,k", [(1, 1), (2, 1), (2, 2), (5, 2), (8, 1), (8, 2), (13, 2), (16, 1), (16, 2),
                                 (16, 3), (16, 4)])
def test_stats_small_e_coselection_shapes(E, k):
    """Up to 16 experts (the register-histogram kernel; for k <= 2 its
    co-selection counts come from bf16 MMAs over one-hot choice counts):
    ragged token counts that leave partial warps and blocks, repeated experts
    within a token's choices (each pair counts), k = 1, out-of-range ids
    (flagged; only their own pairs are dropped).  Ring slots and window sums
    against the oracle, bit for bit."""
    rng = np.random.default_rng([5, E, k])
    for T in (1, 31, 33, 1000, 4097, 100003):
        st = M.MoEStats(2, E, 3)
        prev = rng.integers(0, E, (T, k)).astype(np.int32)
        cur = rng.integers(0, E, (T, k)).astype(np.int32)
        M.moe_stats_update(st, 0, 0, dev(prev))
        M.moe_stats_update(st, 0, 1, dev(cur), dev(prev))
        ok_check()
        ring_h, hsum, ring_c, csum = st.state_arrays()
        assert np.array_equal(ring_h[0, 0].astype(np.int64), O.histogram(prev, E)), T
        assert np.array_equal(ring_h[1, 0].astype(np.int64), O.histogram(cur, E)), T
        assert np.array_equal(ring_c[0, 0].astype(np.int64), O.coselection(prev, cur, E)), T
        assert np.array_equal(csum[0].astype(np.int64), O.coselection(prev, cur, E)), T
    # an out-of-range id in either layer: flagged, and only its own pairs are left out
    st = M.MoEStats(2, E, 3)
    prev = rng.integers(0, E, (300, k)).astype(np.int32)
    cur = rng.integers(0, E, (300, k)).astype(np.int32)
    prev[7, 0] = E + 3
    cur[11, k - 1] = -1
    M.moe_stats_update(st, 1, 1, dev(cur), dev(prev))
    with pytest.raises(M.MoEError):
        M.moe_check()
    M.moe_check()
    keep_p = (prev >= 0) & (prev < E)
    keep_c = (cur >= 0) & (cur < E)
    want = np.zeros((E, E), np.int64)
    for t in range(300):
        for r1 in range(k):
            for r2 in range(k):
                if keep_p[t, r1] and keep_c[t, r2]:
                    want[prev[t, r1], cur[t, r2]] += 1
    _, _, ring_c, _ = st.state_arrays()
    assert np.array_equal(ring_c[0, 1].astype(np.int64), want)


def test_stats_empty_batch_and_invalid_ids():
    st = M.MoEStats(2, 8, 4)
    e = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    M.moe_stats_update(st, 0, 0, e)
    M.moe_stats_update(st, 0, 1, e, e)
    p, cond, pn = M.moe_predict(st, 0)
    assert np.allclose(host(p), 1 / 8) and np.allclose(host(pn), 1 / 8)
    ok_check()
    bad = dev(np.array([[0, 9]], np.int32))     # 9 is not an expert
    M.moe_stats_update(st, 1, 0, bad)
    with pytest.raises(M.MoEError) as ei:
        M.moe_check()
    assert ei.value.status == M.MOE_ERR_DEVICE
    M.moe_check()  # cleared


# ----------------------------------------------------------------------------
# K4 replicate
# ----------------------------------------------------------------------------
def test_replicate_hand_tables_and_random():
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "replicate_table.json")))
    for case in g["cases"]:
        c, rb, ge = M.moe_replicate(dev(np.array(case["load"], np.int32)), case["total"],
                                    max_copies=case.get("max_copies", -1))
        assert host(c).tolist() == case["copies"]
        assert host(rb).tolist() == case["rep_base"]
        oc, orb, oge = O.replicate(case["load"], case["total"], 6, 5, case.get("max_copies", -1))
        assert np.array_equal(host(ge), oge)
    rng = np.random.default_rng(1)
    for trial in range(200):
        E = int(rng.integers(1, 257))
        A = int(rng.integers(E, 200000))
        load = rng.multinomial(A, rng.dirichlet(np.full(E, rng.uniform(0.05, 2)))).astype(np.int32)
        num, den = [(6, 5), (1, 1), (3, 2), (11, 10)][trial % 4]
        cap = [-1, 0, 1, 3][trial % 4]
        c, rb, ge = M.moe_replicate(dev(load), A, (num, den), cap)
        oc, orb, oge = O.replicate(load, A, num, den, cap)
        assert np.array_equal(host(c), oc) and np.array_equal(host(rb), orb) and np.array_equal(host(ge), oge)
    ok_check()


def test_replicate_rejects_loads_above_total():
    c, rb, ge = M.moe_replicate(dev(np.array([10, 10], np.int32)), 5)
    with pytest.raises(M.MoEError):
        M.moe_check()
    assert host(rb).tolist() == [0, 1, 2]  # no-replication table


# ----------------------------------------------------------------------------
# K5 dispatch
# ----------------------------------------------------------------------------
def _dispatch_check(idx_np, E, x=None, rep_base=None):
    go, perm, inv, xp = M.moe_dispatch(None if x is None else x, dev(idx_np), E,
                                       None if rep_base is None else dev(rep_base))
    ogo, operm, oinv = O.dispatch(idx_np, E, rep_base)
    assert np.array_equal(host(go), ogo)
    assert np.array_equal(host(perm), operm)
    assert np.array_equal(host(inv), oinv)
    if x is not None:
        xb = W.bf16_bits(x)
        assert np.array_equal(W.bf16_bits(xp), O.gather_rows(xb, operm, idx_np.shape[1]))
    return go, perm, inv, xp


@pytest.mark.parametrize("name", [c.name for c in W.CONFIGS])
def test_dispatch_configs(name):
    c = W.config_by_name(name)
    lg = W.make_layer_logits(c, 0, layers=1)[0]
    idx, _ = O.topk_gate(lg, c.k)
    x = W.make_x(c, 0, 0, device="cuda")
    _dispatch_check(idx, c.E, x)
    h = O.histogram(idx, c.E)
    rep = O.replicate(h, idx.size)
    _dispatch_check(idx, c.E, x, rep[1])
    ok_check()


def test_dispatch_edges():
    rng = np.random.default_rng(3)
    # ragged sizes around the 1024-assignment tile, one token, all to one expert, E=256, k=8
    for T, k, E in [(1, 1, 1), (1, 2, 4), (511, 2, 8), (512, 2, 8), (513, 2, 8), (1000, 3, 7),
                    (3000, 8, 256), (4097, 6, 160)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        _dispatch_check(idx, E)
        h = O.histogram(idx, E)
        _dispatch_check(idx, E, None, O.replicate(h, idx.size)[1])
    idx = np.zeros((2000, 1), np.int32)     # every token on expert 0: 2 copies... capped by rule
    rb = np.array([0, 3, 4, 5], np.int32)    # hand-made table: expert 0 has 3 replicas
    _dispatch_check(idx, 3, None, rb)
    x = torch.randn((300, 64), device="cuda").to(torch.bfloat16)
    _dispatch_check(rng.integers(0, 5, (300, 2)).astype(np.int32), 5, x)
    # empty batch
    go, perm, inv, xp = M.moe_dispatch(None, torch.empty((0, 2), dtype=torch.int32, device="cuda"), 8)
    assert host(go).tolist() == [0] * 17
    ok_check()


def test_dispatch_invalid_expert_has_no_slot():
    """An assignment whose expert is out of range is flagged and gets no slot
    (inv_perm -1); every other assignment's slot holds its token's row, and
    perm inverts inv_perm on them."""
    rng = np.random.default_rng(13)
    T, k, E, H = 700, 2, 6, 64
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    bad = [(5, 0), (333, 1), (699, 1)]
    for t, r in bad:
        idx[t, r] = E + 2 if r == 0 else -3
    x = torch.randn((T, H), device="cuda").to(torch.bfloat16)
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), E)
    with pytest.raises(M.MoEError):
        M.moe_check()
    M.moe_check()
    inv_h, perm_h = host(inv), host(perm)
    xh, xph = x.cpu(), xp.cpu()
    for f in range(T * k):
        t, r = divmod(f, k)
        if (t, r) in bad:
            assert inv_h[f] == -1, f
        else:
            s_ = int(inv_h[f])
            assert 0 <= s_ < T * k and perm_h[s_] == f, f
            assert torch.equal(xph[s_], xh[t]), f


# ----------------------------------------------------------------------------
# K6 expert FFN
# ----------------------------------------------------------------------------
def _weights(c, device="cuda"):
    return W.make_weights(c, 0, device=device)


def _ffn_check(c, sample=256, rep=False, seed=0):
    lg = W.make_layer_logits(c, 0, layers=1)[0]
    idx, _ = O.topk_gate(lg, c.k)
    x = W.make_x(c, 0, 0, device="cuda")
    w1, w3, w2 = _weights(c)
    rb = ge = None
    if rep:
        _, rb, ge = O.replicate(O.histogram(idx, c.E), idx.size)
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), c.E, None if rb is None else dev(rb))
    y = M.moe_expert_ffn(xp, go, None if ge is None else dev(ge), None if rb is None else dev(rb),
                         w1, w3, w2, c.act)
    ok_check()
    ogo = host(go)
    G = (2 * c.E) if rep else c.E
    A = idx.size
    rng = np.random.default_rng(seed)
    if sample is None:
        slots = np.arange(A)
    else:
        firsts = [ogo[g] for g in range(G) if ogo[g + 1] > ogo[g]]
        lasts = [ogo[g + 1] - 1 for g in range(G) if ogo[g + 1] > ogo[g]]
        slots = np.unique(np.concatenate([firsts, lasts, rng.integers(0, A, sample)]))
    xb = W.bf16_bits(xp)
    ref = O.expert_ffn(xb, ogo[:G + 1], ge, W.bf16_bits(w1), None if w3 is None else W.bf16_bits(w3),
                       W.bf16_bits(w2), c.act, slots=slots)
    got = O.bf16_to_f64(W.bf16_bits(y)[slots])
    err = rel_fro(got, ref)
    assert err <= FFN_TOL, err
    # every group individually too (a wrong group/expert mapping cannot hide in the average)
    g_of = np.searchsorted(ogo[:G + 1], slots, side="right") - 1
    for g in np.unique(g_of):
        m = g_of == g
        assert rel_fro(got[m], ref[m]) <= FFN_TOL, g
    return err, (go, perm, inv, xp, y, idx, x, (w1, w3, w2), rb, ge)


@pytest.mark.parametrize("ffn_kernel", ["single", "pair"], indirect=True)
def test_ffn_tiny_full(ffn_kernel):
    err, _ = _ffn_check(W.config_by_name("tiny"), sample=None)
    assert err < 1e-2


@pytest.mark.parametrize("name,ffn_kernel", [("moe_gpt_stream", "auto"), ("mixtral_layer", "auto"),
                                              ("deepseekv2_layer", "auto"), ("dbrx_replicated_layer", "auto"),
                                              ("moe_gpt_stream", "single"), ("deepseekv2_layer", "pair")],
                         indirect=["ffn_kernel"])
def test_ffn_full_size_sampled(name, ffn_kernel):
    c = W.config_by_name(name)
    _ffn_check(c, sample=256, rep=c.replicate)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("ffn_kernel", ["single", "pair"], indirect=True)
def test_ffn_ragged_groups_and_partial_tiles(ffn_kernel):
    """Groups of 0, 1, 127, 128, 129 rows; F and H not multiples of the 256 tile."""
    import dataclasses
    c = dataclasses.replace(W.config_by_name("tiny"), name="ragged", E=10, k=1, H=192, F=320, act="swiglu")
    sizes = [0, 1, 127, 128, 129, 300, 255, 256, 257, 513]
    idx = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)])
    np.random.default_rng(0).shuffle(idx)
    idx = idx.reshape(-1, 1)
    T = idx.shape[0]
    x = W.make_x(c, 0, 0, device="cuda", T=T)
    w1, w3, w2 = _weights(c)
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), c.E)
    y = M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, "swiglu")
    ok_check()
    ref = O.expert_ffn(W.bf16_bits(xp), host(go)[:c.E + 1], None, W.bf16_bits(w1), W.bf16_bits(w3),
                       W.bf16_bits(w2), "swiglu")
    got = O.bf16_to_f64(W.bf16_bits(y))
    assert rel_fro(got, ref) <= FFN_TOL
    for g in range(c.E):
        lo, hi = host(go)[g], host(go)[g + 1]
        if hi > lo:
            assert rel_fro(got[lo:hi], ref[lo:hi]) <= FFN_TOL


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("thresh", [0, 64, 1 << 30])
@pytest.mark.parametrize("ffn_kernel", ["single", "pair"], indirect=True)
def test_ffn_small_batch_path_thresholds(thresh, act, ffn_kernel):
    """Experts below small_group_threshold rows take the swap-AB small-batch
    kernel, the rest the grouped kernel: threshold 0 = grouped only, 64 = the
    default split, 2^30 = everything small (groups above 64 rows are then
    split into 64-token chunks).  Every group is checked against the oracle."""
    import dataclasses
    sizes = [0, 1, 15, 16, 17, 63, 64, 65, 127, 200, 300]
    c = dataclasses.replace(W.config_by_name("tiny"), name="small-path", E=len(sizes), k=1, H=192, F=320, act=act)
    idx = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)])
    np.random.default_rng(1).shuffle(idx)
    idx = idx.reshape(-1, 1)
    x = W.make_x(c, 0, 0, device="cuda", T=idx.shape[0])
    w1, w3, w2 = _weights(c)
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), c.E)
    # give the small-batch kernel SMs of its own (the split model may
    # otherwise leave such a small layer to the grouped kernel alone)
    M.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, 8)
    try:
        y = M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, act, small_group_threshold=thresh)
        ok_check()
    finally:
        M.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, 0)
    ref = O.expert_ffn(W.bf16_bits(xp), host(go)[:c.E + 1], None, W.bf16_bits(w1),
                       None if w3 is None else W.bf16_bits(w3), W.bf16_bits(w2), act)
    got = O.bf16_to_f64(W.bf16_bits(y))
    gof = host(go)
    for g in range(c.E):
        lo, hi = gof[g], gof[g + 1]
        if hi > lo:
            assert rel_fro(got[lo:hi], ref[lo:hi]) <= FFN_TOL, (g, sizes[g])


def test_replication_bit_identical_with_small_experts():
    """The tiny workload has both hot experts (replicated) and experts below 64
    rows (small-batch kernel): outputs with and without replication match
    bit for bit."""
    c = W.config_by_name("tiny")
    lg = W.make_layer_logits(c, 0, layers=1)[0]
    x = W.make_x(c, 0, 0, device="cuda")
    w1, w3, w2 = _weights(c)
    idx, w = M.moe_route(dev(lg), c.k)
    h = torch.bincount(idx.reshape(-1).long(), minlength=c.E).to(torch.int32)
    copies, rb, ge = M.moe_replicate(h, idx.numel())
    hh = host(h)
    assert int(host(rb)[-1]) > c.E and (hh < 64).any() and (hh > 0).any()
    outs = []
    for use_rep in (False, True):
        go, perm, inv, xp = M.moe_dispatch(x, idx, c.E, rb if use_rep else None)
        y = M.moe_expert_ffn(xp, go, ge if use_rep else None, rb if use_rep else None, w1, w3, w2, c.act)
        outs.append(M.moe_combine(y, inv, w))
    ok_check()
    assert torch.equal(outs[0], outs[1])


def _rne_bf16(v):
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + ((u >> 16) & 1) + 0x7FFF) >> 16).astype(np.uint16)


def _act_bound(v, x):
    """Half a bf16 ulp of the result (8 significant bits), plus the fp32
    activation's own error: 1e-6 relative, and 3e-7 |x| + 1e-7 absolute.  The
    absolute part covers the erf approximation (|error| <= 1.5e-7, scaled by
    x/2) and the cancellation in 1 + erf for very negative x, where every fp32
    erf has large relative but tiny absolute error."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    half_ulp = np.where(a > 0, 2.0 ** (e - 8), 0.0)
    return half_ulp + 1e-6 * a + 3e-7 * np.abs(x) + 1e-7


@pytest.mark.parametrize("ffn_kernel", ["single", "pair"], indirect=True)
@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_ffn_activation_accuracy_identity_weights(act, ffn_kernel):
    """With identity projections each output is bf16(act(x)) exactly as the
    epilogue computes it: GeLU(x) = x Phi(x) (exact-erf form) or silu(x) * x.
    The GPU value must be the fp64 activation rounded to bf16, up to half an
    ulp plus the error budget of the fp32 activation (see _act_bound).  A tanh
    GeLU (error up to ~1e-3 |x|), a dropped factor or a wrong sign fails."""
    from scipy.special import erf
    E, H, F, T = 2, 64, 128, 512
    eye = torch.eye(H, dtype=torch.float32, device="cuda")
    w1 = torch.zeros((E, H, F), device="cuda")
    w1[:, :, :H] = eye
    w1[:, :, H:] = eye
    w2 = torch.zeros((E, F, H), device="cuda")
    w2[:, :H, :] = eye
    w1, w2 = w1.to(torch.bfloat16), w2.to(torch.bfloat16)
    w3 = w1.clone() if act == "swiglu" else None
    x = torch.linspace(-9.0, 9.0, T * H, device="cuda").reshape(T, H).to(torch.bfloat16)
    idx = torch.arange(T, device="cuda", dtype=torch.int32).remainder(E).reshape(T, 1)
    go, perm, inv, xp = M.moe_dispatch(x, idx, E)
    y = M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, act)
    ok_check()
    xv = O.bf16_to_f64(W.bf16_bits(xp))
    ref = 0.5 * xv * (1.0 + erf(xv / np.sqrt(2.0))) if act == "gelu" else xv / (1.0 + np.exp(-xv)) * xv
    got = O.bf16_to_f64(W.bf16_bits(y))
    err = np.abs(got - ref)
    bound = _act_bound(ref, xv)
    assert np.all(err <= bound), float((err - bound).max())
    # away from the cancellation tail almost every output is the correctly
    # rounded value
    core = np.abs(xv) <= 2.0
    exact = np.mean(got[core] == O.bf16_to_f64(_rne_bf16(ref[core])))
    assert exact > 0.99, exact


# ----------------------------------------------------------------------------
# K7 combine, replication invariance, whole layer
# ----------------------------------------------------------------------------
def test_combine_matches_oracle_on_gpu_y():
    c = W.config_by_name("moe_gpt_stream")
    lg = W.make_layer_logits(c, 0, layers=1)[0]
    idx, w = M.moe_route(dev(lg), c.k)
    A = idx.numel()
    y = torch.randn((A, c.H), device="cuda").to(torch.bfloat16)
    go, perm, inv, _ = M.moe_dispatch(None, idx, c.E)
    out = M.moe_combine(y, inv, w)
    ref = O.combine(W.bf16_bits(y), host(inv), host(w).astype(np.float64))
    got = O.bf16_to_f64(W.bf16_bits(out))
    # one bf16 rounding of an fp32 sum: |err| <= 2^-8 |ref| + fp32 slack
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)
    ok_check()


@pytest.mark.parametrize("ffn_kernel", ["auto", "single"], indirect=True)
def test_replication_output_bit_identical(ffn_kernel):
    c = W.config_by_name("dbrx_replicated_layer")
    lg = W.make_layer_logits(c, 0, layers=1)[0]
    x = W.make_x(c, 0, 0, device="cuda")
    w1, w3, w2 = _weights(c)
    idx, w = M.moe_route(dev(lg), c.k)
    hist = torch.empty(c.E, dtype=torch.int32, device="cuda")
    st = M.MoEStats(1, c.E, 10)
    M.moe_stats_update(st, 0, 0, idx, hist_out=hist)
    copies, rb, ge = M.moe_replicate(hist, idx.numel())
    assert int(host(rb)[-1]) > c.E  # hot experts do get replicas
    outs = []
    for use_rep in (False, True):
        go, perm, inv, xp = M.moe_dispatch(x, idx, c.E, rb if use_rep else None)
        y = M.moe_expert_ffn(xp, go, ge if use_rep else None, rb if use_rep else None, w1, w3, w2, c.act)
        outs.append(M.moe_combine(y, inv, w))
    ok_check()
    assert torch.equal(outs[0], outs[1])


def test_tiny_layer_end_to_end():
    c = W.config_by_name("tiny")
    for j, lg in enumerate(W.make_layer_logits(c, 0)):
        x = W.make_x(c, 0, j, device="cuda")
        w1, w3, w2 = W.make_weights(c, j, device="cuda")
        idx, w = M.moe_route(dev(lg), c.k)
        go, perm, inv, xp = M.moe_dispatch(x, idx, c.E)
        y = M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, c.act)
        out = M.moe_combine(y, inv, w)
        ok_check()
        ref = O.moe_layer(lg, W.bf16_bits(x), c.k, W.bf16_bits(w1), None, W.bf16_bits(w2), c.act)
        assert rel_fro(O.bf16_to_f64(W.bf16_bits(out)), ref["out"]) <= FFN_TOL


# ----------------------------------------------------------------------------
# bounded waits: a wait that runs out is reported, and the context survives
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("ffn_kernel", ["single", "pair"], indirect=True)
def test_ffn_bounded_wait_timeout_is_reported_and_context_survives(ffn_kernel):
    """A one-shot self-test makes CTA (pair) 0 of GEMM1 withhold one
    accumulator-ready signal (a flag nothing else sets): its epilogue's wait
    runs out after ~2 s, the kernel releases TMEM and returns, moe_check
    reports MOE_ERR_TIMEOUT, and the next call on the same context is correct."""
    import time
    c = W.config_by_name("tiny")
    lg = W.make_layer_logits(c, 0, layers=1)[0]
    idx, _ = O.topk_gate(lg, c.k)
    x = W.make_x(c, 0, 0, device="cuda")
    w1, w3, w2 = _weights(c)
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), c.E)
    M.moe_set_option(M.MOE_OPT_FFN_TIMEOUT_SELFTEST, 1)
    t0 = time.time()
    M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, c.act)
    with pytest.raises(M.MoEError) as ei:
        M.moe_check()
    assert ei.value.status == M.MOE_ERR_TIMEOUT
    assert time.time() - t0 < 60
    assert M.moe_get_option(M.MOE_OPT_FFN_TIMEOUT_SELFTEST) == 0   # one-shot
    y = M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, c.act)
    ok_check()
    ref = O.expert_ffn(W.bf16_bits(xp), host(go)[:c.E + 1], None, W.bf16_bits(w1), None, W.bf16_bits(w2), c.act)
    assert rel_fro(O.bf16_to_f64(W.bf16_bits(y)), ref) <= FFN_TOL

"""Backward of the routed expert layer on the GPU (moe_ffn_backward,
moe_route_backward) against the oracle's float64 gradients on the same seeded
bf16 inputs and the same routing.

Tolerances: the GPU rounds dY, the activation, the derivative factors, dz
(dg, du) and dxp to bf16 between its GEMMs (2^-9 relative each, as the
forward rounds its intermediate), so dx and the weight gradients are held to the forward FFN's
2e-2 relative Frobenius error.  dw is an fp32 dot product of bf16 values
(exact products): |error| <= 1e-5 * sum |terms|.  The gate's gradient is fp32
softmax arithmetic: 1e-5 relative to the largest |dw|."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from moe_expert_routing_02_b300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402

GRAD_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _bf16(rng, shape, scale=1.0):
    return (torch.from_numpy(rng.standard_normal(shape).astype(np.float32)) * scale).to(torch.bfloat16).cuda()


def _case(T, E, k, H, F, act, *, seed=0, alpha=1.0, replicate=False, empty=()):
    """Seeded inputs and the routing, shared by both sides."""
    rng = np.random.default_rng(seed)
    logits = W.make_logits(T, E, alpha, seed_key=(seed, 9)) if T else np.zeros((0, E), np.float32)
    logits = np.asarray(logits, np.float32).copy()
    for e in empty:  # experts no token chooses
        logits[:, e] = -1e30
    idx, wf = O.topk_gate(logits, k)
    w32 = wf.astype(np.float32)
    rb = ge = None
    if replicate:
        _, rb, ge = O.replicate(O.histogram(idx, E), max(idx.size, 1))
    go, perm, inv = O.dispatch(idx, E, rb)
    x = _bf16(rng, (T, H))
    dout = _bf16(rng, (T, H))
    y = _bf16(rng, (T * k, H))
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    mk = lambda shape: (torch.randn(shape, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w1 = mk((E, H, F))
    w3 = mk((E, H, F)) if act == "swiglu" else None
    w2 = mk((E, F, H))
    return dict(T=T, E=E, k=k, H=H, F=F, act=act, logits=logits, idx=idx, w=w32, go=go, perm=perm, inv=inv,
                ge=ge, x=x, dout=dout, y=y, w1=w1, w3=w3, w2=w2)


def _gpu(c):
    return M.moe_ffn_backward(c["x"], c["dout"], dev(c["w"]), c["y"], dev(c["perm"]), dev(c["inv"]),
                              dev(c["go"]), None if c["ge"] is None else dev(c["ge"]), c["w1"], c["w3"], c["w2"],
                              c["act"])


def _slot_experts(c):
    A = c["T"] * c["k"]
    go, ge = c["go"], c["ge"]
    G = len(go) - 1 if ge is not None else c["E"]
    ex = np.empty(A, np.int64)
    for g in range(G):
        ex[go[g]:go[g + 1]] = ge[g] if ge is not None else g
    return ex


def _oracle(c):
    T, k = c["T"], c["k"]
    b = lambda t: O.bf16_to_f64(W.bf16_bits(t))
    xp = b(c["x"])[c["perm"].astype(np.int64) // k]
    dY, dw = O.combine_backward(b(c["dout"]), W.bf16_bits(c["y"]), c["inv"], c["w"])
    dxp, dw1, dw3, dw2 = O.expert_ffn_backward_f64(xp, _slot_experts(c), b(c["w1"]),
                                                   None if c["w3"] is None else b(c["w3"]), b(c["w2"]), c["act"], dY)
    dx = O.scatter_sum(dxp, c["inv"], T, k)
    return dx, dw, dw1, dw3, dw2


def _dw_bound(c):
    """sum_h |dout[t,h] y[slot(t,r),h]| for every (t, r)."""
    b = lambda t: np.abs(O.bf16_to_f64(W.bf16_bits(t)))
    d, yy = b(c["dout"]), b(c["y"])
    T, k = c["T"], c["k"]
    return np.stack([np.sum(d * yy[c["inv"][np.arange(T) * k + r]], axis=1) for r in range(k)], axis=1)


def _check(c):
    got = _gpu(c)
    M.moe_check()
    dw, dw1, dw3, dw2 = (None if t is None else host(t) for t in got[1:])
    rdx, rdw, rdw1, rdw3, rdw2 = _oracle(c)
    if c["T"]:
        assert rel_fro(O.bf16_to_f64(W.bf16_bits(got[0])), rdx) <= GRAD_TOL
        assert np.all(np.abs(dw - rdw) <= 1e-5 * _dw_bound(c) + 1e-30)
    for g, r in ((dw1, rdw1), (dw2, rdw2)) + (((dw3, rdw3),) if c["act"] == "swiglu" else ()):
        for e in range(c["E"]):
            if not np.any(r[e]):
                assert not np.any(g[e]), e  # an expert without rows: exactly zero
            else:
                assert rel_fro(g[e], r[e]) <= GRAD_TOL, e
    return got


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_tiny_matches_oracle(act):
    _check(_case(256, 8, 2, 64, 128, act, seed=1))


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_ragged_shapes(act):
    """H and F not multiples of the 128 / 256 tiles (partial m- and n-tiles in
    every GEMM), skewed routing, two experts without rows."""
    _check(_case(300, 6, 2, 192, 320, act, seed=2, alpha=1.5, empty=(1, 4)))


def test_replica_groups_reduce_into_the_expert():
    """With replica groups, every row adds into its expert's one gradient:
    the same result as without replication."""
    c = _case(512, 8, 2, 128, 192, "gelu", seed=3, alpha=1.6, replicate=True)
    assert c["ge"] is not None and len(set(c["ge"][c["ge"] >= 0])) < np.sum(c["ge"] >= 0)
    got = _check(c)
    c2 = dict(c)
    c2["go"], c2["perm"], c2["inv"] = O.dispatch(c["idx"], c["E"])
    c2["ge"] = None
    got2 = _gpu(c2)
    M.moe_check()
    for a, b in zip(got[2:], got2[2:]):
        if a is not None:
            assert rel_fro(host(a), host(b)) <= 1e-2


def test_moe_gpt_stream_layer_slice():
    """moe_gpt_stream's expert shapes (E=16, k=2, H=1024, F=2048, GeLU) on 2048 tokens."""
    c = W.config_by_name("moe_gpt_stream")
    _check(_case(2048, c.E, c.k, c.H, c.F, c.act, seed=4, alpha=1.2))


def test_swiglu_expert_shapes():
    _check(_case(1024, 8, 2, 512, 1024, "swiglu", seed=5, alpha=1.1))


def test_full_size_sampled():
    """The full moe_gpt_stream layer (T = 16384): sampled token gradients and
    weight-gradient entries, each computed by the oracle from the rows it
    depends on."""
    cfg = W.config_by_name("moe_gpt_stream")
    c = _case(cfg.T, cfg.E, cfg.k, cfg.H, cfg.F, cfg.act, seed=6, alpha=1.2)
    got = _gpu(c)
    M.moe_check()
    T, k = c["T"], c["k"]
    b = lambda t: O.bf16_to_f64(W.bf16_bits(t))
    x, dout, yv = b(c["x"]), b(c["dout"]), W.bf16_bits(c["y"])
    w1, w2 = b(c["w1"]), b(c["w2"])
    ex = _slot_experts(c)
    rng = np.random.default_rng(11)
    toks = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, 30)]))
    dxg = O.bf16_to_f64(W.bf16_bits(got[0]))
    for t in toks:
        slots = c["inv"][t * k:(t + 1) * k]
        dY, _ = O.combine_backward(dout[t:t + 1], yv[slots], np.arange(k), c["w"][t:t + 1])
        # the token's k rows against their own experts' weights only
        dxp, _, _, _ = O.expert_ffn_backward_f64(x[np.full(k, t)], np.arange(k), w1[ex[slots]], None,
                                                 w2[ex[slots]], c["act"], dY)
        assert rel_fro(dxg[t], dxp.sum(0)) <= GRAD_TOL, t
    # weight-gradient entries: the FFN separates over its F columns, so column
    # f of dW1[e] and row f of dW2[e] follow from the expert's rows with F = 1
    dw1g, dw2g = host(got[2]), host(got[4])
    for e in rng.choice(c["E"], 3, replace=False):
        rows = np.nonzero(ex == e)[0]
        tok = c["perm"][rows].astype(np.int64) // k
        r = c["perm"][rows].astype(np.int64) % k
        dY = c["w"][tok, r].astype(np.float64)[:, None] * dout[tok]
        for f in rng.integers(0, c["F"], 3):
            _, d1, _, d2 = O.expert_ffn_backward_f64(x[tok], np.zeros(rows.size, np.int64),
                                                     w1[e][:, f:f + 1][None], None, w2[e][f:f + 1][None],
                                                     c["act"], dY)
            assert rel_fro(dw1g[e][:, f], d1[0][:, 0]) <= GRAD_TOL, (e, f)
            assert rel_fro(dw2g[e][f], d2[0][0]) <= GRAD_TOL, (e, f)


def test_no_tokens_gives_zero_weight_gradients():
    c = _case(0, 4, 2, 64, 64, "swiglu", seed=7)
    got = _gpu(c)
    M.moe_check()
    for t in got[2:]:
        assert not torch.any(t)


def test_experts_not_adjacent_is_flagged():
    c = _case(64, 4, 1, 64, 64, "gelu", seed=8)
    A = 64
    c["go"] = np.array([0, 16, 32, 48, A, A, A, A, A], np.int32)
    c["ge"] = np.array([0, 1, 0, 2, -1, -1, -1, -1], np.int32)  # expert 0 in two runs
    c["idx"] = None
    with pytest.raises(M.MoEError) as ei:
        _gpu(c)
        M.moe_check()
    assert ei.value.status == M.MOE_ERR_DEVICE


@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("T,E,k", [(1000, 8, 2), (257, 160, 6), (64, 256, 8), (33, 16, 1)])
def test_route_backward(T, E, k, renorm):
    rng = np.random.default_rng(T + E)
    logits = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    idx, _ = O.topk_gate(logits, k, renorm)
    dw = rng.standard_normal((T, k)).astype(np.float32)
    got = host(M.moe_route_backward(dev(logits), dev(idx.astype(np.int32)), dev(dw), renorm))
    M.moe_check()
    ref = O.router_backward(logits, idx, dw, renorm)
    assert np.max(np.abs(got - ref)) <= 1e-5 * max(1.0, float(np.max(np.abs(dw))))
    if renorm:
        off = np.ones((T, E), bool)
        off[np.arange(T)[:, None], idx] = False
        assert not np.any(got[off])


def test_backward_rejects_bad_arguments():
    c = _case(64, 4, 2, 64, 64, "swiglu", seed=9)
    with pytest.raises(M.MoEError):  # SwiGLU without w3
        M.moe_ffn_backward(c["x"], c["dout"], dev(c["w"]), c["y"], dev(c["perm"]), dev(c["inv"]), dev(c["go"]),
                           None, c["w1"], None, c["w2"], "swiglu")
    assert M.moe_ffn_backward_workspace_bytes(64, 2, 4, 60, 64) == 0


@pytest.mark.parametrize("replicate,physical", [(True, False), (False, False), (True, True)])
def test_layer_step_backward(replicate, physical):
    """MoELayerStep.run(save=True) for every layer of a stream, then the
    layers' backward in reverse order, each against the oracle's gradients of
    that layer's own routing."""
    from moe_expert_routing_02_b300.layer import MoELayerStep
    c = W.config_by_name("tiny")
    st = M.MoEStats(c.L, c.E, c.window)
    step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, st, replicate=replicate, physical_replicas=physical)
    lgs = [torch.from_numpy(l).cuda() for l in W.make_layer_logits(c, 0)]
    xs = [W.make_x(c, 0, j, device="cuda") for j in range(c.L)]
    ws = [W.make_weights(c, j, device="cuda") for j in range(c.L)]
    if physical:
        ws = [MoELayerStep.replica_buffers(w) for w in ws]
    saved = []
    for j in range(c.L):
        out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda")
        step.run(0, j, lgs[j], xs[j], ws[j], out, save=True)
        saved.append(step.saved)
    M.moe_check()
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    for j in reversed(range(c.L)):
        dout = torch.randn((c.T, c.H), generator=g, device="cuda").to(torch.bfloat16)
        dx, dl, (dw1, _, dw2) = step.backward(saved[j], lgs[j], xs[j], ws[j], dout)
        M.moe_check()
        sv = saved[j]
        cs = dict(T=c.T, E=c.E, k=c.k, H=c.H, F=c.F, act=c.act, w=host(sv.w), go=host(sv.go), perm=host(sv.perm),
                  inv=host(sv.inv), ge=None if sv.ge is None else host(sv.ge), x=xs[j], dout=dout, y=sv.y,
                  w1=ws[j][0][:c.E], w3=None, w2=ws[j][2][:c.E])
        rdx, rdw, rdw1, _, rdw2 = _oracle(cs)
        assert rel_fro(O.bf16_to_f64(W.bf16_bits(dx)), rdx) <= GRAD_TOL, j
        assert rel_fro(host(dw1), rdw1) <= GRAD_TOL and rel_fro(host(dw2), rdw2) <= GRAD_TOL, j
        oi, _ = O.topk_gate(host(lgs[j]), c.k)
        assert np.array_equal(host(sv.idx), oi)
        rdl = O.router_backward(host(lgs[j]), oi, rdw)
        assert np.max(np.abs(host(dl) - rdl)) <= 1e-4 * max(1.0, float(np.max(np.abs(rdw)))), j


@pytest.mark.parametrize("T,E,k,H,F,act", [
    (100, 256, 8, 64, 64, "gelu"),      # the largest E and k, most experts with a few rows or none
    (77, 1, 1, 128, 64, "swiglu"),      # one expert: every row in one unit
    (1, 4, 2, 64, 128, "gelu"),         # one token
    (513, 3, 3, 64, 192, "swiglu"),     # k = E: every token chooses every expert
])
def test_edge_shapes(T, E, k, H, F, act):
    _check(_case(T, E, k, H, F, act, seed=T + E))


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_accumulate_adds_to_the_weight_gradients(act):
    """MOE_BWD_ACCUMULATE_WGRAD: a second call adds its weight gradients to the
    first's (the wgrad is deterministic, so the sum is exactly twice one
    call's); dx and dw are written, not added."""
    c = _case(300, 6, 2, 128, 192, act, seed=21, alpha=1.3, empty=(2,))
    one = _gpu(c)
    M.moe_check()
    out = tuple(None if t is None else t.clone() for t in one)
    got = M.moe_ffn_backward(c["x"], c["dout"], dev(c["w"]), c["y"], dev(c["perm"]), dev(c["inv"]), dev(c["go"]),
                             None, c["w1"], c["w3"], c["w2"], act, out=out, accumulate=True)
    M.moe_check()
    assert torch.equal(got[0], one[0]) and torch.equal(got[1], one[1])
    for a, b in zip(got[2:], one[2:]):
        if b is not None:
            assert torch.equal(a, 2 * b)
    with pytest.raises(ValueError):
        M.moe_ffn_backward(c["x"], c["dout"], dev(c["w"]), c["y"], dev(c["perm"]), dev(c["inv"]), dev(c["go"]),
                           None, c["w1"], c["w3"], c["w2"], act, accumulate=True)


def test_backward_in_a_cuda_graph():
    """The backward (eight launches, no host synchronisation) captured in a
    CUDA graph and replayed gives the eager results bit for bit."""
    c = _case(2048, 16, 2, 1024, 2048, "gelu", seed=22, alpha=1.2)
    eager = _gpu(c)
    lg = dev(c["logits"])
    idx = dev(c["idx"].astype(np.int32))
    dl_eager = M.moe_route_backward(lg, idx, eager[1])
    M.moe_check()
    T, k, E, H, F = c["T"], c["k"], c["E"], c["H"], c["F"]
    ws = torch.empty(M.moe_ffn_backward_workspace_bytes(T, k, E, H, F), dtype=torch.uint8, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    out = (torch.empty((T, H), dtype=torch.bfloat16, device="cuda"), torch.empty((T, k), **f32),
           torch.empty((E, H, F), **f32), None, torch.empty((E, F, H), **f32))
    dl = torch.empty((T, E), **f32)
    args = [dev(a) for a in (c["w"], c["perm"], c["inv"], c["go"])]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            M.moe_ffn_backward(c["x"], c["dout"], args[0], c["y"], args[1], args[2], args[3], None, c["w1"], None,
                               c["w2"], "gelu", workspace=ws, out=out)
            M.moe_route_backward(lg, idx, out[1], out=dl)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    M.moe_check()
    for a, b in zip(out, eager):
        if b is not None:
            assert torch.equal(a, b)
    assert torch.equal(dl, dl_eager)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_bf16_weight_gradients_are_the_fp32_ones_rounded(act):
    """MOE_BWD_WGRAD_BF16: every weight-gradient entry is the fp32 result
    rounded once to bf16 (round to nearest even), bit for bit; accumulation
    with bf16 output is refused."""
    c = _case(300, 6, 2, 128, 192, act, seed=23, alpha=1.3, empty=(4,))
    f = _gpu(c)
    b = M.moe_ffn_backward(c["x"], c["dout"], dev(c["w"]), c["y"], dev(c["perm"]), dev(c["inv"]), dev(c["go"]),
                           None, c["w1"], c["w3"], c["w2"], act, wgrad_bf16=True)
    M.moe_check()
    assert torch.equal(b[0], f[0]) and torch.equal(b[1], f[1])
    for gb, gf in zip(b[2:], f[2:]):
        if gf is not None:
            assert gb.dtype == torch.bfloat16 and torch.equal(gb, gf.to(torch.bfloat16))
    with pytest.raises(ValueError):
        M.moe_ffn_backward(c["x"], c["dout"], dev(c["w"]), c["y"], dev(c["perm"]), dev(c["inv"]), dev(c["go"]),
                           None, c["w1"], c["w3"], c["w2"], act, out=b, accumulate=True, wgrad_bf16=True)

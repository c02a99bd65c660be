"""moe_expert_ffn_gather (the FFN reading token rows in place through the
dispatch permutation) against moe_expert_ffn on the copied rows, bit for bit,
and against the oracle; the layer step with and without the gather."""
import dataclasses

import numpy as np
import pytest

from oracle import moe_oracle as O
from moe_expert_routing_02_b300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402
from moe_expert_routing_02_b300.layer import MoELayerStep  # noqa: E402

FFN_TOL = 2e-2
KERNELS = {"auto": 0, "single": 1, "pair": 2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()
    yield
    torch.cuda.synchronize()


@pytest.fixture
def ffn_kernel(request):
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, KERNELS[request.param])
    yield request.param
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, M.MOE_FFN_KERNEL_AUTO)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _both(x, idx, E, weights, act, rb=None, ge=None, thresh=64):
    """(y from the copied rows, y gathered, group offsets, xp)."""
    w1, w3, w2 = weights
    go, perm, inv, xp = M.moe_dispatch(x, idx, E, rb)
    y_copy = M.moe_expert_ffn(xp, go, ge, rb, w1, w3, w2, act, small_group_threshold=thresh)
    y_gat = M.moe_expert_ffn_gather(x, perm, idx.shape[1], go, ge, rb, w1, w3, w2, act,
                                    small_group_threshold=thresh)
    M.moe_check()
    return y_copy, y_gat, go, xp


@pytest.mark.parametrize("name,ffn_kernel", [("tiny", "single"), ("tiny", "pair"), ("moe_gpt_stream", "auto"),
                                              ("moe_gpt_stream", "single"), ("mixtral_layer", "auto"),
                                              ("deepseekv2_layer", "auto"), ("deepseekv2_layer", "pair"),
                                              ("dbrx_replicated_layer", "auto")],
                         indirect=["ffn_kernel"])
def test_gather_bit_identical_and_oracle(name, ffn_kernel):
    c = W.config_by_name(name)
    lg = W.make_layer_logits(c, 0, layers=1)[0]
    idx, _ = O.topk_gate(lg, c.k)
    rb = ge = None
    if c.replicate:
        _, rb, ge = O.replicate(O.histogram(idx, c.E), idx.size)
    x = W.make_x(c, 0, 0, device="cuda")
    weights = W.make_weights(c, 0, device="cuda")
    y_copy, y_gat, go, xp = _both(x, dev(idx), c.E, weights, c.act, None if rb is None else dev(rb),
                                  None if ge is None else dev(ge))
    assert torch.equal(y_copy, y_gat)
    # sampled slots (each group's first and last row, plus random ones) against the oracle
    G = 2 * c.E if c.replicate else c.E
    ogo = host(go)[:G + 1]
    nonempty = [g for g in range(G) if ogo[g + 1] > ogo[g]]
    rng = np.random.default_rng(3)
    slots = np.unique(np.concatenate([[ogo[g] for g in nonempty], [ogo[g + 1] - 1 for g in nonempty],
                                      rng.integers(0, idx.size, 128)]))
    w1, w3, w2 = weights
    ref = O.expert_ffn(W.bf16_bits(xp), ogo, ge, W.bf16_bits(w1), None if w3 is None else W.bf16_bits(w3),
                       W.bf16_bits(w2), c.act, slots=slots)
    assert rel_fro(O.bf16_to_f64(W.bf16_bits(y_gat)[slots]), ref) <= FFN_TOL
    del y_copy, y_gat, xp, weights
    torch.cuda.empty_cache()


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("thresh", [0, 64, 1 << 30])
@pytest.mark.parametrize("ffn_kernel", ["single", "pair"], indirect=True)
def test_gather_ragged_groups_all_paths(thresh, act, ffn_kernel):
    """Groups of 0..300 rows (partial tiles, rows past the last group) through
    the grouped and the small-batch kernels, k = 2 so that the source row is
    perm // k, checked bit for bit and per group against the oracle."""
    sizes = [0, 1, 3, 15, 16, 17, 63, 64, 65, 127, 129, 200, 301]
    E = len(sizes)
    c = dataclasses.replace(W.config_by_name("tiny"), name="gather-ragged", E=E, k=2, H=192, F=320, act=act)
    # each token picks two distinct experts; the expert sizes follow `sizes` (k * T rows in all)
    flat = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)])
    if flat.size % 2:
        flat = np.concatenate([flat, [E - 1]]).astype(np.int32)
    # sorted by expert, row i pairs with row i + n/2: no expert holds half the
    # rows, so the two always differ; then shuffle tokens and the order within each
    n = flat.size
    assert np.bincount(flat).max() < n // 2
    pairs = np.stack([flat[: n // 2], flat[n // 2:]], axis=1)
    rng = np.random.default_rng(5)
    pairs = pairs[rng.permutation(n // 2)]
    swap = rng.integers(0, 2, n // 2).astype(bool)
    pairs[swap] = pairs[swap][:, ::-1]
    assert (pairs[:, 0] != pairs[:, 1]).all()
    idx = pairs.astype(np.int32)
    x = W.make_x(c, 0, 0, device="cuda", T=idx.shape[0])
    weights = W.make_weights(c, 0, device="cuda")
    y_copy, y_gat, go, xp = _both(x, dev(idx), E, weights, act, thresh=thresh)
    assert torch.equal(y_copy, y_gat)
    w1, w3, w2 = weights
    gof = host(go)[:E + 1]
    ref = O.expert_ffn(W.bf16_bits(xp), gof, None, W.bf16_bits(w1), None if w3 is None else W.bf16_bits(w3),
                       W.bf16_bits(w2), act)
    got = O.bf16_to_f64(W.bf16_bits(y_gat))
    for g in range(E):
        lo, hi = gof[g], gof[g + 1]
        if hi > lo:
            assert rel_fro(got[lo:hi], ref[lo:hi]) <= FFN_TOL, g


def test_gather_empty_batch_and_invalid_permutation():
    c = W.config_by_name("tiny")
    w1, w3, w2 = W.make_weights(c, 0, device="cuda")
    go = torch.zeros(c.E + 1, dtype=torch.int32, device="cuda")
    x0 = torch.empty((0, c.H), dtype=torch.bfloat16, device="cuda")
    y0 = M.moe_expert_ffn_gather(x0, torch.empty(0, dtype=torch.int32, device="cuda"), c.k, go, None, None,
                                 w1, w3, w2, c.act)
    assert y0.shape == (0, c.H)
    M.moe_check()
    # a permutation entry past T*k is invalid device data: flagged, row 0 read instead, no fault
    lg = W.make_layer_logits(c, 0, layers=1)[0]
    idx, _ = O.topk_gate(lg, c.k)
    x = W.make_x(c, 0, 0, device="cuda")
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), c.E)
    bad = perm.clone()
    bad[5] = idx.size + 7
    M.moe_expert_ffn_gather(x, bad, c.k, go, None, None, w1, w3, w2, c.act)
    with pytest.raises(M.MoEError) as ei:
        M.moe_check()
    assert ei.value.status == M.MOE_ERR_DEVICE
    # the context is still usable and a valid call is clean again
    y = M.moe_expert_ffn_gather(x, perm, c.k, go, None, None, w1, w3, w2, c.act)
    M.moe_check()
    assert torch.equal(y, M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, c.act))


@pytest.mark.parametrize("name", ["tiny", "moe_gpt_stream"])
def test_layer_step_gather_and_copy_identical(name):
    """Two iterations of the layer stream with the four front/FFN variants
    (fused or separate front, gathered or copied rows): identical outputs."""
    c = W.config_by_name(name)
    L = min(c.L, 3)
    weights = [W.make_weights(c, j, device="cuda") for j in range(L)]
    outs = {}
    for fused in (True, False):
        for gather in (True, False):
            st = M.MoEStats(L, c.E, c.window)
            step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, stats=st, replicate=True, fused=fused,
                                gather=gather)
            res = []
            for it in range(2):
                lgs = W.make_layer_logits(c, it, layers=L)
                for j in range(L):
                    out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda")
                    step.run(it, j, dev(lgs[j]), W.make_x(c, it, j, device="cuda"), weights[j], out)
                    res.append(out)
            M.moe_check()
            outs[(fused, gather)] = res
    base = outs[(False, False)]
    for key, res in outs.items():
        for a, b in zip(res, base):
            assert torch.equal(a, b), key


def test_layer_step_prediction_driven_replication_same_output():
    """Replicas from the previous layer's prediction (with and without a copies
    budget, fused and separate calls) leave the layer output unchanged."""
    c = W.config_by_name("moe_gpt_stream")
    L = 3
    weights = [W.make_weights(c, j, device="cuda") for j in range(L)]
    outs = {}
    for key, kw in {"hist": dict(), "pred": dict(replicate_from="prediction"),
                    "pred_budget": dict(replicate_from="prediction", budget=1),
                    "pred_unfused": dict(replicate_from="prediction", fused=False)}.items():
        st = M.MoEStats(L, c.E, c.window)
        step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, stats=st, replicate=True, **kw)
        res = []
        for it in range(2):
            lgs = W.make_layer_logits(c, it, layers=L)
            for j in range(L):
                out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda")
                step.run(it, j, dev(lgs[j]), W.make_x(c, it, j, device="cuda"), weights[j], out)
                res.append(out)
        M.moe_check()
        outs[key] = res
    for key, res in outs.items():
        for a, b in zip(res, outs["hist"]):
            assert torch.equal(a, b), key


@pytest.mark.parametrize("chunks", [2, 4])
def test_chunked_pipeline_same_output(chunks):
    """EPS-MoE pipeline over token chunks on two streams: bit-identical to the
    one-shot layer step, statistics included."""
    from moe_expert_routing_02_b300.layer import ChunkedLayerStep
    c = W.config_by_name("moe_gpt_stream")
    L = 2
    weights = [W.make_weights(c, j, device="cuda") for j in range(L)]
    st_a = M.MoEStats(L, c.E, c.window)
    st_b = M.MoEStats(L, c.E, c.window)
    a = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, stats=st_a, replicate=True)
    b = ChunkedLayerStep(c.T, c.E, c.k, c.H, c.F, c.act, st_b, chunks=chunks)
    for it in (60, 61):
        lgs = W.make_layer_logits(c, it, layers=L)
        for j in range(L):
            x = W.make_x(c, it, j, device="cuda")
            oa = torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda")
            ob = torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda")
            a.run(it, j, dev(lgs[j]), x, weights[j], oa)
            b.run(it, j, dev(lgs[j]), x, weights[j], ob)
            torch.cuda.synchronize()
            assert torch.equal(oa, ob), (it, j)
            assert torch.equal(a.hist, b.hist) and torch.equal(a.rep_base, b.rep_base)
    M.moe_check()
    sa, sb = st_a.export_state(), st_b.export_state()
    assert sa == sb

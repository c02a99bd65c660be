"""Physical replica copies (moe_replicate_weights) and the FFN over weight
slots (moe_expert_ffn_slots): the copies equal their experts, the slot map
follows the documented layout, and the output equals the aliasing FFN's bit
for bit."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from moe_expert_routing_02_b300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402
from moe_expert_routing_02_b300.layer import MoELayerStep  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def _slots(w, rb):
    E = w.shape[0]
    w_all = torch.empty((2 * E - 1,) + tuple(w.shape[1:]), dtype=w.dtype, device=w.device)
    w_all[:E].copy_(w)
    gs = M.moe_replicate_weights(rb, w_all)
    return w_all, gs


@pytest.mark.parametrize("name", ["tiny", "moe_gpt_stream", "dbrx_replicated_layer"])
def test_physical_replicas_bit_identical(name):
    c = W.config_by_name(name)
    it = 60 if name == "moe_gpt_stream" else 0   # the stream's skew ramps up over 50 iterations
    lg = W.make_layer_logits(c, it, layers=1)[0]
    idx, _ = O.topk_gate(lg, c.k)
    copies, rb, ge = O.replicate(O.histogram(idx, c.E), idx.size)
    assert int(copies.sum()) > 0
    x = W.make_x(c, 0, 0, device="cuda")
    w1, w3, w2 = W.make_weights(c, 0, device="cuda")
    rbd, ged = dev(rb), dev(ge)
    w1a, gs = _slots(w1, rbd)
    w2a, gs2 = _slots(w2, rbd)
    w3a = None
    if w3 is not None:
        w3a, _ = _slots(w3, rbd)
    M.moe_check()
    # slot map: documented layout
    gsh = host(gs)
    E = c.E
    for e in range(E):
        for q in range(rb[e + 1] - rb[e]):
            want = e if q == 0 else E + (rb[e] - e) + q - 1
            assert gsh[rb[e] + q] == want
    assert (gsh[rb[E]:] == -1).all() and np.array_equal(gsh, host(gs2))
    # every used slot holds its expert's weights
    for g in range(int(rb[E])):
        assert torch.equal(w1a[int(gsh[g])], w1[int(ge[g])])
        assert torch.equal(w2a[int(gsh[g])], w2[int(ge[g])])
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), E, rbd)
    y_alias = M.moe_expert_ffn(xp, go, ged, rbd, w1, w3, w2, c.act)
    y_phys = M.moe_expert_ffn_slots(xp, go, gs, w1a, w3a, w2a, c.act)
    M.moe_check()
    assert torch.equal(y_alias, y_phys)
    del w1a, w2a, w3a
    torch.cuda.empty_cache()


def test_replicate_weights_without_replicas_and_bad_args():
    E = 8
    rb = torch.arange(E + 1, dtype=torch.int32, device="cuda")      # no replicas
    w = torch.randn((2 * E - 1, 64, 64), device="cuda").to(torch.bfloat16)
    before = w.clone()
    gs = M.moe_replicate_weights(rb, w)
    M.moe_check()
    assert torch.equal(w, before)
    assert host(gs).tolist() == list(range(E)) + [-1] * E
    with pytest.raises(M.MoEError):   # rows * cols not a multiple of 8
        M.lib()
        import ctypes
        M._check(M.lib().moe_replicate_weights(ctypes.c_void_p(rb.data_ptr()), E, ctypes.c_void_p(w.data_ptr()),
                                               3, 3, None, None), "moe_replicate_weights")


def test_layer_step_physical_replicas_same_output():
    c = W.config_by_name("moe_gpt_stream")
    L = 2
    weights = [W.make_weights(c, j, device="cuda") for j in range(L)]
    outs = {}
    for phys in (False, True):
        st = M.MoEStats(L, c.E, c.window)
        step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, stats=st, replicate=True, physical_replicas=phys)
        res = []
        for it in (60, 61):   # skewed iterations: hot experts get replicas
            lgs = W.make_layer_logits(c, it, layers=L)
            for j in range(L):
                out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda")
                wj = MoELayerStep.replica_buffers(weights[j]) if phys else weights[j]
                step.run(it, j, dev(lgs[j]), W.make_x(c, it, j, device="cuda"), wj, out)
                res.append(out)
        M.moe_check()
        outs[phys] = res
    for a, b in zip(outs[False], outs[True]):
        assert torch.equal(a, b)

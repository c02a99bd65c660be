"""Host logic of the layer orchestrator (layer.MoELayerStep) without a GPU:
the library's launch entry points are replaced by a recorder that keeps each
call's name and arguments, and the CUDA-tensor check is relaxed to accept CPU
tensors.  Checked: the order of the calls per layer (fused front or the
seven separate calls), that layer j reads layer j-1's choices from the other
half of the ping-pong buffers, that prediction-driven replication hands layer
j the p_next written at layer j-1, that the last layer asks for no next-layer
prediction, and the calls of the backward."""
import ctypes

import pytest

torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402
from moe_expert_routing_02_b300 import _build, layer as LY  # noqa: E402
from moe_expert_routing_02_b300 import workloads as W  # noqa: E402

HOST_ONLY = {"moe_workspace_bytes", "moe_ffn_backward_workspace_bytes", "moe_ffn_launches", "moe_status_string",
             "moe_last_error"}

# argument positions in the C signatures (include/moe.h)
FRONT = dict(idx_prev=10, rep_share=15, idx=17, w=18, hist=19, p_seq=20, cond=21, p_next=22, rep_base=24,
             group_expert=25, go=26, perm=27, inv=28, xp=29)
FFN = dict(xp=0, go=1, group_expert=2, rep_base=3, y=13)
COMBINE = dict(y=0, inv=1, w=2, out=6)


@pytest.fixture()
def calls(monkeypatch):
    _build.build()
    real = M.lib()
    rec = []

    class Recorder:
        def __getattr__(self, name):
            if name in HOST_ONLY:
                return getattr(real, name)

            def launch(*args):
                rec.append((name, [a.value if isinstance(a, ctypes.c_void_p) else a for a in args]))
                return M.MOE_OK
            return launch

    def dev_any(t, dtype, name, ndim=None):
        if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_contiguous():
            raise ValueError(name)
        if ndim is not None and t.dim() != ndim:
            raise ValueError(name)
        return t

    monkeypatch.setattr(M, "lib", lambda: Recorder())
    monkeypatch.setattr(M, "_dev", dev_any)
    monkeypatch.setattr(M, "_stream", lambda s=None: ctypes.c_void_p(0))
    return rec


class _Stats:
    def __init__(self, L, E, window=10):
        self.L, self.E, self.window = L, E, window
        self.handle = ctypes.c_void_p(0)


def _run(c, step, save=False, predict=True):
    outs = []
    for j in range(c.L):
        lg = torch.from_numpy(W.make_layer_logits(c, 0)[j])
        x = W.make_x(c, 0, j)
        ws = W.make_weights(c, j)
        out = torch.empty((c.T, c.H), dtype=torch.bfloat16)
        step.run(3, j, lg, x, ws, out, save=save, predict=predict)
        outs.append((lg, x, ws, out, step.saved if save else None))
    return outs


def _cfg(L=3):
    import dataclasses
    return dataclasses.replace(W.config_by_name("moe_gpt_stream"), T=256, L=L)


def test_fused_layers_chain_their_buffers(calls):
    c = _cfg()
    step = LY.MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, _Stats(c.L, c.E), device="cpu",
                           replicate_from="prediction")
    _run(c, step)
    names = [n for n, _ in calls]
    assert names == ["moe_layer_front", "moe_expert_ffn", "moe_combine"] * c.L
    fronts = [a for n, a in calls if n == "moe_layer_front"]
    ffns = [a for n, a in calls if n == "moe_expert_ffn"]
    combs = [a for n, a in calls if n == "moe_combine"]
    for j, f in enumerate(fronts):
        assert f[9] == j and f[8] == 3                       # layer, iteration
        if j == 0:
            assert f[FRONT["idx_prev"]] is None and f[FRONT["rep_share"]] is None
        else:
            prev = fronts[j - 1]
            assert f[FRONT["idx_prev"]] == prev[FRONT["idx"]]       # the previous layer's choices
            assert f[FRONT["idx"]] != prev[FRONT["idx"]]            # written into the other buffer
            assert f[FRONT["rep_share"]] == prev[FRONT["p_next"]]   # the prediction made at layer j-1
            assert f[FRONT["p_next"]] != prev[FRONT["p_next"]] or j == c.L - 1
        last = j == c.L - 1
        assert (f[FRONT["cond"]] is None) == last and (f[FRONT["p_next"]] is None) == last
        assert f[FRONT["p_seq"]] is not None
        # the FFN reads what the front wrote, the combine what the FFN wrote
        assert ffns[j][FFN["xp"]] == f[FRONT["xp"]] and ffns[j][FFN["go"]] == f[FRONT["go"]]
        assert ffns[j][FFN["rep_base"]] == f[FRONT["rep_base"]]
        assert ffns[j][FFN["group_expert"]] == f[FRONT["group_expert"]]
        assert combs[j][COMBINE["y"]] == ffns[j][FFN["y"]] and combs[j][COMBINE["inv"]] == f[FRONT["inv"]]
        assert combs[j][COMBINE["w"]] == f[FRONT["w"]]


def test_separate_calls_in_the_pages_order(calls):
    c = _cfg()
    step = LY.MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, _Stats(c.L, c.E), device="cpu", fused=False)
    _run(c, step)
    seven = ["moe_route", "moe_stats_update", "moe_predict", "moe_replicate", "moe_dispatch", "moe_expert_ffn",
             "moe_combine"]
    last = [n for n in seven if n != "moe_predict"]       # no next layer to predict
    assert [n for n, _ in calls] == seven * (c.L - 1) + last
    # the statistics update of layer j gets layer j-1's choices
    upd = [a for n, a in calls if n == "moe_stats_update"]
    route = [a for n, a in calls if n == "moe_route"]
    assert upd[0][4] is None
    for j in range(1, c.L):
        assert upd[j][3] == route[j][5] and upd[j][4] == route[j - 1][5]


def test_gather_and_fused_combine_variants(calls):
    c = _cfg(2)
    step = LY.MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, _Stats(c.L, c.E), device="cpu", gather=True)
    _run(c, step)
    assert [n for n, _ in calls] == ["moe_layer_front", "moe_expert_ffn_gather", "moe_combine"] * c.L
    fronts = [a for n, a in calls if n == "moe_layer_front"]
    assert all(f[1] is None and f[FRONT["xp"]] is None for f in fronts)   # no row copy
    calls.clear()
    step = LY.MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, _Stats(c.L, c.E), device="cpu", fuse_combine=True)
    _run(c, step)
    assert [n for n, _ in calls] == ["moe_layer_front", "moe_expert_ffn_combine"] * c.L
    with pytest.raises(ValueError):
        _run(c, step, save=True)


def test_backward_uses_the_saved_routing(calls):
    c = _cfg(2)
    step = LY.MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, _Stats(c.L, c.E), device="cpu")
    runs = _run(c, step, save=True)
    calls.clear()
    lg, x, ws, out, saved = runs[0]
    assert saved.perm.data_ptr() != step.perm.data_ptr()       # a copy, not the live buffer
    dout = torch.zeros((c.T, c.H), dtype=torch.bfloat16)
    step.backward(saved, lg, x, ws, dout)
    assert [n for n, _ in calls] == ["moe_ffn_backward", "moe_route_backward"]
    bwd = calls[0][1]
    assert bwd[4] == saved.perm.data_ptr() and bwd[5] == saved.inv.data_ptr() and bwd[3] == saved.y.data_ptr()
    assert calls[1][1][1] == saved.idx.data_ptr()


def test_prediction_driven_replication_needs_the_prediction():
    c = _cfg(2)
    with pytest.raises(ValueError):
        LY.MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, None, device="cpu", replicate_from="prediction")
    with pytest.raises(ValueError):
        LY.MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, _Stats(c.L, c.E), device="cpu", replicate=False,
                        replicate_from="prediction")
    with pytest.raises(ValueError):     # replication without the statistics that write the histogram
        LY.MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, None, device="cpu")
    LY.MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, None, device="cpu", replicate=False)


def test_layer_without_statistics_makes_route_dispatch_ffn_combine(calls):
    c = _cfg(2)
    step = LY.MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, None, device="cpu", replicate=False)
    _run(c, step)
    assert [n for n, _ in calls] == ["moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine"] * c.L
    assert all(a[6] is None for n, a in calls if n == "moe_dispatch")      # no replica table

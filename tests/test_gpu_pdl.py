"""Programmatic dependent launch (MOE_OPT_PDL) changes only how the layer's
kernels are launched: outputs, window state and replica tables are
bit-identical with it on and off, launched eagerly and replayed from a CUDA
graph."""
import dataclasses

import numpy as np
import pytest

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
    yield
    M.moe_set_option(M.MOE_OPT_PDL, 1)


def _run(c, pdl: int, graph: bool, iters: int = 2):
    M.moe_set_option(M.MOE_OPT_PDL, pdl)
    st = M.MoEStats(c.L, c.E, c.window)
    step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, st)
    lgs = [[torch.from_numpy(l).cuda() for l in W.make_layer_logits(c, it)] for it in range(iters)]
    xs = [W.make_x(c, 0, j, device="cuda") for j in range(c.L)]
    ws = [W.make_weights(c, j, device="cuda") for j in range(c.L)]
    outs = [torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda") for _ in range(c.L)]
    res = []
    for it in range(iters):
        def body():
            for j in range(c.L):
                step.run(it, j, lgs[it][j], xs[j], ws[j], outs[j])
        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    body()
            torch.cuda.current_stream().wait_stream(s)
            g.replay()
        else:
            body()
        torch.cuda.synchronize()
        M.moe_check()
        res.append([o.clone() for o in outs] + [step.rep_base.clone(), step.hist.clone()])
    res.append([torch.from_numpy(np.frombuffer(st.export_state(), dtype=np.uint8).copy())])
    return res


@pytest.mark.parametrize("name,T", [("tiny", None), ("moe_gpt_stream", 2048)])
def test_pdl_on_off_identical(name, T):
    c = W.config_by_name(name)
    c = dataclasses.replace(c, L=3, **({"T": T} if T else {}))
    ref = _run(c, 0, graph=False)
    for pdl, graph in ((1, False), (1, True), (0, True)):
        got = _run(c, pdl, graph)
        for a, b in zip(ref, got):
            for x, y in zip(a, b):
                assert torch.equal(x.cpu(), y.cpu()), (pdl, graph)


def test_pdl_option_roundtrip():
    for v in (0, 1):
        M.moe_set_option(M.MOE_OPT_PDL, v)
        assert M.moe_get_option(M.MOE_OPT_PDL) == v
    with pytest.raises(M.MoEError):
        M.moe_set_option(M.MOE_OPT_PDL, 2)

"""The combine fused into the FFN's second GEMM (moe_expert_ffn_combine)
against the separate calls and the oracle.  It sums w * (fp32 GEMM2 result)
without rounding Y to bf16 first, so it differs from moe_expert_ffn +
moe_combine by about one bf16 rounding: held to 1e-2 relative Frobenius
against them and to the FFN's 2e-2 against the oracle's layer output; for
k <= 2 it is bit-reproducible."""
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def b64(t):
    return O.bf16_to_f64(W.bf16_bits(t))


@pytest.mark.parametrize("T,E,k,H,F,act,alpha,replicate", [
    (256, 8, 2, 64, 128, "gelu", 1.0, True),           # small-batch experts too
    (2048, 16, 2, 1024, 2048, "gelu", 1.2, True),      # moe_gpt_stream's shapes: the CTA-pair kernels
    (1024, 8, 2, 512, 1024, "swiglu", 1.1, False),
    (512, 64, 6, 256, 192, "swiglu", 1.1, False),      # k = 6, most experts small
])
def test_fused_combine_matches_separate_calls_and_oracle(T, E, k, H, F, act, alpha, replicate):
    rng_key = (T, E, k)
    lg = W.make_logits(T, E, alpha, seed_key=rng_key)
    idx, wts = O.topk_gate(lg, k)
    rb = ge = None
    if replicate:
        _, rb, ge = O.replicate(O.histogram(idx, E), idx.size)
    g = torch.Generator(device="cuda")
    g.manual_seed(T + E)
    x = torch.randn((T, H), generator=g, device="cuda").to(torch.bfloat16)
    mk = lambda shape: (torch.randn(shape, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    w1, w2 = mk((E, H, F)), mk((E, F, H))
    w3 = mk((E, H, F)) if act == "swiglu" else None
    rbd, ged = (None, None) if rb is None else (dev(rb), dev(ge))
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), E, rbd)
    wd = dev(wts.astype(np.float32))
    y = M.moe_expert_ffn(xp, go, ged, rbd, w1, w3, w2, act)
    ref_sep = M.moe_combine(y, inv, wd)
    fused = M.moe_expert_ffn_combine(xp, go, ged, rbd, perm, wd, w1, w3, w2, act)
    M.moe_check()
    assert rel_fro(b64(fused), b64(ref_sep)) <= 1e-2
    # the oracle's layer output from the same inputs
    slots = np.arange(T * k)
    yo = O.expert_ffn(W.bf16_bits(xp), M_host(go), None if ge is None else ge, W.bf16_bits(w1),
                      None if w3 is None else W.bf16_bits(w3), W.bf16_bits(w2), act, slots=slots)
    out_o = O.combine(yo, M_host(inv), wts.astype(np.float32))
    assert rel_fro(b64(fused), out_o) <= 2e-2
    if k <= 2:
        again = M.moe_expert_ffn_combine(xp, go, ged, rbd, perm, wd, w1, w3, w2, act)
        M.moe_check()
        assert torch.equal(again, fused)


def M_host(t):
    return t.detach().cpu().numpy()


def test_layer_step_fused_combine():
    from moe_expert_routing_02_b300.layer import MoELayerStep
    c = W.config_by_name("tiny")
    outs = []
    for fuse in (False, True):
        st = M.MoEStats(c.L, c.E, c.window)
        step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, st, fuse_combine=fuse)
        lgs = [torch.from_numpy(l).cuda() for l in W.make_layer_logits(c, 0)]
        res = []
        for j in range(c.L):
            out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda")
            step.run(0, j, lgs[j], W.make_x(c, 0, j, device="cuda"), W.make_weights(c, j, device="cuda"), out)
            res.append(b64(out))
        M.moe_check()
        outs.append(res)
    for a, b in zip(*outs):
        assert rel_fro(b, a) <= 1e-2

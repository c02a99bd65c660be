"""The SM split of an expert-FFN call between the small-batch kernel and the
grouped kernels (MOE_OPT_FFN_SMALL_SMS; EPS-MoE review, "GroupGemm vs
DenseGemm": experts with few tokens take a separate path).

Every split gives the oracle's output within the FFN bar, group by group;
the rows of experts the grouped kernel serves are bit-identical whatever the
split (same kernel, same tiles), and with the small-batch path off (0) every
row comes from the grouped kernel.  Covered for the single-CTA, the CTA-pair
and the fused kernels, GeLU and SwiGLU, with a layer that has experts below
the 64-row threshold, ones just above it, and large ones."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from moe_expert_routing_02_b300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402

FFN_TOL = 2e-2
KERNELS = {"single": 1, "pair": 2, "fused": 3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()
    yield
    M.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, 0)
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, M.MOE_FFN_KERNEL_AUTO)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("kernel", ["single", "pair", "fused"])
@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_split_matches_oracle_and_grouped_rows_are_stable(kernel, act):
    import dataclasses
    sizes = [0, 1, 7, 16, 40, 63, 64, 65, 200, 700, 1500, 3, 30, 900, 50, 2]
    E = len(sizes)
    c = dataclasses.replace(W.config_by_name("tiny"), name="split", E=E, k=1, H=256, F=384, act=act)
    idx = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)])
    np.random.default_rng(5).shuffle(idx)
    idx = idx.reshape(-1, 1)
    x = W.make_x(c, 0, 0, device="cuda", T=idx.shape[0])
    w1, w3, w2 = W.make_weights(c, 0, device="cuda")
    go, perm, inv, xp = M.moe_dispatch(x, torch.from_numpy(idx).cuda(), E)
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, KERNELS[kernel])
    ys = {}
    for sms in (0, 2, 16, 60, -1):
        M.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, sms)
        ys[sms] = M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, act, small_group_threshold=64)
        M.moe_check()
    M.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, 0)
    gof = go.cpu().numpy()
    ref = O.expert_ffn(W.bf16_bits(xp), gof[:E + 1], None, W.bf16_bits(w1),
                       None if w3 is None else W.bf16_bits(w3), W.bf16_bits(w2), act)
    for sms, y in ys.items():
        got = O.bf16_to_f64(W.bf16_bits(y))
        for e in range(E):
            lo, hi = gof[e], gof[e + 1]
            if hi > lo:
                assert _rel(got[lo:hi], ref[lo:hi]) <= FFN_TOL, (sms, e, sizes[e])
        # experts at or above the threshold always take the grouped kernel
        for e in range(E):
            lo, hi = gof[e], gof[e + 1]
            if sizes[e] >= 64:
                assert torch.equal(y[lo:hi], ys[0][lo:hi]), (sms, e)

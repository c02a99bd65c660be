"""The fused FFN kernel (both GEMMs in one launch, tiles interleaved, per-block
completion counters) against the two-launch CTA-pair kernel, bit for bit, and
against the oracle."""
import dataclasses
import time

import numpy as np
import pytest

from oracle import moe_oracle as O
from moe_expert_routing_02_b300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402

FFN_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()
    yield
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, M.MOE_FFN_KERNEL_AUTO)
    torch.cuda.synchronize()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _run(kernel, xp, go, ge, rb, weights, act, thresh=64):
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, kernel)
    try:
        w1, w3, w2 = weights
        y = M.moe_expert_ffn(xp, go, ge, rb, w1, w3, w2, act, small_group_threshold=thresh)
        M.moe_check()
        return y
    finally:
        M.moe_set_option(M.MOE_OPT_FFN_KERNEL, M.MOE_FFN_KERNEL_AUTO)


@pytest.mark.parametrize("name", [c.name for c in W.CONFIGS])
def test_fused_bit_identical_to_two_launches_and_oracle(name):
    c = W.config_by_name(name)
    lg = W.make_layer_logits(c, 0, layers=1)[0]
    idx, _ = O.topk_gate(lg, c.k)
    rb = ge = None
    if c.replicate:
        _, rb, ge = O.replicate(O.histogram(idx, c.E), idx.size)
    x = W.make_x(c, 0, 0, device="cuda")
    weights = W.make_weights(c, 0, device="cuda")
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), c.E, None if rb is None else dev(rb))
    rbd, ged = (None, None) if rb is None else (dev(rb), dev(ge))
    y_pair = _run(M.MOE_FFN_KERNEL_PAIR, xp, go, ged, rbd, weights, c.act)
    y_fused = _run(M.MOE_FFN_KERNEL_FUSED, xp, go, ged, rbd, weights, c.act)
    assert torch.equal(y_pair, y_fused)
    G = 2 * c.E if c.replicate else c.E
    ogo = host(go)[:G + 1]
    nonempty = [g for g in range(G) if ogo[g + 1] > ogo[g]]
    rng = np.random.default_rng(7)
    slots = np.unique(np.concatenate([[ogo[g] for g in nonempty], [ogo[g + 1] - 1 for g in nonempty],
                                      rng.integers(0, idx.size, 128)]))
    w1, w3, w2 = weights
    ref = O.expert_ffn(W.bf16_bits(xp), ogo, ge, W.bf16_bits(w1), None if w3 is None else W.bf16_bits(w3),
                       W.bf16_bits(w2), c.act, slots=slots)
    assert rel_fro(O.bf16_to_f64(W.bf16_bits(y_fused)[slots]), ref) <= FFN_TOL
    del y_pair, y_fused, xp, weights
    torch.cuda.empty_cache()


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("thresh", [0, 64])
def test_fused_ragged_groups(act, thresh):
    """Groups of 0..1500 rows (one-block units, partial blocks, units of many
    blocks, experts below the small-batch threshold) and F, H not multiples of
    the 256-column tile: fused == two launches, and per group against the oracle."""
    sizes = [0, 1, 63, 64, 255, 256, 257, 700, 1500, 129, 511, 3]
    E = len(sizes)
    c = dataclasses.replace(W.config_by_name("tiny"), name="fused-ragged", E=E, k=1, H=192, F=320, act=act)
    idx = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)])
    np.random.default_rng(2).shuffle(idx)
    idx = idx.reshape(-1, 1)
    x = W.make_x(c, 0, 0, device="cuda", T=idx.shape[0])
    weights = W.make_weights(c, 0, device="cuda")
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), E)
    y_pair = _run(M.MOE_FFN_KERNEL_PAIR, xp, go, None, None, weights, act, thresh)
    y_fused = _run(M.MOE_FFN_KERNEL_FUSED, xp, go, None, None, weights, act, thresh)
    assert torch.equal(y_pair, y_fused)
    w1, w3, w2 = weights
    gof = host(go)[:E + 1]
    ref = O.expert_ffn(W.bf16_bits(xp), gof, None, W.bf16_bits(w1), None if w3 is None else W.bf16_bits(w3),
                       W.bf16_bits(w2), act)
    got = O.bf16_to_f64(W.bf16_bits(y_fused))
    for g in range(E):
        lo, hi = gof[g], gof[g + 1]
        if hi > lo:
            assert rel_fro(got[lo:hi], ref[lo:hi]) <= FFN_TOL, g


def test_fused_bounded_wait_timeout_is_reported_and_context_survives():
    """Self-test: pair 0 withholds its first accumulator signal; the fused
    kernel's waits (accumulator and block counters) run out, the kernel
    returns, moe_check reports MOE_ERR_TIMEOUT, and the next call is correct."""
    c = W.config_by_name("moe_gpt_stream")
    T = 4096
    lg = W.make_layer_logits(c, 0, T=T, layers=1)[0]
    idx, _ = O.topk_gate(lg, c.k)
    x = W.make_x(c, 0, 0, device="cuda", T=T)
    weights = W.make_weights(c, 0, device="cuda")
    go, perm, inv, xp = M.moe_dispatch(x, dev(idx), c.E)
    y_ref = _run(M.MOE_FFN_KERNEL_PAIR, xp, go, None, None, weights, c.act)
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, M.MOE_FFN_KERNEL_FUSED)
    try:
        M.moe_set_option(M.MOE_OPT_FFN_TIMEOUT_SELFTEST, 1)
        w1, w3, w2 = weights
        t0 = time.time()
        M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, c.act)
        with pytest.raises(M.MoEError) as ei:
            M.moe_check()
        assert ei.value.status == M.MOE_ERR_TIMEOUT
        assert time.time() - t0 < 60
        y = M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, c.act)
        M.moe_check()
        assert torch.equal(y, y_ref)
    finally:
        M.moe_set_option(M.MOE_OPT_FFN_KERNEL, M.MOE_FFN_KERNEL_AUTO)
        M.moe_set_option(M.MOE_OPT_FFN_TIMEOUT_SELFTEST, 0)

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

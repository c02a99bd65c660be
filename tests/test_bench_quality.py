"""The benchmark's prediction-quality measures agree with the oracle's
definitions (CPU only)."""
import numpy as np

from oracle import moe_oracle as O
import bench


def test_top_overlap_matches_oracle():
    rng = np.random.default_rng(0)
    for _ in range(200):
        E = int(rng.integers(5, 40))
        p = rng.dirichlet(np.ones(E)).astype(np.float32)
        if rng.random() < 0.3:
            p[rng.integers(0, E, 3)] = p[0]          # ties in the prediction
        load = rng.integers(0, 5, E)                 # many ties in the loads
        assert bench._top_overlap(p, load) == O.top_overlap(p, load, 5)


def test_max_group_load():
    load = np.array([10, 7, 0, 3])
    assert bench._max_group_load(load, np.array([0, 0, 0, 0])) == 10
    assert bench._max_group_load(load, np.array([1, 0, 0, 0])) == 7
    assert bench._max_group_load(load, np.array([2, 1, 0, 0])) == 4


def test_routing_summary_from_the_layer_buffers():
    import types
    import torch
    from moe_expert_routing_02_b300 import workloads as W
    c = W.config_by_name("tiny")              # T=256, E=8, k=2: target A/E = 64 rows
    hist = torch.tensor([200, 150, 60, 40, 30, 20, 12, 0], dtype=torch.int32)
    copies = [3, 2, 0, 0, 0, 0, 0, 0]
    rep_base = torch.tensor(np.concatenate([[0], np.cumsum(np.array(copies) + 1)]), dtype=torch.int32)
    rows = [50, 50, 50, 50, 50, 50, 50, 60, 40, 30, 20, 12, 0]     # experts 0 and 1 split into 4 and 3 groups
    go = torch.tensor(np.concatenate([[0], np.cumsum(rows), [512] * (2 * c.E - len(rows))]), dtype=torch.int32)
    step = types.SimpleNamespace(hist=hist, go=go, rep_base=rep_base, replicate=True)
    s = bench.routing_summary(step, c, 64)
    assert s["replica_groups"] == 13 and s["extra_replicas"] == 5
    assert s["load_max_over_mean"] == round(200 / 64, 3)
    assert s["load_stddev_over_mean"] == round(float(np.std(hist.numpy()) / 64), 3)
    assert s["largest_group_over_target"] == round(60 / 64, 3)
    assert s["experts_without_tokens"] == 1
    assert s["small_path_experts"] == 5          # 60, 40, 30, 20, 12 rows
    # a broken buffer gives an error entry, not an exception
    assert "error" in bench.routing_summary(types.SimpleNamespace(), c, 64)


def test_algorithmic_work_matches_the_quoted_figures():
    """The roofline numerators (per-layer bytes of the HBM stages, flops of
    the FFN) for the five workloads, against the per-stage figures quoted for
    them in the build's scope table (route T*E*4 + A*8; dispatch and combine
    about A*H*2 + T*H*2 plus the index traffic; FFN (2 or 3)*2*A*H*F flops),
    each within one unit of its last quoted digit (the figures are rounded or
    truncated)."""
    from moe_expert_routing_02_b300 import workloads as W
    # workload: route (bytes, quoted), dispatch = combine (bytes), FFN (flops)
    quoted = {
        "tiny": ((12e3, 1e3), (0.1e6, 0.1e6), (0.017e9, 0.001e9)),
        "moe_gpt_stream": ((1.31e6, 0.01e6), (101e6, 1e6), (0.275e12, 0.001e12)),
        "mixtral_layer": ((393e3, 1e3), (201e6, 1e6), (5.77e12, 0.01e12)),
        "deepseekv2_layer": ((2.82e6, 0.01e6), (294e6, 1e6), (1.16e12, 0.01e12)),
        "dbrx_replicated_layer": ((393e3, 1e3), (252e6, 1e6), (6.49e12, 0.01e12)),
    }
    for name, ((r, dr), (d, dd), (f, df)) in quoted.items():
        w = bench.algorithmic_work(W.config_by_name(name))
        assert abs(w["route"]["bytes"] - r) <= dr, (name, w["route"])
        assert abs(w["dispatch"]["bytes"] - d) <= dd, (name, w["dispatch"])
        assert abs(w["combine"]["bytes"] - d) <= dd, (name, w["combine"])
        assert abs(w["ffn"]["flops"] - f) <= df, (name, w["ffn"])
        front = sum(w[s]["bytes"] for s in ("route", "stats", "predict", "replicate", "dispatch"))
        assert w["front"]["bytes"] == front
    # the gathered FFN input: dispatch moves no rows, only the index traffic
    g = bench.algorithmic_work(W.config_by_name("moe_gpt_stream"), gather=True)
    assert g["dispatch"]["bytes"] == 3 * 32768 * 4

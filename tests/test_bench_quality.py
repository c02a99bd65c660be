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

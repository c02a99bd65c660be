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

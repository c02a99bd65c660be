"""The layer step exactly as the benchmark runs it, against the oracle chain.

MoELayerStep with its defaults (fused front, the library's FFN kernel choice,
programmatic dependent launch on, replica table from the layer's own
histogram), every iteration replayed from the per-window-slot CUDA graphs of
capture_slot_graphs, is compared with the oracle's gate -> statistics ->
duplicate_experts -> dispatch -> experts -> collect chain (MoE-GPS blog,
section 2.1; PopFetcher review, core method) on the same seeded inputs:

* every layer's output on sampled tokens within the FFN bar (2e-2 relative
  Frobenius against float64), over the whole sample and per group of tokens
  sharing a first choice;
* the window statistics (ring slots and sums) bit-exact after the replays,
  which covers every layer's histogram and co-selection counts;
* the last layers' routing, replica table and permutation bit-exact, and the
  prediction made for the last layer within 1e-6.

The stream workload replays its stationary skewed phase (iterations 50..59,
cycled, as the benchmark does), where hot experts are split into replica
groups; the single-layer workloads run at full size with replication on.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O
from moe_expert_routing_02_b300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402
from moe_expert_routing_02_b300.layer import MoELayerStep, capture_slot_graphs  # noqa: E402

FFN_TOL = 2e-2
PROB_TOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()
    M.moe_set_option(M.MOE_OPT_PDL, 1)
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, M.MOE_FFN_KERNEL_AUTO)
    yield
    torch.cuda.synchronize()


class _ExpertBits:
    """bf16 bit patterns of one expert's weight matrix at a time, fetched
    from the device on demand (the oracle indexes weights by expert; the
    largest workloads hold several GB of them)."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return W.bf16_bits(self.t[int(e)])


def _rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _check_layer_output(out, lg, x, weights, c, rng, n_sample):
    """out [T,H] bf16 of one layer against the oracle chain on sampled
    tokens; returns the oracle's routing of the whole layer."""
    w1, w3, w2 = weights
    tokens = np.unique(np.concatenate([[0, c.T - 1], rng.integers(0, c.T, n_sample)]))
    ref = O.moe_layer(lg, W.bf16_bits(x), c.k, _ExpertBits(w1), None if w3 is None else _ExpertBits(w3),
                      _ExpertBits(w2), c.act, replicate_on=True, tokens=tokens)
    got = O.bf16_to_f64(W.bf16_bits(out[torch.from_numpy(tokens).to(out.device)]))
    assert _rel_fro(got, ref["out"]) <= FFN_TOL
    top1 = ref["idx"][tokens, 0]
    for e in np.unique(top1):
        m = top1 == e
        assert _rel_fro(got[m], ref["out"][m]) <= FFN_TOL, e
    return ref


def _check_tables(step, ref, c):
    """The step's buffers of the last layer it ran against the oracle's."""
    hst = lambda t: t.detach().cpu().numpy()
    assert np.array_equal(hst(step.hist), ref["hist"])
    copies, rb, ge = ref["rep"]
    assert hst(step.copies).tolist() == copies.tolist()
    assert hst(step.rep_base).tolist() == rb.tolist()
    G = int(rb[-1])
    assert hst(step.group_expert)[:G].tolist() == ge[:G].tolist()
    assert np.array_equal(hst(step.go), ref["group_offsets"])
    assert np.array_equal(hst(step.perm), ref["perm"])
    assert np.array_equal(hst(step.inv), ref["inv_perm"])
    assert np.abs(hst(step.w) - ref["w"]).max() <= PROB_TOL
    return G


def test_layer_step_graph_replay_moe_gpt_stream_stationary_phase():
    """Twelve layers at full size (T = 16384, E = 16, top-2, H = 1024,
    F = 2048 GeLU): one eager iteration, then eleven replays of the slot
    graphs (the ring wraps), as the benchmark's warm-up and timed loop do."""
    c = W.config_by_name("moe_gpt_stream")
    dev = torch.device("cuda")
    base = 50
    pool = [W.make_layer_logits(c, base + q) for q in range(c.window)]
    d_logits = [[torch.from_numpy(l).to(dev) for l in it] for it in pool]
    xs = [W.make_x(c, 0, j, device=dev) for j in range(c.L)]
    weights = [W.make_weights(c, j, device=dev) for j in range(c.L)]
    outs = [torch.empty((c.T, c.H), dtype=torch.bfloat16, device=dev) for _ in range(c.L)]
    st = M.MoEStats(c.L, c.E, c.window)
    step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, stats=st, device=dev)

    def run_iteration(q, ev=None):
        for j in range(c.L):
            step.run(base + q, j, d_logits[q % c.window][j], xs[j], weights[j], outs[j])

    run_iteration(0)
    torch.cuda.synchronize()
    M.moe_check()
    graphs, _ = capture_slot_graphs(run_iteration, c.window)
    seq = list(range(1, 12))          # iterations base+1 .. base+11: slots 1..9, 0, 1
    for q in seq:
        graphs[q % c.window].replay()
    torch.cuda.synchronize()
    M.moe_check()

    # the oracle over the same sequence of iterations
    ost = O.WindowStats(c.L, c.E, c.window)
    last = seq[-1]
    pred_last = None
    for q in [0] + seq:
        prev = None
        for j in range(c.L):
            oi, _ = O.topk_gate(pool[q % c.window][j], c.k)
            ost.update(base + q, j, oi, prev)
            if q == last and j == c.L - 2:
                pred_last = ost.predict(j)
            prev = oi
    ring_h, hsum, ring_c, csum = st.state_arrays()
    assert np.array_equal(ring_h.astype(np.int64), ost.h)
    assert np.array_equal(ring_c.astype(np.int64), ost.C)
    for j in range(c.L):
        assert np.array_equal(hsum[j].astype(np.int64), ost.window_hist(j))
    for j in range(c.L - 1):
        assert np.array_equal(csum[j].astype(np.int64), ost.window_cosel(j))

    rng = np.random.default_rng(2)
    refs = []
    for j in range(c.L):
        refs.append(_check_layer_output(outs[j], pool[last % c.window][j], xs[j], weights[j], c, rng, 128))
    # the last layer's tables, the routing of the layer before it (ping-pong
    # buffer) and the prediction made for the last layer
    G = _check_tables(step, refs[-1], c)
    assert G > c.E, "the stationary phase splits hot experts into replica groups"
    assert np.array_equal(step.idx[(c.L - 1) % 2].cpu().numpy(), refs[-1]["idx"])
    assert np.array_equal(step.idx[(c.L - 2) % 2].cpu().numpy(), refs[-2]["idx"])
    op, _, _ = ost.predict(c.L - 1)
    assert np.abs(step.p_seq.cpu().numpy() - op).max() <= PROB_TOL
    assert np.abs(step.pn[(c.L - 2) % 2].cpu().numpy() - pred_last[2]).max() <= PROB_TOL


@pytest.mark.parametrize("name", ["mixtral_layer", "deepseekv2_layer", "dbrx_replicated_layer"])
def test_layer_step_graph_replay_single_layer_workloads(name):
    """Each single-layer workload at full size through the default step:
    one eager call, then a replayed graph of the next window slot."""
    c = W.config_by_name(name)
    dev = torch.device("cuda")
    lgs = [W.make_layer_logits(c, q, layers=1)[0] for q in range(2)]
    d_lgs = [torch.from_numpy(l).to(dev) for l in lgs]
    x = W.make_x(c, 0, 0, device=dev)
    weights = W.make_weights(c, 0, device=dev)
    out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device=dev)
    st = M.MoEStats(1, c.E, c.window)
    step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, stats=st, device=dev)

    def run_iteration(q, ev=None):
        step.run(q, 0, d_lgs[q % 2], x, weights, out)

    run_iteration(0)
    torch.cuda.synchronize()
    M.moe_check()
    graphs, _ = capture_slot_graphs(run_iteration, 2)
    graphs[1].replay()
    torch.cuda.synchronize()
    M.moe_check()
    rng = np.random.default_rng(3)
    ref = _check_layer_output(out, lgs[1], x, weights, c, rng, 48 if c.E > 16 else 96)
    G = _check_tables(step, ref, c)
    # the graph captured last (slot 1) routed into the buffer before the current one
    assert np.array_equal(step.idx[step._cur ^ 1].cpu().numpy(), ref["idx"])
    if name == "dbrx_replicated_layer":
        assert G > c.E, "the heavy skew splits hot experts into replica groups"
    ring_h, hsum, _, _ = st.state_arrays()
    assert np.array_equal(hsum[0].astype(np.int64), O.histogram(O.topk_gate(lgs[0], c.k)[0], c.E)
                          + ref["hist"])
    del graphs, weights
    torch.cuda.empty_cache()

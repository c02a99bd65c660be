"""moe_layer_front on seeded random shapes against the oracle.

Each case draws T, E, k, H, the window length, the replication settings
(threshold, per-expert copy cap, copies budget, replicas from the layer's
histogram or from a predicted popularity) and the logits (Gaussian with a
Zipf bias, a share of exact ties), then runs two layers over several
iterations so the window ring wraps.  Every output of every call is compared
with the oracle: routing (indices bit-exact, weights within 1e-6), the
histogram, the window ring and sums, the prediction (1e-6), the replica table
(MoE-GPS blog section 2.1, duplicate_experts; MoE-MPMC summary, capacity
bound), the dispatch permutation and group offsets, and the dispatched row
copy."""
import numpy as np
import pytest

from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402

PROB_TOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()


def _case(seed):
    rng = np.random.default_rng([7, seed])
    E = int(rng.choice([1, 2, 3, 5, 8, 16, 17, 32, 63, 100, 160, 255, 256]))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.choice([1, 2, 31, 33, 127, 500, 1024, 2049, 4999]))
    H = int(rng.choice([8, 64, 136]))
    s = int(rng.choice([1, 2, 3]))
    num, den = [(6, 5), (1, 1), (3, 2)][int(rng.integers(0, 3))]
    max_copies = int(rng.choice([-1, 0, 1, 3]))
    budget = int(rng.choice([-1, -1, 0, 2, 7]))
    from_prediction = bool(rng.integers(0, 2))
    alpha = float(rng.uniform(0.0, 2.0))
    return rng, dict(E=E, k=k, T=T, H=H, s=s, num=num, den=den, max_copies=max_copies, budget=budget,
                     from_prediction=from_prediction, alpha=alpha)


def _expected_table(load, total, c, E):
    copies, _, _ = O.replicate(load, total, c["num"], c["den"], c["max_copies"])
    copies = O.cap_copies(copies, load, c["budget"])
    rb = np.zeros(E + 1, dtype=np.int64)
    rb[1:] = np.cumsum(copies.astype(np.int64) + 1)
    ge = np.repeat(np.arange(E), copies.astype(np.int64) + 1)
    return copies, rb, ge


@pytest.fixture(params=[1, 0], ids=["one_launch", "two_launches"])
def front_form(request):
    """Both forms of the front: one cooperative launch (where all its blocks
    fit on the device) and the two launches (the default)."""
    M.moe_set_option(M.MOE_OPT_FRONT_ONE_LAUNCH, request.param)
    yield request.param
    M.moe_set_option(M.MOE_OPT_FRONT_ONE_LAUNCH, 0)


@pytest.mark.parametrize("seed", range(40))
def test_front_random_shapes_against_oracle(seed, front_form):
    rng, c = _case(seed)
    E, k, T, H, s = c["E"], c["k"], c["T"], c["H"], c["s"]
    L = 2
    st = M.MoEStats(L, E, s)
    ost = O.WindowStats(L, E, s)
    A = T * k
    bias = -c["alpha"] * np.log(np.arange(1, E + 1, dtype=np.float64))
    for it in range(2 * s + 1):
        prev_d = prev_o = None
        share = None
        for j in range(L):
            lg_np = (rng.standard_normal((T, E)) + bias[None, :]).astype(np.float32)
            lg_np[:, ::3] = np.round(lg_np[:, ::3])                # exact ties
            x = torch.randn((T, H), device="cuda").to(torch.bfloat16)
            use_share = c["from_prediction"] and share is not None and A < (1 << 29)
            b = M.moe_layer_front(torch.from_numpy(lg_np).cuda(), x, st, it, j, k, idx_prev=prev_d,
                                  predict=True, replicate=True, thresh=(c["num"], c["den"]),
                                  max_copies=c["max_copies"], rep_share=share if use_share else None,
                                  budget=c["budget"])
            M.moe_check()
            oi, ow = O.topk_gate(lg_np, k)
            assert np.array_equal(b["idx"].cpu().numpy(), oi), (c, it, j)
            assert np.abs(b["w"].cpu().numpy() - ow).max() <= PROB_TOL
            oh = ost.update(it, j, oi, prev_o)
            assert np.array_equal(b["hist"].cpu().numpy(), oh), (c, it, j)
            ring_h, hsum, ring_c, csum = st.state_arrays()
            assert np.array_equal(ring_h.astype(np.int64), ost.h), (c, it, j)
            assert np.array_equal(ring_c.astype(np.int64), ost.C), (c, it, j)
            op, oc, opn = ost.predict(j)
            assert np.abs(b["p_seq"].cpu().numpy() - op).max() <= PROB_TOL
            if oc is not None:
                assert np.abs(b["cond"].cpu().numpy() - oc).max() <= PROB_TOL
                assert np.abs(b["p_next"].cpu().numpy() - opn).max() <= PROB_TOL
            # the replica table: from the histogram, or from the apportioned shares
            load = O.apportion(share.cpu().numpy(), A) if use_share else oh
            copies, rb, ge = _expected_table(load, A, c, E)
            assert b["copies"].cpu().numpy().tolist() == copies.tolist(), (c, it, j)
            assert b["rep_base"].cpu().numpy().tolist() == rb.tolist(), (c, it, j)
            G = int(rb[-1])
            assert b["group_expert"].cpu().numpy()[:G].tolist() == ge.tolist(), (c, it, j)
            go, perm, inv = O.dispatch(oi, E, rb)
            assert np.array_equal(b["group_offsets"].cpu().numpy(), go), (c, it, j)
            assert np.array_equal(b["perm"].cpu().numpy(), perm), (c, it, j)
            assert np.array_equal(b["inv_perm"].cpu().numpy(), inv), (c, it, j)
            assert torch.equal(b["xp"], x[b["perm"].long() // k]), (c, it, j)
            if j < L - 1:
                share = b["p_next"].clone()
            prev_d, prev_o = b["idx"], oi

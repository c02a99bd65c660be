"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (a framework that owns all device memory, work
enqueued during stream capture, a thread that must not risk cudaMalloc's
device synchronisation).  It keeps its scratch in a static per-device array
instead of a caller workspace; its results must equal moe_dispatch's.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def M():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    import moe_expert_routing_02_b300 as M
    M.lib()
    return M


def _inputs(seed, T, E, k, H):
    from moe_expert_routing_02_b300 import workloads as W
    rng = np.random.default_rng(seed)
    logits = W.make_logits(T, E, 1.3, seed_key=(seed, 77, 0, 0, 0))
    idx = np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)
    x = torch.randn((T, H), device="cuda", generator=torch.Generator("cuda").manual_seed(seed)).to(torch.bfloat16)
    return torch.from_numpy(idx).cuda(), x


def test_noalloc_dispatch_matches_dispatch_on_two_calls(M):
    T, E, k, H = 16384, 16, 2, 1024
    for call, seed in enumerate((1, 2)):  # two calls in a row, different routing
        idx, x = _inputs(seed, T, E, k, H)
        hist = torch.bincount(idx.reshape(-1).long(), minlength=E).to(torch.int32)
        _, rep_base, _ = M.moe_replicate(hist, T * k)
        for rb in (None, rep_base):
            want = M.moe_dispatch(x, idx, E, rb)
            got = M.moe_dispatch_noalloc(x, idx, E, rb)
            M.moe_check()
            for a, b in zip(want, got):
                assert torch.equal(a, b), (call, rb is None)


def test_noalloc_dispatch_through_the_c_abi_rejects_oversize(M):
    L = M.lib()
    # 2^17 * 8 = 1,048,576 assignments over 256 experts: just over the limit
    # (1024-assignment tiles: (1025 + 4) * 256 * 4 bytes > 1 MiB); one
    # assignment past the exact boundary (130,561 * 8) is refused as well.
    # Refused on the host, nothing enqueued.
    fake = ctypes.c_void_p(0x10000)
    for T in (1 << 17, 130561):
        st = L.moe_dispatch_noalloc(None, fake, T, 8, 64, 256, None, fake, fake, fake, None, None)
        assert st == M.MOE_ERR_WORKSPACE
        assert b"scratch" in L.moe_last_error()
    # a size that fits goes through the raw C call and matches moe_dispatch
    idx, _ = _inputs(3, 4097, 160, 6, 64)
    T, k = idx.shape
    A = T * k
    go = torch.empty(2 * 160 + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(A, dtype=torch.int32, device="cuda")
    inv = torch.empty(A, dtype=torch.int32, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        st = L.moe_dispatch_noalloc(None, ctypes.c_void_p(idx.data_ptr()), T, k, 8, 160, None,
                                    ctypes.c_void_p(go.data_ptr()), ctypes.c_void_p(perm.data_ptr()),
                                    ctypes.c_void_p(inv.data_ptr()), None, s)
        assert st == M.MOE_OK
        want = M.moe_dispatch(None, idx, 160)
        M.moe_check()
        assert torch.equal(go, want[0]) and torch.equal(perm, want[1]) and torch.equal(inv, want[2])


def test_noalloc_dispatch_at_the_exact_limit(M):
    """130,560 tokens x top-8 over 256 experts = 1020 tiles of 1024
    assignments: (1020 + 4) * 256 * 4 bytes = exactly 1 MiB of scratch, the
    largest request at E = 256 that is accepted; it must match moe_dispatch."""
    T, E, k = 130560, 256, 8
    assert M.workspace_bytes(M.MOE_OP_DISPATCH, T, k, E) == 1 << 20
    idx, x = _inputs(4, T, E, k, 64)
    for _ in range(2):
        want = M.moe_dispatch(x, idx, E, None)
        got = M.moe_dispatch_noalloc(x, idx, E, None)
        M.moe_check()
        for a, b in zip(want, got):
            assert torch.equal(a, b)

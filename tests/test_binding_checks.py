"""Host-side checks of the Python binding, without a GPU: the library's launch
entry points are replaced by a recorder (its pure host functions, such as the
workspace sizes, stay real) and the CUDA-tensor check is relaxed to accept
CPU tensors, so that only the binding's own argument checks run.  Buffers a
call writes through a raw pointer must be at least the size it writes;
smaller ones are refused before anything is enqueued, larger ones pass."""
import ctypes

import pytest

torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402
from moe_expert_routing_02_b300 import _build  # noqa: E402

HOST_ONLY = {"moe_workspace_bytes", "moe_ffn_backward_workspace_bytes", "moe_ffn_launches", "moe_status_string",
             "moe_last_error"}


@pytest.fixture()
def rec(monkeypatch):
    _build.build()
    real = M.lib()
    calls = []

    class Recorder:
        def __getattr__(self, name):
            if name in HOST_ONLY:
                return getattr(real, name)

            def launch(*args):
                calls.append(name)
                return M.MOE_OK
            return launch

    def dev_any(t, dtype, name, ndim=None):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if ndim is not None and t.dim() != ndim:
            raise ValueError(f"{name} must have {ndim} dims")
        return t

    monkeypatch.setattr(M, "lib", lambda: Recorder())
    monkeypatch.setattr(M, "_dev", dev_any)
    monkeypatch.setattr(M, "_stream", lambda s=None: ctypes.c_void_p(0))
    return calls


class _Stats:
    def __init__(self, L, E):
        self.L, self.E, self.window = L, E, 10
        self.handle = ctypes.c_void_p(0)


T, E, k, H, F = 48, 8, 2, 64, 128
A = T * k
i32, f32, bf = torch.int32, torch.float32, torch.bfloat16


def _z(*shape, dtype=f32):
    return torch.zeros(shape, dtype=dtype)


def test_exact_and_larger_buffers_pass(rec):
    idx = _z(T, k, dtype=i32)
    M.moe_route(_z(T, E), k, idx=idx, w=_z(T, k))
    M.moe_route(_z(T, E), k, idx=_z(T * k + 5, dtype=i32), w=_z(T * k + 5))       # larger is fine
    st = _Stats(3, E)
    M.moe_stats_update(st, 0, 1, idx, idx, hist_out=_z(E, dtype=i32))
    M.moe_predict(st, 0, out=(_z(E), _z(E, E), _z(E)))
    M.moe_replicate(_z(E, dtype=i32), A, out=(_z(E, dtype=i32), _z(E + 1, dtype=i32), _z(2 * E, dtype=i32)))
    x = _z(T, H, dtype=bf)
    go, perm, inv, xp = _z(2 * E + 1, dtype=i32), _z(A, dtype=i32), _z(A, dtype=i32), _z(A, H, dtype=bf)
    M.moe_dispatch(x, idx, E, None, out=(go, perm, inv, xp), workspace=_z(1 << 16, dtype=torch.uint8))
    w1, w2 = _z(E, H, F, dtype=bf), _z(E, F, H, dtype=bf)
    M.moe_expert_ffn(xp, go, None, None, w1, None, w2, "gelu", y=_z(A, H, dtype=bf))
    M.moe_expert_ffn(xp, _z(E + 1, dtype=i32), None, None, w1, None, w2, "gelu")   # E + 1 offsets, no replicas
    M.moe_combine(_z(A, H, dtype=bf), inv, _z(T, k), out=_z(T, H, dtype=bf))
    out = (_z(T, H, dtype=bf), _z(T, k), _z(E, H, F), None, _z(E, F, H))
    M.moe_ffn_backward(x, _z(T, H, dtype=bf), _z(T, k), _z(A, H, dtype=bf), perm, inv, go, None, w1, None, w2,
                       "gelu", out=out, workspace=_z(1 << 22, dtype=torch.uint8))
    M.moe_route_backward(_z(T, E), idx, _z(T, k), out=_z(T, E))
    assert rec == ["moe_route", "moe_route", "moe_stats_update", "moe_predict", "moe_replicate", "moe_dispatch",
                   "moe_expert_ffn", "moe_expert_ffn", "moe_combine", "moe_ffn_backward", "moe_route_backward"]


@pytest.mark.parametrize("case", [
    "route_idx", "route_w", "hist", "cond", "rep_base", "group_expert", "perm", "xp", "ffn_y", "ffn_offsets",
    "combine_out", "combine_y_rows", "dx", "dw1", "dlogits", "front_inv", "front_idx_prev", "slot_map",
    "workspace_dtype",
])
def test_undersized_buffers_are_refused_before_launch(rec, case):
    idx = _z(T, k, dtype=i32)
    x = _z(T, H, dtype=bf)
    st = _Stats(3, E)
    go, perm, inv, xp = _z(2 * E + 1, dtype=i32), _z(A, dtype=i32), _z(A, dtype=i32), _z(A, H, dtype=bf)
    w1, w2 = _z(E, H, F, dtype=bf), _z(E, F, H, dtype=bf)
    ws = _z(1 << 22, dtype=torch.uint8)
    short = {
        "route_idx": lambda: M.moe_route(_z(T, E), k, idx=_z(T, 1, dtype=i32)),
        "route_w": lambda: M.moe_route(_z(T, E), k, w=_z(T * k - 1)),
        "hist": lambda: M.moe_stats_update(st, 0, 0, idx, hist_out=_z(E - 1, dtype=i32)),
        "cond": lambda: M.moe_predict(st, 0, out=(_z(E), _z(E), _z(E))),
        "rep_base": lambda: M.moe_replicate(_z(E, dtype=i32), A, out=(_z(E, dtype=i32), _z(E, dtype=i32),
                                                                       _z(2 * E, dtype=i32))),
        "group_expert": lambda: M.moe_replicate(_z(E, dtype=i32), A, out=(_z(E, dtype=i32), _z(E + 1, dtype=i32),
                                                                           _z(E, dtype=i32))),
        "perm": lambda: M.moe_dispatch(x, idx, E, out=(go, perm[:-1], inv, xp), workspace=ws),
        "xp": lambda: M.moe_dispatch(x, idx, E, out=(go, perm, inv, _z(A - 1, H, dtype=bf)), workspace=ws),
        "ffn_y": lambda: M.moe_expert_ffn(xp, go, None, None, w1, None, w2, "gelu", y=_z(A - 1, H, dtype=bf)),
        "ffn_offsets": lambda: M.moe_expert_ffn(xp, _z(2 * E, dtype=i32), _z(2 * E, dtype=i32), None, w1, None, w2),
        "combine_out": lambda: M.moe_combine(_z(A, H, dtype=bf), inv, _z(T, k), out=_z(T - 1, H, dtype=bf)),
        "combine_y_rows": lambda: M.moe_combine(_z(A - 1, H, dtype=bf), inv, _z(T, k)),
        "dx": lambda: M.moe_ffn_backward(x, x, _z(T, k), None, perm, inv, go, None, w1, None, w2, "gelu",
                                         out=(_z(T - 1, H, dtype=bf), None, _z(E, H, F), None, _z(E, F, H)),
                                         workspace=ws),
        "dw1": lambda: M.moe_ffn_backward(x, x, _z(T, k), None, perm, inv, go, None, w1, None, w2, "gelu",
                                          out=(_z(T, H, dtype=bf), None, _z(E - 1, H, F), None, _z(E, F, H)),
                                          workspace=ws),
        "dlogits": lambda: M.moe_route_backward(_z(T, E), idx, _z(T, k), out=_z(T, E - 1)),
        "front_inv": lambda: M.moe_layer_front(_z(T, E), None, st, 0, 0, k, out={"inv_perm": _z(A - 1, dtype=i32)}),
        "front_idx_prev": lambda: M.moe_layer_front(_z(T, E), None, st, 0, 1, k, idx_prev=_z(T - 1, k, dtype=i32)),
        "slot_map": lambda: M.moe_replicate_weights(_z(E + 1, dtype=i32), None, group_slot=_z(2 * E - 1, dtype=i32)),
        "workspace_dtype": lambda: M.moe_dispatch(x, idx, E, out=(go, perm, inv, xp), workspace=_z(1 << 16)),
    }[case]
    with pytest.raises(ValueError):
        short()
    assert rec == []

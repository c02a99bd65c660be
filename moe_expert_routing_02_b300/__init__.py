"""Python binding of libmoe, the B300 MoE routing-and-expert step.

Argument marshalling only: every function here checks tensor placement and
dtype, passes raw device pointers and the current CUDA stream to the C ABI
(include/moe.h) and returns the output tensors.  All arithmetic runs in the
library's CUDA kernels; there is no CPU fallback, and using any function
without the built library raises.

Functions carry the C names: moe_route, moe_stats_update, moe_predict,
moe_replicate, moe_dispatch, moe_expert_ffn, moe_combine, their fused forms,
the replication and backward calls (plus MoEStats, the owner of the
sliding-window state, and moe_check).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "MoEError", "lib", "library_path", "MoEStats", "moe_check", "moe_error_word", "EXPORTED_SYMBOLS",
    # the seven calls of the layer step
    "moe_route", "moe_stats_update", "moe_predict", "moe_replicate", "moe_dispatch", "moe_expert_ffn",
    "moe_combine",
    # fused forms
    "moe_layer_front", "moe_expert_ffn_gather", "moe_expert_ffn_combine", "moe_dispatch_noalloc",
    # prediction-driven and physical replication
    "moe_predict_decay", "moe_replicate_predicted", "moe_replicate_weights", "moe_expert_ffn_slots",
    # backward
    "moe_ffn_backward", "moe_ffn_backward_workspace_bytes", "moe_route_backward",
    "MOE_BWD_ACCUMULATE_WGRAD", "MOE_BWD_WGRAD_BF16",
    # sizes, options, constants
    "workspace_bytes", "moe_ffn_launches", "moe_layer_front_launches", "moe_set_option", "moe_get_option",
    "MOE_OP_DISPATCH", "MOE_OP_EXPERT_FFN", "MOE_OP_LAYER_FRONT", "MOE_OP_EXPERT_FFN_COMBINE",
    "MOE_ACT_GELU", "MOE_ACT_SWIGLU", "MOE_OPT_FFN_KERNEL", "MOE_FFN_KERNEL_AUTO", "MOE_FFN_KERNEL_SINGLE",
    "MOE_FFN_KERNEL_PAIR", "MOE_FFN_KERNEL_FUSED", "MOE_OPT_FFN_TIMEOUT_SELFTEST", "MOE_OPT_PDL",
    "MOE_OPT_FFN_SMALL_SMS", "MOE_OPT_FRONT_ONE_LAUNCH",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_WORKSPACE, MOE_ERR_DEVICE = range(7)
MOE_ACT_GELU, MOE_ACT_SWIGLU = 0, 1
MOE_OP_DISPATCH, MOE_OP_EXPERT_FFN, MOE_OP_LAYER_FRONT, MOE_OP_EXPERT_FFN_COMBINE = 1, 2, 3, 4
MOE_OPT_FFN_KERNEL, MOE_OPT_FFN_TIMEOUT_SELFTEST, MOE_OPT_PDL, MOE_OPT_FFN_SMALL_SMS = 1, 2, 3, 4
MOE_OPT_FRONT_ONE_LAUNCH = 5
MOE_FFN_KERNEL_AUTO, MOE_FFN_KERNEL_SINGLE, MOE_FFN_KERNEL_PAIR, MOE_FFN_KERNEL_FUSED = 0, 1, 2, 3

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

# name -> (restype, argtypes)
_SIGS = {
    "moe_stats_create": (_I, [ctypes.POINTER(_P), _I, _I, _I, _P]),
    "moe_stats_destroy": (_I, [_P]),
    "moe_route": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_stats_update": (_I, [_P, _I64, _I, _P, _P, _I, _I, _P, _P]),
    "moe_predict": (_I, [_P, _I, _P, _P, _P, _P]),
    "moe_replicate": (_I, [_P, _I, _I64, _I, _I, _I, _P, _P, _P, _P]),
    "moe_dispatch": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_dispatch_noalloc": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "moe_expert_ffn": (_I, [_P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_replicate_weights": (_I, [_P, _I, _P, _I, _I, _P, _P]),
    "moe_expert_ffn_slots": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_ffn_launches": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_layer_front_launches": (_I, [_I, _I, _I, _I]),
    "moe_predict_decay": (_I, [_P, _I, ctypes.c_int64, ctypes.c_double, _P, _P, _P, _P]),
    "moe_replicate_predicted": (_I, [_P, _I, ctypes.c_int64, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_expert_ffn_gather": (_I, [_P, _I, _P, _I, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_combine": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_check": (_I, [_P]),
    "moe_error_word": (_I, [ctypes.POINTER(ctypes.c_uint32)]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_stats_bytes": (_SZ, [_P]),
    "moe_stats_export": (_I, [_P, _P, _SZ]),
    "moe_stats_import": (_I, [_P, _P, _SZ]),
    "moe_version": (ctypes.c_char_p, []),
    "moe_set_option": (_I, [_I, _I]),
    "moe_layer_front": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _I64, _I, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P,
                             _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_get_option": (_I, [_I, ctypes.POINTER(_I)]),
    "moe_ffn_backward_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_expert_ffn_combine": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ,
                                    _P]),
    "moe_ffn_backward": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P,
                              _I, _P, _SZ, _P]),
    "moe_route_backward": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P]),
}
EXPORTED_SYMBOLS = tuple(_SIGS)

_lib = None


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def lib():
    """The loaded libmoe (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"libmoe.so is not built ({library_path}); run "
                               "`python -m moe_expert_routing_02_b300._build`")
        L = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != MOE_OK:
        L = lib()
        raise MoEError(status, f"{what}: {L.moe_status_string(status).decode()}: {L.moe_last_error().decode()}")


def _torch():
    import torch
    return torch


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dev(t, dtype, name, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    return t


def _out(t, dtype, name, numel, ndim=None):
    """A caller-provided output (or an input read by index): a contiguous
    CUDA tensor of `dtype` with room for at least `numel` elements, since
    the kernels reach it through a raw pointer."""
    _dev(t, dtype, name, ndim)
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements; the call needs {numel}")
    return t


def _ws_bytes(workspace) -> int:
    """A workspace is a contiguous uint8 CUDA tensor; its size in bytes."""
    return _dev(workspace, _torch().uint8, "workspace").numel()


def workspace_bytes(op: int, T: int, k: int, E: int, H: int = 64, F: int = 64) -> int:
    return int(lib().moe_workspace_bytes(op, T, k, E, H, F))


# ----------------------------------------------------------------------------
def moe_route(logits, k: int, renorm: bool = True, idx=None, w=None, stream=None):
    """Top-k gate: returns (idx [T,k] int32, w [T,k] float32)."""
    torch = _torch()
    _dev(logits, torch.float32, "logits", 2)
    T, E = logits.shape
    if idx is None:
        idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if w is None:
        w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _out(idx, torch.int32, "idx", T * k)
    _out(w, torch.float32, "w", T * k)
    _check(lib().moe_route(_ptr(logits), T, E, k, int(bool(renorm)), _ptr(idx), _ptr(w), _stream(stream)),
           "moe_route")
    return idx, w


class MoEStats:
    """Owner of the device-side sliding-window statistics (moe_stats_*)."""

    def __init__(self, L: int, E: int, window: int = 10, stream=None):
        self.L, self.E, self.window = L, E, window
        h = ctypes.c_void_p()
        _check(lib().moe_stats_create(ctypes.byref(h), L, E, window, _stream(stream)), "moe_stats_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().moe_stats_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def export_state(self) -> bytes:
        n = int(lib().moe_stats_bytes(self._h))
        buf = ctypes.create_string_buffer(n)
        _check(lib().moe_stats_export(self._h, buf, n), "moe_stats_export")
        return buf.raw

    def import_state(self, data: bytes):
        buf = ctypes.create_string_buffer(bytes(data), len(data))
        _check(lib().moe_stats_import(self._h, buf, len(data)), "moe_stats_import")

    def state_arrays(self):
        """Exported state decoded as NumPy arrays (ring_h, hsum, ring_c, csum)."""
        import numpy as np
        raw = self.export_state()
        hdr = 32
        L, E, s = self.L, self.E, self.window
        off = hdr
        def take(dtype, n):
            nonlocal off
            a = np.frombuffer(raw, dtype=dtype, count=n, offset=off)
            off += a.nbytes
            return a
        hsum = take(np.uint64, L * E).reshape(L, E)
        csum = take(np.uint64, (L - 1) * E * E).reshape(L - 1, E, E)
        ring_h = take(np.uint32, L * s * E).reshape(L, s, E)
        ring_c = take(np.uint32, (L - 1) * s * E * E).reshape(L - 1, s, E, E)
        return ring_h, hsum, ring_c, csum


def moe_stats_update(stats: MoEStats, it: int, layer: int, idx_layer, idx_prev=None, hist_out=None, stream=None):
    """Record one layer's routing; returns hist_out ([E] int32) if given, else None."""
    torch = _torch()
    _dev(idx_layer, torch.int32, "idx_layer", 2)
    T, k = idx_layer.shape
    if idx_prev is not None:
        _dev(idx_prev, torch.int32, "idx_prev", 2)
        if tuple(idx_prev.shape) != (T, k):
            raise ValueError("idx_prev must match idx_layer's shape")
    if hist_out is not None:
        _out(hist_out, torch.int32, "hist_out", stats.E)
    _check(lib().moe_stats_update(stats.handle, int(it), int(layer), _ptr(idx_layer), _ptr(idx_prev), T, k,
                                  _ptr(hist_out), _stream(stream)), "moe_stats_update")
    return hist_out


def moe_predict(stats: MoEStats, layer: int, want_cond: bool = True, want_next: Optional[bool] = None,
                device=None, out=None, stream=None):
    """(p_seq [E], cond [E,E] or None, p_next [E] or None), float32.

    `out` = (p_seq, cond or None, p_next or None) preallocated outputs."""
    torch = _torch()
    E = stats.E
    last = layer == stats.L - 1
    if out is None:
        device = device or torch.device("cuda", torch.cuda.current_device())
        if want_next is None:
            want_next = not last
        p_seq = torch.empty(E, dtype=torch.float32, device=device)
        cond = torch.empty((E, E), dtype=torch.float32, device=device) if (want_cond and not last) else None
        p_next = torch.empty(E, dtype=torch.float32, device=device) if (want_next and not last) else None
    else:
        p_seq, cond, p_next = out
        _out(p_seq, torch.float32, "p_seq", E)
        if cond is not None:
            _out(cond, torch.float32, "cond", E * E)
        if p_next is not None:
            _out(p_next, torch.float32, "p_next", E)
    _check(lib().moe_predict(stats.handle, int(layer), _ptr(p_seq), _ptr(cond), _ptr(p_next), _stream(stream)),
           "moe_predict")
    return p_seq, cond, p_next


def moe_predict_decay(stats: "MoEStats", layer: int, it: int, lam: float, want_cond: bool = True,
                      want_next: Optional[bool] = None, out=None, stream=None):
    """(p_seq [E], cond [E,E] or None, p_next [E] or None) from the
    decay-weighted window (weights lam**age; lam = 1 is moe_predict)."""
    torch = _torch()
    E = stats.E
    last = layer == stats.L - 1
    if want_next is None:
        want_next = not last
    if out is None:
        dev = torch.device("cuda", torch.cuda.current_device())
        p_seq = torch.empty(E, dtype=torch.float32, device=dev)
        cond = torch.empty((E, E), dtype=torch.float32, device=dev) if (want_cond and not last) else None
        p_next = torch.empty(E, dtype=torch.float32, device=dev) if (want_next and not last) else None
    else:
        p_seq, cond, p_next = out
        _out(p_seq, torch.float32, "p_seq", E)
        if cond is not None:
            _out(cond, torch.float32, "cond", E * E)
        if p_next is not None:
            _out(p_next, torch.float32, "p_next", E)
    _check(lib().moe_predict_decay(stats.handle, int(layer), int(it), float(lam), _ptr(p_seq), _ptr(cond),
                                   _ptr(p_next), _stream(stream)), "moe_predict_decay")
    return p_seq, cond, p_next


def moe_replicate_predicted(p_next, total: int, thresh=(6, 5), max_copies: int = -1, budget: int = -1, out=None,
                            stream=None):
    """(load [E], copies [E], rep_base [E+1], group_expert [2E]) int32 from a
    predicted popularity: largest-remainder loads of `total`, the replica rule,
    the copy budget (-1 = none)."""
    torch = _torch()
    _dev(p_next, torch.float32, "p_next", 1)
    E = p_next.numel()
    if out is None:
        out = (torch.empty(E, dtype=torch.int32, device=p_next.device),
               torch.empty(E, dtype=torch.int32, device=p_next.device),
               torch.empty(E + 1, dtype=torch.int32, device=p_next.device),
               torch.empty(2 * E, dtype=torch.int32, device=p_next.device))
    load, copies, rb, ge = out
    for nm, t, n in (("load", load, E), ("copies", copies, E), ("rep_base", rb, E + 1), ("group_expert", ge, 2 * E)):
        _out(t, torch.int32, nm, n)
    _check(lib().moe_replicate_predicted(_ptr(p_next), E, int(total), int(thresh[0]), int(thresh[1]),
                                         int(max_copies), int(budget), _ptr(load), _ptr(copies), _ptr(rb), _ptr(ge),
                                         _stream(stream)), "moe_replicate_predicted")
    return load, copies, rb, ge


def moe_replicate(load, total: int, thresh=(6, 5), max_copies: int = -1, out=None, stream=None):
    """(copies [E], rep_base [E+1], group_expert [2E]) int32."""
    torch = _torch()
    _dev(load, torch.int32, "load", 1)
    E = load.shape[0]
    if out is None:
        out = (torch.empty(E, dtype=torch.int32, device=load.device),
               torch.empty(E + 1, dtype=torch.int32, device=load.device),
               torch.empty(2 * E, dtype=torch.int32, device=load.device))
    copies, rep_base, group_expert = out
    for nm, t, n in (("copies", copies, E), ("rep_base", rep_base, E + 1), ("group_expert", group_expert, 2 * E)):
        _out(t, torch.int32, nm, n)
    _check(lib().moe_replicate(_ptr(load), E, int(total), int(thresh[0]), int(thresh[1]), int(max_copies),
                               _ptr(copies), _ptr(rep_base), _ptr(group_expert), _stream(stream)), "moe_replicate")
    return copies, rep_base, group_expert


def _dispatch_outputs(go, perm, inv, xp, E, A, H):
    torch = _torch()
    _out(go, torch.int32, "group_offsets", 2 * E + 1)
    _out(perm, torch.int32, "perm", A)
    _out(inv, torch.int32, "inv_perm", A)
    if xp is not None:
        _out(xp, torch.bfloat16, "xp", A * H)


def moe_dispatch(x, idx, E: int, rep_base=None, out=None, workspace=None, stream=None):
    """(group_offsets [2E+1], perm [A], inv_perm [A], xp [A,H] or None).

    x may be None for the permutation only."""
    torch = _torch()
    _dev(idx, torch.int32, "idx", 2)
    T, k = idx.shape
    A = T * k
    dev = idx.device
    H = 8
    if x is not None:
        _dev(x, torch.bfloat16, "x", 2)
        H = x.shape[1]
        if x.shape[0] != T:
            raise ValueError("x and idx disagree on T")
    if rep_base is not None:
        _dev(rep_base, torch.int32, "rep_base", 1)
    if out is None:
        out = (torch.empty(2 * E + 1, dtype=torch.int32, device=dev),
               torch.empty(A, dtype=torch.int32, device=dev),
               torch.empty(A, dtype=torch.int32, device=dev),
               None if x is None else torch.empty((A, H), dtype=torch.bfloat16, device=dev))
    go, perm, inv, xp = out
    _dispatch_outputs(go, perm, inv, xp, E, A, H)
    need = workspace_bytes(MOE_OP_DISPATCH, T, k, E)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check(lib().moe_dispatch(_ptr(x), _ptr(idx), T, k, H, E, _ptr(rep_base), _ptr(go), _ptr(perm), _ptr(inv),
                              _ptr(xp), _ptr(workspace), _ws_bytes(workspace), _stream(stream)), "moe_dispatch")
    return go, perm, inv, xp


def moe_dispatch_noalloc(x, idx, E: int, rep_base=None, out=None, stream=None):
    """moe_dispatch with the library's static per-device scratch instead of a
    workspace (for callers that cannot allocate).  `out` = (group_offsets,
    perm, inv_perm, xp or None), allocated here when not given."""
    torch = _torch()
    _dev(idx, torch.int32, "idx", 2)
    T, k = idx.shape
    A = T * k
    dev = idx.device
    H = 8
    if x is not None:
        _dev(x, torch.bfloat16, "x", 2)
        H = x.shape[1]
        if x.shape[0] != T:
            raise ValueError("x and idx disagree on T")
    if rep_base is not None:
        _dev(rep_base, torch.int32, "rep_base", 1)
    if out is None:
        out = (torch.empty(2 * E + 1, dtype=torch.int32, device=dev),
               torch.empty(A, dtype=torch.int32, device=dev),
               torch.empty(A, dtype=torch.int32, device=dev),
               None if x is None else torch.empty((A, H), dtype=torch.bfloat16, device=dev))
    go, perm, inv, xp = out
    _dispatch_outputs(go, perm, inv, xp, E, A, H)
    _check(lib().moe_dispatch_noalloc(_ptr(x), _ptr(idx), T, k, H, E, _ptr(rep_base), _ptr(go), _ptr(perm),
                                      _ptr(inv), _ptr(xp), _stream(stream)), "moe_dispatch_noalloc")
    return go, perm, inv, xp


def moe_layer_front(logits, x, stats: "MoEStats", it: int, layer: int, k: int, idx_prev=None, renorm: bool = True,
                    predict: bool = True, replicate: bool = True, thresh=(6, 5), max_copies: int = -1,
                    rep_share=None, budget: int = -1, out=None, workspace=None, stream=None):
    """Route + stats update + predict + replicate + dispatch of one layer in
    two launches (results identical
    to the separate calls).  Returns a dict of the
    outputs: idx, w, hist, p_seq, cond, p_next, copies, rep_base, group_expert,
    group_offsets, perm, inv_perm, xp (absent ones None).  `out` may hold
    preallocated tensors under those names.  rep_share ([E] float32, e.g. the
    previous layer's p_next) takes the replica table from that prediction
    instead of the layer's own histogram; budget bounds the total copies."""
    torch = _torch()
    _dev(logits, torch.float32, "logits", 2)
    T, E = logits.shape
    dev = logits.device
    H = 8
    if x is not None:
        _dev(x, torch.bfloat16, "x", 2)
        H = x.shape[1]
        if x.shape[0] != T:
            raise ValueError("x and logits disagree on T")
    if idx_prev is not None:
        _out(idx_prev, torch.int32, "idx_prev", T * k, 2)
    last = layer == stats.L - 1
    o = dict(out or {})
    i32, f32 = torch.int32, torch.float32
    def need(name, shape, dtype, cond=True):
        if not cond:
            return None
        if o.get(name) is None:
            o[name] = torch.empty(shape, dtype=dtype, device=dev)
        n = 1
        for d in shape:
            n *= d
        return _out(o[name], dtype, name, n)
    idx = need("idx", (T, k), i32)
    w = need("w", (T, k), f32)
    hist = need("hist", (E,), i32)
    p_seq = need("p_seq", (E,), f32, predict)
    cond = need("cond", (E, E), f32, predict and not last)
    p_next = need("p_next", (E,), f32, predict and not last)
    copies = need("copies", (E,), i32, replicate)
    rep_base = need("rep_base", (E + 1,), i32, replicate)
    group_expert = need("group_expert", (2 * E,), i32, replicate)
    go = need("group_offsets", (2 * E + 1,), i32)
    perm = need("perm", (T * k,), i32)
    inv = need("inv_perm", (T * k,), i32)
    xp = need("xp", (T * k, H), torch.bfloat16, x is not None)
    if workspace is None:
        workspace = torch.empty(max(workspace_bytes(MOE_OP_LAYER_FRONT, T, k, E), 16), dtype=torch.uint8, device=dev)
    if rep_share is not None:
        _out(rep_share, torch.float32, "rep_share", E, 1)
    _check(lib().moe_layer_front(_ptr(logits), _ptr(x), T, E, k, H, int(bool(renorm)), stats.handle, int(it),
                                 int(layer), _ptr(idx_prev), int(bool(replicate)), int(thresh[0]), int(thresh[1]),
                                 int(max_copies), _ptr(rep_share), int(budget), _ptr(idx), _ptr(w), _ptr(hist),
                                 _ptr(p_seq), _ptr(cond),
                                 _ptr(p_next), _ptr(copies), _ptr(rep_base), _ptr(group_expert), _ptr(go),
                                 _ptr(perm), _ptr(inv), _ptr(xp), _ptr(workspace), _ws_bytes(workspace),
                                 _stream(stream)), "moe_layer_front")
    return {"idx": idx, "w": w, "hist": hist, "p_seq": p_seq, "cond": cond, "p_next": p_next, "copies": copies,
            "rep_base": rep_base, "group_expert": group_expert, "group_offsets": go, "perm": perm,
            "inv_perm": inv, "xp": xp}


def moe_expert_ffn(xp, group_offsets, group_expert, rep_base, w1, w3, w2, act: str = "gelu",
                   small_group_threshold: int = 64, y=None, workspace=None, stream=None):
    """Grouped expert FFN: returns y [A, H] bf16."""
    torch = _torch()
    _dev(xp, torch.bfloat16, "xp", 2)
    _dev(w1, torch.bfloat16, "w1", 3)
    _dev(w2, torch.bfloat16, "w2", 3)
    if w3 is not None:
        _dev(w3, torch.bfloat16, "w3", 3)
    _dev(group_offsets, torch.int32, "group_offsets", 1)
    if group_expert is not None:
        _dev(group_expert, torch.int32, "group_expert", 1)
    if rep_base is not None:
        _dev(rep_base, torch.int32, "rep_base", 1)
    A, H = xp.shape
    E, H1, F = w1.shape
    if H1 != H or tuple(w2.shape) != (E, F, H) or (w3 is not None and w3.shape != w1.shape):
        raise ValueError("weight shapes must be w1/w3 [E,H,F], w2 [E,F,H]")
    _out(group_offsets, torch.int32, "group_offsets", (2 * E if group_expert is not None else E) + 1)
    act_id = {"gelu": MOE_ACT_GELU, "swiglu": MOE_ACT_SWIGLU}[act]
    if y is None:
        y = torch.empty((A, H), dtype=torch.bfloat16, device=xp.device)
    _out(y, torch.bfloat16, "y", A * H, 2)
    need = int(lib().moe_workspace_bytes(MOE_OP_EXPERT_FFN, A, 1, E, H, F))
    if workspace is None:
        workspace = torch.empty(max(need, 1024), dtype=torch.uint8, device=xp.device)
    _check(lib().moe_expert_ffn(_ptr(xp), _ptr(group_offsets), _ptr(group_expert), _ptr(rep_base), E, A,
                                _ptr(w1), _ptr(w3), _ptr(w2), H, F, act_id, int(small_group_threshold), _ptr(y),
                                _ptr(workspace), _ws_bytes(workspace), _stream(stream)), "moe_expert_ffn")
    return y


def moe_expert_ffn_gather(x, perm, k: int, group_offsets, group_expert, rep_base, w1, w3, w2, act: str = "gelu",
                          small_group_threshold: int = 64, y=None, workspace=None, stream=None):
    """Grouped expert FFN reading the token rows in place: dispatched row i is
    x[perm[i] // k].  Returns y [T*k, H] bf16, bit-identical to
    moe_expert_ffn on the copied rows."""
    torch = _torch()
    _dev(x, torch.bfloat16, "x", 2)
    _dev(perm, torch.int32, "perm", 1)
    _dev(w1, torch.bfloat16, "w1", 3)
    _dev(w2, torch.bfloat16, "w2", 3)
    if w3 is not None:
        _dev(w3, torch.bfloat16, "w3", 3)
    _dev(group_offsets, torch.int32, "group_offsets", 1)
    if group_expert is not None:
        _dev(group_expert, torch.int32, "group_expert", 1)
    if rep_base is not None:
        _dev(rep_base, torch.int32, "rep_base", 1)
    T, H = x.shape
    E, H1, F = w1.shape
    if H1 != H or tuple(w2.shape) != (E, F, H) or (w3 is not None and w3.shape != w1.shape):
        raise ValueError("weight shapes must be w1/w3 [E,H,F], w2 [E,F,H]")
    if perm.numel() != T * k:
        raise ValueError("perm must hold T*k entries")
    _out(group_offsets, torch.int32, "group_offsets", (2 * E if group_expert is not None else E) + 1)
    act_id = {"gelu": MOE_ACT_GELU, "swiglu": MOE_ACT_SWIGLU}[act]
    if y is None:
        y = torch.empty((T * k, H), dtype=torch.bfloat16, device=x.device)
    _out(y, torch.bfloat16, "y", T * k * H, 2)
    need = int(lib().moe_workspace_bytes(MOE_OP_EXPERT_FFN, T, k, E, H, F))
    if workspace is None:
        workspace = torch.empty(max(need, 1024), dtype=torch.uint8, device=x.device)
    _check(lib().moe_expert_ffn_gather(_ptr(x), T, _ptr(perm), int(k), _ptr(group_offsets), _ptr(group_expert),
                                       _ptr(rep_base), E, _ptr(w1), _ptr(w3), _ptr(w2), H, F, act_id,
                                       int(small_group_threshold), _ptr(y), _ptr(workspace), _ws_bytes(workspace),
                                       _stream(stream)), "moe_expert_ffn_gather")
    return y


def moe_replicate_weights(rep_base, w_all=None, group_slot=None, stream=None):
    """Fill the replica slots of w_all [2E-1, rows, cols] (slots 0..E-1 = the
    experts) from the device table rep_base [E+1]; returns group_slot [2E]."""
    torch = _torch()
    _dev(rep_base, torch.int32, "rep_base", 1)
    E = rep_base.numel() - 1
    rows = cols = 0
    if w_all is not None:
        _dev(w_all, torch.bfloat16, "w_all", 3)
        if w_all.shape[0] != 2 * E - 1:
            raise ValueError("w_all must hold 2E-1 slots")
        rows, cols = int(w_all.shape[1]), int(w_all.shape[2])
    if group_slot is None:
        group_slot = torch.empty(2 * E, dtype=torch.int32, device=rep_base.device)
    _out(group_slot, torch.int32, "group_slot", 2 * E)
    _check(lib().moe_replicate_weights(_ptr(rep_base), E, _ptr(w_all), rows, cols, _ptr(group_slot),
                                       _stream(stream)), "moe_replicate_weights")
    return group_slot


def moe_expert_ffn_slots(xp, group_offsets, group_slot, w1, w3, w2, act: str = "gelu",
                         small_group_threshold: int = 64, y=None, workspace=None, stream=None):
    """Grouped expert FFN where group g reads weight slot group_slot[g]."""
    torch = _torch()
    _dev(xp, torch.bfloat16, "xp", 2)
    _dev(group_offsets, torch.int32, "group_offsets", 1)
    _dev(group_slot, torch.int32, "group_slot", 1)
    A, H = xp.shape
    _dev(w1, torch.bfloat16, "w1", 3)
    _dev(w2, torch.bfloat16, "w2", 3)
    if w3 is not None:
        _dev(w3, torch.bfloat16, "w3", 3)
    S, H1, F = w1.shape
    if H1 != H or tuple(w2.shape) != (S, F, H) or (w3 is not None and w3.shape != w1.shape):
        raise ValueError("weight shapes must be w1/w3 [S,H,F], w2 [S,F,H]")
    G = group_slot.numel()
    _out(group_offsets, torch.int32, "group_offsets", G + 1)
    act_id = {"gelu": MOE_ACT_GELU, "swiglu": MOE_ACT_SWIGLU}[act]
    if y is None:
        y = torch.empty((A, H), dtype=torch.bfloat16, device=xp.device)
    _out(y, torch.bfloat16, "y", A * H, 2)
    need = int(lib().moe_workspace_bytes(MOE_OP_EXPERT_FFN, A, 1, max((G + 1) // 2, 1), H, F))
    if workspace is None:
        workspace = torch.empty(max(need, 1024), dtype=torch.uint8, device=xp.device)
    _check(lib().moe_expert_ffn_slots(_ptr(xp), _ptr(group_offsets), _ptr(group_slot), G, S, A, _ptr(w1), _ptr(w3),
                                      _ptr(w2), H, F, act_id, int(small_group_threshold), _ptr(y), _ptr(workspace),
                                      _ws_bytes(workspace), _stream(stream)), "moe_expert_ffn_slots")
    return y


def moe_expert_ffn_combine(xp, group_offsets, group_expert, rep_base, perm, w, w1, w3, w2, act: str = "gelu",
                           small_group_threshold: int = 64, out=None, workspace=None, stream=None):
    """moe_expert_ffn then moe_combine in one call, the combine in the second
    GEMM's epilogue: returns out [T, H] bf16."""
    torch = _torch()
    _dev(xp, torch.bfloat16, "xp", 2)
    _dev(group_offsets, torch.int32, "group_offsets", 1)
    _dev(perm, torch.int32, "perm", 1)
    _dev(w, torch.float32, "w", 2)
    _dev(w1, torch.bfloat16, "w1", 3)
    _dev(w2, torch.bfloat16, "w2", 3)
    if w3 is not None:
        _dev(w3, torch.bfloat16, "w3", 3)
    if group_expert is not None:
        _dev(group_expert, torch.int32, "group_expert", 1)
    if rep_base is not None:
        _dev(rep_base, torch.int32, "rep_base", 1)
    A, H = xp.shape
    T, k = w.shape
    E, H1, F = w1.shape
    if (H1 != H or tuple(w2.shape) != (E, F, H) or A != T * k
            or (w3 is not None and w3.shape != w1.shape)):
        raise ValueError("shapes: xp [T*k,H], w [T,k], w1/w3 [E,H,F], w2 [E,F,H]")
    _out(perm, torch.int32, "perm", A)
    _out(group_offsets, torch.int32, "group_offsets", (2 * E if group_expert is not None else E) + 1)
    act_id = {"gelu": MOE_ACT_GELU, "swiglu": MOE_ACT_SWIGLU}[act]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=xp.device)
    _out(out, torch.bfloat16, "out", T * H, 2)
    need = int(lib().moe_workspace_bytes(MOE_OP_EXPERT_FFN_COMBINE, T, k, E, H, F))
    if workspace is None:
        workspace = torch.empty(max(need, 1024), dtype=torch.uint8, device=xp.device)
    _check(lib().moe_expert_ffn_combine(_ptr(xp), _ptr(group_offsets), _ptr(group_expert), _ptr(rep_base), E,
                                        _ptr(perm), _ptr(w), T, k, _ptr(w1), _ptr(w3), _ptr(w2), H, F, act_id,
                                        int(small_group_threshold), _ptr(out), _ptr(workspace), _ws_bytes(workspace),
                                        _stream(stream)), "moe_expert_ffn_combine")
    return out


def moe_ffn_launches(A: int, E: int, H: int, F: int, act: str = "gelu", small_group_threshold: int = 64,
                     gather: bool = False) -> int:
    """Kernel launches of one FFN call under the current options."""
    act_id = {"gelu": MOE_ACT_GELU, "swiglu": MOE_ACT_SWIGLU}[act]
    return int(lib().moe_ffn_launches(int(A), int(E), int(H), int(F), act_id, int(small_group_threshold),
                                      int(bool(gather))))


def moe_layer_front_launches(T: int, E: int, k: int, has_prev: bool = True) -> int:
    """Kernel launches of one moe_layer_front call (T > 0) on the current
    device under the current options: 1 (one cooperative launch) or 2."""
    return int(lib().moe_layer_front_launches(int(T), int(E), int(k), int(bool(has_prev))))


MOE_BWD_ACCUMULATE_WGRAD = 1
MOE_BWD_WGRAD_BF16 = 2


def moe_ffn_backward(x, dout, w, y, perm, inv_perm, group_offsets, group_expert, w1, w3, w2, act: str = "gelu",
                     workspace=None, stream=None, out=None, accumulate: bool = False, wgrad_bf16: bool = False):
    """Backward of dispatch -> expert FFN -> combine for one routing.
    x, dout bf16 [T, H]; w f32 [T, k]; y bf16 [T*k, H] (the forward FFN
    output, or None: no dw); perm, inv_perm, group_offsets, group_expert as
    written by the dispatch.  Returns (dx bf16 [T, H], dw f32 [T, k] or None,
    dw1 f32 [E, H, F], dw3 f32 [E, H, F] or None, dw2 f32 [E, F, H]).
    `out` may give those five tensors to write into; accumulate=True adds
    this batch's weight gradients to what out's dw1, dw3, dw2 hold;
    wgrad_bf16=True returns the weight gradients rounded once to bf16."""
    torch = _torch()
    _dev(x, torch.bfloat16, "x", 2)
    _dev(dout, torch.bfloat16, "dout", 2)
    _dev(w, torch.float32, "w", 2)
    _dev(perm, torch.int32, "perm", 1)
    _dev(inv_perm, torch.int32, "inv_perm", 1)
    _dev(group_offsets, torch.int32, "group_offsets", 1)
    if group_expert is not None:
        _dev(group_expert, torch.int32, "group_expert", 1)
    _dev(w1, torch.bfloat16, "w1", 3)
    _dev(w2, torch.bfloat16, "w2", 3)
    if w3 is not None:
        _dev(w3, torch.bfloat16, "w3", 3)
    if y is not None:
        _dev(y, torch.bfloat16, "y", 2)
    T, H = x.shape
    k = w.shape[1]
    E, H1, F = w1.shape
    if (H1 != H or tuple(w2.shape) != (E, F, H) or tuple(dout.shape) != (T, H) or w.shape[0] != T
            or (w3 is not None and w3.shape != w1.shape)):
        raise ValueError("shapes: x, dout [T,H]; w [T,k]; w1/w3 [E,H,F]; w2 [E,F,H]")
    A = T * k
    _out(perm, torch.int32, "perm", A)
    _out(inv_perm, torch.int32, "inv_perm", A)
    _out(group_offsets, torch.int32, "group_offsets", (2 * E if group_expert is not None else E) + 1)
    if y is not None:
        _out(y, torch.bfloat16, "y", A * H)
    act_id = {"gelu": MOE_ACT_GELU, "swiglu": MOE_ACT_SWIGLU}[act]
    dev = x.device
    if accumulate and out is None:
        raise ValueError("accumulate=True needs `out`: the gradients to add to")
    if accumulate and wgrad_bf16:
        raise ValueError("bf16 weight gradients cannot be accumulated")
    gdt = torch.bfloat16 if wgrad_bf16 else torch.float32
    if out is None:
        f32 = dict(dtype=torch.float32, device=dev)
        out = (torch.empty((T, H), dtype=torch.bfloat16, device=dev),
               torch.empty((T, k), **f32) if y is not None else None,
               torch.empty((E, H, F), dtype=gdt, device=dev),
               torch.empty((E, H, F), dtype=gdt, device=dev) if act == "swiglu" else None,
               torch.empty((E, F, H), dtype=gdt, device=dev))
    dx, dw, dw1, dw3, dw2 = out
    if dx is not None:
        _out(dx, torch.bfloat16, "dx", T * H)
    if dw is not None:
        _out(dw, torch.float32, "dw", T * k)
    for nm, t in (("dw1", dw1), ("dw3", dw3), ("dw2", dw2)):
        if t is not None:
            _out(t, gdt, nm, E * H * F, 3)
    need = int(lib().moe_ffn_backward_workspace_bytes(T, k, E, H, F))
    if workspace is None:
        workspace = torch.empty(max(need, 1024), dtype=torch.uint8, device=dev)
    _check(lib().moe_ffn_backward(_ptr(x), _ptr(dout), _ptr(w), _ptr(y), _ptr(perm), _ptr(inv_perm), T, k,
                                  _ptr(group_offsets), _ptr(group_expert), E, _ptr(w1), _ptr(w3), _ptr(w2), H, F,
                                  act_id, _ptr(dx), _ptr(dw), _ptr(dw1), _ptr(dw3), _ptr(dw2),
                                  (MOE_BWD_ACCUMULATE_WGRAD if accumulate else 0)
                                  | (MOE_BWD_WGRAD_BF16 if wgrad_bf16 else 0), _ptr(workspace),
                                  _ws_bytes(workspace), _stream(stream)), "moe_ffn_backward")
    return dx, dw, dw1, dw3, dw2


def moe_ffn_backward_workspace_bytes(T: int, k: int, E: int, H: int, F: int) -> int:
    return int(lib().moe_ffn_backward_workspace_bytes(int(T), int(k), int(E), int(H), int(F)))


def moe_route_backward(logits, idx, dw, renorm: bool = True, out=None, stream=None):
    """dlogits f32 [T, E]: gradient of the gate weights w.r.t. the logits,
    the chosen experts held fixed."""
    torch = _torch()
    _dev(logits, torch.float32, "logits", 2)
    _dev(idx, torch.int32, "idx", 2)
    _dev(dw, torch.float32, "dw", 2)
    T, E = logits.shape
    k = idx.shape[1]
    if idx.shape[0] != T or tuple(dw.shape) != tuple(idx.shape):
        raise ValueError("shapes: logits [T,E], idx and dw [T,k]")
    if out is None:
        out = torch.empty((T, E), dtype=torch.float32, device=logits.device)
    _out(out, torch.float32, "dlogits", T * E, 2)
    _check(lib().moe_route_backward(_ptr(logits), _ptr(idx), _ptr(dw), T, E, k, int(bool(renorm)), _ptr(out),
                                    _stream(stream)), "moe_route_backward")
    return out


def moe_combine(y, inv_perm, w, out=None, stream=None):
    """out [T, H] bf16 = sum_r w[t,r] * y[inv_perm[t*k+r]]."""
    torch = _torch()
    _dev(y, torch.bfloat16, "y", 2)
    _dev(inv_perm, torch.int32, "inv_perm", 1)
    _dev(w, torch.float32, "w", 2)
    T, k = w.shape
    H = y.shape[1]
    if y.shape[0] < T * k:
        raise ValueError("y must hold the T*k dispatched rows")
    _out(inv_perm, torch.int32, "inv_perm", T * k)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    _out(out, torch.bfloat16, "out", T * H, 2)
    _check(lib().moe_combine(_ptr(y), _ptr(inv_perm), _ptr(w), T, k, H, _ptr(out), _stream(stream)), "moe_combine")
    return out


def moe_set_option(option: int, value: int):
    _check(lib().moe_set_option(int(option), int(value)), "moe_set_option")


def moe_get_option(option: int) -> int:
    v = ctypes.c_int(0)
    _check(lib().moe_get_option(int(option), ctypes.byref(v)), "moe_get_option")
    return int(v.value)


def moe_check(stream=None):
    """Synchronise the stream and raise if a kernel flagged an error."""
    _check(lib().moe_check(_stream(stream)), "moe_check")


def moe_error_word() -> int:
    w = ctypes.c_uint32(0)
    _check(lib().moe_error_word(ctypes.byref(w)), "moe_error_word")
    return int(w.value)

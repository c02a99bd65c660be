"""The C ABI without a GPU: the library loads, exports every function that
include/moe.h declares, and rejects bad arguments on the host before any CUDA
call (so these checks run on a machine with no device)."""
import ctypes
import os
import re
import subprocess

import pytest

import moe_expert_routing_02_b300 as M
from moe_expert_routing_02_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return M.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_seven_calls():
    names = declared_functions()
    for n in ["moe_route", "moe_stats_update", "moe_predict", "moe_replicate", "moe_dispatch",
              "moe_expert_ffn", "moe_combine"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", M.library_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(L, n) is not None
    # the binding knows every declared function
    assert sorted(M.EXPORTED_SYMBOLS) == declared_functions()


def test_library_is_sm103a_and_has_no_torch_in_abi(L):
    assert b"sm_103a" in L.moe_version()
    out = subprocess.run(["nm", "-D", "--undefined-only", M.library_path], capture_output=True, text=True).stdout
    assert "torch" not in out and "c10" not in out


def test_status_strings(L):
    for s in range(7):
        assert L.moe_status_string(s)
    assert L.moe_status_string(99) == b"unknown status"


def test_workspace_bytes(L):
    # dispatch: one int32 counter per (tile of 1024 assignments, expert) + 4E
    assert L.moe_workspace_bytes(M.MOE_OP_DISPATCH, 16384, 2, 16, 1024, 0) == (32 * 16 + 64) * 4
    # ffn: bf16 intermediate [A, F] rounded up to 1 KB, one uint32 counter per
    # 256-row block of the fused kernel (A/256 rounded up, + 2E + 1), plus 1 KB
    assert L.moe_workspace_bytes(M.MOE_OP_EXPERT_FFN, 256, 2, 8, 64, 128) == 512 * 128 * 2 + (2 + 16 + 1) * 4 + 1024
    assert L.moe_workspace_bytes(M.MOE_OP_EXPERT_FFN, 256, 2, 8, 64, 100) == 0   # F not a multiple of 64
    assert L.moe_workspace_bytes(99, 1, 1, 1, 64, 64) == 0
    assert L.moe_workspace_bytes(M.MOE_OP_DISPATCH, 16, 9, 16, 64, 64) == 0       # k > 8


P = ctypes.c_void_p
NULL = P(0)
FAKE = P(0x10000)      # never dereferenced: validation fails first
MISALIGNED = P(0x10004)


def test_route_rejects_bad_arguments(L):
    inv = M.MOE_ERR_INVALID
    assert L.moe_route(FAKE, 16, 0, 1, 1, FAKE, FAKE, NULL) == inv      # E < 1
    assert L.moe_route(FAKE, 16, 257, 1, 1, FAKE, FAKE, NULL) == inv    # E > 256
    assert L.moe_route(FAKE, 16, 8, 9, 1, FAKE, FAKE, NULL) == inv      # k > 8
    assert L.moe_route(FAKE, 16, 4, 5, 1, FAKE, FAKE, NULL) == inv      # k > E
    assert L.moe_route(FAKE, -1, 8, 2, 1, FAKE, FAKE, NULL) == inv      # T < 0
    assert L.moe_route(NULL, 16, 8, 2, 1, FAKE, FAKE, NULL) == inv      # null logits
    assert L.moe_route(MISALIGNED, 16, 8, 2, 1, FAKE, FAKE, NULL) == inv
    assert L.moe_route(FAKE, 1 << 29, 8, 8, 1, FAKE, FAKE, NULL) == inv  # T*k >= 2^31
    assert b"moe_route" in L.moe_last_error()
    assert L.moe_route(NULL, 0, 8, 2, 1, NULL, NULL, NULL) == M.MOE_OK  # empty batch: nothing to do


def test_dispatch_ffn_combine_reject_bad_arguments(L):
    inv = M.MOE_ERR_INVALID
    d = L.moe_dispatch
    assert d(FAKE, FAKE, 16, 2, 12, 8, NULL, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, NULL) == inv  # H % 8
    assert d(FAKE, FAKE, 16, 2, 64, 8, NULL, NULL, FAKE, FAKE, FAKE, FAKE, 1 << 20, NULL) == inv  # null offsets
    assert d(FAKE, FAKE, 16, 2, 64, 8, NULL, FAKE, FAKE, FAKE, NULL, FAKE, 1 << 20, NULL) == inv  # x without xp
    assert d(MISALIGNED, FAKE, 16, 2, 64, 8, NULL, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, NULL) == inv
    assert d(FAKE, FAKE, 16, 2, 64, 8, NULL, FAKE, FAKE, FAKE, FAKE, FAKE, 4, NULL) == M.MOE_ERR_WORKSPACE
    f = L.moe_expert_ffn
    args = [FAKE, FAKE, NULL, NULL, 8, 512, FAKE, NULL, FAKE, 64, 128, M.MOE_ACT_GELU, 64, FAKE, FAKE, 1 << 30, NULL]
    a = list(args); a[9] = 96
    assert f(*a) == inv                                   # H % 64
    a = list(args); a[11] = 7
    assert f(*a) == inv                                   # unknown activation
    a = list(args); a[11] = M.MOE_ACT_SWIGLU
    assert f(*a) == inv                                   # SwiGLU without w3
    a = list(args); a[14] = P(0x10400 + 8)
    assert f(*a) == inv                                   # workspace not 16-byte aligned
    a = list(args); a[15] = 1000
    assert f(*a) == M.MOE_ERR_WORKSPACE
    a = list(args); a[12] = -1
    assert f(*a) == inv
    c = L.moe_combine
    assert c(FAKE, FAKE, FAKE, 16, 0, 64, FAKE, NULL) == inv
    assert c(FAKE, FAKE, FAKE, 16, 2, 60, FAKE, NULL) == inv
    assert c(MISALIGNED, FAKE, FAKE, 16, 2, 64, FAKE, NULL) == inv
    assert c(NULL, NULL, NULL, 0, 2, 64, NULL, NULL) == M.MOE_OK


def test_stats_and_replicate_reject_bad_arguments(L):
    inv = M.MOE_ERR_INVALID
    h = P()
    assert L.moe_stats_create(ctypes.byref(h), 0, 8, 10, NULL) == inv
    assert L.moe_stats_create(ctypes.byref(h), 2, 300, 10, NULL) == inv
    assert L.moe_stats_create(ctypes.byref(h), 2, 8, 0, NULL) == inv
    assert L.moe_stats_create(None, 2, 8, 10, NULL) == inv
    assert L.moe_stats_update(NULL, 0, 0, FAKE, NULL, 4, 2, NULL, NULL) == inv
    assert L.moe_predict(NULL, 0, FAKE, NULL, NULL, NULL) == inv
    r = L.moe_replicate
    assert r(FAKE, 16, 100, 0, 5, -1, FAKE, FAKE, FAKE, NULL) == inv   # bad threshold
    assert r(FAKE, 16, 100, 6, 5, -2, FAKE, FAKE, FAKE, NULL) == inv   # bad cap
    assert r(FAKE, 16, -1, 6, 5, -1, FAKE, FAKE, FAKE, NULL) == inv    # negative total
    assert r(NULL, 16, 100, 6, 5, -1, FAKE, FAKE, FAKE, NULL) == inv
    assert L.moe_stats_bytes(NULL) == 0
    assert L.moe_stats_export(NULL, FAKE, 10) == inv
    assert L.moe_error_word(None) == inv
    assert L.moe_set_option(99, 0) == inv
    assert L.moe_set_option(M.MOE_OPT_FFN_KERNEL, 7) == inv
    assert L.moe_set_option(M.MOE_OPT_FFN_TIMEOUT_SELFTEST, 2) == inv
    v = ctypes.c_int(-1)
    assert L.moe_get_option(M.MOE_OPT_FFN_KERNEL, ctypes.byref(v)) == M.MOE_OK and v.value == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib
    monkeypatch.setattr(M, "_lib", None)
    monkeypatch.setattr(M, "library_path", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        M.lib()

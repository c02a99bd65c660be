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
    # the small-path SM split: 0 (no small-batch path) by default, -1..4096 accepted
    assert L.moe_get_option(M.MOE_OPT_FFN_SMALL_SMS, ctypes.byref(v)) == M.MOE_OK and v.value == 0
    assert L.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, -2) == inv
    assert L.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, 5000) == inv
    assert L.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, 24) == M.MOE_OK
    assert L.moe_get_option(M.MOE_OPT_FFN_SMALL_SMS, ctypes.byref(v)) == M.MOE_OK and v.value == 24
    assert L.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, 0) == M.MOE_OK
    # the one-launch front: off by default, 0 or 1
    assert L.moe_get_option(M.MOE_OPT_FRONT_ONE_LAUNCH, ctypes.byref(v)) == M.MOE_OK and v.value == 0
    assert L.moe_set_option(M.MOE_OPT_FRONT_ONE_LAUNCH, 2) == inv
    assert L.moe_set_option(M.MOE_OPT_FRONT_ONE_LAUNCH, 1) == M.MOE_OK
    assert L.moe_get_option(M.MOE_OPT_FRONT_ONE_LAUNCH, ctypes.byref(v)) == M.MOE_OK and v.value == 1
    assert L.moe_set_option(M.MOE_OPT_FRONT_ONE_LAUNCH, 0) == M.MOE_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib
    monkeypatch.setattr(M, "_lib", None)
    monkeypatch.setattr(M, "library_path", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        M.lib()


ALIGN16_NOT_256 = P(0x10010)


def test_fused_and_prediction_calls_reject_bad_arguments(L):
    inv = M.MOE_ERR_INVALID
    # moe_layer_front: a stats handle is required (its own checks need it)
    front = [FAKE, FAKE, 16, 8, 2, 64, 1, NULL, 0, 0, NULL, 1, 6, 5, -1, NULL, -1] + [FAKE] * 14 + [1 << 20, NULL]
    assert L.moe_layer_front(*front) == inv
    assert b"stats handle" in L.moe_last_error()
    assert L.moe_predict_decay(NULL, 0, 0, 0.5, FAKE, NULL, NULL, NULL) == inv
    rp = L.moe_replicate_predicted
    ok = [FAKE, 16, 1000, 6, 5, -1, -1, FAKE, FAKE, FAKE, FAKE, NULL]
    for pos, bad in ((1, 0), (1, 257), (2, 0), (2, 1 << 29), (3, 0), (4, 1025), (5, -2), (6, -2), (0, NULL),
                     (8, NULL)):
        a = list(ok); a[pos] = bad
        assert rp(*a) == inv, (pos, bad)
    nd = L.moe_dispatch_noalloc
    assert nd(NULL, FAKE, -1, 2, 64, 8, NULL, FAKE, FAKE, FAKE, NULL, NULL) == inv
    assert nd(NULL, FAKE, 16, 9, 64, 16, NULL, FAKE, FAKE, FAKE, NULL, NULL) == inv
    assert nd(NULL, FAKE, 1 << 17, 8, 64, 256, NULL, FAKE, FAKE, FAKE, NULL, NULL) == M.MOE_ERR_WORKSPACE


def test_ffn_variants_reject_bad_arguments(L):
    inv = M.MOE_ERR_INVALID
    gel, swi = M.MOE_ACT_GELU, M.MOE_ACT_SWIGLU
    # moe_expert_ffn_gather(x, T, perm, k, go, ge, rb, E, w1, w3, w2, H, F, act, small, y, ws, ws_bytes, stream)
    g = L.moe_expert_ffn_gather
    ok = [FAKE, 16, FAKE, 2, FAKE, NULL, NULL, 8, FAKE, NULL, FAKE, 64, 128, gel, 64, FAKE, FAKE, 1 << 30, NULL]
    for pos, bad in ((3, 0), (3, 9), (7, 1), (7, 300), (0, NULL), (2, NULL), (1, -1), (11, 96), (12, 100),
                     (13, 7), (14, -1), (13, swi), (15, NULL), (16, NULL), (8, MISALIGNED)):
        a = list(ok); a[pos] = bad
        assert g(*a) == inv, (pos, bad)
    a = list(ok); a[1] = 1 << 28; a[3] = 8
    assert g(*a) == inv                                   # T*k >= 2^31
    a = list(ok); a[17] = 64
    assert g(*a) == M.MOE_ERR_WORKSPACE
    a = list(ok); a[1] = 0
    assert g(*a) == M.MOE_OK                              # empty batch: nothing enqueued
    # moe_expert_ffn_combine(xp, go, ge, rb, E, perm, w, T, k, w1, w3, w2, H, F, act, small, out, ws, ws_bytes, st)
    c = L.moe_expert_ffn_combine
    ok = [FAKE, FAKE, NULL, NULL, 8, FAKE, FAKE, 16, 2, FAKE, NULL, FAKE, 64, 128, gel, 64, FAKE, FAKE, 1 << 30,
          NULL]
    for pos, bad in ((4, 0), (4, 257), (8, 0), (8, 9), (7, -1), (12, 100), (13, 32), (5, NULL), (6, NULL),
                     (16, NULL), (17, NULL), (16, MISALIGNED), (17, ALIGN16_NOT_256), (0, NULL), (14, 7),
                     (14, swi)):
        a = list(ok); a[pos] = bad
        assert c(*a) == inv, (pos, bad)
    a = list(ok); a[18] = 256
    assert c(*a) == M.MOE_ERR_WORKSPACE
    a = list(ok); a[7] = 0
    assert c(*a) == M.MOE_OK
    # moe_expert_ffn_slots(xp, go, group_slot, G, n_slots, A, w1, w3, w2, H, F, act, small, y, ws, ws_bytes, st)
    s = L.moe_expert_ffn_slots
    ok = [FAKE, FAKE, FAKE, 9, 15, 32, FAKE, NULL, FAKE, 64, 128, gel, 64, FAKE, FAKE, 1 << 30, NULL]
    for pos, bad in ((2, NULL), (3, 0), (4, 0), (5, -1), (9, 32), (11, 5), (0, NULL)):
        a = list(ok); a[pos] = bad
        assert s(*a) == inv, (pos, bad)
    a = list(ok); a[5] = 0
    assert s(*a) == M.MOE_OK
    # moe_replicate_weights(rep_base, E, w_all, rows, cols, group_slot, stream)
    r = L.moe_replicate_weights
    assert r(FAKE, 0, FAKE, 64, 64, NULL, NULL) == inv
    assert r(NULL, 8, FAKE, 64, 64, NULL, NULL) == inv
    assert r(FAKE, 8, FAKE, 3, 4, NULL, NULL) == inv       # rows*cols not a multiple of 8
    assert r(FAKE, 8, FAKE, 0, 64, NULL, NULL) == inv
    assert r(FAKE, 8, MISALIGNED, 64, 64, NULL, NULL) == inv


def test_backward_calls_reject_bad_arguments(L):
    inv = M.MOE_ERR_INVALID
    gel, swi = M.MOE_ACT_GELU, M.MOE_ACT_SWIGLU
    wsb = L.moe_ffn_backward_workspace_bytes
    assert wsb(16, 2, 8, 96, 128) == 0 and wsb(16, 0, 8, 64, 128) == 0 and wsb(16, 2, 300, 64, 128) == 0
    assert 0 < wsb(16, 2, 8, 64, 128) < wsb(4096, 2, 8, 64, 128)
    need = wsb(16, 2, 8, 64, 128)
    # moe_ffn_backward(x, dout, w, y, perm, inv, T, k, go, ge, E, w1, w3, w2, H, F, act, dx, dw, dw1, dw3, dw2,
    #                  flags, ws, ws_bytes, stream)
    b = L.moe_ffn_backward
    ok = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 2, FAKE, NULL, 8, FAKE, NULL, FAKE, 64, 128, gel, FAKE, FAKE,
          FAKE, NULL, FAKE, 0, FAKE, 1 << 30, NULL]
    for pos, bad in ((6, -1), (7, 0), (7, 9), (10, 1), (10, 300), (14, 96), (15, 100), (16, 7), (22, 4),
                     (22, M.MOE_BWD_ACCUMULATE_WGRAD | M.MOE_BWD_WGRAD_BF16), (8, NULL), (11, NULL), (13, NULL),
                     (19, NULL), (21, NULL), (23, NULL), (16, swi), (0, NULL), (1, NULL), (2, NULL), (4, NULL),
                     (5, NULL), (17, NULL), (18, NULL), (0, MISALIGNED), (17, MISALIGNED), (19, MISALIGNED),
                     (23, ALIGN16_NOT_256)):
        a = list(ok); a[pos] = bad
        assert b(*a) == inv, (pos, bad)
    a = list(ok); a[24] = need - 1
    assert b(*a) == M.MOE_ERR_WORKSPACE
    # moe_route_backward(logits, idx, dw, T, E, k, renorm, dlogits, stream)
    rb = L.moe_route_backward
    ok = [FAKE, FAKE, FAKE, 16, 8, 2, 1, FAKE, NULL]
    for pos, bad in ((3, -1), (4, 0), (4, 257), (5, 0), (5, 9), (0, NULL), (1, NULL), (2, NULL), (7, NULL)):
        a = list(ok); a[pos] = bad
        assert rb(*a) == inv, (pos, bad)
    a = list(ok); a[3] = 0
    assert rb(*a) == M.MOE_OK


def test_ffn_launch_count_rule(L):
    """The FFN's launch count: the fused kernel (one launch) for
    CTA-pair-sized batches of experts of at most 16 MB, two GEMM launches
    otherwise (the gather path, larger experts, small batches), plus the two
    small-batch launches when the threshold is positive and the small-batch
    path is on (MOE_OPT_FFN_SMALL_SMS not 0; off by default)."""
    n = L.moe_ffn_launches
    gel, swi = M.MOE_ACT_GELU, M.MOE_ACT_SWIGLU
    for opt, small in ((0, 0), (-1, 2), (8, 2)):
        assert L.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, opt) == M.MOE_OK
        assert n(32768, 16, 1024, 2048, gel, 64, 0) == 1 + small    # 8 MB experts: fused
        assert n(32768, 16, 1024, 2048, gel, 0, 0) == 1
        assert n(32768, 16, 1024, 2048, gel, 64, 1) == 2 + small    # gather: two GEMM launches
        assert n(32768, 16, 1024, 8192, gel, 64, 0) == 2 + small    # 32 MB experts
        assert n(32768, 16, 1024, 2048, swi, 64, 0) == 1 + small    # 12 MB
        assert n(32768, 16, 1024, 4096, swi, 64, 0) == 2 + small    # 24 MB
        assert n(1000, 16, 1024, 2048, gel, 64, 0) == 2 + small     # A < 256 E: single-CTA GEMMs
    assert L.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, 0) == M.MOE_OK
    assert n(0, 16, 1024, 2048, gel, 64, 0) == 0
    assert n(32768, 16, 96, 2048, gel, 64, 0) == 0
    assert n(32768, 16, 1024, 2000, gel, 64, 0) == 0
    assert n(32768, 16, 1024, 2048, 7, 64, 0) == 0
    assert n(32768, 16, 1024, 2048, gel, -1, 0) == 0


def test_header_is_plain_c_and_a_c_program_links_and_calls_the_library(L, tmp_path):
    """include/moe.h compiles as C99 and C++17, and a C program (no torch,
    no Python) links libmoe.so and calls host-only entry points."""
    import shutil
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    for lang, std in (("c", "-std=c99"), ("c++", "-std=c++17")):
        r = subprocess.run([gcc if lang == "c" else (shutil.which("g++") or gcc), std, "-Wall", "-Wextra",
                            "-Werror", "-fsyntax-only", "-x", lang, HEADER], capture_output=True, text=True)
        assert r.returncode == 0, (lang, r.stderr)
    src = tmp_path / "use_moe.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "moe.h"
int main(void) {
  /* host-only calls: no device is touched */
  size_t ws = moe_workspace_bytes(MOE_OP_DISPATCH, 16384, 2, 16, 1024, 0);
  moe_status bad = moe_route(NULL, 16, 0, 1, 1, NULL, NULL, NULL);   /* E < 1: refused on the host */
  printf("%s|%zu|%d|%s|%d\n", strstr(moe_version(), "sm_103a") ? "sm_103a" : "?", ws, (int)bad,
         moe_status_string(MOE_ERR_INVALID), moe_ffn_launches(32768, 16, 1024, 2048, MOE_ACT_GELU, 64, 0));
  return 0;
}
''')
    libdir = os.path.dirname(M.library_path)
    exe = tmp_path / "use_moe"
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
                        f"-L{libdir}", "-l:libmoe.so", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    ver, ws, bad, msg, n = out.stdout.strip().split("|")
    assert ver == "sm_103a" and int(ws) == (32 * 16 + 64) * 4
    assert int(bad) == M.MOE_ERR_INVALID and msg and int(n) == 1   # fused; no small-batch path by default


def test_every_entry_point_names_its_passage():
    """Each declaration block of include/moe.h cites the passage of the pages
    it follows (a review, blog or summary, by section), or says that the
    pages have no counterpart / that the call is host-only bookkeeping."""
    src = open(HEADER).read()
    marks = ("review", "blog", "summary", "Prediction Is All", "no counterpart", "Host only", "host only")
    for block in re.split(r"(?=/\* -{10,})", src):
        decls = re.findall(r"\b(moe_\w+)\s*\(", re.sub(r"/\*.*?\*/", "", block, flags=re.S))
        if decls:
            assert any(m in block for m in marks), decls


def test_front_launch_count_refusals(L):
    """moe_layer_front_launches answers 0 for an empty batch and for sizes the
    front refuses, before it queries any device."""
    f = L.moe_layer_front_launches
    assert f(0, 16, 2, 1) == 0          # empty batch: the separate calls run instead
    assert f(-1, 16, 2, 1) == 0
    assert f(1024, 0, 2, 1) == 0        # E out of range
    assert f(1024, 257, 2, 1) == 0
    assert f(1024, 16, 0, 1) == 0       # k out of range
    assert f(1024, 4, 8, 1) == 0        # k > E

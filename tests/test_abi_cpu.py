"""CPU checks of the C ABI: the library builds for sm_103a, loads without a GPU, exports every function
declared in include/specverify.h, and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")
INTERNAL = os.path.join(ROOT, "speculative_decoding_verification_target_gb300", "csrc", "specverify_internal.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_target_gb300 import _build
    _build.build()
    import speculative_decoding_verification_target_gb300 as sv
    return sv.load()


def declared_functions(path=HEADER):
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("spec_verify", "spec_counterfactual_gamma", "spec_cactus_verify", "spec_workspace_size",
              "spec_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    import speculative_decoding_verification_target_gb300 as sv
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
    assert set(sv.EXPORTS) == set(names)


def test_test_hooks_are_outside_the_abi(lib):
    """The tuning hooks live in an internal header: exported, but not declared by the C ABI header."""
    import speculative_decoding_verification_target_gb300 as sv
    hooks = declared_functions(INTERNAL)
    assert set(hooks) == set(sv.TEST_HOOKS)
    assert not set(hooks) & set(declared_functions())
    for n in hooks:
        assert hasattr(lib, n), n


def test_workspace_size(lib):
    import speculative_decoding_verification_target_gb300 as sv

    def expect(B, K, V):
        # header + 8-byte row partials: the statistics pass's segments (fewer than min(warps, pieces) + rows,
        # 1024 CTAs x 16 warps at most) or the gamma kernel's one pair per row of the 2K + 1 of a sequence
        rows = B * (2 * K + 1)
        pieces = rows * ((V + 2047) // 2048)
        return (256 + (min(pieces, 1024 * 16) + rows) * 8 + 15) // 16 * 16

    for B, K, V, N in ((64, 5, 128256, 1), (32, 5, 128256, 7), (256, 8, 151936, 21), (4, 5, 1000, 1), (1, 1, 1, 1)):
        assert sv.workspace_size(B, K, V, N) == expect(B, K, V)
    base = sv.workspace_size(64, 5, 128256, 1)
    assert sv.workspace_size(128, 5, 128256, 1) > base
    assert sv.workspace_size(64, 8, 128256, 1) > base
    assert sv.workspace_size(64, 5, 151936, 1) >= base
    assert sv.workspace_size(0, 5, 1000, 1) == 256


def _call_verify(lib, **kw):
    a = dict(target=1 << 20, draft=1 << 21, dtype=0, tokens=1 << 22, seeds=1 << 23, B=2, K=3, V=1000, T=1.0,
             acc=1 << 24, out=1 << 25, diag=None, ws=1 << 26, wsb=1 << 20, stream=None)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.spec_verify(P(a["target"]), P(a["draft"]), a["dtype"], P(a["tokens"]), P(a["seeds"]), a["B"],
                           a["K"], a["V"], ctypes.c_float(a["T"]), P(a["acc"]), P(a["out"]),
                           P(a["diag"]) if a["diag"] else None, P(a["ws"]), a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(K=0), 1), (dict(K=65), 1), (dict(V=0), 1), (dict(V=262145), 1), (dict(B=-1), 1), (dict(T=0.0), 3),
    (dict(T=-1.0), 1), (dict(T=float("inf")), 1), (dict(T=float("nan")), 1), (dict(dtype=7), 1),
    (dict(target=0), 1), (dict(tokens=0), 1), (dict(ws=0), 1), (dict(ws=(1 << 26) + 4), 1), (dict(wsb=16), 1),
])
def test_host_validation(lib, kw, code):
    assert _call_verify(lib, **kw) == code
    assert lib.spec_last_error()


def test_B_zero_returns_ok_without_gpu(lib):
    assert _call_verify(lib, B=0, target=0, draft=0, tokens=0, seeds=0, acc=0, out=0, ws=0) == 0


def test_counterfactual_and_cactus_validation(lib):
    P = ctypes.c_void_p
    f = ctypes.c_float
    good = P(1 << 20)
    # selected out of range
    rc = lib.spec_counterfactual_gamma(good, good, 0, 3, 2, 2, 100, f(1.0), good, None, 3, good, good, good, good,
                                       None, P(1 << 26), 1 << 20, None)
    assert rc == 1
    rc = lib.spec_counterfactual_gamma(good, good, 0, 0, 2, 2, 100, f(1.0), good, None, -1, None, None, None, None,
                                       None, P(1 << 26), 1 << 20, None)
    assert rc == 1   # N = 0
    rc = lib.spec_cactus_verify(good, good, 0, good, good, 2, 2, 100, f(1.0), f(-0.5), good, good, None, None,
                                P(1 << 26), 1 << 20, None)
    assert rc == 1
    rc = lib.spec_cactus_verify(good, good, 0, good, good, 2, 2, 100, f(1.0), f(float("nan")), good, good, None,
                                None, P(1 << 26), 1 << 20, None)
    assert rc == 1


def test_stats_grid_hook(lib):
    assert lib.spec_debug_set_stats_grid(-1) == -1
    assert lib.spec_debug_set_stats_grid(1025) == -1
    assert lib.spec_debug_set_stats_grid(1024) == 0
    assert lib.spec_debug_set_stats_grid(7) == 0
    assert lib.spec_debug_set_stats_grid(0) == 0


def test_static_scratch_entry_refuses_oversized_calls_without_a_gpu(lib):
    # the static-scratch variant checks its size limit before any CUDA call
    P = ctypes.c_void_p
    good = P(1 << 20)
    st = ctypes.c_uint32(0)
    rc = lib.spec_verify_static(good, good, 0, good, good, 40000, 64, 262144, ctypes.c_float(1.0), good, good, None,
                                ctypes.byref(st), None)
    assert rc == 3
    assert b"static region" in lib.spec_last_error()
    rc = lib.spec_verify_static(None, None, 0, None, None, 0, 5, 1000, ctypes.c_float(1.0), None, None, None, None,
                                None)
    assert rc == 0   # B = 0 is a no-op
    rc = lib.spec_verify_static(good, good, 0, good, good, 2, 0, 1000, ctypes.c_float(1.0), good, good, None, None,
                                None)
    assert rc == 1


def test_no_cpu_fallback(lib, tmp_path):
    """The product path has no CPU route: host tensors are refused before any call, and a missing library
    makes loading fail loudly instead of computing anything elsewhere."""
    import torch
    import speculative_decoding_verification_target_gb300 as sv
    B, K, V = 2, 3, 64
    t = torch.zeros((B, K + 1, V), dtype=torch.float32)
    d = torch.zeros((B, K, V), dtype=torch.float32)
    tok = torch.zeros((B, K), dtype=torch.int32)
    seeds = torch.zeros(B, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sv.verify(t, d, tok, seeds)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sv.cactus_verify(t, d, tok, seeds, 0.5)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sv.greedy_verify(t, tok)
    saved_path, saved_lib = sv._build.LIB, sv._lib
    try:
        sv._build.LIB = str(tmp_path / "missing" / "libspecverify.so")
        sv._lib = None
        with pytest.raises(ImportError, match="no CPU fallback"):
            sv.load()
    finally:
        sv._build.LIB, sv._lib = saved_path, saved_lib


def test_filter_workspace_size(lib):
    """spec_verify_filtered's workspace: spec_verify's, then one float threshold and one float pair (the kept
    logits' max and sum) per target and draft row, then per target row a count and up to 1024 kept logits
    (index and value) for the draw, each region on 256 bytes. No copy of the logits."""
    import speculative_decoding_verification_target_gb300 as sv
    up = lambda x: (x + 255) // 256 * 256
    for B, K, V in ((64, 5, 128256), (4, 3, 1000), (1, 64, 262144), (3, 1, 7)):
        rows, rows_a = B * (2 * K + 1), B * (K + 1)
        thr = up(sv.workspace_size(B, K, V, 1))
        ms = up(thr + 4 * rows)
        ln = up(ms + 8 * rows)
        li = up(ln + 4 * rows_a)
        lx = up(li + 4 * 1024 * rows_a)
        for dt in (0, 1):
            assert lib.spec_filter_workspace_size(B, K, V, dt) == up(lx + 4 * 1024 * rows_a)
        if V >= 100000:   # a few percent of the bf16 logits it filters
            assert lib.spec_filter_workspace_size(B, K, V, 0) < 2 * V * rows // 20
    assert lib.spec_filter_workspace_size(4, 3, 0, 0) == 0
    assert lib.spec_filter_workspace_size(4, 3, 1000, 7) == 0
    assert lib.spec_filter_workspace_size(-1, 3, 1000, 0) == 0


@pytest.mark.parametrize("top_k,top_p,wsb,code", [
    (-1, 1.0, 1 << 20, 1), (5, 0.0, 1 << 20, 1), (5, 1.5, 1 << 20, 1), (5, float("nan"), 1 << 20, 1),
    (5, 0.9, 64, 1),
])
def test_filtered_host_validation(lib, top_k, top_p, wsb, code):
    P = ctypes.c_void_p
    r = lib.spec_verify_filtered(P(1 << 20), P(1 << 21), 0, P(1 << 22), P(1 << 23), 2, 3, 1000, ctypes.c_float(1.0),
                                 top_k, ctypes.c_float(top_p), P(1 << 24), P(1 << 25), None, P(1 << 26), wsb, None)
    assert r == code
    assert lib.spec_last_error()

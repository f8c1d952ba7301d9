"""fp64 CPU oracle for speculative-sampling verification -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``spec_oracle.c`` (plain C, fp64); this module compiles it with gcc and
marshals numpy arrays through ctypes. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path never does.

Logit arrays are numpy ``uint16`` (bf16 bit patterns) or ``float32``; the C side converts every
element exactly to double.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py`` against what the pages
fix (the cat/dog/fish worked example of the lossless-proof tutorial, its perfect-draft and
disjoint-support special cases, the two pitfalls as mutations a chi-square test must reject, exact
enumeration of output laws, the Cactus closed-form invariants) and against the published Philox4x32-10
known-answer vectors.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB = os.path.join(_HERE, "libspec_oracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP32 = 1


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into libspec_oracle.so next to it (gcc, OpenMP). Returns the path."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + ".tmp.%d" % os.getpid()
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    i32, u32, u64, f64 = ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double
    lib.spec_oracle_philox4x32_10.argtypes = [P, P, P]
    lib.spec_oracle_philox4x32_10.restype = None
    lib.spec_oracle_uniform.argtypes = [u64, u32, u32, u32]
    lib.spec_oracle_uniform.restype = f64
    lib.spec_oracle_softmax.argtypes = [P, i32, f64, P]
    lib.spec_oracle_softmax.restype = None
    lib.spec_oracle_inverse_cdf.argtypes = [P, i32, f64, P]
    lib.spec_oracle_inverse_cdf.restype = i32
    lib.spec_oracle_sample_one.argtypes = [P, P, i32, i32, f64, f64, i32, P, P, P, P, P]
    lib.spec_oracle_sample_one.restype = i32
    lib.spec_oracle_cactus_h.argtypes = [P, i32, i32, f64, P]
    lib.spec_oracle_cactus_h.restype = f64
    lib.spec_oracle_verify.argtypes = [i32, P, P, P, P, P, i32, i32, i32, f64, i32, P, P, P, P, P, i32]
    lib.spec_oracle_verify.restype = i32
    lib.spec_oracle_greedy.argtypes = [i32, P, P, i32, i32, i32, P, P, i32]
    lib.spec_oracle_greedy.restype = i32
    lib.spec_oracle_accept_length.argtypes = [P, i32, i32, i32, P, P]
    lib.spec_oracle_accept_length.restype = None
    lib.spec_oracle_normalhedge.argtypes = [P, P, P, i32]
    lib.spec_oracle_normalhedge.restype = i32
    lib.spec_oracle_normalhedge_scale.argtypes = [P, i32]
    lib.spec_oracle_normalhedge_scale.restype = f64
    lib.spec_oracle_hedge_feedback.argtypes = [P, P, i32, i32, i32, i32, i32, P, P]
    lib.spec_oracle_hedge_feedback.restype = i32
    lib.spec_oracle_filter_row.argtypes = [P, i32, f64, i32, f64, P, P, P]
    lib.spec_oracle_filter_row.restype = f64
    lib.spec_oracle_verify_filtered.argtypes = [i32, P, P, P, P, i32, i32, i32, f64, i32, f64, P, P, P, P, P, P, P]
    lib.spec_oracle_verify_filtered.restype = i32
    lib.spec_oracle_cactus.argtypes = [i32, P, P, P, P, P, i32, i32, i32, f64, f64, P, P, P, P, P, P, i32]
    lib.spec_oracle_cactus.restype = i32
    lib.spec_oracle_cactus_ex.argtypes = [i32, P, P, P, P, P, i32, i32, i32, f64, f64, i32, P, P, P, P, P, P, i32]
    lib.spec_oracle_cactus_ex.restype = i32
    lib.spec_oracle_cactus_kl.argtypes = [f64, f64]
    lib.spec_oracle_cactus_kl.restype = f64
    lib.spec_oracle_cactus_gamma_kl.argtypes = [f64, f64]
    lib.spec_oracle_cactus_gamma_kl.restype = f64
    lib.spec_oracle_cactus_h_mode.argtypes = [P, i32, i32, f64, i32, P]
    lib.spec_oracle_cactus_h_mode.restype = f64
    lib.spec_oracle_counterfactual.argtypes = [i32, P, P, i32, i32, i32, i32, f64, P, P, i32, P, P, P,
                                               P, P, P, P, P, i32]
    lib.spec_oracle_counterfactual.restype = i32
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, BF16
    if a.dtype == np.float32:
        return a, FP32
    raise TypeError("logits must be uint16 (bf16 bit patterns) or float32, got %s" % a.dtype)


def philox4x32_10(ctr, key):
    """Philox4x32-10 block: 4 x uint32 counter, 2 x uint32 key -> 4 x uint32."""
    lib = _load()
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib.spec_oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, seq: int, pos: int, stream: int) -> float:
    return _load().spec_oracle_uniform(seed, seq, pos, stream)


def softmax(x, T: float = 1.0):
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    p = np.empty_like(x)
    lib.spec_oracle_softmax(_ptr(x), x.size, T, _ptr(p))
    return p


def inverse_cdf(w, target: float):
    lib = _load()
    w = np.ascontiguousarray(w, dtype=np.float64)
    m = np.zeros(1)
    x = lib.spec_oracle_inverse_cdf(_ptr(w), w.size, target, _ptr(m))
    return x, float(m[0])


def sample_one(h, pd, t: int, r: float, u: float, mutation: int = 0):
    """One SpecSampleOne step. Returns (token, accepted, Z, accept_margin, cdf_margin)."""
    lib = _load()
    h = np.ascontiguousarray(h, dtype=np.float64)
    pd = np.ascontiguousarray(pd, dtype=np.float64)
    acc = np.zeros(1, dtype=np.int32)
    z = np.zeros(1)
    am = np.zeros(1)
    cm = np.zeros(1)
    scratch = np.empty(h.size)
    tok = lib.spec_oracle_sample_one(_ptr(h), _ptr(pd), h.size, t, r, u, mutation, _ptr(acc), _ptr(z),
                                     _ptr(am), _ptr(cm), _ptr(scratch))
    return tok, bool(acc[0]), float(z[0]), float(am[0]), float(cm[0])


def cactus_h(pt, n: int, delta: float, exact: bool = False):
    """Cactus target distribution for candidate n (Taylor gamma*, or the root of the divergence constraint
    with exact=True). Returns (h, gamma_star)."""
    lib = _load()
    pt = np.ascontiguousarray(pt, dtype=np.float64)
    h = np.empty_like(pt)
    g = lib.spec_oracle_cactus_h_mode(_ptr(pt), pt.size, n, delta, 1 if exact else 0, _ptr(h))
    return h, g


def cactus_kl(q: float, g: float) -> float:
    """KL(h || target) of the Cactus target with h_n = g for a candidate of target probability q."""
    return _load().spec_oracle_cactus_kl(q, g)


def cactus_gamma_kl(q: float, delta: float) -> float:
    """gamma* as the root of the divergence constraint (no Taylor step), clamped to [q, 1]."""
    return _load().spec_oracle_cactus_gamma_kl(q, delta)


def _t32(temperature):
    """A temperature or a divergence budget as the C ABI of the CUDA path receives it (a 32-bit float), so
    that both sides compute with the same number."""
    return float(np.float32(temperature))


def _seq_index(seq_index, B):
    if seq_index is None:
        return None
    s = np.ascontiguousarray(seq_index, dtype=np.int32)
    assert s.shape == (B,)
    return s


def verify(target, draft, tokens, seeds, temperature=1.0, seq_index=None, mutation=0, nthreads=0):
    """Standard speculative sampling. target [B,K+1,V], draft [B,K,V], tokens [B,K], seeds [B]."""
    lib = _load()
    target, dt = _logits(target)
    draft, dd = _logits(draft)
    assert dt == dd
    B, K1, V = target.shape
    K = K1 - 1
    assert draft.shape == (B, K, V)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    seeds = np.ascontiguousarray(seeds, dtype=np.uint64)
    si = _seq_index(seq_index, B)
    out = dict(accept_len=np.zeros(B, np.int32), out_tokens=np.zeros((B, K + 1), np.int32),
               diag=np.zeros((B, K, 4)), accept_margin=np.zeros((B, K)), cdf_margin=np.zeros(B))
    rc = lib.spec_oracle_verify(dt, _ptr(target), _ptr(draft), _ptr(tokens), _ptr(seeds), _ptr(si), B, K, V,
                                _t32(temperature), mutation, _ptr(out["accept_len"]),
                                _ptr(out["out_tokens"]), _ptr(out["diag"]), _ptr(out["accept_margin"]),
                                _ptr(out["cdf_margin"]), nthreads)
    if rc != 0:
        raise ValueError("oracle verify rejected its arguments")
    return out


def greedy(target, tokens, nthreads=0):
    """Greedy verification (temperature 0): accept a draft token iff it is the target row's argmax (smallest
    index among ties); emit the argmax of the first rejecting row, or of row K. target [B,K+1,V]."""
    lib = _load()
    target, dt = _logits(target)
    B, K1, V = target.shape
    K = K1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    out = dict(accept_len=np.zeros(B, np.int32), out_tokens=np.zeros((B, K + 1), np.int32))
    rc = lib.spec_oracle_greedy(dt, _ptr(target), _ptr(tokens), B, K, V, _ptr(out["accept_len"]),
                                _ptr(out["out_tokens"]), nthreads)
    if rc != 0:
        raise ValueError("oracle greedy rejected its arguments")
    return out


def accept_length(gamma):
    """HedgeSpec accept-length estimate and loss from gamma [N, B, K] (reading: 1 + sum_k prod_{j<=k} gamma_j;
    the page's display is missing). Returns (est [N, B], loss [N, B])."""
    lib = _load()
    g = np.ascontiguousarray(gamma, dtype=np.float64)
    N, B, K = g.shape
    est = np.empty((N, B))
    loss = np.empty((N, B))
    lib.spec_oracle_accept_length(_ptr(g), N, B, K, _ptr(est), _ptr(loss))
    return est, loss


def normalhedge(regret, loss, weights):
    """One NormalHedge round (Chaudhuri, Freund, Hsu 2009): regret += (weights . loss) - loss, then the new
    weights. Returns (regret, weights, c) as new arrays (c = 0 when no regret is positive)."""
    lib = _load()
    R = np.array(regret, dtype=np.float64)
    p = np.array(weights, dtype=np.float64)
    l_ = np.ascontiguousarray(loss, dtype=np.float64)
    if lib.spec_oracle_normalhedge(_ptr(R), _ptr(l_), _ptr(p), R.size) != 0:
        raise ValueError("normalhedge: N must be in [1, 64]")
    return R, p, lib.spec_oracle_normalhedge_scale(_ptr(R), R.size)


def hedge_feedback(gamma, accept_len, objective=0):
    """NormalHedge under delayed, censored feedback, one learner per sequence (reading of the HedgeSpec notes'
    Key design 3; see spec_oracle_hedge_feedback). gamma [T, N, B, K] (the counterfactual gamma of T rounds),
    accept_len [T, B]; objective 0: loss 1 - gamma per revealed level, 1: the accept-length loss over a window
    of K revealed levels. Returns (weights [T, B, N] after each round, applied [T, B])."""
    lib = _load()
    g = np.ascontiguousarray(gamma, dtype=np.float64)
    T, N, B, K = g.shape
    L = np.ascontiguousarray(accept_len, dtype=np.int32)
    assert L.shape == (T, B)
    w = np.zeros((T, B, N))
    a = np.zeros((T, B), np.int32)
    if lib.spec_oracle_hedge_feedback(_ptr(g), _ptr(L), T, N, B, K, int(objective), _ptr(w), _ptr(a)) != 0:
        raise ValueError("hedge_feedback rejected its arguments")
    return w, a


def filter_row(x, temperature=1.0, top_k=0, top_p=1.0):
    """Standardised-sampling filter of one row of logits: top-k then top-p, ties at a threshold kept.
    Returns (filtered logits with -inf outside the kept set, threshold, top-p margin)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    sc = np.empty_like(x)
    m = np.zeros(1)
    thr = lib.spec_oracle_filter_row(_ptr(x), x.size, _t32(temperature), int(top_k), float(top_p), _ptr(out),
                                     _ptr(m), _ptr(sc))
    return out, thr, float(m[0])


def verify_filtered(target, draft, tokens, seeds, temperature=1.0, top_k=0, top_p=1.0):
    """Standard speculative sampling on the standardised rows (every target and draft row filtered by
    filter_row with the same temperature, top_k and top_p). Adds thr and pmargin [B*(K+1) + B*K] (target
    rows, then draft rows) to the verify outputs."""
    lib = _load()
    target, dt = _logits(target)
    draft, dd = _logits(draft)
    assert dt == dd
    B, K1, V = target.shape
    K = K1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    seeds = np.ascontiguousarray(seeds, dtype=np.uint64)
    R = B * (2 * K + 1)
    out = dict(accept_len=np.zeros(B, np.int32), out_tokens=np.zeros((B, K + 1), np.int32),
               diag=np.zeros((B, K, 4)), accept_margin=np.zeros((B, K)), cdf_margin=np.zeros(B),
               thr=np.zeros(R), pmargin=np.zeros(R))
    rc = lib.spec_oracle_verify_filtered(dt, _ptr(target), _ptr(draft), _ptr(tokens), _ptr(seeds), B, K, V,
                                         _t32(temperature), int(top_k), float(top_p), _ptr(out["accept_len"]),
                                         _ptr(out["out_tokens"]), _ptr(out["diag"]), _ptr(out["accept_margin"]),
                                         _ptr(out["cdf_margin"]), _ptr(out["thr"]), _ptr(out["pmargin"]))
    if rc != 0:
        raise ValueError("oracle verify_filtered rejected its arguments")
    return out


def cactus(target, draft, tokens, seeds, delta, temperature=1.0, seq_index=None, nthreads=0, exact=False):
    """Cactus constrained acceptance; same layout as verify plus delta (exact=True: gamma* as the root of the
    divergence constraint instead of its Taylor closed form)."""
    lib = _load()
    target, dt = _logits(target)
    draft, dd = _logits(draft)
    assert dt == dd
    B, K1, V = target.shape
    K = K1 - 1
    assert draft.shape == (B, K, V)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    seeds = np.ascontiguousarray(seeds, dtype=np.uint64)
    si = _seq_index(seq_index, B)
    out = dict(accept_len=np.zeros(B, np.int32), out_tokens=np.zeros((B, K + 1), np.int32),
               diag=np.zeros((B, K, 4)), gamma_star=np.zeros((B, K)), accept_margin=np.zeros((B, K)),
               cdf_margin=np.zeros(B))
    rc = lib.spec_oracle_cactus_ex(dt, _ptr(target), _ptr(draft), _ptr(tokens), _ptr(seeds), _ptr(si), B, K, V,
                                _t32(temperature), _t32(delta), 1 if exact else 0, _ptr(out["accept_len"]),
                                _ptr(out["out_tokens"]), _ptr(out["diag"]), _ptr(out["gamma_star"]),
                                _ptr(out["accept_margin"]), _ptr(out["cdf_margin"]), nthreads)
    if rc != 0:
        raise ValueError("oracle cactus rejected its arguments")
    return out


def counterfactual(target, drafters, temperature=1.0, selected=-1, tokens=None, seeds=None, seq_index=None,
                   nthreads=0):
    """HedgeSpec counterfactual gamma for N drafters; target [B,K+1,V], drafters [N,B,K,V].

    Returns gamma [N,B,K], tv [N,B,K], loss = 1 - gamma, and with selected >= 0 the verify outputs of
    drafter `selected`'s chain."""
    lib = _load()
    target, dt = _logits(target)
    drafters, dd = _logits(drafters)
    assert dt == dd
    B, K1, V = target.shape
    K = K1 - 1
    N = drafters.shape[0]
    assert drafters.shape == (N, B, K, V)
    out = dict(gamma=np.zeros((N, B, K)), tv=np.zeros((N, B, K)))
    tok = sd = si = None
    if selected >= 0:
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        sd = np.ascontiguousarray(seeds, dtype=np.uint64)
        si = _seq_index(seq_index, B)
        out.update(accept_len=np.zeros(B, np.int32), out_tokens=np.zeros((B, K + 1), np.int32),
                   diag=np.zeros((B, K, 4)), accept_margin=np.zeros((B, K)), cdf_margin=np.zeros(B))
    rc = lib.spec_oracle_counterfactual(dt, _ptr(target), _ptr(drafters), N, B, K, V, _t32(temperature),
                                        _ptr(out["gamma"]), _ptr(out["tv"]), selected, _ptr(tok), _ptr(sd),
                                        _ptr(si), _ptr(out.get("accept_len")), _ptr(out.get("out_tokens")),
                                        _ptr(out.get("diag")), _ptr(out.get("accept_margin")),
                                        _ptr(out.get("cdf_margin")), nthreads)
    if rc != 0:
        raise ValueError("oracle counterfactual rejected its arguments")
    out["loss"] = 1.0 - out["gamma"]
    return out

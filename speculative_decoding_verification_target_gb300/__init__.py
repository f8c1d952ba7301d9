"""GB300 speculative-sampling verification: Python binding of the C ABI in include/specverify.h.

Argument marshalling only: every step of verification runs in the CUDA kernels of libspecverify.so.
Tensors are torch CUDA tensors (torch provides device memory and streams); outputs are allocated here
when not given. There is no CPU path: if the library is missing, importing the calls raises.

    verify(target, draft, tokens, seeds, temperature)            standard speculative sampling
    cactus_verify(target, draft, tokens, seeds, delta, temperature)  Cactus constrained acceptance
    counterfactual_gamma(target, drafters, temperature, selected, tokens, seeds)  HedgeSpec gamma
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

SPEC_OK, SPEC_ERR_INVALID, SPEC_ERR_CUDA, SPEC_ERR_UNSUPPORTED = 0, 1, 2, 3
STATUS_BAD_TOKEN, STATUS_TIMEOUT = 1, 2
EXPORTS = ("spec_workspace_size", "spec_verify", "spec_counterfactual_gamma", "spec_cactus_verify", "spec_cactus_kl_verify",
           "spec_greedy_verify", "spec_accept_length_estimate",
           "spec_normalhedge_update", "spec_filter_workspace_size", "spec_verify_filtered",
           "spec_read_status", "spec_clear_status", "spec_last_error", "spec_verify_static",
           "spec_hedge_feedback_state_size", "spec_hedge_feedback_init", "spec_hedge_feedback_push")
# tuning and test hooks (csrc/specverify_internal.h): exported by the library, not part of the C ABI
TEST_HOOKS = ("spec_debug_set_stats_grid", "spec_debug_last_plan", "spec_debug_exp2ff", "spec_debug_set_draw_tau",
              "spec_debug_set_gamma_one_launch")

_lib = None


class SpecError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("spec status %d: %s" % (code, msg))
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Loads libspecverify.so (built by __graft_entry__.build() or _build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        if build_if_missing:
            _build.build()
        else:
            raise ImportError("libspecverify.so is not built (run __graft_entry__.build()); there is no CPU fallback")
    lib = ctypes.CDLL(_build.LIB)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.spec_workspace_size.argtypes = [I, I, I, I]
    lib.spec_workspace_size.restype = Z
    lib.spec_verify.argtypes = [P, P, I, P, P, I, I, I, F, P, P, P, P, Z, P]
    lib.spec_verify.restype = I
    lib.spec_counterfactual_gamma.argtypes = [P, P, I, I, I, I, I, F, P, P, I, P, P, P, P, P, P, Z, P]
    lib.spec_counterfactual_gamma.restype = I
    lib.spec_cactus_verify.argtypes = [P, P, I, P, P, I, I, I, F, F, P, P, P, P, P, Z, P]
    lib.spec_cactus_verify.restype = I
    lib.spec_cactus_kl_verify.argtypes = [P, P, I, P, P, I, I, I, F, F, P, P, P, P, P, Z, P]
    lib.spec_cactus_kl_verify.restype = I
    lib.spec_greedy_verify.argtypes = [P, I, P, I, I, I, P, P, P, Z, P]
    lib.spec_greedy_verify.restype = I
    lib.spec_accept_length_estimate.argtypes = [P, I, I, I, P, P, P]
    lib.spec_accept_length_estimate.restype = I
    lib.spec_normalhedge_update.argtypes = [P, P, P, I, P]
    lib.spec_normalhedge_update.restype = I
    lib.spec_filter_workspace_size.argtypes = [I, I, I, I]
    lib.spec_filter_workspace_size.restype = Z
    lib.spec_verify_filtered.argtypes = [P, P, I, P, P, I, I, I, F, I, F, P, P, P, P, Z, P]
    lib.spec_verify_filtered.restype = I
    lib.spec_hedge_feedback_state_size.argtypes = [I, I, I]
    lib.spec_hedge_feedback_state_size.restype = Z
    lib.spec_hedge_feedback_init.argtypes = [P, I, I, I, I, P]
    lib.spec_hedge_feedback_init.restype = I
    lib.spec_hedge_feedback_push.argtypes = [P, P, P, I, I, I, P, P, P]
    lib.spec_hedge_feedback_push.restype = I
    lib.spec_read_status.argtypes = [P, P, P]
    lib.spec_read_status.restype = I
    lib.spec_clear_status.argtypes = [P, P]
    lib.spec_clear_status.restype = I
    lib.spec_last_error.argtypes = []
    lib.spec_last_error.restype = ctypes.c_char_p
    lib.spec_debug_set_stats_grid.argtypes = [I]
    lib.spec_debug_set_stats_grid.restype = I
    lib.spec_debug_last_plan.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.spec_debug_last_plan.restype = I
    lib.spec_debug_set_draw_tau.argtypes = [F]
    lib.spec_debug_set_draw_tau.restype = I
    lib.spec_debug_set_gamma_one_launch.argtypes = [I]
    lib.spec_debug_set_gamma_one_launch.restype = I
    lib.spec_debug_exp2ff.argtypes = [P, P, P, P, I, F, P]
    lib.spec_debug_exp2ff.restype = I
    lib.spec_verify_static.argtypes = [P, P, I, P, P, I, I, I, F, P, P, P, ctypes.POINTER(ctypes.c_uint32), P]
    lib.spec_verify_static.restype = I
    _lib = lib
    return lib


def _check(code):
    if code != SPEC_OK:
        raise SpecError(code, load().spec_last_error().decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return 0
    if t.dtype == torch.float32:
        return 1
    raise TypeError("logits must be bfloat16 or float32, got %s" % t.dtype)


def _need(t, name, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def workspace_size(B, K, V, N=1) -> int:
    return int(load().spec_workspace_size(B, K, V, N))


def new_workspace(B, K, V, N=1, device=None):
    """Device workspace for calls up to these sizes, with its status word cleared."""
    ws = torch.zeros(workspace_size(B, K, V, N), dtype=torch.uint8, device=device or "cuda")
    return ws


def read_status(ws, stream=None) -> int:
    out = ctypes.c_uint32(0)
    _check(load().spec_read_status(_p(ws), ctypes.byref(out), _stream(stream)))
    return out.value


def clear_status(ws, stream=None):
    _check(load().spec_clear_status(_p(ws), _stream(stream)))


def set_stats_grid(ctas: int):
    """Tuning / test hook: CTAs of the statistics pass of verify / cactus_verify (0 = automatic)."""
    if load().spec_debug_set_stats_grid(int(ctas)) != 0:
        raise ValueError("unsupported statistics grid %r" % ctas)


def set_gamma_one_launch(on: bool):
    """Tuning / test hook: run counterfactual_gamma with a selected drafter as one cooperative launch (gamma,
    a grid barrier, then the chain) instead of the gamma kernel followed by the draw kernel."""
    if load().spec_debug_set_gamma_one_launch(1 if on else 0) != 0:
        raise ValueError("unsupported value %r" % on)


def last_plan() -> dict:
    """Tuning / test hook: the launch plan of the last call on this thread."""
    out = (ctypes.c_int * 5)()
    load().spec_debug_last_plan(out)
    return dict(stages=out[1], ctas=out[2], kernel=out[3], pieces=out[4])


def _outputs(B, K, device, accept_len, out_tokens, diag, want_diag):
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=device)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=device)
    if diag is None and want_diag:
        diag = torch.empty((B, K, 4), dtype=torch.float32, device=device)
    return accept_len, out_tokens, diag


def verify(target, draft, tokens, seeds, temperature=1.0, *, accept_len=None, out_tokens=None, diag=None,
           want_diag=True, workspace=None, stream=None):
    """Standard speculative sampling. target [B,K+1,V], draft [B,K,V] (bf16 or fp32), tokens int32 [B,K],
    seeds int64/uint64 [B]. Returns dict(accept_len, out_tokens, diag)."""
    B, K1, V = target.shape
    K = K1 - 1
    _need(target, "target")
    _need(draft, "draft", target.dtype, (B, K, V))
    _need(tokens, "tokens", torch.int32, (B, K))
    _need(seeds, "seeds", None, (B,))
    accept_len, out_tokens, diag = _outputs(B, K, target.device, accept_len, out_tokens, diag, want_diag)
    ws = workspace if workspace is not None else new_workspace(B, K, V, 1, target.device)
    _check(load().spec_verify(_p(target), _p(draft), _dtype_code(target), _p(tokens), _p(seeds), B, K, V,
                              float(temperature), _p(accept_len), _p(out_tokens), _p(diag), _p(ws), ws.numel(),
                              _stream(stream)))
    return dict(accept_len=accept_len, out_tokens=out_tokens, diag=diag, workspace=ws)


def cactus_verify(target, draft, tokens, seeds, delta, temperature=1.0, *, accept_len=None, out_tokens=None,
                  diag=None, gamma_star=None, want_diag=True, workspace=None, stream=None, exact_kl=False):
    """Cactus constrained acceptance with divergence budget delta; same layout as verify. exact_kl=True uses
    gamma* as the root of the KL constraint (spec_cactus_kl_verify) instead of its Taylor closed form."""
    B, K1, V = target.shape
    K = K1 - 1
    _need(target, "target")
    _need(draft, "draft", target.dtype, (B, K, V))
    _need(tokens, "tokens", torch.int32, (B, K))
    _need(seeds, "seeds", None, (B,))
    accept_len, out_tokens, diag = _outputs(B, K, target.device, accept_len, out_tokens, diag, want_diag)
    if gamma_star is None:
        gamma_star = torch.empty((B, K), dtype=torch.float32, device=target.device)
    ws = workspace if workspace is not None else new_workspace(B, K, V, 1, target.device)
    fn = load().spec_cactus_kl_verify if exact_kl else load().spec_cactus_verify
    _check(fn(_p(target), _p(draft), _dtype_code(target), _p(tokens), _p(seeds), B, K, V, float(temperature),
              float(delta), _p(accept_len), _p(out_tokens), _p(diag), _p(gamma_star), _p(ws), ws.numel(),
              _stream(stream)))
    return dict(accept_len=accept_len, out_tokens=out_tokens, diag=diag, gamma_star=gamma_star, workspace=ws)


def greedy_verify(target, tokens, *, accept_len=None, out_tokens=None, workspace=None, stream=None):
    """Greedy (temperature 0) verification: accept a draft token iff it is the target row's argmax; emit the
    argmax of the first rejecting row (or of row K). target [B,K+1,V], tokens [B,K]."""
    B, K1, V = target.shape
    K = K1 - 1
    _need(target, "target")
    _need(tokens, "tokens", torch.int32, (B, K))
    accept_len, out_tokens, _ = _outputs(B, K, target.device, accept_len, out_tokens, None, False)
    ws = workspace if workspace is not None else new_workspace(B, K, V, 1, target.device)
    _check(load().spec_greedy_verify(_p(target), _dtype_code(target), _p(tokens), B, K, V, _p(accept_len),
                                     _p(out_tokens), _p(ws), ws.numel(), _stream(stream)))
    return dict(accept_len=accept_len, out_tokens=out_tokens, workspace=ws)


def accept_length_estimate(gamma, *, est=None, loss=None, want_loss=True, stream=None):
    """HedgeSpec accept-length estimate 1 + sum_k prod_{j<=k} gamma_j and loss K + 1 - est from gamma [N,B,K]."""
    N, B, K = gamma.shape
    _need(gamma, "gamma", torch.float32, (N, B, K))
    if est is None:
        est = torch.empty((N, B), dtype=torch.float32, device=gamma.device)
    if loss is None and want_loss:
        loss = torch.empty((N, B), dtype=torch.float32, device=gamma.device)
    _check(load().spec_accept_length_estimate(_p(gamma), N, B, K, _p(est), _p(loss), _stream(stream)))
    return dict(est=est, loss=loss)


def normalhedge_update(regret, loss, weights, stream=None):
    """One NormalHedge round in place: regret += weights . loss - loss, weights <- the next distribution."""
    N = regret.shape[0]
    for t, nm in ((regret, "regret"), (loss, "loss"), (weights, "weights")):
        _need(t, nm, torch.float32, (N,))
    _check(load().spec_normalhedge_update(_p(regret), _p(loss), _p(weights), N, _stream(stream)))


class HedgeFeedback:
    """NormalHedge learners (one per sequence) under delayed, censored feedback: each round, push the round's
    counterfactual gamma [N, B, K] and the selected drafter's accepted lengths [B]; the revealed levels are
    queued and every available loss is applied (objective 0: 1 - gamma per level; 1: the accept-length loss
    over a window of K levels). `weights` [B, N] is the distribution for the next round."""

    def __init__(self, N, B, K, objective=0, device=None, stream=None):
        self.N, self.B, self.K = N, B, K
        lib = load()
        n = int(lib.spec_hedge_feedback_state_size(N, B, K))
        if n == 0 and B > 0:
            raise ValueError("unsupported sizes N=%d B=%d K=%d" % (N, B, K))
        dev = device or "cuda"
        self.state = torch.zeros(max(n, 16), dtype=torch.uint8, device=dev)
        self.weights = torch.full((B, N), 1.0 / N, dtype=torch.float32, device=dev)
        self.applied = torch.zeros(B, dtype=torch.int32, device=dev)
        _check(lib.spec_hedge_feedback_init(_p(self.state), N, B, K, int(objective), _stream(stream)))

    def push(self, gamma, accept_len, stream=None):
        _need(gamma, "gamma", torch.float32, (self.N, self.B, self.K))
        _need(accept_len, "accept_len", torch.int32, (self.B,))
        _check(load().spec_hedge_feedback_push(_p(self.state), _p(gamma), _p(accept_len), self.N, self.B, self.K,
                                               _p(self.weights), _p(self.applied), _stream(stream)))
        return self.weights

    def status(self):
        """Per-sequence status words (bit 1: a round with an accepted length outside [0, K] was skipped)."""
        n = self.state.numel() // max(self.B, 1)
        return self.state.view(self.B, n)[:, 16:20].contiguous().view(torch.int32).view(-1).cpu()


def verify_filtered(target, draft, tokens, seeds, temperature=1.0, top_k=0, top_p=1.0, *, accept_len=None,
                    out_tokens=None, diag=None, want_diag=True, workspace=None, stream=None):
    """Standard speculative sampling on standardised rows: top-k then top-p folded into the target and the
    draft row alike (ties at a threshold kept). Same layout and outputs as verify."""
    B, K1, V = target.shape
    K = K1 - 1
    _need(target, "target")
    _need(draft, "draft", target.dtype, (B, K, V))
    _need(tokens, "tokens", torch.int32, (B, K))
    _need(seeds, "seeds", None, (B,))
    accept_len, out_tokens, diag = _outputs(B, K, target.device, accept_len, out_tokens, diag, want_diag)
    lib = load()
    if workspace is None:
        n = lib.spec_filter_workspace_size(B, K, V, _dtype_code(target))
        workspace = torch.zeros(n, dtype=torch.uint8, device=target.device)
    _check(lib.spec_verify_filtered(_p(target), _p(draft), _dtype_code(target), _p(tokens), _p(seeds), B, K, V,
                                    float(temperature), int(top_k), float(top_p), _p(accept_len), _p(out_tokens),
                                    _p(diag), _p(workspace), workspace.numel(), _stream(stream)))
    return dict(accept_len=accept_len, out_tokens=out_tokens, diag=diag, workspace=workspace)


def counterfactual_gamma(target, drafters, temperature=1.0, selected=-1, tokens=None, seeds=None, *, gamma=None,
                         loss=None, want_loss=True, accept_len=None, out_tokens=None, diag=None, want_diag=True,
                         workspace=None, stream=None):
    """HedgeSpec counterfactual gamma. target [B,K+1,V], drafters [N,B,K,V]. With selected >= 0 the chain of
    drafter `selected` is verified in the same pass (tokens, seeds required)."""
    B, K1, V = target.shape
    K = K1 - 1
    N = drafters.shape[0]
    _need(target, "target")
    _need(drafters, "drafters", target.dtype, (N, B, K, V))
    dev = target.device
    if gamma is None:
        gamma = torch.empty((N, B, K), dtype=torch.float32, device=dev)
    if loss is None and want_loss:
        loss = torch.empty((N, B, K), dtype=torch.float32, device=dev)
    out = dict(gamma=gamma, loss=loss)
    if selected >= 0:
        _need(tokens, "tokens", torch.int32, (B, K))
        _need(seeds, "seeds", None, (B,))
        accept_len, out_tokens, diag = _outputs(B, K, dev, accept_len, out_tokens, diag, want_diag)
        out.update(accept_len=accept_len, out_tokens=out_tokens, diag=diag)
    ws = workspace if workspace is not None else new_workspace(B, K, V, N, dev)
    _check(load().spec_counterfactual_gamma(_p(target), _p(drafters), _dtype_code(target), N, B, K, V,
                                            float(temperature), _p(gamma), _p(loss), int(selected), _p(tokens),
                                            _p(seeds), _p(out.get("accept_len")), _p(out.get("out_tokens")),
                                            _p(out.get("diag")), _p(ws), ws.numel(), _stream(stream)))
    out["workspace"] = ws
    return out

"""GPU parity at the limits the C ABI accepts: K = 64 draft positions, V = 262144 logits a row (128 pieces
of 2048, the most a draw CTA keeps), N = 64 drafters. Each case runs the fp64 oracle on the same seeded
inputs; the sizes stay small in B so that it finishes in seconds.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import PROB_TOL, assert_chain, assert_diag, host, oracle_verify, to_device

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_target_gb300")

K_MAX, V_MAX, N_MAX = 64, 262144, 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    sv.load(build_if_missing=True)
    sv.set_stats_grid(0)
    yield


def small(V, B, K, sigma=1.5, sigmas=None, selected=0, T=1.0, seed=29):
    sig = tuple(sigmas) if sigmas is not None else (sigma,)
    return workloads.Workload("limits", B=B, K=K, V=V, N=len(sig), temperature=T, draft_sigmas=sig,
                              selected=selected, gen_seed=seed)


@pytest.mark.parametrize("sigma", [0.0, 0.02, 1.5])
def test_verify_at_max_K_and_V(sigma):
    """K = 64 positions over V = 262144: the chain warp's second pass over positions 32..63, the draw's
    largest piece count, and (sigma 0, a draft equal to the target) every position accepted and the draw
    from the bonus row. Both launches: with diag (every row pair) and without (the one drawn pair)."""
    w = small(V_MAX, B=3, K=K_MAX, sigma=max(sigma, 1e-3))
    inp = workloads.make(w)
    if sigma == 0.0:
        inp["draft"] = inp["target"][:, :w.K].clone()
    ref = oracle_verify(inp)
    g = to_device(inp)
    full = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature)
    lean = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature, want_diag=False)
    torch.cuda.synchronize()
    assert_diag(full, ref)
    assert_chain(full, ref, w.K)
    assert_chain(lean, ref, w.K)
    assert sv.read_status(full["workspace"]) == 0
    if sigma == 0.0:
        assert np.all(full["accept_len"].cpu().numpy() == K_MAX)


@pytest.mark.parametrize("delta", [0.0, 0.5])
@pytest.mark.parametrize("exact_kl", [False, True])
def test_cactus_at_max_K_and_V(delta, exact_kl):
    w = small(V_MAX, B=2, K=K_MAX, sigma=0.3)
    inp = workloads.make(w)
    ref = oracle.cactus(host(inp["target"]), host(inp["draft"]), inp["tokens"].numpy(),
                        inp["seeds"].numpy().astype(np.uint64), delta, w.temperature, exact=exact_kl)
    g = to_device(inp)
    out = sv.cactus_verify(g["target"], g["draft"], g["tokens"], g["seeds"], delta, w.temperature, exact_kl=exact_kl)
    torch.cuda.synchronize()
    assert np.abs(out["gamma_star"].cpu().numpy() - ref["gamma_star"]).max() <= PROB_TOL
    assert_diag(out, ref)
    assert_chain(out, ref, w.K)


def test_greedy_at_max_K_and_V():
    """Draft tokens that are the target's argmax at every position: the whole chain of 64 is accepted and
    the bonus row's argmax is emitted; then one position is changed, which must stop the chain there."""
    w = small(V_MAX, B=3, K=K_MAX)
    inp = workloads.make(w)
    # the argmax of the values (first index among equal maxima), from float copies of the logits
    tok = inp["target"].float()[:, :w.K].argmax(dim=2).numpy().astype(np.int32)
    tok[1, 40] = (tok[1, 40] + 1) % w.V
    ref = oracle.greedy(host(inp["target"]), tok)
    out = sv.greedy_verify(inp["target"].cuda(), torch.from_numpy(tok).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(out["accept_len"].cpu().numpy(), ref["accept_len"])
    assert np.array_equal(out["out_tokens"].cpu().numpy(), ref["out_tokens"])
    assert ref["accept_len"][0] == K_MAX and ref["accept_len"][1] == 40


@pytest.mark.parametrize("selected", [-1, N_MAX - 1])
def test_counterfactual_at_max_N(selected):
    """64 drafters (the most the API takes) over a short vocabulary, with and without the fused chain of
    the last drafter."""
    sig = tuple(0.2 + 0.1 * i for i in range(N_MAX))
    w = small(4096, B=2, K=3, sigmas=sig, selected=max(selected, 0))
    inp = workloads.make(w)
    ref = oracle.counterfactual(host(inp["target"]), host(inp["drafters"]), w.temperature, selected,
                                inp["tokens"].numpy(), inp["seeds"].numpy().astype(np.uint64))
    g = to_device(inp)
    out = sv.counterfactual_gamma(g["target"], g["drafters"], w.temperature, selected, g["tokens"], g["seeds"])
    torch.cuda.synchronize()
    assert sv.read_status(out["workspace"]) == 0
    assert np.abs(out["gamma"].cpu().numpy() - ref["gamma"]).max() <= PROB_TOL
    if selected >= 0:
        assert_diag(out, ref)
        assert_chain(out, ref, w.K)


def test_counterfactual_at_max_K_and_V():
    """Two drafters with K = 64 over V = 262144: rows of 128 pieces, 8 per warp of the gamma kernel, most of
    them re-read from L2 in pass 2 (the tensor-memory share holds two per warp)."""
    w = small(V_MAX, B=1, K=K_MAX, sigmas=(0.3, 2.0), selected=0)
    inp = workloads.make(w)
    ref = oracle.counterfactual(host(inp["target"]), host(inp["drafters"]), w.temperature, 0,
                                inp["tokens"].numpy(), inp["seeds"].numpy().astype(np.uint64))
    g = to_device(inp)
    out = sv.counterfactual_gamma(g["target"], g["drafters"], w.temperature, 0, g["tokens"], g["seeds"])
    torch.cuda.synchronize()
    assert sv.read_status(out["workspace"]) == 0
    assert np.abs(out["gamma"].cpu().numpy() - ref["gamma"]).max() <= PROB_TOL
    assert_diag(out, ref)
    assert_chain(out, ref, w.K)


def test_accept_length_at_max_N_and_K():
    gen = torch.Generator().manual_seed(7)
    gam = torch.rand((N_MAX, 5, K_MAX), generator=gen, dtype=torch.float32) ** 0.1
    est = sv.accept_length_estimate(gam.cuda())
    torch.cuda.synchronize()
    e_ref, l_ref = oracle.accept_length(gam.numpy().astype(np.float64))
    assert np.abs(est["est"].cpu().numpy() - e_ref).max() <= 1e-4
    assert np.abs(est["loss"].cpu().numpy() - l_ref).max() <= 1e-4


def test_filtered_at_max_K_and_V():
    """Top-k then top-p on both rows of every position, K = 64 over V = 262144."""
    w = small(V_MAX, B=2, K=K_MAX, sigma=0.5, T=0.9)
    inp = workloads.make(w)
    ref = oracle.verify_filtered(host(inp["target"]), host(inp["draft"]), inp["tokens"].numpy(),
                                 inp["seeds"].numpy().astype(np.uint64), w.temperature, 5000, 0.9)
    g = to_device(inp)
    out = sv.verify_filtered(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature, 5000, 0.9)
    torch.cuda.synchronize()
    assert_diag(out, ref)
    assert_chain(out, ref, w.K)
    assert sv.read_status(out["workspace"]) == 0

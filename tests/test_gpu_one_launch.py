"""The counterfactual call with a selected drafter as ONE cooperative launch (gamma for every drafter, a grid
barrier, then the selected drafter's chain and draw on one CTA per sequence), against the fp64 oracle and
against the two-launch path (gamma kernel, then draw kernel), which runs the same gamma and per-piece draw
arithmetic and so gives the same bits."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import PROB_TOL, assert_chain, assert_diag, host, to_device

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_target_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    sv.load(build_if_missing=True)
    sv.set_stats_grid(0)
    yield
    sv.set_gamma_one_launch(False)


def both_paths(g, w):
    """(two-launch outputs, one-launch outputs) of the same call."""
    outs = []
    for one in (False, True):
        sv.set_gamma_one_launch(one)
        try:
            o = sv.counterfactual_gamma(g["target"], g["drafters"], w.temperature, w.selected, g["tokens"],
                                        g["seeds"])
            torch.cuda.synchronize()
            plan = sv.last_plan()
        finally:
            sv.set_gamma_one_launch(False)
        assert plan["kernel"] == (5 if one else 2)
        assert sv.read_status(o["workspace"]) == 0
        outs.append(o)
    return outs


def assert_same(a, b):
    for k in ("gamma", "loss", "accept_len", "out_tokens", "diag"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("V,dtype,sigmas,B,K,selected", [
    (5000, "bf16", (0.5, 1.0, 2.0, 4.0), 5, 4, 1),
    (33336, "bf16", (0.7, 1.5, 3.0), 8, 5, 2),
    (4096, "fp32", (1.0, 2.0), 6, 3, 0),
    (128256, "bf16", (1.5, 3.0), 3, 2, 1),
    (1000, "bf16", (1.0, 2.0), 300, 2, 0),   # more sequences than CTAs: each CTA draws several
])
def test_one_launch_small(V, dtype, sigmas, B, K, selected):
    w = workloads.Workload("t", B=B, K=K, V=V, N=len(sigmas), dtype=dtype, temperature=0.9, peaks=5,
                           draft_sigmas=sigmas, selected=selected, gen_seed=23)
    inp = workloads.make(w)
    ref = oracle.counterfactual(host(inp["target"]), host(inp["drafters"]), w.temperature, selected,
                                inp["tokens"].numpy(), inp["seeds"].numpy().astype(np.uint64))
    two, one = both_paths(to_device(inp), w)
    assert np.abs(one["gamma"].cpu().numpy() - ref["gamma"]).max() <= PROB_TOL
    assert_diag(one, ref)
    assert_chain(one, ref, w.K)
    assert_same(two, one)


def test_one_launch_named_full():
    """Config 3 (N = 7, B = 32, K = 5, V = 128256): every sequence against the oracle."""
    w = workloads.WORKLOADS["hedgespec_n7_b32_k5"]
    inp = workloads.make(w, device="cuda")
    two, one = both_paths(inp, w)
    ref = oracle.counterfactual(host(inp["target"]), host(inp["drafters"]), w.temperature, w.selected,
                                inp["tokens"].cpu().numpy(), inp["seeds"].cpu().numpy().astype(np.uint64))
    assert np.abs(one["gamma"].cpu().numpy() - ref["gamma"]).max() <= PROB_TOL
    assert_diag(one, ref)
    assert_chain(one, ref, w.K)
    assert_same(two, one)


def test_one_launch_large_pool_sampled():
    """Config 5 (N = 21, B = 256, K = 8, V = 151936): gamma everywhere and 16 sampled sequences' chains against
    the oracle; the whole batch against the two-launch path."""
    w = workloads.WORKLOADS["hedgespec_n21_b256_k8"]
    inp = workloads.make(w, device="cuda")
    two, one = both_paths(inp, w)
    sel = torch.arange(5, w.B, 16)
    selc = sel.cuda()
    ref = oracle.counterfactual(host(inp["target"][selc]), host(inp["drafters"][:, selc]), w.temperature,
                                w.selected, inp["tokens"][selc].cpu().numpy(),
                                inp["seeds"][selc].cpu().numpy().astype(np.uint64), seq_index=sel.numpy())
    assert np.abs(one["gamma"][:, selc].cpu().numpy() - ref["gamma"]).max() <= PROB_TOL
    sub = {k: one[k][selc] for k in ("accept_len", "out_tokens", "diag")}
    assert_diag(sub, ref)
    assert_chain(sub, ref, w.K)
    assert_same(two, one)


def test_one_launch_repeated_calls_reuse_the_barrier():
    """The grid barrier's words return to their start after each call: back-to-back calls on one workspace
    give the same outputs and leave the status word clear."""
    w = workloads.Workload("t", B=40, K=3, V=20000, N=2, dtype="bf16", temperature=1.0, peaks=5,
                           draft_sigmas=(1.0, 2.0), selected=1, gen_seed=5)
    g = to_device(workloads.make(w))
    ws = sv.new_workspace(w.B, w.K, w.V, w.N, "cuda")
    sv.set_gamma_one_launch(True)
    try:
        outs = [sv.counterfactual_gamma(g["target"], g["drafters"], w.temperature, w.selected, g["tokens"],
                                        g["seeds"], workspace=ws) for _ in range(4)]
        torch.cuda.synchronize()
    finally:
        sv.set_gamma_one_launch(False)
    assert sv.read_status(ws) == 0
    for o in outs[1:]:
        assert_same(outs[0], o)

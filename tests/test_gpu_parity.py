"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Small cases span several 2048-logit pieces, forced statistics grids (rows cut into per-warp segments at
different places), a ragged last piece, unaligned rows (V not a multiple of 8: element-wise loads instead of
bulk copies) and fp32 logits; the five named workloads run at full size (the largest checked on a stated
sample of sequences through seq_index).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import (PROB_TOL, assert_chain, assert_diag, host, oracle_verify, to_device)

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_target_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    sv.load(build_if_missing=True)
    yield
    sv.set_stats_grid(0)


@pytest.fixture(autouse=True)
def _auto_grid():
    sv.set_stats_grid(0)
    yield
    sv.set_stats_grid(0)


def small(V, B=6, K=4, dtype="bf16", T=1.0, sigma=1.5, peaks=5, N=1, sigmas=None, selected=0, seed=11):
    sig = tuple(sigmas) if sigmas is not None else (sigma,)
    return workloads.Workload("t", B=B, K=K, V=V, N=len(sig), dtype=dtype, temperature=T, peaks=peaks,
                              draft_sigmas=sig, selected=selected, gen_seed=seed)


# ------------------------------------------------------------------------------------------------
# standard verification
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("V,C,dtype", [
    (1000, 0, "fp32"), (1000, 0, "bf16"), (4099, 0, "bf16"), (4099, 4, "bf16"), (8192, 2, "fp32"),
    (20000, 8, "bf16"), (20001, 8, "bf16"), (65536, 0, "bf16"), (128256, 0, "bf16"), (151936, 0, "bf16"),
    (3000, 16, "bf16"),
])
def test_verify_small(V, C, dtype):
    sv.set_stats_grid(C)   # C CTAs in the statistics pass: every warp's run spans several rows
    w = small(V, dtype=dtype, T=0.8)
    inp = workloads.make(w)
    ref = oracle_verify(inp)
    g = to_device(inp)
    out = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature)
    torch.cuda.synchronize()
    assert_diag(out, ref)
    assert_chain(out, ref, w.K)
    assert sv.read_status(out["workspace"]) == 0


def test_verify_deterministic():
    w = small(30011, B=16, K=5)
    g = to_device(workloads.make(w))
    a = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"])
    b = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"])
    torch.cuda.synchronize()
    for k in ("accept_len", "out_tokens", "diag"):
        assert torch.equal(a[k], b[k])


def test_verify_stats_grid_invariance():
    """The statistics grid only changes where the rows are cut into per-warp segments (summation order):
    every grid meets the oracle bar, and the probabilities agree within the tolerance."""
    w = small(50000, B=8, K=3)
    inp = workloads.make(w)
    ref = oracle_verify(inp)
    g = to_device(inp)
    outs = []
    for ctas in (1, 3, 5, 37, 0):
        sv.set_stats_grid(ctas)
        o = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"])
        torch.cuda.synchronize()
        if ctas:
            assert 1 <= sv.last_plan()["ctas"] <= ctas
        assert_diag(o, ref)
        assert_chain(o, ref, w.K)
        assert sv.read_status(o["workspace"]) == 0
        outs.append(o)
    for o in outs[1:]:
        assert torch.allclose(o["diag"], outs[0]["diag"], atol=PROB_TOL, rtol=0)


def test_verify_fewer_pieces_than_warps():
    """One sequence of one draft over a 1000-token vocabulary: three pieces in all, so most warps of the
    statistics grid have no run; and a grid of one CTA over many rows."""
    for B, K, V, ctas in ((1, 1, 1000, 0), (1, 1, 1000, 4), (12, 7, 3000, 1)):
        sv.set_stats_grid(ctas)
        w = small(V, B=B, K=K)
        inp = workloads.make(w)
        ref = oracle_verify(inp)
        g = to_device(inp)
        out = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature)
        torch.cuda.synchronize()
        assert_diag(out, ref)
        assert_chain(out, ref, w.K)
        assert sv.read_status(out["workspace"]) == 0


@pytest.mark.parametrize("name", ["tiny_sps_v1000", "sps_llama3_b64_k5"])
def test_verify_named_workloads_full(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make(w, device="cuda")
    ref = oracle_verify(inp)
    out = sv.verify(inp["target"], inp["draft"], inp["tokens"], inp["seeds"], w.temperature)
    torch.cuda.synchronize()
    assert_diag(out, ref)
    assert_chain(out, ref, w.K)


# ------------------------------------------------------------------------------------------------
# edge cases
# ------------------------------------------------------------------------------------------------
def test_B_zero_is_noop():
    t = torch.zeros((0, 3, 100), dtype=torch.bfloat16, device="cuda")
    d = torch.zeros((0, 2, 100), dtype=torch.bfloat16, device="cuda")
    tok = torch.zeros((0, 2), dtype=torch.int32, device="cuda")
    seeds = torch.zeros(0, dtype=torch.int64, device="cuda")
    ws = sv.new_workspace(1, 2, 100)
    out = sv.verify(t, d, tok, seeds, workspace=ws)
    assert out["accept_len"].numel() == 0


def test_vocab_of_one_and_two():
    for V in (1, 2):
        w = small(V, B=5, K=3, peaks=0)
        inp = workloads.make(w)
        ref = oracle_verify(inp)
        g = to_device(inp)
        out = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"])
        torch.cuda.synchronize()
        assert_diag(out, ref)
        assert_chain(out, ref, w.K)
    # V = 1: every draft is the only token, always accepted, Z = 0
    assert np.all(out["accept_len"].cpu().numpy() >= 0)


def test_perfect_draft_always_accepts():
    w = small(7000, B=8, K=5)
    inp = workloads.make(w)
    inp["draft"] = inp["target"][:, :w.K].clone()
    ref = oracle_verify(inp)
    g = to_device(inp)
    out = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"])
    torch.cuda.synchronize()
    assert np.all(out["accept_len"].cpu().numpy() == w.K)
    assert np.all(out["diag"].cpu().numpy()[..., 2] <= 1e-6)
    assert_chain(out, ref, w.K)


def test_disjoint_support_always_rejects():
    B, K, V = 6, 3, 512
    t = torch.full((B, K + 1, V), float("-inf"))
    d = torch.full((B, K, V), float("-inf"))
    gen = torch.Generator().manual_seed(3)
    t[:, :, V // 2:] = torch.randn((B, K + 1, V - V // 2), generator=gen)
    d[:, :, :V // 2] = torch.randn((B, K, V // 2), generator=gen)
    tok = torch.randint(0, V // 2, (B, K), generator=gen, dtype=torch.int32)
    seeds = torch.arange(B, dtype=torch.int64)
    inp = dict(target=t.to(torch.bfloat16), draft=d.to(torch.bfloat16), tokens=tok, seeds=seeds, temperature=1.0)
    ref = oracle_verify(inp)
    g = to_device(inp)
    out = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"])
    torch.cuda.synchronize()
    assert np.all(out["accept_len"].cpu().numpy() == 0)
    assert np.all(out["out_tokens"].cpu().numpy()[:, 0] >= V // 2)
    assert_diag(out, ref)
    assert_chain(out, ref, K)


def test_masked_logits_and_bad_token_status():
    w = small(3000, B=4, K=3)
    inp = workloads.make(w)
    inp["target"][:, :, :100] = float("-inf")
    inp["tokens"][1, 1] = w.V + 5          # out of range: flagged, verified as a zero-probability proposal
    inp["tokens"][2, 0] = -1
    ref = oracle_verify(dict(inp, tokens=inp["tokens"].clamp(0, w.V - 1)))
    g = to_device(inp)
    ws = sv.new_workspace(w.B, w.K, w.V)
    out = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], workspace=ws)
    torch.cuda.synchronize()
    assert sv.read_status(ws) & sv.STATUS_BAD_TOKEN
    d = out["diag"].cpu().numpy()
    assert d[1, 1, 0] == 0.0 and d[1, 1, 1] == 0.0
    assert out["accept_len"][1].item() <= 1 and out["accept_len"][2].item() == 0
    tok = out["out_tokens"].cpu().numpy()
    assert np.all(tok[tok >= 0] >= 100)             # masked tokens are never emitted
    sv.clear_status(ws)
    assert sv.read_status(ws) == 0


def test_invalid_arguments_raise():
    w = small(1000, B=2, K=2)
    g = to_device(workloads.make(w))
    with pytest.raises(sv.SpecError) as e:
        sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], temperature=0.0)
    assert e.value.code == sv.SPEC_ERR_UNSUPPORTED
    with pytest.raises(sv.SpecError) as e:
        sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], temperature=float("nan"))
    assert e.value.code == sv.SPEC_ERR_INVALID
    with pytest.raises(sv.SpecError) as e:
        sv.cactus_verify(g["target"], g["draft"], g["tokens"], g["seeds"], delta=-1.0)
    assert e.value.code == sv.SPEC_ERR_INVALID
    small_ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(sv.SpecError):
        sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], workspace=small_ws)


# ------------------------------------------------------------------------------------------------
# losslessness on the GPU: chi-square of emitted tokens against p_target
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("V", [3, 8, 64])
def test_gpu_chi2_lossless(V):
    from scipy import special, stats
    rng = np.random.default_rng(V)
    n = 1 << 17
    p = special.softmax(rng.normal(0, 1.5, V)).astype(np.float64)
    q = special.softmax(np.log(p) + rng.normal(0, 1.0, V))
    lt = np.log(p).astype(np.float32)
    ld = np.log(q).astype(np.float32)
    t = torch.from_numpy(np.broadcast_to(lt, (n, 2, V)).copy()).cuda()
    d = torch.from_numpy(np.broadcast_to(ld, (n, 1, V)).copy()).cuda()
    tok = torch.from_numpy(rng.choice(V, size=(n, 1), p=q / q.sum()).astype(np.int32)).cuda()
    seeds = torch.full((n,), 12345, dtype=torch.int64, device="cuda")
    out = sv.verify(t, d, tok, seeds, want_diag=False)
    torch.cuda.synchronize()
    first = out["out_tokens"][:, 0].cpu().numpy()
    counts = np.bincount(first, minlength=V)
    pf = np.exp(lt.astype(np.float64))
    pf /= pf.sum()
    assert stats.chisquare(counts, pf * n).pvalue > 1e-6
    # and the rejection rate is Z = 1 - sum min(p, q)
    qf = np.exp(ld.astype(np.float64))
    qf /= qf.sum()
    rej = (out["accept_len"].cpu().numpy() == 0).mean()
    z = np.maximum(pf - qf, 0).sum()
    assert abs(rej - z) < 5 * np.sqrt(z * (1 - z) / n) + 1e-4


# ------------------------------------------------------------------------------------------------
# Cactus
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("delta", [0.0, 0.75, 1.0])
@pytest.mark.parametrize("V,C", [(3000, 0), (40000, 8)])
def test_cactus_small(delta, V, C):
    sv.set_stats_grid(C)
    w = small(V, B=8, K=5, sigma=2.0)
    inp = workloads.make(w)
    ref = oracle.cactus(host(inp["target"]), host(inp["draft"]), inp["tokens"].numpy(),
                        inp["seeds"].numpy().astype(np.uint64), delta, w.temperature)
    g = to_device(inp)
    out = sv.cactus_verify(g["target"], g["draft"], g["tokens"], g["seeds"], delta, w.temperature)
    torch.cuda.synchronize()
    assert np.abs(out["gamma_star"].cpu().numpy() - ref["gamma_star"]).max() <= PROB_TOL
    assert_diag(out, ref)
    assert_chain(out, ref, w.K)


def test_cactus_delta_zero_bit_identical_to_verify():
    w = small(151936, B=6, K=4, sigma=2.0)
    g = to_device(workloads.make(w))
    a = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"])
    c = sv.cactus_verify(g["target"], g["draft"], g["tokens"], g["seeds"], 0.0)
    torch.cuda.synchronize()
    assert torch.equal(a["accept_len"], c["accept_len"])
    assert torch.equal(a["out_tokens"], c["out_tokens"])
    assert torch.equal(a["diag"], c["diag"])


# ------------------------------------------------------------------------------------------------
# Cactus with gamma* as the exact root of its divergence constraint
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("delta", [0.0, 0.05, 0.75, 1.0, 3.0])
@pytest.mark.parametrize("V,dtype", [(3000, "bf16"), (40000, "bf16"), (1000, "fp32")])
def test_cactus_kl_small(delta, V, dtype):
    w = small(V, B=8, K=5, sigma=2.0, dtype=dtype, T=0.8)
    inp = workloads.make(w)
    ref = oracle.cactus(host(inp["target"]), host(inp["draft"]), inp["tokens"].numpy(),
                        inp["seeds"].numpy().astype(np.uint64), delta, w.temperature, exact=True)
    g = to_device(inp)
    out = sv.cactus_verify(g["target"], g["draft"], g["tokens"], g["seeds"], delta, w.temperature, exact_kl=True)
    torch.cuda.synchronize()
    assert np.abs(out["gamma_star"].cpu().numpy() - ref["gamma_star"]).max() <= PROB_TOL
    assert_diag(out, ref)
    assert_chain(out, ref, w.K)
    assert sv.read_status(out["workspace"]) == 0


def test_cactus_kl_delta_zero_bit_identical_to_verify():
    w = small(151936, B=6, K=4, sigma=2.0)
    g = to_device(workloads.make(w))
    a = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"])
    c = sv.cactus_verify(g["target"], g["draft"], g["tokens"], g["seeds"], 0.0, exact_kl=True)
    torch.cuda.synchronize()
    for k in ("accept_len", "out_tokens", "diag"):
        assert torch.equal(a[k], c[k])


def test_cactus_kl_named_workload_sampled():
    """Config 4's shapes with the exact root, every 8th sequence against the oracle; the root never falls
    below the Taylor value where that one is at most 0.5 (the page's Corollary 6)."""
    w = workloads.WORKLOADS["cactus_qwen_b128_m20"]
    inp = workloads.make(w, device="cuda")
    sel = torch.arange(0, w.B, 8)
    for delta in w.deltas:
        out = sv.cactus_verify(inp["target"], inp["draft"], inp["tokens"], inp["seeds"], delta, w.temperature,
                               exact_kl=True)
        tay = sv.cactus_verify(inp["target"], inp["draft"], inp["tokens"], inp["seeds"], delta, w.temperature)
        torch.cuda.synchronize()
        ref = oracle.cactus(host(inp["target"][sel]), host(inp["draft"][sel]), inp["tokens"][sel].cpu().numpy(),
                            inp["seeds"][sel].cpu().numpy().astype(np.uint64), delta, w.temperature,
                            seq_index=sel.numpy(), exact=True)
        sub = {k: out[k][sel.cuda()] for k in ("accept_len", "out_tokens", "diag")}
        assert np.abs(out["gamma_star"][sel.cuda()].cpu().numpy() - ref["gamma_star"]).max() <= PROB_TOL
        assert_diag(sub, ref)
        assert_chain(sub, ref, w.K)
        ge, gt = out["gamma_star"], tay["gamma_star"]
        low = gt <= 0.5
        assert torch.all(ge[low] >= gt[low] - 1e-6)


def test_cactus_named_workload_sampled():
    w = workloads.WORKLOADS["cactus_qwen_b128_m20"]
    inp = workloads.make(w, device="cuda")
    sel = torch.arange(0, w.B, 8)
    for delta in w.deltas:
        out = sv.cactus_verify(inp["target"], inp["draft"], inp["tokens"], inp["seeds"], delta, w.temperature)
        torch.cuda.synchronize()
        ref = oracle.cactus(host(inp["target"][sel]), host(inp["draft"][sel]), inp["tokens"][sel].cpu().numpy(),
                            inp["seeds"][sel].cpu().numpy().astype(np.uint64), delta, w.temperature,
                            seq_index=sel.numpy())
        sub = {k: out[k][sel.cuda()] for k in ("accept_len", "out_tokens", "diag")}
        assert np.abs(out["gamma_star"][sel.cuda()].cpu().numpy() - ref["gamma_star"]).max() <= PROB_TOL
        assert_diag(sub, ref)
        assert_chain(sub, ref, w.K)


# ------------------------------------------------------------------------------------------------
# HedgeSpec counterfactual gamma
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("V,selected", [(5000, -1), (5000, 1), (33333, 2), (33336, 0)])
def test_counterfactual_small(V, selected):
    w = small(V, B=5, K=4, sigmas=(0.5, 1.0, 2.0, 4.0), selected=max(selected, 0))
    inp = workloads.make(w)
    ref = oracle.counterfactual(host(inp["target"]), host(inp["drafters"]), w.temperature, selected,
                                inp["tokens"].numpy(), inp["seeds"].numpy().astype(np.uint64))
    g = to_device(inp)
    out = sv.counterfactual_gamma(g["target"], g["drafters"], w.temperature, selected, g["tokens"], g["seeds"])
    torch.cuda.synchronize()
    gam = out["gamma"].cpu().numpy()
    assert np.abs(gam - ref["gamma"]).max() <= PROB_TOL
    assert np.abs(out["loss"].cpu().numpy() - (1 - ref["gamma"])).max() <= PROB_TOL
    assert np.abs((1 - gam) - ref["tv"]).max() <= PROB_TOL          # gamma = 1 - TV
    if selected >= 0:
        assert_diag(out, ref)
        assert_chain(out, ref, w.K)
        # a plain verify of the selected drafter (the two-kernel path, another summation order) meets the
        # same bar against the same oracle chain
        v = sv.verify(g["target"], g["drafters"][selected].contiguous(), g["tokens"], g["seeds"], w.temperature)
        torch.cuda.synchronize()
        assert_diag(v, ref)
        assert_chain(v, ref, w.K)


@pytest.mark.parametrize("V,dtype,sigmas,B,K,selected", [
    (140000, "bf16", (0.5, 1.5, 3.0), 3, 2, 1),      # 69 pieces a row: pieces past the tensor-memory share
    (70000, "fp32", (1.0, 2.0, 4.0), 3, 2, -1),      # fp32 pieces of 1024 logits, also past the share
    (1000, "fp32", (0.5, 2.0), 4, 5, 0),             # one piece a row: 15 of 16 warps idle
    (20001, "bf16", (0.5, 1.0, 2.0, 3.0, 6.0), 2, 3, 4),   # element-wise loads (V not a multiple of 8)
    (128256, "bf16", (0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0), 24, 5, 2),   # more units than CTAs
])
def test_counterfactual_shapes(V, dtype, sigmas, B, K, selected):
    """The gamma kernel across row lengths, element types and unit counts: every CTA run starting inside a
    position (its own copy of the target row's statistics), rows longer than the tensor-memory share,
    one-piece rows and the element-wise path."""
    w = small(V, B=B, K=K, dtype=dtype, sigmas=sigmas, selected=max(selected, 0))
    inp = workloads.make(w)
    ref = oracle.counterfactual(host(inp["target"]), host(inp["drafters"]), w.temperature, selected,
                                inp["tokens"].numpy(), inp["seeds"].numpy().astype(np.uint64))
    g = to_device(inp)
    out = sv.counterfactual_gamma(g["target"], g["drafters"], w.temperature, selected, g["tokens"], g["seeds"])
    torch.cuda.synchronize()
    assert sv.read_status(out["workspace"]) == 0
    gam = out["gamma"].cpu().numpy()
    assert np.abs(gam - ref["gamma"]).max() <= PROB_TOL
    assert np.abs(out["loss"].cpu().numpy() - (1 - ref["gamma"])).max() <= PROB_TOL
    if selected >= 0:
        assert_diag(out, ref)
        assert_chain(out, ref, w.K)


def test_counterfactual_named_full():
    w = workloads.WORKLOADS["hedgespec_n7_b32_k5"]
    inp = workloads.make(w, device="cuda")
    out = sv.counterfactual_gamma(inp["target"], inp["drafters"], w.temperature, w.selected, inp["tokens"],
                                  inp["seeds"])
    torch.cuda.synchronize()
    ref = oracle.counterfactual(host(inp["target"]), host(inp["drafters"]), w.temperature, w.selected,
                                inp["tokens"].cpu().numpy(), inp["seeds"].cpu().numpy().astype(np.uint64))
    assert np.abs(out["gamma"].cpu().numpy() - ref["gamma"]).max() <= PROB_TOL
    assert_diag(out, ref)
    assert_chain(out, ref, w.K)


def test_large_pool_named_sampled():
    """21 drafters, B=256, K=8, V=151936, T=0.7, fused verify of drafter 4: gamma for every drafter and the
    chain checked on 16 sampled sequences (the oracle on all 256 would take minutes)."""
    w = workloads.WORKLOADS["hedgespec_n21_b256_k8"]
    inp = workloads.make(w, device="cuda")
    out = sv.counterfactual_gamma(inp["target"], inp["drafters"], w.temperature, w.selected, inp["tokens"],
                                  inp["seeds"])
    torch.cuda.synchronize()
    sel = torch.arange(3, w.B, 16)
    selc = sel.cuda()
    ref = oracle.counterfactual(host(inp["target"][selc]), host(inp["drafters"][:, selc]), w.temperature,
                                w.selected, inp["tokens"][selc].cpu().numpy(),
                                inp["seeds"][selc].cpu().numpy().astype(np.uint64), seq_index=sel.numpy())
    assert np.abs(out["gamma"][:, selc].cpu().numpy() - ref["gamma"]).max() <= PROB_TOL
    sub = {k: out[k][selc] for k in ("accept_len", "out_tokens", "diag")}
    assert_diag(sub, ref)
    assert_chain(sub, ref, w.K)
    # properties over the whole batch
    gam = out["gamma"].cpu().numpy()
    assert np.all((gam > 0) & (gam <= 1.0 + 1e-6))
    assert np.all(np.diff(gam.mean(axis=(1, 2))) < 0.05)   # larger drafter noise, lower acceptance (on average)


# ------------------------------------------------------------------------------------------------
# without diag only the row pair of each sequence's draw is re-read (verify, Cactus), and the fused row
# kernel skips the residual masses of accepted positions (counterfactual); the outputs must not change
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("V,B,K,C", [(5000, 16, 6, 0), (50000, 12, 5, 4), (128256, 24, 5, 0)])
def test_verify_without_diag_matches(V, B, K, C):
    sv.set_stats_grid(C)
    w = small(V, B=B, K=K, sigma=1.0)
    g = to_device(workloads.make(w))
    full = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature)
    lean = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature, want_diag=False)
    torch.cuda.synchronize()
    assert torch.equal(full["accept_len"], lean["accept_len"])
    assert torch.equal(full["out_tokens"], lean["out_tokens"])
    acc = full["accept_len"].cpu().numpy()
    assert 0 < acc.mean() < K   # both accepted and rejected positions occur
    ref = oracle_verify(workloads.make(w))
    assert_chain(lean, ref, w.K)


@pytest.mark.parametrize("delta", [0.0, 1.0])
def test_cactus_without_diag_matches(delta):
    w = small(20000, B=16, K=8, sigma=2.0)
    g = to_device(workloads.make(w))
    full = sv.cactus_verify(g["target"], g["draft"], g["tokens"], g["seeds"], delta, w.temperature)
    lean = sv.cactus_verify(g["target"], g["draft"], g["tokens"], g["seeds"], delta, w.temperature, want_diag=False)
    torch.cuda.synchronize()
    assert torch.equal(full["accept_len"], lean["accept_len"])
    assert torch.equal(full["out_tokens"], lean["out_tokens"])


def test_counterfactual_without_diag_matches():
    w = small(33333, B=8, K=5, sigmas=(0.7, 1.5, 3.0), selected=1)
    g = to_device(workloads.make(w))
    full = sv.counterfactual_gamma(g["target"], g["drafters"], w.temperature, w.selected, g["tokens"], g["seeds"])
    lean = sv.counterfactual_gamma(g["target"], g["drafters"], w.temperature, w.selected, g["tokens"], g["seeds"],
                                   want_diag=False)
    torch.cuda.synchronize()
    assert torch.equal(full["accept_len"], lean["accept_len"])
    assert torch.equal(full["out_tokens"], lean["out_tokens"])
    # accepted positions of the selected drafter take the overlap-only pass 2 (h(t) unpatched): same gamma
    # up to rounding
    assert (full["gamma"] - lean["gamma"]).abs().max().item() <= 1e-6


# ------------------------------------------------------------------------------------------------
# the near-tie bar over whole batches: the oracle on every sequence of a named workload
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("name,delta", [
    ("sps_llama3_b64_k5", None), ("hedgespec_n7_b32_k5", None), ("hedgespec_n21_b256_k8", None),
    ("cactus_qwen_b128_m20", 0.0), ("cactus_qwen_b128_m20", 0.75), ("cactus_qwen_b128_m20", 1.0),
])
def test_full_batch_near_ties(name, delta):
    """Every sequence of the workload's base batch against the oracle, with and without diag: tokens and
    accept lengths bit-exact except at near ties, which are counted here; their rate (under 0.01% of
    positions) is asserted over many batches in test_gpu_near_ties.py, since one batch of 2560 positions
    cannot resolve it. The counterfactual workloads check both the plain verify of the selected drafter and
    the chain fused into the gamma call."""
    w = workloads.WORKLOADS[name]
    inp = workloads.make(w, device="cuda")
    draft = inp["drafters"][w.selected].contiguous() if w.N > 1 else inp["draft"]
    tok = inp["tokens"].cpu().numpy()
    seeds = inp["seeds"].cpu().numpy().astype(np.uint64)
    if delta is None:
        ref = oracle.verify(host(inp["target"]), host(draft), tok, seeds, w.temperature)
        out = sv.verify(inp["target"], draft, inp["tokens"], inp["seeds"], w.temperature)
        lean = sv.verify(inp["target"], draft, inp["tokens"], inp["seeds"], w.temperature, want_diag=False)
    else:
        ref = oracle.cactus(host(inp["target"]), host(draft), tok, seeds, delta, w.temperature)
        out = sv.cactus_verify(inp["target"], draft, inp["tokens"], inp["seeds"], delta, w.temperature)
        lean = sv.cactus_verify(inp["target"], draft, inp["tokens"], inp["seeds"], delta, w.temperature,
                                want_diag=False)
    torch.cuda.synchronize()
    assert_diag(out, ref)
    assert_chain(out, ref, w.K, rate=False)
    # the launch the benchmark times (no diag: one draw pass over the row pair of each sequence's draw)
    assert_chain(lean, ref, w.K, rate=False)
    if w.N > 1:
        fused = sv.counterfactual_gamma(inp["target"], inp["drafters"], w.temperature, w.selected, inp["tokens"],
                                        inp["seeds"], want_diag=False)
        torch.cuda.synchronize()
        assert_chain(fused, ref, w.K, rate=False)


# ------------------------------------------------------------------------------------------------
# greedy verification (temperature 0)
# ------------------------------------------------------------------------------------------------
def _greedy_tokens(inp, frac=0.7, seed=5):
    """Draft tokens: the target's argmax with probability frac (so chains get long), else the draft's."""
    gen = torch.Generator().manual_seed(seed)
    t = inp["target"].float().cpu()
    d = inp["draft"].float().cpu()
    K = d.shape[1]
    am_t = t[:, :K].argmax(dim=2)
    am_d = d.argmax(dim=2)
    pick = torch.rand(am_t.shape, generator=gen) < frac
    return torch.where(pick, am_t, am_d).to(torch.int32)


@pytest.mark.parametrize("V,dtype,C", [(1000, "fp32", 0), (3000, "bf16", 0), (4099, "bf16", 3), (20001, "bf16", 0),
                                       (128256, "bf16", 0), (151936, "bf16", 7), (65536, "fp32", 0)])
def test_greedy_small(V, dtype, C):
    sv.set_stats_grid(C)
    w = small(V, B=9, K=5, dtype=dtype)
    inp = workloads.make(w)
    tok = _greedy_tokens(inp)
    ref = oracle.greedy(host(inp["target"]), tok.numpy())
    g = to_device(inp)
    out = sv.greedy_verify(g["target"], tok.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(out["accept_len"].cpu().numpy(), ref["accept_len"])
    assert np.array_equal(out["out_tokens"].cpu().numpy(), ref["out_tokens"])
    assert sv.read_status(out["workspace"]) == 0
    assert ref["accept_len"].max() > 0      # the chains pass accepted positions too


def test_greedy_ties_masked_rows_and_bad_tokens():
    """Rows with several equal largest logits (the smallest index wins), rows of -inf (argmax 0) and draft
    tokens outside [0, V) (a reject, with the status bit)."""
    B, K, V = 12, 4, 9000
    gen = torch.Generator().manual_seed(9)
    tgt = torch.round(torch.randn((B, K + 1, V), generator=gen) * 2) / 2   # coarse grid: many ties
    tgt[:, :, 100] = tgt.max() + 1.0                                          # a tie at 100 and 7000
    tgt[:, :, 7000] = tgt[:, :, 100]
    tgt[3, 1] = float("-inf")                                                 # a fully masked row
    tgt = tgt.to(torch.bfloat16)
    tok = torch.full((B, K), 100, dtype=torch.int32)
    tok[5, 2] = V + 3
    tok[6, 0] = -1
    ref = oracle.greedy(host(tgt), tok.numpy())
    out = sv.greedy_verify(tgt.cuda(), tok.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(out["accept_len"].cpu().numpy(), ref["accept_len"])
    assert np.array_equal(out["out_tokens"].cpu().numpy(), ref["out_tokens"])
    assert out["accept_len"][3].item() == 1 and out["out_tokens"][3, 1].item() == 0
    assert sv.read_status(out["workspace"]) & sv.STATUS_BAD_TOKEN


def test_greedy_named_workload_full():
    w = workloads.WORKLOADS["sps_llama3_b64_k5"]
    inp = workloads.make(w, device="cuda")
    tok = _greedy_tokens(inp)
    ref = oracle.greedy(host(inp["target"]), tok.numpy())
    out = sv.greedy_verify(inp["target"], tok.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(out["accept_len"].cpu().numpy(), ref["accept_len"])
    assert np.array_equal(out["out_tokens"].cpu().numpy(), ref["out_tokens"])
    assert 0 < ref["accept_len"].mean() < w.K


# ------------------------------------------------------------------------------------------------
# HedgeSpec accept-length estimate over the counterfactual gamma
# ------------------------------------------------------------------------------------------------
def test_accept_length_estimate():
    """The epilogue on the GPU's own gamma against the oracle's formula (same input), and end to end on the
    HedgeSpec pool: the estimate from the GPU gamma against the estimate from the oracle's gamma."""
    w = workloads.WORKLOADS["hedgespec_n7_b32_k5"]
    inp = workloads.make(w, device="cuda")
    out = sv.counterfactual_gamma(inp["target"], inp["drafters"], w.temperature, -1)
    est = sv.accept_length_estimate(out["gamma"])
    torch.cuda.synchronize()
    e_ref, l_ref = oracle.accept_length(out["gamma"].cpu().numpy().astype(np.float64))
    assert np.abs(est["est"].cpu().numpy() - e_ref).max() <= 1e-5
    assert np.abs(est["loss"].cpu().numpy() - l_ref).max() <= 1e-5
    ref = oracle.counterfactual(host(inp["target"]), host(inp["drafters"]), w.temperature, -1)
    e_full, _ = oracle.accept_length(ref["gamma"])
    assert np.abs(est["est"].cpu().numpy() - e_full).max() <= w.K * PROB_TOL
    e = est["est"].cpu().numpy()
    assert np.all((e >= 1) & (e <= w.K + 1))
    # drafters with less noise are estimated to keep longer chains, on average
    assert np.all(np.diff(e.mean(axis=1)) < 0)


# ------------------------------------------------------------------------------------------------
# NormalHedge round
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("N", [1, 7, 21, 33, 64])
def test_normalhedge_round(N):
    """Single rounds from random states against the fp64 oracle, then 300 rounds where one drafter has the
    smaller loss: the GPU learner follows the oracle's and concentrates on it."""
    rng = np.random.default_rng(100 + N)
    for _ in range(20):
        R = rng.normal(0, rng.uniform(0.1, 10), N)
        p = rng.dirichlet(np.ones(N))
        loss = rng.uniform(0, 1, N)
        R_ref, p_ref, _ = oracle.normalhedge(R, loss, p)
        Rg = torch.tensor(R, dtype=torch.float32, device="cuda")
        pg = torch.tensor(p, dtype=torch.float32, device="cuda")
        sv.normalhedge_update(Rg, torch.tensor(loss, dtype=torch.float32, device="cuda"), pg)
        torch.cuda.synchronize()
        assert np.abs(Rg.cpu().numpy() - R_ref).max() <= 1e-5 * (1 + np.abs(R_ref).max())
        assert np.abs(pg.cpu().numpy() - p_ref).max() <= 1e-4
    R = np.zeros(N)
    p = np.full(N, 1.0 / N)
    Rg = torch.zeros(N, device="cuda")
    pg = torch.full((N,), 1.0 / N, device="cuda")
    for t in range(300):
        loss = rng.uniform(0, 1, N)
        loss[N // 2] *= 0.4
        R, p, _ = oracle.normalhedge(R, loss, p)
        sv.normalhedge_update(Rg, torch.tensor(loss, dtype=torch.float32, device="cuda"), pg)
    torch.cuda.synchronize()
    assert np.abs(pg.cpu().numpy() - p).max() <= 1e-3
    if N > 1:
        assert int(pg.argmax()) == N // 2


# ------------------------------------------------------------------------------------------------
# standardised sampling: top-k / top-p on both rows
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("V,dtype,top_k,top_p", [
    (3000, "bf16", 50, 1.0), (3000, "bf16", 0, 0.9), (3000, "bf16", 200, 0.8), (20001, "bf16", 7, 0.95),
    (1000, "fp32", 40, 0.9), (1000, "fp32", 0, 0.5), (128256, "bf16", 1000, 0.9), (151936, "bf16", 0, 0.99),
    (128256, "bf16", 64, 0.95), (4096, "bf16", 256, 1.0), (65536, "fp32", 256, 0.7), (2000, "bf16", 257, 1.0),
])
def test_verify_filtered_small(V, dtype, top_k, top_p):
    w = small(V, B=8, K=4, dtype=dtype, T=0.9, sigma=1.0)
    inp = workloads.make(w)
    ref = oracle.verify_filtered(host(inp["target"]), host(inp["draft"]), inp["tokens"].numpy(),
                                 inp["seeds"].numpy().astype(np.uint64), w.temperature, top_k, top_p)
    g = to_device(inp)
    out = sv.verify_filtered(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature, top_k, top_p)
    torch.cuda.synchronize()
    # top-k up to 1024 on rows of whole 16-byte words takes the line-maxima bound kernel (6), the rest the
    # radix threshold kernel alone (7)
    eb = 2 if dtype == "bf16" else 4
    assert sv.last_plan()["kernel"] == (6 if 0 < top_k <= 1024 and top_k < V and (V * eb) % 16 == 0 else 7)
    # A top-p threshold can land one value off the oracle's when the mass boundary falls within fp32
    # resolution of a partial sum; that moves p(t), Z and the CDF by about one element's mass, which the
    # bar's tolerance and near-tie rules cover.
    assert_diag(out, ref)
    assert_chain(out, ref, w.K)
    assert sv.read_status(out["workspace"]) == 0


def test_verify_filtered_ties():
    """Rows with many equal logits: the keys at or above top-k's bound (the k-th largest of the CTA threads'
    own maxima) can outnumber the candidate list, and every copy of the threshold value is kept."""
    B, K, V = 3, 2, 12000
    gen = torch.Generator().manual_seed(3)
    levels = torch.tensor([0.0, 1.0, 2.0, 3.5], dtype=torch.float32)
    target = levels[torch.randint(0, 4, (B, K + 1, V), generator=gen)]
    target[0] = 2.0                                       # one position flat: every key ties
    draft = target[:, :K] + 0.5 * levels[torch.randint(0, 4, (B, K, V), generator=gen)]
    tokens = torch.randint(0, V, (B, K), generator=gen, dtype=torch.int32)
    seeds = torch.arange(B, dtype=torch.int64) + 77
    for top_k, top_p in ((100, 1.0), (7, 0.9), (256, 0.5)):
        for dt in (torch.bfloat16, torch.float32):
            t, d = target.to(dt), draft.to(dt)
            ref = oracle.verify_filtered(host(t), host(d), tokens.numpy(), seeds.numpy().astype(np.uint64), 1.0,
                                         top_k, top_p)
            out = sv.verify_filtered(t.cuda(), d.cuda(), tokens.cuda(), seeds.cuda(), 1.0, top_k, top_p)
            torch.cuda.synchronize()
            assert_diag(out, ref)
            assert_chain(out, ref, K)
            assert sv.read_status(out["workspace"]) == 0


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_verify_filtered_signed_zeros(dt):
    """Thresholds at zero on rows full of +0 and -0: the keys order -0 below +0, the kept set and the row
    normalisers take both (a float comparison), as the oracle's values do."""
    B, K, V = 4, 3, 2000
    gen = torch.Generator().manual_seed(11)
    levels = torch.tensor([-1.0, -0.0, 0.0, 0.5], dtype=torch.float32)
    target = levels[torch.randint(0, 4, (B, K + 1, V), generator=gen)]
    target[:, :, ::97] = 2.0
    draft = levels[torch.randint(0, 4, (B, K, V), generator=gen)]
    tokens = torch.randint(0, V, (B, K), generator=gen, dtype=torch.int32)
    seeds = torch.arange(B, dtype=torch.int64) + 5
    n_pos = int((target[0, 0] > 0).sum())
    for top_k, top_p in ((n_pos + 10, 1.0), (n_pos + 10, 0.97), (900, 0.999)):
        t, d = target.to(dt), draft.to(dt)
        ref = oracle.verify_filtered(host(t), host(d), tokens.numpy(), seeds.numpy().astype(np.uint64), 0.8,
                                     top_k, top_p)
        out = sv.verify_filtered(t.cuda(), d.cuda(), tokens.cuda(), seeds.cuda(), 0.8, top_k, top_p)
        torch.cuda.synchronize()
        assert sv.last_plan()["kernel"] == 6
        assert_diag(out, ref)
        assert_chain(out, ref, K)
        assert sv.read_status(out["workspace"]) == 0


def test_verify_filtered_lean_launch():
    """The launch the benchmark times (no diag, so only the drawn position's pass, from the kept lists) on
    config 2's row shapes against the oracle, and the same tokens as the call with diag."""
    w = small(128256, B=8, K=5, T=1.0, sigma=1.5)
    inp = workloads.make(w)
    ref = oracle.verify_filtered(host(inp["target"]), host(inp["draft"]), inp["tokens"].numpy(),
                                 inp["seeds"].numpy().astype(np.uint64), w.temperature, 64, 0.95)
    g = to_device(inp)
    lean = sv.verify_filtered(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature, 64, 0.95,
                              want_diag=False)
    full = sv.verify_filtered(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature, 64, 0.95)
    torch.cuda.synchronize()
    assert sv.last_plan()["kernel"] == 6
    assert_chain(lean, ref, w.K)
    assert torch.equal(lean["accept_len"], full["accept_len"])
    assert torch.equal(lean["out_tokens"], full["out_tokens"])
    assert sv.read_status(lean["workspace"]) == 0


def test_verify_filtered_without_filters_is_verify():
    w = small(50000, B=6, K=4)
    g = to_device(workloads.make(w))
    a = sv.verify(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature)
    f = sv.verify_filtered(g["target"], g["draft"], g["tokens"], g["seeds"], w.temperature, 0, 1.0)
    torch.cuda.synchronize()
    for k in ("accept_len", "out_tokens", "diag"):
        assert torch.equal(a[k], f[k])


# ------------------------------------------------------------------------------------------------
# the residual draw's float-float exp2 (its large elements), against fp64
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.7, 2.3])
def test_ff_exp2_building_block(T):
    import ctypes
    rng = np.random.default_rng(7)
    n = 1 << 16
    # d = x - M of bf16 logits (exact in float), row offsets l = -log2 S as a float pair
    x = torch.tensor(rng.normal(0, 4, n), dtype=torch.float32).to(torch.bfloat16).float()
    M = torch.tensor(rng.normal(8, 2, n), dtype=torch.float32).to(torch.bfloat16).float()
    d = torch.minimum(x - M, torch.zeros(n))
    l64 = -np.log2(rng.uniform(1.0, 50.0, n))
    l_hi = torch.tensor(l64, dtype=torch.float32)
    l_lo = torch.tensor(l64 - l_hi.double().numpy(), dtype=torch.float32)
    dd, lh, ll = d.cuda(), l_hi.cuda(), l_lo.cuda()
    out = torch.empty(2 * n, dtype=torch.float32, device="cuda")
    lib = sv.load()
    P = ctypes.c_void_p
    rc = lib.spec_debug_exp2ff(P(dd.data_ptr()), P(lh.data_ptr()), P(ll.data_ptr()), P(out.data_ptr()), n,
                               ctypes.c_float(T), P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    o = out.cpu().double().numpy().reshape(n, 2)
    got = o[:, 0] + o[:, 1]
    c = 1.0 / (np.log(2.0) * float(np.float32(T)))   # the temperature as the C ABI receives it
    exact = np.exp2(d.double().numpy() * c + l_hi.double().numpy() + l_lo.double().numpy())
    keep = exact > 1e-30
    rel = np.abs(got[keep] - exact[keep]) / exact[keep]
    assert rel.max() < 1e-10, rel.max()


# ------------------------------------------------------------------------------------------------
# NormalHedge under delayed, censored feedback (one learner per sequence), against the oracle
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("N,B,K,objective", [(3, 5, 5, 0), (21, 8, 8, 0), (7, 4, 5, 1), (64, 3, 8, 1), (2, 6, 1, 1)])
def test_hedge_feedback_queue(N, B, K, objective):
    rng = np.random.default_rng(300 + N + K)
    T = 80
    gamma = rng.uniform(0.05, 0.95, (T, N, B, K))
    gamma[:, N // 2] = np.minimum(gamma[:, N // 2] + 0.1, 1.0)   # one drafter better on average
    L = rng.integers(0, K + 1, (T, B)).astype(np.int32)
    w_ref, a_ref = oracle.hedge_feedback(gamma, L, objective)
    hf = sv.HedgeFeedback(N, B, K, objective)
    worst = 0.0
    for t in range(T):
        g = torch.tensor(gamma[t], dtype=torch.float32, device="cuda")
        w = hf.push(g, torch.tensor(L[t], device="cuda"))
        torch.cuda.synchronize()
        assert np.array_equal(hf.applied.cpu().numpy(), a_ref[t])
        worst = max(worst, float(np.abs(w.cpu().numpy() - w_ref[t]).max()))
    assert worst <= 2e-3, worst
    assert np.all(hf.status().numpy() == 0)


def test_hedge_feedback_bad_length_skips_the_round():
    """An accepted length outside [0, K] skips that sequence's round and sets its status bit; the other
    sequences are unaffected."""
    N, B, K, T = 4, 3, 4, 12
    rng = np.random.default_rng(310)
    gamma = rng.uniform(0.1, 0.9, (T, N, B, K))
    L = rng.integers(0, K + 1, (T, B)).astype(np.int32)
    hf = sv.HedgeFeedback(N, B, K, 0)
    for t in range(T):
        Lt = L[t].copy()
        if t == 5:
            Lt[1] = K + 3
        hf.push(torch.tensor(gamma[t], dtype=torch.float32, device="cuda"), torch.tensor(Lt, device="cuda"))
    torch.cuda.synchronize()
    keep = [t for t in range(T) if t != 5]
    w_ref, a_ref = oracle.hedge_feedback(gamma, L, 0)
    w_skip, a_skip = oracle.hedge_feedback(gamma[keep][:, :, 1:2], L[keep][:, 1:2], 0)
    st = hf.status().numpy()
    assert st[1] == 1 and st[0] == 0 and st[2] == 0
    assert hf.applied.cpu().numpy()[1] == a_skip[-1, 0]
    assert np.abs(hf.weights.cpu().numpy()[1] - w_skip[-1, 0]).max() <= 2e-3
    assert np.abs(hf.weights.cpu().numpy()[[0, 2]] - w_ref[-1, [0, 2]]).max() <= 2e-3

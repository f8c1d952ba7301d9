"""Pins of the fp64 oracle to facts fixed outside itself (CPU only).

Sources: the lossless-proof tutorial "Speculative Decoding 为什么是 Lossless 的 — 详细证明教程" (the
worked cat/dog/fish example of §2.3/§6/§7.1, the special cases of §7.2/§7.3, the pitfalls of §8 Q1/Q2,
the chain of §9.1); the HedgeSpec notes "Not-a-Bandit: Provably No-Regret Drafter Selection in
Speculative Decoding for LLMs" (Key design 1: gamma = 1 - TV); the Cactus notes "Cactus: Accelerating
Auto-Regressive Decoding with Constrained Acceptance Speculative Sampling" (Key design 1-3: gamma*,
closed-form h, delta = 0 is standard speculative sampling, the KL bound when gamma* <= 0.5, and the
Theorem 3 bound KL(h_alg || target) <= KL(draft || target)); and the Philox4x32-10 known answers.

Exact laws are obtained by enumerating the oracle's own decisions over the whole grid of
uniforms (bisection on the monotone accept and inverse-CDF decisions), so a wrong sign, index or term
anywhere in the accept test, the residual or the inverse CDF changes an enumerated probability.
"""
import math
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GRID = 1 << 23          # the oracle's uniforms are (k + 1/2) / 2^23


def _golden_kv(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *vals = line.split()
            d[k] = np.array([float(v) for v in vals])
    return d


# ----------------------------------------------------------------------------------------------
# enumeration helpers (drive the oracle's decisions; no re-implementation of the rule)
# ----------------------------------------------------------------------------------------------
def accept_fraction(h, pd, t):
    """Fraction of the grid uniforms r that the oracle accepts for candidate t."""
    lo, hi = 0, GRID
    while lo < hi:
        mid = (lo + hi) // 2
        _, acc, *_ = oracle.sample_one(h, pd, t, (mid + 0.5) / GRID, 0.5)
        if acc:
            lo = mid + 1
        else:
            hi = mid
    return lo / GRID


def resample_law(h, pd, t, mutation=0):
    """Law of the token the oracle emits after a reject at candidate t, over the u grid."""
    V = len(h)
    r_rej = (GRID - 0.5) / GRID
    _, acc, *_ = oracle.sample_one(h, pd, t, r_rej, 0.5, mutation)
    if acc:
        return None

    def tok(k):
        return oracle.sample_one(h, pd, t, r_rej, (k + 0.5) / GRID, mutation)[0]

    law = np.zeros(V)
    start = 0
    while start < GRID:
        x = tok(start)
        lo, hi = start, GRID          # first k with tok(k) > x
        while lo < hi:
            mid = (lo + hi) // 2
            if tok(mid) > x:
                hi = mid
            else:
                lo = mid + 1
        law[x] += (lo - start) / GRID
        start = lo
    return law


def output_law(h, pd, mutation=0, h_of=None):
    """P(output = x) of one verification step with the draft token t ~ pd, enumerated exactly.
    h_of(t) gives the target distribution used for candidate t (Cactus); default h."""
    V = len(pd)
    law = np.zeros(V)
    for t in range(V):
        if pd[t] == 0.0:
            continue
        ht = h if h_of is None else h_of(t)
        a = accept_fraction(ht, pd, t)
        law[t] += pd[t] * a
        if a < 1.0:
            law += pd[t] * (1.0 - a) * resample_law(ht, pd, t, mutation)
    return law


# ----------------------------------------------------------------------------------------------
# Philox
# ----------------------------------------------------------------------------------------------
def test_philox_known_answers():
    n = 0
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            left, right = line.split("|")
            vals = [int(v, 16) for v in left.split()]
            want = [int(v, 16) for v in right.split()]
            got = oracle.philox4x32_10(vals[:4], vals[4:6])
            assert [int(g) for g in got] == want
            n += 1
    assert n == 3


def test_uniform_grid_and_streams():
    us = [oracle.uniform(s, b, j, st) for s in (0, 1, 2**40 + 3) for b in range(4) for j in range(6) for st in (0, 1)]
    for u in us:
        assert 0.0 < u < 1.0
        k = u * GRID - 0.5
        assert k == int(k)                      # on the (k + 1/2) 2^-23 grid
        assert float(np.float32(u)) == u        # exact in fp32
    assert len(set(us)) == len(us)              # counter and key both reach the output
    w0 = oracle.philox4x32_10([3, 2, 1, 0], [7, 0])[0]
    assert oracle.uniform(7, 2, 3, 1) == ((int(w0) >> 9) + 0.5) / GRID


def test_uniform_is_uniform():
    us = np.array([oracle.uniform(11, b, j, 0) for b in range(200) for j in range(50)])
    assert stats.kstest(us, "uniform").pvalue > 1e-4


# ----------------------------------------------------------------------------------------------
# softmax / inverse CDF against library routines
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_softmax_matches_scipy(T):
    rng = np.random.default_rng(5)
    x = rng.normal(0, 3, 4099)
    assert np.allclose(oracle.softmax(x, T), special.softmax(x / T), rtol=1e-13, atol=1e-300)
    assert np.allclose(oracle.softmax(x + 123.0, T), oracle.softmax(x, T), rtol=1e-12, atol=0)


def test_softmax_masked_logits():
    x = np.array([-np.inf, math.log(0.75), -np.inf, math.log(0.25)])
    p = oracle.softmax(x, 1.0)
    assert p[0] == 0.0 and p[2] == 0.0
    assert np.allclose(p, [0, 0.75, 0, 0.25], atol=1e-15)


def test_inverse_cdf_matches_searchsorted():
    rng = np.random.default_rng(9)
    for _ in range(200):
        w = rng.random(37) * (rng.random(37) > 0.3)
        if w.sum() == 0:
            continue
        target = rng.random() * w.sum()
        x, margin = oracle.inverse_cdf(w, target)
        c = np.cumsum(w)
        assert x == int(np.searchsorted(c, target, side="right"))
        assert w[x] > 0
        assert margin == pytest.approx(min(target - (c[x] - w[x]), c[x] - target), abs=1e-12)


def test_inverse_cdf_never_picks_zero_mass():
    w = np.array([0.0, 0.5, 0.0, 0.5, 0.0])
    for target in [0.0, 0.25, 0.5, 0.75, 0.9999999, 1.0, 1.5]:
        x, _ = oracle.inverse_cdf(w, target)
        assert x in (1, 3)


# ----------------------------------------------------------------------------------------------
# the worked example of the lossless tutorial
# ----------------------------------------------------------------------------------------------
def test_worked_example_quantities():
    g = _golden_kv("sps_worked_example.txt")
    p, q = g["p"], g["q"]
    for t in range(3):
        assert accept_fraction(p, q, t) == pytest.approx(g["a"][t], abs=2.0 / GRID)
        _, _, Z, _, _ = oracle.sample_one(p, q, t, 0.5, 0.5)
        assert Z == pytest.approx(g["Z"][0], abs=1e-15)
    # acceptance path: P(x and accept) = q(x) a(x) = min(p, q)(x)
    for t in range(3):
        assert q[t] * accept_fraction(p, q, t) == pytest.approx(g["p_x_accept"][t], abs=1e-6)
    # reject path only ever emits cat (p' = (1, 0, 0)); dog is the only candidate that can be rejected
    assert resample_law(p, q, 1) == pytest.approx(g["p_prime"], abs=0)
    assert resample_law(p, q, 0) is None and resample_law(p, q, 2) is None
    law = output_law(p, q)
    assert law == pytest.approx(g["p_out"], abs=1e-6)
    # P(x and reject) = (p - q)+
    acc_part = np.array([q[t] * accept_fraction(p, q, t) for t in range(3)])
    assert law - acc_part == pytest.approx(g["p_x_reject"], abs=1e-6)


def test_worked_example_batched_counterfactual():
    g = _golden_kv("sps_worked_example.txt")
    tgt = np.log(np.array([[g["p"], g["p"]]], dtype=np.float64)).astype(np.float32)
    drf = np.log(np.array([[[g["q"]]]], dtype=np.float64)).astype(np.float32)
    out = oracle.counterfactual(tgt, drf)
    assert out["gamma"][0, 0, 0] == pytest.approx(g["p_accept"][0], abs=1e-7)
    assert out["tv"][0, 0, 0] == pytest.approx(1 - g["p_accept"][0], abs=1e-7)
    assert out["loss"][0, 0, 0] == pytest.approx(g["Z"][0], abs=1e-7)


def test_pitfall_q1_resample_from_target_is_biased():
    g = _golden_kv("sps_worked_example.txt")
    law = output_law(g["p"], g["q"], mutation=1)
    assert law[0] == pytest.approx(g["q1_p_cat"][0], abs=1e-6)
    assert abs(law[0] - g["p"][0]) > 0.05


def test_pitfall_q2_absolute_difference_is_biased():
    g = _golden_kv("sps_worked_example.txt")
    law = output_law(g["p"], g["q"], mutation=2)
    assert law[1] > g["p"][1] + 0.05           # dog pushed above 0.3
    assert law.sum() == pytest.approx(1.0, abs=1e-6)


def test_perfect_draft_never_rejects():
    rng = np.random.default_rng(1)
    p = special.softmax(rng.normal(0, 2, 6))
    for t in range(6):
        assert accept_fraction(p, p, t) == 1.0
        _, _, Z, _, _ = oracle.sample_one(p, p, t, 0.5, 0.5)
        assert Z == 0.0
    assert output_law(p, p) == pytest.approx(p, abs=1e-6)


def test_disjoint_support_always_rejects_and_resamples_target():
    p = np.array([0.0, 0.75, 0.25])
    q = np.array([1.0, 0.0, 0.0])
    assert accept_fraction(p, q, 0) == 0.0
    _, _, Z, _, _ = oracle.sample_one(p, q, 0, 0.5, 0.5)
    assert Z == pytest.approx(1.0, abs=1e-15)
    assert resample_law(p, q, 0) == pytest.approx(p, abs=1e-6)
    assert output_law(p, q) == pytest.approx(p, abs=1e-6)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_lossless_exact_enumeration_random(seed):
    rng = np.random.default_rng(100 + seed)
    V = 5
    p = special.softmax(rng.normal(0, 2, V))
    q = special.softmax(rng.normal(0, 2, V))
    if seed == 3:
        p[2] = 0.0
        p /= p.sum()
    assert output_law(p, q) == pytest.approx(p, abs=2e-6)


def test_money_identity_and_one_minus_tv():
    rng = np.random.default_rng(3)
    B, K, V, N = 3, 2, 257, 4
    tgt = rng.normal(0, 3, (B, K + 1, V)).astype(np.float32)
    drf = (tgt[None, :, :K] + rng.normal(0, 1.5, (N, B, K, V))).astype(np.float32)
    out = oracle.counterfactual(tgt, drf, temperature=0.8)
    assert np.all(np.abs(out["gamma"] + out["tv"] - 1.0) < 1e-12)
    assert np.all((out["gamma"] > 0) & (out["gamma"] < 1))
    # Z of the verify path equals 1 - gamma (P(reject) = Z, tutorial §6.4 Step 3a)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    v = oracle.verify(tgt, drf[1], tok, np.arange(B, dtype=np.uint64), temperature=0.8)
    assert np.allclose(v["diag"][:, :, 2], 1.0 - out["gamma"][1], atol=1e-12)


def test_gamma_special_cases():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 2, (1, 2, 16)).astype(np.float32)
    out = oracle.counterfactual(x, x[None, :, :1].copy())
    assert out["gamma"][0, 0, 0] == pytest.approx(1.0, abs=1e-14)
    tgt = np.full((1, 2, 4), -np.inf, np.float32)
    tgt[0, :, 2:] = 0.0
    drf = np.full((1, 1, 1, 4), -np.inf, np.float32)
    drf[0, 0, 0, :2] = 0.0
    out = oracle.counterfactual(tgt, drf)
    assert out["gamma"][0, 0, 0] == 0.0


# ----------------------------------------------------------------------------------------------
# batched sampling: chi-square losslessness, mutations, chain
# ----------------------------------------------------------------------------------------------
def _batch_same_rows(p_rows, q_rows, bonus, n, rng):
    """n sequences sharing the same rows; draft tokens drawn from q with numpy's generator."""
    K = len(q_rows)
    V = len(bonus)
    tgt = np.log(np.array([list(p_rows) + [bonus]] * n)).astype(np.float32)
    drf = np.log(np.array([list(q_rows)] * n)).astype(np.float32)
    tok = np.stack([rng.choice(V, size=n, p=q_rows[j] / q_rows[j].sum()) for j in range(K)], 1).astype(np.int32)
    return tgt, drf, tok


def _chi2_p(counts, probs):
    m = probs > 0
    assert counts[~m].sum() == 0
    exp = probs[m] / probs[m].sum() * counts.sum()
    return stats.chisquare(counts[m], exp).pvalue


def test_chi2_lossless_worked_example_and_mutations():
    g = _golden_kv("sps_worked_example.txt")
    rng = np.random.default_rng(7)
    n = 60000
    tgt, drf, tok = _batch_same_rows([g["p"]], [g["q"]], g["p"], n, rng)
    seeds = np.arange(n, dtype=np.uint64) * 7919 + 5
    p_true = g["p"] / g["p"].sum()
    with np.errstate(divide="ignore"):
        pass
    good = oracle.verify(tgt, drf, tok, seeds)
    c = np.bincount(good["out_tokens"][:, 0], minlength=3)
    assert _chi2_p(c, p_true) > 1e-6
    assert abs(good["accept_len"].mean() - g["p_accept"][0]) < 0.01
    for mut in (1, 2):
        bad = oracle.verify(tgt, drf, tok, seeds, mutation=mut)
        c = np.bincount(bad["out_tokens"][:, 0], minlength=3)
        assert _chi2_p(c, p_true) < 1e-6


def test_chi2_chain_levels():
    rng = np.random.default_rng(8)
    V, K, n = 8, 3, 40000
    P = [special.softmax(rng.normal(0, 1.5, V)) for _ in range(K + 1)]
    Q = [special.softmax(np.log(P[j]) + rng.normal(0, 1.0, V)) for j in range(K)]
    tgt, drf, tok = _batch_same_rows(P[:K], Q, P[K], n, rng)
    seeds = np.full(n, 42, dtype=np.uint64)      # one key; the sequence number in the counter separates them
    out = oracle.verify(tgt, drf, tok, seeds)
    L = out["accept_len"]
    for j in range(K + 1):
        reach = L >= j
        c = np.bincount(out["out_tokens"][reach, j], minlength=V)
        assert reach.sum() > 1000
        assert _chi2_p(c, P[j]) > 1e-6, j
    gam = [np.minimum(P[j], Q[j]).sum() for j in range(K)]
    for j in range(K):
        reach = L >= j
        assert abs((L[reach] > j).mean() - gam[j]) < 4 * math.sqrt(gam[j] * (1 - gam[j]) / reach.sum()) + 1e-3
    assert np.all(out["out_tokens"][np.arange(n), L] >= 0)
    assert all(np.all(out["out_tokens"][L == l, l + 1:] == -1) for l in range(K))


def test_counterfactual_gamma_matches_monte_carlo_acceptance():
    rng = np.random.default_rng(12)
    V, n, N = 16, 30000, 3
    p = special.softmax(rng.normal(0, 2, V))
    qs = [special.softmax(np.log(p) + rng.normal(0, s, V)) for s in (0.5, 1.5, 3.0)]
    tgt = np.log(np.array([[p, p]])).astype(np.float32)
    drf = np.log(np.array(qs))[:, None, None, :].astype(np.float32)
    gam = oracle.counterfactual(tgt, drf)["gamma"][:, 0, 0]
    for i in range(N):
        t2, d2, tok = _batch_same_rows([p], [qs[i]], p, n, rng)
        out = oracle.verify(t2, d2, tok, np.arange(n, dtype=np.uint64))
        rate = out["accept_len"].mean()
        sd = math.sqrt(gam[i] * (1 - gam[i]) / n)
        assert abs(rate - gam[i]) < 4 * sd + 1e-3


def test_seq_index_selects_counter():
    rng = np.random.default_rng(13)
    B, K, V = 6, 3, 50
    tgt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    drf = (tgt[:, :K] + rng.normal(0, 2, (B, K, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    seeds = np.arange(B, dtype=np.uint64) + 9
    full = oracle.verify(tgt, drf, tok, seeds)
    sub = [1, 4]
    part = oracle.verify(tgt[sub], drf[sub], tok[sub], seeds[sub], seq_index=np.array(sub))
    assert np.array_equal(part["out_tokens"], full["out_tokens"][sub])
    assert np.array_equal(part["diag"], full["diag"][sub])


def test_bf16_input_is_exact_conversion():
    rng = np.random.default_rng(14)
    x32 = rng.normal(0, 3, (2, 3, 64)).astype(np.float32)
    bits = (x32.view(np.uint32) >> 16).astype(np.uint16)          # truncate to bf16
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    d32 = (back[:, :2] + 0.5).astype(np.float32)
    dbits = (d32.view(np.uint32) >> 16).astype(np.uint16)
    dback = (dbits.astype(np.uint32) << 16).view(np.float32)
    tok = np.zeros((2, 2), np.int32)
    a = oracle.verify(bits, dbits, tok, np.arange(2, dtype=np.uint64))
    b = oracle.verify(back, dback, tok, np.arange(2, dtype=np.uint64))
    assert np.array_equal(a["diag"], b["diag"]) and np.array_equal(a["out_tokens"], b["out_tokens"])


# ----------------------------------------------------------------------------------------------
# Cactus
# ----------------------------------------------------------------------------------------------
def _kl(a, b):
    m = a > 0
    return float(np.sum(a[m] * np.log(a[m] / b[m])))


def test_cactus_closed_form_invariants():
    rng = np.random.default_rng(20)
    for _ in range(300):
        V = int(rng.integers(2, 12))
        pt = special.softmax(rng.normal(0, rng.uniform(0.2, 4), V))
        n = int(rng.integers(0, V))
        delta = float(rng.choice([0.0, 1e-3, 0.05, 0.3, 0.75, 1.0, 3.0]))
        h, gs = oracle.cactus_h(pt, n, delta)
        assert gs >= pt[n] - 1e-15 and gs <= 1.0
        assert h[n] == gs
        assert np.all(h >= 0) and h.sum() == pytest.approx(1.0, abs=1e-12)
        others = np.arange(V) != n
        if pt[n] < 1:
            assert np.allclose(h[others], pt[others] * (1 - gs) / (1 - pt[n]), rtol=1e-13, atol=0)
        if gs <= 0.5:
            assert _kl(h, pt) <= delta + 1e-12
        if delta == 0.0:
            assert gs == pt[n] and np.array_equal(h, pt)


def test_cactus_bonus_largest_at_half():
    qs = np.linspace(0.01, 0.99, 99)
    bonus = []
    for qv in qs:
        _, gs = oracle.cactus_h(np.array([qv, 1 - qv]), 0, 0.02)
        bonus.append(gs - qv)
    assert qs[int(np.argmax(bonus))] == pytest.approx(0.5, abs=0.011)


def test_cactus_delta_zero_is_standard_sps():
    rng = np.random.default_rng(21)
    B, K, V = 16, 4, 300
    tgt = rng.normal(0, 3, (B, K + 1, V)).astype(np.float32)
    drf = (tgt[:, :K] + rng.normal(0, 2, (B, K, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    seeds = np.arange(B, dtype=np.uint64) * 3 + 1
    a = oracle.verify(tgt, drf, tok, seeds, temperature=0.9)
    c = oracle.cactus(tgt, drf, tok, seeds, 0.0, temperature=0.9)
    for k in ("accept_len", "out_tokens", "diag", "accept_margin", "cdf_margin"):
        assert np.array_equal(a[k], c[k]), k
    assert np.array_equal(c["gamma_star"], c["diag"][:, :, 0])


def test_cactus_raises_acceptance():
    rng = np.random.default_rng(22)
    B, K, V = 64, 5, 200
    tgt = rng.normal(0, 3, (B, K + 1, V)).astype(np.float32)
    drf = (tgt[:, :K] + rng.normal(0, 2, (B, K, V))).astype(np.float32)
    tok = np.stack([[rng.choice(V, p=special.softmax(drf[b, j])) for j in range(K)] for b in range(B)]).astype(np.int32)
    seeds = np.arange(B, dtype=np.uint64)
    L0 = oracle.cactus(tgt, drf, tok, seeds, 0.0)["accept_len"]
    L1 = oracle.cactus(tgt, drf, tok, seeds, 1.0)["accept_len"]
    assert np.all(L1 >= L0)          # same uniforms, gamma* >= p_target(n): acceptance is monotone in delta
    assert L1.mean() > L0.mean()


@pytest.mark.parametrize("delta", [0.0, 0.2, 1.0])
def test_cactus_exact_law_and_theorem3(delta):
    rng = np.random.default_rng(30 + int(10 * delta))
    V = 5
    pt = special.softmax(rng.normal(0, 1.5, V))
    pd = special.softmax(np.log(pt) + rng.normal(0, 1.0, V))
    hs = [oracle.cactus_h(pt, n, delta)[0] for n in range(V)]
    law = output_law(None, pd, h_of=lambda t: hs[t])
    # law of the algorithm, stated directly: accept n w.p. min(1, h_n(n)/pd(n)); else (h_n - pd)+ / Z
    direct = np.zeros(V)
    for n in range(V):
        h = hs[n]
        a = min(1.0, h[n] / pd[n])
        direct[n] += pd[n] * a
        res = np.maximum(h - pd, 0.0)
        if a < 1.0:
            direct += pd[n] * (1 - a) * res / res.sum()
    assert law == pytest.approx(direct, abs=2e-6)
    if delta == 0.0:
        assert law == pytest.approx(pt, abs=2e-6)
    else:
        # Cactus Theorem 3 (translated): D(h_alg || target) <= D(draft || target)
        assert _kl(law, pt) <= _kl(pd, pt) + 1e-6
        # every candidate's own acceptance rises: gamma* >= p_target(n)
        assert law.sum() == pytest.approx(1.0, abs=1e-6)


def test_cactus_batched_chi2():
    rng = np.random.default_rng(40)
    V, n, delta = 6, 50000, 0.5
    pt = special.softmax(rng.normal(0, 1.5, V))
    pd = special.softmax(np.log(pt) + rng.normal(0, 1.2, V))
    hs = [oracle.cactus_h(pt, k, delta)[0] for k in range(V)]
    direct = np.zeros(V)
    for k in range(V):
        h = hs[k]
        a = min(1.0, h[k] / pd[k])
        res = np.maximum(h - pd, 0.0)
        direct[k] += pd[k] * a
        if a < 1.0:
            direct += pd[k] * (1 - a) * res / res.sum()
    tgt, drf, tok = _batch_same_rows([pt], [pd], pt, n, rng)
    out = oracle.cactus(tgt, drf, tok, np.arange(n, dtype=np.uint64) + 77, delta)
    c = np.bincount(out["out_tokens"][:, 0], minlength=V)
    assert _chi2_p(c, direct) > 1e-6
    assert _chi2_p(c, pt) < 1e-6        # lossy by design for delta > 0


# ----------------------------------------------------------------------------------------------
# Cactus gamma* as the root of the divergence constraint (no Taylor step)
# ----------------------------------------------------------------------------------------------
def test_cactus_exact_root_meets_the_constraint():
    """[Cactus] Key design 2: gamma* is the root of D_KL(h || target) = delta on [q(n), 1] (clamped). The
    divergence is recomputed here from the whole distribution h, not from the oracle's two-term form."""
    rng = np.random.default_rng(50)
    for _ in range(400):
        V = int(rng.integers(2, 40))
        pt = special.softmax(rng.normal(0, rng.uniform(0.2, 5), V))
        n = int(rng.integers(0, V))
        delta = float(rng.choice([1e-4, 1e-2, 0.1, 0.5, 0.75, 1.0, 3.0]))
        h, gs = oracle.cactus_h(pt, n, delta, exact=True)
        q = pt[n]
        assert q <= gs <= 1.0
        assert h.sum() == pytest.approx(1.0, abs=1e-12) and h[n] == gs
        if np.log(1.0 / q) > delta:      # a root below 1 exists
            assert _kl(h, pt) == pytest.approx(delta, rel=1e-9, abs=1e-12)
        else:
            assert gs == 1.0
        assert oracle.cactus_kl(q, gs) == pytest.approx(_kl(h, pt), rel=1e-9, abs=1e-13)


def test_cactus_exact_root_against_taylor():
    """Corollary 6 of the page: where the Taylor gamma* is at most 0.5 it meets KL <= delta, so it lies at or
    below the root; as delta -> 0 the two agree to first order (the Taylor step drops an O(delta) term)."""
    rng = np.random.default_rng(51)
    for _ in range(2000):
        q = float(np.exp(rng.uniform(np.log(1e-6), np.log(0.999))))
        delta = float(np.exp(rng.uniform(np.log(1e-8), np.log(3.0))))
        ex = oracle.cactus_gamma_kl(q, delta)
        ty = min(q + np.sqrt(2 * delta * q * (1 - q)), 1.0)
        if ty <= 0.5:
            assert ty <= ex + 1e-15
        if delta <= 1e-6:
            assert abs(ex - ty) <= 10 * delta
    for q in (1e-4, 0.2, 0.6, 0.97):
        assert oracle.cactus_gamma_kl(q, 0.0) == q
        gs = [oracle.cactus_gamma_kl(q, d) for d in (1e-5, 1e-3, 0.1, 0.5, 2.0)]
        assert all(a <= b for a, b in zip(gs, gs[1:]))        # monotone in delta
    assert oracle.cactus_gamma_kl(0.0, 0.5) == 0.0             # q = 0: every g > 0 has infinite divergence
    assert oracle.cactus_gamma_kl(1.0, 0.5) == 1.0


@pytest.mark.parametrize("delta", [0.2, 1.0])
def test_cactus_exact_root_law(delta):
    """The chain with the exact gamma* produces the law its acceptance rule states (exact enumeration), and
    the batched oracle reports the root as gamma*."""
    rng = np.random.default_rng(60 + int(10 * delta))
    V = 5
    pt = special.softmax(rng.normal(0, 1.5, V))
    pd = special.softmax(np.log(pt) + rng.normal(0, 1.0, V))
    hs = [oracle.cactus_h(pt, n, delta, exact=True)[0] for n in range(V)]
    law = output_law(None, pd, h_of=lambda t: hs[t])
    direct = np.zeros(V)
    for n in range(V):
        h = hs[n]
        a = min(1.0, h[n] / pd[n])
        direct[n] += pd[n] * a
        res = np.maximum(h - pd, 0.0)
        if a < 1.0:
            direct += pd[n] * (1 - a) * res / res.sum()
    assert law == pytest.approx(direct, abs=2e-6)
    B, K = 8, 3
    tgt = rng.normal(0, 2, (B, K + 1, 40)).astype(np.float32)
    drf = (tgt[:, :K] + rng.normal(0, 1, (B, K, 40))).astype(np.float32)
    tok = rng.integers(0, 40, (B, K)).astype(np.int32)
    out = oracle.cactus(tgt, drf, tok, np.arange(B, dtype=np.uint64), delta, exact=True)
    for b in range(B):
        for j in range(K):
            q = special.softmax(tgt[b, j].astype(np.float64))[tok[b, j]]
            # the batched entry takes delta as the C ABI does, a 32-bit float
            assert out["gamma_star"][b, j] == pytest.approx(oracle.cactus_gamma_kl(q, float(np.float32(delta))),
                                                            abs=1e-12)


# ----------------------------------------------------------------------------------------------
# greedy verification (temperature 0)
# ----------------------------------------------------------------------------------------------
def _greedy_case(rng, B=24, K=5, V=60, ties=False):
    tgt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    if ties:   # round to a coarse grid so that rows have several equal largest logits
        tgt = np.round(tgt * 2) / 2
    drf = (tgt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    am = tgt.argmax(axis=2)
    # drafts: the target's argmax most of the time, another token otherwise
    tok = np.where(rng.random((B, K)) < 0.7, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    return tgt, drf, tok


def test_greedy_is_the_chain_on_one_hot_rows():
    """The greedy result equals [SpS] §5.1 / §9.1 run on one-hot target and draft rows (logit 0 at the
    argmax, -inf elsewhere), for any seeds: the uniforms and the draft rows drop out."""
    rng = np.random.default_rng(70)
    for ties in (False, True):
        tgt, drf, tok = _greedy_case(rng, ties=ties)
        g = oracle.greedy(tgt, tok)
        am_t = tgt.argmax(axis=2)                # numpy: first index of the largest value
        am_d = drf.argmax(axis=2)
        oh_t = np.full(tgt.shape, -np.inf, dtype=np.float32)
        oh_d = np.full(drf.shape, -np.inf, dtype=np.float32)
        np.put_along_axis(oh_t, am_t[..., None], 0.0, axis=2)
        np.put_along_axis(oh_d, am_d[..., None], 0.0, axis=2)
        for seed0 in (0, 999):
            seeds = np.arange(len(tok), dtype=np.uint64) + seed0
            v = oracle.verify(oh_t, oh_d, tok, seeds)
            assert np.array_equal(v["accept_len"], g["accept_len"])
            assert np.array_equal(v["out_tokens"], g["out_tokens"])


def test_greedy_is_the_low_temperature_limit():
    """With greedy drafts (each draft token the argmax of its draft row) and no ties, the general algorithm
    at T = 1e-3 gives the greedy outputs: q(t) -> 1 and p(t) -> 1 or 0 as T -> 0. (For a token that is the
    argmax of neither row the ratio p(t)/q(t) has no such limit, which is why greedy is defined on the
    one-hot rows.)"""
    rng = np.random.default_rng(71)
    tgt, drf, _ = _greedy_case(rng, B=40)
    tok = drf.argmax(axis=2).astype(np.int32)
    g = oracle.greedy(tgt, tok)
    v = oracle.verify(tgt, drf, tok, np.arange(40, dtype=np.uint64) + 5, temperature=1e-3)
    assert np.array_equal(v["accept_len"], g["accept_len"])
    assert np.array_equal(v["out_tokens"], g["out_tokens"])
    assert 0 < g["accept_len"].mean() < 5


def test_greedy_chain_structure():
    rng = np.random.default_rng(72)
    tgt, _, tok = _greedy_case(rng, B=50, ties=True)
    g = oracle.greedy(tgt, tok)
    am = tgt.argmax(axis=2)
    for b in range(50):
        L = g["accept_len"][b]
        assert np.array_equal(g["out_tokens"][b, :L], tok[b, :L]) and np.all(tok[b, :L] == am[b, :L])
        assert L == 5 or tok[b, L] != am[b, L]
        assert g["out_tokens"][b, L] == am[b, L]
        assert np.all(g["out_tokens"][b, L + 1:] == -1)


# ----------------------------------------------------------------------------------------------
# HedgeSpec accept-length estimate (the page's display is missing: the reading is pinned through its own
# mathematics, not against the paper's formula)
# ----------------------------------------------------------------------------------------------
def test_accept_length_estimate_identities():
    rng = np.random.default_rng(80)
    N, B, K = 3, 7, 6
    g = rng.uniform(0, 1, (N, B, K))
    est, loss = oracle.accept_length(g)
    assert np.all((est >= 1.0) & (est <= K + 1))                        # the range the page states
    assert np.allclose(est + loss, K + 1, atol=1e-14)
    # constant gamma: the geometric series (1 - gamma^(K+1)) / (1 - gamma)
    for gv in (0.0, 0.3, 0.9, 1.0):
        e, _ = oracle.accept_length(np.full((1, 1, K), gv))
        ref = K + 1 if gv == 1.0 else (1 - gv ** (K + 1)) / (1 - gv)
        assert e[0, 0] == pytest.approx(ref, abs=1e-13)


def test_accept_length_estimate_is_the_chain_expectation():
    """Exact enumeration: a chain whose level k is accepted with probability gamma_k (given the levels before
    it) emits 1 + (number of accepted levels) tokens; its expectation is the estimate."""
    rng = np.random.default_rng(81)
    K = 5
    for _ in range(20):
        g = rng.uniform(0, 1, K)
        expect = 0.0
        for outcome in range(2 ** K):
            bits = [(outcome >> k) & 1 for k in range(K)]
            p = np.prod([g[k] if bits[k] else 1 - g[k] for k in range(K)])
            L = next((k for k in range(K) if not bits[k]), K)   # the first reject stops the chain
            expect += p * (1 + L)
        e, _ = oracle.accept_length(g[None, None, :])
        assert e[0, 0] == pytest.approx(expect, abs=1e-12)


def test_accept_length_estimate_matches_simulated_chains():
    """The estimate from the counterfactual gamma of one drafter against the mean length of many simulated
    speculative-sampling chains over the same rows (different uniforms): within 5 standard errors."""
    rng = np.random.default_rng(82)
    K, V, n = 4, 30, 40000
    pt = [special.softmax(rng.normal(0, 1.5, V)) for _ in range(K + 1)]
    pd = [special.softmax(np.log(pt[j]) + rng.normal(0, 0.8, V)) for j in range(K)]
    # gamma at every level: sum_x min(p, q) (the probability of accepting any draft token there)
    gam = np.array([np.minimum(pt[j], pd[j]).sum() for j in range(K)])
    est, _ = oracle.accept_length(gam[None, None, :])
    # independent chains: draft tokens sampled from q at each level, accept with min(1, p/q)
    toks = np.stack([rng.choice(V, size=n, p=pd[j]) for j in range(K)], axis=1)
    acc = rng.uniform(0, 1, (n, K)) < np.stack([np.minimum(1, pt[j][toks[:, j]] / pd[j][toks[:, j]])
                                                for j in range(K)], axis=1)
    L = np.where(acc.all(axis=1), K, np.argmin(acc, axis=1))
    m, se = (1 + L).mean(), (1 + L).std() / np.sqrt(n)
    assert abs(est[0, 0] - m) < 5 * se


# ----------------------------------------------------------------------------------------------
# NormalHedge (Chaudhuri, Freund, Hsu 2009), the learner the HedgeSpec notes name
# ----------------------------------------------------------------------------------------------
def test_normalhedge_scale_and_weights():
    rng = np.random.default_rng(90)
    for _ in range(300):
        N = int(rng.integers(2, 40))
        R = rng.normal(0, rng.uniform(0.1, 20), N)
        p0 = np.full(N, 1.0 / N)
        Rn, p, c = oracle.normalhedge(R, np.zeros(N), p0)       # zero losses: the regrets stay
        assert np.array_equal(Rn, R)
        pos = np.maximum(R, 0)
        if not np.any(pos > 0):
            assert c == 0 and np.allclose(p, 1.0 / N)
            continue
        # the scale solves mean exp(R+^2 / 2c) = e
        assert np.mean(np.exp(pos ** 2 / (2 * c))) == pytest.approx(np.e, rel=1e-10)
        assert p.sum() == pytest.approx(1.0, abs=1e-12) and np.all(p >= 0)
        assert np.all(p[pos == 0] == 0)                            # no weight without positive regret
        w = pos / c * np.exp(pos ** 2 / (2 * c))
        assert np.allclose(p, w / w.sum(), rtol=1e-9, atol=1e-15)


def test_normalhedge_regret_update_and_learning():
    rng = np.random.default_rng(91)
    N, T = 7, 400
    R = np.zeros(N)
    p = np.full(N, 1.0 / N)
    for t in range(T):
        loss = rng.uniform(0, 1, N)
        loss[3] *= 0.5                                   # expert 3 is the best on average
        lp = p @ loss
        Rn, pn, _ = oracle.normalhedge(R, loss, p)
        assert np.allclose(Rn, R + lp - loss, atol=1e-12)
        # shifting every loss by a constant changes neither the regrets nor the weights
        Rs, ps, _ = oracle.normalhedge(R, loss + 3.0, p)
        assert np.allclose(Rs, Rn, atol=1e-9) and np.allclose(ps, pn, atol=1e-9)
        R, p = Rn, pn
    assert np.argmax(p) == 3 and p[3] > 0.5


# ----------------------------------------------------------------------------------------------
# NormalHedge under delayed, censored feedback ([Hedge] Key design 3; reading in spec_oracle_hedge_feedback)
# ----------------------------------------------------------------------------------------------
def _hf_rounds(rng, T, N, B, K, lo=0.05, hi=0.95):
    gamma = rng.uniform(lo, hi, (T, N, B, K))
    L = rng.integers(0, K + 1, (T, B)).astype(np.int32)
    return gamma, L


def _revealed(gamma, L, b):
    """The feedback items of sequence b in order: levels j < min(L_t + 1, K) of each round."""
    T, N, B, K = gamma.shape
    items = []
    for t in range(T):
        for j in range(min(int(L[t, b]) + 1, K)):
            items.append((t, gamma[t, :, b, j]))
    return items


def test_hedge_feedback_reduces_to_normalhedge():
    """Objective 0 is plain NormalHedge over 1 - gamma of the revealed levels, in order; with every level
    revealed (L = K) that is K NormalHedge rounds per round."""
    rng = np.random.default_rng(120)
    T, N, B, K = 12, 5, 3, 4
    gamma, L = _hf_rounds(rng, T, N, B, K)
    L[:, 0] = K                                            # sequence 0: nothing censored
    w, applied = oracle.hedge_feedback(gamma, L, objective=0)
    for b in range(B):
        R, p = np.zeros(N), np.full(N, 1.0 / N)
        items = _revealed(gamma, L, b)
        n = 0
        for t in range(T):
            while n < len(items) and items[n][0] <= t:
                R, p, _ = oracle.normalhedge(R, 1.0 - items[n][1], p)
                n += 1
            assert applied[t, b] == n
            assert np.allclose(w[t, b], p, atol=1e-12)
    assert np.array_equal(applied[:, 0], K * np.arange(1, T + 1))


def test_hedge_feedback_censored_levels_never_count():
    """Levels at or past min(L + 1, K) are censored: any value there leaves every weight unchanged."""
    rng = np.random.default_rng(121)
    T, N, B, K = 15, 6, 4, 5
    gamma, L = _hf_rounds(rng, T, N, B, K)
    for obj in (0, 1):
        w, a = oracle.hedge_feedback(gamma, L, objective=obj)
        g2 = gamma.copy()
        for t in range(T):
            for b in range(B):
                g2[t, :, b, min(int(L[t, b]) + 1, K):] = rng.uniform(0, 1, (N, K - min(int(L[t, b]) + 1, K)))
        w2, a2 = oracle.hedge_feedback(g2, L, objective=obj)
        assert np.array_equal(a, a2) and np.array_equal(w, w2)


def test_hedge_feedback_accept_length_window_and_delay():
    """Objective 1: item n's loss is K + 1 minus the accept-length estimate over items n .. n + K - 1 (the
    estimate pinned by enumeration and simulated chains above); it is applied in the push that delivers item
    n + K - 1, so at most K - 1 items wait after a push and none waits for more than K - 1 later items."""
    rng = np.random.default_rng(122)
    T, N, B, K = 20, 4, 3, 4
    gamma, L = _hf_rounds(rng, T, N, B, K)
    w, applied = oracle.hedge_feedback(gamma, L, objective=1)
    for b in range(B):
        items = _revealed(gamma, L, b)
        G = np.array([it[1] for it in items])               # [n_items, N]
        R, p = np.zeros(N), np.full(N, 1.0 / N)
        n = 0
        for t in range(T):
            arrived = sum(1 for it in items if it[0] <= t)
            assert applied[t, b] == max(0, arrived - K + 1)
            assert arrived - applied[t, b] <= K - 1
            while n + K - 1 < arrived:
                win = G[n:n + K].T[None]                      # [1, N, K]
                est, loss = oracle.accept_length(win)
                R, p, _ = oracle.normalhedge(R, loss[0], p)
                n += 1
            assert np.allclose(w[t, b], p, atol=1e-12)


def test_hedge_feedback_learns_the_best_drafter():
    """A drafter whose gamma is larger at every level ends with most of the weight, under both losses and
    with heavy censoring."""
    rng = np.random.default_rng(123)
    T, N, B, K = 150, 6, 2, 5
    gamma = rng.uniform(0.2, 0.8, (T, N, B, K))
    gamma[:, 2] = np.minimum(gamma[:, 2] + 0.15, 1.0)
    L = rng.integers(0, 3, (T, B)).astype(np.int32)
    for obj in (0, 1):
        w, _ = oracle.hedge_feedback(gamma, L, objective=obj)
        assert np.all(np.argmax(w[-1], axis=1) == 2)
        assert np.all(w[-1][:, 2] > 0.5)


def test_hedge_feedback_rejects_bad_lengths():
    g = np.full((2, 3, 1, 4), 0.5)
    with pytest.raises(ValueError):
        oracle.hedge_feedback(g, np.array([[0], [5]], np.int32))
    with pytest.raises(ValueError):
        oracle.hedge_feedback(g, np.array([[0], [-1]], np.int32))


# ----------------------------------------------------------------------------------------------
# standardised sampling: top-k / top-p folded into both rows
# ----------------------------------------------------------------------------------------------
def test_filter_row_top_k_and_top_p_sets():
    """The kept set, checked by its defining properties: it is an upper set of values; top-k keeps at least
    k and fewer than k strictly above its threshold; top-p's kept mass (renormalised over the top-k set)
    reaches top_p, and dropping its smallest value would fall below top_p."""
    rng = np.random.default_rng(110)
    for _ in range(300):
        V = int(rng.integers(2, 80))
        x = np.round(rng.normal(0, 2, V) * rng.choice([1, 4]), 0) / 2    # coarse: ties are common
        T = float(rng.choice([0.5, 1.0, 2.0]))
        k = int(rng.choice([0, 1, 3, V // 2, V - 1, V]))
        tp = float(rng.choice([1.0, 0.9, 0.5, 0.1, 1e-9]))
        y, thr, _ = oracle.filter_row(x, T, k, tp)
        kept = np.isfinite(y)
        assert np.array_equal(y[kept], x[kept])
        assert kept.any()
        if kept.sum() < V:
            assert x[kept].min() > x[~kept].max()                      # an upper set
        xk = x.copy()
        if 0 < k < V:
            tk = np.sort(x)[::-1][k - 1]
            assert (x >= tk).sum() >= k and (x > tk).sum() < k
            xk = np.where(x >= tk, x, -np.inf)
        if 0 < tp < 1:
            p = special.softmax(xk / T)
            vals = np.unique(x[kept])
            assert p[kept].sum() >= tp - 1e-12
            if len(vals) > 1:
                assert p[kept & (x > vals[0])].sum() < tp + 1e-12   # minimal: the smallest kept value is needed
        if k in (0, V) and tp == 1.0:
            assert kept.all() and thr == -np.inf


def test_verify_filtered_reductions_and_law():
    """No filter is the plain chain; top_k = 1 is greedy (both rows one-hot); the chain on standardised rows
    is lossless for the standardised target (exact law by enumeration)."""
    rng = np.random.default_rng(111)
    B, K, V = 12, 4, 50
    tgt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    drf = (tgt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    tok = np.stack([[rng.choice(V, p=special.softmax(drf[b, j])) for j in range(K)] for b in range(B)]).astype(np.int32)
    seeds = np.arange(B, dtype=np.uint64) + 3
    a = oracle.verify(tgt, drf, tok, seeds, 0.8)
    f = oracle.verify_filtered(tgt, drf, tok, seeds, 0.8, 0, 1.0)
    for key in ("accept_len", "out_tokens", "diag"):
        assert np.array_equal(a[key], f[key]), key
    g = oracle.greedy(tgt, drf.argmax(axis=2).astype(np.int32))
    f1 = oracle.verify_filtered(tgt, drf, drf.argmax(axis=2).astype(np.int32), seeds, 0.8, 1, 1.0)
    assert np.array_equal(g["accept_len"], f1["accept_len"]) and np.array_equal(g["out_tokens"], f1["out_tokens"])
    # the law of one step on standardised rows is the standardised target
    x_t = rng.normal(0, 1.5, 6)
    x_d = x_t + rng.normal(0, 1, 6)
    pt = special.softmax(oracle.filter_row(x_t, 1.0, 4, 0.8)[0])
    pd = special.softmax(oracle.filter_row(x_d, 1.0, 4, 0.8)[0])
    law = output_law(pt, pd)
    assert law == pytest.approx(pt, abs=2e-6)

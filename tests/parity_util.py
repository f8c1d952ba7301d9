"""Helpers shared by the GPU parity tests: run the oracle on the same inputs and compare.

Bar: accept lengths and emitted tokens bit-exact except where the oracle's accept margin |r - h(t)/p_draft(t)|
or its CDF margin (distance of u * Z to the nearer boundary of the chosen token, in probability mass) is
below 1e-5; such near ties are counted and must stay under 0.01% of positions. Probabilities, Z, gamma and
gamma* agree within 1e-5 absolute.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

PROB_TOL = 1e-5
TIE_TOL = 1e-5
TIE_FRACTION = 1e-4


def host(x):
    return workloads.to_numpy_logits(x)


def _filter_near_tie(ref, b, j, K):
    """Standardised sampling: True when a top-p threshold of sequence b's rows at positions 0..j (target and
    draft rows; the bonus row at j = K) was a near tie in the oracle (its pmargin below the tie tolerance).
    Such a threshold can land one value off, which moves p(t), Z and the CDF of that position."""
    pm = ref.get("pmargin")
    if pm is None:
        return False
    B = len(ref["accept_len"])
    rows_t = [b * (K + 1) + i for i in range(min(j, K) + 1)]
    rows_d = [B * (K + 1) + b * K + i for i in range(min(j, K - 1) + 1)]
    return bool(np.any(pm[rows_t + rows_d] < TIE_TOL))


def chain_report(got_len, got_tok, ref, K):
    """Returns (exact, near_tie_mismatches, bad) sequence counts. A mismatch is a near tie when the oracle's
    accept margin at the first disagreeing position, or its CDF margin for a disagreeing draw, is below the
    tie tolerance; with standardised sampling also when a top-p threshold decision of the sequence up to that
    position was a near tie (the oracle's pmargin)."""
    ref_len, ref_tok = ref["accept_len"], ref["out_tokens"]
    am, cm = ref["accept_margin"], ref["cdf_margin"]
    exact = near = 0
    bad = []
    for b in range(len(got_len)):
        if got_len[b] == ref_len[b] and np.array_equal(got_tok[b], ref_tok[b]):
            exact += 1
            continue
        if got_len[b] != ref_len[b]:
            j = int(min(got_len[b], ref_len[b]))
            ok = j < K and am[b, j] < TIE_TOL
        else:
            j = int(ref_len[b])
            ok = cm[b] < TIE_TOL
        if not ok:
            ok = _filter_near_tie(ref, b, j, K)
        if ok:
            near += 1
        else:
            bad.append(b)
    return exact, near, bad


def assert_chain(out, ref, K, positions=None, rate=True):
    """Tokens and accept lengths against the oracle. rate=False only counts the near-tie mismatches (for one
    batch of a pooled measurement, whose rate is asserted over the pool)."""
    got_len = out["accept_len"].cpu().numpy()
    got_tok = out["out_tokens"].cpu().numpy()
    exact, near, bad = chain_report(got_len, got_tok, ref, K)
    positions = positions or len(got_len) * K
    assert not bad, "mismatch away from a near tie at sequences %s: got %s / %s, oracle %s / %s" % (
        bad[:5], got_len[bad[:5]], got_tok[bad[:5]], ref["accept_len"][bad[:5]], ref["out_tokens"][bad[:5]])
    if rate:
        assert near <= TIE_FRACTION * positions, "%d near-tie mismatches in %d positions" % (near, positions)
    # structural checks that hold whatever the ties
    L = got_len
    assert np.all((L >= 0) & (L <= K))
    for b in range(len(L)):
        assert got_tok[b, L[b]] >= 0
        assert np.all(got_tok[b, L[b] + 1:] == -1)
    return exact, near


def assert_diag(out, ref, check_r=True):
    d = out["diag"].cpu().numpy().astype(np.float64)
    r = ref["diag"]
    assert np.abs(d[..., :3] - r[..., :3]).max() <= PROB_TOL, np.abs(d[..., :3] - r[..., :3]).max()
    if check_r:
        assert np.array_equal(d[..., 3], r[..., 3])   # uniforms are exact in fp32


def oracle_verify(inp, seq_index=None, sel=None):
    s = slice(None) if sel is None else sel
    return oracle.verify(host(inp["target"][s]), host(inp["draft"][s]), inp["tokens"][s].cpu().numpy(),
                         inp["seeds"][s].cpu().numpy().astype(np.uint64), inp["temperature"],
                         seq_index=seq_index)


def to_device(inp, device="cuda"):
    out = {}
    for k, v in inp.items():
        out[k] = v.to(device) if torch.is_tensor(v) else v
    if "drafters" in out:
        out["draft"] = out["drafters"][out["selected"]]
    return out

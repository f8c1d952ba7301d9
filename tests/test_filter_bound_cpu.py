"""CPU check of the argument behind the top-k bound kernel: the k-th largest of a row's 128-byte line maxima
bounds the row's k-th largest logit from below, also as the kernel stores it. A model of the kernel's key
arithmetic (order-preserving integer keys, 16-bit line keys that are the upper half of the key for fp32, a
zero maximum taken as -0, a bound of value zero lowered to the key of -0) is run on random and adversarial
rows, and brute force checks that the logits at or above the bound include every logit top-k keeps (by value,
so -0 and +0 tie) and number at least k, and that every line holding one of them reaches the bound."""
import numpy as np
import pytest


def keys(bits, nbits):
    sign = np.uint64(1) << np.uint64(nbits - 1)
    full = (np.uint64(1) << np.uint64(nbits)) - np.uint64(1)
    b = bits.astype(np.uint64)
    return np.where(b & sign, (~b) & full, b | sign)


def value_of(key, nbits, dtype):
    sign = np.uint64(1) << np.uint64(nbits - 1)
    full = (np.uint64(1) << np.uint64(nbits)) - np.uint64(1)
    k = np.uint64(key)
    b = (k & (sign - np.uint64(1))) if (k & sign) else ((~k) & full)
    if nbits == 16:
        return np.array([int(b) << 16], dtype=np.uint32).view(np.float32)[0]
    return np.array([int(b)], dtype=np.uint32).view(np.float32)[0]


def key_at_most(v, nbits):
    v = np.float32(-0.0) if v == 0 else np.float32(v)
    bits = np.array([v], dtype=np.float32).view(np.uint32)[0]
    if nbits == 16:
        bits = bits >> 16
    return int(keys(np.array([bits]), nbits)[0])


def bound_candidates(x, k, nbits):
    """The kernel's bound and the candidates at or above it, for a row x (float32 values, bf16-exact when
    nbits = 16)."""
    bits = x.view(np.uint32)
    if nbits == 16:
        bits = bits >> 16
    kk = keys(bits, nbits)
    per_line = 128 // (nbits // 8)
    n_lines = -(-len(x) // per_line)
    line_key = []
    for l in range(n_lines):
        m = np.max(x[l * per_line:(l + 1) * per_line])
        key = key_at_most(m, nbits)
        line_key.append(key if nbits == 16 else key >> 16)
    line_key = np.array(line_key, dtype=np.uint64)
    bound16 = int(np.sort(line_key)[::-1][k - 1]) if n_lines >= k else 0
    raw = bound16 if nbits == 16 else bound16 << 16
    v = value_of(raw, nbits, np.float32)
    bound = 0 if (raw == 0) else key_at_most(v, nbits)
    bound_line = bound if nbits == 16 else bound >> 16
    cand = kk >= np.uint64(bound)
    lines_in = line_key >= np.uint64(bound_line)
    return cand, lines_in, per_line


def rows(rng, nbits):
    V = 5000
    out = [rng.normal(0, 2, V), rng.normal(0, 2, V) * (rng.random(V) < 0.01)]
    z = rng.choice(np.array([-1.0, -0.0, 0.0, 0.5]), V)
    z[::97] = 2.0
    out.append(z)
    out.append(np.full(V, 1.5))
    out.append(rng.normal(0, 1e-40, V))                      # denormals and zeros around the bound
    out.append(np.round(rng.normal(0, 1, V), 1))              # many ties
    out.append(rng.normal(0, 2, 300))                         # fewer lines than k
    res = []
    for r in out:
        r = np.asarray(r, dtype=np.float32)
        if nbits == 16:                                       # round to bf16 values (truncate the low half)
            r = (r.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
        res.append(r)
    return res


@pytest.mark.parametrize("nbits", [16, 32])
@pytest.mark.parametrize("k", [1, 7, 64, 256, 1024])
def test_line_maxima_bound_keeps_every_top_k_logit(nbits, k):
    rng = np.random.default_rng(k * 31 + nbits)
    for x in rows(rng, nbits):
        if k >= len(x):
            continue
        cand, lines_in, per_line = bound_candidates(x, k, nbits)
        kth = np.sort(x)[::-1][k - 1]                         # the k-th largest value
        kept = x >= kth                                        # top-k keeps ties, -0 == +0
        assert cand.sum() >= k
        assert np.all(cand[kept]), "a kept logit lies below the bound"
        line_of = np.arange(len(x)) // per_line
        assert np.all(lines_in[line_of[cand]]), "a candidate's line was not listed"

"""Pins of the oracle's mid attention and DupUp shortcut (CPU only).

Attention: a single token attends to itself (o = v); identical keys give a
uniform softmax (o = mean of v); a per-query constant added to every score
(a key bias) changes nothing; a brute-force per-row loop on a tiny case; and
the row-sampled form agrees with the whole-matrix form on every sampled row.
DupUp: a brute-force loop over the printed index formula, and the mass
invariant (each source channel feeds ``repeats`` outputs per source pixel).
"""
import math

import numpy as np
import pytest

import oracle
from vae_inputs import Attn, Conv, Norm


def _attn(rng, c, family):
    def lin():
        return Conv(w=rng.standard_normal((c, c, 1, 1)) / math.sqrt(c), b=rng.standard_normal(c) * 0.1)
    norm = Norm(gamma=rng.uniform(0.5, 1.5, c), beta=rng.standard_normal(c) * 0.1 if family == "gn" else None)
    return Attn(norm=norm, q=lin(), k=lin(), v=lin(), o=lin())


def _lin(t, cv):
    return t @ cv.w[:, :, 0, 0].T + cv.b


@pytest.mark.parametrize("family", ["gn", "rms"])
def test_single_token_output_is_v(family):
    rng = np.random.default_rng(21)
    c = 4
    a = _attn(rng, c, family)
    x = rng.standard_normal((c, 1, 1))
    y = oracle.attention(x, a, family, groups=2)
    n = oracle.group_norm(x, 2, a.norm.gamma, a.norm.beta, 1e-6) if family == "gn" else oracle.rms_norm(x, a.norm.gamma)
    v = _lin(n[:, 0, 0][None], a.v)
    ref = x[:, 0, 0] + _lin(v, a.o)[0]
    np.testing.assert_allclose(y[:, 0, 0], ref, rtol=1e-12)


def test_identical_keys_give_uniform_weights():
    rng = np.random.default_rng(22)
    c, h, w = 4, 2, 3
    a = _attn(rng, c, "rms")
    a.k = Conv(w=np.zeros((c, c, 1, 1)), b=rng.standard_normal(c))  # every key is the bias
    x = rng.standard_normal((c, h, w))
    y = oracle.attention(x, a, "rms")
    n = oracle.rms_norm(x, a.norm.gamma).reshape(c, -1).T
    v = _lin(n, a.v)
    o = np.broadcast_to(v.mean(axis=0), v.shape)
    ref = x + _lin(o, a.o).T.reshape(c, h, w)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_score_shift_invariance():
    rng = np.random.default_rng(23)
    c, h, w = 8, 3, 3
    a = _attn(rng, c, "gn")
    x = rng.standard_normal((c, h, w))
    y1 = oracle.attention(x, a, "gn", groups=4)
    a.k = Conv(w=a.k.w, b=a.k.b + rng.standard_normal(c) * 3.0)  # adds q_i.delta to row i
    y2 = oracle.attention(x, a, "gn", groups=4)
    np.testing.assert_allclose(y1, y2, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("family", ["gn", "rms"])
def test_attention_rows_matches_whole_attention(family):
    rng = np.random.default_rng(25)
    c, h, w = 8, 5, 7
    a = _attn(rng, c, family)
    x = rng.standard_normal((c, h, w)) * 2.0
    whole = oracle.attention(x, a, family, groups=4, chunk=4).reshape(c, -1).T
    rows = [0, 3, 17, 34, 20]
    got = oracle.attention_rows(x, a, family, rows, groups=4)
    np.testing.assert_allclose(got, whole[rows], rtol=1e-12, atol=1e-12)


def test_attention_brute_force_rows():
    rng = np.random.default_rng(24)
    c, h, w = 4, 2, 2
    a = _attn(rng, c, "rms")
    x = rng.standard_normal((c, h, w))
    y = oracle.attention(x, a, "rms", chunk=3)
    n = oracle.rms_norm(x, a.norm.gamma).reshape(c, -1).T
    q, k, v = _lin(n, a.q), _lin(n, a.k), _lin(n, a.v)
    m = h * w
    o = np.zeros((m, c))
    for i in range(m):
        s = [sum(q[i, d] * k[j, d] for d in range(c)) / math.sqrt(c) for j in range(m)]
        mx = max(s)
        e = [math.exp(t - mx) for t in s]
        tot = sum(e)
        for j in range(m):
            o[i] += e[j] / tot * v[j]
    ref = x + _lin(o, a.o).T.reshape(c, h, w)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    # rows of the softmax sum to one: o of a constant v is that constant
    a.v = Conv(w=np.zeros((c, c, 1, 1)), b=np.arange(c, dtype=float))
    y3 = oracle.attention(x, a, "rms")
    ref3 = x + _lin(np.tile(np.arange(c, dtype=float), (m, 1)), a.o).T.reshape(c, h, w)
    np.testing.assert_allclose(y3, ref3, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("cin,cout,ft", [(8, 4, 1), (4, 4, 1), (6, 3, 1), (8, 4, 2), (2, 4, 1)])
def test_dupup_brute_force(cin, cout, ft):
    rng = np.random.default_rng(25)
    h, w = 3, 2
    src = rng.standard_normal((cin, h, w))
    d = oracle.dupup(src, cout, ft)
    factor = 4 * ft
    repeats = cout * factor // cin
    for o in range(cout):
        for Y in range(2 * h):
            for X in range(2 * w):
                j = o * factor + (ft - 1) * 4 + 2 * (Y % 2) + (X % 2)
                assert d[o, Y, X] == src[j // repeats, Y // 2, X // 2]


def test_dupup_mass_invariant():
    """ft = 1: every source channel is read exactly ``repeats`` times per source pixel."""
    cin, cout = 8, 4
    repeats = cout * 4 // cin
    src = np.zeros((cin, 1, 1))
    counts = np.zeros(cin)
    for ch in range(cin):
        src[:] = 0
        src[ch] = 1.0
        counts[ch] = oracle.dupup(src, cout, 1).sum()
    assert np.array_equal(counts, np.full(cin, repeats))

"""The folded form the GPU evaluates the mid attention in, checked in float64
against the oracle's literal definition (q, k, v projections, row softmax,
output projection): the key bias shifts every score of a row by the same
amount, which the softmax removes, and the rows of the softmax sum to one, so

    s_ij = (n_i M^T + Wk^T bq) . n_j / sqrt(c),   M = Wk^T Wq
    y_i  = x_i + (sum_j p_ij n_j) (Wo Wv)^T + (Wo bv + bo)

equals the literal attention up to float64 rounding. A dropped query bias, a
transposed fold or the value bias counted twice fails here."""
import numpy as np
import pytest

import oracle
from vae_inputs import Attn, Conv, Norm, bias_vec, conv_weight, rng_for, stream_normal


def _attn(seed, c, family):
    def lin(nm):
        return Conv(w=conv_weight(seed, f"fold.{nm}.{c}", c, c, 1), b=bias_vec(seed, f"fold.{nm}.b.{c}", c))
    g = rng_for(seed, f"fold.n.{c}")
    norm = Norm(gamma=g.uniform(0.5, 1.5, c).astype(np.float32),
                beta=(g.standard_normal(c) * 0.1).astype(np.float32) if family == "gn" else None)
    return Attn(norm=norm, q=lin("q"), k=lin("k"), v=lin("v"), o=lin("o"))


def folded_attention(x, a, family, groups=32):
    c, h, w = x.shape
    m = h * w
    x = x.astype(np.float64)
    n = oracle.group_norm(x, groups, a.norm.gamma, a.norm.beta) if family == "gn" else oracle.rms_norm(x, a.norm.gamma)
    t = n.reshape(c, m).T
    W = {nm: getattr(a, nm).w[:, :, 0, 0].astype(np.float64) for nm in "qkvo"}
    b = {nm: getattr(a, nm).b.astype(np.float64) for nm in "qkvo"}
    qf = t @ (W["k"].T @ W["q"]).T + W["k"].T @ b["q"]
    s = qf @ t.T / np.sqrt(c)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    y = (p @ t) @ (W["o"] @ W["v"]).T + (W["o"] @ b["v"] + b["o"])
    return x + y.T.reshape(c, h, w)


@pytest.mark.parametrize("m,c,family", [(40, 32, "rms"), (64, 64, "gn"), (129, 48, "rms")])
def test_folded_form_equals_literal_attention(m, c, family):
    x = stream_normal(30, f"fold.x.{m}.{c}", (c, m, 1)) * 2.0
    a = _attn(30, c, family)
    ref = oracle.attention(x, a, family)
    got = folded_attention(x, a, family)
    assert np.max(np.abs(got - ref)) <= 1e-11 * np.max(np.abs(ref - x))


def test_fold_needs_the_query_bias_term():
    """Without Wk^T bq the scores change by a per-key amount, which the softmax
    does not remove: the folded form then differs visibly."""
    m, c = 64, 32
    x = stream_normal(31, "fold.x.bq", (c, m, 1))
    a = _attn(31, c, "rms")
    a.q = Conv(w=a.q.w, b=(a.q.b * 50).astype(np.float32))
    ref = oracle.attention(x, a, "rms")
    a0 = Attn(norm=a.norm, q=Conv(w=a.q.w, b=np.zeros_like(a.q.b)), k=a.k, v=a.v, o=a.o)
    got0 = folded_attention(x, a0, "rms")
    assert np.max(np.abs(got0 - ref)) > 1e-3 * np.max(np.abs(ref - x))
    assert np.max(np.abs(folded_attention(x, a, "rms") - ref)) <= 1e-11 * np.max(np.abs(ref - x))

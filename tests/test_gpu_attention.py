"""GPU parity of the mid attention (norm, projections, the scores-softmax
kernel and the P.V kernel, output projection) against the oracle, on the
attention's contribution y - x. Tolerance 5e-3 of max|ref|: the GPU rounds to
f16 (relative 2^-11 each) the normalised rows, the folded weights Wk^T Wq and
Wo Wv, the folded queries, the unnormalised P and the softmax average (or,
with VAE_ATTN_FOLD=0, q, k, v and o), and accumulates in f32; those roundings
stay near 1e-3 of the output scale."""
import numpy as np
import pytest

import oracle
import implicit_gemm_convolution_vae_gb300 as vg
from gpu_common import rel_err, to_dev, torch_mod
from vae_inputs import Attn, Conv, Norm, bias_vec, conv_weight, rng_for, stream_normal

pytestmark = pytest.mark.gpu

ATTN_TOL = 5e-3


def _attn(seed, c, family):
    def lin(nm):
        return Conv(w=conv_weight(seed, f"at.{nm}.{c}", c, c, 1), b=bias_vec(seed, f"at.{nm}.b.{c}", c))
    g = rng_for(seed, f"at.n.{c}")
    norm = Norm(gamma=g.uniform(0.5, 1.5, c).astype(np.float32),
                beta=(g.standard_normal(c) * 0.1).astype(np.float32) if family == "gn" else None)
    return Attn(norm=norm, q=lin("q"), k=lin("k"), v=lin("v"), o=lin("o"))


def run_gpu(x, a, family, groups=32):
    torch = torch_mod()
    xd = to_dev(x.copy())
    w = lambda cv: to_dev(vg.pack_conv1x1(cv.w))
    vg.mid_attention(xd, vg.NORM_GROUP if family == "gn" else vg.NORM_RMS, to_dev(a.norm.gamma),
                     to_dev(a.norm.beta) if a.norm.beta is not None else None,
                     w(a.q), to_dev(a.q.b), w(a.k), to_dev(a.k.b), w(a.v), to_dev(a.v.b), w(a.o), to_dev(a.o.b),
                     groups=groups)
    vg.sync_status()
    return xd.cpu().numpy()


@pytest.mark.parametrize("m,c,family", [(1, 64, "rms"), (5, 32, "gn"), (33, 48, "rms"), (7, 128, "gn"), (200, 192, "rms"), (1024, 512, "gn"),
                                        (1000, 640, "rms"), (2500, 1152, "rms"), (300, 2048, "rms")])
def test_mid_attention(m, c, family):
    x = stream_normal(20, f"attn.x.{m}.{c}", (m, c))
    a = _attn(20, c, family)
    got = run_gpu(x, a, family)
    ref = oracle.attention(x.T.reshape(c, m, 1), a, family, groups=32).reshape(c, m).T
    assert np.isfinite(got).all()
    assert rel_err(got - x, ref - x) <= ATTN_TOL


def test_mid_attention_full_size_qwen_mid():
    """m = 128 x 128 latent tokens, c = 1152: the 1024^2 decoder's mid block."""
    m, c = 16384, 1152
    x = stream_normal(21, "attn.full.x", (m, c)) * 2.0
    a = _attn(21, c, "rms")
    got = run_gpu(x, a, "rms")
    ref = oracle.attention(x.T.reshape(c, 128, 128), a, "rms").reshape(c, m).T
    assert rel_err(got - x, ref - x) <= ATTN_TOL


@pytest.mark.parametrize("m,c", [(1024, 128), (1024, 512), (1024, 1152), (1100, 1152)])
def test_peaked_softmax_rescales(m, c):
    """Scores that grow block after block force the lazy O rescale path (with
    one, two and three value-channel chunks sharing the rescale flags; 1100
    tokens: nine query tiles, so the PV kernel's last CTA pair has one tile)."""
    x = stream_normal(22, f"attn.peak.x.{c}", (m, c))
    x = x + np.linspace(0, 40, m, dtype=np.float32)[:, None] * x[:, :1]
    a = _attn(22, c, "rms")
    a.q = Conv(w=(a.q.w.astype(np.float32) * 4).astype(np.float16), b=a.q.b)
    got = run_gpu(x, a, "rms")
    ref = oracle.attention(x.T.reshape(c, m, 1), a, "rms").reshape(c, m).T
    # Logits here reach the hundreds, so the f16 roundings of the query side
    # (q and k, or the folded weights and queries) move them by up to about
    # |s| * 2^-10 and the sharply peaked softmax passes that on: 1e-2.
    assert rel_err(got - x, ref - x) <= 1e-2


def test_mid_attention_two_query_groups():
    """m = 33000 tokens (258 query tiles, the last one 104 rows): the
    probabilities of all query tiles exceed the 2 GiB workspace cap, so the
    tiles run as two groups (254 + 4); outputs sampled per row (first and last
    rows of both groups and of the ragged last tile)."""
    m, c = 33000, 64
    x = stream_normal(23, "attn.groups.x", (m, c))
    a = _attn(23, c, "rms")
    got = run_gpu(x, a, "rms")
    rows = [0, 1, 127, 128, 254 * 128 - 1, 254 * 128, 254 * 128 + 5, 257 * 128, m - 1]
    ref = oracle.attention_rows(x.T.reshape(c, m, 1), a, "rms", rows)
    assert np.isfinite(got).all()
    assert rel_err(got[rows] - x[rows], ref - x[rows]) <= ATTN_TOL


def test_single_cta_attention_kernels_match_oracle():
    """The scores and PV steps on single CTAs (VAE_ATTN_SCORES_PAIR=0,
    VAE_ATTN_PV_PAIR=0; by default query-tile pairs share them through
    cta_group::2): the attention tests again in a child process, which reads
    the switches once."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, VAE_ATTN_PV_PAIR="0", VAE_ATTN_SCORES_PAIR="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(root, "tests", "test_gpu_attention.py"), "-k",
                        "not full_size and not two_query_groups and not single_cta and not literal"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_literal_projections_match_oracle():
    """The q, k, v projections as written (VAE_ATTN_FOLD=0) instead of the
    folded weights: the attention tests again in a child process."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, VAE_ATTN_FOLD="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(root, "tests", "test_gpu_attention.py"), "-k",
                        "not two_query_groups and not single_cta and not literal"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]

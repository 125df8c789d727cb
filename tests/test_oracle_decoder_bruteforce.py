"""Whole-decoder pins of the oracle: an element-by-element restatement (CPU only).

The oracle's ``decode_gn`` / ``decode_rms`` compose vectorised primitives.
Here both decoders are written a second time, from the pages' definitions,
as plain scalar loops over a pixel-major layout (a dict of pixel -> channel
list; no numpy arithmetic, sums in ``math.fsum``), on tiny random decoders
(non-square latents, affine norms, a channel-changing ResNet, a DupUp with
repeats 2). The two must agree to rounding (1e-9 relative).

Planted mistakes in the restatement (the DupUp shortcut dropped or taken from
the block's output, the up conv reading a normalised stream, SiLU missing
after the output norm, the latent scale/shift skipped, the attention
residual dropped, a ResNet skip dropped, the shortcut conv skipped) each move
the result far outside that tolerance, so the comparison sees every step of
the composition.

Sources:
- ``vae.rs`` (FLUX-class ``AutoencoderKL`` decoder): ``VaeDecoder::decode``,
  ``ResnetBlock::apply``, ``AttnBlock::apply``, ``GroupNorm::apply``,
  ``Conv2d::apply``, ``fn upsample2x``, ``fn silu``.
- ``qi21_vae.rs`` (Qwen-Image-2.1 / Wan-style decoder): ``decode``,
  ``run_blocks`` (ResNets, up conv on the 2x grid, the DupUp shortcut of the
  block input: output channel o at sub-pixel (sy, sx) takes source channel
  (4·ft·o + 4·(ft − 1) + 2·sy + sx) / repeats, ``DUPUP_SRC``), ``qv_rmsn``
  (v·√C / max(‖v‖, 1e-12)·γ), ``fn attention``, ``output_rows``.
"""
import dataclasses
import math

import numpy as np
import pytest

import oracle
from vae_inputs import flux_decoder, qwen_decoder, latent_normal


# ───────────────────── the restatement (pixel-major scalar loops) ─────────────────────
# A feature map is (h, w, px) with px[(y, x)] = list of channel values (floats).

def _to_px(chw):
    c, h, w = chw.shape
    return h, w, {(y, x): [float(chw[k, y, x]) for k in range(c)] for y in range(h) for x in range(w)}


def _to_chw(fm):
    h, w, px = fm
    c = len(px[(0, 0)])
    out = np.zeros((c, h, w))
    for (y, x), v in px.items():
        for k in range(c):
            out[k, y, x] = v[k]
    return out


def _conv(fm, conv, up=False):
    """Conv2d, stride 1, zero padding k//2; with ``up`` the input is first
    nearest-upsampled (pixel (Y, X) of the 2x grid is source pixel (Y//2, X//2))."""
    h, w, px = fm
    W = np.asarray(conv.w, np.float64)
    B = np.asarray(conv.b, np.float64)
    cout, cin, k, _ = W.shape
    H2, W2 = (2 * h, 2 * w) if up else (h, w)
    r = k // 2
    out = {}
    for Y in range(H2):
        for X in range(W2):
            vals = []
            for o in range(cout):
                terms = [float(B[o])]
                for ky in range(k):
                    for kx in range(k):
                        sy, sx = Y + ky - r, X + kx - r
                        if not (0 <= sy < H2 and 0 <= sx < W2):
                            continue  # zero padding
                        src = px[(sy // 2, sx // 2)] if up else px[(sy, sx)]
                        for c in range(cin):
                            terms.append(float(W[o, c, ky, kx]) * src[c])
                vals.append(math.fsum(terms))
            out[(Y, X)] = vals
    return H2, W2, out


def _silu(fm):
    h, w, px = fm
    return h, w, {p: [v / (1.0 + math.exp(-v)) for v in vs] for p, vs in px.items()}


def _group_norm(fm, norm, groups, eps):
    """Per group of C/G consecutive channels: mean and biased variance over the
    group's channels and all pixels; (v - mean)/sqrt(var + eps)*gamma + beta."""
    h, w, px = fm
    c = len(px[(0, 0)])
    per = c // groups
    stats = []
    for g in range(groups):
        vals = [vs[k] for vs in px.values() for k in range(g * per, (g + 1) * per)]
        mean = math.fsum(vals) / len(vals)
        var = math.fsum((v - mean) ** 2 for v in vals) / len(vals)
        stats.append((mean, math.sqrt(var + eps)))
    out = {}
    for p, vs in px.items():
        out[p] = [(vs[k] - stats[k // per][0]) / stats[k // per][1] * float(norm.gamma[k]) + float(norm.beta[k])
                  for k in range(c)]
    return h, w, out


def _rms_norm(fm, norm):
    """Per pixel: v * sqrt(C) / max(||v||_2, 1e-12) * gamma."""
    h, w, px = fm
    out = {}
    for p, vs in px.items():
        c = len(vs)
        nrm = math.sqrt(math.fsum(v * v for v in vs))
        s = math.sqrt(c) / max(nrm, 1e-12)
        out[p] = [vs[k] * s * float(norm.gamma[k]) for k in range(c)]
    return h, w, out


def _add(a, b):
    h, w, pa = a
    _, _, pb = b
    return h, w, {p: [x + y for x, y in zip(pa[p], pb[p])] for p in pa}


def _norm(fm, nm, family, groups, eps):
    return _group_norm(fm, nm, groups, eps) if family == "gn" else _rms_norm(fm, nm)


def _resnet(fm, r, family, groups, eps, mistakes):
    hdn = _conv(_silu(_norm(fm, r.norm1, family, groups, eps)), r.conv1)
    hdn = _conv(_silu(_norm(hdn, r.norm2, family, groups, eps)), r.conv2)
    if "no_resnet_skip" in mistakes:
        return hdn
    skip = fm
    if r.shortcut is not None and "no_shortcut_conv" not in mistakes:
        skip = _conv(fm, r.shortcut)
    elif r.shortcut is not None:  # the planted mistake: the wider input's first channels
        h, w, px = fm
        skip = (h, w, {p: vs[:r.conv2.cout] for p, vs in px.items()})
    return _add(skip, hdn)


def _attention(fm, a, family, groups, eps, mistakes):
    """Single head over all m pixels: n = norm(x) (no SiLU); q, k, v = 1x1 of n;
    o_i = sum_j softmax_j(q_i . k_j / sqrt(C)) v_j; x + 1x1_o(o)."""
    h, w, px = fm
    n = _norm(fm, a.norm, family, groups, eps)
    q = _conv(n, a.q)[2]
    k = _conv(n, a.k)[2]
    v = _conv(n, a.v)[2]
    pix = sorted(px)
    c = len(px[pix[0]])
    o = {}
    for i in pix:
        s = [math.fsum(q[i][t] * k[j][t] for t in range(c)) / math.sqrt(c) for j in pix]
        mx = max(s)
        e = [math.exp(t - mx) for t in s]
        z = math.fsum(e)
        o[i] = [math.fsum(e[jj] / z * v[j][t] for jj, j in enumerate(pix)) for t in range(c)]
    proj = _conv((h, w, o), a.o)
    if "no_attention_residual" in mistakes:
        return proj
    return _add(fm, proj)


def _dupup(cp, out_dim, ft):
    """The block input spread onto the 2x grid with a channel shuffle: output
    channel o at pixel (2y+sy, 2x+sx) takes source channel
    (4*ft*o + 4*(ft-1) + 2*sy + sx) // repeats of pixel (y, x),
    repeats = out_dim*4*ft / in_dim."""
    h, w, px = cp
    cin = len(px[(0, 0)])
    repeats = out_dim * 4 * ft // cin
    out = {}
    for Y in range(2 * h):
        for X in range(2 * w):
            src = px[(Y // 2, X // 2)]
            out[(Y, X)] = [src[(4 * ft * o + 4 * (ft - 1) + 2 * (Y % 2) + (X % 2)) // repeats]
                           for o in range(out_dim)]
    return 2 * h, 2 * w, out


def brute_decode(dec, z, mistakes=()):
    fam, groups, eps = dec.family, dec.groups, dec.eps
    zz = np.asarray(z, np.float64)
    if fam == "gn" and "no_latent_affine" not in mistakes:
        zz = zz / dec.scaling + dec.shift
    fm = _to_px(zz)
    if fam == "rms":
        fm = _conv(fm, dec.post_quant)
    fm = _conv(fm, dec.conv_in)
    fm = _resnet(fm, dec.mid_res1, fam, groups, eps, mistakes)
    fm = _attention(fm, dec.mid_attn, fam, groups, eps, mistakes)
    fm = _resnet(fm, dec.mid_res2, fam, groups, eps, mistakes)
    for u in dec.ups:
        block_in = fm
        for r in u.resnets:
            fm = _resnet(fm, r, fam, groups, eps, mistakes)
        if u.up is not None:
            src = _silu(_norm(fm, u.resnets[-1].norm1, fam, groups, eps)) if "normed_up_input" in mistakes else fm
            y = _conv(src, u.up, up=True)
            if dec.dupup and "no_dupup" not in mistakes:
                y = _add(y, _dupup(fm if "dupup_of_block_output" in mistakes else block_in, u.out_dim, u.ft))
            fm = y
    fm = _norm(fm, dec.norm_out, fam, groups, eps)
    if "no_output_silu" not in mistakes:
        fm = _silu(fm)
    return _to_chw(_conv(fm, dec.conv_out))


# ───────────────────────────── the decoders pinned ─────────────────────────────

def _rms_dec():
    # widths 8 -> 4: the up conv halves the channels; DupUp repeats = 4*4*1/8 = 2
    return qwen_decoder(seed=3, latent_channels=4, widths=(8, 4), nres=2, affine=True)


def _gn_dec():
    # widths 8 -> 4 (reversed block_out): the second block's first ResNet has a 1x1 shortcut
    d = flux_decoder(seed=4, latent_channels=4, block_out=(4, 8), layers_per_block=1, affine=True)
    return dataclasses.replace(d, groups=2, scaling=0.5, shift=0.25)


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


@pytest.mark.parametrize("family", ["rms", "gn"])
def test_decoder_equals_the_elementwise_restatement(family):
    dec = _rms_dec() if family == "rms" else _gn_dec()
    z = latent_normal(7, 4, 3, 2)  # 3 x 2 latent: rows and columns differ
    ref = oracle.decode(dec, z)
    got = brute_decode(dec, z)
    assert ref.shape == got.shape == (3, 6, 4)
    assert np.all(np.isfinite(ref))
    assert _rel(got, ref) < 1e-9


RMS_MISTAKES = ["no_dupup", "dupup_of_block_output", "normed_up_input", "no_output_silu",
                "no_attention_residual", "no_resnet_skip"]
GN_MISTAKES = ["no_latent_affine", "normed_up_input", "no_output_silu", "no_attention_residual",
               "no_resnet_skip", "no_shortcut_conv"]


@pytest.mark.parametrize("family,mistake", [("rms", m) for m in RMS_MISTAKES] + [("gn", m) for m in GN_MISTAKES])
def test_each_planted_mistake_is_seen(family, mistake):
    dec = _rms_dec() if family == "rms" else _gn_dec()
    z = latent_normal(7, 4, 3, 2)
    ref = oracle.decode(dec, z)
    assert _rel(brute_decode(dec, z, (mistake,)), ref) > 1e-4

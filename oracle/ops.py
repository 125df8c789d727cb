"""Oracle primitives (float64, NCHW) — test infrastructure only.

Each function restates one operation of the pages in plain numpy; the
docstring names the passage it follows. Inputs may be any numeric dtype
(f16 weights, f32 streams); everything is promoted to float64 first.
"""
from __future__ import annotations

import numpy as np

_F = np.float64


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=_F)


def silu(v):
    """SiLU, v / (1 + e^-v).

    ``vae.rs``, ``fn silu`` and ``qi21_vae.rs``, ``qv_rmsn`` (its flags-2 branch).
    """
    v = _f64(v)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def upsample2x(x):
    """Nearest-neighbour 2x: dst[c, Y, X] = src[c, Y//2, X//2].

    ``vae.rs``, ``fn upsample2x``. ``x``: [c][h][w] -> [c][2h][2w].
    """
    x = _f64(x)
    return np.repeat(np.repeat(x, 2, axis=1), 2, axis=2)


def conv2d(x, w, b=None, upsample: bool = False, pad: str = "zero"):
    """2-D convolution, stride 1, padding k//2 (cross-correlation, PyTorch order).

    y[o, Y, X] = b[o] + sum_{c, ky, kx} w[o, c, ky, kx] * xt[c, Y+ky-r, X+kx-r],
    r = k//2, where xt is ``x`` (or ``upsample2x(x)`` when ``upsample``) and
    reads outside the grid are 0 (``pad="zero"``), the nearest edge pixel
    (``pad="replicate"``, a clamp on the upsampled grid) or the pixel mirrored
    about the edge, the edge itself not repeated (``pad="reflect"``: index -1
    reads 1, index n reads n - 2; it needs at least two rows and columns).

    ``vae.rs``, ``Conv2d::apply`` (zero padding, pad = k/2, bias added per
    output channel) and ``VaeDecoder::decode`` (upsample, then conv);
    replicate padding from ``s2v_vae.rs``'s causal-replicate conv, read for 2-D;
    reflect padding from ``vae3d.rs``, ``EncConv::apply`` (the encoder's
    stride-1 convs: reflect on H and W by k/2).

    ``x``: [cin][h][w]; ``w``: [cout][cin][k][k]; returns [cout][H][W].
    Each tap is one channel contraction (a matmul) over a shifted view.
    """
    x = upsample2x(x) if upsample else _f64(x)
    w = _f64(w)
    cout, cin, k, k2 = w.shape
    assert k == k2 and x.shape[0] == cin, (w.shape, x.shape)
    _, H, W = x.shape
    r = k // 2
    mode = {"zero": "constant", "replicate": "edge", "reflect": "reflect"}[pad]
    if pad == "reflect":
        assert H >= 2 and W >= 2, "reflect padding needs two rows and columns"
    xp = np.pad(x, ((0, 0), (r, r), (r, r)), mode=mode)
    y = np.zeros((cout, H * W), _F)
    for ky in range(k):
        for kx in range(k):
            tap = xp[:, ky:ky + H, kx:kx + W].reshape(cin, H * W)
            y += w[:, :, ky, kx] @ tap
    if b is not None:
        y += _f64(b)[:, None]
    return y.reshape(cout, H, W)


def conv2d_down(x, w, b=None, pad: str = "reflect"):
    """The encoder's downsample conv: one row and one column padded onto the
    FAR side (bottom and right), then an unpadded stride-2 k x k convolution.

    y[o, Y, X] = b[o] + sum_{c, ky, kx} w[o, c, ky, kx] * xp[c, 2Y+ky, 2X+kx],
    xp = ``x`` with row h and column w appended: mirrored (``pad="reflect"``:
    they repeat rows / columns h - 2 and w - 2), copied from the edge
    (``"replicate"``) or zero (``"zero"``). The output is
    ((h + 1 - k) // 2 + 1) x ((w + 1 - k) // 2 + 1), i.e. h//2 x w//2 for k = 3.

    ``vae3d.rs``, ``reflect_pad_far`` (the far-side reflect pad) and the
    downsample ``EncConv`` (stride 2, pad 0) of ``VideoVaeEncoder``;
    ``s2v_vae.rs``, ``conv_down`` (the stride-2 conv of the encoder's frame).
    ``x``: [cin][h][w]; ``w``: [cout][cin][k][k].
    """
    x = _f64(x)
    w = _f64(w)
    cout, cin, k, k2 = w.shape
    assert k == k2 and x.shape[0] == cin, (w.shape, x.shape)
    _, h, wd = x.shape
    mode = {"zero": "constant", "replicate": "edge", "reflect": "reflect"}[pad]
    assert h >= 2 and wd >= 2, "the far-side pad needs two rows and columns"
    xp = np.pad(x, ((0, 0), (0, 1), (0, 1)), mode=mode)
    Ho, Wo = (h + 1 - k) // 2 + 1, (wd + 1 - k) // 2 + 1
    y = np.zeros((cout, Ho * Wo), _F)
    for ky in range(k):
        for kx in range(k):
            tap = xp[:, ky:ky + 2 * Ho - 1:2, kx:kx + 2 * Wo - 1:2].reshape(cin, Ho * Wo)
            y += w[:, :, ky, kx] @ tap
    if b is not None:
        y += _f64(b)[:, None]
    return y.reshape(cout, Ho, Wo)


def causal_source_frame(f: int, kt: int, t_upsample: bool) -> int:
    """Source frame that output frame ``f``'s temporal tap ``kt`` (0..2) reads.

    The tap sees upsampled frame vf = f + kt - 2, clamped to the first frame
    (causal padding replicates it); with the temporal 2x the upsampled frame vf
    comes from source frame (vf - 1) // 2 + 1 for vf > 0 and 0 for vf = 0, so
    the first frame is not doubled. ``s2v_vae.rs``, module doc (causal
    replicate padding, two frames back) and ``conv_any``'s ``src_f``.
    """
    vf = max(f + kt - 2, 0)
    return (vf - 1) // 2 + 1 if (t_upsample and vf > 0) else vf


def conv3d_causal(x, w, b=None, upsample: bool = False, t_upsample: bool = False, pad: str = "zero"):
    """3x3x3 causal convolution over frames, stride 1.

    y[o, f, Y, X] = b[o] + sum_{kt} conv2d(xt[:, s(f, kt)], w[:, :, kt])[o, Y, X]
    with s = ``causal_source_frame`` and conv2d the 2-D definition above (its
    spatial nearest 2x and zero / replicate padding). Output frames: F, or
    2F - 1 with ``t_upsample``. ``s2v_vae.rs``, the 3x3x3 causal implicit-GEMM
    conv (module doc; ``conv_any``).

    ``x``: [cin][F][h][w]; ``w``: [cout][cin][3][3][3] (kt, ky, kx); returns
    [cout][F'][H][W].
    """
    x = _f64(x)
    w = _f64(w)
    cout, cin, kd, kh, kw = w.shape
    assert (kd, kh, kw) == (3, 3, 3) and x.shape[0] == cin, (w.shape, x.shape)
    F = x.shape[1]
    Fo = 2 * F - 1 if t_upsample else F
    ys = []
    for f in range(Fo):
        y = None
        for kt in range(3):
            t = conv2d(x[:, causal_source_frame(f, kt, t_upsample)], w[:, :, kt], None, upsample, pad)
            y = t if y is None else y + t
        if b is not None:
            y = y + _f64(b)[:, None, None]
        ys.append(y)
    return np.stack(ys, axis=1)


def subpixel_up_weights(w):
    """Summed weights of the up conv's phase (sub-pixel) decomposition.

    With nearest-2x before a 3x3 conv, output (2v+q, 2u+p) reads source row
    v + floor((q + ky - 1) / 2) for tap ky: two distinct rows per parity q (ky 0 |
    ky 1, 2 for q = 0; ky 0, 1 | ky 2 for q = 1), and likewise for columns. The
    taps that read one source pixel are summed:
    ws[q, p, ty, tx] = sum of w[:, :, ky, kx] over ky in R(q, ty), kx in R(p, tx),
    so the parity class is a 2x2 conv on the source grid at rows
    v + ty + (-1 if q == 0 else 0) (the phase decomposition; exact in real arithmetic).
    ``w``: [cout][cin][3][3]; returns [2][2][2][2][cout][cin] (q, p, ty, tx).
    """
    w = _f64(w)
    rows = {0: ([0], [1, 2]), 1: ([0, 1], [2])}
    ws = np.zeros((2, 2, 2, 2) + w.shape[:2], _F)
    for q in range(2):
        for p in range(2):
            for ty in range(2):
                for tx in range(2):
                    for ky in rows[q][ty]:
                        for kx in rows[p][tx]:
                            ws[q, p, ty, tx] += w[:, :, ky, kx]
    return ws


def conv2d_up_subpixel(x, w, b=None, pad: str = "zero"):
    """conv2d(upsample2x(x), w, b) evaluated as four 2x2 convs on the source
    grid with ``subpixel_up_weights`` (a check of that decomposition).

    ``x``: [cin][h][w]; returns [cout][2h][2w].
    """
    x = _f64(x)
    ws = subpixel_up_weights(w)
    cin, h, wd = x.shape
    cout = ws.shape[4]
    mode = {"zero": "constant", "replicate": "edge"}[pad]
    xp = np.pad(x, ((0, 0), (1, 1), (1, 1)), mode=mode)
    y = np.zeros((cout, 2 * h, 2 * wd), _F)
    for q in range(2):
        for p in range(2):
            acc = np.zeros((cout, h * wd), _F)
            for ty in range(2):
                for tx in range(2):
                    oy, ox = ty + (0 if q == 0 else 1), tx + (0 if p == 0 else 1)  # offset into the 1-padded grid
                    tap = xp[:, oy:oy + h, ox:ox + wd].reshape(cin, h * wd)
                    acc += ws[q, p, ty, tx] @ tap
            y[:, q::2, p::2] = acc.reshape(cout, h, wd)
    if b is not None:
        y += _f64(b)[:, None, None]
    return y


def conv2d_at(x, w, b, ys, xs, upsample: bool = False, pad: str = "zero", down: bool = False):
    """``conv2d`` (or, with ``down``, ``conv2d_down``) evaluated only at output
    pixels (ys[i], xs[i]).

    The same definitions, one output pixel at a time, so that very large
    convs can be checked on a sample. ``x`` may be any array indexable as
    [c][y][x] (e.g. a transposed view of an NHWC tensor); only the receptive
    fields of the sampled pixels are read.
    Returns [len(ys)][cout].
    """
    w = _f64(w)
    cout, cin, k, _ = w.shape
    r = k // 2
    h_in, w_in = x.shape[1], x.shape[2]
    H, W = (2 * h_in, 2 * w_in) if upsample else (h_in, w_in)
    assert not (upsample and down)
    ys = np.asarray(ys, np.int64)
    xs = np.asarray(xs, np.int64)
    out = np.zeros((len(ys), cout), _F)
    if b is not None:
        out += _f64(b)[None, :]
    for ky in range(k):
        for kx in range(k):
            if down:  # the far-side pad: source rows 2Y + ky, column 2X + kx
                Y = 2 * ys + ky
                X = 2 * xs + kx
            else:
                Y = ys + ky - r
                X = xs + kx - r
            if pad == "reflect":
                Y = np.where(Y < 0, -Y, Y)
                Y = np.where(Y >= H, 2 * (H - 1) - Y, Y)
                X = np.where(X < 0, -X, X)
                X = np.where(X >= W, 2 * (W - 1) - X, X)
                inside = np.ones(len(ys), bool)
            elif pad == "replicate":
                Y = np.clip(Y, 0, H - 1)
                X = np.clip(X, 0, W - 1)
                inside = np.ones(len(ys), bool)
            else:
                inside = (Y >= 0) & (Y < H) & (X >= 0) & (X < W)
            Yc = np.clip(Y, 0, H - 1)
            Xc = np.clip(X, 0, W - 1)
            if upsample:
                Yc, Xc = Yc // 2, Xc // 2
            vals = np.stack([_f64(x[:, int(a), int(c)]) for a, c in zip(Yc, Xc)])  # [n][cin]
            vals[~inside] = 0.0
            out += vals @ w[:, :, ky, kx].T
    return out


def group_norm(x, groups: int, gamma, beta, eps: float = 1e-6, bias_in=None):
    """GroupNorm over ``groups`` groups of consecutive channels.

    For group g (channels g*C/G .. (g+1)*C/G - 1, all pixels): mean mu and the
    biased variance var (divided by n), then
    y = (v - mu) / sqrt(var + eps) * gamma[c] + beta[c], with v = x + bias_in[c].

    ``vae.rs``, ``GroupNorm::apply`` (f64 statistics, eps inside the root);
    the bias on read follows ``s2v_vae.rs``'s ``s2v_gn_part``/``s2v_gn_apply``.
    ``x``: [c][...spatial]; returns the same shape.
    """
    v = _f64(x)
    c = v.shape[0]
    assert c % groups == 0
    if bias_in is not None:
        v = v + _f64(bias_in).reshape((c,) + (1,) * (v.ndim - 1))
    per = c // groups
    out = np.empty_like(v)
    g_ = _f64(gamma).reshape((c,) + (1,) * (v.ndim - 1))
    b_ = _f64(beta).reshape((c,) + (1,) * (v.ndim - 1))
    for g in range(groups):
        s = v[g * per:(g + 1) * per]
        mu = s.mean()
        var = ((s - mu) ** 2).mean()
        out[g * per:(g + 1) * per] = (s - mu) / np.sqrt(var + eps) * g_[g * per:(g + 1) * per] \
            + b_[g * per:(g + 1) * per]
    return out


def rms_norm(x, gamma, bias_in=None):
    """Per-pixel RMS_norm over the channels (the Wan ``RMS_norm``).

    v = x + bias_in[c]; y = v * sqrt(C) / max(||v||_2, 1e-12) * gamma[c],
    the norm taken over the C channels of one pixel (no padded channels: the
    tensors carry exactly the model's channels).

    ``qi21_vae.rs``, the ``qv_rmsn`` kernel and its module doc.
    ``x``: [c][...spatial]; returns the same shape.
    """
    v = _f64(x)
    c = v.shape[0]
    if bias_in is not None:
        v = v + _f64(bias_in).reshape((c,) + (1,) * (v.ndim - 1))
    nrm = np.sqrt((v * v).sum(axis=0))
    inv = np.sqrt(float(c)) / np.maximum(nrm, 1e-12)
    return v * inv[None] * _f64(gamma).reshape((c,) + (1,) * (v.ndim - 1))


def dupup(src, out_dim: int, ft: int = 1):
    """The DupUp3D shortcut of an up block, as a tensor on the 2x grid.

    d[o, 2y+sy, 2x+sx] = src[j // repeats, y, x] with
    j = o*factor + (ft-1)*4 + 2*sy + sx, factor = 4*ft and
    repeats = out_dim*factor / in_dim (required to divide).

    ``qi21_vae.rs``, ``DUPUP_SRC`` (``qv_dupup``) and its uniform set-up in
    ``run_blocks``. ``src``: [in_dim][h][w] -> [out_dim][2h][2w].
    """
    s = _f64(src)
    cin, h, w = s.shape
    factor = 4 * ft
    assert (out_dim * factor) % cin == 0
    repeats = out_dim * factor // cin
    d = np.empty((out_dim, 2 * h, 2 * w), _F)
    for sy in range(2):
        for sx in range(2):
            for o in range(out_dim):
                j = o * factor + (ft - 1) * 4 + 2 * sy + sx
                d[o, sy::2, sx::2] = s[j // repeats]
    return d


def linear_tokens(t, conv):
    """A 1x1 conv on token-major rows: t [m][cin] -> t @ W^T + b, [m][cout].

    ``vae.rs``, ``AttnBlock::proj`` (weight rows are output channels).
    """
    w = _f64(conv.w).reshape(conv.w.shape[0], conv.w.shape[1])
    return _f64(t) @ w.T + _f64(conv.b)[None, :]


def attention(x, attn, family: str, groups: int = 32, eps: float = 1e-6,
              chunk: int = 1024):
    """Single-head spatial self-attention of the mid block, with its residual.

    n = GroupNorm(x) (FLUX family) or RMS_norm(x)*gamma (Qwen family), no SiLU;
    token-major q, k, v = n W^T + b; A = softmax_row(q k^T / sqrt(C)) with the
    row maximum subtracted before exp; o = A v; y = x + (o W_o^T + b_o).

    ``vae.rs``, ``AttnBlock::apply`` / ``AttnBlock::finish`` and
    ``qi21_vae.rs``, ``fn attention`` (the RMS variant; there the v bias is
    added after P.V, identical in exact arithmetic because rows of A sum to 1).
    ``x``: [c][h][w]; returns [c][h][w]. Query rows are taken ``chunk`` at a time.
    """
    x = _f64(x)
    c, h, w = x.shape
    m = h * w
    if family == "gn":
        n = group_norm(x, groups, attn.norm.gamma, attn.norm.beta, eps)
    else:
        n = rms_norm(x, attn.norm.gamma)
    t = n.reshape(c, m).T
    q = linear_tokens(t, attn.q)
    k = linear_tokens(t, attn.k)
    v = linear_tokens(t, attn.v)
    scale = 1.0 / np.sqrt(float(c))
    o = np.empty((m, c), _F)
    for r0 in range(0, m, chunk):
        s = (q[r0:r0 + chunk] @ k.T) * scale
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        o[r0:r0 + chunk] = p @ v
    y = linear_tokens(o, attn.o)
    return x + y.T.reshape(c, h, w)


def attention_rows(x, attn, family: str, rows, groups: int = 32, eps: float = 1e-6):
    """``attention`` evaluated only at the query tokens ``rows`` (all keys).

    Same definition as ``attention`` (``vae.rs``, ``AttnBlock::apply`` /
    ``finish``; ``qi21_vae.rs``, ``fn attention``); for sampling outputs of
    token counts whose full score matrix is too large to form here.
    ``x``: [c][h][w]; returns [len(rows)][c] (token-major rows of the output).
    """
    x = _f64(x)
    c, h, w = x.shape
    m = h * w
    rows = np.asarray(rows, dtype=np.int64)
    if family == "gn":
        n = group_norm(x, groups, attn.norm.gamma, attn.norm.beta, eps)
    else:
        n = rms_norm(x, attn.norm.gamma)
    t = n.reshape(c, m).T
    q = linear_tokens(t[rows], attn.q)
    k = linear_tokens(t, attn.k)
    v = linear_tokens(t, attn.v)
    s = (q @ k.T) / np.sqrt(float(c))
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=1, keepdims=True)
    y = linear_tokens(p @ v, attn.o)
    return x.reshape(c, m).T[rows] + y

"""Oracle decoders and band planner (float64, NCHW) — test infrastructure only.

Composes the primitives of ``oracle.ops`` in the order the pages give.
``decode_gn`` / ``decode_rms`` are the plain whole-frame definitions;
``decode_rms_banded`` is the exact-halo banded decode, written separately
so that banded == whole-frame pins the band planner.
The whole decoders are pinned against an element-by-element brute-force
restatement on tiny decoders (scalar loops, a pixel-major layout), besides
the pinned parts they compose.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional

import numpy as np

from .ops import conv2d, conv2d_down, silu, group_norm, rms_norm, dupup, attention


def _norm(x, nm, family: str, groups: int, eps: float):
    if family == "gn":
        return group_norm(x, groups, nm.gamma, nm.beta, eps)
    return rms_norm(x, nm.gamma)


def resnet(x, r, family: str, groups: int = 32, eps: float = 1e-6, pad: str = "zero"):
    """One ResNet unit: skip + conv2(silu(norm2(conv1(silu(norm1(x)))))).

    skip = x, or a 1x1 conv of x when the channel count changes.
    ``vae.rs``, ``ResnetBlock::apply`` (GroupNorm family) and
    ``qi21_vae.rs``, ``Rec::resnet`` (RMS_norm family; conv1's bias is
    added on read by the second norm, the same sum). The encoder's ResNets
    (``vae3d.rs``, ``VideoVaeEncoder::encode_tile``) are the same unit with
    reflect-padded 3x3 convs (``pad="reflect"``).
    """
    h = conv2d(silu(_norm(x, r.norm1, family, groups, eps)), r.conv1.w, r.conv1.b, pad=pad)
    h = conv2d(silu(_norm(h, r.norm2, family, groups, eps)), r.conv2.w, r.conv2.b, pad=pad)
    skip = conv2d(x, r.shortcut.w, r.shortcut.b) if r.shortcut is not None else np.asarray(x, np.float64)
    return skip + h


def up_block(x, u, family: str, with_dupup: bool, groups: int = 32, eps: float = 1e-6):
    """An up block: its ResNets, then (if present) conv3x3(upsample2x(x)).

    The up conv reads the raw stream (no norm). With ``with_dupup`` (the
    Qwen/Wan family) the DupUp shortcut of the block's INPUT is added to
    the up conv's output.
    ``vae.rs``, ``VaeDecoder::decode`` (the up-block loop) and
    ``qi21_vae.rs``, ``run_blocks``.
    """
    cp = x
    for r in u.resnets:
        x = resnet(x, r, family, groups, eps)
    if u.up is not None:
        x = conv2d(x, u.up.w, u.up.b, upsample=True)
        if with_dupup:
            x = x + dupup(cp, u.out_dim, u.ft)
    return x


def down_block(x, blk, groups: int = 32, eps: float = 1e-6):
    """An encoder level: its GroupNorm ResNets with reflect-padded convs, then
    (if present) the downsample: the far-side reflect pad and the unpadded
    stride-2 3x3 conv (``conv2d_down``).

    ``vae3d.rs``, ``VideoVaeEncoder::encode_tile`` (the level loop) and
    ``reflect_pad_far``. ``blk`` has ``resnets`` and ``down`` (a conv or None).
    """
    for r in blk.resnets:
        x = resnet(x, r, "gn", groups, eps, pad="reflect")
    if blk.down is not None:
        x = conv2d_down(x, blk.down.w, blk.down.b, pad="reflect")
    return x


def decode_gn(dec, z):
    """FLUX-class decoder: z/scaling + shift -> conv_in -> ResNet -> attention
    -> ResNet -> up blocks -> GroupNorm + SiLU -> conv_out.

    ``vae.rs``, ``VaeDecoder::decode``. ``z``: [zc][h][w] -> [nch][H][W].
    """
    g, e = dec.groups, dec.eps
    x = np.asarray(z, np.float64) / dec.scaling + dec.shift
    x = conv2d(x, dec.conv_in.w, dec.conv_in.b)
    x = resnet(x, dec.mid_res1, "gn", g, e)
    x = attention(x, dec.mid_attn, "gn", g, e)
    x = resnet(x, dec.mid_res2, "gn", g, e)
    for u in dec.ups:
        x = up_block(x, u, "gn", False, g, e)
    x = silu(group_norm(x, g, dec.norm_out.gamma, dec.norm_out.beta, e))
    return conv2d(x, dec.conv_out.w, dec.conv_out.b)


def head_rms(dec, z):
    """The latent-resolution head of the Qwen-style decoder: 1x1 post_quant
    -> conv_in -> RMS-ResNet -> attention -> RMS-ResNet.

    ``qi21_vae.rs``, the whole-frame part of ``decode``.
    """
    x = conv2d(z, dec.post_quant.w, dec.post_quant.b)
    x = conv2d(x, dec.conv_in.w, dec.conv_in.b)
    x = resnet(x, dec.mid_res1, "rms")
    x = attention(x, dec.mid_attn, "rms")
    return resnet(x, dec.mid_res2, "rms")


def decode_rms(dec, z):
    """Qwen-Image-2.1 / Wan-style decoder, whole frame: the head, the up
    blocks with DupUp, then RMS_norm(gamma) + SiLU -> conv_out.

    ``qi21_vae.rs``, ``decode`` / ``run_blocks`` / ``output_rows``.
    """
    x = head_rms(dec, z)
    for u in dec.ups:
        x = up_block(x, u, "rms", dec.dupup)
    x = silu(rms_norm(x, dec.norm_out.gamma))
    return conv2d(x, dec.conv_out.w, dec.conv_out.b)


def decode(dec, z):
    return decode_gn(dec, z) if dec.family == "gn" else decode_rms(dec, z)


# ───────────────────────────── bands ─────────────────────────────
# ``qi21_vae.rs``, the "bands" section: after the mid block every stage is
# spatially local, so blocks S.. can run on horizontal bands. Walking back
# from a band's kept output rows, a 3x3 conv needs one more row each side
# (clipped to the frame) and an upsample halves the row range, rounded
# outward. Rows next to a band edge are wrong (the conv pads there) but
# never reach a kept row.

@dataclass(frozen=True)
class Rows:
    lo: int
    hi: int

    @property
    def n(self) -> int:
        return self.hi - self.lo


def grow(r: Rows, k: int, h: int) -> Rows:
    """Rows [lo-k, hi+k) clipped to [0, h)."""
    return Rows(max(r.lo - k, 0), min(r.hi + k, h))


def half(r: Rows) -> Rows:
    """The source rows of an upsampled range: [lo/2, ceil(hi/2))."""
    return Rows(r.lo // 2, -(-r.hi // 2))


def levels(dec):
    """The resolution level of every up block, and of the output."""
    lv, l = [], 0
    for u in dec.ups:
        lv.append(l)
        l += 1 if u.up is not None else 0
    return lv, l


@dataclass
class Band:
    input: Rows
    feed: List[Optional[Rows]]
    keep: Rows


def plan_band(dec, s: int, keep: Rows, hs) -> Band:
    """Walk back from ``keep`` through conv_out and blocks s.. (last first).

    ``qi21_vae.rs``, ``plan_band``.
    """
    lvl, lf = levels(dec)
    e = grow(keep, dec.conv_out.k // 2, hs[lf])
    feed: List[Optional[Rows]] = [None] * len(dec.ups)
    for i in range(len(dec.ups) - 1, s - 1, -1):
        u = dec.ups[i]
        if u.up is not None:
            a = half(grow(e, u.up.k // 2, hs[lvl[i] + 1]))
            feed[i] = a
            e = a
        convs = sum(r.conv1.k // 2 + r.conv2.k // 2 for r in u.resnets)
        e = grow(e, convs, hs[lvl[i]])
    return Band(input=e, feed=feed, keep=keep)


def plan_bands(dec, s: int, h0: int, nbands: int) -> List[Band]:
    """``nbands`` equal bands of kept output rows: [j*k, min((j+1)*k, H)), k = ceil(H/nbands).

    ``qi21_vae.rs``, ``decode`` (the band split).
    """
    _, lf = levels(dec)
    hs = [h0 << l for l in range(lf + 1)]
    hf = hs[lf]
    k = -(-hf // max(nbands, 1))
    return [plan_band(dec, s, Rows(j * k, min((j + 1) * k, hf)), hs) for j in range(-(-hf // k))]


def run_blocks_window(dec, x, blocks, cur: Rows, feed: Callable[[int, Rows], Rows]):
    """Run up blocks ``blocks`` on ``x`` = rows ``cur`` of the first block's level.

    The convs pad at the window's edges. Block i's up conv reads only rows
    ``feed(i, cur)`` (a sub-range of ``cur``) and so does its DupUp.
    ``qi21_vae.rs``, ``run_blocks``. Returns (x, rows it holds).
    """
    for i in blocks:
        u = dec.ups[i]
        cp = x
        for r in u.resnets:
            x = resnet(x, r, "rms")
        if u.up is not None:
            f = feed(i, cur)
            assert cur.lo <= f.lo and f.hi <= cur.hi and f.n > 0, (f, cur)
            a, b = f.lo - cur.lo, f.hi - cur.lo
            y = conv2d(x[:, a:b], u.up.w, u.up.b, upsample=True)
            if dec.dupup:
                y = y + dupup(cp[:, a:b], u.out_dim, u.ft)
            x = y
            cur = Rows(2 * f.lo, 2 * f.hi)
    return x, cur


def output_rows_window(dec, x, cur: Rows, keep: Rows):
    """RMS_norm + SiLU -> conv_out on rows ``cur``, returning rows ``keep``.

    ``qi21_vae.rs``, ``output_rows``.
    """
    assert cur.lo <= keep.lo and keep.hi <= cur.hi
    y = conv2d(silu(rms_norm(x, dec.norm_out.gamma)), dec.conv_out.w, dec.conv_out.b)
    return y[:, keep.lo - cur.lo:keep.hi - cur.lo]


def decode_rms_banded(dec, z, band_from: int, nbands: int):
    """Banded decode: head and blocks < band_from on the whole frame, the
    rest band by band from the saved stream with exact halos.

    ``qi21_vae.rs``, ``decode`` (the whole part, then the band loop).
    """
    z = np.asarray(z)
    h0 = z.shape[1]
    nb = len(dec.ups)
    s = min(band_from, nb)
    x = head_rms(dec, z)
    x, cur = run_blocks_window(dec, x, range(0, s), Rows(0, h0), lambda i, c: c)
    _, lf = levels(dec)
    hf, wf = h0 << lf, z.shape[2] << lf
    out = np.zeros((dec.conv_out.cout, hf, wf), np.float64)
    if s == nb:
        out[:] = output_rows_window(dec, x, cur, Rows(0, hf))
        return out
    for bd in plan_bands(dec, s, h0, nbands):
        xb = x[:, bd.input.lo - cur.lo:bd.input.hi - cur.lo]
        xb, cb = run_blocks_window(dec, xb, range(s, nb), bd.input, lambda i, c, bd=bd: bd.feed[i])
        out[:, bd.keep.lo:bd.keep.hi] = output_rows_window(dec, xb, cb, bd.keep)
    return out

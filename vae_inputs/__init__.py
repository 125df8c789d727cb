"""Seeded synthetic inputs for the VAE-decoder hot path.

This module is shared by the oracle tests, the GPU parity tests and the
bench. It holds none of the method's arithmetic: only random draws from
numpy's ``default_rng``, the one-time rounding of weights to f16 at draw
time, and the decoder topologies (which layer has which width).

Every tensor gets its own stream: ``rng_for(seed, name)`` seeds
``default_rng`` with ``[seed, crc32(name)]``, so adding a tensor never
shifts the values of another.

Layouts (all plain numpy arrays):
- activations handed to a single conv: NHWC f16 ``[n][h][w][c]``;
- conv weights: OIHW f16 ``[cout][cin][k][k]`` (the PyTorch / diffusers
  order; each side re-lays them out for itself);
- biases, GroupNorm gamma/beta, RMS gamma: f32 ``[c]``;
- latents: NCHW f32 ``[c][h][w]`` (one frame).

Distributions (the readings of the page configs):
- He normal: ``N(0, 2/fan_in)`` with fan_in = cin*k*k, the second
  parameter read as a variance; the single-conv case uses ``N(0, 1/(9*cin))``;
- biases ``N(0, 0.01)`` (variance), i.e. std 0.1;
- GroupNorm gamma = 1, beta = 0 and RMS gamma = 1 unless ``affine=True``
  draws gamma ~ U(0.5, 1.5), beta ~ N(0, 0.1^2);
- conv_out uses half the He std, a fixed constant chosen so that the
  decoded RGB stays mostly inside [-1, 1] (u8 PSNR is taken on that range).
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

__all__ = [
    "rng_for", "f16_normal", "conv_weight", "bias_vec", "conv_case",
    "Conv", "Norm", "Resnet", "Attn", "UpBlock", "DownBlock", "Decoder",
    "flux_decoder", "qwen_decoder", "gn_up_block", "gn_down_block", "latent_normal",
    "latent_channel_stats", "stream_normal",
]


def rng_for(seed: int, name: str) -> np.random.Generator:
    """An independent generator for tensor ``name`` under ``seed``."""
    return np.random.default_rng([int(seed), zlib.crc32(name.encode("utf-8"))])


def f16_normal(seed: int, name: str, shape, std: float, mean: float = 0.0) -> np.ndarray:
    """Normal draws rounded once to IEEE f16 (round to nearest even)."""
    g = rng_for(seed, name)
    return (g.standard_normal(shape) * std + mean).astype(np.float16)


def conv_weight(seed: int, name: str, cout: int, cin: int, k: int,
                var: Optional[float] = None, gain: float = 1.0) -> np.ndarray:
    """OIHW f16 conv weight; default He normal, variance 2/(cin*k*k)."""
    v = 2.0 / (cin * k * k) if var is None else var
    return f16_normal(seed, name, (cout, cin, k, k), gain * np.sqrt(v))


def bias_vec(seed: int, name: str, c: int, var: float = 0.01) -> np.ndarray:
    g = rng_for(seed, name)
    return (g.standard_normal(c) * np.sqrt(var)).astype(np.float32)


def conv_case(seed: int = 0, n: int = 1, h: int = 32, w: int = 32, cin: int = 64,
              cout: int = 64, k: int = 3, wvar: Optional[float] = None,
              name: str = "conv") -> dict:
    """One conv's inputs: x NHWC f16 ~N(0,1), weight OIHW f16, bias f32.

    ``h, w`` are the INPUT grid (for an upsampling conv the output is 2h x 2w).
    The default weight variance is 1/(k*k*cin), the single-conv case's.
    """
    var = 1.0 / (k * k * cin) if wvar is None else wvar
    return {
        "x": f16_normal(seed, name + ".x", (n, h, w, cin), 1.0),
        "w": conv_weight(seed, name + ".w", cout, cin, k, var=var),
        "b": bias_vec(seed, name + ".b", cout),
    }


def stream_normal(seed: int, name: str, shape) -> np.ndarray:
    """An f32 residual-stream tensor ~N(0,1) (NHWC or NCHW as given)."""
    g = rng_for(seed, name)
    return g.standard_normal(shape).astype(np.float32)


def latent_normal(seed: int, c: int, h: int, w: int, name: str = "latent") -> np.ndarray:
    """NCHW f32 latent ~N(0,1) (the FLUX-class case)."""
    return stream_normal(seed, name, (c, h, w))


def latent_channel_stats(seed: int, c: int, h: int, w: int, name: str = "latent") -> np.ndarray:
    """NCHW f32 latent, channel i ~N(mu_i, sigma_i), mu ~U(-1,1), sigma ~U(0.5,2)."""
    g = rng_for(seed, name + ".stats")
    mu = g.uniform(-1.0, 1.0, c)
    sd = g.uniform(0.5, 2.0, c)
    z = rng_for(seed, name).standard_normal((c, h, w))
    return (z * sd[:, None, None] + mu[:, None, None]).astype(np.float32)


# ───────────────────────── decoder descriptions ─────────────────────────

@dataclass
class Conv:
    w: np.ndarray            # f16 [cout][cin][k][k]
    b: np.ndarray            # f32 [cout]

    @property
    def cout(self) -> int:
        return int(self.w.shape[0])

    @property
    def cin(self) -> int:
        return int(self.w.shape[1])

    @property
    def k(self) -> int:
        return int(self.w.shape[2])


@dataclass
class Norm:
    gamma: np.ndarray                  # f32 [c]
    beta: Optional[np.ndarray] = None  # f32 [c]; GroupNorm only


@dataclass
class Resnet:
    norm1: Norm
    conv1: Conv
    norm2: Norm
    conv2: Conv
    shortcut: Optional[Conv] = None    # 1x1 when cin != cout


@dataclass
class Attn:
    norm: Norm
    q: Conv
    k: Conv
    v: Conv
    o: Conv

    @property
    def c(self) -> int:
        return self.q.cout


@dataclass
class UpBlock:
    resnets: List[Resnet]
    up: Optional[Conv] = None          # 3x3 conv applied after nearest-2x
    in_dim: int = 0
    out_dim: int = 0
    ft: int = 1                        # DupUp temporal factor (rms family)


@dataclass
class DownBlock:
    resnets: List[Resnet]
    down: Optional[Conv] = None        # 3x3 stride-2 conv after the far-side pad
    in_dim: int = 0
    out_dim: int = 0


@dataclass
class Decoder:
    family: str                        # "gn" (FLUX-class) or "rms" (Qwen/Wan-style)
    conv_in: Conv
    mid_res1: Resnet
    mid_attn: Attn
    mid_res2: Resnet
    ups: List[UpBlock]
    norm_out: Norm
    conv_out: Conv
    post_quant: Optional[Conv] = None  # rms family: 1x1 before conv_in
    latent_channels: int = 16
    scaling: float = 1.0               # gn family: z/scaling + shift
    shift: float = 0.0
    groups: int = 32
    eps: float = 1e-6
    dupup: bool = False                # rms family: DupUp shortcut on up blocks
    extra: dict = field(default_factory=dict)


def _norm(seed: int, name: str, c: int, family: str, affine: bool) -> Norm:
    if affine:
        g = rng_for(seed, name + ".gamma").uniform(0.5, 1.5, c).astype(np.float32)
        b = (rng_for(seed, name + ".beta").standard_normal(c) * 0.1).astype(np.float32)
    else:
        g = np.ones(c, np.float32)
        b = np.zeros(c, np.float32)
    return Norm(gamma=g, beta=b if family == "gn" else None)


def _conv(seed: int, name: str, cout: int, cin: int, k: int, gain: float = 1.0) -> Conv:
    return Conv(w=conv_weight(seed, name + ".w", cout, cin, k, gain=gain),
                b=bias_vec(seed, name + ".b", cout))


def _resnet(seed: int, name: str, cin: int, cout: int, family: str, affine: bool) -> Resnet:
    return Resnet(
        norm1=_norm(seed, name + ".norm1", cin, family, affine),
        conv1=_conv(seed, name + ".conv1", cout, cin, 3),
        norm2=_norm(seed, name + ".norm2", cout, family, affine),
        conv2=_conv(seed, name + ".conv2", cout, cout, 3),
        shortcut=_conv(seed, name + ".shortcut", cout, cin, 1) if cin != cout else None,
    )


def _attn(seed: int, name: str, c: int, family: str, affine: bool) -> Attn:
    return Attn(norm=_norm(seed, name + ".norm", c, family, affine),
                q=_conv(seed, name + ".q", c, c, 1), k=_conv(seed, name + ".k", c, c, 1),
                v=_conv(seed, name + ".v", c, c, 1), o=_conv(seed, name + ".o", c, c, 1))


def flux_decoder(seed: int = 0, latent_channels: int = 16,
                 block_out=(128, 256, 512, 512), layers_per_block: int = 2,
                 nch: int = 3, affine: bool = False) -> Decoder:
    """FLUX-class AutoencoderKL decoder with random weights.

    conv_in 16->512; mid = ResNet, single-head attention, ResNet at 512;
    up blocks with widths 512, 512, 256, 128 (reversed ``block_out``), each
    ``layers_per_block + 1`` ResNets, all but the last ending in nearest-2x
    + 3x3 conv; GroupNorm(32, 1e-6) + SiLU + conv_out 128->3.
    """
    fam = "gn"
    widths = list(reversed(block_out))
    top = widths[0]
    ups = []
    cur = top
    for i, wd in enumerate(widths):
        res = []
        for r in range(layers_per_block + 1):
            res.append(_resnet(seed, f"up{i}.res{r}", cur, wd, fam, affine))
            cur = wd
        up = _conv(seed, f"up{i}.upconv", wd, wd, 3) if i < len(widths) - 1 else None
        ups.append(UpBlock(resnets=res, up=up, in_dim=wd, out_dim=wd))
    return Decoder(
        family=fam,
        conv_in=_conv(seed, "conv_in", top, latent_channels, 3),
        mid_res1=_resnet(seed, "mid.res1", top, top, fam, affine),
        mid_attn=_attn(seed, "mid.attn", top, fam, affine),
        mid_res2=_resnet(seed, "mid.res2", top, top, fam, affine),
        ups=ups,
        norm_out=_norm(seed, "norm_out", widths[-1], fam, affine),
        conv_out=_conv(seed, "conv_out", nch, widths[-1], 3, gain=0.5),
        latent_channels=latent_channels,
    )


def qwen_decoder(seed: int = 0, latent_channels: int = 16,
                 widths=(1152, 576, 288, 144), nres: int = 3, nch: int = 3,
                 ft: int = 1, affine: bool = False) -> Decoder:
    """Qwen-Image-2.1 / Wan-style decoder with per-pixel RMS_norm and DupUp.

    1x1 post_quant zc->zc, conv_in zc->w0, mid = RMS-ResNet, attention,
    RMS-ResNet at w0; up block i: ``nres`` ResNets w_i->w_i, and for all
    but the last an up conv w_i->w_{i+1} on the 2x grid plus the DupUp
    shortcut of the block input; RMS(gamma)+SiLU + conv_out w_last->3.
    """
    fam = "rms"
    ups = []
    for i, wd in enumerate(widths):
        res = [_resnet(seed, f"up{i}.res{r}", wd, wd, fam, affine) for r in range(nres)]
        if i < len(widths) - 1:
            nxt = widths[i + 1]
            ups.append(UpBlock(resnets=res, up=_conv(seed, f"up{i}.upconv", nxt, wd, 3),
                               in_dim=wd, out_dim=nxt, ft=ft))
        else:
            ups.append(UpBlock(resnets=res, up=None, in_dim=wd, out_dim=wd, ft=ft))
    w0 = widths[0]
    return Decoder(
        family=fam,
        post_quant=_conv(seed, "post_quant", latent_channels, latent_channels, 1),
        conv_in=_conv(seed, "conv_in", w0, latent_channels, 3),
        mid_res1=_resnet(seed, "mid.res1", w0, w0, fam, affine),
        mid_attn=_attn(seed, "mid.attn", w0, fam, affine),
        mid_res2=_resnet(seed, "mid.res2", w0, w0, fam, affine),
        ups=ups,
        norm_out=_norm(seed, "norm_out", widths[-1], fam, affine),
        conv_out=_conv(seed, "conv_out", nch, widths[-1], 3, gain=0.5),
        latent_channels=latent_channels,
        dupup=True,
    )


def gn_up_block(seed: int = 0, c: int = 256, nres: int = 2, affine: bool = False) -> UpBlock:
    """One GroupNorm up block: ``nres`` ResNets c->c, then nearest-2x + 3x3 conv c->c."""
    res = [_resnet(seed, f"blk.res{r}", c, c, "gn", affine) for r in range(nres)]
    return UpBlock(resnets=res, up=_conv(seed, "blk.upconv", c, c, 3), in_dim=c, out_dim=c)


def gn_down_block(seed: int = 0, cin: int = 128, cout: int = 128, nres: int = 2, affine: bool = True,
                  down: bool = True) -> DownBlock:
    """One encoder level: ``nres`` GroupNorm ResNets (the first cin->cout, with
    a 1x1 shortcut when the widths differ), then a stride-2 3x3 conv cout->cout."""
    res = [_resnet(seed, f"enc.res{r}", cin if r == 0 else cout, cout, "gn", affine) for r in range(nres)]
    return DownBlock(resnets=res, down=_conv(seed, "enc.down", cout, cout, 3) if down else None,
                     in_dim=cin, out_dim=cout)

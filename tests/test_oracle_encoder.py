"""Pins of the oracle's encoder-direction ops (CPU only): reflect padding and
the far-side-padded stride-2 downsample conv, and the encoder level built from
them.

Reflect padding mirrors about the edge without repeating it (index -1 reads 1,
index n reads n - 2): a delta tap on a ramp image exposes the mirrored border
directly, a constant image gives sum(w) + b everywhere, and an independent
brute-force loop with its own mirror function agrees on tiny inputs. The
downsample conv is the stride-1 unpadded conv over the far-side-padded grid
taken at odd-free (even) positions; its output is h//2 x w//2; the far edge
reads row h - 2 (reflect), h - 1 (replicate) or 0 (zero); and brute force agrees
for every padding and both parities of h and w. A level whose ResNets have zero
conv2 weights and bias is the downsample conv alone.
"""
import itertools

import numpy as np
import pytest

import oracle
from vae_inputs import gn_down_block, stream_normal


def _mirror(i, n):
    # the definition: reflect about the edges until inside (edge not repeated)
    while i < 0 or i >= n:
        if i < 0:
            i = -i
        if i >= n:
            i = 2 * (n - 1) - i
    return i


def _case(seed, cin=3, cout=2, h=4, w=5, k=3):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((cin, h, w)), rng.standard_normal((cout, cin, k, k)), rng.standard_normal(cout)


def _brute_reflect(x, wt, b):
    cin, h, w = x.shape
    cout, _, k, _ = wt.shape
    r = k // 2
    y = np.zeros((cout, h, w))
    for o, Y, X in itertools.product(range(cout), range(h), range(w)):
        acc = b[o]
        for c, ky, kx in itertools.product(range(cin), range(k), range(k)):
            acc += wt[o, c, ky, kx] * x[c, _mirror(Y + ky - r, h), _mirror(X + kx - r, w)]
        y[o, Y, X] = acc
    return y


def _brute_down(x, wt, b, pad):
    cin, h, w = x.shape
    cout, _, k, _ = wt.shape
    Ho, Wo = (h + 1 - k) // 2 + 1, (w + 1 - k) // 2 + 1
    y = np.zeros((cout, Ho, Wo))
    for o, Y, X in itertools.product(range(cout), range(Ho), range(Wo)):
        acc = b[o]
        for c, ky, kx in itertools.product(range(cin), range(k), range(k)):
            sy, sx = 2 * Y + ky, 2 * X + kx  # rows / columns 0..h of the far-padded grid
            if sy == h or sx == w:
                if pad == "zero":
                    continue
                if pad == "replicate":
                    sy, sx = min(sy, h - 1), min(sx, w - 1)
                else:
                    sy = h - 2 if sy == h else sy
                    sx = w - 2 if sx == w else sx
            acc += wt[o, c, ky, kx] * x[c, sy, sx]
        y[o, Y, X] = acc
    return y


@pytest.mark.parametrize("h,w", [(2, 2), (3, 5), (4, 4), (5, 3)])
def test_reflect_conv_brute_force_tiny(h, w):
    x, wt, b = _case(1, h=h, w=w)
    np.testing.assert_allclose(oracle.conv2d(x, wt, b, pad="reflect"), _brute_reflect(x, wt, b),
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("ky,kx", list(itertools.product(range(3), range(3))))
def test_reflect_delta_tap_on_a_ramp(ky, kx):
    h, w = 5, 6
    ramp = (10.0 * np.arange(h)[:, None] + np.arange(w)[None, :])[None]  # x[Y, X] = 10 Y + X
    wt = np.zeros((1, 1, 3, 3))
    wt[0, 0, ky, kx] = 1.0
    y = oracle.conv2d(ramp, wt, None, pad="reflect")[0]
    for Y, X in itertools.product(range(h), range(w)):
        sy, sx = Y + ky - 1, X + kx - 1
        sy = 1 if sy == -1 else (h - 2 if sy == h else sy)
        sx = 1 if sx == -1 else (w - 2 if sx == w else sx)
        assert y[Y, X] == 10 * sy + sx


def test_reflect_constant_image():
    _, wt, b = _case(2)
    x = np.full((3, 4, 5), -1.25)
    got = oracle.conv2d(x, wt, b, pad="reflect")
    ref = -1.25 * wt.sum(axis=(1, 2, 3)) + b
    np.testing.assert_allclose(got, np.broadcast_to(ref[:, None, None], got.shape), rtol=1e-12, atol=1e-12)


def test_reflect_differs_from_replicate_and_zero_only_at_the_border():
    x, wt, b = _case(3, h=6, w=7)
    r = oracle.conv2d(x, wt, b, pad="reflect")
    for other in ("zero", "replicate"):
        o = oracle.conv2d(x, wt, b, pad=other)
        np.testing.assert_allclose(r[:, 1:-1, 1:-1], o[:, 1:-1, 1:-1], rtol=1e-12, atol=1e-12)
        assert np.abs(r[:, 0, :] - o[:, 0, :]).max() > 1e-3


@pytest.mark.parametrize("pad", ["zero", "replicate", "reflect"])
@pytest.mark.parametrize("h,w", [(2, 2), (4, 6), (5, 4), (7, 7)])
def test_down_conv_brute_force_tiny(pad, h, w):
    x, wt, b = _case(4, h=h, w=w)
    got = oracle.conv2d_down(x, wt, b, pad=pad)
    assert got.shape == (2, h // 2, w // 2)
    np.testing.assert_allclose(got, _brute_down(x, wt, b, pad), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("h,w", [(6, 8), (7, 5)])
def test_down_conv_is_the_padded_stride1_conv_at_even_positions(h, w):
    """Stride 2 = the stride-1 conv over the far-padded grid, sampled at
    (2Y + 1, 2X + 1) of its symmetric-pad-1 form, where no padding is read."""
    x, wt, b = _case(5, h=h, w=w)
    xp = np.concatenate([x, x[:, h - 2:h - 1, :]], axis=1)        # row h = row h - 2
    xp = np.concatenate([xp, xp[:, :, w - 2:w - 1]], axis=2)      # column w = column w - 2
    full = oracle.conv2d(xp, wt, b)                               # (h+1) x (w+1), zero pad 1
    np.testing.assert_allclose(oracle.conv2d_down(x, wt, b, pad="reflect"), full[:, 1::2, 1::2][:, :h // 2, :w // 2],
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("pad,expect", [("reflect", "h-2"), ("replicate", "h-1"), ("zero", "0")])
def test_down_conv_far_edge(pad, expect):
    h, w = 6, 8
    x, _, _ = _case(6, cin=1, h=h, w=w)
    wt = np.zeros((1, 1, 3, 3))
    wt[0, 0, 2, 2] = 1.0
    y = oracle.conv2d_down(x, wt, None, pad=pad)[0]
    ref = {"h-2": x[0, h - 2, w - 2], "h-1": x[0, h - 1, w - 1], "0": 0.0}[expect]
    assert y[-1, -1] == ref
    assert y[0, 0] == x[0, 2, 2]


@pytest.mark.parametrize("down", [False, True])
def test_conv2d_at_matches_the_whole_conv(down):
    x, wt, b = _case(7, cin=4, cout=3, h=9, w=8)
    whole = oracle.conv2d_down(x, wt, b) if down else oracle.conv2d(x, wt, b, pad="reflect")
    H, W = whole.shape[1:]
    ys, xs = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
    got = oracle.conv2d_at(x, wt, b, ys.ravel(), xs.ravel(), pad="reflect", down=down)
    np.testing.assert_allclose(got, whole.reshape(3, -1).T, rtol=1e-12, atol=1e-12)


def test_down_block_with_silent_resnets_is_the_down_conv():
    blk = gn_down_block(seed=1, cin=32, cout=32, nres=2)
    for r in blk.resnets:
        r.conv2.w = np.zeros_like(r.conv2.w)
        r.conv2.b = np.zeros_like(r.conv2.b)
    x = np.moveaxis(stream_normal(1, "enc.x", (8, 6, 32)), -1, 0)
    np.testing.assert_allclose(oracle.down_block(x, blk), oracle.conv2d_down(x, blk.down.w, blk.down.b),
                               rtol=1e-12, atol=1e-12)


def test_reflect_needs_two_pixels():
    x, wt, b = _case(8, h=1, w=4)
    with pytest.raises(AssertionError):
        oracle.conv2d(x, wt, b, pad="reflect")
    with pytest.raises(AssertionError):
        oracle.conv2d_down(x, wt, b)

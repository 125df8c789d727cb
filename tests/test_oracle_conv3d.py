"""Pins of the oracle's 3x3x3 causal conv (CPU only).

A single frame reduces it to the 2-D conv with the three temporal taps summed
(every tap reads the one frame); a weight living on one temporal tap shifts
frames by the causal look-back, clamped at the first frame; the temporal 2x
maps output frames 0..4 to source frames 0, 1, 1, 2, 2 (the first frame is not
doubled); a constant volume with replicate padding gives sum(w) + b
everywhere; and an independent brute-force loop agrees on tiny volumes for
every padding / spatial / temporal upsample combination.
"""
import itertools

import numpy as np
import pytest

import oracle


def _case(seed, cin=3, cout=2, F=3, h=4, w=5):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((cin, F, h, w))
    wt = rng.standard_normal((cout, cin, 3, 3, 3))
    b = rng.standard_normal(cout)
    return x, wt, b


@pytest.mark.parametrize("up,pad", [(False, "zero"), (True, "zero"), (False, "replicate"), (True, "replicate")])
def test_single_frame_is_the_2d_conv_of_the_summed_taps(up, pad):
    x, wt, b = _case(1, F=1)
    got = oracle.conv3d_causal(x, wt, b, upsample=up, pad=pad)
    ref = oracle.conv2d(x[:, 0], wt.sum(axis=2), b, upsample=up, pad=pad)
    assert got.shape[1] == 1
    np.testing.assert_allclose(got[:, 0], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("kt,look_back", [(2, 0), (1, 1), (0, 2)])
def test_one_temporal_tap_shifts_frames_causally(kt, look_back):
    x, wt, b = _case(2, F=5)
    w1 = np.zeros_like(wt)
    w1[:, :, kt] = wt[:, :, kt]
    got = oracle.conv3d_causal(x, w1, b)
    for f in range(5):
        ref = oracle.conv2d(x[:, max(f - look_back, 0)], wt[:, :, kt], b)
        np.testing.assert_allclose(got[:, f], ref, rtol=1e-12, atol=1e-12)


def test_temporal_upsample_frame_map():
    x, wt, b = _case(3, F=3)
    w1 = np.zeros_like(wt)
    w1[:, :, 2] = wt[:, :, 2]  # the current frame only
    got = oracle.conv3d_causal(x, w1, b, t_upsample=True)
    assert got.shape[1] == 5
    for f, s in enumerate([0, 1, 1, 2, 2]):
        np.testing.assert_allclose(got[:, f], oracle.conv2d(x[:, s], wt[:, :, 2], b), rtol=1e-12, atol=1e-12)
    # and the look-back two frames behind output frame 4 is source frame 1
    w0 = np.zeros_like(wt)
    w0[:, :, 0] = wt[:, :, 0]
    got0 = oracle.conv3d_causal(x, w0, None, t_upsample=True)
    np.testing.assert_allclose(got0[:, 4], oracle.conv2d(x[:, 1], wt[:, :, 0]), rtol=1e-12, atol=1e-12)


def test_constant_volume_with_replicate_padding():
    x, wt, b = _case(4)
    x = np.full_like(x, 0.75)
    got = oracle.conv3d_causal(x, wt, b, upsample=True, t_upsample=True, pad="replicate")
    ref = 0.75 * wt.sum(axis=(1, 2, 3, 4)) + b
    np.testing.assert_allclose(got, np.broadcast_to(ref[:, None, None, None], got.shape), rtol=1e-12, atol=1e-12)


def _brute(x, wt, b, up, t_up, pad):
    cin, F, h, w = x.shape
    cout = wt.shape[0]
    H, W = (2 * h, 2 * w) if up else (h, w)
    Fo = 2 * F - 1 if t_up else F
    y = np.zeros((cout, Fo, H, W))
    for o, f, Y, X in itertools.product(range(cout), range(Fo), range(H), range(W)):
        acc = b[o]
        for kt, ky, kx in itertools.product(range(3), range(3), range(3)):
            vf = f + kt - 2
            if vf < 0:
                vf = 0
            sf = vf if not t_up else (0 if vf == 0 else (vf - 1) // 2 + 1)
            yy, xx = Y + ky - 1, X + kx - 1
            if pad == "zero" and not (0 <= yy < H and 0 <= xx < W):
                continue
            yy = min(max(yy, 0), H - 1)
            xx = min(max(xx, 0), W - 1)
            sy, sx = (yy // 2, xx // 2) if up else (yy, xx)
            for c in range(cin):
                acc += wt[o, c, kt, ky, kx] * x[c, sf, sy, sx]
        y[o, f, Y, X] = acc
    return y


@pytest.mark.parametrize("up,t_up,pad", list(itertools.product([False, True], [False, True], ["zero", "replicate"])))
def test_brute_force_tiny(up, t_up, pad):
    x, wt, b = _case(5, cin=2, cout=2, F=3, h=3, w=4)
    got = oracle.conv3d_causal(x, wt, b, upsample=up, t_upsample=t_up, pad=pad)
    np.testing.assert_allclose(got, _brute(x, wt, b, up, t_up, pad), rtol=1e-12, atol=1e-12)

"""Pins of the oracle's conv, upsample and padding (CPU only).

Each check is chosen so that a plausible mistake fails at least one:
a dropped tap (hand example, brute force), a flipped kernel (delta taps),
a transposed weight (cin != cout brute force), a wrong upsample index
(printed example, brute force with Y//2), a wrong border (zero vs
replicate brute force, constant image), a wrong bias axis (brute force).
"""
import itertools

import numpy as np
import pytest

import oracle
from conftest import load_golden


def brute_conv(x, w, b, upsample=False, pad="zero"):
    """Independent direct sum: explicit loops over every index."""
    cin, h, wd = x.shape
    cout, _, k, _ = w.shape
    H, W = (2 * h, 2 * wd) if upsample else (h, wd)
    r = k // 2
    y = np.zeros((cout, H, W))
    for o in range(cout):
        for Y in range(H):
            for X in range(W):
                acc = 0.0 if b is None else float(b[o])
                for c in range(cin):
                    for ky in range(k):
                        for kx in range(k):
                            yy, xx = Y + ky - r, X + kx - r
                            if pad == "replicate":
                                yy = min(max(yy, 0), H - 1)
                                xx = min(max(xx, 0), W - 1)
                            elif not (0 <= yy < H and 0 <= xx < W):
                                continue
                            if upsample:
                                yy, xx = yy // 2, xx // 2
                            acc += float(w[o, c, ky, kx]) * float(x[c, yy, xx])
                y[o, Y, X] = acc
    return y


def test_hand_reference_printed_values():
    g = load_golden("conv2d_hand_reference.json")
    x = np.array(g["x"], float)[None]
    w = np.array(g["weight"], float)
    y = oracle.conv2d(x, w, np.array(g["bias"]))
    for p in g["printed"]:
        assert y[0, p["y"], p["x"]] == p["value"]


def test_upsample_printed_values():
    g = load_golden("upsample_nearest.json")
    y = oracle.upsample2x(np.array(g["x"], float)[None])
    assert np.array_equal(y[0], np.array(g["printed"], float))


@pytest.mark.parametrize("upsample,pad,k,cin,cout,h,w", [
    (False, "zero", 3, 2, 3, 4, 5),
    (False, "replicate", 3, 3, 2, 5, 3),
    (True, "zero", 3, 2, 2, 3, 2),
    (True, "replicate", 3, 2, 3, 2, 3),
    (False, "zero", 1, 3, 2, 3, 4),
    (False, "zero", 3, 1, 1, 1, 1),
])
def test_brute_force_tiny(upsample, pad, k, cin, cout, h, w):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((cin, h, w))
    wt = rng.standard_normal((cout, cin, k, k))
    b = rng.standard_normal(cout)
    got = oracle.conv2d(x, wt, b, upsample=upsample, pad=pad)
    ref = brute_conv(x, wt, b, upsample=upsample, pad=pad)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("ky,kx", list(itertools.product(range(3), range(3))))
def test_delta_tap_is_a_shift(ky, kx):
    """A single tap (ky,kx) with an identity channel map reads x[Y+ky-1, X+kx-1]."""
    rng = np.random.default_rng(ky * 3 + kx)
    c, h, w = 2, 5, 6
    x = rng.standard_normal((c, h, w))
    wt = np.zeros((c, c, 3, 3))
    for i in range(c):
        wt[i, i, ky, kx] = 1.0
    y = oracle.conv2d(x, wt, None)
    ref = np.zeros_like(x)
    dy, dx = ky - 1, kx - 1
    for Y in range(h):
        for X in range(w):
            if 0 <= Y + dy < h and 0 <= X + dx < w:
                ref[:, Y, X] = x[:, Y + dy, X + dx]
    assert np.array_equal(y, ref)


def test_centre_tap_identity_plus_bias():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 4, 4))
    wt = np.zeros((3, 3, 3, 3))
    for i in range(3):
        wt[i, i, 1, 1] = 1.0
    b = np.array([0.5, -1.0, 2.0])
    np.testing.assert_array_equal(oracle.conv2d(x, wt, b), x + b[:, None, None])


def test_linearity_in_x_and_w():
    rng = np.random.default_rng(2)
    x1, x2 = rng.standard_normal((2, 3, 6, 5))
    w1, w2 = rng.standard_normal((2, 4, 3, 3, 3))
    a, c = 0.7, -1.3
    lhs = oracle.conv2d(a * x1 + c * x2, w1, None)
    rhs = a * oracle.conv2d(x1, w1, None) + c * oracle.conv2d(x2, w1, None)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    lhs = oracle.conv2d(x1, a * w1 + c * w2, None)
    rhs = a * oracle.conv2d(x1, w1, None) + c * oracle.conv2d(x1, w2, None)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


def test_replicate_constant_image():
    """With replicate padding a constant image gives sum(w)*const + b everywhere."""
    rng = np.random.default_rng(3)
    x = np.full((2, 5, 4), 1.5)
    wt = rng.standard_normal((3, 2, 3, 3))
    b = rng.standard_normal(3)
    for up in (False, True):
        y = oracle.conv2d(x, wt, b, upsample=up, pad="replicate")
        ref = wt.sum(axis=(1, 2, 3)) * 1.5 + b
        np.testing.assert_allclose(y, np.broadcast_to(ref[:, None, None], y.shape), rtol=1e-13)


def test_upsampled_constant_stays_constant():
    x = np.full((1, 3, 3), 2.0)
    assert np.array_equal(oracle.upsample2x(x), np.full((1, 6, 6), 2.0))


def test_upsample_conv_equals_materialised_upsample():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 4, 5))
    wt = rng.standard_normal((2, 3, 3, 3))
    b = rng.standard_normal(2)
    for pad in ("zero", "replicate"):
        a = oracle.conv2d(x, wt, b, upsample=True, pad=pad)
        c = oracle.conv2d(oracle.upsample2x(x), wt, b, upsample=False, pad=pad)
        np.testing.assert_array_equal(a, c)


@pytest.mark.parametrize("upsample,pad", [(False, "zero"), (True, "zero"), (False, "replicate"), (True, "replicate")])
def test_conv2d_at_matches_full(upsample, pad):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 6, 7))
    wt = rng.standard_normal((3, 4, 3, 3))
    b = rng.standard_normal(3)
    full = oracle.conv2d(x, wt, b, upsample=upsample, pad=pad)
    H, W = full.shape[1:]
    ys = rng.integers(0, H, 40)
    xs = rng.integers(0, W, 40)
    ys[:4] = [0, 0, H - 1, H - 1]
    xs[:4] = [0, W - 1, 0, W - 1]
    got = oracle.conv2d_at(x, wt, b, ys, xs, upsample=upsample, pad=pad)
    np.testing.assert_allclose(got, full[:, ys, xs].T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("pad", ["zero", "replicate"])
def test_subpixel_decomposition_of_the_up_conv_is_exact(pad):
    """The up conv as four 2x2 convs with summed weights (the phase form) equals
    conv(upsample2x(x)) in exact arithmetic: f64 agreement to 1e-12."""
    rng = np.random.default_rng(41)
    x = rng.standard_normal((3, 5, 6))
    w = rng.standard_normal((4, 3, 3, 3))
    b = rng.standard_normal(4)
    ref = oracle.conv2d(x, w, b, upsample=True, pad=pad)
    got = oracle.conv2d_up_subpixel(x, w, b, pad=pad)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_subpixel_weights_sum_to_the_kernel():
    """Each parity class's four summed taps hold all nine weights once."""
    rng = np.random.default_rng(42)
    w = rng.standard_normal((2, 3, 3, 3))
    ws = oracle.subpixel_up_weights(w)
    for q in range(2):
        for p in range(2):
            np.testing.assert_allclose(ws[q, p].sum(axis=(0, 1)), w.sum(axis=(2, 3)), rtol=1e-12, atol=1e-12)
    # parity (0, 0): top-left tap alone, then the 1x2 / 2x1 / 2x2 sums
    np.testing.assert_allclose(ws[0, 0, 0, 0], w[:, :, 0, 0])
    np.testing.assert_allclose(ws[0, 0, 1, 1], w[:, :, 1:, 1:].sum(axis=(2, 3)))

"""Pins of the oracle's band planner, ResNet skip path and banded decode (CPU only).

The band planner is pinned by the page's printed walk-back values and by
the invariant the pages state: a banded decode with exact halos equals the
whole-frame decode. Both decoders here are the oracle's, so the invariant
is checked to 1e-10 (not bit for bit: BLAS may block a smaller matmul
differently, which moves the last bits; a wrong halo moves values by O(1)).
"""
import dataclasses

import numpy as np
import pytest

import oracle
from oracle import Rows
from conftest import load_golden
from vae_inputs import (Conv, Resnet, UpBlock, Decoder, Norm, qwen_decoder, flux_decoder,
                        latent_channel_stats, latent_normal)


def test_band_walk_back_printed_values():
    g = load_golden("band_rows_walk_back.json")
    keep = Rows(*g["keep"])
    e = oracle.grow(keep, 1, g["frame_rows"])
    e = oracle.grow(e, 0, g["frame_rows"])
    a = oracle.half(oracle.grow(e, 1, g["frame_rows"]))
    assert a == Rows(*g["printed_feed"])
    assert oracle.grow(a, 2, g["frame_rows"] // 2) == Rows(*g["printed_input"])
    ec = g["edge_case"]
    assert oracle.grow(Rows(*ec["rows"]), ec["k"], ec["h"]) == Rows(*ec["printed"])


def _conv(c_out, c_in, k, rng):
    return Conv(w=rng.standard_normal((c_out, c_in, k, k)).astype(np.float16), b=np.zeros(c_out, np.float32))


def test_plan_band_matches_printed_walk_back():
    """plan_band on the printed stage list: one ResNet then the up conv, a final
    block without ResNets, conv_out."""
    g = load_golden("band_rows_walk_back.json")
    rng = np.random.default_rng(0)
    n = Norm(gamma=np.ones(4, np.float32))
    res = Resnet(norm1=n, conv1=_conv(4, 4, 3, rng), norm2=n, conv2=_conv(4, 4, 3, rng))
    dec = Decoder(family="rms", conv_in=_conv(4, 4, 3, rng), mid_res1=res, mid_attn=None, mid_res2=res,
                  ups=[UpBlock(resnets=[res], up=_conv(4, 4, 3, rng), in_dim=4, out_dim=4),
                       UpBlock(resnets=[], up=None, in_dim=4, out_dim=4)],
                  norm_out=n, conv_out=_conv(3, 4, 3, rng))
    bd = oracle.plan_band(dec, 0, Rows(*g["keep"]), [g["frame_rows"] // 2, g["frame_rows"]])
    assert bd.feed[0] == Rows(*g["printed_feed"])
    assert bd.input == Rows(*g["printed_input"])


def test_plan_bands_cover_the_frame():
    dec = qwen_decoder(seed=0, widths=(32, 16, 16, 16), nres=1)
    for nb in (1, 2, 3, 5):
        bands = oracle.plan_bands(dec, 1, 6, nb)
        rows = [r for b in bands for r in range(b.keep.lo, b.keep.hi)]
        assert rows == list(range(48))


def test_resnet_skip_path():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 3, 3))
    n = Norm(gamma=np.ones(4, np.float32))
    zero = Conv(w=np.zeros((4, 4, 3, 3), np.float16), b=np.zeros(4, np.float32))
    r = Resnet(norm1=n, conv1=_conv(4, 4, 3, rng), norm2=n, conv2=zero)
    np.testing.assert_array_equal(oracle.resnet(x, r, "rms"), x)
    zero6 = Conv(w=np.zeros((6, 6, 3, 3), np.float16), b=np.zeros(6, np.float32))
    sc = _conv(6, 4, 1, rng)
    r2 = Resnet(norm1=n, conv1=_conv(6, 4, 3, rng), norm2=Norm(gamma=np.ones(6, np.float32)), conv2=zero6, shortcut=sc)
    np.testing.assert_allclose(oracle.resnet(x, r2, "rms"), oracle.conv2d(x, sc.w, sc.b), rtol=1e-14)


def _tiny_qwen():
    return qwen_decoder(seed=3, widths=(32, 16, 16), nres=1)


@pytest.mark.parametrize("band_from,nbands", [(0, 3), (1, 4), (2, 2), (3, 2)])
def test_banded_equals_whole(band_from, nbands):
    dec = _tiny_qwen()
    z = latent_channel_stats(0, 16, 6, 5)
    whole = oracle.decode_rms(dec, z)
    banded = oracle.decode_rms_banded(dec, z, band_from=band_from, nbands=nbands)
    assert whole.shape == (3, 24, 20)
    np.testing.assert_allclose(banded, whole, rtol=0, atol=1e-10 * np.abs(whole).max())


def test_banded_with_a_wrong_halo_differs():
    """The banded == whole pin is sensitive: dropping one halo row breaks it."""
    dec = _tiny_qwen()
    z = latent_channel_stats(0, 16, 6, 5)
    whole = oracle.decode_rms(dec, z)
    orig = oracle.decoder.grow
    try:
        oracle.decoder.grow = lambda r, k, h: orig(r, max(k - 1, 0), h)
        bad = oracle.decode_rms_banded(dec, z, band_from=0, nbands=3)
    finally:
        oracle.decoder.grow = orig
    assert np.abs(bad - whole).max() > 1e-3


def test_flux_decoder_shapes_and_finite():
    dec = flux_decoder(seed=1, block_out=(32, 32, 32, 32), layers_per_block=1)
    z = latent_normal(1, 16, 3, 4)
    y = oracle.decode_gn(dec, z)
    assert y.shape == (3, 24, 32)
    assert np.isfinite(y).all()

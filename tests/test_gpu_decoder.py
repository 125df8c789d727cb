"""Whole-decoder GPU parity against the oracle (u8 PSNR >= 60 dB), the
up-block configuration built from the library's ops, band-vs-whole
bit-exactness (torch.equal) including the 2048^2 and 1536x2752 frames, banded
decodes of those frames against the oracle's bands, and the host-buffer
(end-to-end) call."""
import numpy as np
import pytest

import oracle
import implicit_gemm_convolution_vae_gb300 as vg
from gpu_common import psnr_u8, rel_err, report_parity, saturated_fraction, to_dev, torch_mod
from vae_inputs import (flux_decoder, gn_up_block, latent_channel_stats, latent_normal, qwen_decoder,
                        stream_normal)

pytestmark = pytest.mark.gpu

PSNR_MIN = 60.0


def gpu_decode(dec, z, opts=None):
    torch = torch_mod()
    D = vg.Decoder(dec)
    out = D.decode(to_dev(z), opts=opts)
    vg.sync_status()
    return out, D


def check_psnr(got, ref, case=None):
    assert np.isfinite(got).all()
    rec = report_parity(case or "decode", got, ref)
    assert rec["saturated_fraction"] < 0.05
    assert rec["psnr_u8_db"] >= PSNR_MIN, rec
    return rec["psnr_u8_db"]


def test_flux_decoder_tiny():
    dec = flux_decoder(seed=1, block_out=(32, 32, 32, 32), layers_per_block=1)
    z = latent_normal(1, 16, 4, 5)
    out, _ = gpu_decode(dec, z)
    check_psnr(out.cpu().numpy(), oracle.decode_gn(dec, z), "flux_decoder_tiny")


def test_flux_decoder_config3():
    """FLUX-class AutoencoderKL, latent [16,32,32] -> RGB 256^2, random He-normal weights."""
    dec = flux_decoder(seed=0)
    z = latent_normal(0, 16, 32, 32)
    out, _ = gpu_decode(dec, z)
    check_psnr(out.cpu().numpy(), oracle.decode_gn(dec, z), "flux_decoder_256")


def test_qwen_decoder_tiny():
    dec = qwen_decoder(seed=2, widths=(64, 32, 32, 16), nres=1)
    z = latent_channel_stats(2, 16, 6, 5)
    out, _ = gpu_decode(dec, z)
    check_psnr(out.cpu().numpy(), oracle.decode_rms(dec, z), "qwen_decoder_tiny")


def test_qwen_decoder_config4_architecture_256():
    """The 1024^2 decoder's exact widths (1152, 576, 288, 144; 3 ResNets) at latent 32^2."""
    dec = qwen_decoder(seed=0)
    z = latent_channel_stats(0, 16, 32, 32)
    out, _ = gpu_decode(dec, z)
    check_psnr(out.cpu().numpy(), oracle.decode_rms(dec, z), "qwen_decoder_256")


def test_subpixel_up_convs_in_both_families():
    """VAE_DECODE_SUBPIXEL_UP: the up convs as four 2x2 convs with summed weights
    (only the f16 rounding of the sums differs from the plain definition), for the
    FLUX-class decoder at config 3 and the 1024^2 decoder's widths at latent 32^2."""
    dec = flux_decoder(seed=0)
    z = latent_normal(0, 16, 32, 32)
    out, _ = gpu_decode(dec, z, opts=vg.Decoder.opts(subpixel=True))
    check_psnr(out.cpu().numpy(), oracle.decode_gn(dec, z), "flux_decoder_256_subpixel_up")
    dec = qwen_decoder(seed=0)
    z = latent_channel_stats(0, 16, 32, 32)
    out, _ = gpu_decode(dec, z, opts=vg.Decoder.opts(subpixel=True))
    check_psnr(out.cpu().numpy(), oracle.decode_rms(dec, z), "qwen_decoder_256_subpixel_up")


def test_up_block_config2():
    """One GroupNorm up block at 128^2 x 256 (2 ResNets, nearest-2x + conv), composed
    from the library's GroupNorm, conv and cast entry points."""
    torch = torch_mod()
    blk = gn_up_block(seed=0, c=256, nres=2)
    x = stream_normal(0, "cfg2.x", (128, 128, 256))
    xd = to_dev(x.copy()).reshape(1, 128 * 128, 256)
    for r in blk.resnets:
        xn = vg.groupnorm_silu(xd, 32, to_dev(r.norm1.gamma), to_dev(r.norm1.beta), silu=True)
        h = vg.conv3x3_nhwc(xn.reshape(1, 128, 128, 256), to_dev(vg.pack_conv3x3(r.conv1.w)), to_dev(r.conv1.b))
        xn = vg.groupnorm_silu(h.reshape(1, -1, 256), 32, to_dev(r.norm2.gamma), to_dev(r.norm2.beta), silu=True)
        vg.conv3x3_nhwc(xn.reshape(1, 128, 128, 256), to_dev(vg.pack_conv3x3(r.conv2.w)), to_dev(r.conv2.b),
                        residual=xd.reshape(1, 128, 128, 256), out=xd.reshape(1, 128, 128, 256))
    xs = vg.cast_f16(xd, 256, scale=2.0 ** -8)
    y = vg.conv3x3_nhwc(xs.reshape(1, 128, 128, 256), to_dev(vg.pack_conv3x3(blk.up.w)), to_dev(blk.up.b),
                        upsample=True, oscale=256.0)
    vg.sync_status()
    ref = oracle.up_block(np.moveaxis(x, -1, 0), blk, "gn", False)
    got = np.moveaxis(y[0].cpu().numpy(), -1, 0)
    # Five f16-input convs in a chain: each conv's inputs carry one f16 rounding (2^-11) and the
    # GroupNorm statistics are f32; 1e-2 of max|ref| bounds their composition.
    assert rel_err(got, ref) <= 1e-2


BAND_CASES = [(0, 3, 0), (1, 4, 0), (2, 2, 0), (3, 5, 0), (2, 0, 40), (1, 0, 7)]


@pytest.mark.parametrize("band_from,nbands,band_rows", BAND_CASES)
def test_banded_decode_is_bit_identical(band_from, nbands, band_rows):
    torch = torch_mod()
    dec = qwen_decoder(seed=4, widths=(64, 32, 32, 16), nres=2)
    z = latent_channel_stats(4, 16, 12, 10)
    whole, D = gpu_decode(dec, z)
    banded = D.decode(to_dev(z), opts=vg.Decoder.opts(band_from=band_from, nbands=nbands, band_rows=band_rows))
    vg.sync_status()
    assert torch.equal(whole, banded)


@pytest.mark.parametrize("h0,w0", [(256, 256), (192, 344)])
def test_banded_decode_bit_identical_at_full_frames(h0, w0):
    """2048^2 and 1536x2752 with the 1024^2 decoder's widths: 3 bands from up block 2."""
    torch = torch_mod()
    dec = qwen_decoder(seed=0)
    z = latent_channel_stats(5, 16, h0, w0)
    D = vg.Decoder(dec)
    opts = vg.Decoder.opts(band_from=2, nbands=3)
    assert D.workspace_bytes(h0, w0, opts) < D.workspace_bytes(h0, w0)
    whole = D.decode(to_dev(z))
    banded = D.decode(to_dev(z), opts=opts)
    vg.sync_status()
    assert torch.isfinite(whole).all().item()
    assert torch.equal(whole, banded)


@pytest.mark.parametrize("h0,w0", [(256, 256), (192, 344)])
def test_banded_decode_matches_oracle_bands_at_full_frames(h0, w0):
    """2048^2 and 1536x2752 frames, 3 bands from up block 2, against the
    oracle's own banded decode (its exact-halo planner). The decoder keeps the
    1024^2 decoder's structure (3 ResNets per block, three up blocks with
    DupUp, mid attention over all 65536 / 66048 latent tokens) at narrow widths;
    the halos depend on the structure, not on the widths. The oracle's f64
    softmax over 65536^2 scores dominates its ~50 s."""
    dec = qwen_decoder(seed=6, widths=(32, 16, 16, 16), nres=3)
    z = latent_channel_stats(6, 16, h0, w0)
    D = vg.Decoder(dec)
    got = D.decode(to_dev(z), opts=vg.Decoder.opts(band_from=2, nbands=3))
    vg.sync_status()
    ref = oracle.decode_rms_banded(dec, z, 2, 3)
    assert got.shape == ref.shape == (3, 8 * h0, 8 * w0)
    check_psnr(got.cpu().numpy(), ref, f"qwen_narrow_banded_{8 * h0}x{8 * w0}")


def test_host_buffer_decode_matches_device_decode():
    torch = torch_mod()
    dec = qwen_decoder(seed=6, widths=(64, 32, 32, 16), nres=1)
    z = latent_channel_stats(6, 16, 8, 8)
    dev_out, D = gpu_decode(dec, z)
    zh = torch.from_numpy(z).pin_memory()
    oh = torch.empty(dev_out.shape, dtype=torch.float32).pin_memory()
    ws = torch.empty(D.workspace_bytes(8, 8), dtype=torch.uint8, device="cuda")
    D.decode_host(zh, oh, ws)
    assert torch.equal(oh, dev_out.cpu())


@pytest.mark.parametrize("widths,nres,hw", [((64, 32, 32, 16), 2, (12, 10)), ((1152, 576, 288, 144), 3, (16, 16)),
                                            ((1152, 576, 288, 144), 2, (20, 18))])
def test_fused_norms_are_bit_identical_to_separate_norms(widths, nres, hw):
    """RMS_norm fused into the producing conv's epilogue (the staged two-pass
    form on rows of >= 128 pixels, the register form on narrower ones) gives the
    same bits as the standalone RMS_norm kernel (one shared evaluation order)."""
    torch = torch_mod()
    dec = qwen_decoder(seed=7, widths=widths, nres=nres)
    z = latent_channel_stats(7, 16, *hw)
    separate, D = gpu_decode(dec, z, opts=vg.Decoder.opts(fuse=False))
    forced = D.decode(to_dev(z), opts=vg.Decoder.opts(fuse=True))
    default = D.decode(to_dev(z))
    vg.sync_status()
    assert torch.equal(forced, separate)
    assert torch.equal(default, separate)


def test_gn_family_rejects_bands():
    dec = flux_decoder(seed=1, block_out=(32, 32, 32, 32), layers_per_block=1)
    D = vg.Decoder(dec)
    with pytest.raises(vg.VaeError) as e:
        D.decode(to_dev(latent_normal(1, 16, 4, 4)), opts=vg.Decoder.opts(band_from=1, nbands=2))
    assert e.value.code == -7


@pytest.mark.parametrize("family", ["rms", "gn"])
def test_graph_replay_matches_eager_decode(family):
    """A decode captured as a CUDA graph gives the eager decode's bits, and a
    replay after the latent buffer's contents change decodes the new latent."""
    torch = torch_mod()
    if family == "rms":
        dec = qwen_decoder(seed=8, widths=(64, 32, 32, 16), nres=1)
        z1, z2 = latent_channel_stats(8, 16, 6, 5), latent_channel_stats(9, 16, 6, 5)
    else:
        dec = flux_decoder(seed=8, block_out=(32, 32, 32, 32), layers_per_block=1)
        z1, z2 = latent_normal(8, 16, 6, 5), latent_normal(9, 16, 6, 5)
    D = vg.Decoder(dec)
    zd = to_dev(z1)
    out = torch.empty((3, 48, 40), dtype=torch.float32, device="cuda")
    ws = torch.empty(D.workspace_bytes(6, 5), dtype=torch.uint8, device="cuda")
    g = D.graph(zd, out, ws)
    out.fill_(float("nan"))
    g.launch()
    vg.sync_status()
    assert torch.equal(out, D.decode(to_dev(z1)))
    zd.copy_(to_dev(z2))
    g.launch()
    g.launch()
    vg.sync_status()
    assert torch.equal(out, D.decode(to_dev(z2)))


@pytest.mark.parametrize("family,band_from,nbands", [("gn", 0, 1), ("rms", 0, 1), ("rms", 1, 3), ("rms", 2, 4)])
def test_cast_fused_into_the_last_resnet_conv_is_bit_identical(family, band_from, nbands):
    """By default the last ResNet conv of an up block stores the up conv's guarded
    f16 input itself ((conv + bias + skip) * 2^-8 rounded to f16); with fusion off a
    separate cast kernel reads the f32 stream. Same bits, whole frame and in bands
    (where the up conv reads only the feed rows of the conv's whole row range)."""
    torch = torch_mod()
    if family == "gn":
        dec = flux_decoder(seed=5, block_out=(32, 32, 64, 64), layers_per_block=1)
        z = latent_normal(5, 16, 6, 10)
    else:
        dec = qwen_decoder(seed=6, widths=(64, 32, 32, 16), nres=2)
        z = latent_channel_stats(6, 16, 12, 10)
    kw = dict(band_from=band_from, nbands=nbands)
    separate, D = gpu_decode(dec, z, opts=vg.Decoder.opts(fuse=False, **kw))
    fused = D.decode(to_dev(z), opts=vg.Decoder.opts(**kw))
    vg.sync_status()
    assert torch.equal(fused, separate)

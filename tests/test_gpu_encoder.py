"""GPU parity of the encoder-direction convs (through the C ABI) against the
oracle: reflect padding and the far-side-padded stride-2 downsample, element
by element on small, ragged and multi-tile shapes (every padding mode, even
and odd sizes, the 2x2 minimum, every epilogue variant), on sampled pixels at
the 1024^2 encoder-level sizes, and an encoder level (GroupNorm ResNets with
reflect-padded convs, then the downsample) composed from the library's ops.
Outputs start as NaN so an unwritten element fails."""
import numpy as np
import pytest

import oracle
import implicit_gemm_convolution_vae_gb300 as vg
from gpu_common import CONV_TOL, rel_err, sentinel_like, to_dev, torch_mod
from vae_inputs import conv_case, f16_normal, gn_down_block, stream_normal

pytestmark = pytest.mark.gpu


def _run(case, pad="zero", down=False, silu=False, out_f16=False, residual=None, oscale=1.0):
    torch = torch_mod()
    n, h, wd, _ = case["x"].shape
    cout = case["w"].shape[0]
    H, W = (h // 2, wd // 2) if down else (h, wd)
    out = sentinel_like((n, H, W, cout), torch.float16 if out_f16 else torch.float32)
    vg.conv3x3_nhwc(to_dev(case["x"]), to_dev(vg.pack_conv3x3(case["w"])), to_dev(case["b"]),
                    residual=None if residual is None else to_dev(residual), out=out, oscale=oscale,
                    replicate=pad == "replicate", reflect=pad == "reflect", down=down, silu=silu, out_f16=out_f16)
    vg.sync_status()
    return out.float().cpu().numpy()


def _ref(case, pad="zero", down=False, silu=False, residual=None):
    outs = []
    for i in range(case["x"].shape[0]):
        xc = np.moveaxis(case["x"][i].astype(np.float64), -1, 0)
        y = oracle.conv2d_down(xc, case["w"], case["b"], pad=pad) if down else \
            oracle.conv2d(xc, case["w"], case["b"], pad=pad)
        y = np.moveaxis(y, 0, -1)
        if residual is not None:
            y = y + residual[i]
        if silu:
            y = oracle.silu(y)
        outs.append(y)
    return np.stack(outs)


SHAPES = [
    # n, h, w, cin, cout
    (1, 2, 2, 16, 16),
    (1, 3, 3, 16, 48),
    (1, 2, 7, 48, 16),
    (2, 7, 33, 16, 144),
    (1, 33, 8, 144, 16),
    (1, 6, 200, 32, 64),
    (1, 5, 257, 64, 3),
    (1, 4, 260, 128, 128),
    (1, 9, 40, 80, 320),
    # rows of >= 128 pixels (the halo boxes with the mirrored edge columns): exactly one
    # tile wide, a one-pixel last tile, two tiles, a 16-channel K remainder, two N tiles
    (1, 3, 128, 64, 64),
    (2, 4, 129, 32, 48),
    (1, 3, 256, 128, 144),
    (1, 5, 150, 80, 64),
    (1, 4, 129, 144, 144),
    (1, 3, 256, 208, 96),
    (1, 3, 140, 64, 256),
    # the downsample's TMA path (even widths, >= 128 output columns): a 3-tile row with
    # a ragged last tile, and 258 columns (129 outputs: its reflect form gathers)
    (1, 5, 600, 32, 48),
    (1, 4, 258, 64, 64),
]


@pytest.mark.parametrize("n,h,w,cin,cout", SHAPES)
def test_reflect_conv_shapes(n, h, w, cin, cout):
    case = conv_case(seed=11, n=n, h=h, w=w, cin=cin, cout=cout, name=f"refl.{n}.{h}.{w}.{cin}.{cout}")
    got = _run(case, pad="reflect")
    assert not np.isnan(got).any()
    assert rel_err(got, _ref(case, pad="reflect")) <= CONV_TOL


@pytest.mark.parametrize("pad", ["zero", "replicate", "reflect"])
@pytest.mark.parametrize("n,h,w,cin,cout", SHAPES)
def test_down_conv_shapes(n, h, w, cin, cout, pad):
    case = conv_case(seed=12, n=n, h=h, w=w, cin=cin, cout=cout, name=f"down.{n}.{h}.{w}.{cin}.{cout}")
    got = _run(case, pad=pad, down=True)
    assert got.shape == (n, h // 2, w // 2, cout)
    assert not np.isnan(got).any()
    assert rel_err(got, _ref(case, pad=pad, down=True)) <= CONV_TOL


@pytest.mark.parametrize("down", [False, True])
@pytest.mark.parametrize("silu,out_f16,with_res", [(True, False, True), (False, True, False), (True, True, True)])
def test_encoder_conv_epilogues(down, silu, out_f16, with_res):
    case = conv_case(seed=13, n=1, h=18, w=134, cin=64, cout=96, name="enc.epi")
    H, W = (9, 67) if down else (18, 134)
    res = stream_normal(13, "enc.epi.res", (1, H, W, 96)) if with_res else None
    got = _run(case, pad="reflect", down=down, silu=silu, out_f16=out_f16, residual=res)
    ref = _ref(case, pad="reflect", down=down, silu=silu, residual=res)
    # f16 output adds one rounding (at most 2^-11 of max|ref| ~ 4.9e-4), inside the per-conv bound
    assert rel_err(got, ref) <= CONV_TOL


def test_reflect_conv_in_place_residual():
    torch = torch_mod()
    case = conv_case(seed=14, n=1, h=20, w=150, cin=128, cout=128, name="enc.inplace")
    res = stream_normal(14, "enc.inplace.res", (1, 20, 150, 128))
    y = to_dev(res.copy())
    vg.conv3x3_nhwc(to_dev(case["x"]), to_dev(vg.pack_conv3x3(case["w"])), to_dev(case["b"]), residual=y, out=y,
                    reflect=True)
    vg.sync_status()
    assert rel_err(y.cpu().numpy(), _ref(case, pad="reflect", residual=res)) <= CONV_TOL


def _sample_points(H, W, n, seed):
    rng = np.random.default_rng(seed)
    ys = list(rng.integers(0, H, n))
    xs = list(rng.integers(0, W, n))
    for y in (0, 1, H // 2, H - 2, H - 1):
        for x in (0, 1, 127, 128, W // 2, W - 129, W - 128, W - 1):
            ys.append(y)
            xs.append(x)
    return np.array(ys), np.array(xs)


@pytest.mark.parametrize("stage", ["resnet_1024_reflect", "down_1024_to_512"])
def test_full_size_encoder_stage_sampled(stage):
    """The 1024^2 encoder level: a 128 -> 128 reflect-padded 3x3 conv at 1024^2, and
    the 128 -> 128 downsample 1024^2 -> 512^2, as the bench times them."""
    torch = torch_mod()
    h = w = 1024
    cin = cout = 128
    down = stage.startswith("down")
    x = f16_normal(15, f"enc.full.{stage}.x", (1, h, w, cin), 1.0)
    wt = f16_normal(15, f"enc.full.{stage}.w", (cout, cin, 3, 3), (2.0 / (9 * cin)) ** 0.5)
    b = (stream_normal(15, f"enc.full.{stage}.b", (cout,)) * 0.1).astype(np.float32)
    H, W = (h // 2, w // 2) if down else (h, w)
    out = sentinel_like((1, H, W, cout), torch.float32)
    vg.conv3x3_nhwc(to_dev(x), to_dev(vg.pack_conv3x3(wt)), to_dev(b), out=out, reflect=True, down=down)
    vg.sync_status()
    assert not torch.isnan(out).any().item()
    ys, xs = _sample_points(H, W, 400, 16)
    got = out[0, torch.from_numpy(ys).cuda(), torch.from_numpy(xs).cuda()].cpu().numpy()
    ref = oracle.conv2d_at(np.moveaxis(x[0], -1, 0), wt, b, ys, xs, pad="reflect", down=down)
    assert rel_err(got, ref) <= CONV_TOL


@pytest.mark.parametrize("cin,cout,h,w", [(64, 128, 64, 64), (128, 128, 130, 66)])
def test_encoder_level_from_library_ops(cin, cout, h, w):
    """One encoder level (2 GroupNorm ResNets with reflect-padded 3x3 convs, the
    first with a 1x1 shortcut when the widths differ, then the far-side-padded
    stride-2 conv), composed from the library's GroupNorm, conv, 1x1 and cast
    entry points, against the oracle's level."""
    torch = torch_mod()
    blk = gn_down_block(seed=17, cin=cin, cout=cout, nres=2)
    x = stream_normal(17, "enc.level.x", (h, w, cin))
    xd = to_dev(x.copy()).reshape(1, h * w, cin)
    c = cin
    for r in blk.resnets:
        xn = vg.groupnorm_silu(xd, 32, to_dev(r.norm1.gamma), to_dev(r.norm1.beta), silu=True)
        hb = vg.conv3x3_nhwc(xn.reshape(1, h, w, c), to_dev(vg.pack_conv3x3(r.conv1.w)), to_dev(r.conv1.b),
                             reflect=True)
        hn = vg.groupnorm_silu(hb.reshape(1, -1, cout), 32, to_dev(r.norm2.gamma), to_dev(r.norm2.beta), silu=True)
        if r.shortcut is not None:
            xs = vg.cast_f16(xd, c)
            skip = vg.conv1x1(xs.reshape(h * w, c), to_dev(vg.pack_conv1x1(r.shortcut.w)), to_dev(r.shortcut.b))
            skip = skip.reshape(1, h, w, cout)
        else:
            skip = xd.reshape(1, h, w, cout)
        y = torch.empty((1, h, w, cout), dtype=torch.float32, device="cuda")
        vg.conv3x3_nhwc(hn.reshape(1, h, w, cout), to_dev(vg.pack_conv3x3(r.conv2.w)), to_dev(r.conv2.b),
                        residual=skip, out=y, reflect=True)
        xd = y.reshape(1, h * w, cout)
        c = cout
    xs = vg.cast_f16(xd, cout)
    out = vg.conv3x3_nhwc(xs.reshape(1, h, w, cout), to_dev(vg.pack_conv3x3(blk.down.w)), to_dev(blk.down.b),
                          reflect=True, down=True)
    vg.sync_status()
    ref = oracle.down_block(np.moveaxis(x, -1, 0), blk)
    got = np.moveaxis(out[0].cpu().numpy(), -1, 0)
    assert got.shape == ref.shape == (cout, h // 2, w // 2)
    # Five f16-input convs in a chain (each input rounded to f16 once) with f32
    # GroupNorm statistics: 1e-2 of max|ref| bounds their composition.
    assert rel_err(got, ref) <= 1e-2

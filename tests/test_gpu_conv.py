"""GPU parity of the implicit-GEMM conv (through the C ABI) against the oracle.

Element by element on small and ragged shapes (several M and N tiles, a
ragged tail, K chunks shorter than 64 channels, every padding/upsample
combination, every epilogue variant), and on sampled pixels at the
full 1024^2 stage sizes in the launch configuration the bench times.
Outputs start as NaN so an unwritten element fails.
"""
import numpy as np
import pytest

import oracle
import implicit_gemm_convolution_vae_gb300 as vg
from gpu_common import CONV_TOL, rel_err, sentinel_like, to_dev, torch_mod
from vae_inputs import conv_case, f16_normal, stream_normal

pytestmark = pytest.mark.gpu


def _run(case, upsample=False, replicate=False, silu=False, out_f16=False, residual=None, oscale=1.0):
    torch = torch_mod()
    x = to_dev(case["x"])
    w = to_dev(vg.pack_conv3x3(case["w"]))
    b = to_dev(case["b"])
    n, h, wd, _ = case["x"].shape
    cout = case["w"].shape[0]
    H, W = (2 * h, 2 * wd) if upsample else (h, wd)
    out = sentinel_like((n, H, W, cout), torch.float16 if out_f16 else torch.float32)
    res = None if residual is None else to_dev(residual)
    vg.conv3x3_nhwc(x, w, b, residual=res, out=out, oscale=oscale, upsample=upsample, replicate=replicate,
                    silu=silu, out_f16=out_f16)
    vg.sync_status()
    return out.float().cpu().numpy()


def _ref(case, upsample=False, replicate=False, silu=False, residual=None):
    outs = []
    for i in range(case["x"].shape[0]):
        xc = np.moveaxis(case["x"][i].astype(np.float64), -1, 0)
        y = oracle.conv2d(xc, case["w"], case["b"], upsample=upsample, pad="replicate" if replicate else "zero")
        y = np.moveaxis(y, 0, -1)
        if residual is not None:
            y = y + residual[i]
        if silu:
            y = oracle.silu(y)
        outs.append(y)
    return np.stack(outs)


@pytest.mark.parametrize("variant", ["zero", "upsample", "replicate", "upsample_replicate"])
def test_single_conv_config(variant):
    """The 32x32x64 -> 64 conv (and its 16x16 -> 32x32 upsample fold), seed 0."""
    up = variant.startswith("upsample")
    rep = variant.endswith("replicate")
    h = 16 if up else 32
    case = conv_case(seed=0, h=h, w=h, cin=64, cout=64, name=f"cfg1.{'up' if up else 'plain'}")
    got = _run(case, upsample=up, replicate=rep)
    ref = _ref(case, upsample=up, replicate=rep)
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= CONV_TOL


SHAPES = [
    # n, h, w, cin, cout
    (1, 1, 1, 16, 16),
    (1, 2, 3, 16, 48),
    (1, 3, 7, 48, 16),
    (2, 7, 33, 16, 144),
    (1, 33, 7, 144, 16),
    (1, 5, 200, 32, 64),
    (1, 3, 256, 64, 3),
    (1, 4, 130, 144, 288),
    (1, 9, 40, 80, 320),
    # cin % 64 == 16 on rows of >= 128 pixels: the 16-channel remainder stage
    (1, 6, 200, 80, 64),
    (2, 5, 128, 208, 144),
    (1, 3, 300, 144, 3),
]


@pytest.mark.parametrize("n,h,w,cin,cout", SHAPES)
@pytest.mark.parametrize("up,rep", [(False, False), (True, False), (False, True), (True, True)])
def test_conv_shapes(n, h, w, cin, cout, up, rep):
    case = conv_case(seed=1, n=n, h=h, w=w, cin=cin, cout=cout, name=f"shape.{n}.{h}.{w}.{cin}.{cout}")
    got = _run(case, upsample=up, replicate=rep)
    ref = _ref(case, upsample=up, replicate=rep)
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= CONV_TOL


@pytest.mark.parametrize("silu,out_f16,with_res", [(True, False, False), (False, True, False),
                                                   (False, False, True), (True, True, True)])
def test_conv_epilogue(silu, out_f16, with_res):
    case = conv_case(seed=2, h=12, w=150, cin=48, cout=96, name="epi")
    res = stream_normal(2, "epi.res", (1, 12, 150, 96)) if with_res else None
    got = _run(case, silu=silu, out_f16=out_f16, residual=res, oscale=1.0)
    ref = _ref(case, silu=silu, residual=res)
    assert not np.isnan(got).any()
    # f16 output adds one rounding (at most 2^-11 of max|ref| ~ 4.9e-4), inside the per-conv bound
    assert rel_err(got, ref) <= CONV_TOL


def test_conv_in_place_residual_and_oscale():
    """y = oscale*acc + b + y (the stream update x += conv(..)), with a 2^8 guard undo."""
    torch = torch_mod()
    case = conv_case(seed=3, h=8, w=64, cin=32, cout=32, name="inplace")
    xs = (case["x"].astype(np.float32) * 2.0 ** -8).astype(np.float16)
    stream = stream_normal(3, "inplace.s", (1, 8, 64, 32))
    y = to_dev(stream.copy())
    vg.conv3x3_nhwc(to_dev(xs), to_dev(vg.pack_conv3x3(case["w"])), to_dev(case["b"]), residual=y, out=y,
                    oscale=256.0)
    vg.sync_status()
    xc = np.moveaxis(xs[0].astype(np.float64), -1, 0) * 256.0
    ref = np.moveaxis(oracle.conv2d(xc, case["w"], case["b"]), 0, -1)[None] + stream
    assert rel_err(y.cpu().numpy(), ref) <= CONV_TOL


@pytest.mark.parametrize("m,cin,cout", [(1, 16, 16), (100, 16, 16), (1000, 512, 256), (333, 1152, 1152),
                                        (4096, 144, 3)])
def test_conv1x1(m, cin, cout):
    torch = torch_mod()
    x = f16_normal(4, f"c11.x.{m}", (m, cin), 1.0)
    w = f16_normal(4, f"c11.w.{cin}", (cout, cin, 1, 1), (1.0 / cin) ** 0.5)
    b = stream_normal(4, f"c11.b.{cout}", (cout,)) * 0.1
    out = sentinel_like((m, cout), torch.float32)
    vg.conv1x1(to_dev(x), to_dev(vg.pack_conv1x1(w)), to_dev(b.astype(np.float32)), out=out)
    vg.sync_status()
    ref = x.astype(np.float64) @ w[:, :, 0, 0].astype(np.float64).T + b
    got = out.cpu().numpy()
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= CONV_TOL


# The 1x1 convs over one row of pixels run on CTA pairs (adjacent 128-pixel
# tiles share each weight tile): the attention projections' shapes (q / k: f16
# rows, N tiles of 192; v^T: 9 pixel tiles, so one pair holds a single tile,
# N tiles of 256; the output projection added in place onto the f32 stream), a
# ragged N tile, a 16-channel tail chunk, and the single-CTA kernel on the same
# inputs for comparison.
@pytest.mark.parametrize("m,cin,cout,f16,inplace", [(16384, 1152, 1152, True, False),
                                                    (1152, 1152, 16384, True, False),
                                                    (16384, 1152, 1152, False, True),
                                                    (333, 256, 200, False, True),
                                                    (700, 80, 48, True, False),
                                                    (5000, 144, 3, False, False)])
def test_conv1x1_pair_gemm(m, cin, cout, f16, inplace):
    torch = torch_mod()
    x = f16_normal(5, f"pg.x.{m}.{cin}", (m, cin), 1.0)
    w = f16_normal(5, f"pg.w.{cout}.{cin}", (cout, cin, 1, 1), (1.0 / cin) ** 0.5)
    b = (stream_normal(5, f"pg.b.{cout}", (cout,)) * 0.1).astype(np.float32)
    ref = x.astype(np.float64) @ w[:, :, 0, 0].astype(np.float64).T + b
    if inplace:
        s0 = stream_normal(5, f"pg.s.{m}.{cout}", (m, cout)).astype(np.float32)
        out = to_dev(s0.copy())
        vg.conv1x1(to_dev(x), to_dev(vg.pack_conv1x1(w)), to_dev(b), residual=out, out=out)
        ref = ref + s0
    else:
        out = sentinel_like((m, cout), torch.float16 if f16 else torch.float32)
        vg.conv1x1(to_dev(x), to_dev(vg.pack_conv1x1(w)), to_dev(b), out=out, out_f16=f16)
    vg.sync_status()
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert rel_err(got, ref) <= CONV_TOL


def _sample_points(H, W, n, seed):
    rng = np.random.default_rng(seed)
    ys = list(rng.integers(0, H, n))
    xs = list(rng.integers(0, W, n))
    for y in (0, 1, H // 2, H - 2, H - 1):
        for x in (0, 1, 127, 128, W // 2, W - 129, W - 128, W - 1):
            ys.append(y)
            xs.append(x)
    return np.array(ys), np.array(xs)


@pytest.mark.parametrize("stage", ["b3_resnet_1024", "b2_upconv_512_to_1024"])
def test_full_size_stage_sampled(stage):
    """The 1024^2 stages: 144->144 3x3 at 1024^2, and the 288->144 up conv 512^2 -> 1024^2."""
    torch = torch_mod()
    if stage == "b3_resnet_1024":
        h = w = 1024
        cin, cout, up = 144, 144, False
    else:
        h = w = 512
        cin, cout, up = 288, 144, True
    x = f16_normal(5, f"full.{stage}.x", (1, h, w, cin), 1.0)
    wt = f16_normal(5, f"full.{stage}.w", (cout, cin, 3, 3), (2.0 / (9 * cin)) ** 0.5)
    b = (stream_normal(5, f"full.{stage}.b", (cout,)) * 0.1).astype(np.float32)
    H, W = (2 * h, 2 * w) if up else (h, w)
    out = sentinel_like((1, H, W, cout), torch.float32)
    vg.conv3x3_nhwc(to_dev(x), to_dev(vg.pack_conv3x3(wt)), to_dev(b), out=out, upsample=up)
    vg.sync_status()
    assert not torch.isnan(out).any().item()
    ys, xs = _sample_points(H, W, 400, 6)
    got = out[0, torch.from_numpy(ys).cuda(), torch.from_numpy(xs).cuda()].cpu().numpy()
    ref = oracle.conv2d_at(np.moveaxis(x[0], -1, 0), wt, b, ys, xs, upsample=up)
    assert rel_err(got, ref) <= CONV_TOL


@pytest.mark.parametrize("n,h,w,cin,cout", SHAPES)
@pytest.mark.parametrize("rep", [False, True])
def test_subpixel_up_conv_matches_the_plain_definition(n, h, w, cin, cout, rep):
    """The up conv's sub-pixel form (summed weights, four 2x2 convs) against the
    oracle's conv(upsample2x(x)): the f16 rounding of the weight sums stays well
    inside the conv tolerance."""
    torch = torch_mod()
    case = conv_case(seed=1, n=n, h=h, w=w, cin=cin, cout=cout, name=f"shape.{n}.{h}.{w}.{cin}.{cout}")
    ws = vg.pack_subpixel_weights(to_dev(vg.pack_conv3x3(case["w"])))
    out = sentinel_like((n, 2 * h, 2 * w, cout), torch.float32)
    vg.conv3x3_nhwc(to_dev(case["x"]), ws, to_dev(case["b"]), out=out, upsample=True, replicate=rep, subpixel=True)
    vg.sync_status()
    got = out.cpu().numpy()
    assert not np.isnan(got).any()
    assert rel_err(got, _ref(case, upsample=True, replicate=rep)) <= CONV_TOL


def test_subpixel_up_conv_full_size_sampled():
    """The 512^2 -> 1024^2, 288 -> 144 up conv of the 1024^2 decoder in the sub-pixel form."""
    torch = torch_mod()
    h = w = 512
    cin, cout = 288, 144
    x = f16_normal(7, "sub.x", (1, h, w, cin), 1.0)
    wt = f16_normal(7, "sub.w", (cout, cin, 3, 3), (2.0 / (9 * cin)) ** 0.5)
    b = (stream_normal(7, "sub.b", (cout,)) * 0.1).astype(np.float32)
    ws = vg.pack_subpixel_weights(to_dev(vg.pack_conv3x3(wt)))
    out = sentinel_like((1, 2 * h, 2 * w, cout), torch.float32)
    vg.conv3x3_nhwc(to_dev(x), ws, to_dev(b), out=out, upsample=True, subpixel=True)
    vg.sync_status()
    assert not torch.isnan(out).any().item()
    ys, xs = _sample_points(2 * h, 2 * w, 400, 8)
    got = out[0, torch.from_numpy(ys).cuda(), torch.from_numpy(xs).cuda()].cpu().numpy()
    ref = oracle.conv2d_at(np.moveaxis(x[0], -1, 0), wt, b, ys, xs, upsample=True)
    assert rel_err(got, ref) <= CONV_TOL


@pytest.mark.parametrize("n,h,w,cin,cout,kw", [
    (1, 6, 256, 144, 144, {}),                    # staged two-pass epilogue (rows of >= 128 pixels)
    (2, 5, 130, 144, 144, {}),                    # CTA pairs over an odd tile-row count, two images
    (1, 5, 200, 64, 64, {}),                      # ragged last tile
    (2, 9, 40, 32, 48, {}),                       # rows shorter than a tile: the register form
    (1, 4, 130, 80, 16, {"reflect": True}),
    (1, 8, 300, 64, 144, {"down": True}),
])
@pytest.mark.parametrize("with_y", [False, True])
def test_conv_with_fused_rmsnorm_is_bit_identical(n, h, w, cin, cout, kw, with_y):
    """vae_conv3x3_nhwc_rms gives the same bits as vae_conv3x3_nhwc followed by
    vae_rmsnorm_silu (one shared evaluation order), with and without the f32 output."""
    torch = torch_mod()
    case = conv_case(seed=31, n=n, h=h, w=w, cin=cin, cout=cout, name=f"rmsf.{n}.{h}.{w}.{cin}.{cout}")
    x = to_dev(case["x"])
    wt = to_dev(vg.pack_conv3x3(case["w"]))
    b = to_dev(case["b"])
    gamma = to_dev((1.0 + 0.25 * stream_normal(31, "rmsf.gamma", (cout,))).astype(np.float32))
    y_ref = vg.conv3x3_nhwc(x, wt, b, **kw)
    ref = vg.rmsnorm_silu(y_ref.reshape(-1, cout), gamma, silu=True)
    y = sentinel_like(tuple(y_ref.shape), torch.float32) if with_y else None
    got = vg.conv3x3_nhwc_rms(x, wt, gamma, b, y=y, silu=True, **kw)
    vg.sync_status()
    assert torch.equal(got.reshape(-1, cout), ref)
    if with_y:
        assert torch.equal(y, y_ref)

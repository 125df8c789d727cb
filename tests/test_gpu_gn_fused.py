"""GroupNorm with its statistics taken in the producing conv's epilogue
(vae_conv3x3_nhwc_gn + vae_groupnorm_apply), through the C ABI.

- The conv output is bit-identical to the plain conv's (vae_conv3x3_nhwc):
  the epilogue computes the same values and only also reduces them.
- The normalised f16 output matches the oracle's GroupNorm of the oracle's
  conv (f64) within the conv tolerance composed with one f16 rounding.
- The statistics match a float64 evaluation of the GroupNorm definition on the
  conv's own f32 output, and the fused pipeline matches the standalone
  GroupNorm kernels on that output to within one f16 ulp.
Group widths 4, 8, 16 and 32 channels (one, two and four groups per
16-channel chunk, and groups spanning two chunks), ragged rows, rows shorter
than a tile, the upsample fold, reflect padding, the downsample, residuals
(separate and in place), SiLU and two images.
"""
import numpy as np
import pytest

import oracle
import implicit_gemm_convolution_vae_gb300 as vg
from gpu_common import CONV_TOL, rel_err, to_dev, torch_mod
from vae_inputs import conv_case, stream_normal

pytestmark = pytest.mark.gpu

CASES = [
    # n, h, w, cin, cout, groups, flags
    (1, 16, 256, 64, 128, 32, ""),          # 4-channel groups, TMA epilogue
    (1, 9, 200, 128, 256, 32, "res"),       # 8-channel groups, ragged last tile, separate residual
    (1, 6, 130, 64, 512, 32, "inplace"),    # 16-channel groups, in-place residual, 2 N tiles
    (1, 5, 128, 64, 1024, 32, ""),          # 32-channel groups spanning two chunks
    (2, 12, 40, 32, 128, 32, "silu"),       # rows shorter than a tile (multi-row tiles), two images
    (1, 8, 70, 64, 128, 32, "up"),          # the upsample fold (parity classes)
    (1, 7, 150, 64, 256, 32, "reflect"),    # reflect padding (halo stages + fixer warp)
    (1, 20, 300, 64, 128, 32, "down"),      # the encoder's downsample (gather path)
    (1, 4, 160, 32, 64, 1, ""),             # one group of all 64 channels
]


def _flags(f):
    return dict(upsample="up" in f, reflect="reflect" in f, down="down" in f, silu="silu" in f)


def _oracle_conv(case, f, res):
    outs = []
    for i in range(case["x"].shape[0]):
        xc = np.moveaxis(case["x"][i].astype(np.float64), -1, 0)
        if "down" in f:
            y = oracle.conv2d_down(xc, case["w"], case["b"], pad="zero")
        else:
            y = oracle.conv2d(xc, case["w"], case["b"], upsample="up" in f,
                              pad="reflect" if "reflect" in f else "zero")
        if res is not None:
            y = y + np.moveaxis(res[i], -1, 0)
        if "silu" in f:
            y = oracle.silu(y)
        outs.append(y)
    return np.stack(outs)  # [n][c][H][W]


@pytest.mark.parametrize("n,h,w,cin,cout,groups,f", CASES)
def test_fused_groupnorm_statistics(n, h, w, cin, cout, groups, f):
    torch = torch_mod()
    case = conv_case(seed=21, n=n, h=h, w=w, cin=cin, cout=cout, name=f"gnf.{n}.{h}.{w}.{cin}.{cout}.{f}")
    H, W = (2 * h, 2 * w) if "up" in f else ((h // 2, w // 2) if "down" in f else (h, w))
    res = stream_normal(21, f"gnf.res.{f}", (n, H, W, cout)) if ("res" in f or "inplace" in f) else None
    x = to_dev(case["x"])
    wt = to_dev(vg.pack_conv3x3(case["w"]))
    b = to_dev(case["b"])
    kw = _flags(f)
    # the plain conv, for bit-identity of the output
    plain = vg.conv3x3_nhwc(x, wt, b, residual=None if res is None else to_dev(res), **kw)
    if "inplace" in f:
        y = to_dev(res.copy())
        y, stats = vg.conv3x3_nhwc_gn(x, wt, groups, b, residual=y, out=y, **kw)
    else:
        y, stats = vg.conv3x3_nhwc_gn(x, wt, groups, b, residual=None if res is None else to_dev(res), **kw)
    gamma = to_dev((1.0 + 0.25 * stream_normal(21, "gnf.gamma", (cout,))).astype(np.float32))
    beta = to_dev((0.1 * stream_normal(21, "gnf.beta", (cout,))).astype(np.float32))
    yn = vg.groupnorm_apply(y.reshape(n, H * W, cout), groups, stats, gamma, beta, silu=True)
    ref_gpu_gn = vg.groupnorm_silu(y.reshape(n, H * W, cout), groups, gamma, beta, silu=True)
    vg.sync_status()
    assert torch.equal(y, plain)

    # statistics against a float64 evaluation of the definition on the conv's own output
    yy = y.double().cpu().numpy().reshape(n, H * W, groups, cout // groups)
    mean = yy.mean(axis=(1, 3))
    var = ((yy - mean[:, None, :, None]) ** 2).mean(axis=(1, 3))
    st = stats.double().cpu().numpy()
    assert np.abs(st[..., 0] - mean).max() <= 1e-5 * (np.abs(mean) + np.sqrt(var)).max()
    np.testing.assert_allclose(st[..., 1], 1.0 / np.sqrt(var + 1e-6), rtol=1e-4)

    # the fused pipeline and the standalone GroupNorm agree to within one f16 ulp
    a = yn.float().cpu().numpy()
    bb = ref_gpu_gn.float().cpu().numpy()
    assert np.abs(a - bb).max() <= 2.0 ** -10 * max(1.0, np.abs(bb).max())

    # against the oracle: GroupNorm(+SiLU) of the oracle's conv (image 0)
    g_np = gamma.cpu().numpy()
    ref = oracle.silu(oracle.group_norm(_oracle_conv(case, f, res)[0], groups, g_np, beta.cpu().numpy()))
    got = np.moveaxis(a[0].reshape(H, W, cout), -1, 0)
    # the conv's error (<= 2e-3 of max|y|, in the value and in the group mean) is scaled by
    # rstd * |gamma| in the normalised output; plus one f16 rounding of that output
    tol = 2 * CONV_TOL * float(np.abs(yy[0]).max() * st[0, :, 1].max() * np.abs(g_np).max()) + \
        2.0 ** -10 * np.abs(ref).max()
    assert np.abs(got - ref).max() <= tol


def test_gn_conv_rejects_unsupported_groups_and_flags():
    torch = torch_mod()
    x = torch.zeros((1, 4, 4, 16), dtype=torch.float16, device="cuda")
    w = torch.zeros((48, 3, 3, 16), dtype=torch.float16, device="cuda")
    with pytest.raises(vg.VaeError) as e:  # 48 / 32 groups is not a whole channel count
        vg.conv3x3_nhwc_gn(x, w, 32)
    assert e.value.code == -2
    with pytest.raises(vg.VaeError):       # 48 / 4 = 12 channels per group: not 4, 8 or a multiple of 16
        vg.conv3x3_nhwc_gn(x, w, 4)
    L = vg.lib()
    assert L.vae_conv3x3_nhwc_gn(x.data_ptr(), 1, 4, 4, 16, w.data_ptr(), None, None, x.data_ptr(), 48, 1.0,
                                 vg.OUT_F16, 3, 1e-6, x.data_ptr(), x.data_ptr(), 1 << 20, None) == -1

"""GPU parity of the 3x3x3 causal conv (through the C ABI) against the oracle.

Element by element: one and several frames, two volumes per batch, rows of
fewer and more than 128 pixels (per-tap tiles and three-tap halo stages, a
ragged last tile), 16-channel remainders, every combination of the spatial
and temporal 2x with zero and replicate padding, and the epilogue variants.
Outputs start as NaN so an unwritten element fails.
"""
import numpy as np
import pytest

import oracle
import implicit_gemm_convolution_vae_gb300 as vg
from gpu_common import CONV_TOL, rel_err, sentinel_like, to_dev, torch_mod
from vae_inputs import f16_normal, stream_normal

pytestmark = pytest.mark.gpu


def _case(name, n, F, h, w, cin, cout):
    x = f16_normal(30, f"c3d.{name}.x", (n, F, h, w, cin), 1.0)
    wt = f16_normal(30, f"c3d.{name}.w", (cout, cin, 3, 3, 3), (1.0 / (27 * cin)) ** 0.5)
    b = (stream_normal(30, f"c3d.{name}.b", (cout,)) * 0.1).astype(np.float32)
    return x, wt, b


def _run(x, wt, b, up, t_up, rep, silu=False, out_f16=False, residual=None):
    torch = torch_mod()
    n, F, h, w, _ = x.shape
    cout = wt.shape[0]
    Fo = 2 * F - 1 if t_up else F
    H, W = (2 * h, 2 * w) if up else (h, w)
    out = sentinel_like((n, Fo, H, W, cout), torch.float16 if out_f16 else torch.float32)
    vg.conv3d_causal_ndhwc(to_dev(x), to_dev(vg.pack_conv3d(wt)), to_dev(b),
                           residual=None if residual is None else to_dev(residual), out=out, upsample=up,
                           t_upsample=t_up, replicate=rep, silu=silu, out_f16=out_f16)
    vg.sync_status()
    return out.float().cpu().numpy()


def _ref(x, wt, b, up, t_up, rep):
    outs = []
    for i in range(x.shape[0]):
        xc = np.moveaxis(x[i].astype(np.float64), -1, 0)  # [cin][F][h][w]
        y = oracle.conv3d_causal(xc, wt, b, upsample=up, t_upsample=t_up, pad="replicate" if rep else "zero")
        outs.append(np.moveaxis(y, 0, -1))
    return np.stack(outs)


SHAPES = [
    # name, n, F, h, w, cin, cout
    ("one_frame", 1, 1, 3, 5, 16, 16),
    ("narrow", 1, 3, 5, 7, 16, 32),
    ("halo", 2, 4, 3, 130, 64, 48),
    ("rem16", 1, 3, 2, 200, 144, 144),
    ("cin80", 1, 2, 6, 40, 80, 16),
]
VARIANTS = [(False, False, False), (True, False, False), (False, True, False), (True, True, False),
            (False, False, True), (True, True, True)]


@pytest.mark.parametrize("name,n,F,h,w,cin,cout", SHAPES)
@pytest.mark.parametrize("up,t_up,rep", VARIANTS)
def test_conv3d_shapes(name, n, F, h, w, cin, cout, up, t_up, rep):
    x, wt, b = _case(name, n, F, h, w, cin, cout)
    got = _run(x, wt, b, up, t_up, rep)
    ref = _ref(x, wt, b, up, t_up, rep)
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= CONV_TOL


@pytest.mark.parametrize("silu,out_f16,with_res", [(True, False, False), (False, True, False), (False, False, True),
                                                   (True, True, True)])
def test_conv3d_epilogue(silu, out_f16, with_res):
    x, wt, b = _case("epi", 1, 3, 4, 136, 32, 32)
    res = stream_normal(31, "c3d.epi.res", (1, 3, 4, 136, 32)) if with_res else None
    got = _run(x, wt, b, False, False, False, silu=silu, out_f16=out_f16, residual=res)
    ref = _ref(x, wt, b, False, False, False)
    if res is not None:
        ref = ref + res
    if silu:
        ref = oracle.silu(ref)
    tol = 2e-3 if out_f16 else CONV_TOL  # f16 output: one more rounding (2^-11 relative)
    assert rel_err(got, ref) <= tol


def test_conv3d_in_place_residual():
    """The residual may be the output itself (the add runs as an L2 reduction)."""
    torch = torch_mod()
    x, wt, b = _case("inplace", 1, 2, 3, 160, 48, 64)
    res = stream_normal(32, "c3d.inplace.res", (1, 2, 3, 160, 64))
    y = to_dev(res.copy())
    vg.conv3d_causal_ndhwc(to_dev(x), to_dev(vg.pack_conv3d(wt)), to_dev(b), residual=y, out=y)
    vg.sync_status()
    ref = _ref(x, wt, b, False, False, False) + res
    assert rel_err(y.cpu().numpy(), ref) <= CONV_TOL

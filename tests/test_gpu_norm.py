"""GPU parity of RMS_norm, GroupNorm and the guarded cast against the oracle."""
import numpy as np
import pytest

import oracle
import implicit_gemm_convolution_vae_gb300 as vg
from gpu_common import NORM_TOL, rel_err, sentinel_like, to_dev, torch_mod
from vae_inputs import rng_for, stream_normal

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m,c", [(1, 4), (7, 16), (1000, 144), (513, 288), (300, 576), (257, 1152),
                                 (100, 4096)])
@pytest.mark.parametrize("silu,with_bias", [(False, False), (True, True)])
def test_rmsnorm(m, c, silu, with_bias):
    torch = torch_mod()
    x = stream_normal(10, f"rms.x.{m}.{c}", (m, c)) * 3.0 + 0.5
    gam = rng_for(10, f"rms.g.{c}").uniform(0.5, 1.5, c).astype(np.float32)
    bia = (rng_for(10, f"rms.b.{c}").standard_normal(c) * 0.2).astype(np.float32) if with_bias else None
    out = sentinel_like((m, c), torch.float16)
    vg.rmsnorm_silu(to_dev(x), to_dev(gam), bias_in=None if bia is None else to_dev(bia), silu=silu, out=out)
    vg.sync_status()
    ref = oracle.rms_norm(x.T, gam, bias_in=bia).T
    if silu:
        ref = oracle.silu(ref)
    got = out.float().cpu().numpy()
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= NORM_TOL


def test_rmsnorm_zero_row():
    torch = torch_mod()
    x = np.zeros((3, 64), np.float32)
    out = vg.rmsnorm_silu(to_dev(x), to_dev(np.ones(64, np.float32)))
    vg.sync_status()
    assert (out.float().cpu().numpy() == 0).all()


@pytest.mark.parametrize("n,hw,c,groups", [(1, 1, 32, 32), (1, 100, 64, 32), (2, 1000, 128, 32),
                                           (1, 16384, 256, 32), (1, 4096, 512, 32), (1, 333, 96, 3),
                                           (1, 50, 4096, 32)])
@pytest.mark.parametrize("silu,with_bias", [(True, False), (False, True)])
def test_groupnorm(n, hw, c, groups, silu, with_bias):
    torch = torch_mod()
    x = stream_normal(11, f"gn.x.{n}.{hw}.{c}", (n, hw, c)) * 2.0 + 3.0
    g = rng_for(11, f"gn.g.{c}")
    gam = g.uniform(0.5, 1.5, c).astype(np.float32)
    bet = (g.standard_normal(c) * 0.1).astype(np.float32)
    bia = (g.standard_normal(c) * 0.3).astype(np.float32) if with_bias else None
    out = sentinel_like((n, hw, c), torch.float16)
    vg.groupnorm_silu(to_dev(x), groups, to_dev(gam), to_dev(bet), eps=1e-6,
                      bias_in=None if bia is None else to_dev(bia), silu=silu, out=out)
    vg.sync_status()
    got = out.float().cpu().numpy()
    assert not np.isnan(got).any()
    for i in range(n):
        ref = oracle.group_norm(x[i].T, groups, gam, bet, 1e-6, bias_in=bia).T
        if silu:
            ref = oracle.silu(ref)
        assert rel_err(got[i], ref) <= NORM_TOL


def test_groupnorm_large_mean_small_spread():
    """Shifted sums keep the variance right when |mean| >> std."""
    torch = torch_mod()
    x = stream_normal(12, "gn.off", (1, 20000, 128)) * 0.01 + 300.0
    gam = np.ones(128, np.float32)
    bet = np.zeros(128, np.float32)
    out = vg.groupnorm_silu(to_dev(x), 32, to_dev(gam), to_dev(bet))
    vg.sync_status()
    ref = oracle.group_norm(x[0].T, 32, gam, bet, 1e-6).T
    assert rel_err(out.float().cpu().numpy()[0], ref) <= 5e-3


@pytest.mark.parametrize("count,c,scale", [(64, 16, 1.0), (1000 * 144, 144, 2.0 ** -8), (333 * 1152, 1152, 1.0)])
def test_cast(count, c, scale):
    torch = torch_mod()
    x = stream_normal(13, f"cast.{count}", (count // c, c)) * 100.0
    b = (stream_normal(13, f"cast.b.{c}", (c,))).astype(np.float32)
    out = vg.cast_f16(to_dev(x), c, bias=to_dev(b), scale=scale)
    vg.sync_status()
    # the kernel's own f32 arithmetic, then one IEEE round to nearest even
    ref = ((x + b) * np.float32(scale)).astype(np.float16)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), ref.view(np.uint16))

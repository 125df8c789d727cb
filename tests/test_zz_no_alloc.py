"""The GroupNorm entry point that allocates nothing (its scratch is a fixed
device array inside the library), for callers that cannot allocate device
memory. Called through the C ABI; its output must match the workspace
entry point's, and the oracle's GroupNorm (+SiLU), on two calls in a row (the
second sees the first call's leftovers in the shared array). This file is
collected last."""
import numpy as np
import pytest

import oracle
import implicit_gemm_convolution_vae_gb300 as vg
from gpu_common import NORM_TOL, rel_err, to_dev, torch_mod
from vae_inputs import rng_for, stream_normal

pytestmark = pytest.mark.gpu


def _case(seed, n, hw, c):
    x = stream_normal(seed, f"noalloc.x.{seed}", (n, hw, c)) * 1.5 + 0.25
    g = rng_for(seed, f"noalloc.g.{seed}")
    return (x, g.uniform(0.5, 1.5, c).astype(np.float32), (g.standard_normal(c) * 0.1).astype(np.float32),
            (g.standard_normal(c) * 0.2).astype(np.float32))


def test_static_groupnorm_matches_workspace_groupnorm_twice():
    torch = torch_mod()
    L = vg.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for seed, (n, hw, c, silu) in enumerate([(1, 16384, 256, 1), (2, 3000, 128, 0)]):
        x, gam, bet, bia = _case(seed, n, hw, c)
        xd, gd, bd, bid = to_dev(x), to_dev(gam), to_dev(bet), to_dev(bia)
        got = torch.full((n, hw, c), float("nan"), dtype=torch.float16, device="cuda")
        rc = L.vae_groupnorm_silu_static(xd.data_ptr(), n, hw, c, 32, 1e-6, bid.data_ptr(), gd.data_ptr(),
                                         bd.data_ptr(), silu, 1.0, got.data_ptr(), stream)
        assert rc == 0, vg.last_error()
        ref = vg.groupnorm_silu(xd, 32, gd, bd, eps=1e-6, bias_in=bid, silu=bool(silu))
        vg.sync_status()
        g, r = got.float().cpu().numpy(), ref.float().cpu().numpy()
        assert not np.isnan(g).any()
        assert rel_err(g, r) <= NORM_TOL
        # the oracle: GroupNorm(32) of x + bias over each image's pixels, then SiLU
        for i in range(n):
            o = oracle.group_norm(x[i].T, 32, gam, bet, eps=1e-6, bias_in=bia)
            if silu:
                o = oracle.silu(o)
            assert rel_err(g[i], o.T) <= NORM_TOL


def test_static_groupnorm_rejects_calls_beyond_its_scratch():
    torch = torch_mod()
    L = vg.lib()
    x = torch.zeros((1, 4096, 1024), device="cuda")
    y = torch.zeros((1, 4096, 1024), dtype=torch.float16, device="cuda")
    g = torch.ones(1024, device="cuda")
    rc = L.vae_groupnorm_silu_static(x.data_ptr(), 1, 4096, 1024, 512, 1e-6, None, g.data_ptr(), g.data_ptr(), 0,
                                     1.0, y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == -4
    assert "scratch" in vg.last_error()

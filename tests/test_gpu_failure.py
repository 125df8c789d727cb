"""Failure detection on the GPU without a fault: a bounded device wait that
nothing completes runs out, the kernel records the timeout and returns, the
host reads VAE_ERR_DEVICE_TIMEOUT, and the context stays usable."""
import numpy as np
import pytest

import implicit_gemm_convolution_vae_gb300 as vg
from gpu_common import to_dev, torch_mod
from vae_inputs import conv_case

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    torch_mod()
    rc = vg.selftest_wait_timeout(2_000_000)  # 2 ms
    assert rc == -6, vg.last_error()
    assert "bounded device wait" in vg.last_error()
    # the status word was cleared and the device still computes
    assert vg.sync_status() == 0
    case = conv_case(seed=0, h=8, w=8, cin=16, cout=16)
    y = vg.conv3x3_nhwc(to_dev(case["x"]), to_dev(vg.pack_conv3x3(case["w"])), to_dev(case["b"]))
    vg.sync_status()
    assert np.isfinite(y.cpu().numpy()).all()


def test_invalid_arguments_enqueue_nothing():
    torch = torch_mod()
    x = torch.zeros((1, 4, 4, 15), dtype=torch.float16, device="cuda")
    w = torch.zeros((16, 3, 3, 15), dtype=torch.float16, device="cuda")
    with pytest.raises(vg.VaeError) as e:
        vg.conv3x3_nhwc(x, w)
    assert e.value.code == -2
    out = torch.full((4, 64), 7.0, dtype=torch.float16, device="cuda")
    with pytest.raises(vg.VaeError):
        vg.rmsnorm_silu(torch.zeros((4, 62), device="cuda"), torch.ones(62, device="cuda"), out=out[:, :62].contiguous())
    assert (out.float() == 7.0).all().item()

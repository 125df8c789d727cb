"""The benchmarked workload itself against the oracle: the Qwen-style decoder
(widths 1152, 576, 288, 144; three ResNets per block; mid attention over all
16384 latent tokens) decoding a [16, 128, 128] latent to a whole 1024^2 RGB
frame, checked at u8 PSNR >= 60 dB with fewer than 5 % saturated pixels.

The float64 oracle does ~14.7 TFLOP here (about two minutes on 16 host
cores), so this file is collected after the other GPU tests. It prints the
PSNR, the raw f32 max|d|/max|ref| and the oracle's time and thread count; with
VAE_PARITY_LOG=<path> it also appends them to that file as one JSON line.
"""
import os
import time

import numpy as np
import pytest

import oracle
import implicit_gemm_convolution_vae_gb300 as vg
from gpu_common import report_parity, to_dev, torch_mod
from vae_inputs import latent_channel_stats, qwen_decoder

pytestmark = pytest.mark.gpu

PSNR_MIN = 60.0


def _threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    return os.cpu_count()


def test_qwen_decoder_whole_frame_1024_matches_oracle():
    torch = torch_mod()
    dec = qwen_decoder(seed=0)
    z = latent_channel_stats(0, 16, 128, 128)
    D = vg.Decoder(dec)
    got = D.decode(to_dev(z))
    vg.sync_status()
    got = got.cpu().numpy()
    assert got.shape == (3, 1024, 1024)
    assert np.isfinite(got).all()
    t0 = time.perf_counter()
    ref = oracle.decode_rms(dec, z)
    oracle_s = time.perf_counter() - t0
    rec = report_parity("qwen_decoder_1024_whole_frame", got, ref, oracle_s=round(oracle_s, 2),
                        oracle_threads=_threads(), host_cores=os.cpu_count())
    assert rec["saturated_fraction"] < 0.05
    assert rec["psnr_u8_db"] >= PSNR_MIN, rec

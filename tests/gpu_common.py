"""Helpers of the GPU parity tests: device transfer, tolerances, sentinels,
and the record of whole-decoder parity figures."""
import json
import os

import numpy as np

# Per conv, from the hot path's stated target: max|d| / max|ref| <= 2e-3,
# the oracle run on the same f16-rounded inputs and weights.
CONV_TOL = 2e-3
# f16 outputs of the norms: one rounding to f16 (relative 2^-11 ~ 4.9e-4 of
# each element) plus f32 statistics; bounded well inside 1e-3 of max|ref|.
NORM_TOL = 1e-3


def torch_mod():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("these tests need a CUDA device (GB300, sm_103a)")
    return torch


def to_dev(a, dtype=None):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def sentinel_like(shape, dtype):
    """A CUDA tensor filled with NaN, so unwritten outputs are caught."""
    torch = torch_mod()
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


def u8(y):
    """RGB in about [-1, 1] -> u8 levels: round(clamp((y+1)/2, 0, 1) * 255)."""
    return np.round(np.clip((np.asarray(y, np.float64) + 1.0) / 2.0, 0.0, 1.0) * 255.0)


def psnr_u8(got, ref):
    mse = float(np.mean((u8(got) - u8(ref)) ** 2))
    return float("inf") if mse == 0 else 10.0 * np.log10(255.0 ** 2 / mse)


def saturated_fraction(ref):
    r = np.asarray(ref)
    return float(np.mean((r <= -1.0) | (r >= 1.0)))


def report_parity(case, got, ref, **extra):
    """Prints one JSON line with a decode's u8 PSNR, raw max|d|/max|ref| and
    saturated fraction (and appends it to $VAE_PARITY_LOG when that is set);
    returns the record."""
    rec = {"case": case, "psnr_u8_db": round(psnr_u8(got, ref), 3), "max_rel_err_f32": rel_err(got, ref),
           "saturated_fraction": saturated_fraction(ref), **extra}
    print(json.dumps(rec))
    log = os.environ.get("VAE_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps(rec) + "\n")
    return rec

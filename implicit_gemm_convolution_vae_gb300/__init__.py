"""Python binding of ``libvae_igemm.so``, the sm_103a image-VAE decoder hot path.

Argument marshalling only: every step of the computation runs in the CUDA
library through its C ABI (``include/vae_igemm.h``); PyTorch provides the
device memory and the stream. There is no CPU fallback: if the library is
not built, or no sm_103a device is present, calls raise ``VaeError``.

Layouts follow the C ABI: activations NHWC, conv weights f16
``[cout][3][3][cin]`` (3x3) or ``[cout][cin]`` (1x1), streams f32, conv
inputs f16.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from .build import LIB_PATH, build  # noqa: F401  (build is re-exported)

__all__ = [
    "VaeError", "lib", "version", "last_error", "sync_status", "set_wait_timeout_ns",
    "selftest_wait_timeout", "conv3x3_nhwc", "conv3x3_nhwc_rms", "conv3x3_nhwc_gn", "conv3x3_gn_workspace_bytes", "groupnorm_apply",
    "conv1x1", "rmsnorm_silu", "groupnorm_silu",
    "groupnorm_workspace_bytes", "cast_f16", "mid_attention", "mid_attention_workspace_bytes",
    "Decoder", "DecodeGraph", "pack_conv3x3", "pack_conv1x1",
    "UPSAMPLE2X", "PAD_REPLICATE", "PAD_REFLECT", "DOWNSAMPLE2X", "EPI_SILU", "OUT_F16", "FAMILY_GN", "FAMILY_RMS",
    "NORM_GROUP", "NORM_RMS",
]

UPSAMPLE2X, PAD_REPLICATE, EPI_SILU, OUT_F16, UPSAMPLE_T2X, UPSAMPLE2X_SUBPIXEL = 1, 2, 16, 32, 64, 128
PAD_REFLECT, DOWNSAMPLE2X = 256, 512
FAMILY_GN, FAMILY_RMS = 0, 1
NORM_GROUP, NORM_RMS = 0, 1

STATUS_NAMES = {0: "VAE_OK", -1: "VAE_ERR_ARG", -2: "VAE_ERR_SHAPE", -3: "VAE_ERR_ALIGN",
                -4: "VAE_ERR_NOMEM", -5: "VAE_ERR_CUDA", -6: "VAE_ERR_DEVICE_TIMEOUT",
                -7: "VAE_ERR_UNSUPPORTED"}


class VaeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_LIB = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

# Every exported function with its argument types (restype int unless noted).
SIGNATURES = {
    "vae_version": ([], ctypes.c_char_p),
    "vae_last_error": ([], ctypes.c_char_p),
    "vae_sync_status": ([_P], _I),
    "vae_set_wait_timeout_ns": ([ctypes.c_ulonglong], _I),
    "vae_selftest_wait_timeout": ([ctypes.c_ulonglong, _P], _I),
    "vae_conv3x3_nhwc": ([_P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _F, ctypes.c_uint, _P], _I),
    "vae_conv3d_causal_ndhwc": ([_P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _I, _F, ctypes.c_uint, _P], _I),
    "vae_pack_subpixel_weights": ([_P, _I, _I, _P, _P], _I),
    "vae_conv1x1": ([_P, _I, _I, _P, _P, _P, _P, _I, _F, ctypes.c_uint, _P], _I),
    "vae_conv3x3_nhwc_rms": ([_P, _I, _I, _I, _I, _P, _P, _P, _I, _F, ctypes.c_uint, _P, _I, _P, _P], _I),
    "vae_conv3x3_gn_workspace_bytes": ([_I, _I, _I, _I, _I, ctypes.c_uint], _SZ),
    "vae_conv3x3_nhwc_gn": ([_P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _F, ctypes.c_uint, _I, _F, _P, _P, _SZ, _P], _I),
    "vae_groupnorm_apply": ([_P, _I, _I, _I, _I, _P, _P, _P, _I, _F, _P, _P], _I),
    "vae_rmsnorm_silu": ([_P, _I, _I, _P, _P, _I, _F, _P, _P], _I),
    "vae_groupnorm_workspace_bytes": ([_I, _I, _I, _I], _SZ),
    "vae_groupnorm_silu": ([_P, _I, _I, _I, _I, _F, _P, _P, _P, _I, _F, _P, _P, _SZ, _P], _I),
    "vae_groupnorm_silu_static": ([_P, _I, _I, _I, _I, _F, _P, _P, _P, _I, _F, _P, _P], _I),
    "vae_cast_f16": ([_P, _SZ, _I, _P, _F, _P, _P], _I),
    "vae_mid_attention_workspace_bytes": ([_I, _I, _I], _SZ),
    "vae_mid_attention": ([_P, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], _I),
    "vae_decoder_create": ([_P, ctypes.POINTER(_P)], _I),
    "vae_decoder_destroy": ([_P], _I),
    "vae_decode_workspace": ([_P, _I, _I, _P, ctypes.POINTER(_SZ)], _I),
    "vae_decode": ([_P, _P, _I, _I, _P, _P, _P, _SZ, _P], _I),
    "vae_decode_host": ([_P, _P, _I, _I, _P, _P, _P, _SZ, _P], _I),
    "vae_decode_profile": ([_P, _P, _I, ctypes.POINTER(_I)], _I),
    "vae_decode_graph_create": ([_P, _P, _I, _I, _P, _P, _P, _SZ, _P, ctypes.POINTER(_P)], _I),
    "vae_decode_graph_launch": ([_P, _P], _I),
    "vae_decode_graph_destroy": ([_P], _I),
}


def lib():
    """The loaded library (raises if it was not built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise VaeError(-5, f"{os.path.basename(LIB_PATH)} is not built; run "
                               "`python -m implicit_gemm_convolution_vae_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(L, name, None)
            if fn is None:
                continue
            fn.argtypes = args
            fn.restype = res
        _LIB = L
    return _LIB


def version() -> str:
    return lib().vae_version().decode()


def last_error() -> str:
    return lib().vae_last_error().decode()


def _check(rc: int):
    if rc != 0:
        raise VaeError(rc, last_error())


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t, dtype, name, ndim=None):
    import torch
    if t is None:
        return
    if not t.is_cuda:
        raise VaeError(-1, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise VaeError(-1, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise VaeError(-1, f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise VaeError(-2, f"{name} must have {ndim} dims, got {t.dim()}")


def sync_status(stream=None) -> int:
    """Synchronise the stream; raises VaeError(VAE_ERR_DEVICE_TIMEOUT) if a device wait ran out."""
    rc = lib().vae_sync_status(_stream(stream))
    _check(rc)
    return rc


def set_wait_timeout_ns(ns: int) -> None:
    _check(lib().vae_set_wait_timeout_ns(int(ns)))


def selftest_wait_timeout(timeout_ns: int = 1_000_000, stream=None) -> int:
    """Runs the bounded-wait self test; returns its status code (expected -6)."""
    return lib().vae_selftest_wait_timeout(int(timeout_ns), _stream(stream))


def pack_subpixel_weights(w, stream=None):
    """f16 [cout][3][3][cin] -> the up conv's sub-pixel weights f16 [cout][16][cin] (device)."""
    import torch
    _need(w, torch.float16, "w", 4)
    cout, _, _, cin = w.shape
    ws = torch.empty((cout, 16, cin), dtype=torch.float16, device=w.device)
    _check(lib().vae_pack_subpixel_weights(_ptr(w), cout, cin, _ptr(ws), _stream(stream)))
    return ws


def conv3x3_nhwc(x, w, bias=None, residual=None, out=None, oscale: float = 1.0, upsample: bool = False,
                 replicate: bool = False, silu: bool = False, out_f16: bool = False, subpixel: bool = False,
                 reflect: bool = False, down: bool = False, stream=None):
    """3x3 implicit-GEMM conv. x f16 [n][h][w][cin]; w f16 [cout][3][3][cin], or with
    ``subpixel`` (an up conv) the summed weights [cout][16][cin] of pack_subpixel_weights.
    ``reflect``: mirror padding; ``down``: the encoder's far-side-padded stride-2
    downsample (output [n][h//2][w//2][cout])."""
    import torch
    _need(x, torch.float16, "x", 4)
    _need(w, torch.float16, "w", 3 if subpixel else 4)
    _need(bias, torch.float32, "bias", 1)
    n, h, wd, cin = x.shape
    cout = w.shape[0]
    if tuple(w.shape[1:]) != ((16, cin) if subpixel else (3, 3, cin)):
        raise VaeError(-2, f"w has the wrong shape {tuple(w.shape)}")
    H, W = (2 * h, 2 * wd) if upsample else ((h // 2, wd // 2) if down else (h, wd))
    odt = torch.float16 if out_f16 else torch.float32
    if out is None:
        out = torch.empty((n, H, W, cout), dtype=odt, device=x.device)
    _need(out, odt, "out")
    _need(residual, torch.float32, "residual")
    for t, nm in ((out, "out"), (residual, "residual")):
        if t is not None and t.numel() != n * H * W * cout:
            raise VaeError(-2, f"{nm} must hold [n][{H}][{W}][{cout}], got {tuple(t.shape)}")
    flags = (UPSAMPLE2X if upsample else 0) | (PAD_REPLICATE if replicate else 0) | \
            (EPI_SILU if silu else 0) | (OUT_F16 if out_f16 else 0) | (UPSAMPLE2X_SUBPIXEL if subpixel else 0) | \
            (PAD_REFLECT if reflect else 0) | (DOWNSAMPLE2X if down else 0)
    _check(lib().vae_conv3x3_nhwc(_ptr(x), n, h, wd, cin, _ptr(w), _ptr(bias), _ptr(residual), _ptr(out),
                                  cout, float(oscale), flags, _stream(stream)))
    return out


def conv3x3_nhwc_gn(x, w, groups: int, bias=None, residual=None, out=None, oscale: float = 1.0,
                    upsample: bool = False, replicate: bool = False, reflect: bool = False, down: bool = False,
                    silu: bool = False, eps: float = 1e-6, workspace=None, stream=None):
    """3x3 conv (f32 output) that also returns the GroupNorm statistics of its
    output: (y [n][H][W][cout] f32, stats [n][groups][2] f32 = (mean, rstd))."""
    import torch
    _need(x, torch.float16, "x", 4)
    _need(w, torch.float16, "w", 4)
    _need(bias, torch.float32, "bias", 1)
    n, h, wd, cin = x.shape
    cout = w.shape[0]
    if tuple(w.shape[1:]) != (3, 3, cin):
        raise VaeError(-2, f"w has the wrong shape {tuple(w.shape)}")
    H, W = (2 * h, 2 * wd) if upsample else ((h // 2, wd // 2) if down else (h, wd))
    if out is None:
        out = torch.empty((n, H, W, cout), dtype=torch.float32, device=x.device)
    _need(out, torch.float32, "out")
    _need(residual, torch.float32, "residual")
    for t, nm in ((out, "out"), (residual, "residual")):
        if t is not None and t.numel() != n * H * W * cout:
            raise VaeError(-2, f"{nm} must hold [n][{H}][{W}][{cout}], got {tuple(t.shape)}")
    flags = (UPSAMPLE2X if upsample else 0) | (PAD_REPLICATE if replicate else 0) | (EPI_SILU if silu else 0) | \
            (PAD_REFLECT if reflect else 0) | (DOWNSAMPLE2X if down else 0)
    need = conv3x3_gn_workspace_bytes(n, h, wd, cout, groups, flags)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    stats = torch.empty((n, groups, 2), dtype=torch.float32, device=x.device)
    _check(lib().vae_conv3x3_nhwc_gn(_ptr(x), n, h, wd, cin, _ptr(w), _ptr(bias), _ptr(residual), _ptr(out), cout,
                                     float(oscale), flags, int(groups), float(eps), _ptr(stats), _ptr(workspace),
                                     workspace.numel(), _stream(stream)))
    return out, stats


def conv3x3_nhwc_rms(x, w, gamma, bias=None, out=None, y=None, oscale: float = 1.0, silu: bool = True,
                     replicate: bool = False, reflect: bool = False, down: bool = False, stream=None):
    """3x3 conv with RMS_norm(+SiLU) of each output pixel in its epilogue: f16
    [n][H][W][cout] (and, if ``y`` is given, the f32 conv output into it)."""
    import torch
    _need(x, torch.float16, "x", 4)
    _need(w, torch.float16, "w", 4)
    _need(gamma, torch.float32, "gamma", 1)
    _need(bias, torch.float32, "bias", 1)
    n, h, wd, cin = x.shape
    cout = w.shape[0]
    if tuple(w.shape[1:]) != (3, 3, cin):
        raise VaeError(-2, f"w has the wrong shape {tuple(w.shape)}")
    H, W = (h // 2, wd // 2) if down else (h, wd)
    if out is None:
        out = torch.empty((n, H, W, cout), dtype=torch.float16, device=x.device)
    _need(out, torch.float16, "out")
    _need(y, torch.float32, "y")
    for t, nm in ((out, "out"), (y, "y")):
        if t is not None and t.numel() != n * H * W * cout:
            raise VaeError(-2, f"{nm} must hold [n][{H}][{W}][{cout}], got {tuple(t.shape)}")
    flags = (PAD_REPLICATE if replicate else 0) | (PAD_REFLECT if reflect else 0) | (DOWNSAMPLE2X if down else 0)
    _check(lib().vae_conv3x3_nhwc_rms(_ptr(x), n, h, wd, cin, _ptr(w), _ptr(bias), _ptr(y), cout, float(oscale),
                                      flags, _ptr(gamma), 1 if silu else 0, _ptr(out), _stream(stream)))
    return out


def conv3x3_gn_workspace_bytes(n: int, h: int, w: int, cout: int, groups: int, flags: int = 0) -> int:
    return int(lib().vae_conv3x3_gn_workspace_bytes(n, h, w, cout, groups, flags))


def groupnorm_apply(x, groups: int, stats, gamma, beta, silu: bool = False, out_scale: float = 1.0, out=None,
                    stream=None):
    """GroupNorm from precomputed statistics. x f32 [n][hw][c] -> f16 [n][hw][c]."""
    import torch
    _need(x, torch.float32, "x", 3)
    _need(stats, torch.float32, "stats")
    _need(gamma, torch.float32, "gamma", 1)
    _need(beta, torch.float32, "beta", 1)
    n, hw, c = x.shape
    if stats.numel() != n * groups * 2:
        raise VaeError(-2, f"stats must hold [n][{groups}][2], got {tuple(stats.shape)}")
    if out is None:
        out = torch.empty((n, hw, c), dtype=torch.float16, device=x.device)
    _need(out, torch.float16, "out")
    _check(lib().vae_groupnorm_apply(_ptr(x), n, hw, c, groups, _ptr(stats), _ptr(gamma), _ptr(beta),
                                     1 if silu else 0, float(out_scale), _ptr(out), _stream(stream)))
    return out


def conv3d_causal_ndhwc(x, w, bias=None, residual=None, out=None, oscale: float = 1.0, upsample: bool = False,
                        t_upsample: bool = False, replicate: bool = False, silu: bool = False,
                        out_f16: bool = False, stream=None):
    """3x3x3 causal conv over frames. x f16 [n][f][h][w][cin]; w f16 [cout][3][3][3][cin]."""
    import torch
    _need(x, torch.float16, "x", 5)
    _need(w, torch.float16, "w", 5)
    _need(bias, torch.float32, "bias", 1)
    n, f, h, wd, cin = x.shape
    cout = w.shape[0]
    if tuple(w.shape[1:]) != (3, 3, 3, cin):
        raise VaeError(-2, f"w must be [cout][3][3][3][{cin}], got {tuple(w.shape)}")
    F = 2 * f - 1 if t_upsample else f
    H, W = (2 * h, 2 * wd) if upsample else (h, wd)
    odt = torch.float16 if out_f16 else torch.float32
    if out is None:
        out = torch.empty((n, F, H, W, cout), dtype=odt, device=x.device)
    _need(out, odt, "out")
    _need(residual, torch.float32, "residual")
    flags = (UPSAMPLE2X if upsample else 0) | (UPSAMPLE_T2X if t_upsample else 0) | \
            (PAD_REPLICATE if replicate else 0) | (EPI_SILU if silu else 0) | (OUT_F16 if out_f16 else 0)
    _check(lib().vae_conv3d_causal_ndhwc(_ptr(x), n, f, h, wd, cin, _ptr(w), _ptr(bias), _ptr(residual), _ptr(out),
                                         cout, float(oscale), flags, _stream(stream)))
    return out


def conv1x1(x, w, bias=None, residual=None, out=None, oscale: float = 1.0, silu: bool = False,
            out_f16: bool = False, stream=None):
    """1x1 conv (GEMM). x f16 [m][cin]; w f16 [cout][cin]."""
    import torch
    _need(x, torch.float16, "x", 2)
    _need(w, torch.float16, "w", 2)
    _need(bias, torch.float32, "bias", 1)
    m, cin = x.shape
    cout = w.shape[0]
    odt = torch.float16 if out_f16 else torch.float32
    if out is None:
        out = torch.empty((m, cout), dtype=odt, device=x.device)
    _need(out, odt, "out")
    _need(residual, torch.float32, "residual")
    flags = (EPI_SILU if silu else 0) | (OUT_F16 if out_f16 else 0)
    _check(lib().vae_conv1x1(_ptr(x), m, cin, _ptr(w), _ptr(bias), _ptr(residual), _ptr(out), cout,
                             float(oscale), flags, _stream(stream)))
    return out


def rmsnorm_silu(x, gamma, bias_in=None, silu: bool = False, out_scale: float = 1.0, out=None, stream=None):
    """Per-pixel RMS_norm. x f32 [m][c] -> f16 [m][c]."""
    import torch
    _need(x, torch.float32, "x", 2)
    _need(gamma, torch.float32, "gamma", 1)
    _need(bias_in, torch.float32, "bias_in", 1)
    m, c = x.shape
    if out is None:
        out = torch.empty((m, c), dtype=torch.float16, device=x.device)
    _need(out, torch.float16, "out")
    _check(lib().vae_rmsnorm_silu(_ptr(x), m, c, _ptr(bias_in), _ptr(gamma), int(silu), float(out_scale),
                                  _ptr(out), _stream(stream)))
    return out


def groupnorm_workspace_bytes(n: int, hw: int, c: int, groups: int) -> int:
    return int(lib().vae_groupnorm_workspace_bytes(n, hw, c, groups))


def groupnorm_silu(x, groups: int, gamma, beta, eps: float = 1e-6, bias_in=None, silu: bool = False,
                   out_scale: float = 1.0, out=None, workspace=None, stream=None):
    """GroupNorm. x f32 [n][hw][c] -> f16 [n][hw][c]."""
    import torch
    _need(x, torch.float32, "x", 3)
    _need(gamma, torch.float32, "gamma", 1)
    _need(beta, torch.float32, "beta", 1)
    _need(bias_in, torch.float32, "bias_in", 1)
    n, hw, c = x.shape
    if out is None:
        out = torch.empty((n, hw, c), dtype=torch.float16, device=x.device)
    _need(out, torch.float16, "out")
    nb = groupnorm_workspace_bytes(n, hw, c, groups)
    if workspace is None:
        workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=x.device)
    _check(lib().vae_groupnorm_silu(_ptr(x), n, hw, c, groups, float(eps), _ptr(bias_in), _ptr(gamma),
                                    _ptr(beta), int(silu), float(out_scale), _ptr(out), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def cast_f16(x, c: int, bias=None, scale: float = 1.0, out=None, stream=None):
    """(x + bias[c]) * scale -> f16, elementwise over a [.., c] f32 tensor."""
    import torch
    _need(x, torch.float32, "x")
    _need(bias, torch.float32, "bias", 1)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    _need(out, torch.float16, "out")
    _check(lib().vae_cast_f16(_ptr(x), x.numel(), c, _ptr(bias), float(scale), _ptr(out), _stream(stream)))
    return out


def mid_attention_workspace_bytes(m: int, c: int, groups: int = 32) -> int:
    return int(lib().vae_mid_attention_workspace_bytes(m, c, groups))


def mid_attention(x, norm_kind: int, gamma, beta, wq, bq, wk, bk, wv, bv, wo, bo, groups: int = 32,
                  eps: float = 1e-6, workspace=None, stream=None):
    """In-place mid self-attention on x f32 [m][c]; w* f16 [c][c], b* f32 [c]."""
    import torch
    _need(x, torch.float32, "x", 2)
    for nm, t in (("wq", wq), ("wk", wk), ("wv", wv), ("wo", wo)):
        _need(t, torch.float16, nm, 2)
    m, c = x.shape
    nb = mid_attention_workspace_bytes(m, c, groups)
    if workspace is None:
        workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=x.device)
    _check(lib().vae_mid_attention(_ptr(x), m, c, int(norm_kind), groups, float(eps), _ptr(gamma), _ptr(beta),
                                   _ptr(wq), _ptr(bq), _ptr(wk), _ptr(bk), _ptr(wv), _ptr(bv), _ptr(wo),
                                   _ptr(bo), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)))
    return x


# ───────────────────────────── weight layouts ─────────────────────────────

def pack_conv3x3(w_oihw: np.ndarray) -> np.ndarray:
    """OIHW [cout][cin][3][3] -> the kernel's [cout][3][3][cin] (a permutation)."""
    return np.ascontiguousarray(np.asarray(w_oihw).transpose(0, 2, 3, 1))


def pack_conv3d(w_oidhw: np.ndarray) -> np.ndarray:
    """OIDHW [cout][cin][3][3][3] -> the kernel's [cout][3][3][3][cin] (a permutation)."""
    return np.ascontiguousarray(np.asarray(w_oidhw).transpose(0, 2, 3, 4, 1))


def pack_conv1x1(w_oihw: np.ndarray) -> np.ndarray:
    """OIHW [cout][cin][1][1] -> [cout][cin]."""
    w = np.asarray(w_oihw)
    return np.ascontiguousarray(w.reshape(w.shape[0], w.shape[1]))


# ───────────────────────────── whole decoder ─────────────────────────────

class _ConvDesc(ctypes.Structure):
    _fields_ = [("w", _P), ("b", _P), ("cout", _I), ("cin", _I), ("k", _I)]


class _NormDesc(ctypes.Structure):
    _fields_ = [("gamma", _P), ("beta", _P)]


class _ResnetDesc(ctypes.Structure):
    _fields_ = [("norm1", _NormDesc), ("conv1", _ConvDesc), ("norm2", _NormDesc), ("conv2", _ConvDesc),
                ("shortcut", _ConvDesc)]


class _AttnDesc(ctypes.Structure):
    _fields_ = [("norm", _NormDesc), ("q", _ConvDesc), ("k", _ConvDesc), ("v", _ConvDesc), ("o", _ConvDesc)]


class _UpDesc(ctypes.Structure):
    _fields_ = [("resnets", ctypes.POINTER(_ResnetDesc)), ("n_resnets", _I), ("up", _ConvDesc),
                ("in_dim", _I), ("out_dim", _I), ("ft", _I)]


class _DecoderDesc(ctypes.Structure):
    _fields_ = [("family", _I), ("latent_channels", _I), ("scaling", _F), ("shift", _F), ("groups", _I),
                ("eps", _F), ("dupup", _I), ("post_quant", _ConvDesc), ("conv_in", _ConvDesc),
                ("mid_res1", _ResnetDesc), ("mid_attn", _AttnDesc), ("mid_res2", _ResnetDesc),
                ("ups", ctypes.POINTER(_UpDesc)), ("n_ups", _I), ("norm_out", _NormDesc),
                ("conv_out", _ConvDesc)]


DECODE_PROFILE = 1
DECODE_NO_FUSION = 2
DECODE_FUSE_NORM = 4
DECODE_SUBPIXEL_UP = 8
DECODE_PROFILE_FULLRES = 16
STAGE_NAMES = {0: "conv3x3", 1: "conv1x1", 2: "norm", 3: "cast", 4: "attention", 5: "layout", 6: "copy"}


class StageRecord(ctypes.Structure):
    _fields_ = [("kind", _I), ("launches", _I), ("h", _I), ("w", _I), ("cin", _I), ("cout", _I),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double), ("ms", ctypes.c_float)]


class DecodeOpts(ctypes.Structure):
    _fields_ = [("band_from", _I), ("nbands", _I), ("band_rows", _I), ("guard_log2", _I),
                ("flags", ctypes.c_uint)]


class Decoder:
    """A decoder handle built from a host description.

    ``desc`` is any object with the attributes of ``vae_decoder_desc``
    (family "gn"/"rms", conv_in, mid_res1, mid_attn, mid_res2, ups,
    norm_out, conv_out, post_quant, latent_channels, scaling, shift, groups,
    eps, dupup), whose convs carry ``w`` (f16 OIHW numpy) and ``b`` (f32) and
    whose norms carry ``gamma`` / ``beta``. The library copies the weights to
    the current device in its own layouts.
    """

    def __init__(self, desc):
        self._keep = []
        d = _DecoderDesc()
        d.family = FAMILY_GN if desc.family == "gn" else FAMILY_RMS
        d.latent_channels = int(desc.latent_channels)
        d.scaling = float(getattr(desc, "scaling", 1.0))
        d.shift = float(getattr(desc, "shift", 0.0))
        d.groups = int(getattr(desc, "groups", 32))
        d.eps = float(getattr(desc, "eps", 1e-6))
        d.dupup = int(bool(getattr(desc, "dupup", False)))
        d.post_quant = self._conv(getattr(desc, "post_quant", None))
        d.conv_in = self._conv(desc.conv_in)
        d.mid_res1 = self._resnet(desc.mid_res1)
        a = desc.mid_attn
        d.mid_attn = _AttnDesc(self._norm(a.norm), self._conv(a.q), self._conv(a.k), self._conv(a.v),
                               self._conv(a.o))
        d.mid_res2 = self._resnet(desc.mid_res2)
        ups = (_UpDesc * len(desc.ups))()
        for i, u in enumerate(desc.ups):
            res = (_ResnetDesc * max(1, len(u.resnets)))()
            for j, r in enumerate(u.resnets):
                res[j] = self._resnet(r)
            self._keep.append(res)
            ups[i] = _UpDesc(ctypes.cast(res, ctypes.POINTER(_ResnetDesc)), len(u.resnets), self._conv(u.up),
                             int(u.in_dim), int(u.out_dim), int(getattr(u, "ft", 1)))
        self._keep.append(ups)
        d.ups = ctypes.cast(ups, ctypes.POINTER(_UpDesc))
        d.n_ups = len(desc.ups)
        d.norm_out = self._norm(desc.norm_out)
        d.conv_out = self._conv(desc.conv_out)
        self.nch = int(desc.conv_out.w.shape[0])
        self.latent_channels = d.latent_channels
        self.n_up = sum(1 for u in desc.ups if u.up is not None)
        h = _P()
        _check(lib().vae_decoder_create(ctypes.byref(d), ctypes.byref(h)))
        self._h = h
        self._keep = None  # the library copied everything

    def _arr(self, a, dtype):
        if a is None:
            return None
        a = np.ascontiguousarray(np.asarray(a, dtype=dtype))
        self._keep.append(a)
        return a.ctypes.data

    def _conv(self, c):
        if c is None:
            return _ConvDesc(None, None, 0, 0, 0)
        w = np.asarray(c.w, dtype=np.float16)
        return _ConvDesc(self._arr(w.view(np.uint16), np.uint16), self._arr(c.b, np.float32),
                         int(w.shape[0]), int(w.shape[1]), int(w.shape[2]))

    def _norm(self, n):
        return _NormDesc(self._arr(n.gamma, np.float32), self._arr(getattr(n, "beta", None), np.float32))

    def _resnet(self, r):
        return _ResnetDesc(self._norm(r.norm1), self._conv(r.conv1), self._norm(r.norm2), self._conv(r.conv2),
                           self._conv(r.shortcut))

    @staticmethod
    def opts(band_from: int = 0, nbands: int = 0, band_rows: int = 0, guard_log2: int = 8,
             profile=False, fuse: Optional[bool] = None, subpixel: bool = False) -> DecodeOpts:
        """profile: False, True (events around every stage) or "fullres" (only around
        the full-resolution ResNet convs). fuse: None (the library's default:
        separate norms), True (a ResNet's second RMS_norm fused into its first
        conv wherever one CTA holds a pixel's channels), False (separate norms)."""
        prof = (DECODE_PROFILE if profile else 0) | (DECODE_PROFILE_FULLRES if profile == "fullres" else 0)
        fz = 0 if fuse is None else (DECODE_FUSE_NORM if fuse else DECODE_NO_FUSION)
        return DecodeOpts(band_from, nbands, band_rows, guard_log2,
                          prof | fz | (DECODE_SUBPIXEL_UP if subpixel else 0))

    def profile(self):
        """Stage records of the most recent profiled decode, as dicts (synchronises)."""
        n = _I()
        _check(lib().vae_decode_profile(self._h, None, 0, ctypes.byref(n)))
        arr = (StageRecord * max(1, n.value))()
        _check(lib().vae_decode_profile(self._h, ctypes.cast(arr, _P), n.value, ctypes.byref(n)))
        return [{"kind": STAGE_NAMES.get(r.kind, r.kind), "launches": r.launches, "h": r.h, "w": r.w,
                 "cin": r.cin, "cout": r.cout, "flops": r.flops, "bytes": r.bytes, "ms": r.ms}
                for r in arr[:n.value]]

    def workspace_bytes(self, h0: int, w0: int, opts: Optional[DecodeOpts] = None) -> int:
        n = _SZ()
        _check(lib().vae_decode_workspace(self._h, h0, w0, ctypes.byref(opts) if opts else None,
                                          ctypes.byref(n)))
        return int(n.value)

    def graph(self, z, out, workspace, opts: Optional[DecodeOpts] = None, stream=None) -> "DecodeGraph":
        """Capture the decode of ``z`` into ``out`` (both CUDA, fixed from now on) as a
        CUDA graph; ``DecodeGraph.launch()`` replays it. Runs one eager decode first."""
        import torch
        _need(z, torch.float32, "z", 3)
        _need(out, torch.float32, "out", 3)
        zc, h0, w0 = z.shape
        g = _P()
        _check(lib().vae_decode_graph_create(self._h, _ptr(z), h0, w0, _ptr(out), ctypes.byref(opts) if opts else None,
                                             _ptr(workspace), workspace.numel(), _stream(stream), ctypes.byref(g)))
        return DecodeGraph(g, (z, out, workspace))

    def decode(self, z, out=None, opts: Optional[DecodeOpts] = None, workspace=None, stream=None):
        """z f32 [zc][h0][w0] (CUDA) -> out f32 [nch][h0<<ups][w0<<ups] (CUDA)."""
        import torch
        _need(z, torch.float32, "z", 3)
        zc, h0, w0 = z.shape
        H, W = h0 << self.n_up, w0 << self.n_up
        if out is None:
            out = torch.empty((self.nch, H, W), dtype=torch.float32, device=z.device)
        _need(out, torch.float32, "out", 3)
        if workspace is None:
            workspace = torch.empty(max(self.workspace_bytes(h0, w0, opts), 16), dtype=torch.uint8,
                                    device=z.device)
        _check(lib().vae_decode(self._h, _ptr(z), h0, w0, _ptr(out), ctypes.byref(opts) if opts else None,
                                _ptr(workspace), workspace.numel(), _stream(stream)))
        return out

    def decode_host(self, z_host: np.ndarray, out_host: np.ndarray, workspace, opts=None, stream=None):
        """End-to-end call with host (ideally pinned) buffers; synchronises the stream."""
        zc, h0, w0 = z_host.shape
        _check(lib().vae_decode_host(self._h, z_host.ctypes.data if isinstance(z_host, np.ndarray)
                                     else z_host.data_ptr(), h0, w0,
                                     out_host.ctypes.data if isinstance(out_host, np.ndarray)
                                     else out_host.data_ptr(),
                                     ctypes.byref(opts) if opts else None, _ptr(workspace), workspace.numel(),
                                     _stream(stream)))
        return out_host

    def close(self):
        if getattr(self, "_h", None):
            lib().vae_decoder_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DecodeGraph:
    """A captured decode (see ``Decoder.graph``); keeps its buffers alive."""

    def __init__(self, handle, keep):
        self._g = handle
        self._keep = keep

    def launch(self, stream=None):
        _check(lib().vae_decode_graph_launch(self._g, _stream(stream)))

    def __del__(self):
        if getattr(self, "_g", None) is not None and _LIB is not None:
            lib().vae_decode_graph_destroy(self._g)
            self._g = None

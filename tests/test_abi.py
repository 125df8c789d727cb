"""The C-ABI library builds, loads and exports every entry point the header
declares, and rejects bad arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import implicit_gemm_convolution_vae_gb300 as vg
from implicit_gemm_convolution_vae_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vae_igemm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int|size_t)\s+(vae_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    build()
    return vg.lib()


def test_header_declares_the_hot_path(L):
    names = declared_functions()
    for required in ("vae_conv3x3_nhwc", "vae_conv1x1", "vae_groupnorm_silu", "vae_rmsnorm_silu",
                     "vae_mid_attention", "vae_decode", "vae_decoder_create", "vae_decoder_destroy",
                     "vae_decode_workspace", "vae_last_error", "vae_sync_status"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    for n in declared_functions():
        assert n in vg.SIGNATURES, f"binding has no signature for {n}"


def test_version(L):
    assert "sm_103a" in vg.version()


FAKE = 1 << 20  # a non-NULL, aligned address never dereferenced: validation fails first


def test_conv_rejects_bad_shapes_and_flags(L):
    assert L.vae_conv3x3_nhwc(FAKE, 1, 4, 4, 15, FAKE, None, None, FAKE, 16, 1.0, 0, None) == -2
    assert "multiple of 16" in vg.last_error()
    assert L.vae_conv3x3_nhwc(FAKE, 1, 0, 4, 16, FAKE, None, None, FAKE, 16, 1.0, 0, None) == -2
    assert L.vae_conv3x3_nhwc(None, 1, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, 0, None) == -1
    assert L.vae_conv3x3_nhwc(FAKE, 1, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, 1 << 12, None) == -1
    assert L.vae_conv3x3_nhwc(FAKE + 8, 1, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, 0, None) == -3
    assert L.vae_conv1x1(FAKE, 10, 16, FAKE, None, None, FAKE, 16, 1.0, vg.UPSAMPLE2X, None) == -1
    assert L.vae_conv1x1(FAKE, 10, 16, FAKE, None, None, FAKE, 0, 1.0, 0, None) == -2


def test_conv_rejects_bad_padding_and_downsample_combinations(L):
    c = L.vae_conv3x3_nhwc
    refl, rep, up, down = vg.PAD_REFLECT, vg.PAD_REPLICATE, vg.UPSAMPLE2X, vg.DOWNSAMPLE2X
    assert c(FAKE, 1, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, refl | rep, None) == -1
    assert "one padding" in vg.last_error()
    assert c(FAKE, 1, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, refl | up, None) == -1
    assert c(FAKE, 1, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, down | up, None) == -1
    assert c(FAKE, 1, 1, 4, 16, FAKE, None, None, FAKE, 16, 1.0, refl, None) == -2
    assert c(FAKE, 1, 4, 1, 16, FAKE, None, None, FAKE, 16, 1.0, down, None) == -2
    assert "h, w >= 2" in vg.last_error()
    # the 3x3x3 conv has no reflect padding or downsample flag
    c3 = L.vae_conv3d_causal_ndhwc
    assert c3(FAKE, 1, 2, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, refl, None) == -1
    assert c3(FAKE, 1, 2, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, down, None) == -1


def test_conv3d_rejects_bad_shapes_and_flags(L):
    c3 = L.vae_conv3d_causal_ndhwc
    assert c3(FAKE, 1, 0, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, 0, None) == -1   # no frames
    assert c3(FAKE, 1, 2, 4, 4, 15, FAKE, None, None, FAKE, 16, 1.0, 0, None) == -2   # cin % 16
    assert c3(FAKE, 1, 2, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, 1 << 9, None) == -1
    assert c3(None, 1, 2, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, 0, None) == -1
    # the temporal 2x flag belongs to the 3x3x3 conv only
    assert L.vae_conv3x3_nhwc(FAKE, 1, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, vg.UPSAMPLE_T2X, None) == -1


def test_norms_reject_bad_shapes(L):
    assert L.vae_rmsnorm_silu(FAKE, 4, 6, None, FAKE, 0, 1.0, FAKE, None) == -2
    assert L.vae_rmsnorm_silu(None, 4, 8, None, FAKE, 0, 1.0, FAKE, None) == -1
    assert L.vae_groupnorm_silu(FAKE, 1, 16, 100, 32, 1e-6, None, FAKE, FAKE, 1, 1.0, FAKE, FAKE, 1 << 20, None) == -2
    assert L.vae_groupnorm_workspace_bytes(1, 16, 100, 32) == 0
    assert L.vae_groupnorm_workspace_bytes(1, 16384, 256, 32) > 0
    ws = L.vae_groupnorm_workspace_bytes(1, 1024, 128, 32)
    assert L.vae_groupnorm_silu(FAKE, 1, 1024, 128, 32, 1e-6, None, FAKE, FAKE, 1, 1.0, FAKE, FAKE, ws - 16,
                                None) == -4
    assert L.vae_cast_f16(FAKE, 30, 6, None, 1.0, FAKE, None) == -2


def test_attention_and_decoder_reject_bad_arguments(L):
    assert L.vae_mid_attention_workspace_bytes(1024, 100, 32) == 0
    assert L.vae_mid_attention_workspace_bytes(1024, 48, 32) > 0
    assert L.vae_mid_attention_workspace_bytes(1024, 48, 16) > 0
    assert L.vae_mid_attention_workspace_bytes(1024, 512, 32) > 0
    assert L.vae_mid_attention(FAKE, 16, 100, 1, 32, 1e-6, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               FAKE, FAKE, FAKE, 1 << 30, None) == -2
    assert L.vae_mid_attention(FAKE, 16, 128, 5, 32, 1e-6, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               FAKE, FAKE, FAKE, 1 << 30, None) == -1
    out = ctypes.c_void_p()
    assert L.vae_decoder_create(None, ctypes.byref(out)) == -1
    assert L.vae_decode(None, FAKE, 4, 4, FAKE, None, FAKE, 1 << 20, None) == -1
    n = ctypes.c_size_t()
    assert L.vae_decode_workspace(None, 4, 4, None, ctypes.byref(n)) == -1


def test_no_cpu_fallback_without_a_gpu(L):
    """Valid arguments without a usable GPU: an error code, never a CPU result."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = L.vae_conv3x3_nhwc(FAKE, 1, 4, 4, 16, FAKE, None, None, FAKE, 16, 1.0, 0, None)
    assert rc in (-5, -7)

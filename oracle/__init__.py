"""CPU f64 oracle for the image-VAE decoder hot path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product path (the CUDA library and its
Python binding) never imports, links or executes anything here, and this
package imports nothing from the product.

What it is: a plain, slow, obviously correct NCHW implementation in float64
of what the decoder computes, written from the pages' own definitions:

- ``vae.rs`` (cortiq-engine 0.7.6, the FLUX-class ``AutoencoderKL`` decoder):
  ``Conv2d::apply``, ``GroupNorm::apply``, ``silu``, ``upsample2x``,
  ``ResnetBlock::apply``, ``AttnBlock::apply``, ``VaeDecoder::decode``;
- ``qi21_vae.rs`` (cortiq-engine 0.8.3, the resident Qwen-Image-2.1 decoder):
  the ``qv_rmsn`` RMS_norm, the ``qv_dupup`` DupUp3D shortcut, ``Rec::resnet``,
  ``attention``, ``run_blocks``, ``output_rows`` and the band planner
  (``grow``, ``half``, ``plan_band``);
- ``s2v_vae.rs`` (cortiq-engine 0.8.72): replicate padding, read for 2-D as a
  clamp to the edge of the (upsampled) grid; the 3x3x3 causal conv;
- ``vae3d.rs`` (cortiq-engine 0.5.87, the video VAE's encoder half):
  reflect padding (``EncConv::apply``), the far-side reflect pad of the
  stride-2 downsample (``reflect_pad_far``) and the encoder level loop.

A library primitive (numpy's matmul) serves as the channel contraction of a
conv tap and of the attention products; nothing is blocked, fused or
reordered beyond what the definitions state, except that the attention is
evaluated a block of query rows at a time (each row's arithmetic is the
same as the unblocked one; only the memory held at once changes).

Scalings that are exact powers of two on the GPU (the 2^-g range guard of
the f16 casts and its 2^g undo in the conv epilogue) are the identity in
exact arithmetic and do not appear here.

Pins (``tests/test_oracle_*.py``): the pages' printed worked examples
(``tests/golden/``), independent brute-force loops on tiny inputs, delta
kernels, linearity, closed forms of the norms and of SiLU, attention
invariants, the DupUp index formula, and banded == whole-frame decoding.
The whole decoders (``decode_gn``, ``decode_rms``) are pinned against an
element-by-element brute-force restatement of both decoders on tiny random
decoders (scalar loops over a pixel-major layout), with planted composition
mistakes that the comparison must see; no trained weights or third-party
decoder exist here to compare with.
"""
from .ops import (conv2d, conv2d_at, conv2d_down, conv3d_causal, causal_source_frame, subpixel_up_weights, conv2d_up_subpixel,
                  upsample2x, silu, group_norm, rms_norm, dupup, attention, attention_rows, linear_tokens)
from .decoder import (resnet, up_block, down_block, decode_gn, decode_rms, decode, Rows, grow, half,
                      levels, plan_band, plan_bands, decode_rms_banded, head_rms,
                      run_blocks_window, output_rows_window)

__all__ = [
    "conv2d", "conv2d_at", "conv2d_down", "conv3d_causal", "causal_source_frame", "subpixel_up_weights", "conv2d_up_subpixel",
    "upsample2x", "silu", "group_norm", "rms_norm", "dupup",
    "attention", "attention_rows", "linear_tokens", "resnet", "up_block", "down_block", "decode_gn", "decode_rms", "decode",
    "Rows", "grow", "half", "levels", "plan_band", "plan_bands", "decode_rms_banded",
    "head_rms", "run_blocks_window", "output_rows_window",
]

// Internal interface of the implicit-GEMM conv kernel, shared by the public
// conv entry points, the mid attention and the decoder driver.
#pragma once

#include "vae_common.cuh"

namespace vae {

struct ConvArgs {
    const void* x = nullptr;     // f16 NHWC [n][h_in][w_in][cin]
    int n = 1, h_in = 0, w_in = 0, cin = 0;
    const void* w = nullptr;     // f16 [cout][taps][cin]
    int cout = 0;
    int taps = 9;                // 9 (3x3), 1 (1x1) or 27 (3x3x3 causal over frames)
    // 3x3x3 causal conv: x holds n images of frames_in frames ([n][frames_in][h][w][cin]);
    // y holds n images of frames_out = t_up ? 2 * frames_in - 1 : frames_in frames.
    int frames_in = 1;
    bool t_up = false;
    // The up conv (up, taps 9) as four 2x2 convs on the source grid: w holds the
    // summed weights [cout][16][cin], tap (q*2+p)*4 + ty*2 + tx (vae_pack_subpixel_weights).
    bool subpix = false;
    const float* bias = nullptr;
    const float* residual = nullptr;  // f32 NHWC [n][H][W][cout]; may alias y
    void* y = nullptr;
    float oscale = 1.0f;
    bool up = false, rep = false, silu = false, out_f16 = false;
    // f16 output only: the stored value is the epilogue's value times out_scale
    // (the decoder's 2^-g range guard, exact), as the guarded cast would store it.
    float out_scale = 1.0f;
    // Reflect padding (mirror about the edge, the edge not repeated).
    bool refl = false;
    // The encoder's downsample: x padded by one row and column on the far side
    // (zero / rep / refl), then an unpadded stride-2 conv; output h_in/2 x w_in/2.
    bool down = false;
    bool no_halo = false;        // force the per-tap A path (tests and sweeps)
    bool no_pair = false;        // force the single-CTA kernel
    // NCHW f32 output of output rows [keep_lo, keep_hi) at destination row
    // (Y - keep_lo + dst_row0), channel planes `plane` floats apart.
    // keep_hi <= keep_lo means all rows of an [n][cout][H][W] tensor.
    bool out_nchw = false;
    int keep_lo = 0, keep_hi = 0, dst_row0 = 0;
    long long plane = 0;
    // DupUp3D add of the up conv: src f32 NHWC [n][h_in][w_in][dup_cin];
    // output channel o of parity (q, p) adds
    // src[..., (o*dup_factor + dup_ftoff + 2q + p) / dup_repeats].
    const float* dup_src = nullptr;
    int dup_cin = 0, dup_factor = 0, dup_repeats = 0, dup_ftoff = 0;
    // Fused RMS_norm (+SiLU) of each output pixel into rms_out, f16
    // [n][H][W][cout] (cout % 16 == 0, cout <= 144); y (f32) may then be NULL.
    const float* rms_gamma = nullptr;
    void* rms_out = nullptr;
    bool rms_silu = false;
    // GroupNorm partial statistics of the f32 output (2-D 3x3 convs): records
    // float4 (count, mean, M2, 0) at [n][conv_gn_chunks(...)][gn_groups],
    // each written once; statistics of the values stored in y.
    void* gn_part = nullptr;
    int gn_groups = 0;
};

// Records per image of the GroupNorm statistics epilogue: 4 per M tile.
int conv_gn_chunks(int h_in, int w_in, bool up, bool down);

int conv_validate(const ConvArgs& a);
// w [cout][3][3][cin] f16 -> the sub-pixel form's summed weights [cout][16][cin] f16.
int pack_subpixel_run(const void* w, int cout, int cin, void* ws, cudaStream_t stream);
int conv_run(const ConvArgs& a, cudaStream_t stream);

}  // namespace vae

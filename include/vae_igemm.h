/*
 * vae_igemm.h — C ABI of the GB300 (sm_103a) image-VAE decoder hot path.
 *
 * The operations restate the image-VAE decoders of the cortiq-engine pages:
 * "qi21_vae.rs" (the resident Qwen-Image-2.1 decoder: NHWC implicit-GEMM
 * 3x3 convs with the nearest-2x upsample folded into the A-tile gather,
 * the qv_rmsn RMS_norm, the qv_dupup DupUp3D shortcut, the band planner) and
 * "vae.rs" (the FLUX-class AutoencoderKL decoder: Conv2d::apply,
 * GroupNorm::apply, AttnBlock::apply, VaeDecoder::decode), with replicate
 * padding from "s2v_vae.rs".
 *
 * Conventions for every entry point below:
 *  - Pointers named *_dev are CUDA device memory owned by the caller. The
 *    library never frees or keeps them past the call (the decoder handle owns
 *    only its own packed weights).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream). No call synchronises the stream except vae_sync_status and
 *    vae_decode_host.
 *  - Return value: VAE_OK (0) or a negative vae_status. Every shape, flag and
 *    alignment is validated before anything is enqueued: on an error nothing
 *    was launched and outputs are untouched. vae_last_error() gives the text.
 *  - f16 tensors are IEEE binary16 (passed as void* / uint16_t bits); f32 is
 *    IEEE binary32. "NHWC" = [n][h][w][c], c contiguous.
 *  - Device-side waits are bounded (vae_set_wait_timeout_ns). A wait that
 *    runs out makes the kernel record VAE_ERR_DEVICE_TIMEOUT in the device
 *    status word and return; vae_sync_status() reports it.
 *  - There is no CPU fallback: without a usable sm_103a GPU every compute
 *    call returns VAE_ERR_CUDA.
 */
#ifndef VAE_IGEMM_H
#define VAE_IGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* vae_stream_t;

typedef enum {
    VAE_OK = 0,
    VAE_ERR_ARG = -1,            /* NULL where a pointer is required, bad flag, bad enum */
    VAE_ERR_SHAPE = -2,          /* unsupported or inconsistent sizes */
    VAE_ERR_ALIGN = -3,          /* a pointer is not 16-byte aligned */
    VAE_ERR_NOMEM = -4,          /* workspace too small / host allocation failed */
    VAE_ERR_CUDA = -5,           /* a CUDA runtime/driver call failed (text in vae_last_error) */
    VAE_ERR_DEVICE_TIMEOUT = -6, /* a bounded device wait ran out */
    VAE_ERR_UNSUPPORTED = -7     /* no sm_103a device */
} vae_status;

/* Conv flags. */
enum {
    VAE_UPSAMPLE2X = 1,     /* nearest-2x of the input folded into the gather: output is 2h x 2w */
    VAE_PAD_REPLICATE = 2,  /* out-of-grid reads take the nearest edge pixel (default: zero) */
    VAE_EPI_SILU = 16,      /* SiLU v/(1+e^-v) applied last in the epilogue */
    VAE_OUT_F16 = 32,       /* store the output as f16 (default f32) */
    VAE_UPSAMPLE_T2X = 64,  /* 3x3x3 conv only: causal temporal 2x folded into the gather */
    VAE_UPSAMPLE2X_SUBPIXEL = 128, /* with VAE_UPSAMPLE2X: the up conv as four 2x2 convs (w_dev from
                                      vae_pack_subpixel_weights); 4/9 of the MACs, weight sums rounded */
    VAE_PAD_REFLECT = 256,  /* out-of-grid reads mirror about the edge, the edge not repeated
                               (-1 reads 1, n reads n - 2); needs h_in, w_in >= 2 */
    VAE_DOWNSAMPLE2X = 512  /* the encoder's downsample: one row and column padded on the far
                               side only, then an unpadded stride-2 3x3 conv: output h_in/2 x w_in/2 */
};

/* Library version string and the compute capability it was built for. */
const char* vae_version(void);

/* Thread-local text of the last error returned on this thread ("" if none). */
const char* vae_last_error(void);

/* Synchronises `stream`, reads and clears the device status word of the
 * current device. Returns VAE_OK or VAE_ERR_DEVICE_TIMEOUT (a kernel gave up a
 * bounded wait since the last call) or VAE_ERR_CUDA. */
int vae_sync_status(vae_stream_t stream);

/* Upper bound, in nanoseconds of %globaltimer, on any single device-side wait
 * of later launches from this process (default 4e9). 0 restores the default. */
int vae_set_wait_timeout_ns(unsigned long long ns);

/* Failure-detection self test: launches one CTA that waits (bounded by
 * timeout_ns) on an mbarrier phase nothing completes, then returns. The
 * kernel records VAE_ERR_DEVICE_TIMEOUT; this call synchronises and returns
 * what vae_sync_status reports (VAE_ERR_DEVICE_TIMEOUT when the path works).
 * No fault, trap or hang is involved. */
int vae_selftest_wait_timeout(unsigned long long timeout_ns, vae_stream_t stream);

/*
 * 3x3 convolution, stride 1, padding 1, as an implicit GEMM on tcgen05.
 *   y[p, o] = SiLU?( oscale * sum_{tap, c} xt[p + d_tap, c] * w[o, tap, c]
 *                    + bias[o] + residual[p, o] )
 * where xt is x, or nearest-2x(x) with VAE_UPSAMPLE2X, and reads outside the
 * (upsampled) grid are 0, or with VAE_PAD_REPLICATE the nearest edge pixel, or
 * with VAE_PAD_REFLECT the pixel mirrored about the edge.
 * With VAE_DOWNSAMPLE2X (the encoder's downsample) output (Y, X) reads source
 * (2Y + ky, 2X + kx) of x padded by one row and column on the far side (by the
 * padding flag: zero, replicate or reflect); H = h_in / 2, W = w_in / 2 (floor).
 * ("vae.rs" Conv2d::apply; "qi21_vae.rs" conv_s and the module doc's
 * implicit-GEMM recipe; "s2v_vae.rs" replicate padding and conv_down;
 * "vae3d.rs" EncConv::apply (reflect) and reflect_pad_far.)
 *
 *   x_dev     f16 NHWC [n][h_in][w_in][cin], 16-byte aligned.
 *   w_dev     f16 [cout][3][3][cin] (tap-major: K index = (ky*3+kx)*cin + c), or with
 *             VAE_UPSAMPLE2X_SUBPIXEL the summed weights of vae_pack_subpixel_weights.
 *   bias_dev  f32 [cout] or NULL (no bias).
 *   residual_dev  f32 NHWC [n][H][W][cout] or NULL; may equal y_dev (in place).
 *   y_dev     NHWC [n][H][W][cout], f32, or f16 with VAE_OUT_F16;
 *             H = h_in, W = w_in, or 2*h_in, 2*w_in with VAE_UPSAMPLE2X,
 *             or h_in/2, w_in/2 with VAE_DOWNSAMPLE2X.
 *   oscale    multiplies the f32 accumulator (the undo of a 2^-g input guard).
 * Requirements: n, h_in, w_in >= 1; cin % 16 == 0, 16 <= cin <= 8192;
 * 1 <= cout <= 2^20; x_dev, w_dev 16-byte aligned. Outputs of any cout are
 * supported (vector stores when cout % 16 == 0). VAE_PAD_REFLECT and
 * VAE_DOWNSAMPLE2X need h_in, w_in >= 2; at most one padding flag; the
 * upsample and the downsample exclude each other, and reflect padding does not
 * combine with the upsample (VAE_ERR_ARG / VAE_ERR_SHAPE otherwise).
 */
int vae_conv3x3_nhwc(const void* x_dev, int n, int h_in, int w_in, int cin,
                     const void* w_dev, const float* bias_dev, const float* residual_dev,
                     void* y_dev, int cout, float oscale, unsigned flags, vae_stream_t stream);

/*
 * 1x1 convolution = plain GEMM over m pixels, the same kernel with one tap.
 *   y[p, o] = SiLU?( oscale * sum_c x[p, c] * w[o, c] + bias[o] + residual[p, o] )
 * ("qi21_vae.rs" conv mode 0: post_quant, the guarded shortcut, attention
 * q/k/v/proj; "vae.rs" AttnBlock::proj.)
 *   x_dev f16 [m][cin]; w_dev f16 [cout][cin]; bias_dev f32 [cout] or NULL;
 *   residual_dev f32 [m][cout] or NULL (may equal y_dev); y_dev [m][cout]
 *   f32 or f16 (VAE_OUT_F16). Flags: VAE_EPI_SILU, VAE_OUT_F16 only.
 * Requirements as vae_conv3x3_nhwc; m >= 1.
 */
/*
 * 3x3 conv with RMS_norm(+SiLU) of each output pixel fused into its epilogue
 * ("qi21_vae.rs" qv_rmsn applied to the conv's output; the decoders use it for
 * a ResNet's first conv, whose output only feeds that norm):
 *   v = oscale * sum x~ * w + bias;  rms_dev[p, c] = f16( SiLU?( v[c] * sqrt(C) / max(||v||, 1e-12) * gamma[c] ) )
 * with the standalone vae_rmsnorm_silu's exact evaluation order (same bits as
 * vae_conv3x3_nhwc followed by vae_rmsnorm_silu with out_scale 1).
 *   y_dev     f32 NHWC [n][H][W][cout] also stored when non-NULL, else only rms_dev.
 *   rms_dev   f16 NHWC [n][H][W][cout]; gamma_dev f32 [cout]; 16-byte aligned.
 * Requirements as vae_conv3x3_nhwc plus 16 <= cout <= 144, cout % 16 == 0 (one
 * CTA holds all of a pixel's channels); no residual, no upsample. Flags:
 * VAE_PAD_REPLICATE, VAE_PAD_REFLECT, VAE_DOWNSAMPLE2X. Rows of >= 128 pixels
 * with y_dev NULL take the staged two-pass epilogue (TMEM read twice, f16 rows
 * stored by TMA); other cases keep the pixel's row in registers.
 */
int vae_conv3x3_nhwc_rms(const void* x_dev, int n, int h_in, int w_in, int cin, const void* w_dev,
                         const float* bias_dev, float* y_dev, int cout, float oscale, unsigned flags,
                         const float* gamma_dev, int silu, void* rms_dev, vae_stream_t stream);

/*
 * Sub-pixel (phase) form of the nearest-2x up conv (an optional speed-up, not
 * on the pages): output (2v+q, 2u+p) reads source rows
 * v + floor((q + ky - 1) / 2), so the three ky taps land on two source rows per
 * parity q (ky {0} | {1, 2} for q = 0, {0, 1} | {2} for q = 1), and likewise the
 * columns. Summing the weights that read one source pixel turns each parity
 * class into a 2x2 conv on the source grid: exact in real arithmetic, 4/9 of the
 * MACs; the sums are rounded to f16 once, which changes the rounding.
 *   w_dev      f16 [cout][3][3][cin] (the vae_conv3x3_nhwc layout).
 *   w_sub_dev  f16 [cout][16][cin], tap (q*2+p)*4 + ty*2 + tx; caller-owned.
 * Use with vae_conv3x3_nhwc(..., VAE_UPSAMPLE2X | VAE_UPSAMPLE2X_SUBPIXEL).
 * Requirements: 1 <= cout <= 2^20, 1 <= cin <= 8192, 16-byte aligned pointers.
 */
int vae_pack_subpixel_weights(const void* w_dev, int cout, int cin, void* w_sub_dev, vae_stream_t stream);

/*
 * 3x3x3 causal convolution over frames, the same implicit GEMM with 27 taps
 * ("s2v_vae.rs" module doc and conv_any: the conv mode 3 of zi_mm, its causal
 * two-frame look-back, the replicate padding and the nearest upsample in the
 * gather, src_f for the temporal 2x):
 *   y[b, f, Y, X, o] = SiLU?( oscale * sum_{kt, ky, kx, c} xt[b, s(f, kt), Y + ky - 1, X + kx - 1, c]
 *                              * w[o, kt, ky, kx, c] + bias[o] + residual[b, f, Y, X, o] )
 * with the temporal tap kt = 0, 1, 2 reading upsampled frame vf = max(f + kt - 2, 0)
 * (causal: frames before the first replicate it) and s(f, kt) = vf, or with
 * VAE_UPSAMPLE_T2X the source frame (vf > 0 ? (vf - 1) / 2 + 1 : 0).
 * Spatially as vae_conv3x3_nhwc: xt is x or nearest-2x(x) with
 * VAE_UPSAMPLE2X; reads outside the (upsampled) grid are 0 or, with
 * VAE_PAD_REPLICATE, the nearest edge pixel.
 *   x_dev     f16 [n][f_in][h_in][w_in][cin], 16-byte aligned.
 *   w_dev     f16 [cout][3][3][3][cin] (K index = ((kt*3+ky)*3+kx)*cin + c).
 *   bias_dev  f32 [cout] or NULL.
 *   residual_dev  f32 [n][F][H][W][cout] or NULL; may equal y_dev.
 *   y_dev     [n][F][H][W][cout] f32, or f16 with VAE_OUT_F16; F = f_in, or
 *             2*f_in - 1 with VAE_UPSAMPLE_T2X; H, W as vae_conv3x3_nhwc.
 * Flags: VAE_UPSAMPLE2X, VAE_UPSAMPLE_T2X, VAE_PAD_REPLICATE, VAE_EPI_SILU,
 * VAE_OUT_F16. Requirements as vae_conv3x3_nhwc, and f_in >= 1.
 */
int vae_conv3d_causal_ndhwc(const void* x_dev, int n, int f_in, int h_in, int w_in, int cin,
                            const void* w_dev, const float* bias_dev, const float* residual_dev,
                            void* y_dev, int cout, float oscale, unsigned flags, vae_stream_t stream);

int vae_conv1x1(const void* x_dev, int m, int cin, const void* w_dev,
                const float* bias_dev, const float* residual_dev, void* y_dev, int cout,
                float oscale, unsigned flags, vae_stream_t stream);

/*
 * Per-pixel RMS_norm (+ bias on read, optional SiLU) -> f16:
 *   v = x[p, :] + bias_in;  y[p, c] = SiLU?( v[c] * sqrt(C) / max(||v||_2, 1e-12) * gamma[c] ) * out_scale
 * ("qi21_vae.rs" qv_rmsn.)
 *   x_dev f32 [m][c]; bias_in_dev f32 [c] or NULL; gamma_dev f32 [c];
 *   y_dev f16 [m][c]. Requirements: m >= 1, c % 4 == 0, 4 <= c <= 16384;
 *   pointers 16-byte aligned.
 */
int vae_rmsnorm_silu(const float* x_dev, int m, int c, const float* bias_in_dev,
                     const float* gamma_dev, int silu, float out_scale, void* y_dev,
                     vae_stream_t stream);

/*
 * GroupNorm(groups) over each image (+ bias on read, optional SiLU) -> f16:
 *   v = x + bias_in; per (image, group g of c/groups consecutive channels):
 *   mean mu and biased variance var over hw * c/groups values;
 *   y = SiLU?( (v - mu) / sqrt(var + eps) * gamma[c] + beta[c] ) * out_scale
 * ("vae.rs" GroupNorm::apply; "s2v_vae.rs" s2v_gn_part / s2v_gn_fin /
 * s2v_gn_apply.) Statistics: per-chunk (count, mean, M2) partials in f32
 * merged with Chan's formula.
 *   x_dev f32 NHWC [n][hw][c]; gamma/beta f32 [c]; bias_in f32 [c] or NULL;
 *   y_dev f16 [n][hw][c]; workspace_dev of at least
 *   vae_groupnorm_workspace_bytes(n, hw, c, groups) bytes, 16-byte aligned,
 *   contents ignored on entry.
 * Requirements: c % groups == 0, c % 4 == 0, 4 <= c <= 4096, 1 <= groups <= 1024.
 */
size_t vae_groupnorm_workspace_bytes(int n, int hw, int c, int groups);
int vae_groupnorm_silu(const float* x_dev, int n, int hw, int c, int groups, float eps,
                       const float* bias_in_dev, const float* gamma_dev, const float* beta_dev,
                       int silu, float out_scale, void* y_dev,
                       void* workspace_dev, size_t workspace_bytes, vae_stream_t stream);

/*
 * GroupNorm with its statistics taken by the conv that produces its input (an
 * optional restructuring, not on the pages): the two-pass GroupNorm of
 * "s2v_vae.rs" (s2v_gn_part reads the tensor for per-block partial sums,
 * s2v_gn_apply reads it again to normalise) loses its first read because the
 * 3x3 conv's epilogue, which holds every output value in registers anyway,
 * emits the partial statistics of what it stores.
 *
 * vae_conv3x3_nhwc_gn: the conv of vae_conv3x3_nhwc (f32 output only), and
 *   gn_stats_dev f32 [n][groups][2] = (mean, 1 / sqrt(var + eps)) of the
 *   stored output per (image, group of cout/groups consecutive channels),
 *   biased variance over H * W * cout/groups values ("vae.rs"
 *   GroupNorm::apply). Each epilogue warp writes one record per group for
 *   its 32 pixels into workspace_dev: shifted sums (count, K, sum (v - K),
 *   sum (v - K)^2), K one of the group's values; a second kernel turns them
 *   into (count, mean, M2) and merges them with Chan's formula in a fixed
 *   order (deterministic).
 *   Flags: VAE_UPSAMPLE2X, VAE_PAD_REPLICATE, VAE_PAD_REFLECT,
 *   VAE_DOWNSAMPLE2X, VAE_EPI_SILU (statistics of the SiLU output then).
 *   workspace_dev: >= vae_conv3x3_gn_workspace_bytes(...) bytes, 16-byte
 *   aligned, contents ignored on entry. Requirements as vae_conv3x3_nhwc plus
 *   cout % 16 == 0 and cout / groups in {4, 8} or a multiple of 16 (every
 *   group of the FLUX-class widths 128 / 256 / 512 with 32 groups).
 * vae_groupnorm_apply: y = SiLU?((x - mean) * rstd * gamma[c] + beta[c]) * out_scale
 *   -> f16, one read of x, with gn_stats_dev from vae_conv3x3_nhwc_gn.
 *   x_dev f32 [n][hw][c]; y_dev f16 [n][hw][c]; 16-byte aligned;
 *   c % 4 == 0, c % groups == 0.
 */
size_t vae_conv3x3_gn_workspace_bytes(int n, int h_in, int w_in, int cout, int groups, unsigned flags);
int vae_conv3x3_nhwc_gn(const void* x_dev, int n, int h_in, int w_in, int cin, const void* w_dev,
                        const float* bias_dev, const float* residual_dev, float* y_dev, int cout,
                        float oscale, unsigned flags, int groups, float eps, float* gn_stats_dev,
                        void* workspace_dev, size_t workspace_bytes, vae_stream_t stream);
int vae_groupnorm_apply(const float* x_dev, int n, int hw, int c, int groups, const float* gn_stats_dev,
                        const float* gamma_dev, const float* beta_dev, int silu, float out_scale,
                        void* y_dev, vae_stream_t stream);

/*
 * GroupNorm exactly as vae_groupnorm_silu, for callers that cannot allocate
 * device memory. The pages have no counterpart to this entry point.
 *
 * Some callers have no way to hand this library a workspace: an inference
 * engine's plugin whose only memory is what the engine planned ahead of time,
 * or a serving loop that must never call cudaMalloc because an allocation can
 * synchronise the whole device and stall every stream in flight. This variant
 * needs no workspace and allocates nothing: its partial statistics live in a
 * fixed 512 KB array of device memory that the library defines at file scope;
 * every GPU that loads the library holds that array until the process exits.
 *
 * Limit: calls whose statistics need more than 512 KB of scratch (see
 * vae_groupnorm_workspace_bytes; every call with groups <= 32 and n <= 416
 * fits) return VAE_ERR_NOMEM without launching anything.
 * Set-up: the first call on each device looks the array's device address up
 * (with that device current); make that first call before any stream capture.
 * Sharing: all calls use the same array and it keeps the last call's
 * contents (each call overwrites every entry it reads, so nothing needs to
 * start at zero). Calls that may overlap on the GPU (different streams, or
 * different host threads) race on the array and must be serialised by the
 * caller.
 * Arguments, layouts, requirements and errors otherwise as vae_groupnorm_silu.
 */
int vae_groupnorm_silu_static(const float* x_dev, int n, int hw, int c, int groups, float eps,
                              const float* bias_in_dev, const float* gamma_dev, const float* beta_dev,
                              int silu, float out_scale, void* y_dev, vae_stream_t stream);

/*
 * f32 -> f16 cast of the raw residual stream with its range guard:
 *   y[i] = (x[i] + bias[i % c]) * scale            (scale normally 2^-g)
 * ("qi21_vae.rs" qv_cast and the guard() doc.)
 *   x_dev f32 [count]; bias_dev f32 [c] or NULL; y_dev f16 [count];
 *   count % c == 0, c % 4 == 0, pointers 16-byte aligned.
 */
int vae_cast_f16(const float* x_dev, size_t count, int c, const float* bias_dev,
                 float scale, void* y_dev, vae_stream_t stream);

/* Mid self-attention norm kinds. */
enum { VAE_NORM_GROUP = 0, VAE_NORM_RMS = 1 };

/*
 * Single-head spatial self-attention of the decoder's mid block, in place on
 * the f32 residual stream:
 *   n = GroupNorm(x) or RMS_norm(x)*gamma (no SiLU); q,k,v = n W^T + b;
 *   o = softmax(q k^T / sqrt(c)) v; x += o W_o^T + b_o.
 * ("vae.rs" AttnBlock::apply / finish; "qi21_vae.rs" attention.)
 * Computed in a folded form that is exact in real arithmetic: the key bias
 * adds the same amount to every score of a row, which the softmax removes,
 * and the rows of the softmax sum to one, so with M = Wk^T Wq and
 * Wov = Wo Wv (f16, formed on the device each call)
 *   s_ij = (n_i M^T + Wk^T bq) . n_j,   x_i += (sum_j p_ij n_j) Wov^T + (Wo bv + bo).
 * (VAE_ATTN_FOLD=0 in the environment runs the q, k, v projections as written.)
 * Scores and the online softmax run in one tcgen05 kernel that writes P (f16)
 * to the workspace; a second kernel forms P.V; the projections run on the
 * implicit-GEMM kernel.
 *   x_dev f32 [m][c] (tokens = pixels of one image); w*_dev f16 [c][c]
 *   (row = output channel), 16-byte aligned; b*_dev f32 [c]; norm_beta_dev
 *   ignored for RMS.
 *   workspace_dev >= vae_mid_attention_workspace_bytes(m, c, groups) (which
 *   sizes for GroupNorm when c % groups == 0, else for RMS_norm), 16-byte
 *   aligned.
 * Requirements: c % 16 == 0, 16 <= c <= 2048, m >= 1. Errors: VAE_ERR_ARG
 * (NULL pointer, norm kind), VAE_ERR_SHAPE, VAE_ERR_ALIGN, VAE_ERR_NOMEM
 * (workspace too small); argument checks fail before anything is launched.
 */
size_t vae_mid_attention_workspace_bytes(int m, int c, int groups);
int vae_mid_attention(float* x_dev, int m, int c, int norm_kind, int groups, float eps,
                      const float* norm_gamma_dev, const float* norm_beta_dev,
                      const void* wq_dev, const float* bq_dev, const void* wk_dev, const float* bk_dev,
                      const void* wv_dev, const float* bv_dev, const void* wo_dev, const float* bo_dev,
                      void* workspace_dev, size_t workspace_bytes, vae_stream_t stream);

/* ───────────────────────────── whole decoder ───────────────────────────── */

/* Host-side description of a decoder, mirroring "vae.rs" VaeChainArgs and
 * its Vae*Ref structs. All pointers are HOST memory read only during
 * vae_decoder_create (which copies and re-lays the weights on the device). */
typedef struct {
    const uint16_t* w;  /* f16 bits, OIHW [cout][cin][k][k]; NULL = this conv is absent */
    const float* b;     /* f32 [cout] */
    int cout, cin, k;   /* k = 1 or 3 */
} vae_conv_desc;

typedef struct {
    const float* gamma; /* f32 [c] */
    const float* beta;  /* f32 [c]; GroupNorm only (NULL for RMS_norm) */
} vae_norm_desc;

typedef struct {
    vae_norm_desc norm1;
    vae_conv_desc conv1;
    vae_norm_desc norm2;
    vae_conv_desc conv2;
    vae_conv_desc shortcut; /* 1x1 when cin != cout; w = NULL otherwise */
} vae_resnet_desc;

typedef struct {
    vae_norm_desc norm;
    vae_conv_desc q, k, v, o; /* 1x1, c -> c */
} vae_attn_desc;

typedef struct {
    const vae_resnet_desc* resnets;
    int n_resnets;
    vae_conv_desc up;  /* 3x3 conv after nearest-2x; w = NULL: no upsample */
    int in_dim, out_dim;
    int ft;            /* DupUp temporal factor (1 for images) */
} vae_up_desc;

enum { VAE_FAMILY_GN = 0, VAE_FAMILY_RMS = 1 };

typedef struct {
    int family;            /* VAE_FAMILY_GN (FLUX-class) or VAE_FAMILY_RMS (Qwen/Wan-style) */
    int latent_channels;
    float scaling, shift;  /* GN family: z/scaling + shift before conv_in */
    int groups;            /* GroupNorm groups (GN family) */
    float eps;             /* GroupNorm eps */
    int dupup;             /* RMS family: add the DupUp shortcut after each up conv */
    vae_conv_desc post_quant; /* RMS family 1x1 before conv_in; w = NULL: none */
    vae_conv_desc conv_in;
    vae_resnet_desc mid_res1;
    vae_attn_desc mid_attn;
    vae_resnet_desc mid_res2;
    const vae_up_desc* ups;
    int n_ups;
    vae_norm_desc norm_out;
    vae_conv_desc conv_out;
} vae_decoder_desc;

typedef struct vae_decoder* vae_decoder_t;

/* Validates `desc`, copies every weight to the current device in the
 * kernels' layouts and returns a handle. */
int vae_decoder_create(const vae_decoder_desc* desc, vae_decoder_t* out);
int vae_decoder_destroy(vae_decoder_t dec);

typedef struct {
    int band_from;   /* RMS family: up blocks >= band_from run in horizontal bands */
    int nbands;      /* number of equal kept-row bands (0 or 1 with band_rows 0: whole frame) */
    int band_rows;   /* alternative to nbands: at most this many kept rows per band */
    int guard_log2;  /* f16 range guard g of the raw-stream casts (default 8 when < 0) */
    unsigned flags;  /* 0, or VAE_DECODE_PROFILE (| VAE_DECODE_PROFILE_FULLRES) | VAE_DECODE_FUSE_NORM |
                        VAE_DECODE_NO_FUSION | VAE_DECODE_SUBPIXEL_UP */
} vae_decode_opts;

/* vae_decode_opts.flags: record CUDA events around every stage of this
 * decode (read back with vae_decode_profile). */
enum {
    VAE_DECODE_PROFILE = 1,
    /* Run every RMS_norm as its own kernel (the default); overrides
     * VAE_DECODE_FUSE_NORM. Also cast the stream to the up convs' guarded f16
     * input in a separate kernel; by default the last ResNet conv of an up block
     * stores that f16 input itself ((conv + bias + skip) * 2^-g rounded to f16,
     * the same bits) and the f32 stream it would replace is not written. */
    VAE_DECODE_NO_FUSION = 2,
    /* Compute a ResNet's second RMS_norm (+SiLU) in the epilogue of its first
     * conv where one CTA holds all <= 144 channels of a pixel (vae_conv3x3_nhwc_rms:
     * on rows of >= 128 pixels two passes over the accumulator in TMEM with f16
     * rows stored by TMA, else a register-held pixel row), instead of writing the
     * f32 conv output and normalising it in a separate kernel. Same bits either
     * way. Off by default: on GB300 the conv with the norm in its epilogue takes
     * longer than the conv plus the separate norm. */
    VAE_DECODE_FUSE_NORM = 4,
    /* Run the up convs in their sub-pixel form (four 2x2 convs with summed
     * weights, see vae_pack_subpixel_weights): 4/9 of their MACs, the weight sums
     * rounded to f16 once. Off by default (it changes the rounding). */
    VAE_DECODE_SUBPIXEL_UP = 8,
    /* With VAE_DECODE_PROFILE: record events only around the full-resolution
     * ResNet convs (3x3, cin == cout, output rows as wide as the image), so a
     * timed decode carries 2 events per such launch instead of 2 per stage. */
    VAE_DECODE_PROFILE_FULLRES = 16
};

/* Stage kinds of a profiled decode. */
enum {
    VAE_STAGE_CONV3X3 = 0,   /* one implicit-GEMM 3x3 conv launch (incl. up convs) */
    VAE_STAGE_CONV1X1 = 1,   /* one 1x1 conv launch (post_quant, shortcut) */
    VAE_STAGE_NORM = 2,      /* RMS_norm (1 launch) or GroupNorm (3 launches) */
    VAE_STAGE_CAST = 3,      /* guarded f32 -> f16 cast of the raw stream */
    VAE_STAGE_ATTENTION = 4, /* the whole mid attention (norm, projections, fused core) */
    VAE_STAGE_LAYOUT = 5,    /* latent NCHW f32 -> NHWC f16 */
    VAE_STAGE_COPY = 6       /* band input rows copied from the saved stream */
};

/* One stage of a profiled decode. `flops` are the algorithmic FLOPs
 * (2*M*N*K with real channels, upsample convs counted on the output grid;
 * attention 4*m^2*c plus 2*m*c^2 per projection); `bytes` the algorithmic
 * HBM bytes of bandwidth-bound stages (0 for convs). */
typedef struct {
    int kind;
    int launches;
    int h, w;       /* output grid of the stage */
    int cin, cout;  /* channels */
    double flops;
    double bytes;
    float ms;       /* device time between the stage's start and end events */
} vae_stage_record;

/* Records accumulate over every decode run with VAE_DECODE_PROFILE on this
 * handle. This call synchronises on their events and sets *n_recs to how many
 * there are; with max_recs > 0 it copies up to max_recs of them (in launch
 * order) and then clears them all (max_recs = 0 only counts). Not thread-safe
 * per handle. */
int vae_decode_profile(vae_decoder_t dec, vae_stage_record* recs, int max_recs, int* n_recs);

/* Device workspace (bytes) vae_decode needs for an h0 x w0 latent. */
int vae_decode_workspace(vae_decoder_t dec, int h0, int w0, const vae_decode_opts* opts,
                         size_t* bytes);

/*
 * Decode one latent frame ("qi21_vae.rs" decode, "vae.rs" VaeDecoder::decode).
 *   z_dev   f32 NCHW [latent_channels][h0][w0] (device)
 *   out_dev f32 NCHW [nch][h0 << ups][w0 << ups] (device), nch = conv_out cout
 *   opts    NULL = whole frame, guard 8.
 * A banded decode writes the same kept rows bit for bit as the whole-frame one.
 */
int vae_decode(vae_decoder_t dec, const float* z_dev, int h0, int w0, float* out_dev,
               const vae_decode_opts* opts, void* workspace_dev, size_t workspace_bytes,
               vae_stream_t stream);

/* As vae_decode with HOST z and out: copies z in, decodes, copies out and
 * synchronises `stream` (the end-to-end call). */
int vae_decode_host(vae_decoder_t dec, const float* z_host, int h0, int w0, float* out_host,
                    const vae_decode_opts* opts, void* workspace_dev, size_t workspace_bytes,
                    vae_stream_t stream);

/*
 * A decode captured once as a CUDA graph and replayed: the buffers (z_dev,
 * out_dev, workspace_dev), the sizes and the options are fixed at capture;
 * every launch reads z_dev and writes out_dev as vae_decode would (same bits).
 * Replays skip the host's per-kernel work and the launch gaps between the
 * decode's ~70 kernels, which matters for small frames.
 * vae_decode_graph_create runs one eager vae_decode on `stream` (validating
 * every argument and doing the one-time kernel set-up), then captures the
 * decode on a private stream; no profile flag. The graph may be launched on
 * any stream of the same device; the caller orders it against other work on
 * the buffers. Errors as vae_decode; on error *graph is NULL.
 */
typedef struct vae_decode_graph* vae_decode_graph_t;
int vae_decode_graph_create(vae_decoder_t dec, const float* z_dev, int h0, int w0, float* out_dev,
                            const vae_decode_opts* opts, void* workspace_dev, size_t workspace_bytes,
                            vae_stream_t stream, vae_decode_graph_t* graph);
int vae_decode_graph_launch(vae_decode_graph_t graph, vae_stream_t stream);
int vae_decode_graph_destroy(vae_decode_graph_t graph);

#ifdef __cplusplus
}
#endif

#endif /* VAE_IGEMM_H */

// NHWC implicit-GEMM convolution (3x3 or 1x1, stride 1) on sm_103a tensor cores.
//
// What it computes ("vae.rs" Conv2d::apply; "qi21_vae.rs" conv_s and the
// module doc's implicit-GEMM recipe): GEMM with M = output pixels,
// N = cout, K = taps * cin in (tap, channel) order, f16 inputs, f32
// accumulation in tensor memory, and a fused epilogue
//   y = SiLU?(oscale * acc + bias + residual [+ DupUp(src)])  -> f32 | f16 | NCHW f32.
//
// How (a GB300 design, not the pages' wgpu one):
//  - M tiles are R rows x Wt columns of a "virtual grid" (R*Wt <= 128). For a
//    plain conv the virtual grid is the output grid. For the nearest-2x fold
//    it is the SOURCE grid, taken once per output parity class (q, p): output
//    (2v+q, 2u+p) reads, for tap (ky, kx), source (v + dy, u + dx) with
//    dy = floor((q+ky-1)/2), dx = floor((p+kx-1)/2). So every tap of every
//    tile is a dense rectangular box of the f16 input and the whole gather
//    is a 4-D TMA tile load; zero padding comes from TMA's out-of-bounds fill.
//  - Replicate padding and the encoder's stride-2 downsample remap source
//    coordinates per pixel, which a box cannot express; those launches use
//    128 gather threads instead (one A row each, 16-byte loads, stores into the
//    128B-swizzled layout). Reflect padding on rows of >= 128 pixels keeps the
//    halo boxes: the producer mirrors the row coordinate, and a fixer warp
//    copies the mirrored edge column inside each landed box (column -1 <- 1,
//    W <- W - 2) and passes the stage on to the MMA thread (whose own proxy
//    fence would stall the tensor pipe); smaller grids gather.
//  - The encoder's stride-2 downsample on even widths with >= 128 output
//    columns: x viewed as (channel, column parity, W/2, row, image) makes tap
//    (ky, kx) of 128 output pixels one box (parity kx & 1, first column
//    u0 + kx / 2, row 2v + ky); the far-side pad is TMA's zero fill, or, for
//    reflect padding, the mirrored row coordinate and one row copy by the
//    fixer warp (column W <- W - 2 sits one row before it in the kx = 2 box).
//  - B (weights [cout][taps][cin]) is a 3-D TMA tile load per (tap, chunk).
//  - One elected thread issues tcgen05.mma (M=128, N=BN, K=16 steps) into one
//    of two TMEM accumulators; four epilogue warps drain the other
//    (tcgen05.ld), so the epilogue of tile i overlaps the MMAs of tile i+1.
//  - Persistent CTAs (one per SM) walk the tile list with a fixed stride; an
//    S-stage mbarrier ring pipelines TMA against the MMAs.
//  - Each output element's value depends only on its own receptive field and
//    the K order, never on the tile it falls in, so banded decodes are
//    bit-identical to whole-frame ones.
//  - Every wait is bounded (mbar_wait); on a timeout the CTA drains its own
//    TMA copies and MMAs, frees TMEM and returns with the status recorded.
#include <algorithm>
#include <cstdio>
#include <cmath>
#include <cstdlib>

#include "vae_conv.h"
#include "vae_norm.h"
#include "vae_rms.cuh"

namespace vae {

namespace {

constexpr int kBK = 64;                // channels per K chunk (one 128-byte swizzle row)
constexpr int kBM = 128;               // M tile (UMMA M)
constexpr int kABytes = kBM * kBK * 2; // 16 KB
constexpr int kMaxStages = 12;       // B (or shared A+B) ring slots
constexpr int kMaxAStages = 4;       // A halo ring slots (halo mode)
constexpr int kHaloRows = 130;       // one output row segment of 128 pixels + a pixel each side
constexpr int kHaloBytes = 17408;    // 130 rows x 128 B, rounded up to 1024 B
constexpr int kTail = 512;           // barriers, TMEM slot and abort flag
constexpr int kRemAStride = 4352;    // one 16-channel halo box (130 rows x 32 B), rounded up to 256 B
constexpr uint32_t kRemABytes = kHaloRows * 32;
constexpr int kStgBytes = 2048;      // 32 pixels x 16 f32 channels, 64-byte swizzle

// Kernel variants: A tile per tap by TMA; A tile per tap by gather threads
// (replicate padding); one A "halo" box per (ky, chunk) shared by the three
// kx taps through descriptor start offsets of whole 128-byte rows.
constexpr int kModeTma = 0, kModeGather = 1, kModeHalo = 2;
// Variants (the kernel's kVar): 0 the 2-D conv, 1 the 3x3x3 conv, 2 the
// sub-pixel up conv, 3 the 2-D conv whose epilogue also emits GroupNorm
// partial statistics of its output.
constexpr bool is_2d(int var) { return var == 0 || var == 3; }
constexpr int kEpiWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kGatherWarp0 = 6;
constexpr int kMaxSmem = 232448;       // 227 KB opt-in per CTA
#ifndef VAE_GEMM_PAIR_KS
#define VAE_GEMM_PAIR_KS 2
#endif
constexpr int kGemmPairKs = VAE_GEMM_PAIR_KS;  // 64-channel chunks per stage of the pair GEMM
#ifndef VAE_GEMM_PAIR_PREFETCH
#define VAE_GEMM_PAIR_PREFETCH 1
#endif
constexpr bool kGemmPairPrefetch = VAE_GEMM_PAIR_PREFETCH != 0;  // L2 prefetch of the A rows one tile ahead

struct ConvParams {
    int n, hv, wv;        // images, virtual grid rows/cols (= input grid)
    int cin, cout, taps;  // taps: 9 or 1
    int up, rep;          // nearest-2x fold, replicate padding
    int refl, down;       // reflect padding; the stride-2 downsample (far-side pad; virtual grid = output)
    int down_tma;         // the downsample's taps as TMA boxes of a (channel, column parity, W/2, row, image) view
    int hs, ws;           // source grid of the gather (= hv, wv except for the downsample)
    int H, W;             // output grid
    int R, Wt;            // tile rows, tile cols on the virtual grid
    int tiles_x, tiles_y, npar;
    int n_tiles, BN, acc_stride;
    int kchunks, total_tiles, stages;
    int frames_out, frames_in, t_up, nkt;  // 3-D causal conv: output / input frames per image, temporal 2x,
                                            // temporal taps (3; 1 for 2-D convs, whose frames are 1)
    int n_in;             // input images (batch x input frames; = n for 2-D convs)
    int subpix;           // up conv as four 2x2 convs on the source grid (weights [cout][16][cin]):
                          // tap (ty, tx) of parity class par reads source (v + dymin + ty, u + dxmin + tx)
    int rem16, kfull;     // three-tap halo stages with cin % 64 == 16: kfull 64-channel chunks, then one
                          // stage of 16-channel boxes (32-byte swizzle) for all three ky and nine taps
    int halo, a_stages;   // halo mode: a_stages halo boxes; B ring of `stages` x ks taps
                          // (ks == 3: box slot i belongs to stage i, one barrier pair)
    int ks;               // K chunks per pipeline stage (per-tap A path: 1 or 2; pair GEMM mode: up to kGemmPairKs)
    int pair;             // CTA-pair kernel: each CTA holds BN/2 rows of B (b_rows)
    int gemm;             // pair kernel on a 1x1 conv over one row of pixels (a plain GEMM): the two CTAs
                          // take adjacent 128-pixel column tiles; a stage holds ks 64-channel chunks
    int stg_bytes;        // epilogue staging boxes in shared memory (0 without the TMA epilogue)
    int b_rows, typ_tiles, pair_tiles;
    uint32_t a_tx;        // bytes one A box delivers
    const __half* x;      // gather source
    const float* bias;
    const float* residual;
    void* y;
    float oscale;
    int silu, out_f16, vec_ok;
    float out_scale;      // f16 output: stored value x out_scale
    int res_prefetch;     // L2-prefetch each tile's residual span (one row, all channels)
    int dup_prefetch;     // L2-prefetch each tile's DupUp source span (one source row)
    int dup_step;         // DupUp: source channel = dup_base[2q+p] + dup_step * o (1 or 2), or 0
    int dup_base[4];
    int dup_v8;           // DupUp rows 32-byte aligned: 32-byte loads of the source window
    int v8_ok;            // f32 y / residual rows 32-byte aligned: 32-byte accesses
    int epi_tma;          // epilogue writes through staged TMA boxes: 1 store, 2 add onto y (residual == y),
                          // 3 the fused RMS_norm's f16 rows (rms_out)
    int bias_smem;        // the bias (cout floats) is copied to shared memory at kernel start
    // NCHW output of kept rows (conv_out): rows [keep_lo, keep_hi) land at
    // destination row (Y - keep_lo + dst_row0) of planes `plane` floats apart.
    int out_nchw, keep_lo, keep_hi, dst_row0;
    long long plane;
    // DupUp add (the RMS-family up conv): src f32 [n][hv][wv][dup_cin].
    const float* dup_src;
    int dup_cin, dup_factor, dup_repeats, dup_ftoff;
    // Fused RMS_norm of the output pixel (cout <= kRmsMaxC, one N tile): f16
    // SiLU?(y * sqrt(C) / max(||y||, 1e-12) * gamma) into rms_out [pixels][cout].
    const float* rms_gamma;
    __half* rms_out;
    int rms_silu;
    // GroupNorm partial statistics of the output (variant 3): per (image,
    // chunk = M tile * 4 + epilogue warp, group) one record (count, K, S1, S2):
    // shifted sums S1 = sum (v - K), S2 = sum (v - K)^2.
    float4* gn_part;
    int gn_groups, gn_cpg, gn_nchunks;
    DevStatus* status;
    unsigned long long timeout_ns;
};

struct TileInfo {
    int img, par, v0, u0, n0;
};

// kT3: the 3x3x3 conv's instantiation (temporal taps, frames); the 2-D
// kernels compile without any of it.
template <bool kT3 = false>
__device__ __forceinline__ TileInfo decode_tile(const ConvParams& p, int t) {
    TileInfo ti;
    const int nt = t % p.n_tiles;
    int r = t / p.n_tiles;
    const int tx = r % p.tiles_x;
    r /= p.tiles_x;
    if (kT3 && p.frames_out > 1) {
        // frames vary faster than rows: the tiles in flight hold a few rows of
        // every frame, so the three temporal taps' source rows stay in L2
        const int f = r % p.frames_out;
        r /= p.frames_out;
        ti.par = r % p.npar;
        r /= p.npar;
        const int ty = r % p.tiles_y;
        ti.img = (r / p.tiles_y) * p.frames_out + f;
        ti.v0 = ty * p.R;
        ti.u0 = tx * p.Wt;
        ti.n0 = nt * p.BN;
        return ti;
    }
    ti.par = r % p.npar;
    r /= p.npar;
    const int ty = r % p.tiles_y;
    ti.img = r / p.tiles_y;
    ti.v0 = ty * p.R;
    ti.u0 = tx * p.Wt;
    ti.n0 = nt * p.BN;
    return ti;
}

// Weight tap (second coordinate of the B tensor) of kernel tap `tap` for parity
// class `par`: the sub-pixel weights hold four taps per parity class.
__device__ __forceinline__ int b_tap(const ConvParams& p, int par, int tap) { return p.subpix ? par * 4 + tap : tap; }

// Source image of output image `img` for temporal tap kt (0..2, frame f + kt - 2):
// causal, the frames before the first replicate it; with the temporal 2x the
// upsampled frame vf comes from source frame vf > 0 ? (vf - 1) / 2 + 1 : 0.
// 2-D convs (one frame) use kt = 2 only: the image itself.
template <bool kT3>
__device__ __forceinline__ int src_img(const ConvParams& p, int img, int kt) {
    if (!kT3 || p.frames_out == 1) return img;
    const int b = img / p.frames_out, f = img - b * p.frames_out;
    const int vf = max(f - 2 + kt, 0);
    const int sf = p.t_up ? (vf > 0 ? (vf - 1) / 2 + 1 : 0) : vf;
    return b * p.frames_in + sf;
}

// Source offset of tap `tap` for parity class `par` (see the file comment);
// a 3x3x3 tap is kt * 9 + ky * 3 + kx.
__device__ __forceinline__ void tap_offset(const ConvParams& p, int tap, int par, int& dy, int& dx) {
    if (p.taps == 1) {
        dy = 0;
        dx = 0;
        return;
    }
    if (p.subpix) {  // four taps per parity class: rows / columns (q|p == 0 ? -1 : 0) + {0, 1}
        dy = ((par >> 1) == 0 ? -1 : 0) + tap / 2;
        dx = ((par & 1) == 0 ? -1 : 0) + tap % 2;
        return;
    }
    const int ky = (tap % 9) / 3, kx = tap % 3;
    if (p.up) {
        const int q = par >> 1, pp = par & 1;
        dy = (q + ky + 1) / 2 - 1;
        dx = (pp + kx + 1) / 2 - 1;
    } else {
        dy = ky - 1;
        dx = kx - 1;
    }
}

struct Smem {
    uint8_t* a;          // stages x 16 KB, or (halo mode) a_stages x kHaloBytes
    uint8_t* b;          // stages x BN*128 B
    uint8_t* stg;        // epilogue staging, 2 KB per epilogue warp (epi_tma)
    float* bias;         // [cout] copy of the bias (bias_smem)
    uint64_t* full;      // [stages]
    uint64_t* empty;     // [stages]
    uint64_t* afull;     // [a_stages] (halo mode)
    uint64_t* aempty;    // [a_stages] (halo mode)
    uint64_t* accf;      // [2]
    uint64_t* acce;      // [2]
    uint64_t* drain;     // [1]
    uint64_t* fixed;     // [stages] (reflect padding: the fixer warp hands each stage to the MMA thread)
    uint64_t* xbar;      // [4] (pair kernel, fused RMS_norm: the two warps of a lane quadrant trade sums)
    uint32_t* tmem_slot;
    int* abort_flag;
};

__device__ __forceinline__ Smem carve(uint8_t* raw, const ConvParams& p) {
    Smem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.a = base;
    s.b = base + (p.halo ? p.a_stages * kHaloBytes : p.stages * p.ks * kABytes);
    s.stg = s.b + p.stages * p.ks * p.b_rows * 128;
    s.bias = reinterpret_cast<float*>(s.stg + p.stg_bytes);
    uint8_t* tail = reinterpret_cast<uint8_t*>(s.bias) + (p.bias_smem ? (p.cout * 4 + 15) / 16 * 16 : 0);
    uint64_t* bars = reinterpret_cast<uint64_t*>(tail);
    s.full = bars;
    s.empty = bars + kMaxStages;
    s.afull = bars + 2 * kMaxStages;
    s.aempty = s.afull + kMaxAStages;
    s.accf = s.aempty + kMaxAStages;
    s.acce = s.accf + 2;
    s.drain = s.acce + 2;
    s.fixed = s.drain + 1;
    s.xbar = s.fixed + kMaxStages;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.xbar + 4);
    s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
    return s;
}

// Reflect padding inside a landed halo box whose row 0 holds source column
// `cbase`: the rows of columns -1 and W take columns 1 and W - 2 (generic-proxy
// copies; the caller fences before the MMAs read the box). kRow = 128: a
// 64-channel box, 128-byte swizzle, 1024-byte aligned, so row r's 16-byte
// chunk j sits at r * 128 + ((j ^ (r & 7)) * 16). kRow = 32: a 16-channel box,
// 32-byte swizzle, 256-byte aligned: chunk j of row r at r * 32 + ((j ^ ((r >> 2) & 1)) * 16).
// Returns whether it wrote anything.
// Copies row rs of a 1024-byte-aligned, 128-byte-swizzled box onto row rd.
__device__ __forceinline__ void copy_row_sw128(uint8_t* box, int rs, int rd) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(box + sw128_off(static_cast<uint32_t>(rd), static_cast<uint32_t>(j))) =
            *reinterpret_cast<const uint4*>(box + sw128_off(static_cast<uint32_t>(rs), static_cast<uint32_t>(j)));
}

template <int kRow>
__device__ __forceinline__ bool reflect_fix_box(uint8_t* box, int cbase, int W) {
    bool fixed = false;
    auto off = [](int r, int j) -> uint32_t {
        return kRow == 128 ? sw128_off(static_cast<uint32_t>(r), static_cast<uint32_t>(j))
                           : static_cast<uint32_t>(r * 32 + ((j ^ ((r >> 2) & 1)) << 4));
    };
    auto copy_row = [&](int rs, int rd) {
#pragma unroll
        for (int j = 0; j < kRow / 16; ++j)
            *reinterpret_cast<uint4*>(box + off(rd, j)) = *reinterpret_cast<const uint4*>(box + off(rs, j));
        fixed = true;
    };
    if (cbase <= -1) copy_row(1 - cbase, -1 - cbase);
    if (W - cbase <= kHaloRows - 1) copy_row(W - 2 - cbase, W - cbase);
    return fixed;
}

// Waits on a barrier during the final drain: bounded, but not cut short by
// the abort flag (the point is to let in-flight async work land).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const ConvParams& p) {
    int never = 0;
    (void)mbar_wait(bar, parity, &never, p.timeout_ns, p.status, kWhereDrain);
}

// ───────────────────────────── roles ─────────────────────────────

// kVar: 0 the 2-D conv, 1 the 3x3x3 conv (temporal taps), 2 the sub-pixel up
// conv (2 x 2 taps per parity class). Each is its own instantiation.
template <int kMode, int kVar>
__device__ void role_producer(const ConvParams& p, const Smem& s, const CUtensorMap* mapA,
                              const CUtensorMap* mapB, const CUtensorMap* mapA16, const CUtensorMap* mapB16) {
    const uint64_t pol_w = policy_evict_last();
    const uint64_t pol_a = policy_evict_normal();
    const uint32_t b_bytes = static_cast<uint32_t>(p.BN) * 128u;
    int stage = 0, astage = 0;
    uint32_t phase = 0, aphase = 0;
    uint32_t armed = 0, arm_par = 0, aarmed = 0, aarm_par = 0;
    bool ok = true;
    // Arms the next B-ring slot for `tx` bytes; returns its barrier, or 0 on abort.
    auto next_b = [&](uint32_t tx, uint32_t* slot) -> uint32_t {
        if (!mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, s.abort_flag, p.timeout_ns, p.status,
                       kWhereProducerEmpty)) {
            ok = false;
            return 0u;
        }
        const uint32_t fb = smem_u32(&s.full[stage]);
        mbar_arrive_expect_tx(fb, tx);
        armed |= 1u << stage;
        arm_par = (arm_par & ~(1u << stage)) | (phase << stage);
        *slot = static_cast<uint32_t>(stage);
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
        }
        return fb;
    };
    for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        constexpr bool kT3 = kVar == 1;
        constexpr int NK = kVar == 2 ? 2 : 3;  // ky and kx taps per stage row
        const TileInfo ti = decode_tile<kT3>(p, t);
        if (p.res_prefetch) {
            // The tile's residual rows, one contiguous span, are pulled into L2 now
            // so the epilogue (a mainloop later) reads them at L2 latency.
            const int npx = min(p.Wt, p.wv - ti.u0);
            const long long pix0 = (static_cast<long long>(ti.img) * p.H + ti.v0) * p.W + ti.u0;
            prefetch_l2_bulk(p.residual + pix0 * p.cout, static_cast<uint32_t>(npx * p.cout * 4));
        }
        if (p.dup_prefetch) {  // likewise the DupUp source pixels of the tile (source grid)
            const int npx = min(p.Wt, p.wv - ti.u0);
            const long long pix0 = (static_cast<long long>(ti.img) * p.hv + ti.v0) * p.wv + ti.u0;
            prefetch_l2_bulk(p.dup_src + pix0 * p.dup_cin, static_cast<uint32_t>(npx * p.dup_cin * 4));
        }
        if (kMode == kModeHalo && p.ks == 3) {
            // one stage = the halo box of (ky, chunk) and the three kx taps' weights
            const int q = ti.par >> 1, pp = ti.par & 1;
            const int dxmin = (p.up && pp == 1) ? 0 : -1;
            const int kc_end = p.rem16 ? p.kfull : p.kchunks;
            const int nkt = kT3 ? p.nkt : 1;
            const int dymin = q == 0 ? -1 : 0;  // the sub-pixel variant's first source row
            for (int kt = 0; kt < nkt && ok; ++kt) {
                const int simg = src_img<kT3>(p, ti.img, kt + 3 - nkt);
                for (int ky = 0; ky < NK && ok; ++ky) {
                    const int dy = kVar == 2 ? dymin + ky : (p.up ? (q + ky + 1) / 2 - 1 : ky - 1);
                    int sy = ti.v0 + dy;
                    if (is_2d(kVar) && p.refl) sy = sy < 0 ? -sy : (sy >= p.hs ? 2 * (p.hs - 1) - sy : sy);
                    for (int kc = 0; kc < kc_end && ok; ++kc) {
                        uint32_t slot;
                        const uint32_t fb = next_b(p.a_tx + static_cast<uint32_t>(NK) * b_bytes, &slot);
                        if (!ok) break;
                        tma_load_4d(smem_u32(s.a + slot * kHaloBytes), mapA, fb, kc * kBK, ti.u0 + dxmin, sy,
                                    simg, pol_a);
                        for (int kx = 0; kx < NK; ++kx)
                            tma_load_3d(smem_u32(s.b + (slot * 3 + kx) * p.BN * 128), mapB, fb, kc * kBK,
                                        kVar == 2 ? ti.par * 4 + ky * 2 + kx : kt * 9 + ky * 3 + kx, ti.n0, pol_w);
                    }
                }
                if (p.rem16 && ok) {
                    // the last 16 channels of all ky rows and (ky, kx) taps in one stage
                    uint32_t slot;
                    const uint32_t fb = next_b(static_cast<uint32_t>(NK) * kRemABytes +
                                                   static_cast<uint32_t>(NK * NK) * static_cast<uint32_t>(p.BN) * 32u,
                                               &slot);
                    if (ok) {
                        for (int ky = 0; ky < NK; ++ky) {
                            const int dy = kVar == 2 ? dymin + ky : (p.up ? (q + ky + 1) / 2 - 1 : ky - 1);
                            int sy = ti.v0 + dy;
                            if (is_2d(kVar) && p.refl) sy = sy < 0 ? -sy : (sy >= p.hs ? 2 * (p.hs - 1) - sy : sy);
                            tma_load_4d(smem_u32(s.a + slot * kHaloBytes + ky * kRemAStride), mapA16, fb,
                                        p.kfull * kBK, ti.u0 + dxmin, sy, simg, pol_a);
                        }
                        for (int tap = 0; tap < NK * NK; ++tap)
                            tma_load_3d(smem_u32(s.b + slot * 3 * p.BN * 128 + tap * p.BN * 32), mapB16, fb,
                                        p.kfull * kBK, kVar == 2 ? ti.par * 4 + tap : kt * 9 + tap, ti.n0, pol_w);
                    }
                }
            }
        } else if (kMode == kModeHalo) {
            const int q = ti.par >> 1, pp = ti.par & 1;
            const int dxmin = (p.up && pp == 1) ? 0 : -1;
            const int nkt = kT3 ? p.nkt : 1;
            for (int kt = 0; kt < nkt && ok; ++kt) {
                const int simg = src_img<kT3>(p, ti.img, kt + 3 - nkt);
                for (int ky = 0; ky < 3 && ok; ++ky) {
                    const int dy = p.up ? (q + ky + 1) / 2 - 1 : ky - 1;
                    for (int kc = 0; kc < p.kchunks && ok; ++kc) {
                        if (!mbar_wait(smem_u32(&s.aempty[astage]), aphase ^ 1u, s.abort_flag, p.timeout_ns,
                                       p.status, kWhereProducerEmpty)) {
                            ok = false;
                            break;
                        }
                        const uint32_t afb = smem_u32(&s.afull[astage]);
                        mbar_arrive_expect_tx(afb, p.a_tx);
                        aarmed |= 1u << astage;
                        aarm_par = (aarm_par & ~(1u << astage)) | (aphase << astage);
                        tma_load_4d(smem_u32(s.a + astage * kHaloBytes), mapA, afb, kc * kBK, ti.u0 + dxmin,
                                    ti.v0 + dy, simg, pol_a);
                        if (++astage == p.a_stages) {
                            astage = 0;
                            aphase ^= 1u;
                        }
                        for (int kx = 0; kx < 3; ++kx) {
                            uint32_t slot;
                            const uint32_t fb = next_b(b_bytes, &slot);
                            if (!ok) break;
                            tma_load_3d(smem_u32(s.b + slot * p.BN * 128), mapB, fb, kc * kBK, kt * 9 + ky * 3 + kx,
                                        ti.n0, pol_w);
                        }
                    }
                }
            }
        } else {
            for (int tap = 0; tap < p.taps && ok; ++tap) {
                int dy, dx;
                tap_offset(p, tap, ti.par, dy, dx);
                const int simg = src_img<kT3>(p, ti.img, p.taps == 27 ? tap / 9 : 2);
                for (int kc = 0; kc < p.kchunks; kc += p.ks) {
                    // one stage = up to ks consecutive 64-channel chunks of this tap
                    const int nck = min(p.ks, p.kchunks - kc);
                    uint32_t slot;
                    const uint32_t fb =
                        next_b(static_cast<uint32_t>(nck) * (b_bytes + (kMode == kModeGather ? 0u : p.a_tx)), &slot);
                    if (!ok) break;
                    for (int h = 0; h < nck; ++h) {
                        if (kMode == kModeTma && is_2d(kVar) && p.down_tma) {
                            // tap (ky, kx) = (dy + 1, dx + 1): column parity kx & 1, first column u0 + kx / 2
                            int sy = 2 * ti.v0 + dy + 1;
                            if (p.refl && sy >= p.hs) sy = 2 * (p.hs - 1) - sy;
                            tma_load_5d(smem_u32(s.a + (slot * p.ks + h) * kABytes), mapA, fb, (kc + h) * kBK,
                                        (dx + 1) & 1, ti.u0 + ((dx + 1) >> 1), sy, simg, pol_a);
                        } else if (kMode == kModeTma)
                            tma_load_4d(smem_u32(s.a + (slot * p.ks + h) * kABytes), mapA, fb, (kc + h) * kBK,
                                        ti.u0 + dx, ti.v0 + dy, simg, pol_a);
                        tma_load_3d(smem_u32(s.b + (slot * p.ks + h) * p.BN * 128), mapB, fb, (kc + h) * kBK,
                                    b_tap(p, ti.par, tap), ti.n0, pol_w);
                    }
                }
            }
        }
    }
    // Let every copy this thread started land before the CTA can exit.
    for (int st = 0; st < p.stages; ++st)
        if (armed & (1u << st)) drain_wait(smem_u32(&s.full[st]), (arm_par >> st) & 1u, p);
    if (kMode == kModeHalo)
        for (int st = 0; st < p.a_stages; ++st)
            if (aarmed & (1u << st)) drain_wait(smem_u32(&s.afull[st]), (aarm_par >> st) & 1u, p);
}

// One thread per A row: gathers the row's 64-channel slice for each
// (tap, chunk) with clamped (replicate), mirrored (reflect) or zero-filled
// (zero) borders. The downsample's row v reads source rows 2v + ky (the far
// side padded by one); every other conv's reads v + dy.
template <int kVar>
__device__ void role_gather(const ConvParams& p, const Smem& s, int gt) {
    constexpr bool kT3 = kVar == 1;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile<kT3>(p, t);
        const int rr = gt / p.Wt, cc = gt % p.Wt;
        const int v = ti.v0 + rr, u = ti.u0 + cc;
        const bool rowvalid = gt < p.R * p.Wt && v < p.hv && u < p.wv;
        for (int tap = 0; tap < p.taps && ok; ++tap) {
            int dy, dx;
            tap_offset(p, tap, ti.par, dy, dx);
            const int simg = src_img<kT3>(p, ti.img, p.taps == 27 ? tap / 9 : 2);
            int sy = p.down ? 2 * v + dy + 1 : v + dy, sx = p.down ? 2 * u + dx + 1 : u + dx;
            bool inb;
            if (p.rep) {
                sy = min(max(sy, 0), p.hs - 1);
                sx = min(max(sx, 0), p.ws - 1);
                inb = rowvalid;
            } else if (p.refl) {  // at most one pixel outside (hs, ws >= 2): one mirror suffices
                sy = sy < 0 ? -sy : (sy >= p.hs ? 2 * (p.hs - 1) - sy : sy);
                sx = sx < 0 ? -sx : (sx >= p.ws ? 2 * (p.ws - 1) - sx : sx);
                inb = rowvalid;
            } else {
                inb = rowvalid && sy >= 0 && sy < p.hs && sx >= 0 && sx < p.ws;
            }
            const __half* src =
                p.x + ((static_cast<long long>(simg) * p.hs + (inb ? sy : 0)) * p.ws + (inb ? sx : 0)) *
                          p.cin;
            for (int kc = 0; kc < p.kchunks; ++kc) {
                if (!mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, s.abort_flag, p.timeout_ns,
                               p.status, kWhereGatherEmpty)) {
                    ok = false;
                    break;
                }
                uint8_t* dst = s.a + stage * kABytes;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c = kc * kBK + j * 8;
                    uint4 val = make_uint4(0u, 0u, 0u, 0u);
                    if (inb && c < p.cin) val = __ldg(reinterpret_cast<const uint4*>(src + c));
                    *reinterpret_cast<uint4*>(dst + sw128_off(static_cast<uint32_t>(gt), j)) = val;
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&s.full[stage]));
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
}

// Reflect padding on the three-tap halo stages: for every stage, in ring order,
// waits for the landed copies, mirrors the edge columns of edge tiles' boxes,
// and hands the stage to the MMA thread (the `fixed` barrier completes once per
// use of a slot, in lockstep with `full`).
__device__ void role_fixer(const ConvParams& p, const Smem& s) {
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    if (!p.halo) {
        // the reflect-padded downsample's per-tap stages: in the last column tile
        // the kx = 2 boxes' row of column W takes column W - 2 (the row before it)
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            const TileInfo ti = decode_tile<false>(p, t);
            const int i = p.wv - 1 - ti.u0;  // the row holding the last output pixel
            const bool edge = (p.ws % 2 == 0) && i >= 1 && i < kBM;
            for (int tap = 0; tap < p.taps && ok; ++tap)
                for (int kc = 0; kc < p.kchunks; kc += p.ks) {
                    if (!mbar_wait(smem_u32(&s.full[stage]), phase, s.abort_flag, p.timeout_ns, p.status,
                                   kWhereFixer)) {
                        ok = false;
                        break;
                    }
                    if (edge && tap % 3 == 2) {
                        const int nck = min(p.ks, p.kchunks - kc);
                        for (int h = 0; h < nck; ++h) copy_row_sw128(s.a + (stage * p.ks + h) * kABytes, i - 1, i);
                        fence_proxy_async_smem();
                    }
                    mbar_arrive(smem_u32(&s.fixed[stage]));
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
        }
        return;
    }
    for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile<false>(p, t);
        const bool edge = ti.u0 == 0 || ti.u0 + kBM >= p.ws;
        const int nfull = 3 * (p.rem16 ? p.kfull : p.kchunks);
        for (int i = 0; i < nfull + (p.rem16 ? 1 : 0); ++i) {
            if (!mbar_wait(smem_u32(&s.full[stage]), phase, s.abort_flag, p.timeout_ns, p.status, kWhereFixer)) {
                ok = false;
                break;
            }
            if (edge) {
                uint8_t* box = s.a + stage * kHaloBytes;
                bool fixed = false;
                if (i < nfull) {
                    fixed = reflect_fix_box<128>(box, ti.u0 - 1, p.ws);
                } else {  // the 16-channel remainder stage: one 32-byte-swizzled box per ky
                    for (int ky = 0; ky < 3; ++ky) fixed |= reflect_fix_box<32>(box + ky * kRemAStride, ti.u0 - 1, p.ws);
                }
                if (fixed) fence_proxy_async_smem();
            }
            mbar_arrive(smem_u32(&s.fixed[stage]));
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

template <int kVar>
__device__ void role_mma(const ConvParams& p, const Smem& s, uint32_t tmem_base) {
    constexpr bool kT3 = kVar == 1;
    constexpr int NK = kVar == 2 ? 2 : 3;  // ky and kx taps per stage row
    const uint32_t idesc = idesc_f16_f32(kBM, p.BN);
    int stage = 0, astage = 0;
    uint32_t phase = 0, aphase = 0;
    int accbuf = 0;
    uint32_t accphase = 0;
    bool ok = true;
    // Issues the MMAs of one B-ring slot: chunk kc0 (and the next ones of the
    // slot, per-tap path) against the A tile at `a_addr` (halo) or in the slot.
    // reflect-padded downsample: stages come through the fixer warp
    const uint64_t* tap_ready = (is_2d(kVar) && p.refl && p.down_tma) ? s.fixed : s.full;
    // Three-tap halo stages: descriptors of slot 0 and slot strides. The
    // start-address field counts 16-byte units and every address here stays
    // below 2^18 bytes, so offsets add without carry.
    const uint64_t h_a128 = sw128_kmajor_desc(smem_u32(s.a));
    const uint64_t h_b128 = sw128_kmajor_desc(smem_u32(s.b));
    const uint64_t h_a32 = sw32_kmajor_desc(smem_u32(s.a));
    const uint64_t h_b32 = sw32_kmajor_desc(smem_u32(s.b));
    const uint32_t h_aslot = kHaloBytes >> 4;
    const uint32_t h_bslot = static_cast<uint32_t>(3 * p.BN * 128) >> 4;
    const uint32_t h_btap = static_cast<uint32_t>(p.BN * 128) >> 4;
    const uint32_t h_btap16 = static_cast<uint32_t>(p.BN * 32) >> 4;
    uint32_t h_soff_a = 0, h_soff_b = 0;  // the current slot's offsets, in descriptor units
    auto h_advance = [&]() {
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
            h_soff_a = 0;
            h_soff_b = 0;
        } else {
            h_soff_a += h_aslot;
            h_soff_b += h_bslot;
        }
    };
    auto mma_slot = [&](uint32_t d, bool halo_a, uint32_t a_addr, int kc0, int nck, int& kit) {
        if (!mbar_wait(smem_u32(&tap_ready[stage]), phase, s.abort_flag, p.timeout_ns, p.status, kWhereMmaFull)) {
            ok = false;
            return;
        }
        tc_fence_after();
        for (int h = 0; h < nck; ++h) {
            const int nk = min(4, (p.cin - (kc0 + h) * kBK) / 16);
            const uint64_t ad = sw128_kmajor_desc(halo_a ? a_addr : smem_u32(s.a + (stage * p.ks + h) * kABytes));
            const uint64_t bd = sw128_kmajor_desc(smem_u32(s.b + (stage * p.ks + h) * p.BN * 128));
            for (int k = 0; k < nk; ++k)
                umma_f16(d, ad + static_cast<uint64_t>(2 * k), bd + static_cast<uint64_t>(2 * k), idesc,
                         (kit | h | k) != 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&s.empty[stage]));
        ++kit;
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
        }
    };
    for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        if (!mbar_wait(smem_u32(&s.acce[accbuf]), accphase ^ 1u, s.abort_flag, p.timeout_ns, p.status,
                       kWhereMmaAccEmpty))
            break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(accbuf * p.acc_stride);
        int kit = 0;
        if (p.halo && p.ks == 3) {
            // Three-tap stages with running descriptors (slot strides added, no
            // per-stage recomputation): the issuing thread's own work between
            // MMAs bounds this loop at N <= 144.
            const int pp = (p.up || kVar == 2) ? decode_tile<kT3>(p, t).par & 1 : 0;
            const int dxmin = (p.up && pp == 1) ? 0 : -1;
            const int kc_end = p.rem16 ? p.kfull : p.kchunks;
            const int nk_last = min(4, (p.cin - (kc_end - 1) * kBK) / 16);
            // reflect padding: the fixer warp has mirrored the edge columns; wait for it
            const uint64_t* ready = (is_2d(kVar) && p.refl) ? s.fixed : s.full;
            uint32_t rel[NK];  // row offset of tap kx inside the halo box, in box rows
#pragma unroll
            for (int kx = 0; kx < NK; ++kx)
                rel[kx] = static_cast<uint32_t>(kVar == 2 ? kx : (p.up ? (pp + kx + 1) / 2 - 1 : kx - 1) - dxmin);
            uint32_t acc = 0u;  // the tile's first MMA overwrites the accumulator
            for (int kt = 0; kt < (kT3 ? p.nkt : 1) && ok; ++kt) {  // temporal taps (3-D); one pass for 2-D
                for (int ky = 0; ky < NK && ok; ++ky) {
                    for (int kc = 0; kc < kc_end; ++kc) {
                        if (!mbar_wait(smem_u32(&ready[stage]), phase, s.abort_flag, p.timeout_ns, p.status,
                                       kWhereMmaFull)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = h_a128 + h_soff_a;
                        const uint64_t bd = h_b128 + h_soff_b;
                        if (kc + 1 < kc_end || nk_last == 4) {
#pragma unroll
                            for (int kx = 0; kx < NK; ++kx)
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    umma_f16(d, ad + rel[kx] * 8u + 2u * k, bd + kx * h_btap + 2u * k, idesc, acc);
                                    acc = 1u;
                                }
                        } else {
                            for (int kx = 0; kx < NK; ++kx)
                                for (int k = 0; k < nk_last; ++k) {
                                    umma_f16(d, ad + rel[kx] * 8u + 2u * k, bd + kx * h_btap + 2u * k, idesc, acc);
                                    acc = 1u;
                                }
                        }
                        umma_commit(smem_u32(&s.empty[stage]));
                        h_advance();
                    }
                }
                if (p.rem16 && ok) {
                    if (!mbar_wait(smem_u32(&ready[stage]), phase, s.abort_flag, p.timeout_ns, p.status,
                                   kWhereMmaFull)) {
                        ok = false;
                    } else {
                        tc_fence_after();
                        // one K = 16 step per tap; the 64-channel chunks came first, so always accumulate:
                        // box ky at ky * kRemAStride, 32-byte rows; tap (ky, kx) weights at (ky * NK + kx) * BN * 32
                        const uint64_t ad = h_a32 + h_soff_a;
                        const uint64_t bd = h_b32 + h_soff_b;
#pragma unroll
                        for (int ky = 0; ky < NK; ++ky)
#pragma unroll
                            for (int kx = 0; kx < NK; ++kx)
                                umma_f16(d, ad + static_cast<uint32_t>(ky * (kRemAStride >> 4)) + rel[kx] * 2u,
                                         bd + static_cast<uint32_t>(ky * NK + kx) * h_btap16, idesc, 1u);
                        umma_commit(smem_u32(&s.empty[stage]));
                        h_advance();
                    }
                }
            }
        } else if (p.halo) {
            const int pp = decode_tile<kT3>(p, t).par & 1;
            const int dxmin = (p.up && pp == 1) ? 0 : -1;
            for (int kt = 0; kt < (kT3 ? p.nkt : 1) && ok; ++kt)
                for (int ky = 0; ky < 3 && ok; ++ky) {
                    for (int kc = 0; kc < p.kchunks && ok; ++kc) {
                        if (!mbar_wait(smem_u32(&s.afull[astage]), aphase, s.abort_flag, p.timeout_ns, p.status,
                                       kWhereMmaFull)) {
                            ok = false;
                            break;
                        }
                        const uint32_t abase = smem_u32(s.a + astage * kHaloBytes);
                        for (int kx = 0; kx < 3 && ok; ++kx) {
                            const int dx = p.up ? (pp + kx + 1) / 2 - 1 : kx - 1;
                            // a whole-row offset: the tensor core swizzles on absolute address bits
                            mma_slot(d, true, abase + static_cast<uint32_t>((dx - dxmin) * 128), kc, 1, kit);
                        }
                        if (!ok) break;
                        umma_commit(smem_u32(&s.aempty[astage]));
                        if (++astage == p.a_stages) {
                            astage = 0;
                            aphase ^= 1u;
                        }
                    }
                }
        } else {
            for (int tap = 0; tap < p.taps && ok; ++tap)
                for (int kc = 0; kc < p.kchunks && ok; kc += p.ks) mma_slot(d, false, 0u, kc, min(p.ks, p.kchunks - kc), kit);
        }
        if (!ok) break;
        umma_commit(smem_u32(&s.accf[accbuf]));
        accbuf ^= 1;
        if (accbuf == 0) accphase ^= 1u;
    }
    // Every MMA this thread issued must finish before TMEM and SMEM go away.
    umma_commit(smem_u32(s.drain));
    drain_wait(smem_u32(s.drain), 0u, p);
}

__device__ __forceinline__ void store_chunk(const ConvParams& p, long long pix, int o0, float (&v)[16],
                                            int Y, int X, int img) {
    if (p.out_nchw) {
        if (Y < p.keep_lo || Y >= p.keep_hi) return;
        float* y = static_cast<float*>(p.y);
        const long long rowoff = static_cast<long long>(Y - p.keep_lo + p.dst_row0) * p.W + X;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int o = o0 + i;
            if (o < p.cout) y[(static_cast<long long>(img) * p.cout + o) * p.plane + rowoff] = v[i];
        }
        return;
    }
    const bool full = p.vec_ok && (o0 + 16 <= p.cout);
    if (p.out_f16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= p.out_scale;
        __half* y = static_cast<__half*>(p.y) + pix * p.cout + o0;
        if (full) {
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                __half2 t = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
                h[i] = *reinterpret_cast<uint32_t*>(&t);
            }
            reinterpret_cast<uint4*>(y)[0] = make_uint4(h[0], h[1], h[2], h[3]);
            reinterpret_cast<uint4*>(y)[1] = make_uint4(h[4], h[5], h[6], h[7]);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (o0 + i < p.cout) y[i] = __float2half_rn(v[i]);
        }
    } else {
        float* y = static_cast<float*>(p.y) + pix * p.cout + o0;
        if (full && p.v8_ok) {
            st_v8_f32(y, v);
            st_v8_f32(y + 8, v + 8);
        } else if (full) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                reinterpret_cast<float4*>(y)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (o0 + i < p.cout) y[i] = v[i];
        }
    }
}

// The epilogue value of 16 output channels o0.. of one pixel: oscale * acc +
// bias + residual + DupUp, then SiLU (channels >= cout are left unspecified).
// `pre_res`, when given, holds the chunk's 16 residual values already loaded.
// kWide: the register-hungrier 32-byte DupUp window loads (off in the
// 320-thread gather kernel).
template <bool kWide = true>
__device__ __forceinline__ void compute_chunk(const ConvParams& p, const TileInfo& ti, const uint32_t (&r)[16],
                                              int o0, int v, int u, int q, int pp, long long pix, float (&val)[16],
                                              const float* pre_res = nullptr, const float* sbias = nullptr) {
#pragma unroll
    for (int i = 0; i < 16; ++i) val[i] = __uint_as_float(r[i]) * p.oscale;
    const bool full = p.vec_ok && (o0 + 16 <= p.cout);
    if (sbias != nullptr && full) {  // the shared-memory copy of the bias
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 b = reinterpret_cast<const float4*>(sbias + o0)[i];
            val[4 * i] += b.x;
            val[4 * i + 1] += b.y;
            val[4 * i + 2] += b.z;
            val[4 * i + 3] += b.w;
        }
    } else if (p.bias != nullptr) {
        if (full) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 b = __ldg(reinterpret_cast<const float4*>(p.bias + o0) + i);
                val[4 * i] += b.x;
                val[4 * i + 1] += b.y;
                val[4 * i + 2] += b.z;
                val[4 * i + 3] += b.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (o0 + i < p.cout) val[i] += __ldg(p.bias + o0 + i);
        }
    }
    if (pre_res != nullptr) {
#pragma unroll
        for (int i = 0; i < 16; ++i) val[i] += pre_res[i];
    } else if (p.residual != nullptr && p.epi_tma != 2) {
        const float* rs = p.residual + pix * p.cout + o0;
        if (full && p.v8_ok) {
            float r8[16];
            ld_v8_f32(rs, r8);
            ld_v8_f32(rs + 8, r8 + 8);
#pragma unroll
            for (int i = 0; i < 16; ++i) val[i] += r8[i];
        } else if (full) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 b = reinterpret_cast<const float4*>(rs)[i];
                val[4 * i] += b.x;
                val[4 * i + 1] += b.y;
                val[4 * i + 2] += b.z;
                val[4 * i + 3] += b.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (o0 + i < p.cout) val[i] += rs[i];
        }
    }
    if (p.dup_src != nullptr && full && p.dup_step != 0) {
        // Division-free form: the 16 source channels are base + step * o, step
        // 1 or 2, so the loads have constant offsets and all go out at once.
        const float* row = p.dup_src + ((static_cast<long long>(ti.img) * p.hv + v) * p.wv + u) * p.dup_cin;
        const int b = p.dup_base[2 * q + pp];
        if (kWide && p.dup_v8 && p.dup_step == 2 && b <= 1) {
            // the 32 floats from 2*o0 (128-byte aligned) cover b + 2i, i < 16
            float t[32];
            const float* a0 = row + 2 * o0;
#pragma unroll
            for (int k = 0; k < 4; ++k) ld_v8_f32_ro(a0 + 8 * k, t + 8 * k);
            if (b != 0) {
#pragma unroll
                for (int i = 0; i < 16; ++i) val[i] += t[2 * i + 1];
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) val[i] += t[2 * i];
            }
        } else if (kWide && p.dup_v8 && p.dup_step == 1 && b == 0) {
            float t[16];
            ld_v8_f32_ro(row + o0, t);
            ld_v8_f32_ro(row + o0 + 8, t + 8);
#pragma unroll
            for (int i = 0; i < 16; ++i) val[i] += t[i];
        } else {
            const float* ds = row + static_cast<long long>(o0) * p.dup_step + b;
            if (p.dup_step == 2) {
#pragma unroll
                for (int i = 0; i < 16; ++i) val[i] += __ldg(ds + 2 * i);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) val[i] += __ldg(ds + i);
            }
        }
    } else if (p.dup_src != nullptr) {
        const float* ds =
            p.dup_src + ((static_cast<long long>(ti.img) * p.hv + v) * p.wv + u) * p.dup_cin;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int o = o0 + i;
            if (o < p.cout) {
                const int jj = o * p.dup_factor + p.dup_ftoff + 2 * q + pp;
                val[i] += __ldg(ds + jj / p.dup_repeats);
            }
        }
    }
    if (p.silu) {
#pragma unroll
        for (int i = 0; i < 16; ++i) val[i] = silu_f(val[i]);
    }
}

// Per-lane shifted sums of a group wider than 16 channels, carried across the
// chunks the group spans (K: the shift, the same in every lane).
struct GnRun {
    float K, a, q;
};

// GroupNorm partial statistics of one 16-channel chunk (channels o0..o0+15)
// of this warp's 32 pixels, as shifted sums: per group (part) of W channels,
// K = lane 0's value of the part's first channel (lane 0 is valid whenever any
// lane is: invalid pixels trail), S1 = sum (v - K) and S2 = sum (v - K)^2 over
// the valid pixels, reduced across the warp with independent shuffle chains
// (the epilogue warp is alone on its scheduler, so it pays latency, not
// issue slots). Lane 0 writes one record (count, K, S1, S2) per group; the
// merge turns it into (count, mean, M2). `npx`: the warp's valid pixels.
template <int W>
__device__ __forceinline__ void gn_chunk_w(const ConvParams& p, const TileInfo& ti, const float (&val)[16],
                                           bool valid, int o0, int chunk, int lane, float npx, GnRun& run) {
    constexpr int G = 16 / W;
    float4* rec = p.gn_part + (static_cast<long long>(ti.img) * p.gn_nchunks + chunk) * p.gn_groups;
    if (W < 16 || p.gn_cpg == 16) {
        float K[G], a[G], q[G];
#pragma unroll
        for (int k = 0; k < G; ++k) K[k] = __shfl_sync(0xffffffffu, val[k * W], 0);
#pragma unroll
        for (int k = 0; k < G; ++k) {
            float sa = 0.f, sq = 0.f;
#pragma unroll
            for (int i = 0; i < W; ++i) {
                const float d = val[k * W + i] - K[k];
                sa += d;
                sq += d * d;
            }
            a[k] = valid ? sa : 0.f;
            q[k] = valid ? sq : 0.f;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int k = 0; k < G; ++k) {
                a[k] += __shfl_xor_sync(0xffffffffu, a[k], off);
                q[k] += __shfl_xor_sync(0xffffffffu, q[k], off);
            }
        if (lane == 0) {
            const int g0 = o0 / p.gn_cpg;
#pragma unroll
            for (int k = 0; k < G; ++k) rec[g0 + k] = make_float4(npx * W, K[k], a[k], q[k]);
        }
    } else {
        if (o0 % p.gn_cpg == 0) run = GnRun{__shfl_sync(0xffffffffu, val[0], 0), 0.f, 0.f};
        if (valid) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float d = val[i] - run.K;
                run.a += d;
                run.q += d * d;
            }
        }
        if ((o0 + 16) % p.gn_cpg == 0) {
            float a = run.a, q = run.q;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, off);
                q += __shfl_xor_sync(0xffffffffu, q, off);
            }
            if (lane == 0) rec[o0 / p.gn_cpg] = make_float4(npx * p.gn_cpg, run.K, a, q);
        }
    }
}

// The same statistics for the staged TMA epilogue, read back from the warp's
// staging box (32 pixels x 16 channels, 64-byte swizzle: pixel r's channel j at
// r * 64 + (((j >> 2) ^ ((r >> 1) & 3)) * 16) + (j & 3) * 4) instead of being
// shuffled out of registers: lane l sums channel l & 15 over one half of the
// pixels (the halves read rows of opposite parity, so the two half-warps hit
// disjoint banks), then log2(W) + 1 shuffle rounds combine a group's lanes.
// Invalid pixels (r >= npx) trail and are skipped. Returns after the record
// of each completed group is written by its leader lane.
__device__ __forceinline__ void gn_chunk_stg(const ConvParams& p, const TileInfo& ti, const uint8_t* box, int o0,
                                             int chunk, int lane, int npx, GnRun& run) {
    const int j = lane & 15, h = lane >> 4;
    const int cpg = p.gn_cpg;
    const int w = cpg < 16 ? cpg : 16;  // channels of each group part in this chunk
    const uint32_t sb = smem_u32(box);
    const uint32_t jo = static_cast<uint32_t>((j & 3) * 4);
    // all 16 loads go out back to back (every row is inside the box; invalid rows are masked below)
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = h * 16 + ((i + h) & 15);
        v[i] = ld_shared_f32(sb + static_cast<uint32_t>(r * 64) +
                             (static_cast<uint32_t>((j >> 2) ^ ((r >> 1) & 3)) << 4) + jo);
    }
    float K;
    if (w < 16 || cpg == 16) {
        const int jg = j & ~(w - 1);  // the part's first channel, pixel 0
        K = ld_shared_f32(sb + (static_cast<uint32_t>(jg >> 2) << 4) + static_cast<uint32_t>((jg & 3) * 4));
    } else {
        if (o0 % cpg == 0) run = GnRun{ld_shared_f32(sb), 0.f, 0.f};  // pixel 0, channel 0
        K = run.K;
    }
    float a0 = 0.f, a1 = 0.f, q0 = 0.f, q1 = 0.f;
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const int r0 = h * 16 + ((i + h) & 15), r1 = h * 16 + ((i + 1 + h) & 15);
        const float d0 = r0 < npx ? v[i] - K : 0.f;
        const float d1 = r1 < npx ? v[i + 1] - K : 0.f;
        a0 += d0;
        q0 += d0 * d0;
        a1 += d1;
        q1 += d1 * d1;
    }
    float a = a0 + a1, q = q0 + q1;
    float4* rec = p.gn_part + (static_cast<long long>(ti.img) * p.gn_nchunks + chunk) * p.gn_groups;
    if (w < 16 || cpg == 16) {
        a += __shfl_xor_sync(0xffffffffu, a, 16);
        q += __shfl_xor_sync(0xffffffffu, q, 16);
        for (int off = 1; off < w; off <<= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, off);
            q += __shfl_xor_sync(0xffffffffu, q, off);
        }
        if (h == 0 && (j & (w - 1)) == 0) rec[(o0 + j) / cpg] = make_float4(static_cast<float>(npx * w), K, a, q);
    } else {
        run.a += a;
        run.q += q;
        if ((o0 + 16) % cpg == 0) {
            a = run.a;
            q = run.q;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, off);
                q += __shfl_xor_sync(0xffffffffu, q, off);
            }
            if (lane == 0) rec[o0 / cpg] = make_float4(static_cast<float>(npx * cpg), K, a, q);
        }
    }
}

__device__ __forceinline__ void gn_chunk(const ConvParams& p, const TileInfo& ti, const float (&val)[16], bool valid,
                                         int o0, int ew, int lane, float npx, GnRun& run) {
    const int mt = ((ti.v0 / p.R) * p.npar + ti.par) * p.tiles_x + ti.u0 / p.Wt;  // M tile within the image
    const int chunk = mt * kEpiWarps + ew;
    if (p.gn_cpg == 4)
        gn_chunk_w<4>(p, ti, val, valid, o0, chunk, lane, npx, run);
    else if (p.gn_cpg == 8)
        gn_chunk_w<8>(p, ti, val, valid, o0, chunk, lane, npx, run);
    else
        gn_chunk_w<16>(p, ti, val, valid, o0, chunk, lane, npx, run);
}

template <bool kWide = true>
__device__ __forceinline__ void epilogue_chunk(const ConvParams& p, const TileInfo& ti, const uint32_t (&r)[16],
                                               int o0, int v, int u, int q, int pp, int Y, int X,
                                               long long pix) {
    float val[16];
    compute_chunk<kWide>(p, ti, r, o0, v, u, q, pp, pix, val);
    store_chunk(p, pix, o0, val, Y, X, ti.img);
}

constexpr int kRmsMaxC = 144;  // fused RMS_norm keeps one pixel's channels in registers

// Whole-row epilogue with a fused RMS_norm: all cout (<= 144) channels of the
// pixel stay in registers, the f32 output is stored if requested, and the
// normalised f16 row is written with the standalone kernel's exact arithmetic
// order (vae_rms.cuh), so fused and unfused decodes agree bit for bit.
__device__ __forceinline__ void epilogue_rms_row(const ConvParams& p, const TileInfo& ti, uint32_t tbase, bool valid,
                                                 int v, int u, int q, int pp, int Y, int X, long long pix) {
    float row[kRmsMaxC];
#pragma unroll
    for (int c = 0; c < kRmsMaxC / 16; ++c) {
        if (c * 16 < p.BN) {  // warp-uniform
            uint32_t r[16];
            __syncwarp();
            tmem_ld16(tbase + static_cast<uint32_t>(c * 16), r);
            tmem_ld_wait();
            float val[16];
            compute_chunk(p, ti, r, c * 16, v, u, q, pp, pix, val);
#pragma unroll
            for (int i = 0; i < 16; ++i) row[c * 16 + i] = val[i];
            if (valid && p.y != nullptr) store_chunk(p, pix, c * 16, val, Y, X, ti.img);
        }
    }
    if (!valid) return;
    constexpr int G = rms_lanes(kRmsMaxC);  // 4: the standalone kernel's lanes for c <= 144
    const int c4 = p.cout / 4;
    float part[G];
#pragma unroll
    for (int l = 0; l < G; ++l) {
        part[l] = 0.f;
#pragma unroll
        for (int k = 0; k < kRmsMaxC / (4 * G); ++k) {
            const int i = l + k * G;
            if (i < c4) part[l] = rms_acc4(part[l], row[4 * i], row[4 * i + 1], row[4 * i + 2], row[4 * i + 3]);
        }
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1)
#pragma unroll
        for (int l = 0; l < off; ++l) part[l] = __fadd_rn(part[l], part[l + off]);
    const float inv = rms_inv(part[0], p.cout);
    __half* dst = p.rms_out + pix * p.cout;
#pragma unroll
    for (int c = 0; c < kRmsMaxC / 16; ++c) {
        if (c * 16 >= p.cout) break;
        uint32_t h[8];
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
            const int o = c * 16 + 4 * i4;
            const float4 g = __ldg(reinterpret_cast<const float4*>(p.rms_gamma + o));
            float a[4] = {rms_apply(row[o], inv, g.x), rms_apply(row[o + 1], inv, g.y),
                          rms_apply(row[o + 2], inv, g.z), rms_apply(row[o + 3], inv, g.w)};
            if (p.rms_silu) {
#pragma unroll
                for (int e = 0; e < 4; ++e) a[e] = silu_f(a[e]);
            }
            __half2 t0 = __floats2half2_rn(a[0], a[1]);
            __half2 t1 = __floats2half2_rn(a[2], a[3]);
            h[2 * i4] = *reinterpret_cast<uint32_t*>(&t0);
            h[2 * i4 + 1] = *reinterpret_cast<uint32_t*>(&t1);
        }
        reinterpret_cast<uint4*>(dst + c * 16)[0] = make_uint4(h[0], h[1], h[2], h[3]);
        reinterpret_cast<uint4*>(dst + c * 16)[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
}

// Fused RMS_norm through the staged TMA epilogue (one-row tiles, one N tile,
// no f32 output, no residual): a first pass over the accumulator's 16-column
// chunks forms the pixel's sum of squares in the standalone kernel's exact order
// (4 partial sums: channel quad i goes to part[i % 4], chunks in order, then
// the butterfly), a second pass reloads the chunks from TMEM, recomputes the
// same values, normalises them and stores f16 boxes (32 pixels x 16 channels,
// 32-byte rows, 32-byte swizzle) with TMA. No pixel row is held in registers.
__device__ __forceinline__ void epilogue_tma_rms_row(const ConvParams& p, const TileInfo& ti, uint32_t tbase, bool valid,
                                                     int v, int u, int q, int pp, long long pix, uint8_t* stg,
                                                     const CUtensorMap* mapY, int ew, int lane,
                                                     const float* sbias = nullptr) {
    const int nch = p.cout / 16;
    float part[4] = {0.f, 0.f, 0.f, 0.f};
    auto acc_chunk = [&](int c, uint32_t (&acc)[16]) {
        float val[16];
        compute_chunk(p, ti, acc, c * 16, v, u, q, pp, pix, val, nullptr, sbias);
#pragma unroll
        for (int l = 0; l < 4; ++l) part[l] = rms_acc4(part[l], val[4 * l], val[4 * l + 1], val[4 * l + 2], val[4 * l + 3]);
    };
    for (int c = 0; c < nch; ++c) {  // pass 1 (two chunks per TMEM wait measured slower)
        uint32_t acc[16];
        __syncwarp();
        tmem_ld16(tbase + static_cast<uint32_t>(c * 16), acc);
        tmem_ld_wait_regs(acc);
        acc_chunk(c, acc);
    }
    part[0] = __fadd_rn(part[0], part[2]);
    part[1] = __fadd_rn(part[1], part[3]);
    part[0] = __fadd_rn(part[0], part[1]);
    const float inv = rms_inv(part[0], p.cout);
    const uint32_t sbase = smem_u32(stg + ew * kStgBytes);
    const int seg = ti.u0 + ew * 32;
    const uint32_t row_off = static_cast<uint32_t>(lane) * 32u;
    const uint32_t sw = static_cast<uint32_t>((lane >> 2) & 1);
    for (int c = 0; c < nch; ++c) {
        uint32_t acc[16];
        __syncwarp();
        tmem_ld16(tbase + static_cast<uint32_t>(c * 16), acc);
        tmem_ld_wait_regs(acc);
        float val[16];
        compute_chunk(p, ti, acc, c * 16, v, u, q, pp, pix, val, nullptr, sbias);
        uint32_t h[8];
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
            const int o = c * 16 + 4 * i4;
            const float4 g = __ldg(reinterpret_cast<const float4*>(p.rms_gamma + o));
            float a[4] = {rms_apply(val[4 * i4], inv, g.x), rms_apply(val[4 * i4 + 1], inv, g.y),
                          rms_apply(val[4 * i4 + 2], inv, g.z), rms_apply(val[4 * i4 + 3], inv, g.w)};
            if (p.rms_silu) {
#pragma unroll
                for (int e = 0; e < 4; ++e) a[e] = silu_f(a[e]);
            }
            __half2 t0 = __floats2half2_rn(a[0], a[1]);
            __half2 t1 = __floats2half2_rn(a[2], a[3]);
            h[2 * i4] = *reinterpret_cast<uint32_t*>(&t0);
            h[2 * i4 + 1] = *reinterpret_cast<uint32_t*>(&t1);
        }
        if (lane == 0) bulk_wait_read_all();  // the previous box left this warp's buffer
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2; ++k)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sbase + row_off +
                                                                        ((static_cast<uint32_t>(k) ^ sw) << 4)),
                         "r"(h[4 * k]), "r"(h[4 * k + 1]), "r"(h[4 * k + 2]), "r"(h[4 * k + 3])
                         : "memory");
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && seg < p.wv) {
            tma_store_4d(mapY, sbase, c * 16, seg, ti.v0, ti.img);
            bulk_commit_group();
        }
    }
    (void)valid;
}

// Epilogue of one accumulator row (pixel) without a fused norm. kPipe: the
// register-hungry pipelined residual path (off in the 320-thread gather kernel).
// c0, cstep: this warp's 16-column chunks are c0, c0 + cstep, ... (the pair
// kernel splits a tile's chunks between two warps per lane quadrant).
template <bool kPipe, bool kGn = false>
__device__ __forceinline__ void epilogue_plain_row(const ConvParams& p, const TileInfo& ti, uint32_t tbase, bool valid,
                                                   int v, int u, int q, int pp, int Y, int X, long long pix,
                                                   int ew = 0, int lane = 0, const float* sbias = nullptr,
                                                   int c0 = 0, int cstep = 1) {
    GnRun run{0.f, 0.f, 0.f};
    const float npx = kGn ? static_cast<float>(__popc(__ballot_sync(0xffffffffu, valid))) : 0.f;
    if (kPipe && p.residual != nullptr && p.v8_ok && !p.out_nchw) {
        // Residual loads run two chunks ahead of their use (a three-slot
        // register ring), so three are in flight instead of one. j counts this
        // warp's chunks: chunk c0 + j * cstep.
        const int nchunk = p.BN / 16;
        const int nch = nchunk > c0 ? (nchunk - c0 + cstep - 1) / cstep : 0;
        float r0[16], r1[16], r2[16];
        auto ld = [&](int j, float* rr) {
            const int c = c0 + j * cstep;
            if (valid && j < nch && ti.n0 + c * 16 < p.cout) {
                const float* rs = p.residual + pix * p.cout + ti.n0 + c * 16;
                ld_v8_f32(rs, rr);
                ld_v8_f32(rs + 8, rr + 8);
            }
        };
        auto step = [&](int j, const float* rr) {
            if (j >= nch) return;  // warp-uniform
            const int c = c0 + j * cstep;
            uint32_t acc[16];
            __syncwarp();
            tmem_ld16(tbase + static_cast<uint32_t>(c * 16), acc);
            tmem_ld_wait();
            const int o0 = ti.n0 + c * 16;
            if (kGn) {
                if (o0 >= p.cout) return;  // warp-uniform
                float val[16];
                if (valid) {
                    compute_chunk(p, ti, acc, o0, v, u, q, pp, pix, val, rr, sbias);
                    store_chunk(p, pix, o0, val, Y, X, ti.img);
                }
                gn_chunk(p, ti, val, valid, o0, ew, lane, npx, run);
            } else if (valid && o0 < p.cout) {
                float val[16];
                compute_chunk(p, ti, acc, o0, v, u, q, pp, pix, val, rr, sbias);
                store_chunk(p, pix, o0, val, Y, X, ti.img);
            }
        };
        ld(0, r0);
        ld(1, r1);
        for (int c = 0; c < nch; c += 3) {
            ld(c + 2, r2);
            step(c, r0);
            ld(c + 3, r0);
            step(c + 1, r1);
            ld(c + 4, r1);
            step(c + 2, r2);
        }
        return;
    }
    for (int j = c0 * 16; j < p.BN; j += 16 * cstep) {
        uint32_t r[16];
        __syncwarp();
        tmem_ld16(tbase + static_cast<uint32_t>(j), r);
        tmem_ld_wait();
        const int o0 = ti.n0 + j;
        if (kGn) {
            if (o0 >= p.cout) break;  // warp-uniform
            float val[16];
            if (valid) {
                compute_chunk<kPipe>(p, ti, r, o0, v, u, q, pp, pix, val);
                store_chunk(p, pix, o0, val, Y, X, ti.img);
            }
            gn_chunk(p, ti, val, valid, o0, ew, lane, npx, run);
        } else if (valid && o0 < p.cout) {
            epilogue_chunk<kPipe>(p, ti, r, o0, v, u, q, pp, Y, X, pix);
        }
    }
}

// Epilogue of one accumulator row through TMA: each warp stages its 32 pixels x
// 16 channels (64-byte swizzle) and one lane issues a bulk tensor store, or an
// f32 add onto y when y is the residual (the add then happens in L2: y + (acc *
// oscale + bias), the same two roundings as the register path). No global
// loads or per-lane stores: the warp's traffic is whole 2 KB boxes.
template <bool kGn = false>
__device__ __forceinline__ void epilogue_tma_row(const ConvParams& p, const TileInfo& ti, uint32_t tbase, int v, int u,
                                                 int q, int pp, long long pix, uint8_t* stg, const CUtensorMap* mapY,
                                                 int ew, int lane, bool valid = true, const float* sbias = nullptr) {
    GnRun run{0.f, 0.f, 0.f};
    const int npx_i = kGn ? __popc(__ballot_sync(0xffffffffu, valid)) : 0;
    const uint32_t sbase = smem_u32(stg + ew * kStgBytes);
    const int seg = ti.u0 + ew * 32;  // first pixel of this warp's 32 (warp-uniform)
    const uint32_t row_off = static_cast<uint32_t>(lane) * 64u;
    const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
    const int nch = (min(p.BN, p.cout - ti.n0) + 15) / 16;  // 16-column chunks of this tile
    auto process = [&](int c, uint32_t (&acc)[16]) {
        const int o0 = ti.n0 + c * 16;
        // pixels past the row's end read no residual or DupUp source; their values are not stored
        float val[16];
        if (valid) {
            compute_chunk(p, ti, acc, o0, v, u, q, pp, pix, val, nullptr, sbias);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) val[i] = 0.f;
        }
        if (lane == 0) bulk_wait_read_all();  // the previous box left this warp's buffer
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 4; ++k)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(sbase + row_off +
                                                                        ((static_cast<uint32_t>(k) ^ sw) << 4)),
                         "f"(val[4 * k]), "f"(val[4 * k + 1]), "f"(val[4 * k + 2]), "f"(val[4 * k + 3])
                         : "memory");
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && seg < p.wv) {
            if (p.epi_tma == 2)
                tma_reduce_add_4d(mapY, sbase, o0, seg, ti.v0, ti.img);
            else if (p.up)  // output pixels 2u + pp of row 2v + q: the (parity, W/2) view
                tma_store_5d(mapY, sbase, o0, pp, seg, 2 * ti.v0 + q, ti.img);
            else
                tma_store_4d(mapY, sbase, o0, seg, ti.v0, ti.img);
            bulk_commit_group();
        }
        if (kGn) {  // the statistics read the staged box (alongside the store's own read)
            const int mt = ((ti.v0 / p.R) * p.npar + ti.par) * p.tiles_x + ti.u0 / p.Wt;
            gn_chunk_stg(p, ti, stg + ew * kStgBytes, o0, mt * kEpiWarps + ew, lane, npx_i, run);
        }
    };
    for (int c = 0; c < nch; ++c) {
        uint32_t acc[16];
        __syncwarp();
        tmem_ld16(tbase + static_cast<uint32_t>(c * 16), acc);
        tmem_ld_wait_regs(acc);
        process(c, acc);
    }
}

template <int kMode, bool kRms, int kVar>
__device__ void role_epilogue(const ConvParams& p, const Smem& s, uint32_t tmem_base, int ew, int lane,
                              const CUtensorMap* mapY) {
    const int row = ew * 32 + lane;
    int accbuf = 0;
    uint32_t accphase = 0;
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const TileInfo ti = decode_tile<kVar == 1>(p, t);
        if (!warp_all(mbar_wait(smem_u32(&s.accf[accbuf]), accphase, s.abort_flag, p.timeout_ns, p.status,
                                kWhereEpiAccFull)))
            break;
        tc_fence_after();
        const int rr = row / p.Wt, cc = row % p.Wt;
        const int v = ti.v0 + rr, u = ti.u0 + cc;
        const bool valid = row < p.R * p.Wt && v < p.hv && u < p.wv;
        const int q = ti.par >> 1, pp = ti.par & 1;
        const int Y = p.up ? 2 * v + q : v;
        const int X = p.up ? 2 * u + pp : u;
        const long long pix = (static_cast<long long>(ti.img) * p.H + Y) * p.W + X;
        const uint32_t tbase =
            tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(accbuf * p.acc_stride);
        if (kRms && kMode != kModeGather && p.epi_tma == 3) {
            epilogue_tma_rms_row(p, ti, tbase, valid, v, u, q, pp, pix, s.stg, mapY, ew, lane,
                                 p.bias_smem ? s.bias : nullptr);
        } else if (kRms) {
            epilogue_rms_row(p, ti, tbase, valid, v, u, q, pp, Y, X, pix);
        } else if (kMode != kModeGather && p.epi_tma) {
            epilogue_tma_row<kVar == 3>(p, ti, tbase, v, u, q, pp, pix, s.stg, mapY, ew, lane, valid,
                                        p.bias_smem ? s.bias : nullptr);
        } else {
            epilogue_plain_row<kMode != kModeGather, kVar == 3>(p, ti, tbase, valid, v, u, q, pp, Y, X, pix, ew,
                                                                 lane, p.bias_smem ? s.bias : nullptr);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&s.acce[accbuf]));
        accbuf ^= 1;
        if (accbuf == 0) accphase ^= 1u;
    }
    if (p.epi_tma && lane == 0) bulk_wait_all();  // boxes read and written before the CTA exits
}

// kRms: the fused RMS_norm epilogue (a separate instantiation, so the other
// kernels do not carry its 144-value row in registers).
template <int kMode, bool kRms, int kVar>
__global__ void __launch_bounds__(kMode == kModeGather ? 320 : 224, 1)
    conv_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const __grid_constant__ CUtensorMap mapA16, const __grid_constant__ CUtensorMap mapB16,
                const __grid_constant__ CUtensorMap mapY, const ConvParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw, p);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        *s.abort_flag = 0;
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(smem_u32(&s.full[i]), kMode == kModeGather ? 129u : 1u);
            mbar_init(smem_u32(&s.empty[i]), 1u);
        }
        if (kMode == kModeHalo && p.ks != 3)  // the separate halo-box ring
            for (int i = 0; i < p.a_stages; ++i) {
                mbar_init(smem_u32(&s.afull[i]), 1u);
                mbar_init(smem_u32(&s.aempty[i]), 1u);
            }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s.accf[i]), 1u);
            mbar_init(smem_u32(&s.acce[i]), static_cast<uint32_t>(kEpiWarps * 32));
        }
        mbar_init(smem_u32(s.drain), 1u);
        if (kMode != kModeGather && p.refl)
            for (int i = 0; i < p.stages; ++i) mbar_init(smem_u32(&s.fixed[i]), 1u);
        fence_mbar_init();
    }
    const uint32_t tmem_cols = p.acc_stride * 2 <= 32 ? 32u
                               : p.acc_stride * 2 <= 64 ? 64u
                               : p.acc_stride * 2 <= 128 ? 128u
                               : p.acc_stride * 2 <= 256 ? 256u
                                                          : 512u;
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(s.tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        if (kMode != kModeGather) tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB);
        if (p.rem16) {
            tma_prefetch_desc(&mapA16);
            tma_prefetch_desc(&mapB16);
        }
        if (p.epi_tma) tma_prefetch_desc(&mapY);
    }
    // everything above touches only shared memory, TMEM and kernel parameters
    pdl_wait();
    if (p.bias_smem)  // visible to the epilogue after the __syncthreads below
        for (int i = threadIdx.x; i < p.cout; i += blockDim.x) s.bias[i] = __ldg(p.bias + i);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s.tmem_slot;

    if (warp < kEpiWarps) {
        role_epilogue<kMode, kRms, kVar>(p, s, tmem_base, warp, lane, &mapY);
    } else if (warp == kProducerWarp) {
        if (lane == 0) role_producer<kMode, kVar>(p, s, &mapA, &mapB, &mapA16, &mapB16);
    } else if (warp == kMmaWarp) {
        if (lane == 0) role_mma<kVar>(p, s, tmem_base);
    } else if (kMode == kModeGather && warp >= kGatherWarp0) {
        role_gather<kVar>(p, s, (warp - kGatherWarp0) * 32 + lane);
    } else if (kMode != kModeGather && is_2d(kVar) && warp == kGatherWarp0) {
        if (lane == 0) role_fixer(p, s);  // launched only for reflect padding
    }
    // this CTA's work is done: the next grid may launch (it waits for this one to finish)
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}


// ───────────────────────────── CTA-pair kernel ─────────────────────────────
// A cluster of two CTAs (the two SMs of a TPC) computes two 128-pixel row tiles
// (rows 2j and 2j + 1 of one column block and parity class) with
// tcgen05.mma.cta_group::2 (M = 256): each CTA holds its own A halo boxes and
// HALF of every weight tile (BN/2 rows) at the same shared-memory offsets, and
// receives its own 128 x BN accumulator in TMEM. Per SM this halves both the
// weight bytes taken in from L2 and the B operand bytes the tensor core reads
// from shared memory, which measured as the two limits of the single-CTA
// kernel at 144 channels (its MMAs issue at ~86 cycles for 72 cycles of tensor
// work; the pair's at 72).
//
// Stages are the three-tap halo stages of the single-CTA kernel (one 130-pixel
// box per (ky, 64-channel chunk) and the three kx taps' weight halves, 12 pair
// MMAs), with the exact 16-channel remainder stage when cin % 64 == 16.
// Barriers: both CTAs' copies complete on the EVEN CTA's full barrier, armed
// once by the even producer for the bytes of both; the even CTA's MMA thread
// commits with multicast to the empty and accumulator-full barriers of both
// CTAs; every epilogue warp of both CTAs arrives on the even CTA's
// accumulator-empty barrier. The odd CTA learns its copies landed from its
// empty barriers (the MMAs that read them completed). The ring's waits (full,
// empty) order only async-proxy traffic (TMA writes, tensor-core reads) and
// take CTA scope; the accumulator handshakes, which order generic TMEM reads
// against MMAs across the pair, take cluster scope.
//
// Eight epilogue warps per CTA: warp w drains TMEM lane quadrant w % 4 (its 32
// pixels) and every other 16-column chunk starting at w / 4, through a
// double-buffered 2 KB staging box (one TMA store in flight while the next
// box is written), so the epilogue keeps up with the doubled MMA rate.
constexpr int kPairEpiWarps = 8;
constexpr int kPairProducerWarp = 8;
constexpr int kPairMmaWarp = 9;
constexpr int kPairThreads = 320;
constexpr int kPairStgBytes = kPairEpiWarps * 2 * kStgBytes;  // two boxes per epilogue warp

__device__ __forceinline__ TileInfo decode_pair_tile(const ConvParams& p, int t, int rank) {
    TileInfo ti;
    const int nt = t % p.n_tiles;
    int r = t / p.n_tiles;
    if (p.gemm) {  // column tiles 2j and 2j + 1 of the one-row grid (typ_tiles = column pairs)
        const int ptx = r % p.typ_tiles;
        ti.img = r / p.typ_tiles;
        ti.par = 0;
        ti.v0 = 0;
        ti.u0 = (2 * ptx + rank) * p.Wt;
        ti.n0 = nt * p.BN;
        return ti;
    }
    const int tx = r % p.tiles_x;
    r /= p.tiles_x;
    ti.par = r % p.npar;
    r /= p.npar;
    const int typ = r % p.typ_tiles;
    ti.img = r / p.typ_tiles;
    ti.v0 = (2 * typ + rank) * p.R;  // same column block and parity, rows 2*typ and 2*typ+1
    ti.u0 = tx * p.Wt;
    ti.n0 = nt * p.BN;
    return ti;
}

__device__ void pair_producer(const ConvParams& p, const Smem& s, const CUtensorMap* mapA, const CUtensorMap* mapB,
                              const CUtensorMap* mapA16, const CUtensorMap* mapB16, int rank) {
    const uint64_t pol_w = policy_evict_last();
    const uint64_t pol_a = policy_evict_normal();
    const uint32_t b_bytes = static_cast<uint32_t>(p.b_rows) * 128u;
    const int boff = rank * p.b_rows;
    int stage = 0;
    uint32_t phase = 0, armed = 0, arm_par = 0;
    bool ok = true;
    // Waits for a free slot; the even CTA arms its (shared) full barrier for
    // the bytes of both CTAs. Returns the full barrier's cluster address.
    auto next_slot = [&](uint32_t tx, uint32_t* slot) -> uint32_t {
        if (!mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, s.abort_flag, p.timeout_ns, p.status,
                               kWhereProducerEmpty)) {
            ok = false;
            return 0u;
        }
        const uint32_t fb = smem_u32(&s.full[stage]);
        if (rank == 0) mbar_arrive_expect_tx(fb, 2u * tx);
        armed |= 1u << stage;
        arm_par = (arm_par & ~(1u << stage)) | (phase << stage);
        *slot = static_cast<uint32_t>(stage);
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
        }
        return mapa_shared(fb, 0u);
    };
    const int kc_end = p.rem16 ? p.kfull : p.kchunks;
    for (int t = blockIdx.x >> 1; t < p.pair_tiles && ok; t += gridDim.x >> 1) {
        const TileInfo ti = decode_pair_tile(p, t, rank);
        if (p.res_prefetch && ti.v0 < p.hv) {
            const int npx = min(p.Wt, p.wv - ti.u0);
            const long long pix0 = (static_cast<long long>(ti.img) * p.H + ti.v0) * p.W + ti.u0;
            prefetch_l2_bulk(p.residual + pix0 * p.cout, static_cast<uint32_t>(npx * p.cout * 4));
        }
        if (p.dup_prefetch && ti.v0 < p.hv) {
            const int npx = min(p.Wt, p.wv - ti.u0);
            const long long pix0 = (static_cast<long long>(ti.img) * p.hv + ti.v0) * p.wv + ti.u0;
            prefetch_l2_bulk(p.dup_src + pix0 * p.dup_cin, static_cast<uint32_t>(npx * p.dup_cin * 4));
        }
        if (p.gemm) {
            // The N tiles of a column pair run side by side (N varies fastest), so their first
            // touch of each A chunk waits on HBM. The pair whose next tile is the first N tile
            // of its column pair asks L2 for that tile's A rows one tile ahead (and for its
            // first tile at the start); the others then find them in L2.
            if (kGemmPairPrefetch) {
                const int step = static_cast<int>(gridDim.x >> 1);
                for (int tn = (t == static_cast<int>(blockIdx.x >> 1) ? t : t + step); tn <= t + step; tn += step) {
                    if (tn >= p.pair_tiles || tn % p.n_tiles != 0) continue;
                    const TileInfo tj = decode_pair_tile(p, tn, rank);
                    if (tj.u0 < p.wv)
                        prefetch_l2_bulk(p.x + (static_cast<long long>(tj.img) * p.wv + tj.u0) * p.cin,
                                         static_cast<uint32_t>(min(p.Wt, p.wv - tj.u0) * p.cin * 2));
                }
            }
            // ks chunks per stage: chunk i of slot j at A slot (j * ks + i), B slot (j * ks + i)
            for (int kc = 0; kc < p.kchunks && ok; kc += p.ks) {
                const int nc = min(p.ks, p.kchunks - kc);
                uint32_t slot;
                const uint32_t fb = next_slot(static_cast<uint32_t>(nc) * (p.a_tx + b_bytes), &slot);
                if (!ok) break;
                for (int i = 0; i < nc; ++i) {
                    const uint32_t j = slot * static_cast<uint32_t>(p.ks) + static_cast<uint32_t>(i);
                    tma_load_4d_pair(smem_u32(s.a + j * kABytes), mapA, fb, (kc + i) * kBK, ti.u0, 0, ti.img,
                                     pol_a);
                    tma_load_3d_pair(smem_u32(s.b + j * b_bytes), mapB, fb, (kc + i) * kBK, 0, ti.n0 + boff,
                                     pol_w);
                }
            }
            continue;
        }
        const int q = ti.par >> 1, pp = ti.par & 1;
        const int dxmin = (p.up && pp == 1) ? 0 : -1;
        for (int ky = 0; ky < 3 && ok; ++ky) {
            const int dy = p.up ? (q + ky + 1) / 2 - 1 : ky - 1;
            for (int kc = 0; kc < kc_end && ok; ++kc) {
                uint32_t slot;
                const uint32_t fb = next_slot(p.a_tx + 3u * b_bytes, &slot);
                if (!ok) break;
                tma_load_4d_pair(smem_u32(s.a + slot * kHaloBytes), mapA, fb, kc * kBK, ti.u0 + dxmin, ti.v0 + dy,
                                 ti.img, pol_a);
                for (int kx = 0; kx < 3; ++kx)
                    tma_load_3d_pair(smem_u32(s.b + (slot * 3 + kx) * p.b_rows * 128), mapB, fb, kc * kBK,
                                     ky * 3 + kx, ti.n0 + boff, pol_w);
            }
        }
        if (p.rem16 && ok) {
            // the last 16 channels of all three ky rows and all nine taps in one stage
            uint32_t slot;
            const uint32_t fb = next_slot(3u * kRemABytes + 9u * static_cast<uint32_t>(p.b_rows) * 32u, &slot);
            if (ok) {
                for (int ky = 0; ky < 3; ++ky) {
                    const int dy = p.up ? (q + ky + 1) / 2 - 1 : ky - 1;
                    tma_load_4d_pair(smem_u32(s.a + slot * kHaloBytes + ky * kRemAStride), mapA16, fb,
                                     p.kfull * kBK, ti.u0 + dxmin, ti.v0 + dy, ti.img, pol_a);
                }
                for (int tap = 0; tap < 9; ++tap)
                    tma_load_3d_pair(smem_u32(s.b + slot * 3 * p.b_rows * 128 + tap * p.b_rows * 32), mapB16, fb,
                                     p.kfull * kBK, tap, ti.n0 + boff, pol_w);
            }
        }
    }
    // Let every copy this CTA started land before it can exit: the even CTA
    // sees them on its full barriers; the odd CTA on its empty barriers (the
    // MMAs that read a slot complete only after that slot's copies landed).
    for (int st = 0; st < p.stages; ++st)
        if (armed & (1u << st))
            drain_wait(smem_u32(rank == 0 ? &s.full[st] : &s.empty[st]), (arm_par >> st) & 1u, p);
}

// Even CTA: one thread issues the pair MMAs (M = 256). This thread's own
// work bounds the loop (measured: a tcgen05.mma takes ~78 cycles to issue
// against 72 cycles of tensor work at N = 144, and every stage adds its
// barrier wait and commit), so the loop carries the shared-memory descriptors
// as running values (slot strides added, nothing recomputed per stage) and
// keeps the work between MMAs to the descriptor adds.
__device__ void pair_mma(const ConvParams& p, const Smem& s, uint32_t tmem_base) {
    const uint32_t idesc = idesc_f16_f32(2 * kBM, p.BN);
    // Descriptors of slot 0; the start-address field counts 16-byte units and
    // every address here stays below 2^18 bytes, so offsets add without carry.
    const uint64_t a128 = sw128_kmajor_desc(smem_u32(s.a));
    const uint64_t b128 = sw128_kmajor_desc(smem_u32(s.b));
    const uint64_t a32 = sw32_kmajor_desc(smem_u32(s.a));
    const uint64_t b32 = sw32_kmajor_desc(smem_u32(s.b));
    // a slot: one halo box (three kx taps), or in GEMM mode ks A chunks; b slot: three taps or ks chunks
    const uint32_t a_slot = p.gemm ? static_cast<uint32_t>(p.ks * kABytes) >> 4 : kHaloBytes >> 4;
    const uint32_t b_slot = static_cast<uint32_t>((p.gemm ? p.ks : 3) * p.b_rows * 128) >> 4;
    const uint32_t b_tap = static_cast<uint32_t>(p.b_rows * 128) >> 4;
    const uint32_t g_a_chunk = static_cast<uint32_t>(kABytes) >> 4;
    const int g_nk_last = min(4, (p.cin - (p.kchunks - 1) * kBK + 15) / 16);  // GEMM mode: K steps of the last chunk
    const uint32_t b_tap16 = static_cast<uint32_t>(p.b_rows * 32) >> 4;
    const int kc_end = p.rem16 ? p.kfull : p.kchunks;
    const int nk_last = min(4, (p.cin - (kc_end - 1) * kBK) / 16);  // K steps of the last 64-channel chunk
    int stage = 0;
    uint32_t phase = 0, soff_a = 0, soff_b = 0;  // this slot's offsets, in descriptor units
    auto advance = [&]() {
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
            soff_a = 0;
            soff_b = 0;
        } else {
            soff_a += a_slot;
            soff_b += b_slot;
        }
    };
    int accbuf = 0;
    uint32_t accphase = 0;
    bool ok = true;
    for (int t = blockIdx.x >> 1; t < p.pair_tiles && ok; t += gridDim.x >> 1) {
        if (!mbar_wait_cluster(smem_u32(&s.acce[accbuf]), accphase ^ 1u, s.abort_flag, p.timeout_ns, p.status,
                               kWhereMmaAccEmpty))
            break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(accbuf * p.acc_stride);
        if (p.gemm) {
            uint32_t acc = 0u;
            for (int kc = 0; kc < p.kchunks; kc += p.ks) {
                if (!mbar_wait(smem_u32(&s.full[stage]), phase, s.abort_flag, p.timeout_ns, p.status,
                               kWhereMmaFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = a128 + soff_a;
                const uint64_t bd = b128 + soff_b;
                const int nc = min(p.ks, p.kchunks - kc);
                if (nc == p.ks && (kc + nc < p.kchunks || g_nk_last == 4)) {
#pragma unroll 3
                    for (int i = 0; i < p.ks; ++i)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            umma_f16_pair(d, ad + static_cast<uint32_t>(i) * g_a_chunk + 2u * k,
                                          bd + static_cast<uint32_t>(i) * b_tap + 2u * k, idesc, acc);
                            acc = 1u;
                        }
                } else {
                    for (int i = 0; i < nc; ++i) {
                        const int nk = kc + i + 1 < p.kchunks ? 4 : g_nk_last;
                        for (int k = 0; k < nk; ++k) {
                            umma_f16_pair(d, ad + static_cast<uint32_t>(i) * g_a_chunk + 2u * k,
                                          bd + static_cast<uint32_t>(i) * b_tap + 2u * k, idesc, acc);
                            acc = 1u;
                        }
                    }
                }
                umma_commit_pair(smem_u32(&s.empty[stage]));
                advance();
            }
            if (!ok) break;
            umma_commit_pair(smem_u32(&s.accf[accbuf]));
            accbuf ^= 1;
            if (accbuf == 0) accphase ^= 1u;
            continue;
        }
        const int pp = p.up ? decode_pair_tile(p, t, 0).par & 1 : 0;  // (the divisions only where parity matters)
        const int dxmin = (p.up && pp == 1) ? 0 : -1;
        // row offset of tap kx inside the halo box, in 128-byte rows
        uint32_t rel[3];
#pragma unroll
        for (int kx = 0; kx < 3; ++kx) rel[kx] = static_cast<uint32_t>((p.up ? (pp + kx + 1) / 2 - 1 : kx - 1) - dxmin);
        uint32_t acc = 0u;  // the tile's first MMA overwrites the accumulator
        for (int ky = 0; ky < 3 && ok; ++ky)
            for (int kc = 0; kc < kc_end; ++kc) {
                if (!mbar_wait(smem_u32(&s.full[stage]), phase, s.abort_flag, p.timeout_ns, p.status,
                               kWhereMmaFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = a128 + soff_a;
                const uint64_t bd = b128 + soff_b;
                if (kc + 1 < kc_end || nk_last == 4) {
#pragma unroll
                    for (int kx = 0; kx < 3; ++kx)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            umma_f16_pair(d, ad + rel[kx] * 8u + 2u * k, bd + kx * b_tap + 2u * k, idesc, acc);
                            acc = 1u;
                        }
                } else {
                    for (int kx = 0; kx < 3; ++kx)
                        for (int k = 0; k < nk_last; ++k) {
                            umma_f16_pair(d, ad + rel[kx] * 8u + 2u * k, bd + kx * b_tap + 2u * k, idesc, acc);
                            acc = 1u;
                        }
                }
                umma_commit_pair(smem_u32(&s.empty[stage]));
                advance();
            }
        if (p.rem16 && ok) {
            if (!mbar_wait(smem_u32(&s.full[stage]), phase, s.abort_flag, p.timeout_ns, p.status,
                           kWhereMmaFull)) {
                ok = false;
            } else {
                tc_fence_after();
                // one K = 16 step per tap (the 64-channel chunks came first: always accumulate):
                // box ky at ky * kRemAStride, 32-byte rows; tap (ky, kx) weights at (ky * 3 + kx) * b_rows * 32
                const uint64_t ad = a32 + soff_a;
                const uint64_t bd = b32 + soff_b;
#pragma unroll
                for (int ky = 0; ky < 3; ++ky)
#pragma unroll
                    for (int kx = 0; kx < 3; ++kx)
                        umma_f16_pair(d, ad + static_cast<uint32_t>(ky * (kRemAStride >> 4)) + rel[kx] * 2u,
                                      bd + static_cast<uint32_t>(ky * 3 + kx) * b_tap16, idesc, 1u);
                umma_commit_pair(smem_u32(&s.empty[stage]));
                advance();
            }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&s.accf[accbuf]));
        accbuf ^= 1;
        if (accbuf == 0) accphase ^= 1u;
    }
    umma_commit_pair(smem_u32(s.drain));
    drain_wait(smem_u32(s.drain), 0u, p);
}

// One accumulator row (pixel) of a pair tile through TMA: this warp's chunks
// half, half + 2, ... each staged as a 32-pixel x 16-channel box (64-byte
// swizzle) in one of the warp's two buffers and stored (or, when y is the
// residual, added onto y in L2) by one bulk tensor operation; a buffer is
// rewritten only after the store issued from it two boxes earlier has read it.
__device__ __forceinline__ void pair_epi_tma_row(const ConvParams& p, const TileInfo& ti, uint32_t tbase, int v,
                                                 int u, int q, int pp, long long pix, uint8_t* stg,
                                                 const CUtensorMap* mapY, int quad, int half, int lane, bool valid,
                                                 const float* sbias, uint32_t& nbox) {
    const int seg = ti.u0 + quad * 32;  // first pixel of this warp's 32 (warp-uniform)
    const bool store = seg < p.wv && ti.v0 < p.hv;
    const uint32_t row_off = static_cast<uint32_t>(lane) * 64u;
    const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
    const int nch = (min(p.BN, p.cout - ti.n0) + 15) / 16;  // 16-column chunks of this tile
    for (int c = half; c < nch; c += 2) {
        uint32_t acc[16];
        __syncwarp();
        tmem_ld16(tbase + static_cast<uint32_t>(c * 16), acc);
        tmem_ld_wait_regs(acc);
        const int o0 = ti.n0 + c * 16;
        float val[16];
        if (valid) {
            compute_chunk(p, ti, acc, o0, v, u, q, pp, pix, val, nullptr, sbias);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) val[i] = 0.f;
        }
        const uint32_t sbase = smem_u32(stg + (nbox & 1u) * kStgBytes);
        if (lane == 0) bulk_wait_read_1();  // the store issued from this buffer two boxes ago has read it
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 4; ++k)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(sbase + row_off +
                                                                        ((static_cast<uint32_t>(k) ^ sw) << 4)),
                         "f"(val[4 * k]), "f"(val[4 * k + 1]), "f"(val[4 * k + 2]), "f"(val[4 * k + 3])
                         : "memory");
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && store) {
            if (p.epi_tma == 2)
                tma_reduce_add_4d(mapY, sbase, o0, seg, ti.v0, ti.img);
            else if (p.up)  // output pixels 2u + pp of row 2v + q: the (parity, W/2) view
                tma_store_5d(mapY, sbase, o0, pp, seg, 2 * ti.v0 + q, ti.img);
            else
                tma_store_4d(mapY, sbase, o0, seg, ti.v0, ti.img);
        }
        if (lane == 0) bulk_commit_group();  // (an empty group when nothing was stored keeps the count)
        ++nbox;
    }
}

// The fused RMS_norm of a pair tile's pixel (one N tile holds all cout <= 144
// channels; f16 rows only, no residual). The sum of squares follows the
// standalone kernel's order (channel quad i into partial sum i % 4, chunks in
// order, then the butterfly) while each warp of the lane quadrant reads only
// its own chunks (half, half + 2, ...): it puts each chunk's four quad sums in
// free TMEM columns of its lanes (two sets by tile parity), the two warps meet
// on a bounded barrier, and each then adds all chunks' quad sums in order. Then
// it reloads its chunks from TMEM (faster, measured, than holding them in
// registers through the exchange), normalises them and stores them as 32-pixel
// x 16-channel f16 boxes (32-byte rows, 32-byte swizzle) from two 1 KB staging
// buffers.
__device__ __forceinline__ void pair_epi_tma_rms_row(const ConvParams& p, const TileInfo& ti, uint32_t tbase,
                                                     uint32_t xbase, int v, int u, int q, int pp, long long pix,
                                                     uint8_t* stg, const CUtensorMap* mapY, int quad, int half,
                                                     int lane, const float* sbias, uint32_t& nbox, uint64_t* xbar,
                                                     volatile int* abort_flag, uint32_t& xphase) {
    const int nch = p.cout / 16;
    for (int c = half; c < nch; c += 2) {
        uint32_t acc[16];
        __syncwarp();
        tmem_ld16(tbase + static_cast<uint32_t>(c * 16), acc);
        tmem_ld_wait_regs(acc);
        float val[16];
        compute_chunk(p, ti, acc, c * 16, v, u, q, pp, pix, val, nullptr, sbias);
        float qs[4];
#pragma unroll
        for (int l = 0; l < 4; ++l) qs[l] = rms_acc4(0.f, val[4 * l], val[4 * l + 1], val[4 * l + 2], val[4 * l + 3]);
        tmem_st4(xbase + static_cast<uint32_t>(c * 4), qs);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(smem_u32(xbar));
    const bool met = warp_all(mbar_wait(smem_u32(xbar), xphase & 1u, abort_flag, p.timeout_ns, p.status,
                                        kWhereEpiAccFull));
    ++xphase;
    tc_fence_after();
    float part[4] = {0.f, 0.f, 0.f, 0.f};
    if (met) {
        for (int c = 0; c < nch; ++c) {
            uint32_t r[4];
            tmem_ld4(xbase + static_cast<uint32_t>(c * 4), r);
            tmem_ld_wait_regs4(r);
#pragma unroll
            for (int l = 0; l < 4; ++l) part[l] = __fadd_rn(part[l], __uint_as_float(r[l]));
        }
    }
    part[0] = __fadd_rn(part[0], part[2]);
    part[1] = __fadd_rn(part[1], part[3]);
    part[0] = __fadd_rn(part[0], part[1]);
    const float inv = rms_inv(part[0], p.cout);
    const int seg = ti.u0 + quad * 32;
    const bool store = seg < p.wv && ti.v0 < p.hv;
    const uint32_t row_off = static_cast<uint32_t>(lane) * 32u;
    const uint32_t sw = static_cast<uint32_t>((lane >> 2) & 1);
    for (int c = half; c < nch; c += 2) {
        uint32_t acc[16];
        __syncwarp();
        tmem_ld16(tbase + static_cast<uint32_t>(c * 16), acc);
        tmem_ld_wait_regs(acc);
        float val[16];
        compute_chunk(p, ti, acc, c * 16, v, u, q, pp, pix, val, nullptr, sbias);
        uint32_t hv[8];
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
            const int o = c * 16 + 4 * i4;
            const float4 g = __ldg(reinterpret_cast<const float4*>(p.rms_gamma + o));
            float a[4] = {rms_apply(val[4 * i4], inv, g.x), rms_apply(val[4 * i4 + 1], inv, g.y),
                          rms_apply(val[4 * i4 + 2], inv, g.z), rms_apply(val[4 * i4 + 3], inv, g.w)};
            if (p.rms_silu) {
#pragma unroll
                for (int e = 0; e < 4; ++e) a[e] = silu_f(a[e]);
            }
            __half2 t0 = __floats2half2_rn(a[0], a[1]);
            __half2 t1 = __floats2half2_rn(a[2], a[3]);
            hv[2 * i4] = *reinterpret_cast<uint32_t*>(&t0);
            hv[2 * i4 + 1] = *reinterpret_cast<uint32_t*>(&t1);
        }
        const uint32_t sbase = smem_u32(stg + (nbox & 1u) * (kStgBytes / 2));
        if (lane == 0) bulk_wait_read_1();  // the store issued from this buffer two boxes ago has read it
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2; ++k)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sbase + row_off +
                                                                        ((static_cast<uint32_t>(k) ^ sw) << 4)),
                         "r"(hv[4 * k]), "r"(hv[4 * k + 1]), "r"(hv[4 * k + 2]), "r"(hv[4 * k + 3])
                         : "memory");
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && store) tma_store_4d(mapY, sbase, c * 16, seg, ti.v0, ti.img);
        if (lane == 0) bulk_commit_group();
        ++nbox;
    }
}

// kRms: the fused RMS_norm instantiation (its register-held chunks would
// otherwise crowd the plain epilogues' registers).
template <bool kRms>
__device__ void pair_epilogue(const ConvParams& p, const Smem& s, uint32_t tmem_base, int w, int lane, int rank,
                              const CUtensorMap* mapY) {
    const int quad = w & 3, half = w >> 2;
    const int row = quad * 32 + lane;
    uint8_t* stg = s.stg + w * 2 * kStgBytes;
    const float* sbias = p.bias_smem ? s.bias : nullptr;
    uint32_t nbox = 0, xphase = 0;
    int accbuf = 0;
    uint32_t accphase = 0;
    for (int t = blockIdx.x >> 1; t < p.pair_tiles; t += gridDim.x >> 1) {
        const TileInfo ti = decode_pair_tile(p, t, rank);
        if (!warp_all(mbar_wait_cluster(smem_u32(&s.accf[accbuf]), accphase, s.abort_flag, p.timeout_ns, p.status,
                                        kWhereEpiAccFull)))
            break;
        tc_fence_after();
        const int v = ti.v0, u = ti.u0 + row;
        const bool valid = v < p.hv && u < p.wv && ti.img < p.n;
        const int q = ti.par >> 1, pp = ti.par & 1;
        const int Y = p.up ? 2 * v + q : v;
        const int X = p.up ? 2 * u + pp : u;
        const long long pix = (static_cast<long long>(ti.img) * p.H + Y) * p.W + X;
        const uint32_t tbase =
            tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(accbuf * p.acc_stride);
        if (kRms) {
            // the quad-sum exchange columns follow the two accumulators, one set per tile parity
            const uint32_t xbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                   static_cast<uint32_t>(2 * p.acc_stride + (xphase & 1u) * 4 * (p.BN / 16));
            pair_epi_tma_rms_row(p, ti, tbase, xbase, v, u, q, pp, pix, stg, mapY, quad, half, lane, sbias, nbox,
                                 &s.xbar[quad], s.abort_flag, xphase);
        }
        else if (p.epi_tma)
            pair_epi_tma_row(p, ti, tbase, v, u, q, pp, pix, stg, mapY, quad, half, lane, valid, sbias, nbox);
        else
            epilogue_plain_row<true>(p, ti, tbase, valid, v, u, q, pp, Y, X, pix, 0, lane, sbias, half, 2);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&s.acce[accbuf]), 0u));
        accbuf ^= 1;
        if (accbuf == 0) accphase ^= 1u;
    }
    if (p.epi_tma && lane == 0) bulk_wait_all();  // boxes read and written before the CTA exits
}

template <bool kRms>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    conv_pair_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                     const __grid_constant__ CUtensorMap mapA16, const __grid_constant__ CUtensorMap mapB16,
                     const __grid_constant__ CUtensorMap mapY, const ConvParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw, p);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int rank = static_cast<int>(cluster_ctarank());
    if (threadIdx.x == 0) {
        *s.abort_flag = 0;
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(smem_u32(&s.full[i]), 1u);  // the even producer's arrive; both CTAs' bytes as transactions
            mbar_init(smem_u32(&s.empty[i]), 1u);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s.accf[i]), 1u);
            mbar_init(smem_u32(&s.acce[i]), static_cast<uint32_t>(2 * kPairEpiWarps));
        }
        mbar_init(smem_u32(s.drain), 1u);
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&s.xbar[i]), 64u);  // both warps of a lane quadrant
        fence_mbar_init();
    }
    // two accumulators, and with the fused RMS_norm two sets of quad-sum exchange columns
    const int tcols = 2 * p.acc_stride + (p.epi_tma == 3 ? 8 * (p.BN / 16) : 0);
    const uint32_t tmem_cols = tcols <= 32 ? 32u
                               : tcols <= 64 ? 64u
                               : tcols <= 128 ? 128u
                               : tcols <= 256 ? 256u
                                              : 512u;
    if (warp == kPairMmaWarp) {
        tmem_alloc_pair(smem_u32(s.tmem_slot), tmem_cols);
        tmem_relinquish_pair();
    }
    if (warp == kPairProducerWarp && lane == 0) {
        tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB);
        if (p.rem16) {
            tma_prefetch_desc(&mapA16);
            tma_prefetch_desc(&mapB16);
        }
        if (p.epi_tma) tma_prefetch_desc(&mapY);
    }
    // everything above touches only shared memory, TMEM and kernel parameters
    pdl_wait();
    if (p.bias_smem)  // visible to the epilogue after the barriers below
        for (int i = threadIdx.x; i < p.cout; i += blockDim.x) s.bias[i] = __ldg(p.bias + i);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers and TMEM exist before any remote arrive or pair MMA
    tc_fence_after();
    const uint32_t tmem_base = *s.tmem_slot;

    if (warp < kPairEpiWarps) {
        pair_epilogue<kRms>(p, s, tmem_base, warp, lane, rank, &mapY);
    } else if (warp == kPairProducerWarp) {
        if (lane == 0) pair_producer(p, s, &mapA, &mapB, &mapA16, &mapB16, rank);
    } else if (warp == kPairMmaWarp) {
        if (lane == 0 && rank == 0) pair_mma(p, s, tmem_base);
    }
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the even CTA's MMAs into both TMEMs are done; no remote arrives remain
    if (warp == kPairMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, tmem_cols);
    }
}

// The CTA-pair kernel takes the convs it covers unless VAE_CONV_CTA_PAIR=0 is
// set in the environment (the single-CTA kernel then runs them; for tests and
// measurements).
bool cta_pair_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("VAE_CONV_CTA_PAIR");
        return !(e != nullptr && e[0] == '0');
    }();
    return on;
}

// N tile width. halo3: the tile can use three-tap halo stages, which need
// BN <= 144 for three stages to fit; measured on GB300 they beat the widest
// per-tap tiles (BN = 256) by 1.3-1.7x at 288, 576 and 1152 output channels
// and tie at 192 and 768, while BN = 256 stays ahead when cout is a multiple of
// 256 (256, 512, 1024).
// The N tile of at most 144 columns with the least padding (ties: the widest).
int choose_bn_small(int cout) {
    const int c16 = (cout + 15) / 16 * 16;
    if (c16 <= 144) return c16;
    int best = 144, best_cost = (c16 + 143) / 144 * 144;
    for (int bn = 144; bn >= 64; bn -= 16) {
        const int cost = (c16 + bn - 1) / bn * bn;
        if (cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

// N tile of the pair GEMM (M = 256, N <= 256): the least padding, ties to the
// widest (1152 -> 192, 16384 -> 256, 576 -> 192).
int choose_bn_pair_gemm(int cout) {
    const int c16 = (cout + 15) / 16 * 16;
    if (c16 <= 256) return c16;
    int best = 256, best_cost = (c16 + 255) / 256 * 256;
    for (int bn = 256; bn >= 128; bn -= 16) {
        const int cost = (c16 + bn - 1) / bn * bn;
        if (cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

int choose_bn(int cout, bool halo3) {
    const int c16 = (cout + 15) / 16 * 16;
    if (halo3 && c16 % 256 != 0) {
        if (c16 <= 144) return c16;
        int best = 144, best_cost = (c16 + 143) / 144 * 144;
        for (int bn = 144; bn >= 64; bn -= 16) {
            const int cost = (c16 + bn - 1) / bn * bn;
            if (cost < best_cost) {
                best = bn;
                best_cost = cost;
            }
        }
        return best;
    }
    if (c16 <= 256) return c16;
    if (c16 >= 1024) return 256;  // widest MMA; measured faster at 1152 despite a ragged last tile
    int best = 256, best_cost = (c16 + 255) / 256 * 256;
    for (int bn = 256; bn >= 64; bn -= 16) {
        const int cost = (c16 + bn - 1) / bn * bn;
        if (cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

template <bool kRms>
int launch_pair(const ConvParams& p, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& ma16,
                const CUtensorMap& mb16, const CUtensorMap& my, size_t smem, int grid, cudaStream_t stream) {
    static CtxOnce attr_set;
    int dev = 0;
    VAE_CUDA_CHECK(cudaGetDevice(&dev));
    if (!attr_set.done(dev)) {
        VAE_CUDA_CHECK(
            cudaFuncSetAttribute(conv_pair_kernel<kRms>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem));
        attr_set.mark(dev);
    }
    VAE_CUDA_CHECK(launch_kernel(conv_pair_kernel<kRms>, dim3(grid), dim3(kPairThreads), smem, stream, ma, mb, ma16,
                                 mb16, my, p));
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

template <int kMode, bool kRms, int kVar = 0>
int launch(const ConvParams& p, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& ma16,
           const CUtensorMap& mb16, const CUtensorMap& my, size_t smem, int grid, cudaStream_t stream) {
    static CtxOnce attr_set;
    int dev = 0;
    VAE_CUDA_CHECK(cudaGetDevice(&dev));
    if (!attr_set.done(dev)) {
        VAE_CUDA_CHECK(
            cudaFuncSetAttribute(conv_kernel<kMode, kRms, kVar>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem));
        attr_set.mark(dev);
    }
    const int threads = kMode == kModeGather ? 320 : (p.refl ? 224 : 192);
    VAE_CUDA_CHECK(launch_kernel(conv_kernel<kMode, kRms, kVar>, dim3(grid), dim3(threads), smem, stream, ma, mb, ma16,
                                 mb16, my, p));
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

}  // namespace

// The epilogue reads the bias from a shared-memory copy (VAE_CONV_BIAS_SMEM=0
// turns it off): the global loads miss the small L1 left beside the pipeline's
// shared memory. Neutral for the plain 1024^2 conv (0.324 ms either way), 7 %
// faster for the epilogue-bound fused RMS_norm conv (0.466 against 0.498 ms).
bool bias_smem_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("VAE_CONV_BIAS_SMEM");
        return !(e != nullptr && e[0] == '0');
    }();
    return on;
}

int conv_gn_chunks(int h_in, int w_in, bool up, bool down) {
    // the tiling of conv_run: the virtual grid, its tile shape and the parity classes
    const int hv = down ? h_in / 2 : h_in, wv = down ? w_in / 2 : w_in;
    if (hv < 1 || wv < 1) return -1;
    const int Wt = wv >= kBM ? kBM : wv, R = wv >= kBM ? 1 : kBM / wv;
    const long long tiles = static_cast<long long>((hv + R - 1) / R) * (up ? 4 : 1) * ((wv + Wt - 1) / Wt);
    return tiles * kEpiWarps >= (1LL << 31) ? -1 : static_cast<int>(tiles * kEpiWarps);
}

int conv_validate(const ConvArgs& a) {
    if (a.x == nullptr || a.w == nullptr)
        return set_error(VAE_ERR_ARG, "conv: x and w must be non-NULL");
    if (a.taps != 1 && a.taps != 9 && a.taps != 27) return set_error(VAE_ERR_ARG, "conv: taps must be 1, 9 or 27");
    if (a.frames_in < 1 || (a.taps != 27 && (a.frames_in != 1 || a.t_up)))
        return set_error(VAE_ERR_ARG, "conv: frames_in=%d / temporal upsample need the 3x3x3 conv", a.frames_in);
    if (a.taps == 27 && (a.rms_out != nullptr || a.dup_src != nullptr || a.out_nchw))
        return set_error(VAE_ERR_ARG, "conv: the 3x3x3 conv has no fused norm, DupUp or NCHW output");
    if (a.subpix && (!a.up || a.taps != 9 || a.rms_out != nullptr))
        return set_error(VAE_ERR_ARG, "conv: the sub-pixel form is the 3x3 up conv's (no fused norm)");
    if (a.out_scale != 1.0f && (!a.out_f16 || !(a.out_scale > 0.0f) || !std::isfinite(a.out_scale)))
        return set_error(VAE_ERR_ARG, "conv: an output scale needs f16 output and a finite positive value");
    if (a.n < 1 || a.h_in < 1 || a.w_in < 1)
        return set_error(VAE_ERR_SHAPE, "conv: n=%d h=%d w=%d must be >= 1", a.n, a.h_in, a.w_in);
    if (a.cin < 16 || a.cin % 16 != 0 || a.cin > 8192)
        return set_error(VAE_ERR_SHAPE, "conv: cin=%d must be a multiple of 16 in [16, 8192]", a.cin);
    if (a.cout < 1 || a.cout > (1 << 20))
        return set_error(VAE_ERR_SHAPE, "conv: cout=%d out of [1, 2^20]", a.cout);
    if (a.taps == 1 && (a.up || a.rep || a.refl || a.down))
        return set_error(VAE_ERR_ARG, "conv1x1: no upsample, downsample or padding mode");
    if (static_cast<int>(a.rep) + static_cast<int>(a.refl) > 1)
        return set_error(VAE_ERR_ARG, "conv: at most one padding mode (replicate or reflect)");
    if (a.refl && a.up) return set_error(VAE_ERR_ARG, "conv: reflect padding does not combine with the upsample");
    if (a.down && (a.up || a.taps != 9 || a.subpix))
        return set_error(VAE_ERR_ARG, "conv: the downsample is a plain 3x3 conv (no upsample)");
    if (a.taps == 27 && a.refl) return set_error(VAE_ERR_ARG, "conv: the 3x3x3 conv takes zero or replicate padding");
    if ((a.refl || a.down) && (a.h_in < 2 || a.w_in < 2))
        return set_error(VAE_ERR_SHAPE, "conv: reflect padding and the downsample need h, w >= 2 (h=%d w=%d)",
                         a.h_in, a.w_in);
    if (a.down && a.dup_src != nullptr) return set_error(VAE_ERR_ARG, "conv: no DupUp on the downsample");
    if (a.gn_part != nullptr) {
        if (a.taps != 9 || a.subpix || a.out_f16 || a.out_nchw || a.rms_out != nullptr || a.y == nullptr)
            return set_error(VAE_ERR_ARG, "conv: GroupNorm statistics need a 2-D 3x3 conv with an f32 output");
        const int cpg = a.gn_groups >= 1 && a.cout % a.gn_groups == 0 ? a.cout / a.gn_groups : 0;
        if (a.cout % 16 != 0 || !(cpg == 4 || cpg == 8 || (cpg > 0 && cpg % 16 == 0)))
            return set_error(VAE_ERR_SHAPE,
                             "conv: GroupNorm statistics need cout %% 16 == 0 and C/groups in {4, 8} or a multiple "
                             "of 16 (cout=%d groups=%d)", a.cout, a.gn_groups);
        if (!aligned16(a.gn_part)) return set_error(VAE_ERR_ALIGN, "conv: the statistics workspace must be 16-byte aligned");
    }
    if (!aligned16(a.x) || !aligned16(a.w))
        return set_error(VAE_ERR_ALIGN, "conv: x and w must be 16-byte aligned");
    const long long H = a.up ? 2LL * a.h_in : a.h_in, W = a.up ? 2LL * a.w_in : a.w_in;
    const long long F = a.t_up ? 2LL * a.frames_in - 1 : a.frames_in;
    if (static_cast<long long>(a.n) * F * H * W >= (1LL << 31) || static_cast<long long>(a.w_in) >= (1LL << 31) ||
        static_cast<long long>(a.n) * a.frames_in * a.h_in * a.w_in >= (1LL << 31))
        return set_error(VAE_ERR_SHAPE, "conv: too many pixels");
    if (a.out_nchw && (a.out_f16 || a.residual != nullptr))
        return set_error(VAE_ERR_ARG, "conv: NCHW output is f32 without residual");
    if (a.rms_out != nullptr) {
        if (a.rms_gamma == nullptr || !aligned16(a.rms_gamma) || a.cout > 144 || a.cout % 16 != 0 || a.out_nchw ||
            a.out_f16 || a.silu)
            return set_error(VAE_ERR_ARG, "conv: the fused RMS_norm needs gamma, cout %% 16 == 0, cout <= 144, f32 y");
        if (!aligned16(a.rms_out)) return set_error(VAE_ERR_ALIGN, "conv: rms_out must be 16-byte aligned");
    } else if (a.y == nullptr) {
        return set_error(VAE_ERR_ARG, "conv: y must be non-NULL");
    }
    if (a.dup_src != nullptr) {
        if (!a.up || a.dup_cin < 1 || a.dup_repeats < 1 || a.dup_factor < 1)
            return set_error(VAE_ERR_ARG, "conv: DupUp needs the upsample fold and a valid shuffle");
        const long long jmax = static_cast<long long>(a.cout - 1) * a.dup_factor + a.dup_ftoff + 3;
        if (jmax / a.dup_repeats >= a.dup_cin)
            return set_error(VAE_ERR_SHAPE, "conv: DupUp reads past the source channels");
    }
    return VAE_OK;
}

int conv_run(const ConvArgs& a, cudaStream_t stream) {
    int rc = conv_validate(a);
    if (rc != VAE_OK) return rc;
    rc = check_device();
    if (rc != VAE_OK) return rc;
    DevStatus* st = device_status_ptr();
    if (st == nullptr) return VAE_ERR_CUDA;
    const int nsm = sm_count();
    if (nsm <= 0) return set_error(VAE_ERR_CUDA, "conv: no SM count");

    ConvParams p{};
    p.frames_in = a.frames_in;
    p.t_up = a.t_up ? 1 : 0;
    p.frames_out = a.t_up ? 2 * a.frames_in - 1 : a.frames_in;
    p.nkt = a.taps == 27 ? 3 : 1;
    p.n = a.n * p.frames_out;  // output images: the tile space
    p.n_in = a.n * a.frames_in;
    p.hs = a.h_in;
    p.ws = a.w_in;
    p.down = a.down ? 1 : 0;
    p.refl = a.refl ? 1 : 0;
    p.hv = a.down ? a.h_in / 2 : a.h_in;  // the downsample tiles its output grid
    p.wv = a.down ? a.w_in / 2 : a.w_in;
    p.cin = a.cin;
    p.cout = a.cout;
    p.subpix = a.subpix ? 1 : 0;
    p.taps = a.subpix ? 4 : a.taps;  // taps per parity class
    p.up = a.up ? 1 : 0;
    p.rep = a.rep ? 1 : 0;
    p.H = p.up ? 2 * a.h_in : p.hv;
    p.W = p.up ? 2 * a.w_in : p.wv;
    // per-pixel source remaps: gather threads (reflect only where no halo box can serve)
    const bool refl_halo = a.refl && !a.down && !a.no_halo && a.taps == 9 && p.wv >= kBM;
    // the downsample as TMA boxes: even widths, one-row tiles; with reflect padding
    // the last tile must hold at least two output pixels (the fix copies within a box)
    const bool down_tma = a.down && !a.rep && a.taps == 9 && a.w_in % 2 == 0 && p.wv >= kBM &&
                          (!a.refl || (p.wv - 1) % kBM != 0);
    const bool gather = a.rep || (a.down && !down_tma) || (a.refl && !a.down && !refl_halo);
    if (p.wv >= kBM) {
        p.Wt = kBM;
        p.R = 1;
    } else {
        p.Wt = p.wv;
        p.R = kBM / p.wv;
    }
    p.tiles_x = (p.wv + p.Wt - 1) / p.Wt;
    p.tiles_y = (p.hv + p.R - 1) / p.R;
    p.npar = p.up ? 4 : 1;
    // Geometry that allows a halo box: a tile is 128 pixels of one row, 3x3 taps,
    // zero padding (the TMA box fills out-of-range pixels with zeros).
    const bool halo_geom = !gather && !a.down && !a.no_halo && (a.taps == 9 || a.taps == 27) && p.R == 1 &&
                           p.Wt == kBM;
    // reflect padding needs the three-tap halo stages (the edge fix runs per stage): N <= 144
    p.BN = refl_halo ? choose_bn_small(a.cout) : choose_bn(a.cout, halo_geom);
    p.b_rows = p.BN;
    p.n_tiles = (a.cout + p.BN - 1) / p.BN;
    p.acc_stride = (p.BN + 31) / 32 * 32;
    p.kchunks = (a.cin + kBK - 1) / kBK;
    const long long m_tiles = static_cast<long long>(p.n) * p.tiles_y * p.npar * p.tiles_x;
    const long long total = m_tiles * p.n_tiles;
    if (total >= (1LL << 31)) return set_error(VAE_ERR_SHAPE, "conv: too many tiles");
    p.total_tiles = static_cast<int>(total);
    // Two K chunks per stage halve the per-stage barrier/commit overhead of the
    // MMA thread (measured +10-21 % on the wide convs) when two such stages fit.
    p.ks = 1;
    if (!gather && p.kchunks >= 2 && 2 * 2 * (kABytes + p.BN * 128) <= kMaxSmem - 1024 - kTail) p.ks = 2;
    const int stage_bytes = p.ks * (kABytes + p.BN * 128);
    p.stages = std::min(kMaxStages, (kMaxSmem - 1024 - kTail) / stage_bytes);
    p.a_tx = static_cast<uint32_t>(128 * p.Wt * p.R);
    p.x = static_cast<const __half*>(a.x);
    p.bias = a.bias;
    p.residual = a.residual;
    p.y = a.y;
    p.oscale = a.oscale;
    p.silu = a.silu ? 1 : 0;
    p.out_f16 = a.out_f16 ? 1 : 0;
    p.out_scale = a.out_scale;
    p.vec_ok = (a.cout % 16 == 0) && (a.y == nullptr || aligned16(a.y)) && (a.residual == nullptr || aligned16(a.residual)) &&
               (a.bias == nullptr || aligned16(a.bias));
    p.v8_ok = p.vec_ok && (a.y == nullptr || (reinterpret_cast<uintptr_t>(a.y) & 31) == 0) &&
              (a.residual == nullptr || (reinterpret_cast<uintptr_t>(a.residual) & 31) == 0) ? 1 : 0;
    p.res_prefetch = (p.residual != nullptr && p.vec_ok && p.R == 1 && !p.up && p.n_tiles == 1 &&
                      static_cast<long long>(p.Wt) * a.cout * 4 < (1LL << 31))
                         ? 1
                         : 0;
    p.out_nchw = a.out_nchw ? 1 : 0;
    p.keep_lo = a.keep_lo;
    p.keep_hi = a.keep_hi;
    p.dst_row0 = a.dst_row0;
    p.plane = a.plane;
    if (p.out_nchw && p.keep_hi <= p.keep_lo) {
        p.keep_lo = 0;
        p.keep_hi = p.H;
        p.dst_row0 = 0;
        p.plane = static_cast<long long>(p.H) * p.W;
    }
    p.dup_src = a.dup_src;
    p.dup_cin = a.dup_cin;
    p.dup_factor = a.dup_factor;
    p.dup_repeats = a.dup_repeats;
    p.dup_ftoff = a.dup_ftoff;
    // (o*F + off)/R = o*(F/R) + off/R exactly when R divides F.
    p.dup_step = 0;
    if (a.dup_src != nullptr && a.dup_factor % a.dup_repeats == 0 && a.dup_factor / a.dup_repeats <= 2) {
        p.dup_step = a.dup_factor / a.dup_repeats;
        for (int c = 0; c < 4; ++c) p.dup_base[c] = (a.dup_ftoff + c) / a.dup_repeats;
    }
    p.dup_v8 = (a.dup_src != nullptr && a.dup_cin % 8 == 0 && (reinterpret_cast<uintptr_t>(a.dup_src) & 31) == 0) ? 1 : 0;
    p.dup_prefetch = (a.dup_src != nullptr && p.R == 1 && a.dup_cin % 4 == 0 && aligned16(a.dup_src) &&
                      static_cast<long long>(p.Wt) * a.dup_cin * 4 < (1LL << 31))
                         ? 1
                         : 0;
    p.rms_gamma = a.rms_gamma;
    p.rms_out = static_cast<__half*>(a.rms_out);
    p.rms_silu = a.rms_silu ? 1 : 0;
    p.gn_part = static_cast<float4*>(a.gn_part);
    if (a.gn_part != nullptr) {
        p.gn_groups = a.gn_groups;
        p.gn_cpg = a.cout / a.gn_groups;
        p.gn_nchunks = p.tiles_y * p.npar * p.tiles_x * kEpiWarps;
        if (p.gn_cpg > 16 && p.BN % p.gn_cpg != 0)
            return set_error(VAE_ERR_SHAPE, "conv: a group of %d channels straddles the %d-column N tiles", p.gn_cpg,
                             p.BN);
    }
    p.status = st;
    p.timeout_ns = wait_timeout_ns();

    CUtensorMap ma{}, mb{}, ma16{}, mb16{}, my{};
    const int wtaps = a.subpix ? 16 : a.taps;  // weight taps: the sub-pixel form holds 4 per parity class
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(a.cin), static_cast<uint64_t>(wtaps),
                                  static_cast<uint64_t>(a.cout)};
        const uint64_t strides[2] = {static_cast<uint64_t>(a.cin) * 2, static_cast<uint64_t>(wtaps) * a.cin * 2};
        const uint32_t box[3] = {static_cast<uint32_t>(kBK), 1u, static_cast<uint32_t>(p.BN)};
        rc = encode_tiled(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.w, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != VAE_OK) return rc;
    }
    int mode = gather ? kModeGather : kModeTma;
    // Halo stages: three-tap stages whenever three fit (any cin); otherwise one
    // tap per stage, which measured faster than per-tap A tiles only for
    // narrow inputs (cin <= 192).
    const int st3 = (kMaxSmem - 1024 - kTail) / (kHaloBytes + 3 * p.BN * 128);
    // (The one-tap halo ring has no sub-pixel form: that variant takes the halo
    // path only with three-tap stages.)
    if (mode == kModeTma && halo_geom && (st3 >= 3 || (a.cin <= 192 && !a.subpix && !a.refl))) {
        // one 130-pixel halo box per (ky, chunk), shared by the three kx taps
        const uint64_t dims[4] = {static_cast<uint64_t>(a.cin), static_cast<uint64_t>(p.wv),
                                  static_cast<uint64_t>(p.hv), static_cast<uint64_t>(p.n_in)};
        const uint64_t strides[3] = {static_cast<uint64_t>(a.cin) * 2, static_cast<uint64_t>(p.wv) * a.cin * 2,
                                     static_cast<uint64_t>(p.hv) * p.wv * a.cin * 2};
        const uint32_t box[4] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(kHaloRows), 1u, 1u};
        if (encode_tiled(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, a.x, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) == VAE_OK) {
            mode = kModeHalo;
            p.halo = 1;
            p.a_tx = static_cast<uint32_t>(kHaloRows * 128);
            // Preferred: a stage holds the halo box and all three kx taps (12
            // MMAs per 64-channel chunk) when three such stages fit; else one
            // tap per stage with a separate ring of halo boxes.
            if (st3 >= 3) {
                p.ks = 3;
                p.stages = std::min(kMaxStages, st3);
                p.a_stages = p.stages;
                if (a.cin % kBK == 16 && a.cin > kBK) {
                    // exact 16-channel boxes for the remainder instead of zero-filled 64-channel ones
                    const uint32_t box16[4] = {16u, static_cast<uint32_t>(kHaloRows), 1u, 1u};
                    const uint64_t bdims[3] = {static_cast<uint64_t>(a.cin), static_cast<uint64_t>(wtaps),
                                               static_cast<uint64_t>(a.cout)};
                    const uint64_t bstrides[2] = {static_cast<uint64_t>(a.cin) * 2,
                                                  static_cast<uint64_t>(wtaps) * a.cin * 2};
                    const uint32_t bbox16[3] = {16u, 1u, static_cast<uint32_t>(p.BN)};
                    if (encode_tiled(&ma16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, a.x, dims, strides, box16,
                                     CU_TENSOR_MAP_SWIZZLE_32B) == VAE_OK &&
                        encode_tiled(&mb16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.w, bdims, bstrides, bbox16,
                                     CU_TENSOR_MAP_SWIZZLE_32B) == VAE_OK) {
                        p.rem16 = 1;
                        p.kfull = a.cin / kBK;
                    } else {
                        clear_error();
                    }
                }
            } else {
                p.ks = 1;
                p.a_stages = 3;
                p.stages = std::min(kMaxStages, (kMaxSmem - 1024 - kTail - p.a_stages * kHaloBytes) / (p.BN * 128));
            }
        } else {
            clear_error();
        }
    }
    if (a.refl && !a.down && mode != kModeHalo) {
        // only the halo stages carry the reflect fix: anything else gathers
        mode = kModeGather;
        p.ks = 1;
        p.stages = std::min(kMaxStages, (kMaxSmem - 1024 - kTail) / (kABytes + p.BN * 128));
    }
    if (mode == kModeTma && down_tma) {
        // x as (channel, column parity, W/2, row, image): pixel (row, 2j + parity)
        const uint64_t dims[5] = {static_cast<uint64_t>(a.cin), 2u, static_cast<uint64_t>(a.w_in / 2),
                                  static_cast<uint64_t>(a.h_in), static_cast<uint64_t>(p.n_in)};
        const uint64_t strides[4] = {static_cast<uint64_t>(a.cin) * 2, static_cast<uint64_t>(a.cin) * 4,
                                     static_cast<uint64_t>(a.w_in) * a.cin * 2,
                                     static_cast<uint64_t>(a.h_in) * a.w_in * a.cin * 2};
        const uint32_t box[5] = {static_cast<uint32_t>(kBK), 1u, static_cast<uint32_t>(kBM), 1u, 1u};
        if (encode_tiled(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, a.x, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) == VAE_OK) {
            p.down_tma = 1;
        } else {
            clear_error();
            mode = kModeGather;
            p.ks = 1;
            p.stages = std::min(kMaxStages, (kMaxSmem - 1024 - kTail) / (kABytes + p.BN * 128));
        }
    } else if (mode == kModeTma) {
        const uint64_t dims[4] = {static_cast<uint64_t>(a.cin), static_cast<uint64_t>(p.wv),
                                  static_cast<uint64_t>(p.hv), static_cast<uint64_t>(p.n_in)};
        const uint64_t strides[3] = {static_cast<uint64_t>(a.cin) * 2, static_cast<uint64_t>(p.wv) * a.cin * 2,
                                     static_cast<uint64_t>(p.hv) * p.wv * a.cin * 2};
        const uint32_t box[4] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(p.Wt),
                                 static_cast<uint32_t>(p.R), 1u};
        if (encode_tiled(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, a.x, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) != VAE_OK) {
            clear_error();
            mode = kModeGather;  // shapes TMA cannot describe: gather threads build the A tiles
            p.ks = 1;
            p.stages = std::min(kMaxStages, (kMaxSmem - 1024 - kTail) / (kABytes + p.BN * 128));
        }
    }
    const int grid = static_cast<int>(std::min<long long>(total, nsm));
    // The staged TMA epilogue's output view: a 128-pixel row segment, plain f32
    // output written whole (no residual) or added onto itself (residual == y, no
    // SiLU after). The add-reduction keeps the register path's rounding order
    // only without upsampling and DupUp (whose add comes after the residual's).
    const bool res_self = a.residual != nullptr && a.residual == a.y && !a.silu && !p.up && a.dup_src == nullptr;
    auto encode_epi = [&]() -> bool {
        if (!(mode != kModeGather && p.R == 1 && p.Wt == kBM && !p.out_f16 && !p.out_nchw && a.rms_out == nullptr &&
              a.cout % 16 == 0 && a.y != nullptr && aligned16(a.y) &&
              (a.residual == nullptr || res_self || a.gn_part != nullptr)))
            return false;
        int erc;
        if (p.up) {  // y viewed as (channel, column parity, W/2, row, image)
            const uint64_t dims[5] = {static_cast<uint64_t>(a.cout), 2u, static_cast<uint64_t>(p.W / 2),
                                      static_cast<uint64_t>(p.H), static_cast<uint64_t>(p.n)};
            const uint64_t strides[4] = {static_cast<uint64_t>(a.cout) * 4, static_cast<uint64_t>(a.cout) * 8,
                                         static_cast<uint64_t>(p.W) * a.cout * 4,
                                         static_cast<uint64_t>(p.H) * p.W * a.cout * 4};
            const uint32_t box[5] = {16u, 1u, 32u, 1u, 1u};
            erc = encode_tiled(&my, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, a.y, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_64B);
        } else {
            const uint64_t dims[4] = {static_cast<uint64_t>(a.cout), static_cast<uint64_t>(p.W),
                                      static_cast<uint64_t>(p.H), static_cast<uint64_t>(p.n)};
            const uint64_t strides[3] = {static_cast<uint64_t>(a.cout) * 4, static_cast<uint64_t>(p.W) * a.cout * 4,
                                         static_cast<uint64_t>(p.H) * p.W * a.cout * 4};
            const uint32_t box[4] = {16u, 32u, 1u, 1u};
            erc = encode_tiled(&my, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.y, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_64B);
        }
        if (erc != VAE_OK) {
            clear_error();
            return false;
        }
        return true;
    };
    // CTA pairs for a 1x1 conv over one row of pixels (the plain GEMMs
    // [pixels][cin] x [cout][cin]^T): adjacent 128-pixel column tiles share every
    // weight tile, half in each SM; a stage holds kGemmPairKs 64-channel chunks.
    if (cta_pair_enabled() && !a.no_pair && a.taps == 1 && mode == kModeTma && p.hv == 1 && p.R == 1 &&
        p.Wt == kBM && p.tiles_x >= 2 && !p.up && !a.subpix && !a.refl && !a.down && !a.rep &&
        a.gn_part == nullptr && a.rms_out == nullptr && !p.out_nchw && a.dup_src == nullptr && nsm >= 2) {
        ConvParams q = p;
        q.pair = 1;
        q.gemm = 1;
        q.BN = choose_bn_pair_gemm(a.cout);
        q.b_rows = q.BN / 2;
        q.n_tiles = (a.cout + q.BN - 1) / q.BN;
        q.acc_stride = (q.BN + 31) / 32 * 32;
        q.typ_tiles = (q.tiles_x + 1) / 2;  // column-tile pairs
        const long long pt = static_cast<long long>(q.n) * q.typ_tiles * q.n_tiles;
        if (pt >= (1LL << 31)) return set_error(VAE_ERR_SHAPE, "conv: too many tiles");
        q.pair_tiles = static_cast<int>(pt);
        q.halo = 0;
        q.a_stages = 0;
        q.rem16 = 0;
        q.a_tx = static_cast<uint32_t>(kABytes);
        q.res_prefetch = 0;
        CUtensorMap pb{};
        const uint64_t bdims[3] = {static_cast<uint64_t>(a.cin), 1u, static_cast<uint64_t>(a.cout)};
        const uint64_t bstrides[2] = {static_cast<uint64_t>(a.cin) * 2, static_cast<uint64_t>(a.cin) * 2};
        const uint32_t bbox[3] = {static_cast<uint32_t>(kBK), 1u, static_cast<uint32_t>(q.b_rows)};
        bool ok = encode_tiled(&pb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.w, bdims, bstrides, bbox,
                               CU_TENSOR_MAP_SWIZZLE_128B) == VAE_OK;
        if (ok) {
            CUtensorMap pmy{};
            q.epi_tma = 0;
            q.stg_bytes = 0;
            {
                const ConvParams keep = p;  // encode_epi() reads p; the pair shares its output view
                p = q;
                if (encode_epi()) {
                    q.epi_tma = res_self ? 2 : 1;
                    q.stg_bytes = kPairStgBytes;
                    pmy = my;
                }
                p = keep;
            }
            const size_t bias_bytes = static_cast<size_t>(a.cout * 4 + 15) / 16 * 16;
            q.bias_smem = (bias_smem_enabled() && a.bias != nullptr && aligned16(a.bias)) ? 1 : 0;
            const size_t fixed = 1024 + static_cast<size_t>(q.stg_bytes) + (q.bias_smem ? bias_bytes : 0) + kTail;
            for (q.ks = std::min(kGemmPairKs, q.kchunks); q.ks >= 1; --q.ks) {
                const size_t stage_bytes =
                    static_cast<size_t>(q.ks) * (static_cast<size_t>(kABytes) + static_cast<size_t>(q.b_rows) * 128u);
                const int st = static_cast<int>((kMaxSmem - fixed) / stage_bytes);
                if (st >= 3 || (q.ks == 1 && st >= 2)) {
                    q.stages = std::min(kMaxStages, st);
                    const size_t smem = fixed + static_cast<size_t>(q.stages) * stage_bytes;
                    const int pgrid = 2 * static_cast<int>(std::min<long long>(pt, nsm / 2));
                    return launch_pair<false>(q, ma, pb, ma, pb, pmy, smem, pgrid, stream);
                }
            }
        }
        clear_error();
    }
    // CTA pairs (cta_group::2): two row tiles of one column block share every
    // weight tile, half in each SM, on the three-tap halo stages. Plain 2-D 3x3
    // convs with zero padding (with or without the nearest-2x fold) whose
    // images have at least two tile rows; everything else runs on single CTAs.
    // The fused RMS_norm rides along when one N tile holds a pixel's channels and
    // the conv writes only the normalised f16 rows.
    const bool pair_rms = a.rms_out != nullptr && a.y == nullptr && a.residual == nullptr && a.dup_src == nullptr &&
                          !a.up && a.cout <= 144 && a.cout % 16 == 0 && aligned16(a.rms_gamma) &&
                          aligned16(a.rms_out);
    if (cta_pair_enabled() && halo_geom && !a.no_pair && (mode == kModeTma || mode == kModeHalo) && a.taps == 9 &&
        !a.subpix && !a.refl && !a.down && a.gn_part == nullptr && (a.rms_out == nullptr || pair_rms) &&
        p.tiles_y >= 2 && nsm >= 2) {
        ConvParams q = p;
        q.pair = 1;
        q.BN = choose_bn_small(a.cout);
        q.b_rows = q.BN / 2;
        q.n_tiles = (a.cout + q.BN - 1) / q.BN;
        q.acc_stride = (q.BN + 31) / 32 * 32;
        q.typ_tiles = (q.tiles_y + 1) / 2;
        const long long pt = static_cast<long long>(q.n) * q.typ_tiles * q.npar * q.tiles_x * q.n_tiles;
        if (pt >= (1LL << 31)) return set_error(VAE_ERR_SHAPE, "conv: too many tiles");
        q.pair_tiles = static_cast<int>(pt);
        q.halo = 1;
        q.ks = 3;
        q.a_tx = static_cast<uint32_t>(kHaloRows * 128);
        q.res_prefetch = (q.residual != nullptr && q.vec_ok && !q.up && q.n_tiles == 1 &&
                          static_cast<long long>(q.Wt) * a.cout * 4 < (1LL << 31))
                             ? 1
                             : 0;
        CUtensorMap pa{}, pb{}, pa16{}, pb16{};
        bool ok = true;
        {  // one 130-pixel halo box per (ky, chunk) of this CTA's row tile
            const uint64_t dims[4] = {static_cast<uint64_t>(a.cin), static_cast<uint64_t>(q.wv),
                                      static_cast<uint64_t>(q.hv), static_cast<uint64_t>(q.n_in)};
            const uint64_t strides[3] = {static_cast<uint64_t>(a.cin) * 2, static_cast<uint64_t>(q.wv) * a.cin * 2,
                                         static_cast<uint64_t>(q.hv) * q.wv * a.cin * 2};
            const uint32_t box[4] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(kHaloRows), 1u, 1u};
            ok = encode_tiled(&pa, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, a.x, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B) == VAE_OK;
            const uint64_t bdims[3] = {static_cast<uint64_t>(a.cin), 9u, static_cast<uint64_t>(a.cout)};
            const uint64_t bstrides[2] = {static_cast<uint64_t>(a.cin) * 2, static_cast<uint64_t>(9) * a.cin * 2};
            const uint32_t bbox[3] = {static_cast<uint32_t>(kBK), 1u, static_cast<uint32_t>(q.b_rows)};
            ok = ok && encode_tiled(&pb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.w, bdims, bstrides, bbox,
                                    CU_TENSOR_MAP_SWIZZLE_128B) == VAE_OK;
            q.rem16 = 0;
            q.kfull = 0;
            if (ok && a.cin % kBK == 16 && a.cin > kBK) {
                // exact 16-channel boxes for the remainder instead of zero-filled 64-channel ones
                const uint32_t box16[4] = {16u, static_cast<uint32_t>(kHaloRows), 1u, 1u};
                const uint32_t bbox16[3] = {16u, 1u, static_cast<uint32_t>(q.b_rows)};
                if (encode_tiled(&pa16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, a.x, dims, strides, box16,
                                 CU_TENSOR_MAP_SWIZZLE_32B) == VAE_OK &&
                    encode_tiled(&pb16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.w, bdims, bstrides, bbox16,
                                 CU_TENSOR_MAP_SWIZZLE_32B) == VAE_OK) {
                    q.rem16 = 1;
                    q.kfull = a.cin / kBK;
                }
            }
        }
        if (ok) {
            CUtensorMap pmy{};
            q.epi_tma = 0;
            q.stg_bytes = 0;
            {
                // encode_epi() reads p; the pair shares its output view
                const ConvParams keep = p;
                p = q;
                if (pair_rms) {
                    const uint64_t dims[4] = {static_cast<uint64_t>(a.cout), static_cast<uint64_t>(q.W),
                                              static_cast<uint64_t>(q.H), static_cast<uint64_t>(q.n)};
                    const uint64_t strides[3] = {static_cast<uint64_t>(a.cout) * 2,
                                                 static_cast<uint64_t>(q.W) * a.cout * 2,
                                                 static_cast<uint64_t>(q.H) * q.W * a.cout * 2};
                    const uint32_t box[4] = {16u, 32u, 1u, 1u};
                    if (encode_tiled(&pmy, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, a.rms_out, dims, strides, box,
                                     CU_TENSOR_MAP_SWIZZLE_32B) == VAE_OK) {
                        q.epi_tma = 3;
                        q.stg_bytes = kPairStgBytes;
                    } else {
                        ok = false;
                    }
                } else if (encode_epi()) {
                    q.epi_tma = res_self ? 2 : 1;
                    q.stg_bytes = kPairStgBytes;
                    pmy = my;
                }
                p = keep;
            }
            const size_t bias_bytes = static_cast<size_t>(a.cout * 4 + 15) / 16 * 16;
            q.bias_smem = (bias_smem_enabled() && a.bias != nullptr && aligned16(a.bias)) ? 1 : 0;
            const size_t stage_bytes = static_cast<size_t>(kHaloBytes) + 3u * static_cast<size_t>(q.b_rows) * 128u;
            const size_t fixed = 1024 + static_cast<size_t>(q.stg_bytes) + (q.bias_smem ? bias_bytes : 0) + kTail;
            const int st = static_cast<int>((kMaxSmem - fixed) / stage_bytes);
            if (ok && st >= 3) {
                q.stages = std::min(kMaxStages, st);
                q.a_stages = q.stages;
                const size_t smem = fixed + static_cast<size_t>(q.stages) * stage_bytes;
                const int pgrid = 2 * static_cast<int>(std::min<long long>(pt, nsm / 2));
                return q.epi_tma == 3 ? launch_pair<true>(q, pa, pb, pa16, pb16, pmy, smem, pgrid, stream)
                                      : launch_pair<false>(q, pa, pb, pa16, pb16, pmy, smem, pgrid, stream);
            }
        }
        clear_error();
    }
    size_t ring = mode == kModeHalo
                      ? static_cast<size_t>(p.a_stages) * kHaloBytes + static_cast<size_t>(p.stages) * p.ks * p.BN * 128
                      : static_cast<size_t>(p.stages) * p.ks * (kABytes + p.BN * 128);
    if (1024 + ring + kEpiWarps * kStgBytes + kTail <= kMaxSmem && encode_epi())
        // with statistics the values are needed in registers: the residual is read, not added
        p.epi_tma = res_self && a.gn_part == nullptr ? 2 : 1;
    // Fused RMS_norm with f16 rows only (a ResNet's first conv): staged f16 TMA boxes.
    if (mode != kModeGather && !p.epi_tma && a.rms_out != nullptr && a.y == nullptr && a.residual == nullptr &&
        a.dup_src == nullptr && !p.up && p.R == 1 && p.Wt == kBM && p.n_tiles == 1 && a.cout % 16 == 0 &&
        aligned16(a.rms_gamma) && 1024 + ring + kEpiWarps * kStgBytes + kTail <= kMaxSmem) {
        const uint64_t dims[4] = {static_cast<uint64_t>(a.cout), static_cast<uint64_t>(p.W),
                                  static_cast<uint64_t>(p.H), static_cast<uint64_t>(p.n)};
        const uint64_t strides[3] = {static_cast<uint64_t>(a.cout) * 2, static_cast<uint64_t>(p.W) * a.cout * 2,
                                     static_cast<uint64_t>(p.H) * p.W * a.cout * 2};
        const uint32_t box[4] = {16u, 32u, 1u, 1u};
        if (encode_tiled(&my, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, a.rms_out, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_32B) == VAE_OK)
            p.epi_tma = 3;
        else
            clear_error();
    }
    p.stg_bytes = p.epi_tma ? kEpiWarps * kStgBytes : 0;
    size_t smem = 1024 + ring + p.stg_bytes + kTail;
    // A shared-memory copy of the bias where it fits: the epilogue's bias reads
    // otherwise miss the small L1 left beside the pipeline's shared memory.
    const size_t bias_bytes = static_cast<size_t>(a.cout * 4 + 15) / 16 * 16;
    if (bias_smem_enabled() && a.bias != nullptr && aligned16(a.bias) && smem + bias_bytes <= kMaxSmem) {
        p.bias_smem = 1;
        smem += bias_bytes;
    }
    if (a.taps == 27) {  // the 3x3x3 instantiations (no fused norm)
        if (mode == kModeHalo) return launch<kModeHalo, false, 1>(p, ma, mb, ma16, mb16, my, smem, grid, stream);
        if (mode == kModeGather) return launch<kModeGather, false, 1>(p, ma, mb, ma, mb, my, smem, grid, stream);
        return launch<kModeTma, false, 1>(p, ma, mb, ma, mb, my, smem, grid, stream);
    }
    if (a.gn_part != nullptr) {  // the 2-D conv with the GroupNorm statistics epilogue
        if (mode == kModeHalo) return launch<kModeHalo, false, 3>(p, ma, mb, ma16, mb16, my, smem, grid, stream);
        if (mode == kModeGather) return launch<kModeGather, false, 3>(p, ma, mb, ma, mb, my, smem, grid, stream);
        return launch<kModeTma, false, 3>(p, ma, mb, ma, mb, my, smem, grid, stream);
    }
    if (a.subpix) {  // the sub-pixel up conv instantiations
        if (mode == kModeHalo) return launch<kModeHalo, false, 2>(p, ma, mb, ma16, mb16, my, smem, grid, stream);
        if (mode == kModeGather) return launch<kModeGather, false, 2>(p, ma, mb, ma, mb, my, smem, grid, stream);
        return launch<kModeTma, false, 2>(p, ma, mb, ma, mb, my, smem, grid, stream);
    }
    if (p.rms_out != nullptr) {
        if (mode == kModeHalo) return launch<kModeHalo, true>(p, ma, mb, ma16, mb16, my, smem, grid, stream);
        if (mode == kModeGather) return launch<kModeGather, true>(p, ma, mb, ma, mb, my, smem, grid, stream);
        return launch<kModeTma, true>(p, ma, mb, ma, mb, my, smem, grid, stream);
    }
    if (mode == kModeHalo) return launch<kModeHalo, false>(p, ma, mb, ma16, mb16, my, smem, grid, stream);
    if (mode == kModeGather) return launch<kModeGather, false>(p, ma, mb, ma, mb, my, smem, grid, stream);
    return launch<kModeTma, false>(p, ma, mb, ma, mb, my, smem, grid, stream);
}

// Summed weights of the up conv's sub-pixel form: w [cout][9][cin] (tap
// ky*3+kx) -> ws [cout][16][cin] (tap (q*2+p)*4 + ty*2 + tx). Row ty of parity q
// collects ky in {0} | {1, 2} (q = 0) or {0, 1} | {2} (q = 1); columns alike.
// Summed in f32 in (ky, kx) order, rounded to f16 once.
__global__ void pack_subpixel_kernel(const __half* __restrict__ w, int cout, int cin, __half* __restrict__ ws) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<long long>(cout) * cin) return;
    const int o = static_cast<int>(i / cin), c = static_cast<int>(i % cin);
    float t[9];
#pragma unroll
    for (int k = 0; k < 9; ++k) t[k] = __half2float(w[(static_cast<long long>(o) * 9 + k) * cin + c]);
    // first and last source row (tap index range) of row ty for parity q
    const int lo[2][2] = {{0, 1}, {0, 2}}, hi[2][2] = {{0, 2}, {1, 2}};
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
#pragma unroll
            for (int ty = 0; ty < 2; ++ty)
#pragma unroll
                for (int tx = 0; tx < 2; ++tx) {
                    float acc = 0.f;
                    for (int ky = lo[q][ty]; ky <= hi[q][ty]; ++ky)
                        for (int kx = lo[pp][tx]; kx <= hi[pp][tx]; ++kx) acc += t[ky * 3 + kx];
                    ws[(static_cast<long long>(o) * 16 + (q * 2 + pp) * 4 + ty * 2 + tx) * cin + c] = __float2half_rn(acc);
                }
}

int pack_subpixel_run(const void* w, int cout, int cin, void* ws, cudaStream_t stream) {
    if (w == nullptr || ws == nullptr) return set_error(VAE_ERR_ARG, "pack_subpixel: w and ws must be non-NULL");
    if (cout < 1 || cout > (1 << 20) || cin < 1 || cin > 8192)
        return set_error(VAE_ERR_SHAPE, "pack_subpixel: cout=%d cin=%d", cout, cin);
    int rc = check_device();
    if (rc != VAE_OK) return rc;
    const long long n = static_cast<long long>(cout) * cin;
    pack_subpixel_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
        static_cast<const __half*>(w), cout, cin, static_cast<__half*>(ws));
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

}  // namespace vae

using namespace vae;

extern "C" {

int vae_conv3x3_nhwc(const void* x_dev, int n, int h_in, int w_in, int cin, const void* w_dev,
                     const float* bias_dev, const float* residual_dev, void* y_dev, int cout, float oscale,
                     unsigned flags, vae_stream_t stream) {
    clear_error();
    if (flags & ~static_cast<unsigned>(VAE_UPSAMPLE2X | VAE_UPSAMPLE2X_SUBPIXEL | VAE_PAD_REPLICATE | VAE_EPI_SILU |
                                       VAE_OUT_F16 | VAE_PAD_REFLECT | VAE_DOWNSAMPLE2X))
        return set_error(VAE_ERR_ARG, "vae_conv3x3_nhwc: unknown flag bits 0x%x", flags);
    if ((flags & VAE_UPSAMPLE2X_SUBPIXEL) && !(flags & VAE_UPSAMPLE2X))
        return set_error(VAE_ERR_ARG, "vae_conv3x3_nhwc: the sub-pixel form needs VAE_UPSAMPLE2X");
    ConvArgs a{};
    a.x = x_dev;
    a.n = n;
    a.h_in = h_in;
    a.w_in = w_in;
    a.cin = cin;
    a.w = w_dev;
    a.cout = cout;
    a.taps = 9;
    a.subpix = (flags & VAE_UPSAMPLE2X_SUBPIXEL) != 0;
    a.bias = bias_dev;
    a.residual = residual_dev;
    a.y = y_dev;
    a.oscale = oscale;
    a.up = (flags & VAE_UPSAMPLE2X) != 0;
    a.rep = (flags & VAE_PAD_REPLICATE) != 0;
    a.refl = (flags & VAE_PAD_REFLECT) != 0;
    a.down = (flags & VAE_DOWNSAMPLE2X) != 0;
    a.silu = (flags & VAE_EPI_SILU) != 0;
    a.out_f16 = (flags & VAE_OUT_F16) != 0;
    return conv_run(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t vae_conv3x3_gn_workspace_bytes(int n, int h_in, int w_in, int cout, int groups, unsigned flags) {
    clear_error();
    const int nch = conv_gn_chunks(h_in, w_in, (flags & VAE_UPSAMPLE2X) != 0, (flags & VAE_DOWNSAMPLE2X) != 0);
    if (n < 1 || nch < 1 || groups < 1 || cout < 1 || cout % groups != 0) return 0;
    return static_cast<size_t>(n) * nch * groups * sizeof(float4);
}

int vae_conv3x3_nhwc_gn(const void* x_dev, int n, int h_in, int w_in, int cin, const void* w_dev,
                        const float* bias_dev, const float* residual_dev, float* y_dev, int cout, float oscale,
                        unsigned flags, int groups, float eps, float* gn_stats_dev, void* workspace_dev,
                        size_t ws_bytes, vae_stream_t stream) {
    clear_error();
    if (flags & ~static_cast<unsigned>(VAE_UPSAMPLE2X | VAE_PAD_REPLICATE | VAE_EPI_SILU | VAE_PAD_REFLECT |
                                       VAE_DOWNSAMPLE2X))
        return set_error(VAE_ERR_ARG, "vae_conv3x3_nhwc_gn: unsupported flag bits 0x%x", flags);
    if (gn_stats_dev == nullptr || workspace_dev == nullptr)
        return set_error(VAE_ERR_ARG, "vae_conv3x3_nhwc_gn: gn_stats and workspace must be non-NULL");
    const size_t need = vae_conv3x3_gn_workspace_bytes(n, h_in, w_in, cout, groups, flags);
    if (need == 0) return set_error(VAE_ERR_SHAPE, "vae_conv3x3_nhwc_gn: n=%d h=%d w=%d cout=%d groups=%d", n, h_in,
                                    w_in, cout, groups);
    if (ws_bytes < need)
        return set_error(VAE_ERR_NOMEM, "vae_conv3x3_nhwc_gn: workspace %zu bytes < %zu needed", ws_bytes, need);
    ConvArgs a{};
    a.x = x_dev;
    a.n = n;
    a.h_in = h_in;
    a.w_in = w_in;
    a.cin = cin;
    a.w = w_dev;
    a.cout = cout;
    a.taps = 9;
    a.bias = bias_dev;
    a.residual = residual_dev;
    a.y = y_dev;
    a.oscale = oscale;
    a.up = (flags & VAE_UPSAMPLE2X) != 0;
    a.rep = (flags & VAE_PAD_REPLICATE) != 0;
    a.refl = (flags & VAE_PAD_REFLECT) != 0;
    a.down = (flags & VAE_DOWNSAMPLE2X) != 0;
    a.silu = (flags & VAE_EPI_SILU) != 0;
    a.gn_part = workspace_dev;
    a.gn_groups = groups;
    if (!(eps >= 0.f)) return set_error(VAE_ERR_ARG, "vae_conv3x3_nhwc_gn: eps must be >= 0");
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int rc = conv_run(a, st);
    if (rc != VAE_OK) return rc;
    return gn_stats_from_records(workspace_dev, n, conv_gn_chunks(h_in, w_in, a.up, a.down), groups, eps,
                                 gn_stats_dev, st);
}

int vae_conv3x3_nhwc_rms(const void* x_dev, int n, int h_in, int w_in, int cin, const void* w_dev,
                         const float* bias_dev, float* y_dev, int cout, float oscale, unsigned flags,
                         const float* gamma_dev, int silu, void* rms_dev, vae_stream_t stream) {
    clear_error();
    if (flags & ~static_cast<unsigned>(VAE_PAD_REPLICATE | VAE_PAD_REFLECT | VAE_DOWNSAMPLE2X))
        return set_error(VAE_ERR_ARG, "vae_conv3x3_nhwc_rms: unsupported flag bits 0x%x", flags);
    if (rms_dev == nullptr) return set_error(VAE_ERR_ARG, "vae_conv3x3_nhwc_rms: rms_dev must be non-NULL");
    ConvArgs a{};
    a.x = x_dev;
    a.n = n;
    a.h_in = h_in;
    a.w_in = w_in;
    a.cin = cin;
    a.w = w_dev;
    a.cout = cout;
    a.taps = 9;
    a.bias = bias_dev;
    a.y = y_dev;
    a.oscale = oscale;
    a.rep = (flags & VAE_PAD_REPLICATE) != 0;
    a.refl = (flags & VAE_PAD_REFLECT) != 0;
    a.down = (flags & VAE_DOWNSAMPLE2X) != 0;
    a.rms_out = rms_dev;
    a.rms_gamma = gamma_dev;
    a.rms_silu = silu != 0;
    return conv_run(a, reinterpret_cast<cudaStream_t>(stream));
}

int vae_pack_subpixel_weights(const void* w_dev, int cout, int cin, void* w_sub_dev, vae_stream_t stream) {
    clear_error();
    if (!aligned16(w_dev) || !aligned16(w_sub_dev))
        return set_error(VAE_ERR_ALIGN, "vae_pack_subpixel_weights: pointers must be 16-byte aligned");
    return pack_subpixel_run(w_dev, cout, cin, w_sub_dev, reinterpret_cast<cudaStream_t>(stream));
}

int vae_conv3d_causal_ndhwc(const void* x_dev, int n, int f_in, int h_in, int w_in, int cin, const void* w_dev,
                            const float* bias_dev, const float* residual_dev, void* y_dev, int cout, float oscale,
                            unsigned flags, vae_stream_t stream) {
    clear_error();
    if (flags & ~static_cast<unsigned>(VAE_UPSAMPLE2X | VAE_UPSAMPLE_T2X | VAE_PAD_REPLICATE | VAE_EPI_SILU |
                                       VAE_OUT_F16))
        return set_error(VAE_ERR_ARG, "vae_conv3d_causal_ndhwc: unknown flag bits 0x%x", flags);
    ConvArgs a{};
    a.x = x_dev;
    a.n = n;
    a.frames_in = f_in;
    a.t_up = (flags & VAE_UPSAMPLE_T2X) != 0;
    a.h_in = h_in;
    a.w_in = w_in;
    a.cin = cin;
    a.w = w_dev;
    a.cout = cout;
    a.taps = 27;
    a.bias = bias_dev;
    a.residual = residual_dev;
    a.y = y_dev;
    a.oscale = oscale;
    a.up = (flags & VAE_UPSAMPLE2X) != 0;
    a.rep = (flags & VAE_PAD_REPLICATE) != 0;
    a.silu = (flags & VAE_EPI_SILU) != 0;
    a.out_f16 = (flags & VAE_OUT_F16) != 0;
    return conv_run(a, reinterpret_cast<cudaStream_t>(stream));
}

int vae_conv1x1(const void* x_dev, int m, int cin, const void* w_dev, const float* bias_dev,
                const float* residual_dev, void* y_dev, int cout, float oscale, unsigned flags,
                vae_stream_t stream) {
    clear_error();
    if (flags & ~static_cast<unsigned>(VAE_EPI_SILU | VAE_OUT_F16))
        return set_error(VAE_ERR_ARG, "vae_conv1x1: only VAE_EPI_SILU and VAE_OUT_F16 apply (0x%x)", flags);
    ConvArgs a{};
    a.x = x_dev;
    a.n = 1;
    a.h_in = 1;
    a.w_in = m;
    a.cin = cin;
    a.w = w_dev;
    a.cout = cout;
    a.taps = 1;
    a.bias = bias_dev;
    a.residual = residual_dev;
    a.y = y_dev;
    a.oscale = oscale;
    a.silu = (flags & VAE_EPI_SILU) != 0;
    a.out_f16 = (flags & VAE_OUT_F16) != 0;
    return conv_run(a, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

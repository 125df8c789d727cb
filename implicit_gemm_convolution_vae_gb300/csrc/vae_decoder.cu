// The whole decoder on one GPU: handle creation (weights copied to the
// device in the kernels' layouts), workspace sizing and the decode driver
// with exact-halo horizontal bands.
//
// Follows "vae.rs" VaeDecoder::decode (FLUX-class GroupNorm family) and
// "qi21_vae.rs" decode / run_blocks / output_rows / plan_band (Qwen/Wan RMS
// family with DupUp and bands). Per stage:
//   ResNet: norm1+SiLU -> f16, conv1 (+bias) -> f32, norm2+SiLU -> f16,
//           conv2 (+bias +skip, in the epilogue) -> stream; the 1x1 shortcut
//           reads the raw stream cast to f16 with the 2^-g guard and undoes
//           it with oscale = 2^g.
//   Up conv: raw stream cast with the guard (written as f16 by the epilogue
//           of the block's last conv2 unless fusion is off), 3x3 conv with the
//           nearest-2x fold, + bias (+ the DupUp shortcut of the block input)
//           in the epilogue.
//   Output: norm_out+SiLU -> f16, conv_out (few channels) as one 1x1 GEMM with
//           its nine taps folded into the output channels, then a tap-sum
//           kernel writes NCHW f32 kept rows (+ bias).
// Banded decoding runs the head and blocks < band_from on the whole frame,
// then each band from the saved stream rows its plan needs; every kernel is
// row-local with a per-pixel result independent of tiling, so kept rows are
// bit-identical to the whole-frame decode.
//
// The driver runs twice over the same code: a dry run records the size of
// every logical buffer, a real run launches. The workspace layout therefore
// always matches what the launches use.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "vae_attn.h"
#include "vae_conv.h"
#include "vae_norm.h"

namespace vae {

struct DConv {
    __half* w = nullptr;  // [cout][k][k][cin]
    float* b = nullptr;
    int cout = 0, cin = 0, k = 0;
    bool present() const { return w != nullptr; }
};
struct DNorm {
    float* gamma = nullptr;
    float* beta = nullptr;
    int c = 0;
};
struct DRes {
    DNorm n1, n2;
    DConv c1, c2, sc;
};
struct DAttn {
    DNorm n;
    DConv q, k, v, o;
    // the folded weights (Wk^T Wq, Wo Wv f16 [c][c]; Wk^T bq, Wo bv + bo f32 [c]),
    // formed once at creation; NULL when the projections run as written
    __half* wqk = nullptr;
    __half* wov = nullptr;
    float* bqk = nullptr;
    float* bov = nullptr;
};
struct DUp {
    std::vector<DRes> res;
    DConv up;
    __half* wsub = nullptr;  // the up conv's sub-pixel weights [cout][16][cin] (VAE_DECODE_SUBPIXEL_UP)
    int in_dim = 0, out_dim = 0, ft = 1;
};

}  // namespace vae

struct vae_decoder {
    int family = 0, zc = 0, groups = 32, dupup = 0, device = 0;
    float scaling = 1.f, shift = 0.f, eps = 1e-6f;
    vae::DConv pq, conv_in, conv_out;
    // conv_out with its nine taps folded into the output channels: a 1x1 conv
    // [9 * cout rounded up to 16][cin], row t * cout + o = tap t of output o.
    vae::DConv conv_out_t;
    vae::DRes mid1, mid2;
    vae::DAttn attn;
    std::vector<vae::DUp> ups;
    vae::DNorm norm_out;
    std::vector<void*> allocs;
    // profiling of the most recent VAE_DECODE_PROFILE decode
    std::vector<cudaEvent_t> events;
    std::vector<vae_stage_record> recs;
    std::vector<int> rec_ev;  // first event index of each record (start, start + 1 = end)
};

namespace vae {

namespace {

// ───────────────────────────── conv_out tap sum ─────────────────────────────
// The second half of conv_out with its taps folded into N: z [rows][w][np]
// holds, for every pixel and tap t = 3 * ky + kx, the channel contraction of
// that tap (z[p][t * cout + o]). Output pixel (Y, X), channel o:
// bias[o] + sum over (ky, kx) of z[(Y + ky - 1, X + kx - 1)][t * cout + o], taps
// outside the rows' window or the width read zero (the conv's zero padding),
// summed in (ky, kx) order. Kept rows [keep_lo, keep_hi) of the window land at
// destination row (Y - keep_lo + dst_row0) of NCHW planes `plane` floats apart.
__global__ void __launch_bounds__(256) tapsum_nchw_kernel(const float* __restrict__ z, int rows, int w, int cout,
                                                          int np, const float* __restrict__ bias, int keep_lo,
                                                          int keep_hi, float* __restrict__ out, int dst_row0,
                                                          long long plane) {
    pdl_wait();
    const long long npx = static_cast<long long>(keep_hi - keep_lo) * w;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < npx;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int Y = keep_lo + static_cast<int>(i / w), X = static_cast<int>(i % w);
        for (int o = 0; o < cout; ++o) {
            float acc = 0.f;
            for (int ky = 0; ky < 3; ++ky) {
                const int yy = Y + ky - 1;
                if (yy < 0 || yy >= rows) continue;
                for (int kx = 0; kx < 3; ++kx) {
                    const int xx = X + kx - 1;
                    if (xx < 0 || xx >= w) continue;
                    acc = __fadd_rn(acc, __ldg(z + (static_cast<long long>(yy) * w + xx) * np + (ky * 3 + kx) * cout + o));
                }
            }
            out[o * plane + static_cast<long long>(Y - keep_lo + dst_row0) * w + X] = __fadd_rn(acc, __ldg(bias + o));
        }
    }
}

int tapsum_nchw_run(const float* z, int rows, int w, int cout, int np, const float* bias, int keep_lo, int keep_hi,
                    float* out, int dst_row0, long long plane, cudaStream_t stream) {
    const long long npx = static_cast<long long>(keep_hi - keep_lo) * w;
    if (npx <= 0) return VAE_OK;
    const int grid = static_cast<int>(std::min<long long>((npx + 255) / 256, 1LL << 20));
    VAE_CUDA_CHECK(launch_kernel(tapsum_nchw_kernel, dim3(grid), dim3(256), 0, stream, z, rows, w, cout, np, bias,
                                 keep_lo, keep_hi, out, dst_row0, plane));
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

// ───────────────────────────── handle creation ─────────────────────────────

struct Uploader {
    vae_decoder* d;
    int rc = VAE_OK;

    template <typename T>
    T* put(const void* host, size_t bytes) {
        if (rc != VAE_OK) return nullptr;
        void* p = nullptr;
        cudaError_t e = cudaMalloc(&p, std::max<size_t>(bytes, 16));
        if (e != cudaSuccess) {
            rc = set_error(VAE_ERR_NOMEM, "decoder_create: cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
            return nullptr;
        }
        d->allocs.push_back(p);
        e = cudaMemcpy(p, host, bytes, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            rc = set_error(VAE_ERR_CUDA, "decoder_create: cudaMemcpy: %s", cudaGetErrorString(e));
            return nullptr;
        }
        return static_cast<T*>(p);
    }

    DConv conv(const vae_conv_desc& c, const char* what, bool required = true) {
        DConv o;
        if (rc != VAE_OK) return o;
        if (c.w == nullptr) {
            if (required) rc = set_error(VAE_ERR_ARG, "decoder_create: %s has no weights", what);
            return o;
        }
        if ((c.k != 1 && c.k != 3) || c.cout < 1 || c.cin < 16 || c.cin % 16 != 0 || c.b == nullptr) {
            rc = set_error(VAE_ERR_SHAPE, "decoder_create: %s k=%d cout=%d cin=%d (cin %% 16 == 0 needed)", what,
                           c.k, c.cout, c.cin);
            return o;
        }
        const int kk = c.k * c.k;
        std::vector<uint16_t> packed(static_cast<size_t>(c.cout) * kk * c.cin);
        for (int o_ = 0; o_ < c.cout; ++o_)
            for (int ci = 0; ci < c.cin; ++ci)
                for (int t = 0; t < kk; ++t)
                    packed[(static_cast<size_t>(o_) * kk + t) * c.cin + ci] =
                        c.w[(static_cast<size_t>(o_) * c.cin + ci) * kk + t];
        o.w = put<__half>(packed.data(), packed.size() * 2);
        o.b = put<float>(c.b, static_cast<size_t>(c.cout) * 4);
        o.cout = c.cout;
        o.cin = c.cin;
        o.k = c.k;
        return o;
    }

    // The 3x3 conv `c` (few outputs) as a 1x1 conv whose output channel
    // t * cout + o (t = 3 * ky + kx) is tap t of output o, zero rows up to a
    // multiple of 16; no bias (the tap sum adds it).
    DConv taps_folded(const vae_conv_desc& c) {
        DConv o;
        if (rc != VAE_OK || c.w == nullptr || c.k != 3) return o;
        const int n = (9 * c.cout + 15) / 16 * 16;
        std::vector<uint16_t> packed(static_cast<size_t>(n) * c.cin, 0);
        for (int t = 0; t < 9; ++t)
            for (int o_ = 0; o_ < c.cout; ++o_)
                for (int ci = 0; ci < c.cin; ++ci)
                    packed[static_cast<size_t>(t * c.cout + o_) * c.cin + ci] =
                        c.w[(static_cast<size_t>(o_) * c.cin + ci) * 9 + t];
        o.w = put<__half>(packed.data(), packed.size() * 2);
        o.cout = n;
        o.cin = c.cin;
        o.k = 1;
        return o;
    }

    DNorm norm(const vae_norm_desc& n, int c, bool need_beta, const char* what) {
        DNorm o;
        if (rc != VAE_OK) return o;
        if (n.gamma == nullptr || (need_beta && n.beta == nullptr)) {
            rc = set_error(VAE_ERR_ARG, "decoder_create: %s norm parameters missing", what);
            return o;
        }
        o.gamma = put<float>(n.gamma, static_cast<size_t>(c) * 4);
        if (need_beta) o.beta = put<float>(n.beta, static_cast<size_t>(c) * 4);
        o.c = c;
        return o;
    }

    DRes res(const vae_resnet_desc& r, int cin, bool gn, const char* what) {
        DRes o;
        o.c1 = conv(r.conv1, what);
        o.c2 = conv(r.conv2, what);
        o.sc = conv(r.shortcut, what, false);
        if (rc != VAE_OK) return o;
        const int cout = o.c1.cout;
        if (o.c1.k != 3 || o.c2.k != 3 || o.c1.cin != cin || o.c2.cin != cout || o.c2.cout != cout) {
            rc = set_error(VAE_ERR_SHAPE, "decoder_create: %s conv shapes do not chain (cin %d)", what, cin);
            return o;
        }
        if (o.sc.present() ? (o.sc.k != 1 || o.sc.cin != cin || o.sc.cout != cout) : (cin != cout)) {
            rc = set_error(VAE_ERR_SHAPE, "decoder_create: %s needs a 1x1 shortcut %d->%d", what, cin, cout);
            return o;
        }
        o.n1 = norm(r.norm1, cin, gn, what);
        o.n2 = norm(r.norm2, cout, gn, what);
        return o;
    }
};

// ───────────────────────────── decode driver ─────────────────────────────

struct Rows {
    int lo, hi;
    int n() const { return hi - lo; }
};
Rows grow(Rows r, int k, int h) { return Rows{std::max(r.lo - k, 0), std::min(r.hi + k, h)}; }
Rows half_rows(Rows r) { return Rows{r.lo / 2, (r.hi + 1) / 2}; }

enum Buf { kS0, kS1, kS2, kB0, kB1, kB2, kH, kSC, kXN, kXN2, kZ, kATT, kGN, kZIN, kOUT, kTAP, kNBuf };

struct Band {
    Rows input;
    std::vector<Rows> feed;
    Rows keep;
};

// The first of the three stream buffers that is neither `a` nor `b`.
inline int other(int a, int b) {
    for (int i = 0; i < 3; ++i)
        if (i != a && i != b) return i;
    return -1;
}

struct Exec {
    const vae_decoder* d;
    bool dry;
    cudaStream_t st;
    uint8_t* base = nullptr;
    size_t need[kNBuf] = {};
    size_t off[kNBuf] = {};
    float guard = 256.f;
    vae_decoder* prof = nullptr;  // non-null: record events around stages
    int prof_only_w = 0;          // > 0: only the 3x3 convs with cin == cout on rows this wide
    bool fuse = false;            // VAE_DECODE_FUSE_NORM without VAE_DECODE_NO_FUSION
    // Without VAE_DECODE_NO_FUSION the last ResNet of an up block writes its conv2
    // output (the stream only the up conv still reads) straight as the guarded
    // f16 input of the up conv: (acc * oscale + bias + residual) * 2^-g rounded to
    // f16, the value and rounding of the separate cast of the f32 stream.
    bool fuse_cast = true;
    bool subpix = false;          // VAE_DECODE_SUBPIXEL_UP
    // With VAE_DECODE_FUSE_NORM a ResNet's second RMS_norm rides in the epilogue
    // of its first conv (whose f32 output only feeds that norm) when the conv's
    // CTA holds all of a pixel's channels (one N tile of <= 144): on rows of >= 128
    // pixels the staged two-pass epilogue (f16 rows only), else a register-held
    // row. Same bits as the separate norm. Off by default: on GB300 the 1024^2
    // conv with the norm in its (CTA-pair) epilogue takes 0.40 ms against
    // 0.295 + 0.136 ms for the conv and the separate norm, and whole 1024^2
    // decodes measured the same with and without it (12.75-12.95 against
    // 12.76-12.95 ms): the epilogue, which must read every chunk twice, becomes
    // the limit.
    bool fusable(int cout, int w) const {
        (void)w;
        return fuse && d->family == VAE_FAMILY_RMS && cout <= 144 && cout % 16 == 0;
    }

    // Starts a profiled stage; returns its record index (or -1).
    int begin(int kind, int launches, int h, int w, int cin, int cout, double flops, double bytes) {
        if (dry || prof == nullptr) return -1;
        if (prof_only_w > 0 && !(kind == VAE_STAGE_CONV3X3 && w == prof_only_w && cin == cout)) return -1;
        const int i = static_cast<int>(prof->recs.size());
        const size_t ev = prof->rec_ev.size() * 2;
        while (prof->events.size() < ev + 2) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) return -1;
            prof->events.push_back(e);
        }
        vae_stage_record r{};
        r.kind = kind;
        r.launches = launches;
        r.h = h;
        r.w = w;
        r.cin = cin;
        r.cout = cout;
        r.flops = flops;
        r.bytes = bytes;
        prof->recs.push_back(r);
        prof->rec_ev.push_back(static_cast<int>(ev));
        cudaEventRecord(prof->events[ev], st);
        return i;
    }
    void end(int i) {
        if (i < 0) return;
        cudaEventRecord(prof->events[prof->rec_ev[i] + 1], st);
    }

    void* buf(int id, size_t bytes) {
        if (dry) {
            need[id] = std::max(need[id], bytes);
            return reinterpret_cast<void*>(static_cast<uintptr_t>(1) << 20);
        }
        return base + off[id];
    }
    float* f32(int id, size_t count) { return static_cast<float*>(buf(id, count * 4)); }
    __half* f16(int id, size_t count) { return static_cast<__half*>(buf(id, count * 2)); }

    int conv(const ConvArgs& a) {
        if (dry) return conv_validate(a);
        const int H = a.up ? 2 * a.h_in : a.h_in, W = a.up ? 2 * a.w_in : a.w_in;
        const double flops = 2.0 * a.n * H * W * static_cast<double>(a.cout) * a.taps * a.cin;
        const int i = begin(a.taps == 9 ? VAE_STAGE_CONV3X3 : VAE_STAGE_CONV1X1, 1, H, W, a.cin, a.cout, flops, 0.0);
        const int rc = conv_run(a, st);
        end(i);
        return rc;
    }

    // norm (+SiLU) of stream `x` [hw][c] -> f16 `y`.
    int norm(const float* x, long long hw, int c, const DNorm& n, bool silu, __half* y) {
        if (d->family == VAE_FAMILY_GN) {
            GnPlan gp;
            int rc = gn_plan(1, static_cast<int>(hw), c, d->groups, &gp);
            if (rc != VAE_OK) return rc;
            void* ws = buf(kGN, gp.bytes);
            if (dry) return VAE_OK;
            const int i = begin(VAE_STAGE_NORM, 3, static_cast<int>(hw), 1, c, c, 0.0, static_cast<double>(hw) * c * 10.0);
            rc = gn_run(x, 1, static_cast<int>(hw), c, d->groups, d->eps, nullptr, n.gamma, n.beta, silu ? 1 : 0,
                        1.f, y, ws, gp.bytes, st);
            end(i);
            return rc;
        }
        if (dry) return VAE_OK;
        const int i = begin(VAE_STAGE_NORM, 1, static_cast<int>(hw), 1, c, c, 0.0, static_cast<double>(hw) * c * 6.0);
        const int rc = rms_run(x, hw, c, nullptr, n.gamma, silu ? 1 : 0, 1.f, y, st);
        end(i);
        return rc;
    }

    int cast(const float* x, size_t count, int c, float scale, __half* y) {
        if (dry) return VAE_OK;
        const int i = begin(VAE_STAGE_CAST, 1, static_cast<int>(count / c), 1, c, c, 0.0, count * 6.0);
        const int rc = cast_run(x, count, c, nullptr, scale, y, st);
        end(i);
        return rc;
    }

    static ConvArgs c3(const void* x, int h, int w, const DConv& cv, void* y) {
        ConvArgs a{};
        a.x = x;
        a.n = 1;
        a.h_in = h;
        a.w_in = w;
        a.cin = cv.cin;
        a.w = cv.w;
        a.cout = cv.cout;
        a.taps = cv.k * cv.k;
        a.bias = cv.b;
        a.y = y;
        return a;
    }

    // One ResNet on stream `x` (rows h x w, channels r.c1.cin) -> stream `y`
    // (may equal x when the channel count does not change); with `y16` the
    // result goes to y16 instead, as f16 times 2^-g (the guarded cast).
    int resnet(const DRes& r, float* x, float* y, int h, int w, __half* y16 = nullptr) {
        const long long hw = static_cast<long long>(h) * w;
        const int cin = r.c1.cin, cout = r.c1.cout;
        int rc;
        const float* skip = x;
        __half* xn = f16(kXN, hw * std::max(cin, cout));
        if (r.sc.present()) {
            float* s = f32(kSC, hw * cout);
            if ((rc = cast(x, hw * cin, cin, 1.f / guard, xn)) != VAE_OK) return rc;
            ConvArgs a = c3(xn, h, w, r.sc, s);
            a.oscale = guard;
            if ((rc = conv(a)) != VAE_OK) return rc;
            skip = s;
        }
        if ((rc = norm(x, hw, cin, r.n1, true, xn)) != VAE_OK) return rc;
        __half* xmid = f16(kXN2, hw * std::max(cin, cout));
        ConvArgs a1 = c3(xn, h, w, r.c1, nullptr);
        if (fusable(cout, w)) {
            // conv1's output feeds only norm2: the epilogue writes norm2(h), no f32 h
            a1.rms_out = xmid;
            a1.rms_gamma = r.n2.gamma;
            a1.rms_silu = true;
            if ((rc = conv(a1)) != VAE_OK) return rc;
        } else {
            float* hb = f32(kH, hw * cout);
            a1.y = hb;
            if ((rc = conv(a1)) != VAE_OK) return rc;
            if ((rc = norm(hb, hw, cout, r.n2, true, xmid)) != VAE_OK) return rc;
        }
        ConvArgs a = c3(xmid, h, w, r.c2, y);
        a.residual = skip;
        if (y16 != nullptr) {
            a.y = y16;
            a.out_f16 = true;
            a.out_scale = 1.f / guard;
        }
        return conv(a);
    }

    // Up blocks [b0, b1) on a stream held in one of three buffers
    // `bufs` (rows `cur` of the first block's level; buffer row 0 = cur.lo).
    // `feed(i)` = the rows block i feeds to its up conv (nullptr: all).
    int blocks(int b0, int b1, const int bufs[3], int* cur_buf, Rows* cur, int w0,
               const std::vector<Rows>* feed, int* ch) {
        int rc;
        for (int i = b0; i < b1; ++i) {
            const DUp& u = d->ups[i];
            int lvl = 0;
            for (int k = 0; k < i; ++k) lvl += d->ups[k].up.present() ? 1 : 0;
            const int w = w0 << lvl;
            const int h = cur->n();
            const long long hw = static_cast<long long>(h) * w;
            const bool keep_input = u.up.present() && d->dupup;
            const int in_b = *cur_buf;
            const int avoid = keep_input ? in_b : -1;
            int s_b = in_b;
            bool cast_done = false;  // the last ResNet wrote the up conv's guarded f16 input
            for (size_t r = 0; r < u.res.size(); ++r) {
                const DRes& rs = u.res[r];
                const bool fresh = rs.c1.cin != rs.c1.cout || (r == 0 && keep_input);
                const int out_b = fresh ? other(s_b, avoid) : s_b;
                float* xin = f32(bufs[s_b], hw * rs.c1.cin);
                float* xout = f32(bufs[out_b], hw * rs.c1.cout);
                __half* y16 = nullptr;
                if (fuse_cast && u.up.present() && r + 1 == u.res.size()) {
                    y16 = f16(kXN, hw * rs.c1.cout);
                    cast_done = true;
                }
                if ((rc = resnet(rs, xin, xout, h, w, y16)) != VAE_OK) return rc;
                s_b = out_b;
                *ch = rs.c1.cout;
            }
            if (!u.up.present()) {
                *cur_buf = s_b;
                continue;
            }
            const Rows f = feed ? (*feed)[i] : *cur;
            if (f.lo < cur->lo || f.hi > cur->hi || f.n() <= 0)
                return set_error(VAE_ERR_SHAPE, "decode: band feed rows [%d,%d) outside [%d,%d)", f.lo, f.hi, cur->lo,
                                 cur->hi);
            const long long skip_px = static_cast<long long>(f.lo - cur->lo) * w;
            const long long fhw = static_cast<long long>(f.n()) * w;
            const int out_b = other(s_b, avoid);
            float* xs = f32(bufs[s_b], hw * (*ch));
            __half* xn = f16(kXN, hw * (*ch));
            if (cast_done) {
                xn += dry ? 0 : skip_px * (*ch);  // the feed rows of the whole range's f16 stream
            } else if ((rc = cast(xs + (dry ? 0 : skip_px * (*ch)), fhw * (*ch), *ch, 1.f / guard, xn)) != VAE_OK) {
                return rc;
            }
            float* y = f32(bufs[out_b], fhw * 4 * u.up.cout);
            ConvArgs a = c3(xn, f.n(), w, u.up, y);
            a.up = true;
            a.oscale = guard;
            if (subpix && u.wsub != nullptr) {  // the four 2x2 convs with the summed weights
                a.w = u.wsub;
                a.subpix = true;
            }
            if (d->dupup) {
                const float* src = f32(bufs[in_b], hw * u.in_dim);
                a.dup_src = src + (dry ? 0 : skip_px * u.in_dim);
                a.dup_cin = u.in_dim;
                a.dup_factor = 4 * u.ft;
                a.dup_repeats = u.out_dim * 4 * u.ft / u.in_dim;
                a.dup_ftoff = (u.ft - 1) * 4;
            }
            if ((rc = conv(a)) != VAE_OK) return rc;
            *cur_buf = out_b;
            *cur = Rows{2 * f.lo, 2 * f.hi};
            *ch = u.up.cout;
        }
        return VAE_OK;
    }

    // norm_out + SiLU -> conv_out on stream rows `cur` (width w); kept rows
    // `keep` go to `out` [nch][hf][w].
    int output(const float* x, Rows cur, int w, int ch, Rows keep, float* out, int hf) {
        const long long hw = static_cast<long long>(cur.n()) * w;
        __half* xn = f16(kXN, hw * ch);
        int rc = norm(x, hw, ch, d->norm_out, true, xn);
        if (rc != VAE_OK) return rc;
        if (d->conv_out_t.present()) {
            // few output channels: one GEMM with the taps folded into N (9 MMAs per
            // 128 pixels instead of 81 narrow ones), then the 3x3 tap sum + bias
            const int np = d->conv_out_t.cout;
            float* z = f32(kTAP, hw * np);
            ConvArgs a = c3(xn, cur.n(), w, d->conv_out_t, z);
            if (dry) return conv_validate(a);
            const double flops = 2.0 * hw * d->conv_out.cout * 9.0 * ch;
            const int i = begin(VAE_STAGE_CONV3X3, 2, cur.n(), w, ch, d->conv_out.cout, flops, 0.0);
            rc = conv_run(a, st);
            if (rc == VAE_OK)
                rc = tapsum_nchw_run(z, cur.n(), w, d->conv_out.cout, np, d->conv_out.b, keep.lo - cur.lo,
                                     keep.hi - cur.lo, out, keep.lo, static_cast<long long>(hf) * w, st);
            end(i);
            return rc;
        }
        ConvArgs a = c3(xn, cur.n(), w, d->conv_out, out);
        a.out_nchw = true;
        a.keep_lo = keep.lo - cur.lo;
        a.keep_hi = keep.hi - cur.lo;
        a.dst_row0 = keep.lo;
        a.plane = static_cast<long long>(hf) * w;
        return conv(a);
    }
};

int levels_total(const vae_decoder* d) {
    int l = 0;
    for (const DUp& u : d->ups) l += u.up.present() ? 1 : 0;
    return l;
}

std::vector<Band> plan_bands(const vae_decoder* d, int s, int h0, int nbands) {
    const int nb = static_cast<int>(d->ups.size());
    std::vector<int> lvl(nb);
    int l = 0;
    for (int i = 0; i < nb; ++i) {
        lvl[i] = l;
        l += d->ups[i].up.present() ? 1 : 0;
    }
    const int lf = l;
    std::vector<int> hs(lf + 1);
    for (int k = 0; k <= lf; ++k) hs[k] = h0 << k;
    const int hf = hs[lf];
    const int k = (hf + nbands - 1) / nbands;
    std::vector<Band> out;
    for (int j = 0; j * k < hf; ++j) {
        Band b;
        b.keep = Rows{j * k, std::min((j + 1) * k, hf)};
        b.feed.assign(nb, Rows{0, 0});
        Rows e = grow(b.keep, d->conv_out.k / 2, hs[lf]);
        for (int i = nb - 1; i >= s; --i) {
            const DUp& u = d->ups[i];
            if (u.up.present()) {
                Rows a = half_rows(grow(e, u.up.k / 2, hs[lvl[i] + 1]));
                b.feed[i] = a;
                e = a;
            }
            int convs = 0;
            for (const DRes& r : u.res) convs += r.c1.k / 2 + r.c2.k / 2;
            e = grow(e, convs, hs[lvl[i]]);
        }
        b.input = e;
        out.push_back(b);
    }
    return out;
}

// The whole decode, dry or real. `z` NCHW f32 (device), `out` NCHW f32.
int run_decode(Exec& X, int h0, int w0, const vae_decode_opts* opts, const float* z, float* out) {
    const vae_decoder* d = X.d;
    const int nb = static_cast<int>(d->ups.size());
    const int lf = levels_total(d);
    const int hf = h0 << lf, wf = w0 << lf;
    const long long hw0 = static_cast<long long>(h0) * w0;
    int rc;
    X.guard = std::ldexp(1.0f, opts ? (opts->guard_log2 < 0 ? 8 : std::min(opts->guard_log2, 14)) : 8);
    X.fuse = opts != nullptr && (opts->flags & VAE_DECODE_FUSE_NORM) != 0 && (opts->flags & VAE_DECODE_NO_FUSION) == 0;
    X.fuse_cast = opts == nullptr || (opts->flags & VAE_DECODE_NO_FUSION) == 0;
    X.subpix = opts != nullptr && (opts->flags & VAE_DECODE_SUBPIXEL_UP) != 0;
    int nbands = 1;
    if (opts && opts->band_rows > 0) nbands = (hf + opts->band_rows - 1) / opts->band_rows;
    if (opts && opts->nbands > 1) nbands = opts->nbands;
    int s = nb;
    if (nbands > 1) {
        if (d->family != VAE_FAMILY_RMS)
            return set_error(VAE_ERR_UNSUPPORTED,
                             "decode: bands need per-pixel norms (RMS family); GroupNorm statistics are frame-global");
        s = std::min(std::max(opts->band_from, 0), nb);
        if (nbands > hf) nbands = hf;
    }
    // head: latent -> f16 NHWC -> (post_quant) -> conv_in -> mid
    const int s_bufs[3] = {kS0, kS1, kS2};
    __half* zl = X.f16(kZ, hw0 * d->zc);
    if (!X.dry) {
        const float mul = d->family == VAE_FAMILY_GN ? 1.f / d->scaling : 1.f;
        const float add = d->family == VAE_FAMILY_GN ? d->shift : 0.f;
        const int i = X.begin(VAE_STAGE_LAYOUT, 1, h0, w0, d->zc, d->zc, 0.0, hw0 * d->zc * 6.0);
        rc = latent_run(z, d->zc, hw0, mul, add, zl, X.st);
        X.end(i);
        if (rc != VAE_OK) return rc;
    }
    const void* cin_src = zl;
    if (d->pq.present()) {
        __half* xq = X.f16(kXN, hw0 * d->pq.cout);
        ConvArgs a = Exec::c3(zl, h0, w0, d->pq, xq);
        a.out_f16 = true;
        if ((rc = X.conv(a)) != VAE_OK) return rc;
        cin_src = xq;
    }
    int cur_buf = 0;
    int ch = d->conv_in.cout;
    float* x = X.f32(kS0, hw0 * ch);
    if ((rc = X.conv(Exec::c3(cin_src, h0, w0, d->conv_in, x))) != VAE_OK) return rc;
    for (int part = 0; part < 3; ++part) {
        if (part == 1) {
            size_t ab = 0;
            const int kind = d->family == VAE_FAMILY_GN ? VAE_NORM_GROUP : VAE_NORM_RMS;
            if ((rc = attn_workspace_bytes(static_cast<int>(hw0), ch, d->groups, kind, &ab)) != VAE_OK) return rc;
            void* aws = X.buf(kATT, ab);
            float* xa = X.f32(s_bufs[cur_buf], hw0 * ch);
            if (!X.dry) {
                const double m = static_cast<double>(hw0);
                // norm (+ pad rows), q' GEMM, transpose, scores, P.V, output GEMM; as written:
                // the q, k, v GEMMs instead of the q' GEMM and the transpose
                const int i = X.begin(VAE_STAGE_ATTENTION,
                                      (kind == VAE_NORM_GROUP ? 3 : 1) + (d->attn.wqk != nullptr ? 5 : 6) +
                                          (hw0 % 8 ? 1 : 0),
                                      h0, w0, ch, ch, 4.0 * m * m * ch + 4.0 * 2.0 * m * ch * ch, 0.0);
                rc = d->attn.wqk != nullptr
                         ? attn_run_folded(xa, static_cast<int>(hw0), ch, kind, d->groups, d->eps, d->attn.n.gamma,
                                           d->attn.n.beta, d->attn.wqk, d->attn.bqk, d->attn.wov, d->attn.bov, aws,
                                           ab, X.st)
                         : attn_run(xa, static_cast<int>(hw0), ch, kind, d->groups, d->eps, d->attn.n.gamma,
                                    d->attn.n.beta, d->attn.q.w, d->attn.q.b, d->attn.k.w, d->attn.k.b, d->attn.v.w,
                                    d->attn.v.b, d->attn.o.w, d->attn.o.b, aws, ab, X.st);
                X.end(i);
                if (rc != VAE_OK) return rc;
            }
            continue;
        }
        const DRes& r = part == 0 ? d->mid1 : d->mid2;
        const int out_b = r.c1.cin != r.c1.cout ? other(cur_buf, -1) : cur_buf;
        float* xin = X.f32(s_bufs[cur_buf], hw0 * r.c1.cin);
        float* xout = X.f32(s_bufs[out_b], hw0 * r.c1.cout);
        if ((rc = X.resnet(r, xin, xout, h0, w0)) != VAE_OK) return rc;
        cur_buf = out_b;
        ch = r.c1.cout;
    }
    // whole-frame up blocks [0, s)
    Rows cur{0, h0};
    if ((rc = X.blocks(0, s, s_bufs, &cur_buf, &cur, w0, nullptr, &ch)) != VAE_OK) return rc;
    int ls = 0;
    for (int i = 0; i < s; ++i) ls += d->ups[i].up.present() ? 1 : 0;
    const int ws_ = w0 << ls;
    if (s == nb) {
        const float* xs = X.f32(s_bufs[cur_buf], static_cast<size_t>(cur.n()) * ws_ * ch);
        return X.output(xs, cur, wf, ch, Rows{0, hf}, out, hf);
    }
    // bands over blocks [s, nb) from the saved level-s stream
    const float* saved = X.f32(s_bufs[cur_buf], static_cast<size_t>(cur.n()) * ws_ * ch);
    const int b_bufs[3] = {kB0, kB1, kB2};
    const std::vector<Band> bands = plan_bands(d, s, h0, nbands);
    for (const Band& bd : bands) {
        const size_t row_floats = static_cast<size_t>(ws_) * ch;
        float* xb = X.f32(kB0, bd.input.n() * row_floats);
        if (!X.dry) {
            const int i = X.begin(VAE_STAGE_COPY, 1, bd.input.n(), ws_, ch, ch, 0.0,
                                  2.0 * bd.input.n() * row_floats * sizeof(float));
            VAE_CUDA_CHECK(cudaMemcpyAsync(xb, saved + bd.input.lo * row_floats,
                                           bd.input.n() * row_floats * sizeof(float), cudaMemcpyDeviceToDevice,
                                           X.st));
            X.end(i);
        }
        int bcur = 0, bch = ch;
        Rows r = bd.input;
        if ((rc = X.blocks(s, nb, b_bufs, &bcur, &r, w0, &bd.feed, &bch)) != VAE_OK) return rc;
        const float* xo = X.f32(b_bufs[bcur], static_cast<size_t>(r.n()) * wf * bch);
        if ((rc = X.output(xo, r, wf, bch, bd.keep, out, hf)) != VAE_OK) return rc;
    }
    return VAE_OK;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

int plan_workspace(const vae_decoder* d, int h0, int w0, const vae_decode_opts* opts, Exec* X) {
    if (h0 < 1 || w0 < 1) return set_error(VAE_ERR_SHAPE, "decode: latent %dx%d", h0, w0);
    const int lf = levels_total(d);
    if ((static_cast<long long>(h0) << lf) > (1 << 20) || (static_cast<long long>(w0) << lf) > (1 << 20))
        return set_error(VAE_ERR_SHAPE, "decode: frame too large");
    X->dry = true;
    const long long nz = static_cast<long long>(d->zc) * h0 * w0;
    const long long nout = static_cast<long long>(d->conv_out.cout) * (static_cast<long long>(h0) << lf) * (w0 << lf);
    int rc = run_decode(*X, h0, w0, opts, reinterpret_cast<const float*>(1 << 20), reinterpret_cast<float*>(1 << 20));
    if (rc != VAE_OK) return rc;
    X->need[kZIN] = nz * 4;
    X->need[kOUT] = nout * 4;
    X->need[kXN2] = std::max(X->need[kXN], X->need[kXN2]);
    size_t off = 0;
    for (int i = 0; i < kNBuf; ++i) {
        X->off[i] = off;
        off = align256(off + X->need[i]);
    }
    return VAE_OK;
}

size_t total_bytes(const Exec& X) {
    size_t off = 0;
    for (int i = 0; i < kNBuf; ++i) off = align256(off + X.need[i]);
    return off;
}

}  // namespace

}  // namespace vae

using namespace vae;

extern "C" {

int vae_decoder_create(const vae_decoder_desc* desc, vae_decoder_t* out) {
    clear_error();
    if (desc == nullptr || out == nullptr) return set_error(VAE_ERR_ARG, "decoder_create: NULL argument");
    *out = nullptr;
    if (desc->family != VAE_FAMILY_GN && desc->family != VAE_FAMILY_RMS)
        return set_error(VAE_ERR_ARG, "decoder_create: family %d", desc->family);
    if (desc->n_ups < 1 || desc->ups == nullptr) return set_error(VAE_ERR_ARG, "decoder_create: no up blocks");
    int rc = check_device();
    if (rc != VAE_OK) return rc;
    const bool gn = desc->family == VAE_FAMILY_GN;
    if (gn && (desc->groups < 1 || desc->scaling == 0.f))
        return set_error(VAE_ERR_ARG, "decoder_create: GroupNorm family needs groups >= 1 and scaling != 0");
    vae_decoder* d = new (std::nothrow) vae_decoder();
    if (d == nullptr) return set_error(VAE_ERR_NOMEM, "decoder_create: host allocation");
    VAE_CUDA_CHECK(cudaGetDevice(&d->device));
    d->family = desc->family;
    d->zc = desc->latent_channels;
    d->groups = gn ? desc->groups : 32;
    d->eps = desc->eps;
    d->scaling = desc->scaling;
    d->shift = desc->shift;
    d->dupup = (!gn && desc->dupup) ? 1 : 0;
    Uploader U{d};
    d->pq = U.conv(desc->post_quant, "post_quant", false);
    d->conv_in = U.conv(desc->conv_in, "conv_in");
    const int zc_in = d->pq.present() ? d->pq.cout : d->zc;
    if (U.rc == VAE_OK && d->pq.present() && (d->pq.k != 1 || d->pq.cin != d->zc))
        U.rc = set_error(VAE_ERR_SHAPE, "decoder_create: post_quant must be 1x1 from the latent channels");
    if (U.rc == VAE_OK && (d->conv_in.k != 3 || d->conv_in.cin != zc_in))
        U.rc = set_error(VAE_ERR_SHAPE, "decoder_create: conv_in must be 3x3 from %d channels", zc_in);
    int ch = d->conv_in.cout;
    d->mid1 = U.res(desc->mid_res1, ch, gn, "mid_res1");
    if (U.rc == VAE_OK) ch = d->mid1.c1.cout;
    d->attn.n = U.norm(desc->mid_attn.norm, ch, gn, "mid_attn");
    d->attn.q = U.conv(desc->mid_attn.q, "attn.q");
    d->attn.k = U.conv(desc->mid_attn.k, "attn.k");
    d->attn.v = U.conv(desc->mid_attn.v, "attn.v");
    d->attn.o = U.conv(desc->mid_attn.o, "attn.o");
    if (U.rc == VAE_OK) {
        for (const DConv* c : {&d->attn.q, &d->attn.k, &d->attn.v, &d->attn.o})
            if (c->k != 1 || c->cin != ch || c->cout != ch)
                U.rc = set_error(VAE_ERR_SHAPE, "decoder_create: attention projections must be 1x1 %d->%d", ch, ch);
    }
    if (U.rc == VAE_OK && attn_fold_enabled()) {
        // the attention's folded weights, formed once on the device (the weights are fixed)
        const size_t cc = static_cast<size_t>(ch) * ch * 2;
        const size_t cb = (static_cast<size_t>(ch) * 4 + 255) / 256 * 256;
        void* fw = nullptr;
        void* scratch = nullptr;
        if (cudaMalloc(&fw, 2 * cc + 2 * cb) != cudaSuccess) {
            U.rc = set_error(VAE_ERR_NOMEM, "decoder_create: cudaMalloc(%zu) for the folded attention weights",
                             2 * cc + 2 * cb);
        } else {
            d->allocs.push_back(fw);
            uint8_t* f8 = static_cast<uint8_t*>(fw);
            d->attn.wqk = reinterpret_cast<__half*>(f8);
            d->attn.wov = reinterpret_cast<__half*>(f8 + cc);
            d->attn.bqk = reinterpret_cast<float*>(f8 + 2 * cc);
            d->attn.bov = reinterpret_cast<float*>(f8 + 2 * cc + cb);
            if (cudaMalloc(&scratch, 3 * cc) != cudaSuccess) {
                U.rc = set_error(VAE_ERR_NOMEM, "decoder_create: cudaMalloc(%zu) for the weight transposes", 3 * cc);
            } else {
                U.rc = attn_fold_run(ch, d->attn.q.w, d->attn.q.b, d->attn.k.w, d->attn.v.w, d->attn.v.b,
                                     d->attn.o.w, d->attn.o.b, d->attn.wqk, d->attn.wov, d->attn.bqk, d->attn.bov,
                                     static_cast<__half*>(scratch), nullptr);
                if (U.rc == VAE_OK && cudaDeviceSynchronize() != cudaSuccess)
                    U.rc = set_error(VAE_ERR_CUDA, "decoder_create: folding the attention weights failed");
                cudaFree(scratch);
            }
        }
    }
    d->mid2 = U.res(desc->mid_res2, ch, gn, "mid_res2");
    if (U.rc == VAE_OK) ch = d->mid2.c1.cout;
    for (int i = 0; i < desc->n_ups && U.rc == VAE_OK; ++i) {
        const vae_up_desc& ud = desc->ups[i];
        DUp u;
        u.in_dim = ud.in_dim;
        u.out_dim = ud.out_dim;
        u.ft = ud.ft < 1 ? 1 : ud.ft;
        if (ud.n_resnets < 0 || (ud.n_resnets > 0 && ud.resnets == nullptr)) {
            U.rc = set_error(VAE_ERR_ARG, "decoder_create: up block %d resnets", i);
            break;
        }
        const int block_in = ch;
        for (int r = 0; r < ud.n_resnets && U.rc == VAE_OK; ++r) {
            u.res.push_back(U.res(ud.resnets[r], ch, gn, "up block resnet"));
            if (U.rc == VAE_OK) ch = u.res.back().c1.cout;
        }
        u.up = U.conv(ud.up, "up conv", false);
        if (U.rc == VAE_OK && u.up.present()) {
            if (u.up.k != 3 || u.up.cin != ch)
                U.rc = set_error(VAE_ERR_SHAPE, "decoder_create: up conv of block %d must be 3x3 from %d", i, ch);
            if (d->dupup) {
                if (u.in_dim != block_in || u.out_dim != u.up.cout || (u.out_dim * 4 * u.ft) % u.in_dim != 0)
                    U.rc = set_error(VAE_ERR_SHAPE, "decoder_create: DupUp of block %d: in %d out %d ft %d", i,
                                     u.in_dim, u.out_dim, u.ft);
            }
            if (U.rc == VAE_OK) {  // the sub-pixel weights, for decodes that ask for that form
                void* ws = nullptr;
                const size_t bytes = static_cast<size_t>(u.up.cout) * 16 * u.up.cin * 2;
                if (cudaMalloc(&ws, bytes) != cudaSuccess) {
                    U.rc = set_error(VAE_ERR_NOMEM, "decoder_create: cudaMalloc(%zu) for sub-pixel weights", bytes);
                } else {
                    d->allocs.push_back(ws);
                    u.wsub = static_cast<__half*>(ws);
                    U.rc = pack_subpixel_run(u.up.w, u.up.cout, u.up.cin, ws, nullptr);
                    if (U.rc == VAE_OK && cudaDeviceSynchronize() != cudaSuccess)
                        U.rc = set_error(VAE_ERR_CUDA, "decoder_create: packing the sub-pixel weights failed");
                }
            }
            ch = u.up.cout;
        }
        d->ups.push_back(std::move(u));
    }
    d->norm_out = U.norm(desc->norm_out, ch, gn, "norm_out");
    d->conv_out = U.conv(desc->conv_out, "conv_out");
    if (U.rc == VAE_OK && (d->conv_out.k != 3 || d->conv_out.cin != ch))
        U.rc = set_error(VAE_ERR_SHAPE, "decoder_create: conv_out must be 3x3 from %d", ch);
    if (U.rc == VAE_OK && 9 * d->conv_out.cout <= 256) d->conv_out_t = U.taps_folded(desc->conv_out);
    if (U.rc == VAE_OK && gn && ch % d->groups != 0)
        U.rc = set_error(VAE_ERR_SHAPE, "decoder_create: %d channels not divisible by %d groups", ch, d->groups);
    if (U.rc != VAE_OK) {
        const int keep = U.rc;
        std::string msg = vae_last_error();
        vae_decoder_destroy(d);
        return set_error(keep, "%s", msg.c_str());
    }
    *out = d;
    return VAE_OK;
}

int vae_decoder_destroy(vae_decoder_t dec) {
    if (dec == nullptr) return VAE_OK;
    for (cudaEvent_t e : dec->events) cudaEventDestroy(e);
    for (void* p : dec->allocs) cudaFree(p);
    delete dec;
    return VAE_OK;
}

int vae_decode_profile(vae_decoder_t dec, vae_stage_record* recs, int max_recs, int* n_recs) {
    clear_error();
    if (dec == nullptr || n_recs == nullptr || (recs == nullptr && max_recs > 0))
        return set_error(VAE_ERR_ARG, "decode_profile: NULL argument");
    *n_recs = static_cast<int>(dec->recs.size());
    if (dec->recs.empty()) return VAE_OK;
    VAE_CUDA_CHECK(cudaEventSynchronize(dec->events[dec->rec_ev.back() + 1]));
    for (size_t i = 0; i < dec->recs.size(); ++i) {
        float ms = 0.f;
        VAE_CUDA_CHECK(cudaEventElapsedTime(&ms, dec->events[dec->rec_ev[i]], dec->events[dec->rec_ev[i] + 1]));
        dec->recs[i].ms = ms;
        if (static_cast<int>(i) < max_recs) recs[i] = dec->recs[i];
    }
    if (max_recs > 0) {  // a read that copies records also clears them
        dec->recs.clear();
        dec->rec_ev.clear();
    }
    return VAE_OK;
}

int vae_decode_workspace(vae_decoder_t dec, int h0, int w0, const vae_decode_opts* opts, size_t* bytes) {
    clear_error();
    if (dec == nullptr || bytes == nullptr) return set_error(VAE_ERR_ARG, "decode_workspace: NULL argument");
    Exec X{dec, true, nullptr};
    int rc = plan_workspace(dec, h0, w0, opts, &X);
    if (rc != VAE_OK) return rc;
    *bytes = total_bytes(X);
    return VAE_OK;
}

static int decode_impl(vae_decoder_t dec, const float* z, int h0, int w0, float* out, const vae_decode_opts* opts,
                       void* ws, size_t ws_bytes, cudaStream_t st, bool host) {
    if (dec == nullptr || z == nullptr || out == nullptr || ws == nullptr)
        return set_error(VAE_ERR_ARG, "decode: NULL argument");
    if (opts != nullptr &&
        (opts->flags & ~static_cast<unsigned>(VAE_DECODE_PROFILE | VAE_DECODE_NO_FUSION | VAE_DECODE_FUSE_NORM |
                                              VAE_DECODE_SUBPIXEL_UP | VAE_DECODE_PROFILE_FULLRES)) != 0)
        return set_error(VAE_ERR_ARG, "decode: unknown opts.flags 0x%x", opts->flags);
    int rc = check_device();
    if (rc != VAE_OK) return rc;
    Exec X{dec, true, st};
    rc = plan_workspace(dec, h0, w0, opts, &X);
    if (rc != VAE_OK) return rc;
    const size_t need = total_bytes(X);
    if (ws_bytes < need) return set_error(VAE_ERR_NOMEM, "decode: workspace %zu < %zu bytes", ws_bytes, need);
    if (!aligned16(ws)) return set_error(VAE_ERR_ALIGN, "decode: workspace must be 16-byte aligned");
    X.dry = false;
    X.base = static_cast<uint8_t*>(ws);
    const int lf = levels_total(dec);
    if (opts != nullptr && (opts->flags & VAE_DECODE_PROFILE)) {
        X.prof = dec;
        if (opts->flags & VAE_DECODE_PROFILE_FULLRES) X.prof_only_w = w0 << lf;
    }
    const size_t zbytes = static_cast<size_t>(dec->zc) * h0 * w0 * 4;
    const size_t obytes = static_cast<size_t>(dec->conv_out.cout) * (static_cast<size_t>(h0) << lf) * (w0 << lf) * 4;
    const float* zd = z;
    float* od = out;
    if (host) {
        float* zs = reinterpret_cast<float*>(X.base + X.off[kZIN]);
        VAE_CUDA_CHECK(cudaMemcpyAsync(zs, z, zbytes, cudaMemcpyHostToDevice, st));
        zd = zs;
        od = reinterpret_cast<float*>(X.base + X.off[kOUT]);
    }
    rc = run_decode(X, h0, w0, opts, zd, od);
    if (rc != VAE_OK) return rc;
    if (host) {
        VAE_CUDA_CHECK(cudaMemcpyAsync(out, od, obytes, cudaMemcpyDeviceToHost, st));
        return vae_sync_status(reinterpret_cast<vae_stream_t>(st));
    }
    return VAE_OK;
}

int vae_decode(vae_decoder_t dec, const float* z_dev, int h0, int w0, float* out_dev, const vae_decode_opts* opts,
               void* workspace_dev, size_t workspace_bytes, vae_stream_t stream) {
    clear_error();
    return decode_impl(dec, z_dev, h0, w0, out_dev, opts, workspace_dev, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream), false);
}

int vae_decode_host(vae_decoder_t dec, const float* z_host, int h0, int w0, float* out_host,
                    const vae_decode_opts* opts, void* workspace_dev, size_t workspace_bytes, vae_stream_t stream) {
    clear_error();
    return decode_impl(dec, z_host, h0, w0, out_host, opts, workspace_dev, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream), true);
}

struct vae_decode_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

int vae_decode_graph_create(vae_decoder_t dec, const float* z_dev, int h0, int w0, float* out_dev,
                            const vae_decode_opts* opts, void* workspace_dev, size_t workspace_bytes,
                            vae_stream_t stream, vae_decode_graph_t* graph) {
    clear_error();
    if (graph == nullptr) return set_error(VAE_ERR_ARG, "decode_graph_create: NULL graph");
    *graph = nullptr;
    if (opts != nullptr && (opts->flags & VAE_DECODE_PROFILE))
        return set_error(VAE_ERR_ARG, "decode_graph_create: a captured decode records no profile events");
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // One eager decode first: it validates everything and performs the one-time
    // per-kernel set-up, so the capture below records kernel launches only.
    int rc = decode_impl(dec, z_dev, h0, w0, out_dev, opts, workspace_dev, workspace_bytes, st, false);
    if (rc != VAE_OK) return rc;
    cudaStream_t cap;
    VAE_CUDA_CHECK(cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking));
    // the capture stream starts after the eager decode (it reads z and writes the workspace)
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(ev, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cap, ev, 0);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cap);
    if (ev != nullptr) cudaEventDestroy(ev);
    if (e != cudaSuccess) {
        cudaStreamDestroy(cap);
        return set_error(VAE_ERR_CUDA, "decode_graph_create: %s", cudaGetErrorString(e));
    }
    auto* g = new (std::nothrow) vae_decode_graph();
    if (g == nullptr) {
        cudaStreamDestroy(cap);
        return set_error(VAE_ERR_NOMEM, "decode_graph_create: host allocation failed");
    }
    e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
        rc = decode_impl(dec, z_dev, h0, w0, out_dev, opts, workspace_dev, workspace_bytes, cap, false);
        const cudaError_t e2 = cudaStreamEndCapture(cap, &g->graph);
        if (rc == VAE_OK && e2 != cudaSuccess) rc = set_error(VAE_ERR_CUDA, "decode_graph_create: %s",
                                                              cudaGetErrorString(e2));
    } else {
        rc = set_error(VAE_ERR_CUDA, "decode_graph_create: %s", cudaGetErrorString(e));
    }
    if (rc == VAE_OK) {
        e = cudaGraphInstantiate(&g->exec, g->graph, 0);
        if (e != cudaSuccess) rc = set_error(VAE_ERR_CUDA, "decode_graph_create: instantiate: %s", cudaGetErrorString(e));
    }
    cudaStreamDestroy(cap);
    if (rc != VAE_OK) {
        if (g->exec != nullptr) cudaGraphExecDestroy(g->exec);
        if (g->graph != nullptr) cudaGraphDestroy(g->graph);
        delete g;
        return rc;
    }
    *graph = g;
    return VAE_OK;
}

int vae_decode_graph_launch(vae_decode_graph_t graph, vae_stream_t stream) {
    clear_error();
    if (graph == nullptr || graph->exec == nullptr) return set_error(VAE_ERR_ARG, "decode_graph_launch: NULL graph");
    VAE_CUDA_CHECK(cudaGraphLaunch(graph->exec, reinterpret_cast<cudaStream_t>(stream)));
    return VAE_OK;
}

int vae_decode_graph_destroy(vae_decode_graph_t graph) {
    clear_error();
    if (graph == nullptr) return VAE_OK;
    if (graph->exec != nullptr) cudaGraphExecDestroy(graph->exec);
    if (graph->graph != nullptr) cudaGraphDestroy(graph->graph);
    delete graph;
    return VAE_OK;
}

}  // extern "C"

// Bandwidth-bound kernels that feed the convs: per-pixel RMS_norm,
// GroupNorm(32) (partial statistics -> Chan merge -> apply), the guarded
// f32->f16 cast of the raw stream, and the latent's NCHW f32 -> NHWC f16
// layout. All read f32 with 128-bit loads and write f16 with 64-bit stores.
#include <algorithm>
#include <mutex>

#include "vae_norm.h"
#include "vae_rms.cuh"

namespace vae {

namespace {

__device__ __forceinline__ uint2 pack4_f16(float a, float b, float c, float d) {
    __half2 lo = __floats2half2_rn(a, b);
    __half2 hi = __floats2half2_rn(c, d);
    return make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
}

// ───────────────────────────── RMS_norm ─────────────────────────────
// "qi21_vae.rs" qv_rmsn: v = x + bias; y = v * sqrt(C) / max(||v||, 1e-12) * gamma,
// optional SiLU, f16. G lanes per pixel (a power of two <= 32), each lane
// walking the pixel's float4s with stride G; a shuffle tree sums the squares.
template <int G>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x, long long m, int c,
                                                      const float* __restrict__ bias,
                                                      const float* __restrict__ gamma, int silu,
                                                      float out_scale, __half* __restrict__ y) {
    pdl_wait();
    const int c4 = c / 4;
    const int lane = threadIdx.x % G;
    const long long group = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / G;
    const long long ngroups = static_cast<long long>(gridDim.x) * blockDim.x / G;
    const float sc = sqrtf(static_cast<float>(c));
    for (long long pix = group; pix < m; pix += ngroups) {
        const float4* xr = reinterpret_cast<const float4*>(x + pix * c);
        float ss = 0.f;
        for (int i = lane; i < c4; i += G) {
            float4 v = __ldg(xr + i);
            if (bias != nullptr) {
                const float4 b = __ldg(reinterpret_cast<const float4*>(bias) + i);
                v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
            }
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off, G);
        const float inv = sc / fmaxf(sqrtf(ss), 1e-12f);
        uint2* yr = reinterpret_cast<uint2*>(y + pix * c);
        for (int i = lane; i < c4; i += G) {
            float4 v = __ldg(xr + i);
            if (bias != nullptr) {
                const float4 b = __ldg(reinterpret_cast<const float4*>(bias) + i);
                v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
            }
            const float4 g = __ldg(reinterpret_cast<const float4*>(gamma) + i);
            float o[4] = {v.x * inv * g.x, v.y * inv * g.y, v.z * inv * g.z, v.w * inv * g.w};
            if (silu) {
#pragma unroll
                for (int k = 0; k < 4; ++k) o[k] = silu_f(o[k]);
            }
            yr[i] = pack4_f16(o[0] * out_scale, o[1] * out_scale, o[2] * out_scale, o[3] * out_scale);
        }
    }
}

// The same RMS_norm with the pixel held in registers: G lanes per pixel, one
// pixel per lane group (no grid-stride loop, so every group's loads are in
// flight at once), each lane loading its <= kRmsV float4s before any use;
// x is read from memory once. Used when c/4 <= kRmsV * 32.
constexpr int kRmsV = 9;
// Threads per block of the register kernel: 128 measured 1-8 % faster than 256
// or 512 on GB300 (RMS_norm of 128^2 x 1152 ... 1024^2 x 144).
constexpr int kRmsBlock = 128;

template <int G>
__global__ void __launch_bounds__(256) rmsnorm_reg_kernel(const float* __restrict__ x, long long m, int c,
                                                          const float* __restrict__ bias,
                                                          const float* __restrict__ gamma, int silu,
                                                          float out_scale, __half* __restrict__ y) {
    pdl_wait();
    const int c4 = c / 4;
    const int lane = threadIdx.x % G;
    const long long pix = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / G;
    const bool live = pix < m;
    const float4* xr = reinterpret_cast<const float4*>(x + (live ? pix : 0) * c);
    float4 v[kRmsV];
#pragma unroll
    for (int k = 0; k < kRmsV; ++k) {
        const int i = lane + k * G;
        v[k] = (live && i < c4) ? __ldg(xr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kRmsV; ++k) {
        const int i = lane + k * G;
        if (bias != nullptr && i < c4) {
            const float4 b = __ldg(reinterpret_cast<const float4*>(bias) + i);
            v[k].x += b.x; v[k].y += b.y; v[k].z += b.z; v[k].w += b.w;
        }
        if (i < c4) ss = rms_acc4(ss, v[k].x, v[k].y, v[k].z, v[k].w);
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off, G));
    if (!live) return;
    const float inv = rms_inv(ss, c);
    uint2* yr = reinterpret_cast<uint2*>(y + pix * c);
#pragma unroll
    for (int k = 0; k < kRmsV; ++k) {
        const int i = lane + k * G;
        if (i >= c4) continue;
        const float4 g = __ldg(reinterpret_cast<const float4*>(gamma) + i);
        float o[4] = {rms_apply(v[k].x, inv, g.x), rms_apply(v[k].y, inv, g.y), rms_apply(v[k].z, inv, g.z),
                      rms_apply(v[k].w, inv, g.w)};
        if (silu) {
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = silu_f(o[e]);
        }
        yr[i] = pack4_f16(__fmul_rn(o[0], out_scale), __fmul_rn(o[1], out_scale), __fmul_rn(o[2], out_scale),
                          __fmul_rn(o[3], out_scale));
    }
}

// ───────────────────────────── GroupNorm ─────────────────────────────
// "vae.rs" GroupNorm::apply and "s2v_vae.rs" s2v_gn_part / s2v_gn_fin /
// s2v_gn_apply. Pass 1: block (chunk, image) reduces its rows; thread t
// owns float4 column t % tpr of rows t / tpr, t / tpr + rpar, ... and keeps,
// per owned channel, shifted sums (shift = the first value it read) that it
// turns into (mean, M2). Per group those are merged with Chan's formula into
// the chunk's (mean, M2). Pass 2: one block per (group, image) merges the
// chunks. Pass 3: elementwise normalise, affine, SiLU, f16.

constexpr int kGnThreads = 256;
constexpr int kGnMaxCols = 4;   // float4 columns per thread -> C <= 4 * 4 * 256 = 4096

__device__ __forceinline__ void chan_merge(float& na, float& ma, float& m2a, float nb, float mb, float m2b) {
    if (nb <= 0.f) return;
    const float n = na + nb;
    const float d = mb - ma;
    const float f = nb / n;
    ma += d * f;
    m2a += m2b + d * d * na * f;
    na = n;
}

__global__ void __launch_bounds__(kGnThreads) gn_partial_kernel(const float* __restrict__ x, int hw, int c,
                                                                int groups, int chunk_rows, int nchunks,
                                                                const float* __restrict__ bias,
                                                                float* __restrict__ part) {
    pdl_wait();
    extern __shared__ float sh[];  // [rpar][c] mean, then [rpar][c] M2
    const int chunk = blockIdx.x, img = blockIdx.y;
    const int c4 = c / 4;
    const int tpr = min(c4, kGnThreads);    // threads per row
    const int rpar = kGnThreads / tpr;           // rows processed side by side
    const int t = threadIdx.x;
    const int r0 = chunk * chunk_rows;
    const int r1 = min(r0 + chunk_rows, hw);
    float* shm = sh;
    float* shq = sh + rpar * c;
    const int rl = t / tpr;
    if (rl < rpar) {
        const int col0 = t % tpr;
        const float* xb = x + static_cast<long long>(img) * hw * c;
        for (int k = 0; k < kGnMaxCols; ++k) {
            const int col = col0 + k * tpr;
            if (col >= c4) break;
            float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
            if (bias != nullptr) b = __ldg(reinterpret_cast<const float4*>(bias) + col);
            float K[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
            int cnt = 0;
            for (int r = r0 + rl; r < r1; r += rpar) {
                float4 v = __ldg(reinterpret_cast<const float4*>(xb + static_cast<long long>(r) * c) + col);
                const float vv[4] = {v.x + b.x, v.y + b.y, v.z + b.z, v.w + b.w};
                if (cnt == 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) K[i] = vv[i];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float d = vv[i] - K[i];
                    s1[i] += d;
                    s2[i] += d * d;
                }
                ++cnt;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float n = static_cast<float>(cnt);
                const float mean = cnt > 0 ? K[i] + s1[i] / n : 0.f;
                const float m2 = cnt > 0 ? fmaxf(s2[i] - s1[i] * s1[i] / n, 0.f) : 0.f;
                shm[rl * c + col * 4 + i] = mean;
                shq[rl * c + col * 4 + i] = m2;
            }
        }
    }
    __syncthreads();
    // Per group: merge (count, mean, M2) of its channels x row lanes.
    const int cpg = c / groups;
    for (int g = t; g < groups; g += kGnThreads) {
        float na = 0.f, ma = 0.f, m2a = 0.f;
        for (int l = 0; l < rpar; ++l) {
            const int rows_l = (r1 - r0 - l + rpar - 1) / rpar;
            if (rows_l <= 0) continue;
            for (int ch = g * cpg; ch < (g + 1) * cpg; ++ch)
                chan_merge(na, ma, m2a, static_cast<float>(rows_l), shm[l * c + ch], shq[l * c + ch]);
        }
        float* out = part + ((static_cast<long long>(img) * nchunks + chunk) * groups + g) * 2;
        out[0] = ma;
        out[1] = m2a;
    }
}

__global__ void __launch_bounds__(kGnThreads) gn_finalize_kernel(const float* __restrict__ part, int hw,
                                                                 int groups, int cpg, int chunk_rows,
                                                                 int nchunks, float eps,
                                                                 float* __restrict__ stats) {
    pdl_wait();
    __shared__ float sn[kGnThreads], sm[kGnThreads], sq[kGnThreads];
    const int g = blockIdx.x, img = blockIdx.y, t = threadIdx.x;
    float na = 0.f, ma = 0.f, m2a = 0.f;
    for (int ch = t; ch < nchunks; ch += kGnThreads) {
        const int rows = min(chunk_rows, hw - ch * chunk_rows);
        const float* pp = part + ((static_cast<long long>(img) * nchunks + ch) * groups + g) * 2;
        chan_merge(na, ma, m2a, static_cast<float>(rows) * cpg, pp[0], pp[1]);
    }
    sn[t] = na;
    sm[t] = ma;
    sq[t] = m2a;
    __syncthreads();
    for (int st = kGnThreads / 2; st > 0; st >>= 1) {
        if (t < st) {
            float a = sn[t], b = sm[t], q = sq[t];
            chan_merge(a, b, q, sn[t + st], sm[t + st], sq[t + st]);
            sn[t] = a;
            sm[t] = b;
            sq[t] = q;
        }
        __syncthreads();
    }
    if (t == 0) {
        const float var = sq[0] / sn[0];
        stats[(static_cast<long long>(img) * groups + g) * 2] = sm[0];
        stats[(static_cast<long long>(img) * groups + g) * 2 + 1] = 1.0f / sqrtf(var + eps);
    }
}

// Pass 2 for statistics that a conv epilogue produced: turns each (count, K,
// S1, S2) record of shifted sums [img][nchunks][groups] into (count, mean =
// K + S1/count, M2 = S2 - S1^2/count) and merges those of one (group, image)
// in a fixed order (strided per thread, then a tree), as gn_finalize_kernel does.
__global__ void __launch_bounds__(kGnThreads) gn_finalize_records_kernel(const float4* __restrict__ rec,
                                                                         int nchunks, int groups, float eps,
                                                                         float* __restrict__ stats) {
    pdl_wait();
    __shared__ float sn[kGnThreads], sm[kGnThreads], sq[kGnThreads];
    const int g = blockIdx.x, img = blockIdx.y, t = threadIdx.x;
    float na = 0.f, ma = 0.f, m2a = 0.f;
    const float4* base = rec + static_cast<long long>(img) * nchunks * groups + g;
    constexpr int kU = 8;  // records in flight per thread
    for (int ch0 = t; ch0 < nchunks; ch0 += kU * kGnThreads) {
        float4 r[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int ch = ch0 + u * kGnThreads;
            r[u] = ch < nchunks ? __ldg(base + static_cast<long long>(ch) * groups) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (r[u].x > 0.f)
                chan_merge(na, ma, m2a, r[u].x, r[u].y + r[u].z / r[u].x, fmaxf(r[u].w - r[u].z * r[u].z / r[u].x, 0.f));
    }
    sn[t] = na;
    sm[t] = ma;
    sq[t] = m2a;
    __syncthreads();
    for (int st = kGnThreads / 2; st > 0; st >>= 1) {
        if (t < st) {
            float a = sn[t], b = sm[t], q = sq[t];
            chan_merge(a, b, q, sn[t + st], sm[t + st], sq[t + st]);
            sn[t] = a;
            sm[t] = b;
            sq[t] = q;
        }
        __syncthreads();
    }
    if (t == 0) {
        const float var = sn[0] > 0.f ? sq[0] / sn[0] : 0.f;
        stats[(static_cast<long long>(img) * groups + g) * 2] = sm[0];
        stats[(static_cast<long long>(img) * groups + g) * 2 + 1] = 1.0f / sqrtf(var + eps);
    }
}

// Pass 3: one block row of a 2-D grid per image (blockIdx.y); thread t owns
// float4 column t % tpr of rows t / tpr, t / tpr + rpar, ... so its channels,
// their gamma / beta and their groups' statistics are loaded once and the row
// loop has no index division.
__global__ void __launch_bounds__(256) gn_apply_kernel(const float* __restrict__ x, int hw, int c, int groups,
                                                       const float* __restrict__ bias,
                                                       const float* __restrict__ gamma,
                                                       const float* __restrict__ beta,
                                                       const float* __restrict__ stats, int silu,
                                                       float out_scale, __half* __restrict__ y) {
    pdl_wait();
    const int c4 = c / 4;
    const int cpg = c / groups;
    const int tpr = min(c4, 256);
    const int rpar = 256 / tpr;
    const int t = threadIdx.x;
    const int rl = t / tpr;
    if (rl >= rpar) return;
    const long long img = blockIdx.y;
    const float* xs = x + img * hw * static_cast<long long>(c);
    __half* ys = y + img * hw * static_cast<long long>(c);
    for (int col = t % tpr; col < c4; col += tpr) {
        float b4[4] = {0.f, 0.f, 0.f, 0.f}, sc[4], sh[4];
        if (bias != nullptr) {
            const float4 b = __ldg(reinterpret_cast<const float4*>(bias) + col);
            b4[0] = b.x; b4[1] = b.y; b4[2] = b.z; b4[3] = b.w;
        }
        const float4 ga = __ldg(reinterpret_cast<const float4*>(gamma) + col);
        const float4 be = __ldg(reinterpret_cast<const float4*>(beta) + col);
        const float gg[4] = {ga.x, ga.y, ga.z, ga.w};
        const float bb[4] = {be.x, be.y, be.z, be.w};
        float mu[4], rs[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float* st = stats + (img * groups + (col * 4 + k) / cpg) * 2;
            mu[k] = __ldg(st);
            rs[k] = __ldg(st + 1);
            sc[k] = gg[k];
            sh[k] = bb[k];
        }
        for (long long r = static_cast<long long>(blockIdx.x) * rpar + rl; r < hw;
             r += static_cast<long long>(gridDim.x) * rpar) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(xs + r * c) + col);
            const float vv[4] = {v.x, v.y, v.z, v.w};
            float o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float q = ((vv[k] + b4[k]) - mu[k]) * rs[k] * sc[k] + sh[k];
                if (silu) q = silu_f(q);
                o[k] = q * out_scale;
            }
            reinterpret_cast<uint2*>(ys + r * c)[col] = pack4_f16(o[0], o[1], o[2], o[3]);
        }
    }
}

// ───────────────────────────── cast / layout ─────────────────────────────

// "qi21_vae.rs" qv_cast: y = (x + bias[c]) * scale -> f16.
__global__ void __launch_bounds__(256) cast_kernel(const float* __restrict__ x, long long total4, int c,
                                                   const float* __restrict__ bias, float scale,
                                                   __half* __restrict__ y) {
    pdl_wait();
    const int c4 = c / 4;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total4;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        float4 v = __ldg(reinterpret_cast<const float4*>(x) + i);
        if (bias != nullptr) {
            const float4 b = __ldg(reinterpret_cast<const float4*>(bias) + (i % c4));
            v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
        }
        reinterpret_cast<uint2*>(y)[i] = pack4_f16(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
    }
}

// NCHW f32 [c][h*w] -> NHWC f16 [h*w][c], y = x * mul + add (the GN family's
// z / scaling + shift; mul = 1, add = 0 otherwise).
__global__ void __launch_bounds__(256) latent_nhwc_kernel(const float* __restrict__ z, int c, long long hw,
                                                          float mul, float add, __half* __restrict__ y) {
    pdl_wait();
    const long long total = hw * c;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long p = i / c;
        const int ch = static_cast<int>(i % c);
        y[i] = __float2half_rn(__ldg(z + ch * hw + p) * mul + add);
    }
}

int grid_for(long long work, int per_block) {
    const int nsm = sm_count();
    const long long want = (work + per_block - 1) / per_block;
    return static_cast<int>(std::max<long long>(1, std::min<long long>(want, static_cast<long long>(nsm) * 8)));
}

}  // namespace

// Pass 3's grid: (row blocks, images), about 8 blocks of 256 threads per SM in all.
dim3 gn_apply_grid(int n, int hw, int c) {
    const int c4 = c / 4;
    const int rpar = 256 / std::min(c4, 256);
    const long long rows_per_block_min = rpar;
    long long want = std::max(1LL, (static_cast<long long>(sm_count() > 0 ? sm_count() : 148) * 8 + n - 1) / n);
    want = std::min(want, (static_cast<long long>(hw) + rows_per_block_min - 1) / rows_per_block_min);
    want = std::min(want, 65535LL);
    return dim3(static_cast<unsigned>(want), static_cast<unsigned>(n));
}

int gn_plan(int n, int hw, int c, int groups, GnPlan* plan) {
    if (n < 1 || hw < 1 || c < 4 || c % 4 != 0 || groups < 1 || groups > 1024 || c % groups != 0 ||
        c > 4 * kGnMaxCols * kGnThreads)
        return set_error(VAE_ERR_SHAPE, "groupnorm: n=%d hw=%d c=%d groups=%d unsupported", n, hw, c, groups);
    const int c4 = c / 4;
    const int tpr = std::min(c4, kGnThreads);
    const int rpar = kGnThreads / tpr;
    // About 1216 blocks over all images, at least 8 rows per chunk: a fixed
    // plan (not device dependent), so the workspace size is too.
    long long per_img = std::max(1LL, (1216LL + n - 1) / n);
    long long max_chunks = std::max(1LL, (static_cast<long long>(hw) + 7) / 8);
    int nchunks = static_cast<int>(std::min(per_img, max_chunks));
    int chunk_rows = (hw + nchunks - 1) / nchunks;
    chunk_rows = (chunk_rows + rpar - 1) / rpar * rpar;
    nchunks = (hw + chunk_rows - 1) / chunk_rows;
    plan->nchunks = nchunks;
    plan->chunk_rows = chunk_rows;
    plan->rpar = rpar;
    plan->part_floats = static_cast<size_t>(n) * nchunks * groups * 2;
    plan->stats_floats = static_cast<size_t>(n) * groups * 2;
    plan->bytes = (plan->part_floats + plan->stats_floats) * sizeof(float) + 256;
    return VAE_OK;
}

int gn_run(const float* x, int n, int hw, int c, int groups, float eps, const float* bias, const float* gamma,
           const float* beta, int silu, float out_scale, void* y, void* ws, size_t ws_bytes,
           cudaStream_t stream) {
    GnPlan plan;
    int rc = gn_plan(n, hw, c, groups, &plan);
    if (rc != VAE_OK) return rc;
    if (x == nullptr || gamma == nullptr || beta == nullptr || y == nullptr || ws == nullptr)
        return set_error(VAE_ERR_ARG, "groupnorm: x, gamma, beta, y and workspace must be non-NULL");
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(beta) || !aligned16(y) || !aligned16(ws) ||
        (bias != nullptr && !aligned16(bias)))
        return set_error(VAE_ERR_ALIGN, "groupnorm: pointers must be 16-byte aligned");
    if (ws_bytes < plan.bytes)
        return set_error(VAE_ERR_NOMEM, "groupnorm: workspace %zu bytes < %zu needed", ws_bytes, plan.bytes);
    if (!(eps >= 0.f)) return set_error(VAE_ERR_ARG, "groupnorm: eps must be >= 0");
    rc = check_device();
    if (rc != VAE_OK) return rc;
    float* part = static_cast<float*>(ws);
    float* stats = part + plan.part_floats;
    const size_t shm = static_cast<size_t>(plan.rpar) * c * 2 * sizeof(float);
    if (shm > 48 * 1024) {
        VAE_CUDA_CHECK(cudaFuncSetAttribute(gn_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(shm)));
    }
    VAE_CUDA_CHECK(launch_kernel(gn_partial_kernel, dim3(plan.nchunks, n), dim3(kGnThreads), shm, stream, x, hw, c,
        groups, plan.chunk_rows, plan.nchunks, bias, part));
    VAE_CUDA_CHECK(cudaGetLastError());
    VAE_CUDA_CHECK(launch_kernel(gn_finalize_kernel, dim3(groups, n), dim3(kGnThreads), 0, stream, part, hw, groups,
        c / groups, plan.chunk_rows, plan.nchunks, eps, stats));
    VAE_CUDA_CHECK(cudaGetLastError());
    VAE_CUDA_CHECK(launch_kernel(gn_apply_kernel, dim3(gn_apply_grid(n, hw, c)), dim3(256), 0, stream, x, hw, c,
        groups, bias, gamma, beta, stats, silu, out_scale, static_cast<__half*>(y)));
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

int gn_stats_from_records(const void* rec, int n, int nchunks, int groups, float eps, float* stats,
                          cudaStream_t stream) {
    if (rec == nullptr || stats == nullptr) return set_error(VAE_ERR_ARG, "groupnorm: NULL records or statistics");
    if (n < 1 || nchunks < 1 || groups < 1 || groups > 65535)
        return set_error(VAE_ERR_SHAPE, "groupnorm: n=%d chunks=%d groups=%d", n, nchunks, groups);
    if (!(eps >= 0.f)) return set_error(VAE_ERR_ARG, "groupnorm: eps must be >= 0");
    VAE_CUDA_CHECK(launch_kernel(gn_finalize_records_kernel, dim3(groups, n), dim3(kGnThreads), 0, stream,
        static_cast<const float4*>(rec), nchunks, groups, eps, stats));
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

int gn_apply_run(const float* x, int n, int hw, int c, int groups, const float* stats, const float* gamma,
                 const float* beta, int silu, float out_scale, void* y, cudaStream_t stream) {
    if (x == nullptr || stats == nullptr || gamma == nullptr || beta == nullptr || y == nullptr)
        return set_error(VAE_ERR_ARG, "groupnorm_apply: x, statistics, gamma, beta and y must be non-NULL");
    if (n < 1 || hw < 1 || c < 4 || c % 4 != 0 || groups < 1 || c % groups != 0)
        return set_error(VAE_ERR_SHAPE, "groupnorm_apply: n=%d hw=%d c=%d groups=%d unsupported", n, hw, c, groups);
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(beta) || !aligned16(y))
        return set_error(VAE_ERR_ALIGN, "groupnorm_apply: pointers must be 16-byte aligned");
    int rc = check_device();
    if (rc != VAE_OK) return rc;
    VAE_CUDA_CHECK(launch_kernel(gn_apply_kernel, dim3(gn_apply_grid(n, hw, c)), dim3(256), 0, stream, x, hw, c,
        groups, nullptr, gamma, beta, stats, silu, out_scale, static_cast<__half*>(y)));
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

int rms_run(const float* x, long long m, int c, const float* bias, const float* gamma, int silu,
            float out_scale, void* y, cudaStream_t stream) {
    if (x == nullptr || gamma == nullptr || y == nullptr)
        return set_error(VAE_ERR_ARG, "rmsnorm: x, gamma and y must be non-NULL");
    if (m < 1 || c < 4 || c % 4 != 0 || c > 16384)
        return set_error(VAE_ERR_SHAPE, "rmsnorm: m=%lld c=%d unsupported", m, c);
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(y) || (bias != nullptr && !aligned16(bias)))
        return set_error(VAE_ERR_ALIGN, "rmsnorm: pointers must be 16-byte aligned");
    int rc = check_device();
    if (rc != VAE_OK) return rc;
    const int c4 = c / 4;
    __half* yh = static_cast<__half*>(y);
    if (c4 <= kRmsV * 32) {
        const int G = rms_lanes(c);
        const long long blocks = (m * G + kRmsBlock - 1) / kRmsBlock;
        if (blocks > 0x7fffffffLL) return set_error(VAE_ERR_SHAPE, "rmsnorm: m=%lld too large", m);
        const int grid = static_cast<int>(blocks);
        if (G == 4)
            VAE_CUDA_CHECK(launch_kernel(rmsnorm_reg_kernel<4>, dim3(grid), dim3(kRmsBlock), 0, stream, x, m, c, bias,
                gamma, silu, out_scale, yh));
        else if (G == 8)
            VAE_CUDA_CHECK(launch_kernel(rmsnorm_reg_kernel<8>, dim3(grid), dim3(kRmsBlock), 0, stream, x, m, c, bias,
                gamma, silu, out_scale, yh));
        else if (G == 16)
            VAE_CUDA_CHECK(launch_kernel(rmsnorm_reg_kernel<16>, dim3(grid), dim3(kRmsBlock), 0, stream, x, m, c, bias,
                gamma, silu, out_scale, yh));
        else
            VAE_CUDA_CHECK(launch_kernel(rmsnorm_reg_kernel<32>, dim3(grid), dim3(kRmsBlock), 0, stream, x, m, c, bias,
                gamma, silu, out_scale, yh));
    } else if (c4 >= 128) {
        VAE_CUDA_CHECK(launch_kernel(rmsnorm_kernel<32>, dim3(grid_for(m * 32, 256)), dim3(256), 0, stream, x, m, c,
            bias, gamma, silu, out_scale, yh));
    } else if (c4 >= 32) {
        VAE_CUDA_CHECK(launch_kernel(rmsnorm_kernel<16>, dim3(grid_for(m * 16, 256)), dim3(256), 0, stream, x, m, c,
            bias, gamma, silu, out_scale, yh));
    } else {
        VAE_CUDA_CHECK(launch_kernel(rmsnorm_kernel<8>, dim3(grid_for(m * 8, 256)), dim3(256), 0, stream, x, m, c,
            bias, gamma, silu, out_scale, yh));
    }
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

int cast_run(const float* x, size_t count, int c, const float* bias, float scale, void* y, cudaStream_t stream) {
    if (x == nullptr || y == nullptr) return set_error(VAE_ERR_ARG, "cast: x and y must be non-NULL");
    if (c < 4 || c % 4 != 0 || count % static_cast<size_t>(c) != 0)
        return set_error(VAE_ERR_SHAPE, "cast: count %zu, c %d unsupported", count, c);
    if (!aligned16(x) || !aligned16(y) || (bias != nullptr && !aligned16(bias)))
        return set_error(VAE_ERR_ALIGN, "cast: pointers must be 16-byte aligned");
    int rc = check_device();
    if (rc != VAE_OK) return rc;
    if (count == 0) return VAE_OK;
    const long long total4 = static_cast<long long>(count / 4);
    VAE_CUDA_CHECK(launch_kernel(cast_kernel, dim3(grid_for(total4, 256)), dim3(256), 0, stream, x, total4, c, bias,
        scale, static_cast<__half*>(y)));
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

int latent_run(const float* z, int c, long long hw, float mul, float add, void* y, cudaStream_t stream) {
    VAE_CUDA_CHECK(launch_kernel(latent_nhwc_kernel, dim3(grid_for(hw * c, 256)), dim3(256), 0, stream, z, c, hw, mul,
        add, static_cast<__half*>(y)));
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

// Scratch of vae_groupnorm_silu_static: a fixed array in device memory that
// every GPU loading this library holds until the process exits. Host code
// must not pass the symbol itself to a kernel (on the host it only names a
// stand-in); gn_static_scratch() looks its device address up once per device
// and context (again after a cudaDeviceReset).
constexpr size_t kGnStaticFloats = 131072;  // 512 KB
static __device__ __align__(256) float g_gn_static_scratch[kGnStaticFloats];

static float* gn_static_scratch() {
    static std::mutex mu;
    static float* ptr[64] = {nullptr};
    static CtxOnce once;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error(VAE_ERR_CUDA, "groupnorm_static: cudaGetDevice: %s", cudaGetErrorString(e));
        return nullptr;
    }
    if (dev < 0 || dev >= 64) {
        set_error(VAE_ERR_UNSUPPORTED, "groupnorm_static: device index %d", dev);
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (ptr[dev] == nullptr || !once.done(dev)) {  // first call, or a new context since (cudaDeviceReset)
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_gn_static_scratch);
        if (e != cudaSuccess) {
            set_error(VAE_ERR_CUDA, "groupnorm_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            return nullptr;
        }
        ptr[dev] = static_cast<float*>(p);
        once.mark(dev);
    }
    return ptr[dev];
}

}  // namespace vae

using namespace vae;

extern "C" {

int vae_groupnorm_silu_static(const float* x_dev, int n, int hw, int c, int groups, float eps,
                              const float* bias_in_dev, const float* gamma_dev, const float* beta_dev, int silu,
                              float out_scale, void* y_dev, vae_stream_t stream) {
    clear_error();
    GnPlan plan;
    int rc = gn_plan(n, hw, c, groups, &plan);
    if (rc != VAE_OK) return rc;
    if (plan.bytes > kGnStaticFloats * sizeof(float))
        return set_error(VAE_ERR_NOMEM,
                         "groupnorm_static: n=%d hw=%d groups=%d needs %zu bytes of scratch, more than the fixed "
                         "%zu bytes; use vae_groupnorm_silu with a workspace",
                         n, hw, groups, plan.bytes, kGnStaticFloats * sizeof(float));
    rc = check_device();
    if (rc != VAE_OK) return rc;
    float* ws = gn_static_scratch();
    if (ws == nullptr) return VAE_ERR_CUDA;
    return gn_run(x_dev, n, hw, c, groups, eps, bias_in_dev, gamma_dev, beta_dev, silu, out_scale, y_dev, ws,
                  kGnStaticFloats * sizeof(float), reinterpret_cast<cudaStream_t>(stream));
}

int vae_rmsnorm_silu(const float* x_dev, int m, int c, const float* bias_in_dev, const float* gamma_dev, int silu,
                     float out_scale, void* y_dev, vae_stream_t stream) {
    clear_error();
    return rms_run(x_dev, m, c, bias_in_dev, gamma_dev, silu, out_scale, y_dev,
                   reinterpret_cast<cudaStream_t>(stream));
}

int vae_groupnorm_apply(const float* x_dev, int n, int hw, int c, int groups, const float* gn_stats_dev,
                        const float* gamma_dev, const float* beta_dev, int silu, float out_scale, void* y_dev,
                        vae_stream_t stream) {
    clear_error();
    return gn_apply_run(x_dev, n, hw, c, groups, gn_stats_dev, gamma_dev, beta_dev, silu, out_scale, y_dev,
                        reinterpret_cast<cudaStream_t>(stream));
}

size_t vae_groupnorm_workspace_bytes(int n, int hw, int c, int groups) {
    GnPlan plan;
    if (gn_plan(n, hw, c, groups, &plan) != VAE_OK) return 0;
    return plan.bytes;
}

int vae_groupnorm_silu(const float* x_dev, int n, int hw, int c, int groups, float eps, const float* bias_in_dev,
                       const float* gamma_dev, const float* beta_dev, int silu, float out_scale, void* y_dev,
                       void* workspace_dev, size_t workspace_bytes, vae_stream_t stream) {
    clear_error();
    return gn_run(x_dev, n, hw, c, groups, eps, bias_in_dev, gamma_dev, beta_dev, silu, out_scale, y_dev,
                  workspace_dev, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int vae_cast_f16(const float* x_dev, size_t count, int c, const float* bias_dev, float scale, void* y_dev,
                 vae_stream_t stream) {
    clear_error();
    return cast_run(x_dev, count, c, bias_dev, scale, y_dev, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

// Mid-block single-head spatial self-attention ("vae.rs" AttnBlock::apply /
// finish; "qi21_vae.rs" attention): norm -> q, k, v^T projections (the
// implicit-GEMM kernel with one tap) -> one fused tcgen05 kernel computing
// o = softmax(q k^T / sqrt(c)) v + b_v -> output projection added onto the
// stream by the conv epilogue's residual path.
//
// The fused kernel (one CTA per (128-query tile, value-channel chunk)):
//  - S = Q K_j^T for key block j (128 keys) accumulates in TMEM columns
//    [384, 512) from 64-channel chunks of Q and K streamed by TMA;
//  - four softmax warps (one query row per thread) read S with tcgen05.ld,
//    mask keys >= m, keep a running max m and sum l (online softmax; O is
//    rescaled in TMEM only when the max grows by more than 2^8, so the
//    unnormalised P = 2^(s - m) stays <= 256 in f16), and write P (f16) to
//    shared memory in the K-major 128B-swizzled layout;
//  - O[:, chunk] += P V_j^T[chunk] accumulates in TMEM columns [0, dv) (dv <=
//    384, so c = 1152 takes three chunks and recomputes S per chunk);
//  - the MMA issue order QK(j+1) before PV(j) and one S buffer let the
//    softmax of block j overlap the tensor-core work of blocks j+1 (QK) and
//    j-1 (PV); one P buffer is enough, because PV(j-1) finishes while the
//    softmax of block j is still taking its row maxima, and the 32 KB saved
//    buys a third 64 KB slot of the Q/K/V ring: a key block streams about
//    twice the ring's capacity of Q and K, so the bytes in flight, not the
//    tensor cores, set the pace;
//  - the epilogue writes O / l + b_v as f16 (the v bias is added after P.V,
//    exact because the rows of the softmax sum to one).
// No score matrix is ever written to memory. Every wait is bounded.
#include <algorithm>
#include <cmath>

#include "vae_attn.h"
#include "vae_conv.h"
#include "vae_norm.h"

namespace vae {

namespace {

constexpr int kThreads = 192;
constexpr int kStageBytes = 64 * 1024;  // QK: two (Q, K) 64-channel chunk pairs; PV: one 64-key V^T half
constexpr int kStages = 3;
constexpr int kPBytes = 32 * 1024;  // 128 x 128 f16: two 64-key SW128 atoms
static_assert(1024 + kStages * kStageBytes + kPBytes + 256 <= 232448, "attention shared memory over 227 KB");
constexpr uint32_t kSCol = 384;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxDv = 384;

struct AttnParams {
    int m, c, dv, ndv, nkb, nchunk_c;
    int vbox_rows, vboxes;
    float scale_log2;
    const float* bv;
    __half* out;
    DevStatus* status;
    unsigned long long timeout_ns;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

struct ASmem {
    uint8_t* ring;
    uint8_t* p;
    uint64_t *full, *empty, *s_full, *s_free, *p_full, *pv_done, *drain;
    uint32_t* tmem_slot;
    int* abort_flag;
};

__device__ __forceinline__ ASmem carve_attn(uint8_t* raw) {
    ASmem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.ring = base;
    s.p = base + kStages * kStageBytes;
    uint64_t* b = reinterpret_cast<uint64_t*>(s.p + kPBytes);
    s.full = b;
    s.empty = b + kStages;
    s.s_full = b + 2 * kStages;
    s.s_free = s.s_full + 1;
    s.p_full = s.s_free + 1;   // [2]
    s.pv_done = s.p_full + 2;  // [2]
    s.drain = s.pv_done + 2;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
    return s;
}

__device__ __forceinline__ bool wait_(uint64_t* bar, uint32_t parity, const ASmem& s, const AttnParams& p) {
    return mbar_wait(smem_u32(bar), parity, s.abort_flag, p.timeout_ns, p.status, kWhereAttn);
}

// The same wait taken by a whole warp, with a warp-uniform result.
__device__ __forceinline__ bool wwait_(uint64_t* bar, uint32_t parity, const ASmem& s, const AttnParams& p) {
    return warp_all(wait_(bar, parity, s, p));
}

__device__ void attn_producer(const AttnParams& p, const ASmem& s, const CUtensorMap* mq, const CUtensorMap* mk,
                              const CUtensorMap* mv, int q0, int d0) {
    const uint64_t pol = policy_evict_normal();
    int stage = 0;
    uint32_t phase = 0, armed = 0, arm_par = 0;
    bool ok = true;
    auto next = [&]() {
        if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
        }
    };
    // Chunks cc and cc+1 (when it exists) of Q and of K block j in one stage.
    auto load_qk = [&](int j, int cc) {
        if (!ok) return;
        if (!wait_(&s.empty[stage], phase ^ 1u, s, p)) {
            ok = false;
            return;
        }
        const int nck = min(2, p.nchunk_c - cc);
        const uint32_t fb = smem_u32(&s.full[stage]);
        mbar_arrive_expect_tx(fb, 32768u * static_cast<uint32_t>(nck));
        armed |= 1u << stage;
        arm_par = (arm_par & ~(1u << stage)) | (phase << stage);
        uint8_t* st = s.ring + stage * kStageBytes;
        for (int h = 0; h < nck; ++h) {
            tma_load_2d(smem_u32(st + h * 32768), mq, fb, (cc + h) * 64, q0, pol);
            tma_load_2d(smem_u32(st + h * 32768 + 16384), mk, fb, (cc + h) * 64, j * 128, pol);
        }
        next();
    };
    auto load_v = [&](int j, int half) {
        if (!ok) return;
        if (!wait_(&s.empty[stage], phase ^ 1u, s, p)) {
            ok = false;
            return;
        }
        const uint32_t fb = smem_u32(&s.full[stage]);
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(p.vboxes * p.vbox_rows * 128));
        armed |= 1u << stage;
        arm_par = (arm_par & ~(1u << stage)) | (phase << stage);
        uint8_t* st = s.ring + stage * kStageBytes;
        for (int b = 0; b < p.vboxes; ++b)
            tma_load_2d(smem_u32(st + b * p.vbox_rows * 128), mv, fb, j * 128 + half * 64, d0 + b * p.vbox_rows,
                        pol);
        next();
    };
    for (int cc = 0; cc < p.nchunk_c; cc += 2) load_qk(0, cc);
    for (int j = 0; j < p.nkb && ok; ++j) {
        if (j + 1 < p.nkb)
            for (int cc = 0; cc < p.nchunk_c; cc += 2) load_qk(j + 1, cc);
        load_v(j, 0);
        load_v(j, 1);
    }
    int never = 0;
    for (int st = 0; st < kStages; ++st)
        if (armed & (1u << st))
            (void)mbar_wait(smem_u32(&s.full[st]), (arm_par >> st) & 1u, &never, p.timeout_ns, p.status, kWhereDrain);
}

__device__ void attn_mma(const AttnParams& p, const ASmem& s, uint32_t tmem) {
    const uint32_t id_s = idesc_f16_f32(128, 128);
    const int nsplit = p.dv > 256 ? 2 : 1;
    const int ns = p.dv / nsplit;
    const uint32_t id_o = idesc_f16_f32(128, ns);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    auto next = [&]() {
        if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
        }
    };
    auto issue_qk = [&]() {
        for (int cc = 0; cc < p.nchunk_c && ok; cc += 2) {
            if (!wait_(&s.full[stage], phase, s, p)) {
                ok = false;
                return;
            }
            tc_fence_after();
            uint8_t* st = s.ring + stage * kStageBytes;
            const int nck = min(2, p.nchunk_c - cc);
            for (int h = 0; h < nck; ++h) {
                const uint64_t ad = sw128_kmajor_desc(smem_u32(st + h * 32768));
                const uint64_t bd = sw128_kmajor_desc(smem_u32(st + h * 32768 + 16384));
                for (int k = 0; k < 4; ++k)
                    umma_f16(tmem + kSCol, ad + 2 * k, bd + 2 * k, id_s, (cc | h | k) != 0 ? 1u : 0u);
            }
            umma_commit(smem_u32(&s.empty[stage]));
            next();
        }
        if (ok) umma_commit(smem_u32(s.s_full));
    };
    auto issue_pv = [&](int j) {
        uint8_t* pb = s.p;
        for (int half = 0; half < 2 && ok; ++half) {
            if (!wait_(&s.full[stage], phase, s, p)) {
                ok = false;
                return;
            }
            tc_fence_after();
            uint8_t* st = s.ring + stage * kStageBytes;
            const uint64_t ad = sw128_kmajor_desc(smem_u32(pb + half * 16384));
            for (int k = 0; k < 4; ++k)
                for (int sp = 0; sp < nsplit; ++sp) {
                    const uint64_t bd = sw128_kmajor_desc(smem_u32(st + sp * ns * 128));
                    umma_f16(tmem + static_cast<uint32_t>(sp * ns), ad + 2 * k, bd + 2 * k, id_o,
                             (j | half | k) != 0 ? 1u : 0u);
                }
            umma_commit(smem_u32(&s.empty[stage]));
            next();
        }
        if (ok) umma_commit(smem_u32(&s.pv_done[j & 1]));
    };
    issue_qk();
    for (int j = 0; j < p.nkb && ok; ++j) {
        if (j + 1 < p.nkb) {
            if (!wait_(s.s_free, static_cast<uint32_t>(j & 1), s, p)) break;
            tc_fence_after();
            issue_qk();
        }
        if (!ok) break;
        if (!wait_(&s.p_full[j & 1], static_cast<uint32_t>((j >> 1) & 1), s, p)) break;
        tc_fence_after();
        issue_pv(j);
    }
    umma_commit(smem_u32(s.drain));
    int never = 0;
    (void)mbar_wait(smem_u32(s.drain), 0u, &never, p.timeout_ns, p.status, kWhereDrain);
}

__device__ void attn_softmax(const AttnParams& p, const ASmem& s, uint32_t tmem, int warp, int lane, int q0,
                             int d0) {
    const int r = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + kSCol;
    const uint32_t tO = tmem + lane_off;
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < p.nkb; ++j) {
        if (!wwait_(s.s_full, static_cast<uint32_t>(j & 1), s, p)) {
            ok = false;
            break;
        }
        tc_fence_after();
        float sv[128];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            uint32_t rr[16];
            __syncwarp();
            tmem_ld16(tS + g * 16, rr);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) sv[g * 16 + i] = __uint_as_float(rr[i]);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(s.s_free));
        const int nvalid = min(128, p.m - j * 128);
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 128; ++i) {
            sv[i] = i < nvalid ? sv[i] * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, sv[i]);
        }
        float alpha = 1.f;
        bool resc = false;
        if (j == 0) {
            m_run = mx;
        } else if (mx > m_run + 8.f) {
            alpha = exp2f(m_run - mx);
            m_run = mx;
            resc = true;
        }
        // P and the O accumulator are free once PV(j-1) is done.
        if (j >= 1 && !wwait_(&s.pv_done[(j - 1) & 1], static_cast<uint32_t>(((j - 1) >> 1) & 1), s, p)) {
            ok = false;
            break;
        }
        if (__any_sync(0xffffffffu, resc)) {
            tc_fence_after();
            for (int col = 0; col < p.dv; col += 16) {
                uint32_t rr[16];
                __syncwarp();
                tmem_ld16(tO + col, rr);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
                tmem_st16(tO + col, rr);
            }
            tmem_st_wait();
        }
        l *= alpha;
        float sum = 0.f;
        uint8_t* pb = s.p;
#pragma unroll
        for (int g = 0; g < 16; ++g) {
            uint32_t h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float a = exp2f(sv[g * 8 + 2 * i] - m_run);
                const float b = exp2f(sv[g * 8 + 2 * i + 1] - m_run);
                sum += a + b;
                __half2 t = __floats2half2_rn(a, b);
                h[i] = *reinterpret_cast<uint32_t*>(&t);
            }
            *reinterpret_cast<uint4*>(pb + (g >> 3) * 16384 + sw128_off(static_cast<uint32_t>(r), g & 7)) =
                make_uint4(h[0], h[1], h[2], h[3]);
        }
        l += sum;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&s.p_full[j & 1]));
    }
    if (!ok) return;
    const int jl = p.nkb - 1;
    if (!wwait_(&s.pv_done[jl & 1], static_cast<uint32_t>((jl >> 1) & 1), s, p)) return;
    tc_fence_after();
    const float inv = 1.f / l;
    const int q = q0 + r;
    for (int col = 0; col < p.dv; col += 16) {
        uint32_t rr[16];
        __syncwarp();
        tmem_ld16(tO + col, rr);
        tmem_ld_wait();
        const int d = d0 + col;
        if (q >= p.m || d >= p.c) continue;
        __half* dst = p.out + static_cast<long long>(q) * p.c + d;
        if (d + 16 <= p.c) {
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                __half2 t = __floats2half2_rn(__uint_as_float(rr[2 * i]) * inv + __ldg(p.bv + d + 2 * i),
                                              __uint_as_float(rr[2 * i + 1]) * inv + __ldg(p.bv + d + 2 * i + 1));
                h[i] = *reinterpret_cast<uint32_t*>(&t);
            }
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(h[0], h[1], h[2], h[3]);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(h[4], h[5], h[6], h[7]);
        } else {
            for (int i = 0; i < 16 && d + i < p.c; ++i)
                dst[i] = __float2half_rn(__uint_as_float(rr[i]) * inv + __ldg(p.bv + d + i));
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mv, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    const ASmem s = carve_attn(smem_raw);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int q0 = (blockIdx.x / p.ndv) * 128;
    const int d0 = (blockIdx.x % p.ndv) * p.dv;
    if (threadIdx.x == 0) {
        *s.abort_flag = 0;
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&s.full[i]), 1u);
            mbar_init(smem_u32(&s.empty[i]), 1u);
        }
        mbar_init(smem_u32(s.s_full), 1u);
        mbar_init(smem_u32(s.s_free), 128u);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s.p_full[i]), 128u);
            mbar_init(smem_u32(&s.pv_done[i]), 1u);
        }
        mbar_init(smem_u32(s.drain), 1u);
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(s.tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s.tmem_slot;
    if (warp < 4) {
        attn_softmax(p, s, tmem, warp, lane, q0, d0);
    } else if (warp == 4) {
        if (lane == 0) attn_producer(p, s, &mq, &mk, &mv, q0, d0);
    } else {
        if (lane == 0) attn_mma(p, s, tmem);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

struct AttnLayout {
    int m_pad, ndv, dv;
    size_t xn, q, k, vt, o, gn, total;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

int attn_layout(int m, int c, int groups, int norm_kind, AttnLayout* L) {
    if (m < 1 || c < 16 || c % 16 != 0 || c > 2048)
        return set_error(VAE_ERR_SHAPE, "mid_attention: m=%d c=%d (need c %% 16 == 0, 16 <= c <= 2048)", m, c);
    L->m_pad = (m + 7) / 8 * 8;
    const int nchunk = (c + kMaxDv - 1) / kMaxDv;
    L->dv = ((c + nchunk - 1) / nchunk + 31) / 32 * 32;
    L->ndv = (c + L->dv - 1) / L->dv;
    size_t off = 0;
    L->xn = off;
    off = align256(off + static_cast<size_t>(L->m_pad) * c * 2);
    L->q = off;
    off = align256(off + static_cast<size_t>(m) * c * 2);
    L->k = off;
    off = align256(off + static_cast<size_t>(m) * c * 2);
    L->vt = off;
    off = align256(off + static_cast<size_t>(c) * L->m_pad * 2);
    L->o = off;
    off = align256(off + static_cast<size_t>(m) * c * 2);
    L->gn = off;
    if (norm_kind == VAE_NORM_GROUP) {
        GnPlan gp;
        int rc = gn_plan(1, m, c, groups, &gp);
        if (rc != VAE_OK) return rc;
        off = align256(off + gp.bytes);
    }
    L->total = off;
    return VAE_OK;
}

}  // namespace

int attn_core_run(const __half* q, const __half* k, const __half* vt, int m, int m_pad, int c, const float* bv,
                  __half* out, cudaStream_t stream) {
    int rc = check_device();
    if (rc != VAE_OK) return rc;
    DevStatus* st = device_status_ptr();
    if (st == nullptr) return VAE_ERR_CUDA;
    AttnParams p{};
    p.m = m;
    p.c = c;
    const int nchunk = (c + kMaxDv - 1) / kMaxDv;
    p.dv = ((c + nchunk - 1) / nchunk + 31) / 32 * 32;
    p.ndv = (c + p.dv - 1) / p.dv;
    p.nkb = (m + 127) / 128;
    p.nchunk_c = (c + 63) / 64;  // a partial last chunk reads TMA zero fill
    p.vboxes = p.dv > 256 ? 2 : 1;
    p.vbox_rows = p.dv / p.vboxes;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c)));
    p.bv = bv;
    p.out = out;
    p.status = st;
    p.timeout_ns = wait_timeout_ns();
    CUtensorMap mq{}, mk{}, mv{};
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(c), static_cast<uint64_t>(m)};
        const uint64_t strides[1] = {static_cast<uint64_t>(c) * 2};
        const uint32_t box[2] = {64u, 128u};
        rc = encode_tiled(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != VAE_OK) return rc;
        rc = encode_tiled(&mk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, k, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != VAE_OK) return rc;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(m_pad), static_cast<uint64_t>(c)};
        const uint64_t strides[1] = {static_cast<uint64_t>(m_pad) * 2};
        const uint32_t box[2] = {64u, static_cast<uint32_t>(p.vbox_rows)};
        rc = encode_tiled(&mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, vt, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != VAE_OK) return rc;
    }
    const size_t smem = 1024 + kStages * kStageBytes + kPBytes + 256;
    static bool attr_set[64] = {false};
    int dev = 0;
    VAE_CUDA_CHECK(cudaGetDevice(&dev));
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        VAE_CUDA_CHECK(cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(smem)));
        attr_set[dev] = true;
    }
    const long long grid = static_cast<long long>((m + 127) / 128) * p.ndv;
    attn_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(mq, mk, mv, p);
    VAE_CUDA_CHECK(cudaGetLastError());
    return VAE_OK;
}

int attn_workspace_bytes(int m, int c, int groups, int norm_kind, size_t* bytes) {
    AttnLayout L;
    int rc = attn_layout(m, c, groups, norm_kind, &L);
    if (rc != VAE_OK) return rc;
    *bytes = L.total;
    return VAE_OK;
}

int attn_run(float* x, int m, int c, int norm_kind, int groups, float eps, const float* gamma, const float* beta,
             const void* wq, const float* bq, const void* wk, const float* bk, const void* wv, const float* bv,
             const void* wo, const float* bo, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (x == nullptr || gamma == nullptr || wq == nullptr || wk == nullptr || wv == nullptr || wo == nullptr ||
        bq == nullptr || bk == nullptr || bv == nullptr || bo == nullptr || ws == nullptr)
        return set_error(VAE_ERR_ARG, "mid_attention: a required pointer is NULL");
    if (norm_kind != VAE_NORM_GROUP && norm_kind != VAE_NORM_RMS)
        return set_error(VAE_ERR_ARG, "mid_attention: norm_kind %d", norm_kind);
    if (norm_kind == VAE_NORM_GROUP && beta == nullptr)
        return set_error(VAE_ERR_ARG, "mid_attention: GroupNorm needs beta");
    AttnLayout L;
    int rc = attn_layout(m, c, groups, norm_kind, &L);
    if (rc != VAE_OK) return rc;
    if (ws_bytes < L.total)
        return set_error(VAE_ERR_NOMEM, "mid_attention: workspace %zu < %zu bytes", ws_bytes, L.total);
    if (!aligned16(ws) || !aligned16(x)) return set_error(VAE_ERR_ALIGN, "mid_attention: x/workspace alignment");
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    __half* xn = reinterpret_cast<__half*>(w8 + L.xn);
    __half* q = reinterpret_cast<__half*>(w8 + L.q);
    __half* k = reinterpret_cast<__half*>(w8 + L.k);
    __half* vt = reinterpret_cast<__half*>(w8 + L.vt);
    __half* o = reinterpret_cast<__half*>(w8 + L.o);
    if (norm_kind == VAE_NORM_GROUP)
        rc = gn_run(x, 1, m, c, groups, eps, nullptr, gamma, beta, 0, 1.0f, xn, w8 + L.gn, L.total - L.gn, stream);
    else
        rc = rms_run(x, m, c, nullptr, gamma, 0, 1.0f, xn, stream);
    if (rc != VAE_OK) return rc;
    if (L.m_pad > m)
        VAE_CUDA_CHECK(cudaMemsetAsync(xn + static_cast<size_t>(m) * c, 0,
                                       static_cast<size_t>(L.m_pad - m) * c * 2, stream));
    ConvArgs a{};
    a.taps = 1;
    a.n = 1;
    a.h_in = 1;
    a.cin = c;
    a.out_f16 = true;
    // q, k = xn W^T + b (f16)
    a.x = xn;
    a.w_in = m;
    a.cout = c;
    a.w = wq;
    a.bias = bq;
    a.y = q;
    if ((rc = conv_run(a, stream)) != VAE_OK) return rc;
    a.w = wk;
    a.bias = bk;
    a.y = k;
    if ((rc = conv_run(a, stream)) != VAE_OK) return rc;
    // v^T [c][m_pad] = W_v xn^T (no bias: added after P.V)
    a.x = wv;
    a.w_in = c;
    a.w = xn;
    a.cout = L.m_pad;
    a.bias = nullptr;
    a.y = vt;
    if ((rc = conv_run(a, stream)) != VAE_OK) return rc;
    if ((rc = attn_core_run(q, k, vt, m, L.m_pad, c, bv, o, stream)) != VAE_OK) return rc;
    // x += o W_o^T + b_o
    ConvArgs pr{};
    pr.taps = 1;
    pr.n = 1;
    pr.h_in = 1;
    pr.w_in = m;
    pr.cin = c;
    pr.cout = c;
    pr.x = o;
    pr.w = wo;
    pr.bias = bo;
    pr.residual = x;
    pr.y = x;
    return conv_run(pr, stream);
}

}  // namespace vae

using namespace vae;

extern "C" {

size_t vae_mid_attention_workspace_bytes(int m, int c, int groups) {
    // Enough for either norm kind; channel counts GroupNorm cannot split into
    // `groups` still get the RMS_norm size.
    size_t b = 0;
    if (attn_workspace_bytes(m, c, groups, VAE_NORM_GROUP, &b) == VAE_OK) return b;
    clear_error();
    if (attn_workspace_bytes(m, c, groups, VAE_NORM_RMS, &b) != VAE_OK) return 0;
    return b;
}

int vae_mid_attention(float* x_dev, int m, int c, int norm_kind, int groups, float eps,
                      const float* norm_gamma_dev, const float* norm_beta_dev, const void* wq_dev,
                      const float* bq_dev, const void* wk_dev, const float* bk_dev, const void* wv_dev,
                      const float* bv_dev, const void* wo_dev, const float* bo_dev, void* workspace_dev,
                      size_t workspace_bytes, vae_stream_t stream) {
    clear_error();
    return attn_run(x_dev, m, c, norm_kind, groups, eps, norm_gamma_dev, norm_beta_dev, wq_dev, bq_dev, wk_dev,
                    bk_dev, wv_dev, bv_dev, wo_dev, bo_dev, workspace_dev, workspace_bytes,
                    reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

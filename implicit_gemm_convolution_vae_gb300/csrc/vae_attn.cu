// Mid-block single-head spatial self-attention ("vae.rs" AttnBlock::apply /
// finish; "qi21_vae.rs" attention): norm -> projections (the implicit-GEMM
// kernel with one tap, on CTA pairs) -> o = softmax(q k^T / sqrt(c)) v by two
// tcgen05 kernels -> output projection added onto the stream by the conv
// epilogue's residual path.
//
// Folded form (the default; VAE_ATTN_FOLD=0 runs the projections as written):
// the key bias adds the same amount to every score of a row, which the softmax
// removes, and each softmax row sums to one, so with M = Wk^T Wq the scores are
// q'_i . n_j, q' = n M^T + Wk^T bq, and the output is
// (sum_j p_ij n_j / l_i) (Wo Wv)^T + (Wo bv + bo): keys and values are the
// normalised rows themselves (n, and n^T for the P.V operand).
//
// Scores kernel (clusters of two query tiles, tcgen05.mma.cta_group::2, M = 256;
// a single-CTA form for one tile): S = Q K^T for 256 keys accumulates in one of
// two TMEM buffers from 64-channel chunks of Q and K streamed by TMA (each CTA
// of a pair loads its Q chunk and half of the keys). Eight softmax warps (one
// query row per thread; two warps per TMEM lane quadrant, one per key half)
// read S with tcgen05.ld, mask keys >= m and keep a running max m and sum l
// (online softmax, rescaling only when the max grows by more than 2^8, so the
// unnormalised P = 2^(s - m) stays <= 256 in f16). They write P (f16) to a
// row-major workspace, the factor alpha_j each row's O must be scaled by before
// block j is added (1 when its max did not move), one "some row rescaled" flag
// per lane quadrant and block, and the final l.
//
// PV kernel (clusters of two query tiles per value-channel chunk of <= 384; a
// single-CTA form): O += P_j V_j^T in TMEM from TMA-streamed 64-key halves of
// P and V^T; on a flagged block the row warps scale O by alpha_j after PV(j-1)
// and before PV(j). The epilogue writes O / l (+ b_v when the values carry a
// bias: added after P.V, exact because the rows of the softmax sum to one) as
// f16.
//
// S is computed once however many value chunks c needs (the O accumulator of
// c = 1152 columns cannot live in one SM's 512 TMEM columns, so a fused kernel
// had to recompute S per chunk, doubling the tensor work), at the price of
// writing P (2 bytes per score) once and reading it once per chunk. Query tiles
// run in groups whose P fits a 2 GiB workspace. Every wait is bounded.
#include <algorithm>
#include <cmath>
#include <cstdlib>

#include "vae_attn.h"
#include "vae_conv.h"
#include "vae_norm.h"

namespace vae {

namespace {

constexpr int kThreads = 192;
constexpr int kStageBytes = 64 * 1024;  // PV: a 64-key P half + V^T half
constexpr int kStages = 3;
// scores: one 64-channel chunk of Q (128 rows) and of K (256 keys) per stage
constexpr int kScStageBytes = 48 * 1024;
constexpr int kScStages = 4;
static_assert(kScStages * kScStageBytes <= kStages * kStageBytes, "scores ring over the shared ring bytes");
constexpr int kRingBars = 8;  // barrier slots of each ring array
static_assert(1024 + kStages * kStageBytes + 256 <= 232448, "attention shared memory over 227 KB");
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxDv = 384;
// The value bias, or 0 where the values carry none (the folded form adds it
// through the output projection's bias).
__device__ __forceinline__ float bias_at(const float* b, int i) { return b != nullptr ? __ldg(b + i) : 0.f; }
constexpr int kMaxFlagWords = 256;                   // key blocks <= 8192, i.e. m <= 2^20
constexpr size_t kMaxPBytes = size_t(2) << 30;       // P of one group of query tiles
constexpr int kPHalfBytes = 128 * 64 * 2;            // 128 query rows x 64 keys

struct ScoreParams {
    int m, nkb, nchunk_c;
    int q_tile0;   // first query tile of this group
    int ntiles;    // query tiles of this group (the pair kernel's odd last tile may be missing)
    int kcols;     // P row length (nkb * 128)
    int grows;     // rows of the group buffers (tiles * 128)
    float scale_log2;
    __half* p;        // [grows][kcols]
    float* alpha;     // [nkb][grows]
    float* lsum;      // [grows]
    uint32_t* flags;  // [tiles][nkb][4]
    DevStatus* status;
    unsigned long long timeout_ns;
};

struct PvParams {
    int m, c, dv, ndv, nkb;
    int ntiles;    // query tiles of this group (the pair kernel's odd last tile may be missing)
    int q_tile0, grows;
    int vbox_rows, vboxes;
    const float* alpha;
    const float* lsum;
    const uint32_t* flags;
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

__device__ __forceinline__ void st_v8_b32(void* dst, const uint32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

struct ASmem {
    uint8_t* ring;
    uint64_t *full, *empty;    // [kRingBars]
    uint64_t *s_full, *s_free;  // [2] (scores)
    uint64_t* resc_ready;       // (PV) MMAs up to PV(j-1) done before a flagged block j
    uint64_t* scaled;           // (PV) O scaled by alpha_j
    uint64_t* final;            // (PV) every PV done
    uint64_t* drain;
    uint32_t* tmem_slot;
    int* abort_flag;
};

// ring_bytes: the ring's size; the barriers (<= 256 bytes) follow it.
__device__ __forceinline__ ASmem carve_attn(uint8_t* raw, int ring_bytes = kStages * kStageBytes) {
    ASmem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.ring = base;
    uint64_t* b = reinterpret_cast<uint64_t*>(base + ring_bytes);
    s.full = b;
    s.empty = b + kRingBars;
    s.s_full = b + 2 * kRingBars;
    s.s_free = s.s_full + 2;
    s.resc_ready = s.s_free + 2;
    s.scaled = s.resc_ready + 1;
    s.final = s.scaled + 1;
    s.drain = s.final + 1;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
    return s;
}

__device__ __forceinline__ bool wait_(uint64_t* bar, uint32_t parity, const ASmem& s, DevStatus* st,
                                      unsigned long long timeout) {
    return mbar_wait(smem_u32(bar), parity, s.abort_flag, timeout, st, kWhereAttn);
}

// The same wait taken by a whole warp, with a warp-uniform result.
__device__ __forceinline__ bool wwait_(uint64_t* bar, uint32_t parity, const ASmem& s, DevStatus* st,
                                       unsigned long long timeout) {
    return warp_all(wait_(bar, parity, s, st, timeout));
}

__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

__device__ __forceinline__ bool wait_c(uint64_t* bar, uint32_t parity, const ASmem& s, DevStatus* st,
                                       unsigned long long timeout) {
    return mbar_wait_cluster(smem_u32(bar), parity, s.abort_flag, timeout, st, kWhereAttn);
}

// Ring bookkeeping shared by the producers and MMA threads (N slots).
template <int N>
struct RingT {
    int stage = 0;
    uint32_t phase = 0, armed = 0, arm_par = 0;
    __device__ __forceinline__ void next() {
        if (++stage == N) {
            stage = 0;
            phase ^= 1u;
        }
    }
    __device__ __forceinline__ void arm() {
        armed |= 1u << stage;
        arm_par = (arm_par & ~(1u << stage)) | (phase << stage);
    }
    // Lets every copy this thread started land before the CTA can exit.
    __device__ __forceinline__ void drain(const ASmem& s, DevStatus* st, unsigned long long timeout) const {
        int never = 0;
        for (int i = 0; i < N; ++i)
            if (armed & (1u << i))
                (void)mbar_wait(smem_u32(&s.full[i]), (arm_par >> i) & 1u, &never, timeout, st, kWhereDrain);
    }
};
using Ring = RingT<kStages>;

__device__ __forceinline__ void mma_drain(const ASmem& s, DevStatus* st, unsigned long long timeout) {
    umma_commit(smem_u32(s.drain));
    int never = 0;
    (void)mbar_wait(smem_u32(s.drain), 0u, &never, timeout, st, kWhereDrain);
}

// ───────────────────────────── scores kernel ─────────────────────────────

__device__ void scores_producer(const ScoreParams& p, const ASmem& s, const CUtensorMap* mq, const CUtensorMap* mk,
                                int q0) {
    const uint64_t pol = policy_evict_normal();
    RingT<kScStages> r;
    const int npair = (p.nkb + 1) / 2;
    for (int jj = 0; jj < npair; ++jj)  // 256 keys per pass: each Q chunk serves two key blocks
        for (int cc = 0; cc < p.nchunk_c; ++cc) {
            if (!wait_(&s.empty[r.stage], r.phase ^ 1u, s, p.status, p.timeout_ns)) {
                r.drain(s, p.status, p.timeout_ns);
                return;
            }
            const uint32_t fb = smem_u32(&s.full[r.stage]);
            mbar_arrive_expect_tx(fb, static_cast<uint32_t>(kScStageBytes));
            r.arm();
            uint8_t* st = s.ring + r.stage * kScStageBytes;
            tma_load_2d(smem_u32(st), mq, fb, cc * 64, q0, pol);
            tma_load_2d(smem_u32(st + 16384), mk, fb, cc * 64, jj * 256, pol);  // keys >= m read as zeros
            r.next();
        }
    r.drain(s, p.status, p.timeout_ns);
}

__device__ void scores_mma(const ScoreParams& p, const ASmem& s, uint32_t tmem) {
    const uint32_t id_s = idesc_f16_f32(128, 256);
    const uint64_t q_desc0 = sw128_kmajor_desc(smem_u32(s.ring));  // every ring address stays below 2^18 bytes
    RingT<kScStages> r;
    bool ok = true;
    const int npair = (p.nkb + 1) / 2;
    for (int jj = 0; jj < npair && ok; ++jj) {
        const int b = jj & 1;
        if (jj >= 2) {  // the softmax has read S(jj - 2) out of this buffer
            if (!wait_(&s.s_free[b], static_cast<uint32_t>(((jj - 2) >> 1) & 1), s, p.status, p.timeout_ns)) break;
            tc_fence_after();
        }
        for (int cc = 0; cc < p.nchunk_c; ++cc) {
            if (!wait_(&s.full[r.stage], r.phase, s, p.status, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // slot descriptors as running values (16-byte units: slot r.stage at r.stage * kScStageBytes)
            const uint64_t ad = q_desc0 + static_cast<uint32_t>(r.stage) * (kScStageBytes >> 4);
            const uint64_t bd = ad + (16384u >> 4);
            const uint32_t dS = tmem + static_cast<uint32_t>(b * 256);
            umma_f16(dS, ad, bd, id_s, cc != 0 ? 1u : 0u);  // S(128 x 256) += Q_c K_c^T, K = 16 per step
#pragma unroll
            for (int k = 1; k < 4; ++k) umma_f16(dS, ad + 2u * k, bd + 2u * k, id_s, 1u);
            umma_commit(smem_u32(&s.empty[r.stage]));
            r.next();
        }
        if (ok) umma_commit(smem_u32(&s.s_full[b]));
    }
    mma_drain(s, p.status, p.timeout_ns);
}

// One thread per query row. Per pass of 256 keys (two key blocks): the row max
// from a first read of S, the rescale decision (the running max moves only when
// the new one exceeds it by more than 2^8, so P = 2^(s - m) <= 256 fits f16),
// then a second read of S for P (f16), the row sum and the per-block rescale
// factors and flags the PV kernel replays (the pass's second block never
// rescales).
// Eight softmax warps, one query row per thread: warp w reads TMEM lane
// quadrant w % 4 (its 32 rows) and key half w / 4 (128 of the pass's 256 keys).
// Per pass of 256 keys (two key blocks): the row max from a first read of S;
// the two warps of a quadrant trade their half maxima through shared memory on
// a bounded barrier, so both take the same max and the same rescale decision
// (the running max moves only when the new one exceeds it by more than 2^8, so
// P = 2^(s - m) <= 256 fits f16); then a second read of S for P (f16) and a
// partial row sum. The first half writes the per-block rescale factors and
// flags the PV kernel replays (the pass's second block never rescales); at the
// end the second half's partial sum joins the first's (l = l0 + l1).
// kPair: a CTA of a pair (S arrives by the even CTA's multicast commit; the
// buffer is released on the even CTA's barrier, which counts both CTAs' rows);
// live: this CTA's query tile exists (a missing odd tile of a pair writes
// nothing but still takes part in every barrier).
// 2^x by the PTX approximate base-2 exponential (relative error far below the
// 2^-11 of the f16 P it feeds; results under 2^-126 flush to zero, where f16
// holds nothing either).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr int kScWarps = 8;                       // softmax warps of the scores kernels
constexpr int kScThreads = (kScWarps + 2) * 32;   // + producer + MMA warp
constexpr int kScProducerWarp = kScWarps, kScMmaWarp = kScWarps + 1;

struct ScExchange {
    float* xmax;     // [2 pass parities][2 halves][128 rows]
    float* xl;       // [128 rows]: the second half's partial row sum
    uint64_t* xbar;  // [4]: the two warps (64 threads) of each lane quadrant
};

template <bool kPair>
__device__ void scores_softmax(const ScoreParams& p, const ASmem& s, uint32_t tmem, int warp, int lane, int tl,
                               bool live, const ScExchange& x) {
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;
    const int row = tl * 128 + r;  // row of the group buffers
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    __half* prow = p.p + static_cast<size_t>(row) * p.kcols;
    const uint32_t xb = smem_u32(&x.xbar[quad]);
    uint32_t xph = 0;
    auto exchange = [&]() -> bool {
        mbar_arrive(xb);
        const bool ok = mbar_wait(xb, xph, s.abort_flag, p.timeout_ns, p.status, kWhereAttn);
        xph ^= 1u;
        return warp_all(ok);
    };
    float m_run = -INFINITY, l = 0.f;
    const int npair = (p.nkb + 1) / 2;
    for (int jj = 0; jj < npair; ++jj) {
        const int b = jj & 1;
        const uint32_t par = static_cast<uint32_t>((jj >> 1) & 1);
        if (!(kPair ? warp_all(wait_c(&s.s_full[b], par, s, p.status, p.timeout_ns))
                    : wwait_(&s.s_full[b], par, s, p.status, p.timeout_ns)))
            return;
        tc_fence_after();
        const int kbase = jj * 256 + half * 128;  // this warp's first key
        const uint32_t sb = tmem + lane_off + static_cast<uint32_t>(b * 256 + half * 128);
        // S is read in batches of four 16-column loads under one wait.
        const bool all_in = kbase + 128 <= p.m;  // no key of this half is past m
        float mx = -INFINITY;
        for (int g = 0; g < 8; g += 4) {
            uint32_t rr[4][16];
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 4; ++u) tmem_ld16(sb + static_cast<uint32_t>((g + u) * 16), rr[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) tmem_ld_wait_regs(rr[u]);
            if (all_in) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int i = 0; i < 16; ++i) mx = fmaxf(mx, __uint_as_float(rr[u][i]));
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (kbase + (g + u) * 16 + i < p.m) mx = fmaxf(mx, __uint_as_float(rr[u][i]));
            }
        }
        mx *= p.scale_log2;  // (the scale is positive: the max of the scaled scores)
        float* xm = x.xmax + (jj & 1) * 256;
        xm[half * 128 + r] = mx;
        if (!exchange()) return;
        mx = fmaxf(xm[r], xm[128 + r]);
        float alpha = 1.f;
        bool resc = false;
        if (jj == 0) {
            m_run = mx;
        } else if (mx > m_run + 8.f) {
            alpha = exp2f(m_run - mx);
            m_run = mx;
            resc = true;
        }
        const bool any = __any_sync(0xffffffffu, resc);
        const int j0 = 2 * jj, j1 = 2 * jj + 1;
        if (live && half == 0) {
            if (j0 >= 1) {
                p.alpha[static_cast<size_t>(j0) * p.grows + row] = alpha;
                if (lane == 0) p.flags[(static_cast<size_t>(tl) * p.nkb + j0) * 4 + quad] = any ? 1u : 0u;
            }
            if (j1 < p.nkb) {
                p.alpha[static_cast<size_t>(j1) * p.grows + row] = 1.f;
                if (lane == 0) p.flags[(static_cast<size_t>(tl) * p.nkb + j1) * 4 + quad] = 0u;
            }
        }
        l *= alpha;
        float sum = 0.f;
        const int ngr = live && kbase < p.nkb * 128 ? 8 : 0;  // this half's 16-key groups with P columns
        for (int g = 0; g < ngr; g += 4) {
            uint32_t rr[4][16];
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 4; ++u) tmem_ld16(sb + static_cast<uint32_t>((g + u) * 16), rr[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) tmem_ld_wait_regs(rr[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t h[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int key = kbase + (g + u) * 16 + 2 * i;
                    float a = ex2_approx(fmaf(__uint_as_float(rr[u][2 * i]), p.scale_log2, -m_run));
                    float c = ex2_approx(fmaf(__uint_as_float(rr[u][2 * i + 1]), p.scale_log2, -m_run));
                    if (!all_in) {
                        a = key < p.m ? a : 0.f;
                        c = key + 1 < p.m ? c : 0.f;
                    }
                    sum += a + c;
                    __half2 t = __floats2half2_rn(a, c);
                    h[i] = *reinterpret_cast<uint32_t*>(&t);
                }
                st_v8_b32(prow + kbase + (g + u) * 16, h);
            }
        }
        tc_fence_before();
        if (kPair)
            mbar_arrive_cluster(mapa_shared(smem_u32(&s.s_free[b]), 0u));
        else
            mbar_arrive(smem_u32(&s.s_free[b]));
        l += sum;
    }
    if (half == 1) x.xl[r] = l;
    if (!exchange()) return;
    if (live && half == 0) p.lsum[row] = l + x.xl[r];
}

__global__ void __launch_bounds__(kScThreads, 1)
    attn_scores_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ float xmax[2 * 2 * 128], xl[128];
    __shared__ uint64_t xbar[4];
    const ASmem s = carve_attn(smem_raw);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int tl = blockIdx.x;
    const int q0 = (p.q_tile0 + tl) * 128;
    if (threadIdx.x == 0) {
        *s.abort_flag = 0;
        for (int i = 0; i < kScStages; ++i) {
            mbar_init(smem_u32(&s.full[i]), 1u);
            mbar_init(smem_u32(&s.empty[i]), 1u);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s.s_full[i]), 1u);
            mbar_init(smem_u32(&s.s_free[i]), 32u * kScWarps);
        }
        mbar_init(smem_u32(s.drain), 1u);
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&xbar[i]), 64u);
        fence_mbar_init();
    }
    if (warp == kScMmaWarp) {
        tmem_alloc(smem_u32(s.tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kScProducerWarp && lane == 0) {
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
    }
    pdl_wait();  // q, k come from the projections launched before
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s.tmem_slot;
    if (warp < kScWarps) {
        scores_softmax<false>(p, s, tmem, warp, lane, tl, true, ScExchange{xmax, xl, xbar});
    } else if (warp == kScProducerWarp) {
        if (lane == 0) scores_producer(p, s, &mq, &mk, q0);
    } else {
        if (lane == 0) scores_mma(p, s, tmem);
    }
    pdl_launch_dependents();  // this CTA's work is done
    tc_fence_before();
    __syncthreads();
    if (warp == kScMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ───────────────────────────── PV kernel ─────────────────────────────

__device__ __forceinline__ bool flagged(const uint32_t* fl, int j) { return (fl[j >> 5] >> (j & 31)) & 1u; }

__device__ void pv_producer(const PvParams& p, const ASmem& s, const CUtensorMap* mp, const CUtensorMap* mv, int tl,
                            int d0) {
    const uint64_t pol = policy_evict_normal();
    const uint32_t tx = static_cast<uint32_t>(kPHalfBytes + p.vboxes * p.vbox_rows * 128);
    Ring r;
    for (int j = 0; j < p.nkb; ++j)
        for (int half = 0; half < 2; ++half) {
            if (!wait_(&s.empty[r.stage], r.phase ^ 1u, s, p.status, p.timeout_ns)) {
                r.drain(s, p.status, p.timeout_ns);
                return;
            }
            const uint32_t fb = smem_u32(&s.full[r.stage]);
            mbar_arrive_expect_tx(fb, tx);
            r.arm();
            uint8_t* st = s.ring + r.stage * kStageBytes;
            const int key0 = j * 128 + half * 64;
            tma_load_2d(smem_u32(st), mp, fb, key0, tl * 128, pol);
            for (int b = 0; b < p.vboxes; ++b)
                tma_load_2d(smem_u32(st + kPHalfBytes + b * p.vbox_rows * 128), mv, fb, key0, d0 + b * p.vbox_rows,
                            pol);
            r.next();
        }
    r.drain(s, p.status, p.timeout_ns);
}

__device__ void pv_mma(const PvParams& p, const ASmem& s, uint32_t tmem, const uint32_t* fl) {
    const int nsplit = p.dv > 256 ? 2 : 1;
    const int ns = p.dv / nsplit;
    const uint32_t id_o = idesc_f16_f32(128, ns);
    const uint64_t p_desc0 = sw128_kmajor_desc(smem_u32(s.ring));  // every ring address stays below 2^18 bytes
    const uint32_t v_split = static_cast<uint32_t>(ns * 128) >> 4;   // second V^T half, in descriptor units
    Ring r;
    uint32_t ev = 0;
    bool ok = true;
    for (int j = 0; j < p.nkb && ok; ++j) {
        if (j >= 1 && flagged(fl, j)) {
            // The row warps scale O by alpha_j once PV(j - 1) is done; both
            // sides count these events in the same order.
            umma_commit(smem_u32(s.resc_ready));
            if (!wait_(s.scaled, ev & 1u, s, p.status, p.timeout_ns)) {
                ok = false;
                break;
            }
            ++ev;
            tc_fence_after();
        }
        for (int half = 0; half < 2; ++half) {
            if (!wait_(&s.full[r.stage], r.phase, s, p.status, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // slot descriptors as running values: P half at the slot, V^T halves after it
            const uint64_t ad = p_desc0 + static_cast<uint32_t>(r.stage) * (kStageBytes >> 4);
            const uint64_t bd0 = ad + (static_cast<uint32_t>(kPHalfBytes) >> 4);
            const uint32_t acc0 = (j | half) != 0 ? 1u : 0u;
            if (nsplit == 2) {
                const uint64_t bd1 = bd0 + v_split;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    umma_f16(tmem, ad + 2u * k, bd0 + 2u * k, id_o, k != 0 ? 1u : acc0);
                    umma_f16(tmem + static_cast<uint32_t>(ns), ad + 2u * k, bd1 + 2u * k, id_o, k != 0 ? 1u : acc0);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) umma_f16(tmem, ad + 2u * k, bd0 + 2u * k, id_o, k != 0 ? 1u : acc0);
            }
            umma_commit(smem_u32(&s.empty[r.stage]));
            r.next();
        }
    }
    if (ok) umma_commit(smem_u32(s.final));
    mma_drain(s, p.status, p.timeout_ns);
}

__device__ void pv_rows(const PvParams& p, const ASmem& s, uint32_t tmem, const uint32_t* fl, int warp, int lane,
                        int tl, int d0) {
    const int r = warp * 32 + lane;
    const int row = tl * 128 + r;
    const uint32_t tO = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    uint32_t ev = 0;
    for (int j = 1; j < p.nkb; ++j) {
        if (!flagged(fl, j)) continue;
        if (!wwait_(s.resc_ready, ev & 1u, s, p.status, p.timeout_ns)) return;
        ++ev;
        tc_fence_after();
        const float alpha = p.alpha[static_cast<size_t>(j) * p.grows + row];
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
        tc_fence_before();
        mbar_arrive(smem_u32(s.scaled));
    }
    if (!wwait_(s.final, 0u, s, p.status, p.timeout_ns)) return;
    tc_fence_after();
    const float inv = 1.f / p.lsum[row];
    const int q = (p.q_tile0 + tl) * 128 + r;
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
                __half2 t = __floats2half2_rn(__uint_as_float(rr[2 * i]) * inv + bias_at(p.bv, d + 2 * i),
                                              __uint_as_float(rr[2 * i + 1]) * inv + bias_at(p.bv, d + 2 * i + 1));
                h[i] = *reinterpret_cast<uint32_t*>(&t);
            }
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(h[0], h[1], h[2], h[3]);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(h[4], h[5], h[6], h[7]);
        } else {
            for (int i = 0; i < 16 && d + i < p.c; ++i)
                dst[i] = __float2half_rn(__uint_as_float(rr[i]) * inv + bias_at(p.bv, d + i));
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_pv_kernel(const __grid_constant__ CUtensorMap mp, const __grid_constant__ CUtensorMap mv, const PvParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t fl[kMaxFlagWords];
    const ASmem s = carve_attn(smem_raw);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int tl = blockIdx.x / p.ndv;
    const int d0 = (blockIdx.x % p.ndv) * p.dv;
    const int nwords = (p.nkb + 31) / 32;
    for (int i = threadIdx.x; i < nwords; i += blockDim.x) fl[i] = 0u;
    if (threadIdx.x == 0) {
        *s.abort_flag = 0;
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&s.full[i]), 1u);
            mbar_init(smem_u32(&s.empty[i]), 1u);
        }
        mbar_init(smem_u32(s.resc_ready), 1u);
        mbar_init(smem_u32(s.scaled), 128u);
        mbar_init(smem_u32(s.final), 1u);
        mbar_init(smem_u32(s.drain), 1u);
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(s.tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&mp);
        tma_prefetch_desc(&mv);
    }
    pdl_wait();  // P, the flags and V come from kernels launched before
    __syncthreads();
    // The tile's "some row rescaled at block j" flags, one bit per key block.
    for (int j = 1 + threadIdx.x; j < p.nkb; j += blockDim.x) {
        const uint4 f = *reinterpret_cast<const uint4*>(p.flags + (static_cast<size_t>(tl) * p.nkb + j) * 4);
        if ((f.x | f.y | f.z | f.w) != 0u) atomicOr(&fl[j >> 5], 1u << (j & 31));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s.tmem_slot;
    if (warp < 4) {
        pv_rows(p, s, tmem, fl, warp, lane, tl, d0);
    } else if (warp == 4) {
        if (lane == 0) pv_producer(p, s, &mp, &mv, tl, d0);
    } else {
        if (lane == 0) pv_mma(p, s, tmem, fl);
    }
    pdl_launch_dependents();  // this CTA's work is done
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ───────────────────────── PV kernel on CTA pairs ─────────────────────────
// A cluster of two CTAs computes O for two query tiles (2t, 2t + 1 of the
// group) and one value chunk with tcgen05.mma.cta_group::2 (M = 256): each CTA
// streams its own tile's 64-key P half and HALF of every V^T box (the rows of
// N that the pair MMA takes from it), so per SM a stage carries 40 KB instead
// of 64 KB (the single-CTA kernel is bound by the bytes each SM takes in from
// L2). Both CTAs' copies complete on the even CTA's full barrier (armed once
// for the bytes of both); the even CTA's MMA thread commits with multicast.
// Rescaling follows the union of the two tiles' flags: on a flagged block j
// the row warps of BOTH CTAs scale their O rows (by 1 where their rows did
// not move) and arrive on the even CTA's `scaled` barrier. A missing odd tile
// (an odd tile count) reads zero-filled P, scales by 1 and stores nothing.
constexpr int kPvPairStageBytes = 40 * 1024;  // P half 16 KB + two V^T half boxes of <= 96 rows x 128 B
constexpr int kPvPairStages = 5;
static_assert(1024 + kPvPairStages * kPvPairStageBytes + 256 <= 232448, "PV pair shared memory over 227 KB");

__device__ void pvp_producer(const PvParams& p, const ASmem& s, const CUtensorMap* mp, const CUtensorMap* mv, int tl,
                             int d0, int rank) {
    const uint64_t pol = policy_evict_normal();
    const int nsplit = p.dv > 256 ? 2 : 1;
    const int ns = p.dv / nsplit, hrows = ns / 2;
    const uint32_t tx = static_cast<uint32_t>(kPHalfBytes + nsplit * hrows * 128);
    RingT<kPvPairStages> r;
    for (int j = 0; j < p.nkb; ++j)
        for (int half = 0; half < 2; ++half) {
            if (!wait_(&s.empty[r.stage], r.phase ^ 1u, s, p.status, p.timeout_ns)) {
                j = p.nkb;
                break;
            }
            const uint32_t fb = smem_u32(&s.full[r.stage]);
            if (rank == 0) mbar_arrive_expect_tx(fb, 2u * tx);
            r.arm();
            const uint32_t fbc = mapa_shared(fb, 0u);
            uint8_t* st = s.ring + r.stage * kPvPairStageBytes;
            const int key0 = j * 128 + half * 64;
            tma_load_2d_pair(smem_u32(st), mp, fbc, key0, tl * 128, pol);  // rows past the group read as zeros
            for (int sp = 0; sp < nsplit; ++sp)
                tma_load_2d_pair(smem_u32(st + kPHalfBytes + sp * hrows * 128), mv, fbc, key0,
                                 d0 + sp * ns + rank * hrows, pol);
            r.next();
        }
    // Let every copy land before the CTA can exit: the even CTA sees them on its
    // full barriers, the odd CTA on its empty barriers (the MMAs that read them).
    int never = 0;
    for (int i = 0; i < kPvPairStages; ++i)
        if (r.armed & (1u << i))
            (void)mbar_wait(smem_u32(rank == 0 ? &s.full[i] : &s.empty[i]), (r.arm_par >> i) & 1u, &never,
                            p.timeout_ns, p.status, kWhereDrain);
}

__device__ void pvp_mma(const PvParams& p, const ASmem& s, uint32_t tmem, const uint32_t* fl) {
    const int nsplit = p.dv > 256 ? 2 : 1;
    const int ns = p.dv / nsplit, hrows = ns / 2;
    const uint32_t id_o = idesc_f16_f32(256, ns);
    const uint64_t p_desc0 = sw128_kmajor_desc(smem_u32(s.ring));  // every ring address stays below 2^18 bytes
    const uint32_t v_split = static_cast<uint32_t>(hrows * 128) >> 4;
    RingT<kPvPairStages> r;
    uint32_t ev = 0;
    bool ok = true;
    for (int j = 0; j < p.nkb && ok; ++j) {
        if (j >= 1 && flagged(fl, j)) {
            // both CTAs' row warps scale O once PV(j - 1) is done
            umma_commit_pair(smem_u32(s.resc_ready));
            if (!wait_c(s.scaled, ev & 1u, s, p.status, p.timeout_ns)) {
                ok = false;
                break;
            }
            ++ev;
            tc_fence_after();
        }
        for (int half = 0; half < 2; ++half) {
            if (!wait_(&s.full[r.stage], r.phase, s, p.status, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t ad = p_desc0 + static_cast<uint32_t>(r.stage) * (kPvPairStageBytes >> 4);
            const uint64_t bd0 = ad + (static_cast<uint32_t>(kPHalfBytes) >> 4);
            const uint32_t acc0 = (j | half) != 0 ? 1u : 0u;
            if (nsplit == 2) {
                const uint64_t bd1 = bd0 + v_split;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    umma_f16_pair(tmem, ad + 2u * k, bd0 + 2u * k, id_o, k != 0 ? 1u : acc0);
                    umma_f16_pair(tmem + static_cast<uint32_t>(ns), ad + 2u * k, bd1 + 2u * k, id_o,
                                  k != 0 ? 1u : acc0);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) umma_f16_pair(tmem, ad + 2u * k, bd0 + 2u * k, id_o, k != 0 ? 1u : acc0);
            }
            umma_commit_pair(smem_u32(&s.empty[r.stage]));
            r.next();
        }
    }
    if (ok) umma_commit_pair(smem_u32(s.final));
    umma_commit_pair(smem_u32(s.drain));
    int never = 0;
    (void)mbar_wait(smem_u32(s.drain), 0u, &never, p.timeout_ns, p.status, kWhereDrain);
}

__device__ void pvp_rows(const PvParams& p, const ASmem& s, uint32_t tmem, const uint32_t* fl, int warp, int lane,
                         int tl, int d0, bool live) {
    const int r = warp * 32 + lane;
    const int row = tl * 128 + r;  // row of the group buffers (only read when the tile exists)
    const uint32_t tO = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t scaled_c = mapa_shared(smem_u32(s.scaled), 0u);
    uint32_t ev = 0;
    for (int j = 1; j < p.nkb; ++j) {
        if (!flagged(fl, j)) continue;
        // (arrived by the even CTA's multicast commit: acquire at cluster scope)
        if (!warp_all(wait_c(s.resc_ready, ev & 1u, s, p.status, p.timeout_ns))) return;
        ++ev;
        tc_fence_after();
        const float alpha = live ? p.alpha[static_cast<size_t>(j) * p.grows + row] : 1.f;
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
        tc_fence_before();
        mbar_arrive_cluster(scaled_c);
    }
    if (!warp_all(wait_c(s.final, 0u, s, p.status, p.timeout_ns))) return;
    tc_fence_after();
    if (!live) return;
    const float inv = 1.f / p.lsum[row];
    const int q = (p.q_tile0 + tl) * 128 + r;
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
                __half2 t = __floats2half2_rn(__uint_as_float(rr[2 * i]) * inv + bias_at(p.bv, d + 2 * i),
                                              __uint_as_float(rr[2 * i + 1]) * inv + bias_at(p.bv, d + 2 * i + 1));
                h[i] = *reinterpret_cast<uint32_t*>(&t);
            }
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(h[0], h[1], h[2], h[3]);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(h[4], h[5], h[6], h[7]);
        } else {
            for (int i = 0; i < 16 && d + i < p.c; ++i)
                dst[i] = __float2half_rn(__uint_as_float(rr[i]) * inv + bias_at(p.bv, d + i));
        }
    }
}

// grid: 2 x (tile pairs of the group) x ndv, clusters of 2; p.ntiles = tiles of the group.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_pv_pair_kernel(const __grid_constant__ CUtensorMap mp, const __grid_constant__ CUtensorMap mv,
                        const PvParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t fl[kMaxFlagWords];
    const ASmem s = carve_attn(smem_raw, kPvPairStages * kPvPairStageBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rank = static_cast<int>(cluster_ctarank());
    const int cl = blockIdx.x >> 1;
    const int tl = (cl / p.ndv) * 2 + rank;
    const int d0 = (cl % p.ndv) * p.dv;
    const bool live = tl < p.ntiles;
    const int nwords = (p.nkb + 31) / 32;
    for (int i = threadIdx.x; i < nwords; i += blockDim.x) fl[i] = 0u;
    if (threadIdx.x == 0) {
        *s.abort_flag = 0;
        for (int i = 0; i < kPvPairStages; ++i) {
            mbar_init(smem_u32(&s.full[i]), 1u);
            mbar_init(smem_u32(&s.empty[i]), 1u);
        }
        mbar_init(smem_u32(s.resc_ready), 1u);
        mbar_init(smem_u32(s.scaled), 256u);  // the row threads of both CTAs
        mbar_init(smem_u32(s.final), 1u);
        mbar_init(smem_u32(s.drain), 1u);
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc_pair(smem_u32(s.tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&mp);
        tma_prefetch_desc(&mv);
    }
    pdl_wait();  // P, the flags and V come from kernels launched before
    __syncthreads();
    // The union of the two tiles' "some row rescaled at block j" flags.
    const int t0 = (cl / p.ndv) * 2;
    for (int j = 1 + threadIdx.x; j < p.nkb; j += blockDim.x) {
        uint32_t any = 0u;
        for (int t = t0; t < t0 + 2 && t < p.ntiles; ++t) {
            const uint4 f = *reinterpret_cast<const uint4*>(p.flags + (static_cast<size_t>(t) * p.nkb + j) * 4);
            any |= f.x | f.y | f.z | f.w;
        }
        if (any != 0u) atomicOr(&fl[j >> 5], 1u << (j & 31));
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers and TMEM exist before any remote arrive or pair MMA
    tc_fence_after();
    const uint32_t tmem = *s.tmem_slot;
    if (warp < 4) {
        pvp_rows(p, s, tmem, fl, warp, lane, tl, d0, live);
    } else if (warp == 4) {
        if (lane == 0) pvp_producer(p, s, &mp, &mv, tl, d0, rank);
    } else {
        if (lane == 0 && rank == 0) pvp_mma(p, s, tmem, fl);
    }
    pdl_launch_dependents();  // this CTA's work is done
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the even CTA's MMAs into both TMEMs are done; no remote arrives remain
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

// ─────────────────────── scores kernel on CTA pairs ───────────────────────
// A cluster of two CTAs computes S for two query tiles (2t, 2t + 1 of the
// group) with tcgen05.mma.cta_group::2 (M = 256, N = 256 keys per pass): each
// CTA streams its own tile's 64-channel Q chunk and HALF of the pass's 256 keys
// (the 128 rows of N the pair MMA takes from it), 32 KB per stage per SM
// instead of 48 KB. Both CTAs' copies complete on the even CTA's full barrier;
// the even CTA's MMA thread commits with multicast (ring slots to both empty
// barriers, each S buffer to both CTAs' s_full), and the softmax rows of both
// CTAs release an S buffer on the even CTA's s_free (256 arrivals). The
// softmax itself is the single-CTA kernel's, row for row, so P, the factors
// and the flags are the same bits.
constexpr int kScPairStageBytes = 32 * 1024;  // Q chunk 128 x 64 + K half 128 x 64 (f16)
constexpr int kScPairStages = 6;
static_assert(1024 + kScPairStages * kScPairStageBytes + 256 <= 232448, "scores pair shared memory over 227 KB");
static_assert(kScPairStages <= kRingBars, "scores pair ring over the barrier slots");

__device__ void scp_producer(const ScoreParams& p, const ASmem& s, const CUtensorMap* mq, const CUtensorMap* mk,
                             int q0, int rank) {
    const uint64_t pol = policy_evict_normal();
    RingT<kScPairStages> r;
    const int npair = (p.nkb + 1) / 2;
    bool ok = true;
    for (int jj = 0; jj < npair && ok; ++jj)
        for (int cc = 0; cc < p.nchunk_c; ++cc) {
            if (!wait_(&s.empty[r.stage], r.phase ^ 1u, s, p.status, p.timeout_ns)) {
                ok = false;
                break;
            }
            const uint32_t fb = smem_u32(&s.full[r.stage]);
            if (rank == 0) mbar_arrive_expect_tx(fb, 2u * static_cast<uint32_t>(kScPairStageBytes));
            r.arm();
            const uint32_t fbc = mapa_shared(fb, 0u);
            uint8_t* st = s.ring + r.stage * kScPairStageBytes;
            tma_load_2d_pair(smem_u32(st), mq, fbc, cc * 64, q0, pol);  // rows past m read as zeros
            tma_load_2d_pair(smem_u32(st + 16384), mk, fbc, cc * 64, jj * 256 + rank * 128, pol);
            r.next();
        }
    // every copy lands before the CTA can exit: the even CTA sees them on its
    // full barriers, the odd CTA on its empty barriers (the MMAs that read them)
    int never = 0;
    for (int i = 0; i < kScPairStages; ++i)
        if (r.armed & (1u << i))
            (void)mbar_wait(smem_u32(rank == 0 ? &s.full[i] : &s.empty[i]), (r.arm_par >> i) & 1u, &never,
                            p.timeout_ns, p.status, kWhereDrain);
}

__device__ void scp_mma(const ScoreParams& p, const ASmem& s, uint32_t tmem) {
    const uint32_t id_s = idesc_f16_f32(256, 256);
    const uint64_t q_desc0 = sw128_kmajor_desc(smem_u32(s.ring));  // every ring address stays below 2^18 bytes
    RingT<kScPairStages> r;
    bool ok = true;
    const int npair = (p.nkb + 1) / 2;
    for (int jj = 0; jj < npair && ok; ++jj) {
        const int b = jj & 1;
        if (jj >= 2) {  // both CTAs' softmax rows have read S(jj - 2) out of this buffer
            if (!wait_c(&s.s_free[b], static_cast<uint32_t>(((jj - 2) >> 1) & 1), s, p.status, p.timeout_ns)) break;
            tc_fence_after();
        }
        for (int cc = 0; cc < p.nchunk_c; ++cc) {
            if (!wait_(&s.full[r.stage], r.phase, s, p.status, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t ad = q_desc0 + static_cast<uint32_t>(r.stage) * (kScPairStageBytes >> 4);
            const uint64_t bd = ad + (16384u >> 4);
            const uint32_t dS = tmem + static_cast<uint32_t>(b * 256);
            umma_f16_pair(dS, ad, bd, id_s, cc != 0 ? 1u : 0u);  // S(256 x 256) += Q_c K_c^T
#pragma unroll
            for (int k = 1; k < 4; ++k) umma_f16_pair(dS, ad + 2u * k, bd + 2u * k, id_s, 1u);
            umma_commit_pair(smem_u32(&s.empty[r.stage]));
            r.next();
        }
        if (ok) umma_commit_pair(smem_u32(&s.s_full[b]));
    }
    umma_commit_pair(smem_u32(s.drain));
    int never = 0;
    (void)mbar_wait(smem_u32(s.drain), 0u, &never, p.timeout_ns, p.status, kWhereDrain);
}

// grid: 2 x (tile pairs of the group), clusters of 2; p.ntiles = tiles of the group.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kScThreads, 1)
    attn_scores_pair_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                            const ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ float xmax[2 * 2 * 128], xl[128];
    __shared__ uint64_t xbar[4];
    const ASmem s = carve_attn(smem_raw, kScPairStages * kScPairStageBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rank = static_cast<int>(cluster_ctarank());
    const int tl = (blockIdx.x >> 1) * 2 + rank;
    const bool live = tl < p.ntiles;
    const int q0 = (p.q_tile0 + tl) * 128;
    if (threadIdx.x == 0) {
        *s.abort_flag = 0;
        for (int i = 0; i < kScPairStages; ++i) {
            mbar_init(smem_u32(&s.full[i]), 1u);
            mbar_init(smem_u32(&s.empty[i]), 1u);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s.s_full[i]), 1u);
            mbar_init(smem_u32(&s.s_free[i]), 2u * 32u * kScWarps);  // the softmax rows of both CTAs
        }
        mbar_init(smem_u32(s.drain), 1u);
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&xbar[i]), 64u);
        fence_mbar_init();
    }
    if (warp == kScMmaWarp) {
        tmem_alloc_pair(smem_u32(s.tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == kScProducerWarp && lane == 0) {
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
    }
    pdl_wait();  // q and the keys come from kernels launched before
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers and TMEM exist before any remote arrive or pair MMA
    tc_fence_after();
    const uint32_t tmem = *s.tmem_slot;
    if (warp < kScWarps) {
        scores_softmax<true>(p, s, tmem, warp, lane, tl, live, ScExchange{xmax, xl, xbar});
    } else if (warp == kScProducerWarp) {
        if (lane == 0) scp_producer(p, s, &mq, &mk, q0, rank);
    } else {
        if (lane == 0 && rank == 0) scp_mma(p, s, tmem);
    }
    pdl_launch_dependents();  // this CTA's work is done
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the even CTA's MMAs into both TMEMs are done; no remote arrives remain
    if (warp == kScMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

struct AttnLayout {
    int m_pad, ndv, dv;
    int qtiles, nkb, group;  // query tiles, key blocks, query tiles per scores/PV launch pair
    size_t xn, q, k, vt, o, gn, p, alpha, lsum, flags;
    size_t wqk, wov, bqk, bov, wT;  // the folded weights and the transposes they are made from
    size_t total;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

int attn_layout(int m, int c, int groups, int norm_kind, AttnLayout* L) {
    if (m < 1 || m > kMaxFlagWords * 32 * 128 || c < 16 || c % 16 != 0 || c > 2048)
        return set_error(VAE_ERR_SHAPE, "mid_attention: m=%d c=%d (need 1 <= m <= 2^20, c %% 16 == 0, 16 <= c <= 2048)",
                         m, c);
    L->qtiles = (m + 127) / 128;
    L->nkb = L->qtiles;
    {
        const size_t row_block = static_cast<size_t>(128) * L->nkb * 128 * 2;  // P of one query tile
        L->group = static_cast<int>(std::min<size_t>(L->qtiles, std::max<size_t>(1, kMaxPBytes / row_block)));
    }
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
    const size_t grows = static_cast<size_t>(L->group) * 128;
    L->p = off;
    off = align256(off + grows * L->nkb * 128 * 2);
    L->alpha = off;
    off = align256(off + static_cast<size_t>(L->nkb) * grows * 4);
    L->lsum = off;
    off = align256(off + grows * 4);
    L->flags = off;
    off = align256(off + static_cast<size_t>(L->group) * L->nkb * 4 * 4);
    const size_t cc = static_cast<size_t>(c) * c * 2;
    L->wqk = off;
    off = align256(off + cc);
    L->wov = off;
    off = align256(off + cc);
    L->bqk = off;
    off = align256(off + static_cast<size_t>(c) * 4);
    L->bov = off;
    off = align256(off + static_cast<size_t>(c) * 4);
    L->wT = off;  // the transposed Wq, Wk, Wv, one after another
    off = align256(off + 3 * cc);
    L->total = off;
    return VAE_OK;
}


// out[j][i] = in[i][j] for i < rows, j < cols (f16; rows, cols and both row
// strides multiples of 8, bases 16-byte aligned): 64 x 64 tiles through shared
// memory, 16-byte global accesses on both sides.
__global__ void __launch_bounds__(256)
    transpose_f16_kernel(const __half* __restrict__ in, int rows, int cols, long long ld_in, __half* __restrict__ out,
                         long long ld_out) {
    __shared__ __half2 tile[64][33];  // 64 rows of 64 halves (+1 word: the column reads spread over banks)
    pdl_wait();
    const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
    const int t = threadIdx.x;
    for (int pass = 0; pass < 2; ++pass) {
        const int r = (t >> 3) + 32 * pass, cc = (t & 7) * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r0 + r < rows && c0 + cc < cols)
            v = *reinterpret_cast<const uint4*>(in + static_cast<long long>(r0 + r) * ld_in + c0 + cc);
        tile[r][cc / 2 + 0] = *reinterpret_cast<__half2*>(&v.x);
        tile[r][cc / 2 + 1] = *reinterpret_cast<__half2*>(&v.y);
        tile[r][cc / 2 + 2] = *reinterpret_cast<__half2*>(&v.z);
        tile[r][cc / 2 + 3] = *reinterpret_cast<__half2*>(&v.w);
    }
    __syncthreads();
    for (int pass = 0; pass < 2; ++pass) {
        const int oc = (t >> 3) + 32 * pass, rr = (t & 7) * 8;  // input column, first of 8 input rows
        if (c0 + oc >= cols || r0 + rr >= rows) continue;
        __half h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __half2 w = tile[rr + i][oc / 2];
            h[i] = (oc & 1) ? __high2half(w) : __low2half(w);
        }
        *reinterpret_cast<uint4*>(out + static_cast<long long>(c0 + oc) * ld_out + r0 + rr) =
            *reinterpret_cast<const uint4*>(h);
    }
    pdl_launch_dependents();
}

// The folded biases: bqk = Wk^T bq (rows of Wk^T) and bov = Wo bv + bo, one
// warp per output; each lane sums a strided share of the c products, then the
// lanes combine by a butterfly (a fixed order).
__global__ void __launch_bounds__(256)
    fold_bias_kernel(const __half* __restrict__ wkT, const float* __restrict__ bq, const __half* __restrict__ wo,
                     const float* __restrict__ bv, const float* __restrict__ bo, int c, float* __restrict__ bqk,
                     float* __restrict__ bov) {
    pdl_wait();
    const int w = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (w < 2 * c) {
        const bool second = w >= c;
        const int i = second ? w - c : w;
        const __half* row = (second ? wo : wkT) + static_cast<long long>(i) * c;
        const float* vec = second ? bv : bq;
        float acc = 0.f;
        for (int r = lane; r < c; r += 32) acc = fmaf(__half2float(row[r]), vec[r], acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            if (second)
                bov[i] = acc + bo[i];
            else
                bqk[i] = acc;
        }
    }
    pdl_launch_dependents();
}

int transpose_run(const __half* in, int rows, int cols, long long ld_in, __half* out, long long ld_out,
                  cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>((cols + 63) / 64), static_cast<unsigned>((rows + 63) / 64));
    VAE_CUDA_CHECK(launch_kernel(transpose_f16_kernel, grid, dim3(256), 0, stream, in, rows, cols, ld_in, out, ld_out));
    return VAE_OK;
}

// The CTA-pair scores kernel runs unless VAE_ATTN_SCORES_PAIR=0 is set (tests and measurements).
bool attn_scores_pair_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("VAE_ATTN_SCORES_PAIR");
        return !(e != nullptr && e[0] == '0');
    }();
    return on;
}

// The CTA-pair PV kernel runs unless VAE_ATTN_PV_PAIR=0 is set (tests and measurements).
bool attn_pv_pair_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("VAE_ATTN_PV_PAIR");
        return !(e != nullptr && e[0] == '0');
    }();
    return on;
}

}  // namespace

// The folded form runs unless VAE_ATTN_FOLD=0 is set (tests and measurements).
bool attn_fold_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("VAE_ATTN_FOLD");
        return !(e != nullptr && e[0] == '0');
    }();
    return on;
}

// o = softmax(q k^T / sqrt(c)) v + b_v (f16 [m][c]) with the scratch of L in ws.
static int attn_core_run(const __half* q, const __half* k, const __half* vt, int m, int m_pad, int c, const float* bv,
                         __half* out, const AttnLayout& L, uint8_t* ws, cudaStream_t stream) {
    int rc = check_device();
    if (rc != VAE_OK) return rc;
    DevStatus* st = device_status_ptr();
    if (st == nullptr) return VAE_ERR_CUDA;
    const int grows = L.group * 128;
    const int kcols = L.nkb * 128;
    ScoreParams sp{};
    sp.m = m;
    sp.nkb = L.nkb;
    sp.nchunk_c = (c + 63) / 64;  // a partial last chunk reads TMA zero fill
    sp.kcols = kcols;
    sp.grows = grows;
    sp.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c)));
    sp.p = reinterpret_cast<__half*>(ws + L.p);
    sp.alpha = reinterpret_cast<float*>(ws + L.alpha);
    sp.lsum = reinterpret_cast<float*>(ws + L.lsum);
    sp.flags = reinterpret_cast<uint32_t*>(ws + L.flags);
    sp.status = st;
    sp.timeout_ns = wait_timeout_ns();
    PvParams pp{};
    pp.m = m;
    pp.c = c;
    pp.dv = L.dv;
    pp.ndv = L.ndv;
    pp.nkb = L.nkb;
    pp.grows = grows;
    pp.vboxes = L.dv > 256 ? 2 : 1;
    pp.vbox_rows = L.dv / pp.vboxes;
    pp.alpha = sp.alpha;
    pp.lsum = sp.lsum;
    pp.flags = sp.flags;
    pp.bv = bv;
    pp.out = out;
    pp.status = st;
    pp.timeout_ns = sp.timeout_ns;
    CUtensorMap mq{}, mk{}, mk2{}, mp{}, mv{};
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(c), static_cast<uint64_t>(m)};
        const uint64_t strides[1] = {static_cast<uint64_t>(c) * 2};
        const uint32_t box[2] = {64u, 128u};
        rc = encode_tiled(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != VAE_OK) return rc;
        const uint32_t kbox[2] = {64u, 256u};  // two key blocks per box
        rc = encode_tiled(&mk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, k, dims, strides, kbox, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != VAE_OK) return rc;
        const uint32_t kbox2[2] = {64u, 128u};  // the pair kernel: each CTA loads one key block of the pass
        rc = encode_tiled(&mk2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, k, dims, strides, kbox2,
                          CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != VAE_OK) return rc;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(kcols), static_cast<uint64_t>(grows)};
        const uint64_t strides[1] = {static_cast<uint64_t>(kcols) * 2};
        const uint32_t box[2] = {64u, 128u};
        rc = encode_tiled(&mp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, sp.p, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != VAE_OK) return rc;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(m_pad), static_cast<uint64_t>(c)};
        const uint64_t strides[1] = {static_cast<uint64_t>(m_pad) * 2};
        const uint32_t box[2] = {64u, static_cast<uint32_t>(pp.vbox_rows)};
        rc = encode_tiled(&mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, vt, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != VAE_OK) return rc;
    }
    // The PV kernel on CTA pairs: each CTA loads half of every V^T box (the
    // N rows of the pair MMA it supplies).
    CUtensorMap mv2{};
    {
        const int nsplit = L.dv > 256 ? 2 : 1;
        const uint64_t dims[2] = {static_cast<uint64_t>(m_pad), static_cast<uint64_t>(c)};
        const uint64_t strides[1] = {static_cast<uint64_t>(m_pad) * 2};
        const uint32_t box[2] = {64u, static_cast<uint32_t>(L.dv / nsplit / 2)};
        rc = encode_tiled(&mv2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, vt, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != VAE_OK) return rc;
    }
    const size_t smem = 1024 + kStages * kStageBytes + 256;
    const size_t smem_pair = 1024 + kPvPairStages * kPvPairStageBytes + 256;
    const size_t smem_sc_pair = 1024 + kScPairStages * kScPairStageBytes + 256;
    static CtxOnce attr_set;
    int dev = 0;
    VAE_CUDA_CHECK(cudaGetDevice(&dev));
    if (!attr_set.done(dev)) {
        VAE_CUDA_CHECK(cudaFuncSetAttribute(attn_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(smem)));
        VAE_CUDA_CHECK(cudaFuncSetAttribute(attn_pv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(smem)));
        VAE_CUDA_CHECK(cudaFuncSetAttribute(attn_pv_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(smem_pair)));
        VAE_CUDA_CHECK(cudaFuncSetAttribute(attn_scores_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(smem_sc_pair)));
        attr_set.mark(dev);
    }
    for (int t0 = 0; t0 < L.qtiles; t0 += L.group) {
        const int nt = std::min(L.group, L.qtiles - t0);
        sp.q_tile0 = t0;
        sp.ntiles = nt;
        pp.q_tile0 = t0;
        pp.ntiles = nt;
        if (nt >= 2 && attn_scores_pair_enabled())
            VAE_CUDA_CHECK(launch_kernel(attn_scores_pair_kernel, dim3(static_cast<unsigned>(2 * ((nt + 1) / 2))),
                                         dim3(kScThreads), smem_sc_pair, stream, mq, mk2, sp));
        else
            VAE_CUDA_CHECK(launch_kernel(attn_scores_kernel, dim3(static_cast<unsigned>(nt)), dim3(kScThreads), smem,
                                         stream, mq, mk, sp));
        if (nt >= 2 && attn_pv_pair_enabled())
            VAE_CUDA_CHECK(launch_kernel(attn_pv_pair_kernel, dim3(static_cast<unsigned>(2 * ((nt + 1) / 2) * L.ndv)),
                                         dim3(kThreads), smem_pair, stream, mp, mv2, pp));
        else
            VAE_CUDA_CHECK(launch_kernel(attn_pv_kernel, dim3(static_cast<unsigned>(nt * L.ndv)), dim3(kThreads),
                                         smem, stream, mp, mv, pp));
    }
    return VAE_OK;
}

int attn_workspace_bytes(int m, int c, int groups, int norm_kind, size_t* bytes) {
    AttnLayout L;
    int rc = attn_layout(m, c, groups, norm_kind, &L);
    if (rc != VAE_OK) return rc;
    *bytes = L.total;
    return VAE_OK;
}

namespace {

// Checks the common arguments, runs the norm into xn and zeroes its pad rows.
struct AttnBufs {
    AttnLayout L;
    uint8_t* w8;
    __half *xn, *q, *k, *vt, *o;
};

int attn_begin(float* x, int m, int c, int norm_kind, int groups, float eps, const float* gamma, const float* beta,
               void* ws, size_t ws_bytes, cudaStream_t stream, AttnBufs* B) {
    if (x == nullptr || gamma == nullptr || ws == nullptr)
        return set_error(VAE_ERR_ARG, "mid_attention: a required pointer is NULL");
    if (norm_kind != VAE_NORM_GROUP && norm_kind != VAE_NORM_RMS)
        return set_error(VAE_ERR_ARG, "mid_attention: norm_kind %d", norm_kind);
    if (norm_kind == VAE_NORM_GROUP && beta == nullptr)
        return set_error(VAE_ERR_ARG, "mid_attention: GroupNorm needs beta");
    AttnLayout& L = B->L;
    int rc = attn_layout(m, c, groups, norm_kind, &L);
    if (rc != VAE_OK) return rc;
    if (ws_bytes < L.total)
        return set_error(VAE_ERR_NOMEM, "mid_attention: workspace %zu < %zu bytes", ws_bytes, L.total);
    if (!aligned16(ws) || !aligned16(x)) return set_error(VAE_ERR_ALIGN, "mid_attention: x/workspace alignment");
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    B->w8 = w8;
    B->xn = reinterpret_cast<__half*>(w8 + L.xn);
    B->q = reinterpret_cast<__half*>(w8 + L.q);
    B->k = reinterpret_cast<__half*>(w8 + L.k);
    B->vt = reinterpret_cast<__half*>(w8 + L.vt);
    B->o = reinterpret_cast<__half*>(w8 + L.o);
    if (norm_kind == VAE_NORM_GROUP)
        rc = gn_run(x, 1, m, c, groups, eps, nullptr, gamma, beta, 0, 1.0f, B->xn, w8 + L.gn, L.total - L.gn, stream);
    else
        rc = rms_run(x, m, c, nullptr, gamma, 0, 1.0f, B->xn, stream);
    if (rc != VAE_OK) return rc;
    if (L.m_pad > m)
        VAE_CUDA_CHECK(cudaMemsetAsync(B->xn + static_cast<size_t>(m) * c, 0,
                                       static_cast<size_t>(L.m_pad - m) * c * 2, stream));
    return VAE_OK;
}

ConvArgs gemm_args(const void* x, int rows, int cin, const void* w, int cout, const float* bias, void* y, bool f16) {
    ConvArgs a{};
    a.taps = 1;
    a.n = 1;
    a.h_in = 1;
    a.w_in = rows;
    a.cin = cin;
    a.x = x;
    a.w = w;
    a.cout = cout;
    a.bias = bias;
    a.y = y;
    a.out_f16 = f16;
    return a;
}

// The folded attention on the norm's rows in B (see attn_fold_run).
int attn_folded_core(float* x, int m, int c, const __half* wqk, const float* bqk, const __half* wov, const float* bov,
                     const AttnBufs& B, cudaStream_t stream) {
    int rc;
    // q' = xn M^T + Wk^T bq (f16)
    if ((rc = conv_run(gemm_args(B.xn, m, c, wqk, c, bqk, B.q, true), stream)) != VAE_OK) return rc;
    // xn^T [c][m_pad] (the zeroed pad rows included): the P.V operand
    if ((rc = transpose_run(B.xn, B.L.m_pad, c, c, B.vt, B.L.m_pad, stream)) != VAE_OK) return rc;
    if ((rc = attn_core_run(B.q, B.xn, B.vt, m, B.L.m_pad, c, nullptr, B.o, B.L, B.w8, stream)) != VAE_OK) return rc;
    // x += xbar (Wo Wv)^T + (Wo bv + bo)
    ConvArgs pr = gemm_args(B.o, m, c, wov, c, bov, x, false);
    pr.residual = x;
    return conv_run(pr, stream);
}

}  // namespace

// The folded weights. With q_i = Wq n_i + bq and k_j = Wk n_j + bk, the score
// q_i . k_j = (Wk^T q_i) . n_j + q_i . bk, and the last term is the same for
// every key j of row i, so the softmax drops it: the scores are q'_i . n_j with
// q' = n M^T + Wk^T bq, M = Wk^T Wq. Each row of the softmax sums to one, so
// o_i = Wv (sum_j p_ij n_j / l_i) + bv, and the block's output
// Wo o_i + bo = (Wo Wv) nbar_i + (Wo bv + bo), nbar being the softmax average
// of the normalised rows themselves. Two c x c weight products replace the key
// and value projections of all m tokens; keys and values are the normalised
// rows (xn, and xn^T for the P.V operand). wqk, wov f16 [c][c]; bqk, bov f32
// [c]; scratch 3 c^2 f16 (the transposed Wq, Wk, Wv). All 16-byte aligned.
int attn_fold_run(int c, const void* wq, const float* bq, const void* wk, const void* wv, const float* bv,
                  const void* wo, const float* bo, __half* wqk, __half* wov, float* bqk, float* bov, __half* scratch,
                  cudaStream_t stream) {
    if (wq == nullptr || wk == nullptr || wv == nullptr || wo == nullptr || bq == nullptr || bv == nullptr ||
        bo == nullptr || wqk == nullptr || wov == nullptr || bqk == nullptr || bov == nullptr || scratch == nullptr)
        return set_error(VAE_ERR_ARG, "mid_attention: a required pointer is NULL");
    if (c < 16 || c % 16 != 0 || c > 2048) return set_error(VAE_ERR_SHAPE, "mid_attention: c=%d", c);
    if (!aligned16(wq) || !aligned16(wk) || !aligned16(wv) || !aligned16(wo) || !aligned16(wqk) || !aligned16(wov) ||
        !aligned16(scratch))
        return set_error(VAE_ERR_ALIGN, "mid_attention: the weights must be 16-byte aligned");
    const size_t cc = static_cast<size_t>(c) * c;
    __half* wqT = scratch;
    __half* wkT = scratch + cc;
    __half* wvT = scratch + 2 * cc;
    int rc;
    if ((rc = transpose_run(static_cast<const __half*>(wq), c, c, c, wqT, c, stream)) != VAE_OK) return rc;
    if ((rc = transpose_run(static_cast<const __half*>(wk), c, c, c, wkT, c, stream)) != VAE_OK) return rc;
    if ((rc = transpose_run(static_cast<const __half*>(wv), c, c, c, wvT, c, stream)) != VAE_OK) return rc;
    // M[a][b] = sum_r Wk[r][a] Wq[r][b]: rows of Wk^T against rows of Wq^T
    if ((rc = conv_run(gemm_args(wkT, c, c, wqT, c, nullptr, wqk, true), stream)) != VAE_OK) return rc;
    // (Wo Wv)[a][b] = sum_r Wo[a][r] Wv[r][b]: rows of Wo against rows of Wv^T
    if ((rc = conv_run(gemm_args(wo, c, c, wvT, c, nullptr, wov, true), stream)) != VAE_OK) return rc;
    VAE_CUDA_CHECK(launch_kernel(fold_bias_kernel, dim3(static_cast<unsigned>((2 * c * 32 + 255) / 256)), dim3(256), 0,
                                 stream, static_cast<const __half*>(wkT), bq, static_cast<const __half*>(wo), bv, bo, c,
                                 bqk, bov));
    return VAE_OK;
}

int attn_run_folded(float* x, int m, int c, int norm_kind, int groups, float eps, const float* gamma,
                    const float* beta, const __half* wqk, const float* bqk, const __half* wov, const float* bov,
                    void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (wqk == nullptr || bqk == nullptr || wov == nullptr || bov == nullptr)
        return set_error(VAE_ERR_ARG, "mid_attention: a required pointer is NULL");
    if (!aligned16(wqk) || !aligned16(wov))
        return set_error(VAE_ERR_ALIGN, "mid_attention: the weights must be 16-byte aligned");
    AttnBufs B;
    int rc = attn_begin(x, m, c, norm_kind, groups, eps, gamma, beta, ws, ws_bytes, stream, &B);
    if (rc != VAE_OK) return rc;
    return attn_folded_core(x, m, c, wqk, bqk, wov, bov, B, stream);
}

int attn_run(float* x, int m, int c, int norm_kind, int groups, float eps, const float* gamma, const float* beta,
             const void* wq, const float* bq, const void* wk, const float* bk, const void* wv, const float* bv,
             const void* wo, const float* bo, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (wq == nullptr || wk == nullptr || wv == nullptr || wo == nullptr || bq == nullptr || bk == nullptr ||
        bv == nullptr || bo == nullptr)
        return set_error(VAE_ERR_ARG, "mid_attention: a required pointer is NULL");
    if (!aligned16(wq) || !aligned16(wk) || !aligned16(wv) || !aligned16(wo))
        return set_error(VAE_ERR_ALIGN, "mid_attention: the weights must be 16-byte aligned");
    {
        AttnLayout L;  // shape and workspace checks before anything is launched
        int rc = attn_layout(m, c, groups, norm_kind, &L);
        if (rc != VAE_OK) return rc;
        if (ws != nullptr && ws_bytes < L.total)
            return set_error(VAE_ERR_NOMEM, "mid_attention: workspace %zu < %zu bytes", ws_bytes, L.total);
    }
    AttnBufs B;
    int rc = attn_begin(x, m, c, norm_kind, groups, eps, gamma, beta, ws, ws_bytes, stream, &B);
    if (rc != VAE_OK) return rc;
    const AttnLayout& L = B.L;
    if (attn_fold_enabled()) {
        __half* wqk = reinterpret_cast<__half*>(B.w8 + L.wqk);
        __half* wov = reinterpret_cast<__half*>(B.w8 + L.wov);
        float* bqk = reinterpret_cast<float*>(B.w8 + L.bqk);
        float* bov = reinterpret_cast<float*>(B.w8 + L.bov);
        if ((rc = attn_fold_run(c, wq, bq, wk, wv, bv, wo, bo, wqk, wov, bqk, bov,
                                reinterpret_cast<__half*>(B.w8 + L.wT), stream)) != VAE_OK)
            return rc;
        return attn_folded_core(x, m, c, wqk, bqk, wov, bov, B, stream);
    }
    // The projections as written: q, k = xn W^T + b (f16); v^T [c][m_pad] = W_v xn^T
    // (no bias: added after P.V); x += o W_o^T + b_o.
    if ((rc = conv_run(gemm_args(B.xn, m, c, wq, c, bq, B.q, true), stream)) != VAE_OK) return rc;
    if ((rc = conv_run(gemm_args(B.xn, m, c, wk, c, bk, B.k, true), stream)) != VAE_OK) return rc;
    if ((rc = conv_run(gemm_args(wv, c, c, B.xn, L.m_pad, nullptr, B.vt, true), stream)) != VAE_OK) return rc;
    if ((rc = attn_core_run(B.q, B.k, B.vt, m, L.m_pad, c, bv, B.o, L, B.w8, stream)) != VAE_OK) return rc;
    ConvArgs pr = gemm_args(B.o, m, c, wo, c, bo, x, false);
    pr.residual = x;
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

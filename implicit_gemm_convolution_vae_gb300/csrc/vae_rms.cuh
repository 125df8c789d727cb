// RMS_norm arithmetic shared by the standalone RMS_norm kernel and the conv
// epilogue that fuses it ("qi21_vae.rs" qv_rmsn: v * sqrt(C) / max(||v||, 1e-12)
// * gamma). Both follow one fixed evaluation order with no FMA contraction, so
// a fused and an unfused decode produce the same bits (banded decodes rely on
// per-pixel results that do not depend on which kernel produced them).
//
// Order: the C channels form C/4 float4 columns; "lane" l of G lanes sums its
// columns l, l+G, l+2G, ... in that order, each column adding
// (((x*x + y*y) + z*z) + w*w); the G partial sums are then combined by a
// butterfly (s[l] += s[l + off] for off = G/2 .. 1) and s[0] is the sum.
#pragma once

#include "vae_common.cuh"

namespace vae {

// Lanes per pixel of the standalone kernel for `c` channels when the pixel
// fits in registers (c/4 <= 9 * 32); the fused epilogue reproduces the same G.
__host__ __device__ constexpr int rms_lanes(int c) {
    return (c / 4) <= 36 ? 4 : (c / 4) <= 72 ? 8 : (c / 4) <= 144 ? 16 : 32;
}

__device__ __forceinline__ float rms_acc4(float acc, float x, float y, float z, float w) {
    float t = __fadd_rn(__fmul_rn(x, x), __fmul_rn(y, y));
    t = __fadd_rn(t, __fmul_rn(z, z));
    t = __fadd_rn(t, __fmul_rn(w, w));
    return __fadd_rn(acc, t);
}

__device__ __forceinline__ float rms_inv(float ss, int c) {
    return __fdiv_rn(__fsqrt_rn(static_cast<float>(c)), fmaxf(__fsqrt_rn(ss), 1e-12f));
}

__device__ __forceinline__ float rms_apply(float v, float inv, float g) { return __fmul_rn(__fmul_rn(v, inv), g); }

}  // namespace vae

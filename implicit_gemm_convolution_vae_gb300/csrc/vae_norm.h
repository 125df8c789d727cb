// Internal interface of the bandwidth-bound kernels (norms, casts, layout),
// shared by the public entry points, the mid attention and the decoder.
#pragma once

#include "vae_common.cuh"

namespace vae {

struct GnPlan {
    int nchunks, chunk_rows, rpar;
    size_t part_floats, stats_floats, bytes;
};

int gn_plan(int n, int hw, int c, int groups, GnPlan* plan);
int gn_run(const float* x, int n, int hw, int c, int groups, float eps, const float* bias, const float* gamma,
           const float* beta, int silu, float out_scale, void* y, void* ws, size_t ws_bytes,
           cudaStream_t stream);
// (count, mean, M2) records [n][nchunks][groups] (float4) -> (mean, 1/sqrt(var+eps)) [n][groups][2].
int gn_stats_from_records(const void* rec, int n, int nchunks, int groups, float eps, float* stats,
                          cudaStream_t stream);
int gn_apply_run(const float* x, int n, int hw, int c, int groups, const float* stats, const float* gamma,
                 const float* beta, int silu, float out_scale, void* y, cudaStream_t stream);
int rms_run(const float* x, long long m, int c, const float* bias, const float* gamma, int silu,
            float out_scale, void* y, cudaStream_t stream);
int cast_run(const float* x, size_t count, int c, const float* bias, float scale, void* y, cudaStream_t stream);
int latent_run(const float* z, int c, long long hw, float mul, float add, void* y, cudaStream_t stream);

}  // namespace vae

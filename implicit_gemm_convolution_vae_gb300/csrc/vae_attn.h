// Internal interface of the mid attention, used by the decoder driver.
#pragma once

#include "vae_common.cuh"

namespace vae {

int attn_workspace_bytes(int m, int c, int groups, int norm_kind, size_t* bytes);
int attn_run(float* x, int m, int c, int norm_kind, int groups, float eps, const float* gamma, const float* beta,
             const void* wq, const float* bq, const void* wk, const float* bk, const void* wv, const float* bv,
             const void* wo, const float* bo, void* ws, size_t ws_bytes, cudaStream_t stream);
// The folded weights (M = Wk^T Wq, Wo Wv, Wk^T bq, Wo bv + bo) formed once,
// for callers whose weights stay fixed; scratch holds 3 c^2 f16.
int attn_fold_run(int c, const void* wq, const float* bq, const void* wk, const void* wv, const float* bv,
                  const void* wo, const float* bo, __half* wqk, __half* wov, float* bqk, float* bov, __half* scratch,
                  cudaStream_t stream);
// The attention on weights attn_fold_run formed (same workspace as attn_run).
int attn_run_folded(float* x, int m, int c, int norm_kind, int groups, float eps, const float* gamma,
                    const float* beta, const __half* wqk, const float* bqk, const __half* wov, const float* bov,
                    void* ws, size_t ws_bytes, cudaStream_t stream);
bool attn_fold_enabled();

}  // namespace vae

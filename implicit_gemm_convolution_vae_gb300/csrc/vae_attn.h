// Internal interface of the mid attention, used by the decoder driver.
#pragma once

#include "vae_common.cuh"

namespace vae {

int attn_workspace_bytes(int m, int c, int groups, int norm_kind, size_t* bytes);
int attn_run(float* x, int m, int c, int norm_kind, int groups, float eps, const float* gamma, const float* beta,
             const void* wq, const float* bq, const void* wk, const float* bk, const void* wv, const float* bv,
             const void* wo, const float* bo, void* ws, size_t ws_bytes, cudaStream_t stream);

}  // namespace vae

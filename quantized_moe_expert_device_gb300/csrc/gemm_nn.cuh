// Declarations of the transpose=False gather (gqmm_gather_qmm_nn), shared by api.cu and gemm_nn.cu.
#pragma once

#include "gqmm_internal.cuh"

namespace gqmm {

// y[i, :] = x[i / x_div, :] . deq(W[idx[i]]) for n routed rows; W [E, K, N] quantized along N in
// groups of group_size; rows whose index is >= E are zero.
cudaError_t launch_gemm_nn(const __nv_bfloat16* x, const uint8_t* wq, const __nv_bfloat16* scales,
                           const __nv_bfloat16* biases, const uint32_t* idx, int64_t n, int K, int N, int E,
                           int group_size, int x_div, __nv_bfloat16* y, cudaStream_t s);

}  // namespace gqmm

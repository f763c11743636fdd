// CUDA-core cross-check of the gather matmul: one thread per output element, float32
// accumulation over H with the weight dequantized in float32 (scale * q + bias).  It shares
// nothing with the tensor-core path except the data format, and no entry point of the fast
// path calls it; tests use it to separate data-handling faults from MMA-pipeline faults.
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

__global__ void __launch_bounds__(128) gemm_simt_kernel(const __nv_bfloat16* __restrict__ x,
                                                        const uint8_t* __restrict__ wq,
                                                        const __nv_bfloat16* __restrict__ scales,
                                                        const __nv_bfloat16* __restrict__ biases,
                                                        const uint32_t* __restrict__ idx, int H, int F,
                                                        int E, int gs, int x_div, __nv_bfloat16* __restrict__ y) {
  const int64_t i = blockIdx.x;
  const int f = blockIdx.y * blockDim.x + threadIdx.x;
  if (f >= F) return;
  const uint32_t e = idx ? __ldg(idx + i) : 0u;
  if (e >= (uint32_t)E) {
    y[i * F + f] = __float2bfloat16_rn(0.0f);
    return;
  }
  const int G = H / gs;
  const int64_t wr = (int64_t)e * F + f;
  const uint8_t* wrow = wq + wr * (H / 2);
  const __nv_bfloat16* xr = x + (i / x_div) * H;
  float acc = 0.0f;
  for (int g = 0; g < G; ++g) {
    const float s = __bfloat162float(scales[wr * G + g]);
    const float b = __bfloat162float(biases[wr * G + g]);
    for (int k = 0; k < gs; k += 2) {
      const uint8_t byte = wrow[(g * gs + k) / 2];
      const float w0 = fmaf(s, (float)(byte & 15), b);
      const float w1 = fmaf(s, (float)(byte >> 4), b);
      acc = fmaf(__bfloat162float(xr[g * gs + k]), w0, acc);
      acc = fmaf(__bfloat162float(xr[g * gs + k + 1]), w1, acc);
    }
  }
  y[i * F + f] = __float2bfloat16_rn(acc);
}

}  // namespace

cudaError_t launch_gemm_simt(const __nv_bfloat16* x, const uint8_t* wq, const __nv_bfloat16* scales,
                             const __nv_bfloat16* biases, const uint32_t* idx, int64_t n, int H, int F,
                             int E, int group_size, int x_div, __nv_bfloat16* y, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  dim3 grid((unsigned)n, (unsigned)((F + 127) / 128));
  gemm_simt_kernel<<<grid, 128, 0, s>>>(x, wq, scales, biases, idx, H, F, E, group_size, x_div, y);
  return cudaGetLastError();
}

}  // namespace gqmm

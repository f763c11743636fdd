// gather_qmm with transpose=False: y[i, :] = x[i, :] . deq(W[idx[i]]), where W[e] is [K, N] and
// quantized along N, the layout mx.quantize gives an [E, K, N] weight (mlx PR #4023 "Pick BM
// from rows per expert in gather_qmm_rhs_nax", the author's follow-up: the transpose=false
// shape, used by the backward pass and fine-tuning, has no fast path there).
//
// CUDA cores, one routed row per block row: a thread owns eight adjacent output columns (one
// 32-bit code word per k, so a warp reads 128 contiguous bytes of a weight row), a block 1024
// columns.  The row's x is staged in shared memory 1024 values at a time; each k costs a
// thread one code word, one scale and one bias (its eight columns share a group, since groups
// are at least 32 wide).  With s q + b = 16 s (1 + q/16) - 16 s + b, where 1 + q/16 is exact in
// float32 with the code in the mantissa (0x3F800000 | q << 19), a column costs a shift, a
// masked OR and one FMA, and the k's bias term joins one accumulator shared by the eight:
//     y[c] = sum_k (16 x_k s_k) v_kc + sum_k x_k (b_k - 16 s_k).
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

constexpr int kNnThreads = 128;
constexpr int kNnColsPerThread = 8;
constexpr int kNnChunk = 1024;  // x values staged per pass

__global__ void __launch_bounds__(kNnThreads) gemm_nn_kernel(const __nv_bfloat16* __restrict__ x,
                                                             const uint8_t* __restrict__ wq,
                                                             const __nv_bfloat16* __restrict__ scales,
                                                             const __nv_bfloat16* __restrict__ biases,
                                                             const uint32_t* __restrict__ idx, int K, int N, int E,
                                                             int gs, int x_div, __nv_bfloat16* __restrict__ y) {
  __shared__ float xs[kNnChunk];
  const int64_t i = blockIdx.x;                                  // routed row
  const int w = blockIdx.y * kNnThreads + threadIdx.x;           // code word: columns 8 w .. 8 w + 7
  const int NW = N / kNnColsPerThread;
  const uint32_t e = idx ? __ldg(idx + i) : 0u;
  if (e >= (uint32_t)E) {  // uniform over the block: its row has no expert
    if (w < NW) *reinterpret_cast<uint4*>(y + i * N + (int64_t)w * kNnColsPerThread) = make_uint4(0, 0, 0, 0);
    return;
  }
  const int G = N / gs;
  const int g = (w * kNnColsPerThread) / gs;
  const uint32_t* wrow = reinterpret_cast<const uint32_t*>(wq + (int64_t)e * K * (N / 2)) + w;  // word w of row 0
  const __nv_bfloat16* srow = scales + (int64_t)e * K * G + g;
  const __nv_bfloat16* brow = biases + (int64_t)e * K * G + g;
  const __nv_bfloat16* xrow = x + (i / x_div) * K;
  float acc[kNnColsPerThread];
#pragma unroll
  for (int m = 0; m < kNnColsPerThread; ++m) acc[m] = 0.f;
  float corr = 0.f;  // sum_k x_k (b_k - 16 s_k), shared by the thread's columns
  for (int k0 = 0; k0 < K; k0 += kNnChunk) {
    const int kn = K - k0 < kNnChunk ? K - k0 : kNnChunk;
    __syncthreads();  // the previous chunk is consumed
    for (int t = threadIdx.x; t < kn; t += kNnThreads) xs[t] = __bfloat162float(xrow[k0 + t]);
    __syncthreads();
    if (w < NW) {
      for (int kk = 0; kk < kn; ++kk) {
        const int64_t k = k0 + kk;
        const uint32_t word = __ldg(wrow + k * NW);
        const float s = __bfloat162float(srow[k * G]);
        const float b = __bfloat162float(brow[k * G]);
        const float xk = xs[kk];
        const float a16 = (xk * s) * 16.f;  // exact scaling by 16
        corr = fmaf(xk, b, corr) - a16;
#pragma unroll
        for (int m = 0; m < kNnColsPerThread; ++m) {
          // nibble m to mantissa bits 19..22: 1 + q/16
          const uint32_t bits = 4 * m <= 19 ? (word << (19 - 4 * m)) : (word >> (4 * m - 19));
          acc[m] = fmaf(a16, __uint_as_float((bits & 0x00780000u) | 0x3F800000u), acc[m]);
        }
      }
    }
  }
  if (w < NW) {
    uint32_t o[4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
      o[m] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * m] + corr)) |
             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * m + 1] + corr)) << 16);
    *reinterpret_cast<uint4*>(y + i * N + (int64_t)w * kNnColsPerThread) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_gemm_nn(const __nv_bfloat16* x, const uint8_t* wq, const __nv_bfloat16* scales,
                           const __nv_bfloat16* biases, const uint32_t* idx, int64_t n, int K, int N, int E,
                           int group_size, int x_div, __nv_bfloat16* y, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int NW = N / kNnColsPerThread;
  dim3 grid((unsigned)n, (unsigned)((NW + kNnThreads - 1) / kNnThreads));
  gemm_nn_kernel<<<grid, kNnThreads, 0, s>>>(x, wq, scales, biases, idx, K, N, E, group_size, x_div, y);
  return cudaGetLastError();
}

}  // namespace gqmm

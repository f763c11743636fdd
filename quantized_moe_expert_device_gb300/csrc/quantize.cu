// Affine 4-bit group quantization (mx.quantize(w, group_size=64, bits=4), as called in the
// mlx issue "[CUDA] gather_qmm ~24x slower than equal-FLOPs quantized_matmul on GB10",
// section "Kernel microbenchmark").  Format: see include/gqmm.h.
//
// One thread per group of 64 weights: eight 16-byte loads, float32 min/max, IEEE float32
// divide for the scale (no fast math in this file), round-half-to-even codes computed from
// the stored bfloat16 scale and bias, two 16-byte stores of packed nibbles.  A warp covers
// 32 consecutive groups = 4 KB of contiguous input, so loads and stores are coalesced.
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__global__ void __launch_bounds__(256) quantize_kernel(const __nv_bfloat16* __restrict__ w,
                                                       int64_t n_groups, int64_t G,
                                                       uint8_t* __restrict__ wq,
                                                       __nv_bfloat16* __restrict__ scales,
                                                       __nv_bfloat16* __restrict__ biases) {
  const int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gi >= n_groups) return;
  // Groups are contiguous in memory: group gi = row gi / G, group gi % G, and row r of H
  // elements starts at r * H = r * G * 64, so group gi starts at element gi * 64.
  const uint4* src = reinterpret_cast<const uint4*>(w + gi * 64);
  float v[64];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 u = __ldg(src + c);
    v[c * 8 + 0] = bf16_lo(u.x);
    v[c * 8 + 1] = bf16_hi(u.x);
    v[c * 8 + 2] = bf16_lo(u.y);
    v[c * 8 + 3] = bf16_hi(u.y);
    v[c * 8 + 4] = bf16_lo(u.z);
    v[c * 8 + 5] = bf16_hi(u.z);
    v[c * 8 + 6] = bf16_lo(u.w);
    v[c * 8 + 7] = bf16_hi(u.w);
  }
  float mn = v[0], mx = v[0];
#pragma unroll
  for (int k = 1; k < 64; ++k) {
    mn = v[k] < mn ? v[k] : mn;
    mx = v[k] > mx ? v[k] : mx;
  }
  const float scale32 = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
  const __nv_bfloat16 s_b = __float2bfloat16_rn(scale32);
  const __nv_bfloat16 b_b = __float2bfloat16_rn(mn);  // exact: mn is a bfloat16 value
  const float s = __bfloat162float(s_b);
  const float b = __bfloat162float(b_b);
  scales[gi] = s_b;
  biases[gi] = b_b;

  uint32_t packed[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      int q = 0;
      if (s != 0.0f) {
        q = __float2int_rn(__fdiv_rn(__fsub_rn(v[j * 8 + k], b), s));
        q = q < 0 ? 0 : (q > 15 ? 15 : q);
      }
      word |= (uint32_t)q << (4 * k);  // element 2m in the low nibble of byte m
    }
    packed[j] = word;
  }
  uint4* dst = reinterpret_cast<uint4*>(wq + gi * 32);
  dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  (void)G;
}

}  // namespace

cudaError_t launch_quantize(const __nv_bfloat16* w, int64_t rows, int64_t H, uint8_t* wq,
                            __nv_bfloat16* scales, __nv_bfloat16* biases, cudaStream_t s) {
  const int64_t G = H / 64;
  const int64_t n_groups = rows * G;
  if (n_groups == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (n_groups + threads - 1) / threads;
  quantize_kernel<<<(unsigned)blocks, threads, 0, s>>>(w, n_groups, G, wq, scales, biases);
  return cudaGetLastError();
}

}  // namespace gqmm

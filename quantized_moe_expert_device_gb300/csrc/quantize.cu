// Affine 4-bit group quantization (mx.quantize(w, group_size=64, bits=4), as called in the
// mlx issue "[CUDA] gather_qmm ~24x slower than equal-FLOPs quantized_matmul on GB10",
// section "Kernel microbenchmark"; also 32- and 128-wide groups).  Format: see include/gqmm.h.
//
// One thread per group of GS weights: GS/8 16-byte loads, float32 min/max, IEEE float32
// divide for the scale (no fast math in this file), round-half-to-even codes computed from
// the stored bfloat16 scale and bias, GS/32 16-byte stores of packed nibbles.  A warp covers
// 32 consecutive groups of contiguous input, so loads and stores are coalesced.
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

template <int GS>
__global__ void __launch_bounds__(256) quantize_kernel(const __nv_bfloat16* __restrict__ w, int64_t n_groups,
                                                       uint8_t* __restrict__ wq, __nv_bfloat16* __restrict__ scales,
                                                       __nv_bfloat16* __restrict__ biases) {
  const int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gi >= n_groups) return;
  // Groups are contiguous in memory: group gi = row gi / G, group gi % G, and row r of H
  // elements starts at r * H = r * G * GS, so group gi starts at element gi * GS.
  const uint4* src = reinterpret_cast<const uint4*>(w + gi * GS);
  float v[GS];
#pragma unroll
  for (int c = 0; c < GS / 8; ++c) {
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
  for (int k = 1; k < GS; ++k) {
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

  uint4* dst = reinterpret_cast<uint4*>(wq + gi * (GS / 2));
#pragma unroll
  for (int c = 0; c < GS / 32; ++c) {  // 32 codes = one 16-byte store
    uint32_t packed[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t word = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        int q = 0;
        if (s != 0.0f) {
          q = __float2int_rn(__fdiv_rn(__fsub_rn(v[c * 32 + j * 8 + k], b), s));
          q = q < 0 ? 0 : (q > 15 ? 15 : q);
        }
        word |= (uint32_t)q << (4 * k);  // element 2m in the low nibble of byte m
      }
      packed[j] = word;
    }
    dst[c] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

}  // namespace

cudaError_t launch_quantize(const __nv_bfloat16* w, int64_t rows, int64_t H, int group_size, uint8_t* wq,
                            __nv_bfloat16* scales, __nv_bfloat16* biases, cudaStream_t s) {
  const int64_t n_groups = rows * (H / group_size);
  if (n_groups == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = (unsigned)((n_groups + threads - 1) / threads);
  switch (group_size) {
    case 32: quantize_kernel<32><<<blocks, threads, 0, s>>>(w, n_groups, wq, scales, biases); break;
    case 64: quantize_kernel<64><<<blocks, threads, 0, s>>>(w, n_groups, wq, scales, biases); break;
    case 128: quantize_kernel<128><<<blocks, threads, 0, s>>>(w, n_groups, wq, scales, biases); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gqmm

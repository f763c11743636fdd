// Affine 4-bit group quantization (mx.quantize(w, group_size=64, bits=4), as called in the
// mlx issue "[CUDA] gather_qmm ~24x slower than equal-FLOPs quantized_matmul on GB10",
// section "Kernel microbenchmark"; also 32- and 128-wide groups).  Format: see include/gqmm.h.
//
// One thread per group of GS weights: GS/8 16-byte loads, float32 min/max, IEEE float32
// divide for the scale (no fast math in this file), round-half-to-even codes computed from
// the stored bfloat16 scale and bias, GS/32 16-byte stores of packed nibbles.  A warp covers
// 32 consecutive groups of contiguous input, so loads and stores are coalesced.
#include "formats.cuh"
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

template <int GS, int BITS>
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
  constexpr int LEVELS = (1 << BITS) - 1;
  const float scale32 = __fdiv_rn(__fsub_rn(mx, mn), (float)LEVELS);
  const __nv_bfloat16 s_b = __float2bfloat16_rn(scale32);
  const __nv_bfloat16 b_b = __float2bfloat16_rn(mn);  // exact: mn is a bfloat16 value
  const float s = __bfloat162float(s_b);
  const float b = __bfloat162float(b_b);
  scales[gi] = s_b;
  biases[gi] = b_b;

  // The group's codes as a little-endian bit stream (element k in bits [k BITS, (k + 1) BITS);
  // for 4-bit codes, element 2m in the low nibble of byte m): GS * BITS / 32 whole words.
  constexpr int NWORDS = GS * BITS / 32;
  uint32_t words[NWORDS];
  uint64_t acc = 0;
  int nacc = 0, wi = 0;
#pragma unroll
  for (int k = 0; k < GS; ++k) {
    int q = 0;
    if (s != 0.0f) {
      q = __float2int_rn(__fdiv_rn(__fsub_rn(v[k], b), s));
      q = q < 0 ? 0 : (q > LEVELS ? LEVELS : q);
    }
    acc |= (uint64_t)q << nacc;
    nacc += BITS;
    if (nacc >= 32) {
      words[wi++] = (uint32_t)acc;
      acc >>= 32;
      nacc -= 32;
    }
  }
  if (NWORDS % 4 == 0) {  // the group's codes start on a 16-byte boundary
    uint4* dst = reinterpret_cast<uint4*>(wq + gi * (GS * BITS / 8));
#pragma unroll
    for (int c = 0; c < NWORDS / 4; ++c)
      dst[c] = make_uint4(words[4 * c], words[4 * c + 1], words[4 * c + 2], words[4 * c + 3]);
  } else {
    uint32_t* dst = reinterpret_cast<uint32_t*>(wq + gi * (GS * BITS / 8));
#pragma unroll
    for (int c = 0; c < NWORDS; ++c) dst[c] = words[c];
  }
}

// ---- block-scaled floating-point formats (formats.cuh; the steps of the oracle's reading of
//      OCP MX v1.0 and NVFP4, every operation an IEEE float32 one) ----

__device__ __forceinline__ float pow2f(int k) { return __int_as_float((k + 127) << 23); }  // k in [-126, 127]

// The value nearest to v (ties to the even significand) of a float type with MAN mantissa bits
// and smallest normal exponent EMIN, saturating at +-MAXV; exact in float32 for these types.
template <int MAN, int EMIN>
__device__ __forceinline__ float round_small(float v, float maxv) {
  const float a = fabsf(v);
  if (a == 0.0f) return v;
  if (a >= maxv) return copysignf(maxv, v);
  int e = ilogbf(a);
  if (e < EMIN) e = EMIN;
  float r = rintf(a * pow2f(MAN - e)) * pow2f(e - MAN);  // both products exact; rintf: half to even
  if (r > maxv) r = maxv;
  return copysignf(r, v);
}

__device__ __forceinline__ uint32_t e2m1_code(float r) {  // r exactly representable
  const float a = fabsf(r);
  uint32_t c;
  if (a < 1.0f) {
    c = (uint32_t)(a * 2.0f);  // 0 or 0.5 (subnormal)
  } else {
    const int e = ilogbf(a);
    c = ((uint32_t)(e + 1) << 1) | (uint32_t)((a * pow2f(-e) - 1.0f) * 2.0f);
  }
  return (signbit(r) ? 8u : 0u) | c;
}

__device__ __forceinline__ uint32_t e4m3_code(float r) {  // r exactly representable
  const float a = fabsf(r);
  uint32_t c = 0;
  if (a != 0.0f) {
    const int e = ilogbf(a);
    c = e < -6 ? (uint32_t)(a * 512.0f) : ((uint32_t)(e + 7) << 3) | (uint32_t)((a * pow2f(-e) - 1.0f) * 8.0f);
  }
  return (signbit(r) ? 0x80u : 0u) | c;
}

__device__ __forceinline__ void load_block(const __nv_bfloat16* w, int n, float* v) {
  const uint4* src = reinterpret_cast<const uint4*>(w);
  for (int c = 0; c < n / 8; ++c) {
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
}

// mxfp4 (ELEM8 = false) / mxfp8: one thread per block of 32 weights.
template <bool ELEM8>
__global__ void __launch_bounds__(256) quantize_mx_kernel(const __nv_bfloat16* __restrict__ w, int64_t n_blocks,
                                                          uint8_t* __restrict__ wq, uint8_t* __restrict__ scales) {
  const int64_t bi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (bi >= n_blocks) return;
  float v[32];
  load_block(w + bi * 32, 32, v);
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
  constexpr int EMAX = ELEM8 ? 8 : 2;  // largest exponent of the element type
  int kx = amax > 0.0f ? ilogbf(amax) - EMAX : 0;
  kx = kx < -127 ? -127 : (kx > 127 ? 127 : kx);
  scales[bi] = (uint8_t)(kx + 127);
  uint32_t words[ELEM8 ? 8 : 4] = {};
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const float x = scalbnf(v[k], -kx);  // exact: a power-of-two scale
    const uint32_t c = ELEM8 ? e4m3_code(round_small<3, -6>(x, 448.0f)) : e2m1_code(round_small<1, 0>(x, 6.0f));
    if (ELEM8)
      words[k / 4] |= c << (8 * (k % 4));
    else
      words[k / 8] |= c << (4 * (k % 8));
  }
  uint4* dst = reinterpret_cast<uint4*>(wq + bi * (ELEM8 ? 32 : 16));
  dst[0] = make_uint4(words[0], words[1], words[2], words[3]);
  if (ELEM8) dst[1] = make_uint4(words[ELEM8 ? 4 : 0], words[ELEM8 ? 5 : 0], words[ELEM8 ? 6 : 0], words[ELEM8 ? 7 : 0]);
}

// nvfp4, step 1: the largest magnitude of each tensor (rows_per_tensor rows of H), as the bits of a
// non-negative float32 (ordered like unsigned integers) in tscale, which starts zeroed.
__global__ void __launch_bounds__(256) nv_amax_kernel(const __nv_bfloat16* __restrict__ w, int64_t per_tensor,
                                                      int64_t chunks, float* tscale) {
  const int64_t t = blockIdx.y;
  const int64_t per_chunk = (per_tensor + chunks - 1) / chunks;
  const int64_t i0 = (int64_t)blockIdx.x * per_chunk, i1 = min(per_tensor, i0 + per_chunk);
  const uint16_t* src = reinterpret_cast<const uint16_t*>(w) + t * per_tensor;
  uint32_t m = 0;
  for (int64_t i = i0 + threadIdx.x; i < i1; i += blockDim.x) m = max(m, ((uint32_t)__ldg(src + i) & 0x7FFFu) << 16);
  for (int off = 16; off; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0 && m) atomicMax(reinterpret_cast<unsigned int*>(tscale + t), m);
}

// nvfp4, step 2: tensor scale t = amax / (6 * 448) (1 for an all-zero tensor).
__global__ void nv_tscale_kernel(float* tscale, int64_t n_tensors) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n_tensors) return;
  const float amax = tscale[t];
  tscale[t] = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
}

// nvfp4, step 3: one thread per block of 16 weights: E4M3 scale S of (amax / 6) / t, then each
// weight w / (S t) as E2M1 (codes 0 when S t is 0).
__global__ void __launch_bounds__(256) quantize_nv_kernel(const __nv_bfloat16* __restrict__ w, int64_t n_blocks,
                                                          int64_t blocks_per_tensor, const float* __restrict__ tscale,
                                                          uint8_t* __restrict__ wq, uint8_t* __restrict__ scales) {
  const int64_t bi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (bi >= n_blocks) return;
  float v[16];
  load_block(w + bi * 16, 16, v);
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
  const float t = __ldg(tscale + bi / blocks_per_tensor);
  const float S = round_small<3, -6>(__fdiv_rn(__fdiv_rn(amax, 6.0f), t), 448.0f);
  scales[bi] = (uint8_t)e4m3_code(S);
  const float denom = __fmul_rn(S, t);
  uint32_t words[2] = {0u, 0u};
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t c = denom != 0.0f ? e2m1_code(round_small<1, 0>(__fdiv_rn(v[k], denom), 6.0f)) : 0u;
    words[k / 8] |= c << (4 * (k % 8));
  }
  *reinterpret_cast<uint2*>(wq + bi * 8) = make_uint2(words[0], words[1]);
}

}  // namespace

cudaError_t launch_quantize(const __nv_bfloat16* w, int64_t rows, int64_t H, int group_size, int bits, uint8_t* wq,
                            __nv_bfloat16* scales, __nv_bfloat16* biases, cudaStream_t s) {
  const int64_t n_groups = rows * (H / group_size);
  if (n_groups == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = (unsigned)((n_groups + threads - 1) / threads);
#define GQMM_Q(GS, B) quantize_kernel<GS, B><<<blocks, threads, 0, s>>>(w, n_groups, wq, scales, biases)
  if (bits == 4) {
    switch (group_size) {
      case 32: GQMM_Q(32, 4); break;
      case 64: GQMM_Q(64, 4); break;
      case 128: GQMM_Q(128, 4); break;
      default: return cudaErrorInvalidValue;
    }
  } else {
    if (group_size != 64) return cudaErrorInvalidValue;
    switch (bits) {
      case 2: GQMM_Q(64, 2); break;
      case 3: GQMM_Q(64, 3); break;
      case 5: GQMM_Q(64, 5); break;
      case 6: GQMM_Q(64, 6); break;
      case 8: GQMM_Q(64, 8); break;
      default: return cudaErrorInvalidValue;
    }
  }
#undef GQMM_Q
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp(const __nv_bfloat16* w, int64_t rows, int64_t H, int64_t rows_per_tensor, int kind,
                               uint8_t* wq, uint8_t* scales, float* tscale, cudaStream_t s) {
  const int threads = 256;
  if (rows * H == 0) return cudaSuccess;
  if (kind == kMxfp4 || kind == kMxfp8) {
    const int64_t n_blocks = rows * (H / 32);
    const unsigned blocks = (unsigned)((n_blocks + threads - 1) / threads);
    if (kind == kMxfp4)
      quantize_mx_kernel<false><<<blocks, threads, 0, s>>>(w, n_blocks, wq, scales);
    else
      quantize_mx_kernel<true><<<blocks, threads, 0, s>>>(w, n_blocks, wq, scales);
    return cudaGetLastError();
  }
  if (kind != kNvfp4) return cudaErrorInvalidValue;
  const int64_t n_tensors = rows / rows_per_tensor, per_tensor = rows_per_tensor * H;
  cudaError_t e = cudaMemsetAsync(tscale, 0, sizeof(float) * (size_t)n_tensors, s);
  if (e != cudaSuccess) return e;
  const int64_t chunks = (per_tensor + (1 << 20) - 1) >> 20;  // about 1 M weights per block
  nv_amax_kernel<<<dim3((unsigned)chunks, (unsigned)n_tensors), threads, 0, s>>>(w, per_tensor, chunks, tscale);
  nv_tscale_kernel<<<(unsigned)((n_tensors + threads - 1) / threads), threads, 0, s>>>(tscale, n_tensors);
  const int64_t n_blocks = rows * (H / 16);
  quantize_nv_kernel<<<(unsigned)((n_blocks + threads - 1) / threads), threads, 0, s>>>(w, n_blocks, per_tensor / 16,
                                                                                      tscale, wq, scales);
  return cudaGetLastError();
}

}  // namespace gqmm

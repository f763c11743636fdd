// The MoE expert MLP (gqmm_moe_mlp): gate/up projection -> gating -> down projection, the
// two projections sharing one route sort and one work list.  This file holds the gating step;
// the projections are the gather matmul's kernels, called by api.cu with separate row maps for
// x and y (the first gathers x by the route's permutation and writes its output in sorted
// order, the second reads that sorted intermediate and scatters y back to the routed rows).
// mlx PR #4023 "Pick BM from rows per expert", section Measurement (the projections are timed
// as chained up/down pairs); mlxcel #629 References (a fused switch-GeGLU over gather_qmm).
#include "mlp.cuh"

namespace gqmm {
namespace {

constexpr int kGateThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}
// act(g) * u in fp32.  SiLU: g / (1 + e^-g).  GELU by its definition g * Phi(g) =
// g/2 (1 + erf(g / sqrt 2)), and its tanh form g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))
// (Hendrycks and Gimpel, "Gaussian Error Linear Units"); expf, erff and tanhf are CUDA's.
template <int ACT>
__device__ __forceinline__ float glu(float g, float u) {
  if constexpr (ACT == GQMM_ACT_SILU) {
    return g / (1.f + expf(-g)) * u;
  } else if constexpr (ACT == GQMM_ACT_GELU) {
    constexpr float kInvSqrt2 = 0.70710678118654752f;
    return 0.5f * g * (1.f + erff(g * kInvSqrt2)) * u;
  } else {
    constexpr float kSqrt2OverPi = 0.79788456080286536f;
    return 0.5f * g * (1.f + tanhf(kSqrt2OverPi * (g + 0.044715f * g * g * g))) * u;
  }
}

// h[j, i] = bf16(act(h1[j, i]) * h1[j, I + i]) for the n sorted rows of the gate/up output,
// eight columns per thread and step.  Block 0 also resets the work counter that the second
// projection's tensor-core GEMM takes units from to that GEMM's number of unit workers (this
// kernel starts after the first projection has ended).
template <int ACT>
__global__ void __launch_bounds__(kGateThreads) glu_kernel(const __nv_bfloat16* __restrict__ h1,
                                                           __nv_bfloat16* __restrict__ h, int64_t n, int I,
                                                           WsHeader* header, int workers) {
  grid_dependents_launch();  // the second projection may start its prologue
  if (blockIdx.x == 0 && threadIdx.x == 0) header->next_unit = workers;
  const int64_t per_row = I / 8;
  const int64_t total = n * per_row;
  for (int64_t v = (int64_t)blockIdx.x * kGateThreads + threadIdx.x; v < total; v += (int64_t)gridDim.x * kGateThreads) {
    const int64_t j = v / per_row, c = (v - j * per_row) * 8;
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(h1 + j * 2 * I + c));
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(h1 + j * 2 * I + I + c));
    uint4 o;
    o.x = pack_bf16x2(glu<ACT>(bf16_lo(g.x), bf16_lo(u.x)), glu<ACT>(bf16_hi(g.x), bf16_hi(u.x)));
    o.y = pack_bf16x2(glu<ACT>(bf16_lo(g.y), bf16_lo(u.y)), glu<ACT>(bf16_hi(g.y), bf16_hi(u.y)));
    o.z = pack_bf16x2(glu<ACT>(bf16_lo(g.z), bf16_lo(u.z)), glu<ACT>(bf16_hi(g.z), bf16_hi(u.z)));
    o.w = pack_bf16x2(glu<ACT>(bf16_lo(g.w), bf16_lo(u.w)), glu<ACT>(bf16_hi(g.w), bf16_hi(u.w)));
    *reinterpret_cast<uint4*>(h + j * I + c) = o;
  }
}

}  // namespace

cudaError_t launch_glu(const __nv_bfloat16* h1, __nv_bfloat16* h, int64_t n, int I, int activation,
                       WsHeader* header, int sms, int workers, cudaStream_t s) {
  const int64_t total = n * (I / 8);
  int64_t blocks = (total + kGateThreads - 1) / kGateThreads;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  switch (activation) {
    case GQMM_ACT_SILU: glu_kernel<GQMM_ACT_SILU><<<(unsigned)blocks, kGateThreads, 0, s>>>(h1, h, n, I, header, workers); break;
    case GQMM_ACT_GELU: glu_kernel<GQMM_ACT_GELU><<<(unsigned)blocks, kGateThreads, 0, s>>>(h1, h, n, I, header, workers); break;
    case GQMM_ACT_GELU_TANH:
      glu_kernel<GQMM_ACT_GELU_TANH><<<(unsigned)blocks, kGateThreads, 0, s>>>(h1, h, n, I, header, workers);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gqmm

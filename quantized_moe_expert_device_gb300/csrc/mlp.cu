// The MoE expert MLP (gqmm_moe_mlp): gate/up projection -> SiLU gating -> down projection, the
// two projections sharing one route sort and one work list.  This file holds the gating step;
// the projections are the gather matmul's kernels, called by api.cu with separate row maps for
// x and y (the first gathers x by the route's permutation and writes its output in sorted
// order, the second reads that sorted intermediate and scatters y back to the routed rows).
// mlx PR #4023 "Pick BM from rows per expert", section Measurement (the projections are timed
// as chained up/down pairs); mlxcel #629 References (a fused switch MLP over gather_qmm).
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

constexpr int kGateThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}
// SiLU(g) * u in fp32
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// h[j, i] = bf16(SiLU(h1[j, i]) * h1[j, I + i]) for the n sorted rows of the gate/up output,
// eight columns per thread and step.  Block 0 also resets the work counter that the second
// projection's tensor-core GEMM takes units from (this kernel starts after the first has ended).
__global__ void __launch_bounds__(kGateThreads) swiglu_kernel(const __nv_bfloat16* __restrict__ h1,
                                                              __nv_bfloat16* __restrict__ h, int64_t n, int I,
                                                              WsHeader* header, int sms) {
  grid_dependents_launch();  // the second projection may start its prologue
  if (blockIdx.x == 0 && threadIdx.x == 0) header->next_unit = sms;
  const int64_t per_row = I / 8;
  const int64_t total = n * per_row;
  for (int64_t v = (int64_t)blockIdx.x * kGateThreads + threadIdx.x; v < total; v += (int64_t)gridDim.x * kGateThreads) {
    const int64_t j = v / per_row, c = (v - j * per_row) * 8;
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(h1 + j * 2 * I + c));
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(h1 + j * 2 * I + I + c));
    uint4 o;
    o.x = pack_bf16x2(silu_mul(bf16_lo(g.x), bf16_lo(u.x)), silu_mul(bf16_hi(g.x), bf16_hi(u.x)));
    o.y = pack_bf16x2(silu_mul(bf16_lo(g.y), bf16_lo(u.y)), silu_mul(bf16_hi(g.y), bf16_hi(u.y)));
    o.z = pack_bf16x2(silu_mul(bf16_lo(g.z), bf16_lo(u.z)), silu_mul(bf16_hi(g.z), bf16_hi(u.z)));
    o.w = pack_bf16x2(silu_mul(bf16_lo(g.w), bf16_lo(u.w)), silu_mul(bf16_hi(g.w), bf16_hi(u.w)));
    *reinterpret_cast<uint4*>(h + j * I + c) = o;
  }
}

}  // namespace

cudaError_t launch_swiglu(const __nv_bfloat16* h1, __nv_bfloat16* h, int64_t n, int I, WsHeader* header, int sms,
                          cudaStream_t s) {
  const int64_t total = n * (I / 8);
  int64_t blocks = (total + kGateThreads - 1) / kGateThreads;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  swiglu_kernel<<<(unsigned)blocks, kGateThreads, 0, s>>>(h1, h, n, I, header, sms);
  return cudaGetLastError();
}

}  // namespace gqmm

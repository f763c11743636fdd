// Declarations of the MoE expert MLP (gqmm_moe_mlp), shared by api.cu and mlp.cu.
#pragma once

#include "gqmm_internal.cuh"

namespace gqmm {

// Workspace of the MoE expert MLP: the route/plan region of a gate/up gather (no K split),
// then the gate/up output [n, 2I] and the gated intermediate [n, I], bf16, in sorted row order.
struct MlpLayout {
  WsLayout route;
  size_t h1, h, total;
};
inline MlpLayout mlp_ws_layout(int64_t n, int H, int I, int E) {
  (void)H;
  MlpLayout M;
  M.route = ws_layout(n, 2 * I, E, false);
  size_t off = align256(M.route.total);
  M.h1 = off;
  off = align256(off + (size_t)(n > 0 ? n : 1) * 2 * (size_t)I * 2);
  M.h = off;
  off = align256(off + (size_t)(n > 0 ? n : 1) * (size_t)I * 2);
  M.total = off;
  return M;
}

int moe_mlp_impl(const void* x, const void* wq_gu, const void* sc_gu, const void* bs_gu, const void* wq_dn,
                 const void* sc_dn, const void* bs_dn, const uint32_t* idx, int64_t T, int A, int H, int I, int E,
                 int group_size, int bits, int activation, int sorted, int x_shared, void* y, void* ws,
                 size_t ws_bytes, cudaStream_t s);

// Gating of the MLP's gate/up output (n sorted rows of [g | u]) by a GQMM_ACT_* activation into
// h [n, I] (grid sized for `sms` SMs); also resets header->next_unit to `workers`, the unit
// workers of the down projection's tensor-core GEMM (it starts after the gate/up projection has
// ended).
cudaError_t launch_glu(const __nv_bfloat16* h1, __nv_bfloat16* h, int64_t n, int I, int activation,
                       WsHeader* header, int sms, int workers, cudaStream_t s);

}  // namespace gqmm

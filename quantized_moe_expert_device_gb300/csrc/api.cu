// C ABI of libgqmm (declared in include/gqmm.h): argument validation, workspace layout,
// kernel launches on the caller's stream, device status, instrumentation.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "formats.cuh"
#include "gqmm_internal.cuh"
#include "gemm_nn.cuh"
#include "mlp.cuh"

using namespace gqmm;

namespace {

thread_local std::string t_last_error;
std::atomic<int64_t> g_launches{0};
std::atomic<int> g_test_stall{0};  // gqmm_test_stall_next: GEMM launches left to stall
std::atomic<int64_t> g_dispatch[GQMM_VARIANT_COUNT];

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

int ok() {
  t_last_error.clear();
  return GQMM_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool log_dispatch() {
  static const bool on = [] {
    const char* e = std::getenv("GQMM_LOG_DISPATCH");
    return e && e[0] && e[0] != '0';
  }();
  return on;
}

void count_variant(int v) {
  g_dispatch[v].fetch_add(1, std::memory_order_relaxed);
}

// Device check: the library is built for sm_103a only.
int check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  static std::atomic<int> cached_ok[64];  // zero-initialized; set once a device has passed the check
  if (dev >= 0 && dev < 64 && cached_ok[dev].load(std::memory_order_relaxed) == 1) return GQMM_OK;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (!(major == 10 && minor == 3))
    return fail(GQMM_ERR_DEVICE, "device %d is sm_%d%d; libgqmm is built for sm_103a only", dev, major, minor);
  if (dev >= 0 && dev < 64) cached_ok[dev].store(1, std::memory_order_relaxed);
  return GQMM_OK;
}

// ---- GEMM kernel timer -------------------------------------------------------------------
std::mutex g_timer_mu;
bool g_timer_on = false;
std::vector<std::pair<cudaEvent_t, cudaEvent_t>> g_events;
size_t g_events_used = 0;

bool timer_begin(cudaStream_t s, size_t* slot) {
  std::lock_guard<std::mutex> lk(g_timer_mu);
  if (!g_timer_on || g_events_used >= g_events.size()) return false;  // capacity is set up front
  *slot = g_events_used++;
  cudaEventRecord(g_events[*slot].first, s);
  return true;
}

void timer_end(cudaStream_t s, size_t slot) {
  std::lock_guard<std::mutex> lk(g_timer_mu);
  cudaEventRecord(g_events[slot].second, s);
}

// Affine formats the kernels take: 4-bit codes with 32-, 64- or 128-wide groups; 2-, 3-, 5-, 6- and
// 8-bit codes with 64-wide groups.
int check_affine_format(int group_size, int bits) {
  if (bits == 4 && (group_size == 32 || group_size == 64 || group_size == 128)) return GQMM_OK;
  if ((bits == 2 || bits == 3 || bits == 5 || bits == 6 || bits == 8) && group_size == 64) return GQMM_OK;
  return fail(GQMM_ERR_UNSUPPORTED,
              "need bits=4 with group_size 32, 64 or 128, or bits 2, 3, 5, 6 or 8 with group_size 64 (got %d, %d)",
              group_size, bits);
}

int validate_gather(const void* x, const void* wq, const void* scales, const void* biases,
                    const uint32_t* idx, int64_t T, int A, int H, int F, int E, int group_size,
                    int bits, const void* y) {
  if (!x || !wq || !scales || !biases || !y) return fail(GQMM_ERR_NULL, "x, wq, scales, biases and y must be non-NULL");
  int rc = check_affine_format(group_size, bits);
  if (rc) return rc;
  if (H > 0 && ((int64_t)H * bits / 8) % 16)
    return fail(GQMM_ERR_SHAPE, "a weight row's codes (H*bits/8 = %lld bytes) must be a multiple of 16 bytes",
                (long long)H * bits / 8);
  if (T < 1 || A < 1 || T * (int64_t)A > 2147483647LL)
    return fail(GQMM_ERR_SHAPE, "need T >= 1, A >= 1, T*A < 2^31 (got T=%lld A=%d)", (long long)T, A);
  if (H <= 0 || H % 64 || H % group_size)
    return fail(GQMM_ERR_SHAPE, "H must be a positive multiple of 64 and of group_size (got %d, %d)", H, group_size);
  if (F <= 0 || F % 16) return fail(GQMM_ERR_SHAPE, "F must be a positive multiple of 16 (got %d)", F);
  if (E < 1) return fail(GQMM_ERR_SHAPE, "E must be >= 1 (got %d)", E);
  if (E > GQMM_MAX_EXPERTS) return fail(GQMM_ERR_UNSUPPORTED, "E=%d exceeds %d", E, GQMM_MAX_EXPERTS);
  if ((int64_t)E * F > 2147483647LL) return fail(GQMM_ERR_SHAPE, "E*F must be < 2^31");
  if (!idx && E != 1) return fail(GQMM_ERR_NULL, "idx may be NULL only for the dense case E == 1");
  if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(scales, 16) || !aligned(biases, 16) || !aligned(y, 16))
    return fail(GQMM_ERR_ALIGN, "x, wq, scales, biases and y must be 16-byte aligned");
  if (idx && !aligned(idx, 4)) return fail(GQMM_ERR_ALIGN, "idx must be 4-byte aligned");
  return GQMM_OK;
}

// gqmm_gather_qmm_fp's weights: codes, one scale byte per block, and for nvfp4 a float32 scale
// per expert.
int validate_gather_fp(const void* x, const void* wq, const void* scales, const float* tscale, const uint32_t* idx,
                       int64_t T, int A, int H, int F, int E, int mode, const void* y) {
  if (mode != GQMM_MODE_MXFP4 && mode != GQMM_MODE_NVFP4 && mode != GQMM_MODE_MXFP8)
    return fail(GQMM_ERR_UNSUPPORTED, "mode must be GQMM_MODE_MXFP4, GQMM_MODE_NVFP4 or GQMM_MODE_MXFP8 (got %d)", mode);
  if (!x || !wq || !scales || !y) return fail(GQMM_ERR_NULL, "x, wq, scales and y must be non-NULL");
  if (mode == GQMM_MODE_NVFP4 && !tscale) return fail(GQMM_ERR_NULL, "nvfp4 needs the per-expert scales");
  if (T < 1 || A < 1 || T * (int64_t)A > 2147483647LL)
    return fail(GQMM_ERR_SHAPE, "need T >= 1, A >= 1, T*A < 2^31 (got T=%lld A=%d)", (long long)T, A);
  if (H <= 0 || H % 64) return fail(GQMM_ERR_SHAPE, "H must be a positive multiple of 64 (got %d)", H);
  if (F <= 0 || F % 16) return fail(GQMM_ERR_SHAPE, "F must be a positive multiple of 16 (got %d)", F);
  if (E < 1) return fail(GQMM_ERR_SHAPE, "E must be >= 1 (got %d)", E);
  if (E > GQMM_MAX_EXPERTS) return fail(GQMM_ERR_UNSUPPORTED, "E=%d exceeds %d", E, GQMM_MAX_EXPERTS);
  if ((int64_t)E * F > 2147483647LL) return fail(GQMM_ERR_SHAPE, "E*F must be < 2^31");
  if (!idx && E != 1) return fail(GQMM_ERR_NULL, "idx may be NULL only for the dense case E == 1");
  if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(y, 16) || !aligned(scales, 4) || (tscale && !aligned(tscale, 4)))
    return fail(GQMM_ERR_ALIGN, "x, wq and y must be 16-byte aligned, scales and tscale 4-byte aligned");
  if (idx && !aligned(idx, 4)) return fail(GQMM_ERR_ALIGN, "idx must be 4-byte aligned");
  return GQMM_OK;
}

// gqmm_gather_qmm_nn's weights: W[e] is [K, N] with 4-bit affine codes grouped along N.  The
// tensor-core path copies one k-block (64 k-rows) of a unit's 256 columns per TMA box, so K is
// a multiple of 64 and a code row (N/2 bytes) a multiple of 16 bytes.
int validate_gather_nn(const void* x, const void* wq, const void* scales, const void* biases, const uint32_t* idx,
                       int64_t T, int A, int K, int N, int E, int group_size, int bits, const void* y) {
  if (!x || !wq || !scales || !biases || !y) return fail(GQMM_ERR_NULL, "x, wq, scales, biases and y must be non-NULL");
  if ((group_size != 32 && group_size != 64 && group_size != 128) || bits != 4)
    return fail(GQMM_ERR_UNSUPPORTED, "need group_size 32, 64 or 128 and bits=4 (got %d, %d)", group_size, bits);
  if (T < 1 || A < 1 || T * (int64_t)A > 2147483647LL)
    return fail(GQMM_ERR_SHAPE, "need T >= 1, A >= 1, T*A < 2^31 (got T=%lld A=%d)", (long long)T, A);
  if (K <= 0 || K % 64) return fail(GQMM_ERR_SHAPE, "K must be a positive multiple of 64 (got %d)", K);
  if (N <= 0 || N % 32 || N % group_size)
    return fail(GQMM_ERR_SHAPE, "N must be a positive multiple of 32 and of group_size (got %d, %d)", N, group_size);
  if (E < 1) return fail(GQMM_ERR_SHAPE, "E must be >= 1 (got %d)", E);
  if (E > GQMM_MAX_EXPERTS) return fail(GQMM_ERR_UNSUPPORTED, "E=%d exceeds %d", E, GQMM_MAX_EXPERTS);
  if ((int64_t)E * K > 2147483647LL || (int64_t)E * N > 2147483647LL)
    return fail(GQMM_ERR_SHAPE, "E*K and E*N must be < 2^31");
  if (!idx && E != 1) return fail(GQMM_ERR_NULL, "idx may be NULL only for the dense case E == 1");
  if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(scales, 2) || !aligned(biases, 2) || !aligned(y, 16))
    return fail(GQMM_ERR_ALIGN, "x, wq and y must be 16-byte aligned, scales and biases 2-byte aligned");
  if (idx && !aligned(idx, 4)) return fail(GQMM_ERR_ALIGN, "idx must be 4-byte aligned");
  return GQMM_OK;
}

int validate_shared(int x_shared, const uint32_t* idx) {
  if (x_shared != 0 && x_shared != 1) return fail(GQMM_ERR_SHAPE, "x_shared must be 0 or 1");
  if (x_shared && !idx) return fail(GQMM_ERR_NULL, "x_shared needs idx (a token's rows are its A routed rows)");
  return GQMM_OK;
}

}  // namespace

int gqmm::report_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

namespace gqmm {
namespace {

// Launches one projection (the streaming kernel or the tensor-core GEMM, as `shape` says) with
// the kernel timer around it, and counts and optionally logs the variant.
int launch_projection(const GemmArgs& ga, const UnitShape& shape, int sms, cudaStream_t s, const char* what,
                      int route_variant) {
  size_t slot = 0;
  const bool timed = timer_begin(s, &slot);
  int gemm_launched = 0;
  cudaError_t e;
  if (shape.stream) {
    e = launch_gemv(ga, shape.chunk_rows, sms, s);
    gemm_launched = 1;
  } else {
    GemmArgs a = ga;
    int left = g_test_stall.load();
    while (left > 0 && !g_test_stall.compare_exchange_weak(left, left - 1)) {
    }
    if (left > 0) a.test_stall = 1;
    e = launch_gemm_tc(a, s, &gemm_launched);
  }
  if (timed) timer_end(s, slot);
  g_launches.fetch_add(gemm_launched);
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "grouped GEMM launch: %s", cudaGetErrorString(e));
  const bool stream_mma = shape.stream && gemv_uses_mma(shape.chunk_rows, ga.H, ga.E);
  count_variant(shape.stream ? (stream_mma ? GQMM_VARIANT_GEMV_MMA : GQMM_VARIANT_GEMV)
                : shape.chunk_rows <= kChunkRowsNarrow ? GQMM_VARIANT_GEMM_NARROW : GQMM_VARIANT_GEMM_TC);
  if (ga.ks_cap > 1) count_variant(GQMM_VARIANT_SPLIT_K);
  int workers = sms;
  if (log_dispatch() && !shape.stream) (void)gemm_tc_workers(ga.kind, ga.bits, shape.chunk_rows, &workers);
  if (log_dispatch())
    std::fprintf(stderr, "[gqmm] %s n=%lld H=%d F=%d E=%d route=%s gemm=%s ks_cap=%d workers=%d\n", what,
                 (long long)ga.n, ga.H, ga.F, ga.E,
                 route_variant == GQMM_VARIANT_ROUTE_DENSE ? "dense"
                 : route_variant == GQMM_VARIANT_ROUTE_SORTED ? "sorted"
                 : route_variant == GQMM_VARIANT_ROUTE_FUSED ? "in-kernel" : "unsorted",
                 shape.stream ? (stream_mma ? "stream-mma" : "stream")
                 : shape.chunk_rows <= kChunkRowsNarrow ? "narrow"
                 : shape.chunk_rows <= kChunkRowsMid    ? "mid"
                 : shape.chunk_rows > kChunkRowsWide    ? "pair"
                                                        : "wide",
                 ga.ks_cap, workers);
  return GQMM_OK;
}

}  // namespace
}  // namespace gqmm

int gqmm::gather_qmm_impl(const void* x, const void* wq, const void* scales, const void* biases,
                          const uint32_t* idx, int64_t T, int A, int H, int F, int E, int group_size, int bits,
                          int sorted, int x_shared, void* y, void* ws, size_t ws_bytes, cudaStream_t s,
                          bool allow_split, bool clear_header, int kind, const float* tscale) {
  int rc = kind == kAffine     ? validate_gather(x, wq, scales, biases, idx, T, A, H, F, E, group_size, bits, y)
           : kind == kAffineNn ? validate_gather_nn(x, wq, scales, biases, idx, T, A, H, F, E, group_size, bits, y)
                               : validate_gather_fp(x, wq, scales, tscale, idx, T, A, H, F, E, kind, y);
  if (rc) return rc;
  rc = validate_shared(x_shared, idx);
  if (rc) return rc;
  if (sorted != 0 && sorted != 1) return fail(GQMM_ERR_SHAPE, "sorted must be 0 or 1");
  if (!ws) return fail(GQMM_ERR_NULL, "ws must be non-NULL");
  const int64_t n = T * (int64_t)A;
  const WsLayout L = ws_layout(n, F, E, allow_split);
  UnitShape shape = unit_shape(n, H, F, E);
  if (!allow_split) shape.ksplit = 1;
  const bool affine4 = kind == kAffine && bits == 4;
  // the weight-streaming kernels take 4-bit affine codes in 64-wide groups
  if (group_size != 64 || !affine4) shape.stream = false;
  if (!aligned(ws, 256) || ws_bytes < L.total)
    return fail(GQMM_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", L.total, ws_bytes);
  rc = check_device();
  if (rc) return rc;
  // wide 4-bit affine calls of more than 256 rows per expert run on CTA pairs, in chunks of up to
  // 512 rows, when the device holds any
  if (!shape.stream) {
    int cr = shape.chunk_rows;
    cudaError_t ce = gemm_tc_chunk_rows(kind, kind == kAffine ? bits : 4, shape.chunk_rows, n, E, &cr);
    if (ce != cudaSuccess) return fail(GQMM_ERR_CUDA, "device query: %s", cudaGetErrorString(ce));
    shape.chunk_rows = cr;
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  WsHeader* header = reinterpret_cast<WsHeader*>(w);
  if (clear_header) {
    cudaError_t ce = cudaMemsetAsync(header, 0, sizeof(WsHeader), s);
    if (ce != cudaSuccess) return fail(GQMM_ERR_CUDA, "clearing the workspace header: %s", cudaGetErrorString(ce));
  }

  RouteArgs ra;
  ra.idx = idx;
  ra.n = n;
  ra.E = E;
  ra.sorted = sorted;
  ra.perm = reinterpret_cast<int32_t*>(w + L.perm);
  ra.offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  ra.tile_hist = reinterpret_cast<uint32_t*>(w + L.tile_hist);
  ra.chunks = reinterpret_cast<Chunk*>(w + L.chunks);
  ra.header = header;
  ra.y = static_cast<__nv_bfloat16*>(y);
  ra.F = F;
  ra.n_tiles = L.n_tiles;
  ra.chunk_rows = shape.chunk_rows;
  ra.n_fpairs = (F + kUnitRows - 1) / kUnitRows;
  ra.ks_cap = L.has_acc && !shape.stream ? shape.ksplit : 1;
  int sms = 0;
  cudaError_t e = device_sm_count(&sms);
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  // the plan step starts the tensor-core GEMM's unit counter at its number of unit workers
  int workers = sms;
  if (!shape.stream) {
    e = gemm_tc_workers(kind, kind == kAffine ? bits : 4, shape.chunk_rows, &workers);
    if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  }
  ra.sms = workers;
  // Decode-sized calls on the weight-streaming path need no route kernel: a dense call's plan is
  // the single chunk, and an unsorted routed call of at most kFusedPlanMaxRows rows on the CUDA-core
  // streaming kernel is planned inside that kernel.  Such a call is one programmatic-dependent
  // launch, which the previous call's streaming kernel lets start as its blocks retire.
  const bool fused = shape.stream && idx != nullptr && !sorted && n <= kFusedPlanMaxRows &&
                     !gemv_uses_mma(shape.chunk_rows, H, E);
  const bool route_kernel = !(shape.stream && (idx == nullptr || fused));
  const bool permuted = idx != nullptr && !sorted && !fused;
  if (route_kernel) {
    int launched = 0;
    e = launch_route(ra, s, &launched);
    g_launches.fetch_add(launched);
    if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "route launch: %s", cudaGetErrorString(e));
  }
  const int route_variant = idx == nullptr ? GQMM_VARIANT_ROUTE_DENSE
                            : fused        ? GQMM_VARIANT_ROUTE_FUSED
                            : sorted       ? GQMM_VARIANT_ROUTE_SORTED
                                           : GQMM_VARIANT_ROUTE_UNSORTED;
  count_variant(route_variant);

  GemmArgs ga;
  ga.x = static_cast<const __nv_bfloat16*>(x);
  ga.n = n;
  ga.wq = static_cast<const uint8_t*>(wq);
  ga.scales = static_cast<const __nv_bfloat16*>(scales);
  ga.biases = static_cast<const __nv_bfloat16*>(biases);
  ga.y = static_cast<__nv_bfloat16*>(y);
  ga.perm = permuted ? ra.perm : nullptr;
  ga.y_perm = ga.perm;
  ga.chunks = ra.chunks;
  ga.header = header;
  ga.H = H;
  ga.F = F;
  ga.E = E;
  ga.chunk_rows = shape.chunk_rows;
  ga.ks_cap = ra.ks_cap;
  ga.dense_plan = idx == nullptr ? 1 : 0;
  ga.acc = L.has_acc ? reinterpret_cast<float*>(w + L.acc) : nullptr;
  ga.offsets = ra.offsets;
  ga.group_size = group_size;
  ga.x_div = x_shared ? A : 1;
  ga.idx = idx;
  ga.fused_plan = fused ? 1 : 0;
  ga.kind = kind;
  ga.bits = kind == kAffine ? bits : 4;
  ga.tscale = tscale;
  rc = launch_projection(ga, shape, sms, s, kind == kAffineNn ? "gather_qmm_nn" : "gather_qmm", route_variant);
  if (rc) return rc;
  if (kind == kAffineNn) count_variant(GQMM_VARIANT_NN);
  return ok();
}


int gqmm::moe_mlp_impl(const void* x, const void* wq_gu, const void* sc_gu, const void* bs_gu, const void* wq_dn,
                       const void* sc_dn, const void* bs_dn, const uint32_t* idx, int64_t T, int A, int H, int I, int E,
                       int group_size, int bits, int activation, int sorted, int x_shared, void* y, void* ws,
                       size_t ws_bytes, cudaStream_t s) {
  if (I <= 0 || I > (1 << 29)) return fail(GQMM_ERR_SHAPE, "I must be in [1, 2^29] (got %d)", I);
  if (activation != GQMM_ACT_SILU && activation != GQMM_ACT_GELU && activation != GQMM_ACT_GELU_TANH)
    return fail(GQMM_ERR_UNSUPPORTED, "unknown activation %d", activation);
  if (bits != 4) return fail(GQMM_ERR_UNSUPPORTED, "the expert MLP takes 4-bit codes (got bits=%d)", bits);
  // gate/up projection: K = H, 2I output columns; down projection: K = I, H output columns
  int rc = validate_gather(x, wq_gu, sc_gu, bs_gu, idx, T, A, H, 2 * I, E, group_size, bits, y);
  if (rc) return rc;
  rc = validate_gather(x, wq_dn, sc_dn, bs_dn, idx, T, A, I, H, E, group_size, bits, y);
  if (rc) return rc;
  if (sorted != 0 && sorted != 1) return fail(GQMM_ERR_SHAPE, "sorted must be 0 or 1");
  rc = validate_shared(x_shared, idx);
  if (rc) return rc;
  if (!ws) return fail(GQMM_ERR_NULL, "ws must be non-NULL");
  const int64_t n = T * (int64_t)A;
  const MlpLayout M = mlp_ws_layout(n, H, I, E);
  const WsLayout& L = M.route;
  if (!aligned(ws, 256) || ws_bytes < M.total)
    return fail(GQMM_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", M.total, ws_bytes);
  rc = check_device();
  if (rc) return rc;
  UnitShape shape1 = unit_shape(n, H, 2 * I, E);
  UnitShape shape2 = unit_shape(n, I, H, E);
  shape1.ksplit = shape2.ksplit = 1;  // one work list serves both: no K split, no partial-sum planes
  if (group_size != 64) shape1.stream = shape2.stream = false;  // streaming kernels: 64-wide groups
  uint8_t* w = static_cast<uint8_t*>(ws);
  WsHeader* header = reinterpret_cast<WsHeader*>(w);
  __nv_bfloat16* h1 = reinterpret_cast<__nv_bfloat16*>(w + M.h1);
  __nv_bfloat16* hg = reinterpret_cast<__nv_bfloat16*>(w + M.h);
  int sms = 0;
  cudaError_t e = device_sm_count(&sms);
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "device query: %s", cudaGetErrorString(e));

  RouteArgs ra;
  ra.idx = idx;
  ra.n = n;
  ra.E = E;
  ra.sorted = sorted;
  ra.perm = reinterpret_cast<int32_t*>(w + L.perm);
  ra.offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  ra.tile_hist = reinterpret_cast<uint32_t*>(w + L.tile_hist);
  ra.chunks = reinterpret_cast<Chunk*>(w + L.chunks);
  ra.header = header;
  ra.y = static_cast<__nv_bfloat16*>(y);  // rows with an invalid index are zeroed in the final y
  ra.F = H;
  ra.n_tiles = L.n_tiles;
  ra.chunk_rows = shape1.chunk_rows;
  ra.n_fpairs = (2 * I + kUnitRows - 1) / kUnitRows;
  ra.ks_cap = 1;
  // unit workers of each projection's tensor-core GEMM (the plan step and the gating kernel
  // start the unit counter at these)
  int workers1 = sms, workers2 = sms;
  if (!shape1.stream) e = gemm_tc_workers(kAffine, bits, shape1.chunk_rows, &workers1);
  if (e == cudaSuccess && !shape2.stream) e = gemm_tc_workers(kAffine, bits, shape2.chunk_rows, &workers2);
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  ra.sms = workers1;
  const bool permuted = idx != nullptr && !sorted;
  int launched = 0;
  e = launch_route(ra, s, &launched);
  g_launches.fetch_add(launched);
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "route launch: %s", cudaGetErrorString(e));
  const int route_variant = idx == nullptr ? GQMM_VARIANT_ROUTE_DENSE
                                           : (sorted ? GQMM_VARIANT_ROUTE_SORTED : GQMM_VARIANT_ROUTE_UNSORTED);
  count_variant(route_variant);

  GemmArgs g1;  // gate/up: x gathered by the route's permutation, output in sorted order
  g1.x = static_cast<const __nv_bfloat16*>(x);
  g1.n = n;
  g1.wq = static_cast<const uint8_t*>(wq_gu);
  g1.scales = static_cast<const __nv_bfloat16*>(sc_gu);
  g1.biases = static_cast<const __nv_bfloat16*>(bs_gu);
  g1.y = h1;
  g1.perm = permuted ? ra.perm : nullptr;
  g1.y_perm = nullptr;
  g1.chunks = ra.chunks;
  g1.header = header;
  g1.acc = nullptr;
  g1.offsets = ra.offsets;
  g1.H = H;
  g1.F = 2 * I;
  g1.E = E;
  g1.chunk_rows = shape1.chunk_rows;
  g1.ks_cap = 1;
  g1.dense_plan = idx == nullptr ? 1 : 0;
  g1.group_size = group_size;
  g1.x_div = x_shared ? A : 1;  // the down projection reads the sorted intermediate (x_div 1)
  rc = launch_projection(g1, shape1, sms, s, "moe_mlp gate/up", route_variant);
  if (rc) return rc;

  e = launch_glu(h1, hg, n, I, activation, header, sms, workers2, s);
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "gating launch: %s", cudaGetErrorString(e));
  g_launches.fetch_add(1);

  GemmArgs g2 = g1;  // down: the sorted intermediate in, y scattered to the routed rows
  g2.x = hg;
  g2.wq = static_cast<const uint8_t*>(wq_dn);
  g2.scales = static_cast<const __nv_bfloat16*>(sc_dn);
  g2.biases = static_cast<const __nv_bfloat16*>(bs_dn);
  g2.y = static_cast<__nv_bfloat16*>(y);
  g2.perm = nullptr;
  g2.x_div = 1;
  g2.y_perm = permuted ? ra.perm : nullptr;
  g2.H = I;
  g2.F = H;
  g2.chunk_rows = shape2.chunk_rows;
  rc = launch_projection(g2, shape2, sms, s, "moe_mlp down", route_variant);
  if (rc) return rc;
  return ok();
}

extern "C" {

int gqmm_quantize(const void* w, int64_t rows, int64_t H, int group_size, int bits, void* wq,
                  void* scales, void* biases, gqmm_stream_t stream) {
  if (!w || !wq || !scales || !biases) return fail(GQMM_ERR_NULL, "w, wq, scales, biases must be non-NULL");
  int rc0 = check_affine_format(group_size, bits);
  if (rc0) return rc0;
  if (rows < 0 || H <= 0 || H % group_size)
    return fail(GQMM_ERR_SHAPE, "need rows >= 0 and H a positive multiple of group_size");
  if (!aligned(w, 16) || !aligned(wq, 16)) return fail(GQMM_ERR_ALIGN, "w and wq must be 16-byte aligned");
  if (!aligned(scales, 2) || !aligned(biases, 2)) return fail(GQMM_ERR_ALIGN, "scales and biases must be 2-byte aligned");
  int rc = check_device();
  if (rc) return rc;
  cudaError_t e = launch_quantize(static_cast<const __nv_bfloat16*>(w), rows, H, group_size, bits, static_cast<uint8_t*>(wq),
                                  static_cast<__nv_bfloat16*>(scales), static_cast<__nv_bfloat16*>(biases),
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "quantize launch: %s", cudaGetErrorString(e));
  if (rows * (H / group_size) > 0) g_launches.fetch_add(1);
  return ok();
}

size_t gqmm_workspace_size(int64_t n, int F, int E) {
  if (n < 0 || n > 2147483647LL || F < 0 || E < 1 || E > GQMM_MAX_EXPERTS) return 0;
  return ws_layout(n, F, E).total;
}

int gqmm_route_sort(const uint32_t* idx, int64_t n, int E, int32_t* perm, int32_t* offsets, void* ws,
                    size_t ws_bytes, gqmm_stream_t stream) {
  if (!idx || !perm || !offsets || !ws) return fail(GQMM_ERR_NULL, "idx, perm, offsets and ws must be non-NULL");
  if (n < 0 || n > 2147483647LL) return fail(GQMM_ERR_SHAPE, "n must be in [0, 2^31)");
  if (E < 1) return fail(GQMM_ERR_SHAPE, "E must be >= 1");
  if (E > GQMM_MAX_EXPERTS) return fail(GQMM_ERR_UNSUPPORTED, "E=%d exceeds %d", E, GQMM_MAX_EXPERTS);
  const WsLayout L = ws_layout(n, 1, E);
  if (!aligned(ws, 256) || ws_bytes < L.total)
    return fail(GQMM_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", L.total, ws_bytes);
  int rc = check_device();
  if (rc) return rc;
  uint8_t* w = static_cast<uint8_t*>(ws);
  RouteArgs a;
  a.chunk_rows = kChunkRowsWide;
  a.idx = idx;
  a.n = n;
  a.E = E;
  a.sorted = 0;
  a.perm = perm;
  a.offsets = offsets;
  a.tile_hist = reinterpret_cast<uint32_t*>(w + L.tile_hist);
  a.chunks = nullptr;
  a.header = reinterpret_cast<WsHeader*>(w);
  a.y = nullptr;
  a.F = 0;
  a.n_tiles = L.n_tiles;
  a.n_fpairs = 1;
  a.ks_cap = 1;
  a.sms = 1;
  int launched = 0;
  cudaError_t e = launch_route(a, reinterpret_cast<cudaStream_t>(stream), &launched);
  g_launches.fetch_add(launched);
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "route sort launch: %s", cudaGetErrorString(e));
  count_variant(GQMM_VARIANT_ROUTE_UNSORTED);
  return ok();
}

int gqmm_gather_qmm(const void* x, const void* wq, const void* scales, const void* biases, const uint32_t* idx,
                    int64_t T, int A, int H, int F, int E, int group_size, int bits, int sorted, int x_shared,
                    void* y, void* ws, size_t ws_bytes, gqmm_stream_t stream) {
  return gqmm::gather_qmm_impl(x, wq, scales, biases, idx, T, A, H, F, E, group_size, bits, sorted, x_shared, y, ws,
                               ws_bytes, reinterpret_cast<cudaStream_t>(stream), true);
}

int gqmm_quantize_fp(const void* w, int64_t rows, int64_t H, int64_t rows_per_tensor, int mode, void* wq, void* scales,
                     float* tscale, gqmm_stream_t stream) {
  if (mode != GQMM_MODE_MXFP4 && mode != GQMM_MODE_NVFP4 && mode != GQMM_MODE_MXFP8)
    return fail(GQMM_ERR_UNSUPPORTED, "mode must be GQMM_MODE_MXFP4, GQMM_MODE_NVFP4 or GQMM_MODE_MXFP8 (got %d)", mode);
  if (!w || !wq || !scales) return fail(GQMM_ERR_NULL, "w, wq and scales must be non-NULL");
  if (rows < 0 || H <= 0 || H % 64) return fail(GQMM_ERR_SHAPE, "need rows >= 0 and H a positive multiple of 64");
  if (mode == GQMM_MODE_NVFP4) {
    if (!tscale) return fail(GQMM_ERR_NULL, "nvfp4 needs tscale (one float32 per tensor)");
    if (rows_per_tensor < 1 || rows % rows_per_tensor)
      return fail(GQMM_ERR_SHAPE, "rows must be a multiple of rows_per_tensor >= 1");
    if (rows / rows_per_tensor > 65535) return fail(GQMM_ERR_SHAPE, "at most 65535 tensors");
  }
  if (!aligned(w, 16) || !aligned(wq, 16) || (tscale && !aligned(tscale, 4)))
    return fail(GQMM_ERR_ALIGN, "w and wq must be 16-byte aligned, tscale 4-byte aligned");
  int rc = check_device();
  if (rc) return rc;
  cudaError_t e = launch_quantize_fp(static_cast<const __nv_bfloat16*>(w), rows, H, rows_per_tensor, mode,
                                     static_cast<uint8_t*>(wq), static_cast<uint8_t*>(scales), tscale,
                                     reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "quantize launch: %s", cudaGetErrorString(e));
  if (rows > 0) g_launches.fetch_add(mode == GQMM_MODE_NVFP4 ? 3 : 1);
  return ok();
}

int gqmm_gather_qmm_fp(const void* x, const void* wq, const void* scales, const float* tscale, const uint32_t* idx,
                       int64_t T, int A, int H, int F, int E, int mode, int sorted, int x_shared, void* y, void* ws,
                       size_t ws_bytes, gqmm_stream_t stream) {
  if (mode != GQMM_MODE_MXFP4 && mode != GQMM_MODE_NVFP4 && mode != GQMM_MODE_MXFP8)
    return fail(GQMM_ERR_UNSUPPORTED, "mode must be GQMM_MODE_MXFP4, GQMM_MODE_NVFP4 or GQMM_MODE_MXFP8 (got %d)", mode);
  return gqmm::gather_qmm_impl(x, wq, scales, nullptr, idx, T, A, H, F, E, mode == GQMM_MODE_NVFP4 ? 16 : 32, 4,
                               sorted, x_shared, y, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), true, false,
                               mode, tscale);
}

size_t gqmm_moe_mlp_workspace_size(int64_t n, int H, int I, int E) {
  if (n < 0 || n > 2147483647LL || H < 0 || I < 1 || I > (1 << 29) || E < 1 || E > GQMM_MAX_EXPERTS) return 0;
  return mlp_ws_layout(n, H, I, E).total;
}

int gqmm_moe_mlp(const void* x, const void* wq_gu, const void* sc_gu, const void* bs_gu, const void* wq_dn,
                 const void* sc_dn, const void* bs_dn, const uint32_t* idx, int64_t T, int A, int H, int I, int E,
                 int group_size, int bits, int activation, int sorted, int x_shared, void* y, void* ws,
                 size_t ws_bytes, gqmm_stream_t stream) {
  return gqmm::moe_mlp_impl(x, wq_gu, sc_gu, bs_gu, wq_dn, sc_dn, bs_dn, idx, T, A, H, I, E, group_size, bits,
                            activation, sorted, x_shared, y, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int gqmm_gather_qmm_nn(const void* x, const void* wq, const void* scales, const void* biases, const uint32_t* idx,
                       int64_t T, int A, int K, int N, int E, int group_size, int bits, int sorted, int x_shared,
                       void* y, void* ws, size_t ws_bytes, gqmm_stream_t stream) {
  return gqmm::gather_qmm_impl(x, wq, scales, biases, idx, T, A, K, N, E, group_size, bits, sorted, x_shared, y, ws,
                               ws_bytes, reinterpret_cast<cudaStream_t>(stream), true, false, gqmm::kAffineNn, nullptr);
}

int gqmm_gather_qmm_nn_simt(const void* x, const void* wq, const void* scales, const void* biases,
                            const uint32_t* idx, int64_t T, int A, int K, int N, int E, int group_size, int bits,
                            int x_shared, void* y, gqmm_stream_t stream) {
  if (!x || !wq || !scales || !biases || !y) return fail(GQMM_ERR_NULL, "x, wq, scales, biases and y must be non-NULL");
  if ((group_size != 32 && group_size != 64 && group_size != 128) || bits != 4)
    return fail(GQMM_ERR_UNSUPPORTED, "need group_size 32, 64 or 128 and bits=4 (got %d, %d)", group_size, bits);
  if (T < 1 || A < 1 || T * (int64_t)A > 2147483647LL)
    return fail(GQMM_ERR_SHAPE, "need T >= 1, A >= 1, T*A < 2^31 (got T=%lld A=%d)", (long long)T, A);
  if (K < 1 || K > (1 << 24)) return fail(GQMM_ERR_SHAPE, "K must be in [1, 2^24] (got %d)", K);
  if (N <= 0 || N % group_size || N > (1 << 24))
    return fail(GQMM_ERR_SHAPE, "N must be a positive multiple of group_size, at most 2^24 (got %d)", N);
  if (E < 1) return fail(GQMM_ERR_SHAPE, "E must be >= 1 (got %d)", E);
  if (E > GQMM_MAX_EXPERTS) return fail(GQMM_ERR_UNSUPPORTED, "E=%d exceeds %d", E, GQMM_MAX_EXPERTS);
  if ((int64_t)E * K * N / 2 > (int64_t)1 << 40) return fail(GQMM_ERR_SHAPE, "E*K*N too large");
  if (!idx && E != 1) return fail(GQMM_ERR_NULL, "idx may be NULL only for the dense case E == 1");
  int rc = validate_shared(x_shared, idx);
  if (rc) return rc;
  if (!aligned(x, 2) || !aligned(wq, 16) || !aligned(scales, 2) || !aligned(biases, 2) || !aligned(y, 16))
    return fail(GQMM_ERR_ALIGN, "wq and y must be 16-byte aligned, x, scales and biases 2-byte aligned");
  if (idx && !aligned(idx, 4)) return fail(GQMM_ERR_ALIGN, "idx must be 4-byte aligned");
  rc = check_device();
  if (rc) return rc;
  size_t slot = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool timed = timer_begin(s, &slot);
  cudaError_t e = launch_gemm_nn(static_cast<const __nv_bfloat16*>(x), static_cast<const uint8_t*>(wq),
                                 static_cast<const __nv_bfloat16*>(scales), static_cast<const __nv_bfloat16*>(biases),
                                 idx, T * (int64_t)A, K, N, E, group_size, x_shared ? A : 1,
                                 static_cast<__nv_bfloat16*>(y), s);
  if (timed) timer_end(s, slot);
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "transpose=False launch: %s", cudaGetErrorString(e));
  g_launches.fetch_add(1);
  return ok();
}

int gqmm_gather_qmm_simt(const void* x, const void* wq, const void* scales, const void* biases,
                         const uint32_t* idx, int64_t T, int A, int H, int F, int E, int group_size, int bits,
                         int x_shared, void* y, gqmm_stream_t stream) {
  if (bits != 4) return fail(GQMM_ERR_UNSUPPORTED, "the CUDA-core cross-check takes 4-bit codes (got bits=%d)", bits);
  int rc = validate_gather(x, wq, scales, biases, idx, T, A, H, F, E, group_size, bits, y);
  if (rc) return rc;
  rc = validate_shared(x_shared, idx);
  if (rc) return rc;
  rc = check_device();
  if (rc) return rc;
  cudaError_t e = launch_gemm_simt(static_cast<const __nv_bfloat16*>(x), static_cast<const uint8_t*>(wq),
                                   static_cast<const __nv_bfloat16*>(scales), static_cast<const __nv_bfloat16*>(biases),
                                   idx, T * (int64_t)A, H, F, E, group_size, x_shared ? A : 1,
                                   static_cast<__nv_bfloat16*>(y),
                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "simt launch: %s", cudaGetErrorString(e));
  g_launches.fetch_add(1);
  return ok();
}

int gqmm_device_status(void* ws, gqmm_stream_t stream) {
  if (!ws) return -fail(GQMM_ERR_NULL, "ws must be non-NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return -fail(GQMM_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
  uint32_t st = 0;
  e = cudaMemcpy(&st, ws, sizeof st, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return -fail(GQMM_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  e = cudaMemset(ws, 0, sizeof(uint32_t));
  if (e != cudaSuccess) return -fail(GQMM_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
  ok();
  return (int)st;
}

const char* gqmm_status_string(int status) {
  switch (status) {
    case GQMM_OK: return "ok";
    case GQMM_ERR_NULL: return "a required pointer is NULL";
    case GQMM_ERR_SHAPE: return "a size argument is out of range";
    case GQMM_ERR_UNSUPPORTED: return "unsupported group_size, bits or expert count";
    case GQMM_ERR_ALIGN: return "a pointer is not aligned as required";
    case GQMM_ERR_WORKSPACE: return "workspace too small or misaligned";
    case GQMM_ERR_CUDA: return "CUDA call or kernel launch failed";
    case GQMM_ERR_DEVICE: return "current device is not sm_103";
    case (int)GQMM_STATUS_BAD_INDEX: return "device: an expert index was >= E (rows zeroed)";
    case (int)GQMM_STATUS_NOT_SORTED: return "device: sorted=1 but the indices decrease";
    case (int)GQMM_STATUS_TIMEOUT: return "device: a bounded wait timed out";
    default: return "unknown status";
  }
}

const char* gqmm_last_error(void) { return t_last_error.c_str(); }

int64_t gqmm_launch_count(void) { return g_launches.load(); }

void gqmm_test_stall_next(int n) { g_test_stall.store(n > 0 ? n : 0); }

void gqmm_kernel_timer(int capacity) {
  std::lock_guard<std::mutex> lk(g_timer_mu);
  g_timer_on = capacity > 0;
  g_events_used = 0;
  // Events are created here, outside any timed region.
  while (g_events.size() < (size_t)(capacity > 0 ? capacity : 0)) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) break;
    if (cudaEventCreate(&b) != cudaSuccess) {
      cudaEventDestroy(a);
      break;
    }
    g_events.emplace_back(a, b);
  }
}

int gqmm_kernel_timer_read(int64_t* launches, double* total_ms) {
  std::lock_guard<std::mutex> lk(g_timer_mu);
  double tot = 0.0;
  for (size_t i = 0; i < g_events_used; ++i) {
    cudaError_t e = cudaEventSynchronize(g_events[i].second);
    if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "event sync: %s", cudaGetErrorString(e));
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, g_events[i].first, g_events[i].second);
    if (e != cudaSuccess) return fail(GQMM_ERR_CUDA, "event elapsed: %s", cudaGetErrorString(e));
    tot += ms;
  }
  if (launches) *launches = (int64_t)g_events_used;
  if (total_ms) *total_ms = tot;
  g_events_used = 0;
  return ok();
}

int64_t gqmm_dispatch_count(int variant) {
  if (variant < 0 || variant >= GQMM_VARIANT_COUNT) return -1;
  return g_dispatch[variant].load();
}

}  // extern "C"

// Internal declarations shared by the libgqmm translation units (sm_103a only).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gqmm.h"

namespace gqmm {

// ------------------------------------------------------------------------------------------
// Workspace layout.  Every section starts on a 256-byte boundary.
//   [0, 256)        header: status word, counters written by the route/plan kernels
//   perm            int32 [n]                    sorted position -> flat row
//   offsets         int32 [E + 1]                expert segment starts
//   tile_hist       uint32 [(E + 1) * n_tiles]   per-tile key counts, key-major
//   chunks          Chunk [max_chunks]           work list of (expert, row range)
//   acc             float [ksplit, n, F]         split-K partial sums, one plane per K slice
//                                                (only when split-K can be chosen for these
//                                                sizes; every entry read is written first)
// ------------------------------------------------------------------------------------------
struct WsHeader {
  uint32_t status;    // GQMM_STATUS_* bits, OR-ed by kernels, cleared by gqmm_device_status
  int32_t n_chunks;   // number of valid entries in the chunk list (written by the plan step)
  int32_t ksplit;     // K slices per (chunk, F pair) chosen by the plan step (1 = no split)
  int32_t next_unit;  // work counter of the grouped GEMM's schedulers; the plan step sets it to
                      // the number of unit workers (worker b, a CTA or a CTA pair, takes unit b first)
  int32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

struct Chunk {
  int32_t expert;  // expert id
  int32_t start;   // first sorted position of the chunk
  int32_t rows;    // rows in the chunk, 1..chunk_max_rows
  int32_t pad;
};

constexpr int kRouteThreads = 256;            // threads per route-sort block
constexpr int kRouteTileTiny = 512;          // routing entries per route-sort block, n <= 16384
constexpr int kRouteTileSmall = 1024;         // n <= 65536
constexpr int kRouteTileLarge = 2048;         // and above (keeps the tile table at (E+1)*n/2048)
inline int route_tile(int64_t n) {
  return n <= 16384 ? kRouteTileTiny : n <= 65536 ? kRouteTileSmall : kRouteTileLarge;
}
constexpr int64_t kSmallMaxN = 4096;          // unsorted calls up to this size: one route block
constexpr int64_t kTinyMaxN = 256;            // ... and up to this size: one entry per thread
constexpr int kChunkRowsWide = 256;           // tokens per work unit, wide GEMM variant
constexpr int kChunkRowsPair = 512;           // tokens per work unit, wide GEMM on CTA pairs
constexpr int kChunkRowsMid = 128;            // tokens per work unit, mid GEMM variant
constexpr int kMidMaxAvgRows = 64;            // ... taken up to this many rows per expert on average
constexpr int kChunkRowsNarrow = 32;          // tokens per work unit, narrow GEMM variant
constexpr int kMaxExperts = GQMM_MAX_EXPERTS;
constexpr int kUnitRows = 256;                // weight rows per work unit (two 128-row tiles)
constexpr int kTargetUnits = 2 * 152;         // split K until about this many units exist
constexpr int64_t kSplitMaxRows = 1024;       // split K only for decode-sized calls: the fp32
                                              // partial sums cost n*F*4 bytes per slice

constexpr int kFusedPlanMaxRows = 64;        // routed streaming calls of up to this many rows
                                              // (unsorted) are planned inside the kernel
constexpr int kStreamMaxRows = 8;             // weight-streaming path: a dense call of <= 8 rows,
constexpr int kStreamMoeRows = 2;             // or a routed call in chunks of <= 2 rows

// Rows per chunk of the work list for n routed rows over E experts, a pure function of (n, E)
// so the workspace size (which depends on it) is known before any device work:
//   up to 8 for decode-sized calls (the weight-streaming path: one dense call of n <= 8 rows,
//   or at most 1.5 rows per hit expert on average in chunks of 2, so a second row of an expert
//   does not stream its weights again), else 32 (narrow: at most 32 rows per expert on average),
//   128 (mid: at most 64) or 256 (wide).
inline int chunk_rows_for(int64_t n, int E) {
  const int64_t busy = n < E ? n : E;  // experts that can have rows
  if (busy <= 0) return kChunkRowsWide;
  if (E == 1) {
    if (n <= kStreamMaxRows) return (int)n;
  } else {
    if (2 * n <= 3 * busy) return kStreamMoeRows;
  }
  const int64_t avg = (n + busy - 1) / busy;
  return avg <= kChunkRowsNarrow ? kChunkRowsNarrow : avg <= kMidMaxAvgRows ? kChunkRowsMid : kChunkRowsWide;
}

// How a call is split into work units.  A pure function of the sizes.
struct UnitShape {
  int chunk_rows;  // chunk_rows_for(n, E)
  int ksplit;      // K slices per (chunk, F pair); 1 = no split
  bool stream;     // weight-streaming path (chunk_rows <= kStreamMaxRows and H supported)
};

// Largest K split a call of these sizes may use before the per-H cap (which only lowers it):
// for decode-sized calls with fewer than kTargetUnits units, ceil(2 kTargetUnits / units), at
// most 16; the plan step picks the split within this bound from the actual chunk count.
// The workspace holds this many partial-sum planes.
inline int ksplit_bound(int64_t n, int F, int E, int* chunk_rows_out) {
  const int64_t busy = n < E ? n : E;                  // experts that can have rows
  const int rows = chunk_rows_for(n, E);
  if (chunk_rows_out) *chunk_rows_out = rows;
  const int64_t units = (busy + n / rows) * ((F + kUnitRows - 1) / kUnitRows);  // upper bound
  if (n > kSplitMaxRows || units <= 0 || units >= kTargetUnits) return 1;
  const int64_t ks = (2 * kTargetUnits + units - 1) / units;
  return (int)(ks < 16 ? ks : 16);
}

bool gemv_supported(int rows, int H, int E);

inline UnitShape unit_shape(int64_t n, int H, int F, int E) {
  UnitShape u;
  const int ks = ksplit_bound(n, F, E, &u.chunk_rows);
  u.stream = u.chunk_rows <= kStreamMaxRows && gemv_supported(u.chunk_rows, H, E);
  const int G = H / 64;
  const int ks_max = G / 4 > 1 ? (G / 4 < 16 ? G / 4 : 16) : 1;  // keep >= 4 K blocks per slice
  u.ksplit = ks < ks_max ? ks : ks_max;
  return u;
}

struct WsLayout {
  size_t perm, offsets, tile_hist, chunks, acc, total;
  int64_t n_tiles, max_chunks;
  bool has_acc;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// allow_split = false lays out a workspace for calls that never split K (no sum buffer).
inline WsLayout ws_layout(int64_t n, int F, int E, bool allow_split = true) {
  WsLayout L;
  L.n_tiles = (n + route_tile(n) - 1) / route_tile(n);
  if (L.n_tiles < 1) L.n_tiles = 1;
  // chunks of at most 32 rows where the format has only the narrow variant (or fewer rows)
  const int crows = chunk_rows_for(n, E);
  L.max_chunks = E + n / (crows < kChunkRowsNarrow ? crows : kChunkRowsNarrow) + 1;
  const int ks = allow_split ? ksplit_bound(n, F, E, nullptr) : 1;
  L.has_acc = ks > 1;
  size_t off = sizeof(WsHeader);
  L.perm = off;
  off = align256(off + sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  L.offsets = off;
  off = align256(off + sizeof(int32_t) * (size_t)(E + 1));
  L.tile_hist = off;
  off = align256(off + sizeof(uint32_t) * (size_t)(E + 1) * (size_t)L.n_tiles);
  L.chunks = off;
  off = align256(off + sizeof(Chunk) * (size_t)L.max_chunks);
  L.acc = off;
  if (L.has_acc) off = align256(off + sizeof(float) * (size_t)ks * (size_t)n * (size_t)F);
  L.total = off;
  return L;
}

// Records a printf-style message as the calling thread's gqmm_last_error() and returns code.
int report_error(int code, const char* fmt, ...);

// gqmm_gather_qmm with two switches: allow_split = false never splits K, so its workspace needs
// no split-K sum buffer (ws_layout(n, F, E, false)); clear_header = true zeroes the workspace's
// 256-byte header (status word included) on the stream once every argument has been validated,
// before the first kernel.
int gather_qmm_impl(const void* x, const void* wq, const void* scales, const void* biases, const uint32_t* idx,
                    int64_t T, int A, int H, int F, int E, int group_size, int bits, int sorted, int x_shared,
                    void* y, void* ws, size_t ws_bytes, cudaStream_t s, bool allow_split, bool clear_header = false,
                    int kind = 0, const float* tscale = nullptr);


// ------------------------------------------------------------------------------------------
// Kernel launchers (defined in the .cu files).  All return cudaError_t of the launch.
// ------------------------------------------------------------------------------------------
cudaError_t launch_quantize(const __nv_bfloat16* w, int64_t rows, int64_t H, int group_size, int bits, uint8_t* wq,
                            __nv_bfloat16* scales, __nv_bfloat16* biases, cudaStream_t s);
// Block-scaled floating-point quantization (kind 1 mxfp4, 2 nvfp4, 3 mxfp8; formats.cuh).
cudaError_t launch_quantize_fp(const __nv_bfloat16* w, int64_t rows, int64_t H, int64_t rows_per_tensor, int kind,
                               uint8_t* wq, uint8_t* scales, float* tscale, cudaStream_t s);

struct RouteArgs {
  const uint32_t* idx;  // NULL: dense (E == 1, every row in expert 0)
  int64_t n;
  int E;
  int sorted;           // 1: caller promises nondecreasing idx
  int32_t* perm;        // sorted position -> flat row (unused when rows keep their order)
  int32_t* offsets;     // [E + 1]
  uint32_t* tile_hist;
  Chunk* chunks;        // NULL: no work list wanted (standalone route sort)
  WsHeader* header;
  __nv_bfloat16* y;     // rows with an invalid index are zero-filled here (may be NULL)
  int F;
  int64_t n_tiles;
  int chunk_rows;       // longest chunk of the work list
  int n_fpairs;         // 256-row output tiles per expert (work units per chunk and K slice)
  int ks_cap;           // largest K split the workspace and H allow (1: never split)
  int sms;              // unit workers of the grouped GEMM (its CTAs, or CTA pairs: gemm_tc_workers)
};
// Unsorted: histogram kernel + scan/scatter/plan kernel.  Sorted or dense: one plan kernel.
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, int* kernels_launched);

struct GemmArgs {
  const __nv_bfloat16* x;
  int64_t n;            // rows of x
  const uint8_t* wq;
  const __nv_bfloat16* scales;
  const __nv_bfloat16* biases;
  __nv_bfloat16* y;
  const int32_t* perm;  // rows of x: NULL means sorted position == row of x
  const int32_t* y_perm;  // rows of y: NULL means sorted position == row of y
  const Chunk* chunks;
  WsHeader* header;
  float* acc;           // [ksplit, n, F] split-K partial sums (ks_cap > 1)
  const int32_t* offsets;  // [E + 1]; offsets[E] = valid sorted positions (split-K finalize)
  int H, F, E;
  int chunk_rows;       // rows per chunk: <= kChunkRowsNarrow selects the narrow variant, kChunkRowsMid
                        // the mid one (4-bit affine codes; other formats run such chunks on the wide one)
  int ks_cap;           // > 1: the plan step may split K (header->ksplit) and the finalize runs
  int dense_plan;       // 1: idx is NULL, so the plan is the single chunk (expert 0, start 0, n rows)
  int group_size = 64;  // quantization group along H: 32, 64 or 128 (the streaming kernels: 64)
  int kind = 0;         // weight format (formats.cuh): 0 affine, 1 mxfp4, 2 nvfp4, 3 mxfp8, 4 affine transpose=False
  int bits = 4;         // affine code width: 2, 3, 4, 5, 6 or 8
  const float* tscale = nullptr;  // nvfp4: float32 scale per expert [E]
  int test_stall = 0;   // 1: leave the first k-block's codes uncopied (gqmm_test_stall_next)
  int x_div = 1;        // x row of routed row r: r / x_div (A when the A rows of a token share
                        // one x row, else 1); x has n / x_div rows
  const uint32_t* idx = nullptr;  // routing entries [n] (fused_plan calls)
  int fused_plan = 0;   // 1: a routed decode call (n <= kFusedPlanMaxRows, unsorted) that the
                        // weight-streaming kernel plans itself; no route kernel runs before it
};
// Launches the grouped GEMM (and, when ks_cap > 1, the kernel that turns the partial sums into
// y).  *launched gets the number of kernels enqueued.
cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t s, int* launched);
// Streaming multiprocessors of the current device (queried once per device).
cudaError_t device_sm_count(int* sms);
// Unit workers of the grouped GEMM instance a call of this format and chunk size runs on: the
// CTAs (one per SM), or the CTA pairs of the 4-bit affine pair instance.  The plan step starts
// the GEMM's unit counter (WsHeader::next_unit) at this number.
cudaError_t gemm_tc_workers(int kind, int bits, int chunk_rows, int* workers);
// The chunk size a gather call of n routed rows over E experts uses: kChunkRowsPair for wide 4-bit
// affine calls with more than kChunkRowsWide rows per expert on average (whose experts would
// otherwise be split into several chunks, each dequantizing the expert's weights again) when the
// device runs the pair instance, else chunk_rows.
cudaError_t gemm_tc_chunk_rows(int kind, int bits, int chunk_rows, int64_t n, int E, int* out);

// The weight-streaming kernels for chunks of at most `rows` rows: the CUDA-core kernel (two blocks
// per SM) for routed chunks of 1 or 2 rows and single-row dense calls, the MMA kernel (one block
// per SM) for dense calls of 2 to 8 rows.
bool gemv_fma_supported(int rows, int H);
cudaError_t launch_gemv_fma(const GemmArgs& a, int rows, int sms, cudaStream_t s);
bool gemv_mma_supported(int rows, int H);
cudaError_t launch_gemv_mma(const GemmArgs& a, int rows, int sms, cudaStream_t s);
cudaError_t launch_gemv(const GemmArgs& a, int rows, int sms, cudaStream_t s);
bool gemv_uses_mma(int rows, int H, int E);  // which of the two launch_gemv runs

cudaError_t launch_gemm_simt(const __nv_bfloat16* x, const uint8_t* wq,
                             const __nv_bfloat16* scales, const __nv_bfloat16* biases,
                             const uint32_t* idx, int64_t n, int H, int F, int E, int group_size, int x_div,
                             __nv_bfloat16* y, cudaStream_t s);

// ------------------------------------------------------------------------------------------
// Device helpers: PTX wrappers for mbarrier, TMA, cp.async and tcgen05.
// ------------------------------------------------------------------------------------------
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// kCluster: acquire at cluster scope, for barriers that threads of the other CTA of a pair
// arrive on after writing data the waiter reads.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kCluster) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  }
  return ok != 0;
}

// Upper bound on any single wait inside a kernel.  A correct launch never gets near it;
// hitting it means a producer is missing, and the kernel then unwinds instead of hanging.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Bounded wait for the phase of parity `parity` of barrier `bar` to complete.  Returns
// false if the CTA-wide abort flag is raised or the limit passes (which raises the flag and
// records GQMM_STATUS_TIMEOUT).
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status) {
  if (mbar_try_wait<kCluster>(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait<kCluster>(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(status, GQMM_STATUS_TIMEOUT);
        return false;
      }
    }
  }
}

// Wait used only while unwinding after an abort: bounded, ignores the abort flag.
__device__ __forceinline__ bool mbar_wait_unwind(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async proxy
// (the tensor core reads its operands through the async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled TMA load global -> shared, completion counted on an mbarrier in bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Four rows (r0..r3) of one box-wide column slice starting at element c0, written as four
// consecutive box rows at dst (tile::gather4; the map's box must be one row high).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                                            int32_t r0, int32_t r1, int32_t r2, int32_t r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization
// may start before the previous kernel of the stream ends.  It must wait before it reads
// what that kernel writes; the previous kernel lets it start early by triggering.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Bulk prefetch of [src, src + bytes) into L2 (src 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared of `bytes` bytes (both addresses 16-byte aligned, bytes a
// multiple of 16), completion counted on an mbarrier in bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Named barrier `id` over `nthreads` threads (a multiple of 32) that also ORs `v` over them.
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Wait until at most n (0..7, clamped) of this thread's most recent cp.async groups are pending.
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<7>(); break;
  }
}
// Arrive (without raising the expected count) on `bar` once all of this thread's prior
// cp.async copies have completed.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// ---- tcgen05 (5th-generation tensor core, accumulators in tensor memory) ----

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, f32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// ---- CTA pairs (a cluster of two CTAs on two SMs sharing one MMA: cta_group::2) ----
// The pair's tensor memory is allocated, used and freed with .cta_group::2 throughout: one warp
// of each CTA allocates (collectively), the even CTA issues the MMAs, whose M = 256 rows are the
// even CTA's 128 A rows then the odd CTA's 128, and whose N columns of B are split in halves, the
// first half in the even CTA's shared memory; each CTA's tensor memory holds its own 128 rows of
// the accumulator.  Both CTAs keep operands, barriers and the TMEM address at the same offsets.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of this CTA's shared-memory location `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on a barrier of another CTA of the cluster; this thread's earlier writes (including
// remote ones) are released to the barrier's waiters at cluster scope.  (Costly: the release waits
// for the thread's outstanding writes; used once per work unit.)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Arrive on a barrier of another CTA of the cluster with the default (CTA-scope) semantics: a
// signal that the data it guards is complete, for data the tensor core or the tensor memory
// holds (per-stage and per-accumulator handshakes of a CTA pair).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// Every thread of both CTAs: barrier.cluster (arrive with release, wait with acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T over the pair (M = 256), bf16 in, f32 accumulate.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the barrier at offset `bar` in each CTA of `cta_mask` when every tcgen05
// operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// The same wait, with the loaded registers as operands: their uses cannot be scheduled before it.
__device__ __forceinline__ void tc_wait_ld_regs(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte-swizzle canonical
// layout: rows of 64 bf16 (128 bytes), 8-row groups 1024 bytes apart, 16-byte chunks of
// row r stored at chunk position (c ^ (r % 8)).  The tile must start 1024-byte aligned.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);       // start address, bits 0-13
  d |= (uint64_t)(16u >> 4) << 16;                    // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;                  // stride byte offset: 8-row group pitch
  d |= (uint64_t)1 << 46;                             // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;                             // layout: 128-byte swizzle
  return d;
}

// Shared-memory matrix descriptor for a K-major operand without swizzle: core matrices of 8 rows x
// 16 bytes stored as 128 contiguous bytes; the 16-byte chunks of a row are 128 bytes apart
// (leading byte offset), 8-row groups 1024 bytes apart (stride byte offset): a 128 x 64 bf16
// tile, chunk c of row r at (r / 8) * 1024 + c * 128 + (r % 8) * 16.
__device__ __forceinline__ uint64_t umma_desc_kmajor_interleave(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);       // start address, bits 0-13
  d |= (uint64_t)(128u >> 4) << 16;                   // leading byte offset: K-adjacent chunks
  d |= (uint64_t)(1024u >> 4) << 32;                  // stride byte offset: 8-row group pitch
  d |= (uint64_t)1 << 46;                             // descriptor version (tcgen05); layout 0: no swizzle
  return d;
}

// The same for an MN-major operand in the 128-byte-swizzle canonical layout: atoms of 8 k-rows
// x 64 bf16 along M/N (1024 bytes, 16-byte chunk c of k-row r at chunk position c ^ (r % 8)),
// atoms adjacent along M/N `lbo` bytes apart and atoms adjacent along K (8-row groups) `sbo`
// bytes apart.
__device__ __forceinline__ uint64_t umma_desc_sw128_mn(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);       // start address, bits 0-13
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;        // leading byte offset: M/N atom pitch
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;        // stride byte offset: 8-row group pitch
  d |= (uint64_t)1 << 46;                             // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;                             // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B, f32 D, both operands K-major.
__device__ __forceinline__ uint32_t umma_idesc_bf16(int M, int N) {
  uint32_t d = 0;
  d |= 1u << 4;                          // D format: f32
  d |= 1u << 7;                          // A format: bf16
  d |= 1u << 10;                         // B format: bf16
  d |= (uint32_t)(N >> 3) << 17;         // N / 8
  d |= (uint32_t)(M >> 4) << 24;         // M / 16
  return d;
}
constexpr uint32_t kIdescTransposeA = 1u << 15;  // A is MN-major
constexpr uint32_t kIdescTransposeB = 1u << 16;  // B is MN-major

#endif  // __CUDACC__

}  // namespace gqmm

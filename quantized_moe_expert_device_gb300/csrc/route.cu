// On-device routing: stable counting sort of the routing entries by expert and the
// grouped-GEMM work list built from the resulting segments.
//
// mlxcel #629 "perf(cuda/moe): fix MoE prefill collapse", implementation plan items 2 and
// 4b: host-side sorting/segmentation can serialize the prefill path; sorting tokens by
// expert on the device gives every expert one contiguous block of rows for a single grouped
// GEMM launch.
//
// Unsorted idx (two kernels, no host round trip):
//   1. route_hist:     one block per tile of kRouteTile entries; per-key counts in shared
//                      memory (keys >= E are folded into an extra key E) written key-major.
//   2. route_scatter:  every block scans the key-major table itself (warp-shuffle scan), so
//                      no block waits on another; then it ranks its tile's entries stably
//                      (warp match + per-warp counts) and writes perm.  Block 0 also writes
//                      offsets and the work list.
// Caller-sorted or dense idx: route_plan_sorted finds segment boundaries by binary search,
// checks the sorted promise and writes the work list (one kernel).
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

constexpr int kWarps = kRouteThreads / 32;

// Block-wide exclusive scan of one value per thread using warp shuffles.  `warp_tot` is
// shared scratch of at least NT/32 entries.  Returns the exclusive prefix; *total gets the sum.
template <int NT>
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* warp_tot, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int64_t o = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    constexpr int NW = NT / 32;
    int64_t w = lane < NW ? warp_tot[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t o = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += o;
    }
    if (lane < NW) warp_tot[lane] = w;  // inclusive prefix over warps
  }
  __syncthreads();
  const int64_t warp_prefix = warp == 0 ? 0 : warp_tot[warp - 1];
  *total = warp_tot[NT / 32 - 1];
  __syncthreads();  // warp_tot may be reused by the caller right after
  return warp_prefix + inc - v;
}

// Writes the chunk list for experts [0, E) whose segment e is [seg_start[e], seg_start[e] +
// seg_len[e]).  A segment longer than max_rows is split into equal chunks (sizes differ by at
// most one row) so no chunk leaves most of an MMA tile empty.  Called by one block.
template <int NT>
__device__ void write_plan(const int32_t* seg_start, const int32_t* seg_len, int E, int max_rows, Chunk* chunks,
                           WsHeader* header, int64_t* warp_tot) {
  // Each thread owns a contiguous run of experts so one scan orders all chunks by expert.
  const int per = (E + NT - 1) / NT;
  const int e0 = threadIdx.x * per;
  const int e1 = min(E, e0 + per);
  int64_t my = 0;
  for (int e = e0; e < e1; ++e) my += (seg_len[e] + max_rows - 1) / max_rows;
  int64_t total;
  int64_t at = block_exclusive_scan<NT>(my, warp_tot, &total);
  for (int e = e0; e < e1; ++e) {
    const int len = seg_len[e];
    const int nch = (len + max_rows - 1) / max_rows;
    if (nch == 0) continue;
    const int base = len / nch, rem = len % nch;
    for (int k = 0; k < nch; ++k) {
      Chunk c;
      c.expert = e;
      c.start = seg_start[e] + k * base + min(k, rem);
      c.rows = base + (k < rem ? 1 : 0);
      c.pad = 0;
      chunks[at++] = c;
    }
  }
  if (threadIdx.x == 0) header->n_chunks = (int32_t)total;
}

__device__ __forceinline__ void zero_row(__nv_bfloat16* y, int64_t row, int F) {
  uint4* p = reinterpret_cast<uint4*>(y + row * F);
  for (int c = 0; c < F / 8; ++c) p[c] = make_uint4(0, 0, 0, 0);
}

__global__ void __launch_bounds__(kRouteThreads) route_hist(RouteArgs a) {
  __shared__ uint32_t h[kMaxExperts + 1];
  const int E = a.E;
  for (int k = threadIdx.x; k <= E; k += kRouteThreads) h[k] = 0;
  __syncthreads();
  const int64_t begin = (int64_t)blockIdx.x * kRouteTile;
  const int64_t end = min(a.n, begin + kRouteTile);
  int bad = 0;
  for (int64_t i = begin + threadIdx.x; i < end; i += kRouteThreads) {
    uint32_t key = __ldg(a.idx + i);
    if (key >= (uint32_t)E) {
      key = (uint32_t)E;
      bad = 1;
    }
    atomicAdd(&h[key], 1u);
  }
  bad = __syncthreads_or(bad);
  for (int k = threadIdx.x; k <= E; k += kRouteThreads)
    a.tile_hist[(int64_t)k * a.n_tiles + blockIdx.x] = h[k];
  if (bad && threadIdx.x == 0) atomicOr(&a.header->status, GQMM_STATUS_BAD_INDEX);
}

__global__ void __launch_bounds__(kRouteThreads) route_scatter(RouteArgs a) {
  __shared__ int32_t base[kMaxExperts + 1];      // next perm position for each key, this tile
  __shared__ int32_t seg_start[kMaxExperts + 1]; // first perm position of each key
  __shared__ int32_t seg_len[kMaxExperts + 1];   // rows of each key
  __shared__ int32_t wc[kWarps][kMaxExperts + 2];  // per-warp counts in the current round
  __shared__ int64_t warp_tot[32];

  const int E = a.E;
  const int tile = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // 1. key totals over all tiles and this tile's preceding count, one contiguous key run
  //    per thread, then a block scan over keys gives each key's segment start.
  const int keys = E + 1;
  const int per = (keys + kRouteThreads - 1) / kRouteThreads;
  const int k0 = threadIdx.x * per, k1 = min(keys, k0 + per);
  int64_t my_total = 0;
  for (int k = k0; k < k1; ++k) {
    const uint32_t* row = a.tile_hist + (int64_t)k * a.n_tiles;
    int64_t tot = 0, before = 0;
    for (int64_t t = 0; t < a.n_tiles; ++t) {
      const uint32_t c = row[t];
      tot += c;
      if (t < tile) before += c;
    }
    seg_len[k] = (int32_t)tot;
    base[k] = (int32_t)before;
    my_total += tot;
  }
  int64_t total;
  int64_t run = block_exclusive_scan<kRouteThreads>(my_total, warp_tot, &total);
  for (int k = k0; k < k1; ++k) {
    seg_start[k] = (int32_t)run;
    base[k] += (int32_t)run;
    run += seg_len[k];
  }
  for (int w = 0; w < kWarps; ++w)
    for (int k = threadIdx.x; k <= E + 1; k += kRouteThreads) wc[w][k] = 0;
  __syncthreads();

  if (tile == 0) {
    for (int k = threadIdx.x; k <= E; k += kRouteThreads) a.offsets[k] = seg_start[k];
  }

  // 2. stable scatter: rounds of kRouteThreads consecutive entries.  Within a warp the rank
  //    comes from the match mask; across warps from the per-warp counts of earlier warps.
  const int64_t tile_begin = (int64_t)tile * kRouteTile;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r = 0; r < kRouteTile / kRouteThreads; ++r) {
    const int64_t i = tile_begin + (int64_t)r * kRouteThreads + threadIdx.x;
    const bool valid = i < a.n;
    uint32_t key = (uint32_t)E + 1u;  // sentinel for entries past n: never stored
    if (valid) {
      key = __ldg(a.idx + i);
      if (key > (uint32_t)E) key = (uint32_t)E;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(peers & lt_mask);
    const int cnt = __popc(peers);
    if (valid && rank == 0) wc[warp][key] = cnt;
    __syncthreads();
    if (valid) {
      int pre = 0;
      for (int w = 0; w < warp; ++w) pre += wc[w][key];
      a.perm[base[key] + pre + rank] = (int32_t)i;
      if (key == (uint32_t)E && a.y != nullptr) zero_row(a.y, i, a.F);
    }
    __syncthreads();
    if (valid && rank == 0) {
      atomicAdd(&base[key], cnt);
      wc[warp][key] = 0;
    }
    __syncthreads();
  }

  // 3. work list (block 0)
  if (tile == 0 && a.chunks != nullptr) write_plan<kRouteThreads>(seg_start, seg_len, E, a.chunk_rows, a.chunks, a.header, warp_tot);
}

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) route_plan_sorted(RouteArgs a) {
  __shared__ int32_t seg_start[kMaxExperts + 1];
  __shared__ int32_t seg_len[kMaxExperts + 1];
  __shared__ int64_t warp_tot[32];
  const int E = a.E;
  const int64_t n = a.n;

  int bad = 0, unsorted = 0;
  if (a.idx != nullptr) {
    for (int64_t i = threadIdx.x; i < n; i += kPlanThreads) {
      const uint32_t v = __ldg(a.idx + i);
      if (v >= (uint32_t)E) {
        bad = 1;
        if (a.y != nullptr) zero_row(a.y, i, a.F);
      }
      if (i + 1 < n && v > __ldg(a.idx + i + 1)) unsorted = 1;
    }
  }
  bad = __syncthreads_or(bad);
  unsorted = __syncthreads_or(unsorted);
  if (threadIdx.x == 0) {
    uint32_t bits = (bad ? GQMM_STATUS_BAD_INDEX : 0u) | (unsorted ? GQMM_STATUS_NOT_SORTED : 0u);
    if (bits) atomicOr(&a.header->status, bits);
  }
  if (unsorted) {  // the promise is broken: no segments can be trusted, compute nothing
    for (int e = threadIdx.x; e <= E; e += kPlanThreads) a.offsets[e] = 0;
    if (threadIdx.x == 0) a.header->n_chunks = 0;
    return;
  }
  // Segment starts: first row whose (clamped) key is >= e.
  for (int e = threadIdx.x; e <= E; e += kPlanThreads) {
    int64_t lo = 0, hi = n;
    if (a.idx == nullptr) {
      lo = (e == 0) ? 0 : n;
    } else {
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        uint32_t v = __ldg(a.idx + mid);
        if (v > (uint32_t)E) v = (uint32_t)E;
        if (v < (uint32_t)e) lo = mid + 1; else hi = mid;
      }
    }
    seg_start[e] = (int32_t)lo;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kPlanThreads) seg_len[e] = seg_start[e + 1] - seg_start[e];
  for (int e = threadIdx.x; e <= E; e += kPlanThreads) a.offsets[e] = seg_start[e];
  __syncthreads();
  if (a.chunks != nullptr) write_plan<kPlanThreads>(seg_start, seg_len, E, a.chunk_rows, a.chunks, a.header, warp_tot);
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, int* kernels_launched) {
  *kernels_launched = 0;
  if (a.idx != nullptr && !a.sorted) {
    const unsigned tiles = (unsigned)a.n_tiles;
    route_hist<<<tiles, kRouteThreads, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    route_scatter<<<tiles, kRouteThreads, 0, s>>>(a);
    *kernels_launched = 2;
    return cudaGetLastError();
  }
  route_plan_sorted<<<1, kPlanThreads, 0, s>>>(a);
  *kernels_launched = 1;
  return cudaGetLastError();
}

}  // namespace gqmm

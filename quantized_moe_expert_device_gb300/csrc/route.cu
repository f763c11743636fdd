// On-device routing: stable counting sort of the routing entries by expert and the
// grouped-GEMM work list built from the resulting segments.
//
// mlxcel #629 "perf(cuda/moe): fix MoE prefill collapse", implementation plan items 2 and
// 4b: host-side sorting/segmentation can serialize the prefill path; sorting tokens by
// expert on the device gives every expert one contiguous block of rows for a single grouped
// GEMM launch.
//
// Unsorted idx, decode-sized calls (n <= kTinyMaxN, E <= kSmallMaxE): route_tiny, one block,
// one entry per thread, ranks by loops over the keys in shared memory.
// Unsorted idx, small calls (n <= kSmallMaxN, E <= kSmallMaxE): route_small, one block of
// 1024 threads.  Each warp owns a contiguous range of entries and holds its keys in registers;
// pass 1 counts keys per warp (warp match, no atomics), one scan over (key, warp) gives every
// warp its first position per key, and pass 2 ranks the warp's entries in order.  Three block
// barriers in all, and the index array is read once.
// Unsorted idx, larger calls (two kernels, no host round trip):
//   1. route_hist:     one block per tile of TILE entries (512, 1024 or 2048 by n); per-key
//                      counts in shared memory (keys >= E are folded into an extra key E)
//                      written key-major.
//   2. route_scatter:  every block scans the key-major table itself (warp-shuffle scan), so
//                      no block waits on another; then it ranks its tile's entries stably with
//                      the same per-warp scheme and writes perm.  One extra block writes
//                      offsets and the work list meanwhile.
// The sort is stable: entries of one expert keep their order of flat index.
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

// K slices per (chunk, F pair) for n_units0 = chunks x F pairs work units on `sms` unit workers
// (CTAs or CTA pairs): the split (at most ks_cap) that minimises the waves of units per worker per
// unit of work,
// ceil(n_units0 * ks / sms) / ks, taken only when it saves at least a tenth.
__device__ __forceinline__ int choose_ksplit(int64_t n_units0, int ks_cap, int sms) {
  if (n_units0 <= 0 || ks_cap <= 1 || sms <= 0) return 1;
  int best = 1;
  int64_t best_w = (n_units0 + sms - 1) / sms;
  for (int ks = 2; ks <= ks_cap; ++ks) {
    const int64_t w = (n_units0 * ks + sms - 1) / sms;
    if (w * best * 10 <= best_w * ks * 9) {  // w / ks <= 0.9 * best_w / best
      best = ks;
      best_w = w;
    }
  }
  return best;
}

// Writes the chunk list for experts [0, E) whose segment e is [seg_start[e], seg_start[e] +
// seg_len[e]).  A segment longer than max_rows is split into equal chunks (sizes differ by at
// most one row) so no chunk leaves most of an MMA tile empty.  Chunks are stored largest
// first (a counting sort on the row count; the order among chunks of one size is arbitrary
// and does not affect any result), so the GEMM's schedulers hand out the big units first.
// Also writes the header fields the GEMM reads: chunk count, K split, zeroed work counter.
// Called by one whole block of NT threads.
template <int NT>
__device__ void write_plan(const int32_t* seg_start, const int32_t* seg_len, int E, int max_rows, Chunk* chunks,
                           WsHeader* header, int64_t* warp_tot, int n_fpairs, int ks_cap, int sms) {
  static_assert(NT >= kChunkRowsWide, "one thread per size bucket");
  // chunks with max_rows - b rows (with max_rows - 2b or - 2b - 1 rows for the CTA pairs' chunks of
  // up to 512 rows), then cursors
  __shared__ int32_t bucket[kChunkRowsWide];
  const int sh = max_rows > kChunkRowsWide ? 1 : 0;
  const int nb = ((max_rows - 1) >> sh) + 1;
  for (int b = threadIdx.x; b < kChunkRowsWide; b += NT) bucket[b] = 0;
  __syncthreads();
  const int per = (E + NT - 1) / NT;
  const int e0 = threadIdx.x * per;
  const int e1 = min(E, e0 + per);
  for (int e = e0; e < e1; ++e) {
    const int len = seg_len[e];
    const int nch = (len + max_rows - 1) / max_rows;
    if (nch == 0) continue;
    const int base = len / nch, rem = len % nch;  // rem chunks of base + 1 rows, the rest base
    if (rem) atomicAdd(&bucket[(max_rows - (base + 1)) >> sh], rem);
    if (nch > rem) atomicAdd(&bucket[(max_rows - base) >> sh], nch - rem);
  }
  __syncthreads();
  int64_t total;
  const int64_t at = block_exclusive_scan<NT>(threadIdx.x < nb ? bucket[threadIdx.x] : 0, warp_tot, &total);
  if (threadIdx.x < nb) bucket[threadIdx.x] = (int32_t)at;
  __syncthreads();
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
      chunks[atomicAdd(&bucket[(max_rows - c.rows) >> sh], 1)] = c;
    }
  }
  if (threadIdx.x == 0) {
    header->n_chunks = (int32_t)total;
    header->ksplit = choose_ksplit(total * (int64_t)n_fpairs, ks_cap, sms);
    header->next_unit = sms;  // units below the worker count go to the worker of that index first
  }
}

__device__ __forceinline__ void zero_row(__nv_bfloat16* y, int64_t row, int F) {
  uint4* p = reinterpret_cast<uint4*>(y + row * F);
  for (int c = 0; c < F / 8; ++c) p[c] = make_uint4(0, 0, 0, 0);
}

// Per-warp stable ranking over a contiguous range [w_begin, w_end) of entries, S rounds of
// 32 (S <= MAXS).  Keys (clamped to E; entries past the range get the sentinel E + 1, which
// is never counted or stored) are loaded once into registers, two 16-bit keys per register
// when PACK (E + 1 < 65536).
template <int MAXS, bool PACK>
struct WarpKeys {
  static constexpr int R = PACK ? (MAXS + 1) / 2 : MAXS;
  uint32_t k[R];
  __device__ __forceinline__ uint32_t get(int j) const {
    return PACK ? (k[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu : k[j];
  }
};

template <int MAXS, bool PACK>
__device__ __forceinline__ WarpKeys<MAXS, PACK> load_warp_keys(const uint32_t* idx, int64_t w_begin,
                                                               int64_t w_end, int S, int E, int* bad) {
  const int lane = threadIdx.x & 31;
  WarpKeys<MAXS, PACK> K;
#pragma unroll
  for (int r = 0; r < WarpKeys<MAXS, PACK>::R; ++r) K.k[r] = 0;
#pragma unroll
  for (int j = 0; j < MAXS; ++j) {
    const int64_t i = w_begin + (int64_t)j * 32 + lane;
    uint32_t key = (uint32_t)E + 1u;
    if (j < S && i < w_end) {
      key = __ldg(idx + i);
      if (key >= (uint32_t)E) {
        key = (uint32_t)E;
        *bad = 1;
      }
    }
    if (PACK)
      K.k[j >> 1] |= key << ((j & 1) * 16);
    else
      K.k[j] = key;
  }
  return K;
}

// Lanes of the warp whose key equals this lane's key, from one ballot per key bit (keys
// below 2^nbits).  Cheaper than a warp match, which is a slow instruction when many warps
// of one SM use it.
__device__ __forceinline__ unsigned warp_peers(uint32_t key, int nbits) {
  unsigned m = 0xffffffffu;
  for (int b = 0; b < nbits; ++b) {
    const uint32_t bit = (key >> b) & 1u;
    const unsigned bb = __ballot_sync(0xffffffffu, bit != 0u);
    m &= bit ? bb : ~bb;
  }
  return m;
}

// bits that hold every key including the sentinel E + 1
__device__ __forceinline__ int key_bits(int E) { return 32 - __clz(E + 1); }

// Pass 1: cnt[key] += entries of this warp with that key (cnt is this warp's private row).
template <int MAXS, bool PACK>
__device__ __forceinline__ void warp_count(const WarpKeys<MAXS, PACK>& K, int S, int E, int32_t* cnt) {
  const int nbits = key_bits(E);
#pragma unroll
  for (int j = 0; j < MAXS; ++j) {
    if (j < S) {
      const uint32_t key = K.get(j);
      const unsigned peers = warp_peers(key, nbits);
      if (key <= (uint32_t)E && (threadIdx.x & 31) == __ffs(peers) - 1) cnt[key] += __popc(peers);
      __syncwarp();
    }
  }
}

// Pass 2: next[key] holds this warp's next perm position for each key.
template <int MAXS, bool PACK>
__device__ __forceinline__ void warp_scatter(const WarpKeys<MAXS, PACK>& K, int S, int E, int64_t w_begin, int32_t* next,
                                             int32_t* perm, __nv_bfloat16* y, int F) {
  const int nbits = key_bits(E);
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < MAXS; ++j) {
    if (j < S) {
      const uint32_t key = K.get(j);
      const unsigned peers = warp_peers(key, nbits);
      const bool valid = key <= (uint32_t)E;
      if (valid) {
        const int64_t i = w_begin + (int64_t)j * 32 + lane;
        perm[next[key] + __popc(peers & lt_mask)] = (int32_t)i;
        if (key == (uint32_t)E && y != nullptr) zero_row(y, i, F);
      }
      __syncwarp();
      if (valid && lane == __ffs(peers) - 1) next[key] += __popc(peers);
      __syncwarp();
    }
  }
}

constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallMaxS = 4;                                   // rounds of 32 per warp
constexpr int kSmallMaxE = 256;
static_assert(kSmallMaxN == (int64_t)kSmallWarps * 32 * kSmallMaxS, "small-route capacity");

__global__ void __launch_bounds__(kSmallThreads) route_small(RouteArgs a) {
  grid_dependents_launch();  // the GEMM may start its prologue; it waits before reading the plan
  __shared__ int32_t wc[kSmallWarps][kSmallMaxE + 2];  // per-warp counts, then next positions
  __shared__ int32_t seg_start[kSmallMaxE + 1];
  __shared__ int32_t seg_len[kSmallMaxE + 1];
  __shared__ int64_t warp_tot[32];
  const int E = a.E;
  const int64_t n = a.n;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kSmallWarps * (kSmallMaxE + 2); i += kSmallThreads) (&wc[0][0])[i] = 0;
  // warp ranges: L entries each, a multiple of 32
  const int64_t L = ((n + kSmallWarps - 1) / kSmallWarps + 31) / 32 * 32;
  const int S = (int)(L / 32);
  const int64_t w_begin = (int64_t)warp * L;
  const int64_t w_end = min(n, w_begin + L);
  int bad = 0;
  const WarpKeys<kSmallMaxS, true> K = load_warp_keys<kSmallMaxS, true>(a.idx, w_begin, w_end, S, E, &bad);
  __syncthreads();
  warp_count(K, S, E, wc[warp]);
  bad = __syncthreads_or(bad);
  // key totals, segment starts (block scan over keys), then per-warp first positions
  const int key = threadIdx.x;
  int64_t tot = 0;
  if (key <= E)
    for (int w = 0; w < kSmallWarps; ++w) tot += wc[w][key];
  int64_t total;
  const int64_t start = block_exclusive_scan<kSmallThreads>(tot, warp_tot, &total);
  if (key <= E) {
    seg_start[key] = (int32_t)start;
    seg_len[key] = (int32_t)tot;
    int32_t run = (int32_t)start;
    for (int w = 0; w < kSmallWarps; ++w) {
      const int32_t c = wc[w][key];
      wc[w][key] = run;
      run += c;
    }
    a.offsets[key] = (int32_t)start;
  }
  if (threadIdx.x == 0 && bad) atomicOr(&a.header->status, GQMM_STATUS_BAD_INDEX);
  __syncthreads();
  warp_scatter(K, S, E, w_begin, wc[warp], a.perm, a.y, a.F);
  if (a.chunks != nullptr) write_plan<kSmallThreads>(seg_start, seg_len, E, a.chunk_rows, a.chunks, a.header, warp_tot,
                                 a.n_fpairs, a.ks_cap, a.sms);
}

// Unsorted idx, decode-sized calls (n <= kTinyMaxN, E <= kSmallMaxE): one block of 256 threads,
// one entry per thread.  Every key's count and first position, and every entry's stable rank
// (keys below its own, plus equal keys at lower flat index), are loops over the n keys held in
// shared memory: two block barriers before the plan, and no atomics.
constexpr int kTinyThreads = 256;
static_assert(kTinyMaxN <= kTinyThreads, "one entry per thread");

__global__ void __launch_bounds__(kTinyThreads) route_tiny(RouteArgs a) {
  grid_dependents_launch();  // the GEMM may start its prologue; it waits before reading the plan
  __shared__ int32_t keys[kTinyThreads];
  __shared__ int32_t seg_start[kSmallMaxE + 1];
  __shared__ int32_t seg_len[kSmallMaxE + 1];
  __shared__ int64_t warp_tot[32];
  const int E = a.E, n = (int)a.n, t = threadIdx.x;
  int key = E, bad = 0;
  if (t < n) {
    const uint32_t k = __ldg(a.idx + t);
    bad = k >= (uint32_t)E;
    key = bad ? E : (int)k;  // invalid indices sort last, as key E
  }
  keys[t] = key;
  bad = __syncthreads_or(bad);
  for (int e = t; e <= E; e += kTinyThreads) {
    int cnt = 0, less = 0;
    for (int i = 0; i < n; ++i) {
      const int k = keys[i];
      cnt += k == e;
      less += k < e;
    }
    seg_start[e] = less;
    seg_len[e] = cnt;
    a.offsets[e] = less;
  }
  if (t < n) {
    int rank = 0;
    for (int i = 0; i < n; ++i) {
      const int k = keys[i];
      rank += k < key || (k == key && i < t);
    }
    a.perm[rank] = t;
    if (key == E && a.y != nullptr) zero_row(a.y, t, a.F);
  }
  if (t == 0 && bad) atomicOr(&a.header->status, GQMM_STATUS_BAD_INDEX);
  __syncthreads();
  if (a.chunks != nullptr) write_plan<kTinyThreads>(seg_start, seg_len, E, a.chunk_rows, a.chunks, a.header, warp_tot,
                                 a.n_fpairs, a.ks_cap, a.sms);
}

template <int TILE>
__global__ void __launch_bounds__(kRouteThreads) route_hist(RouteArgs a) {
  grid_dependents_launch();  // route_scatter may launch now; it waits before reading the table
  __shared__ uint32_t h[kMaxExperts + 1];
  const int E = a.E;
  for (int k = threadIdx.x; k <= E; k += kRouteThreads) h[k] = 0;
  __syncthreads();
  const int64_t begin = (int64_t)blockIdx.x * TILE;
  const int64_t end = min(a.n, begin + TILE);
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

template <int TILE>
__global__ void __launch_bounds__(kRouteThreads) route_scatter(RouteArgs a) {
  grid_dependents_launch();  // the GEMM may start its prologue; it waits before reading the plan
  __shared__ int32_t base[kMaxExperts + 1];      // next perm position for each key, this tile
  __shared__ int32_t seg_start[kMaxExperts + 1]; // first perm position of each key
  __shared__ int32_t seg_len[kMaxExperts + 1];   // rows of each key
  __shared__ int32_t wc[kWarps][kMaxExperts + 2];  // per-warp counts, then next positions
  __shared__ int64_t warp_tot[32];

  const int E = a.E;
  const int tile = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The tile's keys do not come from route_hist: every kernel before it (a plain launch) has
  // completed, so they are loaded before the wait and arrive while it lasts.
  constexpr int kWarpRange = TILE / kWarps;
  constexpr int kS = kWarpRange / 32;
  const int64_t w_begin = (int64_t)tile * TILE + (int64_t)warp * kWarpRange;
  const int64_t w_end = min(a.n, w_begin + kWarpRange);
  int bad = 0;  // already reported by route_hist
  const WarpKeys<kS, false> K = load_warp_keys<kS, false>(a.idx, w_begin, w_end, kS, E, &bad);
  grid_dependency_wait();  // route_hist's table is complete and visible

  // 1. key totals over all tiles and this tile's preceding count: a warp per key, its lanes over
  //    the tiles (coalesced loads, several keys in flight), summed by warp reductions; then a
  //    block scan over keys, one contiguous key run per thread, gives each key's segment start.
  const int keys = E + 1;
  const int64_t n_tiles = a.n_tiles;
  constexpr int kKeysInFlight = 8;  // keys per warp whose loads are issued together
  for (int kb = warp; kb < keys; kb += kKeysInFlight * kWarps) {
    uint32_t tot[kKeysInFlight], before[kKeysInFlight];
#pragma unroll
    for (int j = 0; j < kKeysInFlight; ++j) tot[j] = before[j] = 0u;
    for (int64_t t0 = 0; t0 < n_tiles; t0 += 32) {
      const int64_t t = t0 + lane;
      uint32_t c[kKeysInFlight];
#pragma unroll
      for (int j = 0; j < kKeysInFlight; ++j) {
        const int k = kb + j * kWarps;
        c[j] = (k < keys && t < n_tiles) ? __ldcg(a.tile_hist + (int64_t)k * n_tiles + t) : 0u;
      }
#pragma unroll
      for (int j = 0; j < kKeysInFlight; ++j) {
        tot[j] += c[j];
        before[j] += t < tile ? c[j] : 0u;
      }
    }
#pragma unroll
    for (int j = 0; j < kKeysInFlight; ++j) {
      const int k = kb + j * kWarps;
      const uint32_t s_tot = __reduce_add_sync(0xffffffffu, tot[j]);
      const uint32_t s_before = __reduce_add_sync(0xffffffffu, before[j]);
      if (lane == 0 && k < keys) {
        seg_len[k] = (int32_t)s_tot;
        base[k] = (int32_t)s_before;
      }
    }
  }
  __syncthreads();
  const int per = (keys + kRouteThreads - 1) / kRouteThreads;
  const int k0 = threadIdx.x * per, k1 = min(keys, k0 + per);
  int64_t my_total = 0;
  for (int k = k0; k < k1; ++k) my_total += seg_len[k];
  int64_t total;
  int64_t run = block_exclusive_scan<kRouteThreads>(my_total, warp_tot, &total);
  for (int k = k0; k < k1; ++k) {
    seg_start[k] = (int32_t)run;
    base[k] += (int32_t)run;
    run += seg_len[k];
  }
  if (tile == a.n_tiles) {
    // the plan block (one past the tiles): offsets and the work list, while the others rank
    __syncthreads();
    for (int k = threadIdx.x; k <= E; k += kRouteThreads) a.offsets[k] = seg_start[k];
    if (a.chunks != nullptr) write_plan<kRouteThreads>(seg_start, seg_len, E, a.chunk_rows, a.chunks, a.header, warp_tot,
                                   a.n_fpairs, a.ks_cap, a.sms);
    return;
  }
  for (int w = 0; w < kWarps; ++w)
    for (int k = threadIdx.x; k <= E + 1; k += kRouteThreads) wc[w][k] = 0;

  // 2. stable scatter: warp w ranks the tile's entries [w * kWarpRange, (w + 1) * kWarpRange)
  //    in order (keys loaded above); the per-warp counts of pass 1 give each warp its first
  //    position per key.
  __syncthreads();
  warp_count(K, kS, E, wc[warp]);
  __syncthreads();
  for (int k = threadIdx.x; k <= E; k += kRouteThreads) {
    int32_t run = base[k];
    for (int w = 0; w < kWarps; ++w) {
      const int32_t c = wc[w][k];
      wc[w][k] = run;
      run += c;
    }
  }
  __syncthreads();
  warp_scatter(K, kS, E, w_begin, wc[warp], a.perm, a.y, a.F);
}

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) route_plan_sorted(RouteArgs a) {
  grid_dependents_launch();  // the GEMM may start its prologue; it waits before reading the plan
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
  if (unsorted) {
    // The promise is broken: no segment can be trusted, so nothing is computed and y is
    // defined as all zeros (F is a multiple of 16 and y 16-byte aligned: whole 16-byte stores).
    if (a.y != nullptr) {
      uint4* y4 = reinterpret_cast<uint4*>(a.y);
      const int64_t n16 = n * (int64_t)a.F / 8;
      for (int64_t i = threadIdx.x; i < n16; i += kPlanThreads) y4[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int e = threadIdx.x; e <= E; e += kPlanThreads) a.offsets[e] = 0;
    if (threadIdx.x == 0) {
      a.header->n_chunks = 0;
      a.header->ksplit = 1;
      a.header->next_unit = a.sms;
    }
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
  if (a.chunks != nullptr) write_plan<kPlanThreads>(seg_start, seg_len, E, a.chunk_rows, a.chunks, a.header, warp_tot,
                                 a.n_fpairs, a.ks_cap, a.sms);
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, int* kernels_launched) {
  *kernels_launched = 0;
  if (a.idx != nullptr && !a.sorted && a.n <= kTinyMaxN && a.E <= kSmallMaxE) {
    route_tiny<<<1, kTinyThreads, 0, s>>>(a);
    *kernels_launched = 1;
    return cudaGetLastError();
  }
  if (a.idx != nullptr && !a.sorted && a.n <= kSmallMaxN && a.E <= kSmallMaxE) {
    route_small<<<1, kSmallThreads, 0, s>>>(a);
    *kernels_launched = 1;
    return cudaGetLastError();
  }
  if (a.idx != nullptr && !a.sorted) {
    const unsigned tiles = (unsigned)a.n_tiles;
    const int tile = route_tile(a.n);
    if (tile == kRouteTileTiny)
      route_hist<kRouteTileTiny><<<tiles, kRouteThreads, 0, s>>>(a);
    else if (tile == kRouteTileSmall)
      route_hist<kRouteTileSmall><<<tiles, kRouteThreads, 0, s>>>(a);
    else
      route_hist<kRouteTileLarge><<<tiles, kRouteThreads, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // one block per tile, plus the plan block; launched as a programmatic dependent of
    // route_hist (which starts only after the previous call's kernels, as a plain launch)
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles + 1);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (tile == kRouteTileTiny)
      e = cudaLaunchKernelEx(&cfg, route_scatter<kRouteTileTiny>, a);
    else if (tile == kRouteTileSmall)
      e = cudaLaunchKernelEx(&cfg, route_scatter<kRouteTileSmall>, a);
    else
      e = cudaLaunchKernelEx(&cfg, route_scatter<kRouteTileLarge>, a);
    if (e != cudaSuccess) return e;
    *kernels_launched = 2;
    return cudaGetLastError();
  }
  route_plan_sorted<<<1, kPlanThreads, 0, s>>>(a);
  *kernels_launched = 1;
  return cudaGetLastError();
}

}  // namespace gqmm
